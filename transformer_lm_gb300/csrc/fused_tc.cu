// fused_tc.cu -- the fused operator's matrix product with the fp32 operands
// split into bf16 halves inside the kernel (sm_103a, tcgen05 + TMA).
//
// y = gelu_tanh(x W^T + b) for fp32 x (M, K) and W (N, K) (POPCORNBENCH
// "fused Linear + GELU + Softmax": nn.Linear, then GELU), with, per row and
// column tile, the softmax partials (max, sum exp(y - max)); a second pass
// (softmax_finish_k) normalises the rows. Each fp32 value v is written as
// hi + lo with hi = bf16(v) and lo = bf16(v - hi), and x W^T is taken as
// hi.hi + hi.lo + lo.hi on the bf16 tensor cores with fp32 accumulation: only
// lo.lo and the rounding of lo are left out (about 2^-16 of each product).
//
// A CTA pair computes 256 x BN output tiles (cta_group::2 MMAs; each CTA
// holds 128 rows of x and BN/2 rows of W per stage), persistent over the
// tiles; BN is 256, or 224 where 224-wide tiles fill the last round of CTA
// pairs markedly better (1024 x 8192 outputs: 148 tiles on 76 pairs instead
// of 128):
//   warp 0      TMA: per 64-wide k-block, this CTA's 128 x 64 fp32 tile of x
//               and of W (two 32-column boxes each, 128-byte swizzle) into a
//               stage of the shared-memory ring, completing on a local barrier;
//   warps 10-17 convert each landed stage in place: the 256 bytes of fp32 that
//               row r holds become its 128-byte bf16 hi row (over the first box)
//               and its 128-byte bf16 lo row (over the second), both in the
//               128-byte-swizzled K-major layout the MMA reads; two lanes share
//               a row (one per box) and synchronise between reading and writing;
//               then they signal their CTA's conversion barrier (in the second
//               CTA of the pair, warp 1 forwards each completed phase to the
//               leader's barrier: one cluster-scope arrival per stage instead
//               of one per converter warp);
//   warp 1      (leader) issues the 12 MMAs of a stage (3 products x 4 k-steps
//               of 16) into one of two TMEM accumulators and commits the stage
//               back to both CTAs' producers;
//   warps 2-9   epilogue: bias, GELU, the row partials, fp32 TMA stores.
// Every mbarrier wait is bounded; on expiry the CTA records DEVERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace gk {
namespace fsp {

using namespace tc;

constexpr int BM = 128;                  // rows of x per CTA
constexpr int KB = 64;                   // k-block (fp32 elements per stage)
constexpr int OPB = BM * KB * 4;         // bytes of one operand's fp32 stage tile (32 KB)
constexpr int HALF = OPB / 2;            // one 32-column box; later the hi (or lo) tile
constexpr int STAGE = 2 * OPB;           // x tile, then W tile
constexpr int STAGES = 3;
constexpr int EPI_WARPS = 8, CONV_WARPS = 8;
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int NUM_THREADS = 64 + EPI_THREADS + 32 * CONV_WARPS;
constexpr int STG = 32 * 128;            // an epilogue warp's staging: 32 rows x 32 fp32
constexpr int OFF_EPI = STAGES * STAGE;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * STG;
constexpr int BAR_BYTES = 256 + 1024;    // barriers and flags, then per-row softmax partials
constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
constexpr int TMEM_COLS = 512;           // two accumulators of up to 256 columns
constexpr int GROUP_M = 8;               // m-block pairs per rasterisation group

struct Args {
    int M, N, K;
    int num_mp, num_n, num_kb;
    const float* bias;
    float2* part;
    int part_ld;
    unsigned int* err;
};

DEVI void tile_coords(int st, int num_mp, int num_n, int& mp, int& nb) {
    const int per_group = GROUP_M * num_n;
    const int g = st / per_group, idx = st - g * per_group;
    const int first = g * GROUP_M;
    const int gm = min(GROUP_M, num_mp - first);
    mp = first + idx % gm;
    nb = idx / gm;
}

DEVI void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory"); }

// the fp32 value pair (a, b) as bf16 hi and lo words (low half first)
DEVI void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = f2_h2<bf16>(a, b);
    const float2 h = h2_f2<bf16>(hi);
    lo = f2_h2<bf16>(a - h.x, b - h.y);
}

// BN: output columns per tile (BN / 2 rows of W per CTA)
template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fused_split_gemm_k(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmY, const __grid_constant__ Args a) {
    static_assert(BN % 32 == 0 && BN <= 256 && BN >= 128, "tile width");
    constexpr int BNC = BN / 2;                       // rows of W per CTA
    constexpr int STAGE_TX = OPB + BNC * KB * 4;      // bytes landing per stage
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + OFF_BAR;
    uint8_t* bars_ptr = base_ptr + OFF_BAR;
    auto full = [&](int s) { return bars + 8u * s; };                // TMA landed (local)
    auto conv = [&](int s) { return bars + 8u * (STAGES + s); };     // both CTAs converted (leader)
    auto empty = [&](int s) { return bars + 8u * (2 * STAGES + s); };  // MMAs done reading (both)
    auto tfull = [&](int c) { return bars + 8u * (3 * STAGES + c); };
    auto tempty = [&](int c) { return bars + 8u * (3 * STAGES + 2 + c); };
    const uint32_t drain = bars + 8u * (3 * STAGES + 4);
    constexpr int NBARS = 3 * STAGES + 5;
    static_assert(8 * NBARS + 16 <= 256, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);
    float2* row_part = reinterpret_cast<float2*>(bars_ptr + 256);  // [BM]

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank() & 1u;  // 0: the pair leader (issues the MMAs)
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full(s), 1);
            // leader: its converter warps and the peer's forwarder; peer: its converter warps
            mbar_init(conv(s), rank == 0 ? CONV_WARPS + 1 : CONV_WARPS);
            mbar_init(empty(s), 1);
        }
        for (int c = 0; c < 2; c++) {
            mbar_init(tfull(c), 1);
            mbar_init(tempty(c), 2 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *n_issued_smem = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<2>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    const uint32_t tmem_base = *tmem_slot;
    pdl_enter();
    const int num_tiles = a.num_mp * a.num_n;
    const int cid = (int)blockIdx.x / 2, ncl = (int)gridDim.x / 2;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA loads its own rows)
            int stage = 0, n_issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int st = cid; ok && st < num_tiles; st += ncl) {
                int mp, nb;
                tile_coords(st, a.num_mp, a.num_n, mp, nb);
                const int m0 = (mp * 2 + (int)rank) * BM, n0 = nb * BN + (int)rank * BNC;
                for (int kb = 0; kb < a.num_kb; kb++) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t sx = base + stage * STAGE, sw = sx + OPB;
                    const int k0 = kb * KB;
                    mbar_expect_tx(full(stage), STAGE_TX);
                    tma_load_2d(sx, &tmX, full(stage), k0, m0);
                    tma_load_2d(sx + HALF, &tmX, full(stage), k0 + 32, m0);
                    tma_load_2d(sw, &tmW, full(stage), k0, n0);
                    tma_load_2d(sw + HALF, &tmW, full(stage), k0 + 32, n0);
                    ++n_issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            *n_issued_smem = n_issued;
        }
    } else if (warp == 1) {
        if (rank == 1) {
            // ---------------- forwarder (second CTA): each completed local
            // conversion phase becomes one arrival on the leader's barrier
            const uint32_t conv_leader = mapa_rank(conv(0), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int st = cid; ok && st < num_tiles; st += ncl) {
                for (int kb = 0; kb < a.num_kb; kb++) {
                    if (!mbar_wait_warp(conv(stage), phase, abort_flag)) { ok = false; break; }
                    if (lane == 0) mbar_arrive_cluster(conv_leader + 8u * (uint32_t)stage);
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
        if (rank == 0) {
            // ---------------- MMA issuer (the pair leader, a converged warp)
            const uint32_t id = idesc<0>(0, 0, 2 * BM, BN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int st = cid; st < num_tiles; st += ncl) {
                if (!mbar_wait_warp(tempty(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < a.num_kb; kb++) {
                    if (!mbar_wait_warp(conv(stage), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sx = base + stage * STAGE, sw = sx + OPB;
                    const uint64_t xh = sdesc(sx, 16, 1024), xl = sdesc(sx + HALF, 16, 1024);
                    const uint64_t wh = sdesc(sw, 16, 1024), wl = sdesc(sw + HALF, 16, 1024);
#pragma unroll
                    for (int k = 0; k < 4; k++) {  // 16 k per MMA: 32 bytes = 2 descriptor units
                        const uint32_t first = (kb > 0 || k > 0) ? 1u : 0u;
                        umma_warp<0, 2>(d, xh + 2 * k, wh + 2 * k, id, first);
                        umma_warp<0, 2>(d, xh + 2 * k, wl + 2 * k, id, 1u);
                        umma_warp<0, 2>(d, xl + 2 * k, wh + 2 * k, id, 1u);
                    }
                    umma_commit_warp<2>(empty(stage));  // frees the stage in both CTAs
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_warp<2>(tfull(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else if (warp >= 2 + EPI_WARPS) {
        // ---------------- converters: 16 rows per warp and pass; lanes
        // 0-7 / 16-23 read box 0 of rows j, lanes 8-15 / 24-31 box 1 (so the 8
        // lanes of each shared-memory phase touch 8 different bank groups)
        const int cw = warp - 2 - EPI_WARPS;
        const int box = (lane >> 3) & 1;
        const int rsub = (lane & 7) + ((lane >> 4) << 3);  // row within the warp's 16
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int st = cid; ok && st < num_tiles; st += ncl) {
            for (int kb = 0; kb < a.num_kb; kb++) {
                if (!mbar_wait_warp(full(stage), phase, abort_flag)) { ok = false; break; }
                uint8_t* sp = base_ptr + stage * STAGE;
                // 128 + BNC rows (x then W) in groups of 16: 2 passes of 8 warps
#pragma unroll 1
                for (int pass = 0; pass < 2; pass++) {
                    if ((pass * CONV_WARPS + cw) * 16 >= BM + BNC) continue;  // (warp-uniform)
                    const int row = (pass * CONV_WARPS + cw) * 16 + rsub;  // 0..255
                    uint8_t* op = sp + (row >> 7) * OPB;
                    const int r = row & 127;
                    const int sw = r & 7;
                    uint8_t* src = op + box * HALF + r * 128;
                    float4 f[8];
#pragma unroll
                    for (int c = 0; c < 8; c++) f[c] = *reinterpret_cast<const float4*>(src + ((c ^ sw) << 4));
                    // box b holds k = 32 b .. 32 b + 31: hi/lo chunks 4 b .. 4 b + 3
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        split2(f[c].x, f[c].y, hi[2 * c], lo[2 * c]);
                        split2(f[c].z, f[c].w, hi[2 * c + 1], lo[2 * c + 1]);
                    }
                    __syncwarp();  // both halves of every row are read before either is overwritten
                    uint8_t* dh = op + r * 128;
                    uint8_t* dl = op + HALF + r * 128;
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int cc = (box * 4 + q) ^ sw;
                        *reinterpret_cast<uint4*>(dh + (cc << 4)) =
                            make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
                        *reinterpret_cast<uint4*>(dl + (cc << 4)) =
                            make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
                    }
                    __syncwarp();
                }
                // the generic-proxy writes become visible to the MMA's async proxy
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(conv(stage));  // this CTA's barrier
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue warps 2..9: lane quarter q, chunk parity hh
        const int q = warp & 3;
        const int hh = (warp - 2) >> 2;
        const int rl = q * 32 + lane;
        uint8_t* stg = base_ptr + OFF_EPI + (warp - 2) * STG;
        const uint32_t stg_s = base + OFF_EPI + (uint32_t)((warp - 2) * STG);
        const uint32_t tempty_leader = mapa_rank(tempty(0), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool aborted = false;
        for (int st = cid; st < num_tiles; st += ncl) {
            int mp, nb;
            tile_coords(st, a.num_mp, a.num_n, mp, nb);
            const int m0 = (mp * 2 + (int)rank) * BM, n0 = nb * BN;
            const int row = m0 + rl;
            if (!aborted && !mbar_wait_warp(tfull(acc), acc_phase, abort_flag)) aborted = true;
            if (!aborted) tc_fence_after();
            float pmax = -INFINITY, psum = 0.f;
#pragma unroll 1
            for (int j = hh; j < BN / 32 && !aborted; j += 2) {
                const int nc = n0 + j * 32;
                float v[32];
                tmem_ld32(tmem_base + (uint32_t)(acc * BN + j * 32) + ((uint32_t)(q * 32) << 16), v);
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    if (nc + k < a.N) {
                        const float4 bb = __ldg(reinterpret_cast<const float4*>(a.bias + nc + k));
                        v[k] += bb.x; v[k + 1] += bb.y; v[k + 2] += bb.z; v[k + 3] += bb.w;
                    }
                }
                float cm = pmax;
#pragma unroll
                for (int e = 0; e < 32; e++) {
                    v[e] = gelu_fwd(v[e]);
                    if (nc + e < a.N) cm = fmaxf(cm, v[e]);
                }
                if (row < a.M && cm != -INFINITY) {
                    float sum = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; e++) sum += nc + e < a.N ? expf(v[e] - cm) : 0.f;
                    psum = (pmax == -INFINITY ? 0.f : psum * expf(pmax - cm)) + sum;
                    pmax = cm;
                }
                if (lane == 0) bulk_wait_read<0>();  // this warp's previous store has read the buffer
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; k++)
                    *reinterpret_cast<float4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, stg_s, nc, m0 + q * 32);
                    bulk_commit();
                }
            }
            // the accumulator rows are read: release them to the leader's MMA
            if (!aborted) tc_fence_before();
            __syncwarp();
            if (lane == 0 && !aborted) mbar_arrive_cluster_relaxed(tempty_leader + 8u * (uint32_t)acc);
            // merge the two chunk parities of each row: one partial per (row, tile)
            if (hh == 1) row_part[rl] = make_float2(pmax, psum);
            epi_bar();
            if (hh == 0 && row < a.M && !aborted) {
                const float2 o = row_part[rl];
                const float m = fmaxf(pmax, o.x);
                float sum = 0.f;
                if (pmax != -INFINITY) sum += psum * expf(pmax - m);
                if (o.x != -INFINITY) sum += o.y * expf(o.x - m);
                a.part[(size_t)row * a.part_ld + nb] = make_float2(m, sum);
            }
            epi_bar();
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncthreads();
    if (*abort_flag) {
        // drain: every TMA copy this CTA issued has landed, every MMA is done
        if (threadIdx.x == 0) {
            const int n_issued = *n_issued_smem;
            for (int s = 0; s < STAGES; s++) {
                if (n_issued > s) {
                    const int last = s + ((n_issued - 1 - s) / STAGES) * STAGES;
                    mbar_wait_drain(full(s), (uint32_t)((last / STAGES) & 1));
                }
            }
            atomicOr(a.err, DEVERR_TIMEOUT);
        }
        if (warp == 1 && rank == 0) {
            umma_commit_local_warp<2>(drain);
            if (lane == 0) mbar_wait_drain(drain, 0);
            __syncwarp();
        }
        __syncthreads();
    }
    cluster_sync();  // the peer's arrivals and copies are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<2>(tmem_base, TMEM_COLS);
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// fp32 row-major (rows, cols) with row pitch ld; box = 32 columns x box_rows, 128-byte swizzle
static bool make_map_f32(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows, long long ld,
                         uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(p), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fsp

// 224-wide tiles where they take fewer column-tile rounds of the CTA pairs
// than 256-wide ones (rounds x width) and their M x ceil(N/224) partials fit
// within max_partials, else 256
int fused_split_tile_n(int M, int N, long long max_partials) {
    const long long pairs = num_sms() / 2, mp = ((long long)M + 255) / 256;
    auto cost = [&](int bn) {
        const long long tiles = mp * (((long long)N + bn - 1) / bn);
        return ((tiles + pairs - 1) / pairs) * bn;
    };
    const long long parts224 = (long long)M * (((long long)N + 223) / 224);
    return cost(224) < cost(256) && parts224 <= max_partials ? 224 : 256;
}

namespace fsp {
template <int BN>
static int launch_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, Args a, cudaStream_t s) {
    static bool attr = false;
    static int max_clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[3];
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(fused_split_gemm_k<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess)
            return set_error(GPT2_ERR_CUDA, "fused op: shared-memory opt-in failed: %s", cudaGetErrorString(e));
        int n = 0;
        cfg.gridDim = dim3(2 * 64);
        e = cudaOccupancyMaxActiveClusters(&n, (void*)fused_split_gemm_k<BN>, &cfg);
        if (e != cudaSuccess || n < 1)
            return set_error(GPT2_ERR_CUDA, "fused op: no co-resident CTA pair (%s)", cudaGetErrorString(e));
        max_clusters = n;
        attr = true;
    }
    a.num_n = (a.N + BN - 1) / BN;
    const long long tiles = (long long)a.num_mp * a.num_n;
    const long long ncl = tiles < max_clusters ? tiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(2 * ncl));
    cfg.numAttrs += launch_attrs(at + cfg.numAttrs);
    note_launch(1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_split_gemm_k<BN>, tx, tw, ty, a);
    if (e != cudaSuccess) return set_error(GPT2_ERR_CUDA, "fused op: launch failed: %s", cudaGetErrorString(e));
    return GPT2_OK;
}
}  // namespace fsp

int launch_fused_split_gemm(const float* x, const float* W, const float* b, float* y, float* part,
                            int part_ld, int M, int K, int N, int tile_n, cudaStream_t s, unsigned int* err) {
    using namespace fsp;
    if (tile_n != 256 && tile_n != 224) return set_error(GPT2_ERR_CONFIG, "fused op: tile width %d", tile_n);
    if (part_ld < (N + tile_n - 1) / tile_n) return set_error(GPT2_ERR_CONFIG, "fused op: partial rows too short");
    CUtensorMap tx, tw, ty;
    if (!make_map_f32(&tx, x, K, M, K, BM) || !make_map_f32(&tw, W, K, N, K, (uint32_t)(tile_n / 2)) ||
        !make_map_f32(&ty, y, N, M, N, 32))
        return set_error(GPT2_ERR_CUDA, "fused op: tensor map encoding failed");
    Args a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_mp = (M + 2 * BM - 1) / (2 * BM);
    a.num_n = 0;
    a.num_kb = (K + KB - 1) / KB;
    a.bias = b;
    a.part = reinterpret_cast<float2*>(part);
    a.part_ld = part_ld;
    a.err = err;
    return tile_n == 224 ? launch_bn<224>(tx, tw, ty, a, s) : launch_bn<256>(tx, tw, ty, a, s);
}

// the bounded-wait limit of this translation unit's kernels (0: the default)
int set_wait_limit_fused(unsigned long long ns) {
    return tc::set_tu_wait_limit(ns ? ns : tc::WAIT_LIMIT_NS) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gk
