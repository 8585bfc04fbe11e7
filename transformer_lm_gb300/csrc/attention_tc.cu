// attention_tc.cu -- causal flash attention forward on the tcgen05 tensor
// cores (sm_103a), head size 64, bf16 in, fp32 softmax, bf16 out + fp32 LSE.
//
// Computes for every (b, h) and query i: O_i = sum_{j<=i} softmax_j(q_i.k_j /
// sqrt(64)) v_j and LSE_i (llm.c "train_gpt2.cu", attention_forward with
// softmax_forward_kernel5, in flash form: no T x T matrix is stored).
//
// One CTA takes 256 consecutive queries of one (b, h) as two 128-row tiles
// (one TMEM lane = one query row = one thread of its softmax warpgroup):
//   warp 0       TMA: both Q tiles once, then K and V blocks of 128 keys into
//                a 2-stage ring (3-D tensor map over (3C, T, B): rows past the
//                end of a sequence read as zero);
//   warp 1       one thread issues the MMAs: S_t = Q_t K^T (M=128, N=128,
//                K=64) into TMEM, then O_t = P_t V (M=128, N=64, K=128; V is
//                the MN-major operand);
//   warps 2..9   two softmax warpgroups, one per query tile: each thread reads
//                its row of S from TMEM, forms exp2(s - m) and writes the bf16 P
//                row into 128B-swizzled shared memory. O_t accumulates in TMEM
//                across key blocks; a row's reference max m moves only when a
//                block's max exceeds it by more than 8 (so p <= 256), and then
//                the warp rescales its O rows in TMEM between two P.V MMAs.
// All waits are bounded; on expiry the CTA records DEVERR_TIMEOUT, drains its
// copies and MMAs and frees TMEM.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace gk {
namespace fatc {
using namespace tc;

constexpr int HSZ = 64;
constexpr int BQ = 128;          // queries per tile
constexpr int NQT = 2;           // query tiles per CTA
constexpr int BKV = 128;         // keys per block
constexpr int KV_STAGES = 2;
constexpr int TILE_BYTES = 128 * 128;    // 128 rows x 128 bytes (64 bf16)
constexpr int P_BYTES = 2 * TILE_BYTES;  // 128 queries x 128 keys, two 64-key atoms
constexpr int NUM_THREADS = 64 + NQT * 128;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + NQT * TILE_BYTES;
constexpr int OFF_V = OFF_K + KV_STAGES * TILE_BYTES;
constexpr int OFF_P = OFF_V + KV_STAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_P + NQT * P_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr int TMEM_COLS = 512;   // tile t: S at t*192 (128 columns), O at t*192+128 (64)
constexpr float LN2_F = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.f;  // lazy-rescale threshold (log2 units)

struct FwdArgs {
    bf16* out;
    float* lse;
    int T, C, NH;
    float scale_log2;
    unsigned int* err;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    flash_fwd_tc_k(const __grid_constant__ CUtensorMap tm, const __grid_constant__ FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + OFF_BAR;
    uint8_t* bars_ptr = base_ptr + OFF_BAR;
    // barriers
    const uint32_t qfull = bars;
    auto kvfull = [&](int s) { return bars + 8u * (1 + s); };
    auto kvempty = [&](int s) { return bars + 8u * (1 + KV_STAGES + s); };
    auto sfull = [&](int t) { return bars + 8u * (1 + 2 * KV_STAGES + t); };
    auto pfull = [&](int t) { return bars + 8u * (3 + 2 * KV_STAGES + t); };
    auto pempty = [&](int t) { return bars + 8u * (5 + 2 * KV_STAGES + t); };
    auto ofull = [&](int t) { return bars + 8u * (7 + 2 * KV_STAGES + t); };
    const uint32_t drain = bars + 8u * (11 + 2 * KV_STAGES);
    constexpr int NBARS = 12 + 2 * KV_STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int T = a.T, C = a.C;
    const int nqb = (T + NQT * BQ - 1) / (NQT * BQ);
    const int qblk = nqb - 1 - (int)blockIdx.x;  // the longest rows first
    const int b = blockIdx.y / a.NH, h = blockIdx.y % a.NH;
    const int q0 = qblk * NQT * BQ;
    const int nkb_total = (T + BKV - 1) / BKV;
    const int last = min((q0 + NQT * BQ - 1) / BKV, nkb_total - 1);
    const int n = last + 1;  // key blocks this CTA visits

    if (threadIdx.x == 0) {
        mbar_init(qfull, 1);
        for (int s = 0; s < KV_STAGES; s++) {
            mbar_init(kvfull(s), 1);
            mbar_init(kvempty(s), 1);
        }
        for (int t = 0; t < NQT; t++) {
            mbar_init(sfull(t), 1);
            mbar_init(pfull(t), 128);
            mbar_init(pempty(t), 1);
            mbar_init(ofull(t), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *n_issued_smem = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_enter();  // global memory is touched only from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int issued = 0;
            mbar_expect_tx(qfull, NQT * TILE_BYTES);
            for (int t = 0; t < NQT; t++)
                tma_load_3d(base + OFF_Q + t * TILE_BYTES, &tm, qfull, h * HSZ, q0 + t * BQ, b);
            for (int i = 0; i < n; i++) {
                const int st = i % KV_STAGES;
                if (!mbar_wait(kvempty(st), (uint32_t)(((i / KV_STAGES) & 1) ^ 1), abort_flag)) break;
                mbar_expect_tx(kvfull(st), 2 * TILE_BYTES);
                tma_load_3d(base + OFF_K + st * TILE_BYTES, &tm, kvfull(st), C + h * HSZ, i * BKV, b);
                tma_load_3d(base + OFF_V + st * TILE_BYTES, &tm, kvfull(st), 2 * C + h * HSZ, i * BKV, b);
                ++issued;
            }
            *n_issued_smem = issued;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idS = idesc<0>(0, 0, BQ, BKV);
            const uint32_t idPV = idesc<0>(0, 1, BQ, HSZ);
            auto issue_s = [&](int t, int st) {
                const uint32_t d = tmem_base + (uint32_t)(t * 192);
#pragma unroll
                for (int k = 0; k < HSZ / 16; k++)
                    umma<0, 1>(d, sdesc(base + OFF_Q + t * TILE_BYTES + k * 32, 16, 1024),
                               sdesc(base + OFF_K + st * TILE_BYTES + k * 32, 16, 1024), idS,
                               k ? 1u : 0u);
                umma_commit<1>(sfull(t));
            };
            bool ok = mbar_wait(qfull, 0, abort_flag) && mbar_wait(kvfull(0), 0, abort_flag);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < NQT; t++) issue_s(t, 0);
            }
            for (int i = 0; ok && i < n; i++) {
                const int st = i % KV_STAGES;
                for (int t = 0; t < NQT && ok; t++) {
                    if (!mbar_wait(pfull(t), (uint32_t)(i & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(t * 192 + 128);
                    const uint32_t pb = base + OFF_P + t * P_BYTES;
#pragma unroll
                    for (int k = 0; k < BKV / 16; k++)
                        umma<0, 1>(d, sdesc(pb + (k >> 2) * TILE_BYTES + (k & 3) * 32, 16, 1024),
                                   sdesc(base + OFF_V + st * TILE_BYTES + k * 2048, 8192, 1024), idPV,
                                   (i | k) ? 1u : 0u);
                    umma_commit<1>(pempty(t));
                    if (i == n - 1) umma_commit<1>(ofull(t));  // O_t is complete
                    if (i + 1 < n) {
                        const int st1 = (i + 1) % KV_STAGES;
                        if (t == 0) {
                            if (!mbar_wait(kvfull(st1), (uint32_t)(((i + 1) / KV_STAGES) & 1), abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        issue_s(t, st1);
                    }
                }
                umma_commit<1>(kvempty(st));  // K/V of this stage are no longer read
            }
        }
    } else {
        // ---------------- softmax warpgroups
        const int t = (warp - 2) >> 2;
        const int qq = warp & 3;  // TMEM lane quarter
        const int r = qq * 32 + lane;
        const int query = q0 + t * BQ + r;
        const uint32_t tS = tmem_base + (uint32_t)(t * 192) + ((uint32_t)(qq * 32) << 16);
        const uint32_t tO = tS + 128;
        uint8_t* pbuf = base_ptr + OFF_P + t * P_BYTES;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait_warp = [&](uint32_t bar, uint32_t parity) {
            int w = 1;
            if (lane == 0) w = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
            w = __shfl_sync(0xffffffffu, w, 0);
            return w != 0;
        };
        for (int i = 0; i < n; i++) {
            if (!wait_warp(sfull(t), (uint32_t)(i & 1))) { ok = false; break; }
            tc_fence_after();
            const int k0 = i * BKV;
            const bool diag = k0 + BKV - 1 > q0 + t * BQ;  // some key may follow some query
            float va[64], vb[64];
            tmem_ld64(tS, va);
            tmem_ld64(tS + 64, vb);
            // row maximum of the raw scores (the scale is positive)
            float mx = -INFINITY;
            if (!diag) {
#pragma unroll
                for (int j = 0; j < 64; j += 2) mx = fmaxf(mx, fmaxf(va[j], va[j + 1]));
#pragma unroll
                for (int j = 0; j < 64; j += 2) mx = fmaxf(mx, fmaxf(vb[j], vb[j + 1]));
            } else {
                const int lim = query - k0;  // keys k0 + j with j <= lim are visible
#pragma unroll
                for (int j = 0; j < 64; j++) mx = fmaxf(mx, j <= lim ? va[j] : -INFINITY);
#pragma unroll
                for (int j = 0; j < 64; j++) mx = fmaxf(mx, j + 64 <= lim ? vb[j] : -INFINITY);
            }
            mx *= a.scale_log2;
            // P may be overwritten (and O rescaled) once the previous P.V is done
            if (!wait_warp(pempty(t), (uint32_t)((i & 1) ^ 1))) { ok = false; break; }
            if (i == 0) {
                m = mx;
            } else if (__any_sync(0xffffffffu, mx > m + RESCALE_LOG2)) {
                // lazy rescale of this warp's 32 O rows (and row sums)
                const float m_new = fmaxf(m, mx);
                const float f = ex2_approx(m - m_new);
#pragma unroll 1
                for (int hh = 0; hh < HSZ; hh += 16) {
                    float ov[16];
                    tmem_ld16(tO + hh, ov);
#pragma unroll
                    for (int j = 0; j < 16; j++) ov[j] *= f;
                    tmem_st16(tO + hh, ov);
                }
                l *= f;
                m = m_new;
            }
            const float neg = -m;
            float lsum = 0.f;
            auto emit = [&](const float (&vv)[64], int half) {
                const int lim = diag ? query - (k0 + half * 64) : 64;
                // 64 keys = one 128-byte row of atom `half`, eight 16-byte chunks
                uint8_t* atom = pbuf + half * TILE_BYTES + r * 128;
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int j = 8 * u + 2 * e;
                        float p0 = ex2_approx(fmaf(vv[j], a.scale_log2, neg));
                        float p1 = ex2_approx(fmaf(vv[j + 1], a.scale_log2, neg));
                        if (diag) {
                            p0 = j <= lim ? p0 : 0.f;
                            p1 = j + 1 <= lim ? p1 : 0.f;
                        }
                        lsum += p0 + p1;
                        __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
                        pk[e] = *reinterpret_cast<uint32_t*>(&pr);
                    }
                    *reinterpret_cast<uint4*>(atom + ((u ^ (r & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            };
            emit(va, 0);
            emit(vb, 1);
            l += lsum;
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(pfull(t));
        }
        // the last P.V completes O
        if (ok && wait_warp(ofull(t), 0u)) {
            tc_fence_after();
            float ov[64];
            tmem_ld64(tO, ov);
            if (query < T) {
                const float inv = 1.f / l;
                bf16* dst = a.out + ((size_t)b * T + query) * C + (size_t)h * HSZ;
#pragma unroll
                for (int d = 0; d < HSZ; d += 8) {
                    __nv_bfloat162 p0 = __floats2bfloat162_rn(ov[d] * inv, ov[d + 1] * inv);
                    __nv_bfloat162 p1 = __floats2bfloat162_rn(ov[d + 2] * inv, ov[d + 3] * inv);
                    __nv_bfloat162 p2 = __floats2bfloat162_rn(ov[d + 4] * inv, ov[d + 5] * inv);
                    __nv_bfloat162 p3 = __floats2bfloat162_rn(ov[d + 6] * inv, ov[d + 7] * inv);
                    *reinterpret_cast<uint4*>(dst + d) =
                        make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                                   *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
                }
                a.lse[(size_t)blockIdx.y * T + query] = (m + log2f(l)) * LN2_F;
            }
        }
    }

    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) {
            mbar_wait_drain(qfull, 0);
            const int issued = *n_issued_smem;
            for (int s = 0; s < KV_STAGES; s++) {
                if (issued > s) {
                    const int lst = s + ((issued - 1 - s) / KV_STAGES) * KV_STAGES;
                    mbar_wait_drain(kvfull(s), (uint32_t)((lst / KV_STAGES) & 1));
                }
            }
            atomicOr(a.err, DEVERR_TIMEOUT);
        }
        if (threadIdx.x == 32) {
            umma_commit_local<1>(drain);
            mbar_wait_drain(drain, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, TMEM_COLS);
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

}  // namespace fatc

// qkv (B, T, 3C) bf16 viewed as a 3-D tensor (3C, T, B); 64 x 128 x 1 boxes
int launch_flash_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
                            cudaStream_t s, unsigned int* err) {
    using namespace fatc;
    auto fn = encode_fn();
    if (!fn) return set_error(GPT2_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    if ((uintptr_t)qkv % 16 || C % 64)
        return set_error(GPT2_ERR_ALIGN, "flash forward: qkv must be 16-byte aligned and C a multiple of 64");
    CUtensorMap tm;
    cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    cuuint32_t box[3] = {HSZ, BQ, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return set_error(GPT2_ERR_CUDA, "flash forward: tensor map encoding failed");
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(flash_fwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess)
            return set_error(GPT2_ERR_CUDA, "flash forward: shared-memory opt-in failed: %s",
                             cudaGetErrorString(e));
        attr = true;
    }
    FwdArgs a;
    a.out = (bf16*)out;
    a.lse = lse;
    a.T = T;
    a.C = C;
    a.NH = NH;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)HSZ);
    a.err = err;
    dim3 grid((T + NQT * BQ - 1) / (NQT * BQ), B * NH);
    note_launch(1);
    launch_pdl(flash_fwd_tc_k, grid, dim3(NUM_THREADS), SMEM_BYTES, s, tm, a);
    return GPT2_OK;
}

}  // namespace gk
