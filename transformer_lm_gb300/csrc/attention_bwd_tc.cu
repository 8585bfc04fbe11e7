// attention_bwd_tc.cu -- causal flash attention backward on the tcgen05 tensor
// cores (sm_103a), head size 64, bf16 operands, fp32 softmax and accumulators.
//
// With P = softmax(q.k / sqrt(64)) recomputed from the forward's LSE, and
// D_i = sum_d dO_id O_id (the row dot product of the output and its grad):
//   dV_j = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dK_j = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
// (llm.c "train_gpt2.cu", attention_backward with softmax_autoregressive_
// backward_kernel, in flash form: no T x T matrix is stored). The grads are
// written with "=" into dqkv (B, T, 3C).
//
// Two kernels, neither with float atomics, so every run is bit-identical:
//   DKV  one work item per (128-key tile, b, h); it walks the query blocks at
//        and after its keys, with S^T = K Q^T and dP^T = V dO^T in TMEM and
//        dV += P^T dO, dK += dS^T Q accumulating in TMEM;
//   DQ   one work item per (128-query tile, b, h); it walks the key blocks at
//        and before its queries with S = Q K^T, dP = dO V^T and dQ += dS K.
// Roles (608 threads): warp 0 loads by TMA the item's fixed tiles (K, V or Q,
// dO; double-buffered, so the next item's arrive during this one) and the
// streamed Q/dO (or K/V) blocks into a 4-stage ring (and, for DKV, the blocks'
// LSE and D into shared memory); warp 18 issues the S and dP MMAs and warp 1
// the accumulating ones (each loop runs as a whole warp, one elected lane
// issues), so neither chain waits behind the other; warps 2..17 form P and
// dS, four warps per TMEM lane quarter, each on 32 of the 128 columns, and
// write them as bf16 pairs into TMEM, where the accumulating MMAs read them as
// their A operand. The next block's S (and dP) MMA is issued as soon as the
// current one has been read, so it overlaps the current block's softmax. All
// waits are bounded; on expiry the CTA records DEVERR_TIMEOUT, drains its
// copies and MMAs and frees TMEM.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

namespace gk {
namespace fabw {
using namespace tc;

constexpr int HSZ = 64;
constexpr int BLK = 128;                   // rows per work item and columns per block
constexpr int STAGES = 4;
constexpr int TILE = 128 * 128;            // 128 rows x 64 bf16, 128B-swizzled
constexpr int OFF_X = 0;                   // [buffer][2]: K, V (DKV) or Q, dO (DQ) of an item
constexpr int OFF_Y = 4 * TILE;            // ring: stage s holds Y0 at +2s*TILE, Y1 at +(2s+1)*TILE
constexpr int OFF_VEC = OFF_Y + STAGES * 2 * TILE;  // per stage: -LSE*log2(e) [128], D [128]
constexpr int OFF_BAR = OFF_VEC + STAGES * 1024;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr int CW = 16;                     // compute warps (P and dS)
constexpr int CQ = CW / 4;                 // compute warps per TMEM lane quarter
constexpr int COLS = 128 / CQ;             // columns per compute thread
constexpr int QKW = 2 + CW;                // the warp that issues S and dP
constexpr int NUM_THREADS = 64 + 32 * CW + 32;
// TMEM columns: S, P (bf16 pairs, DKV), dS (bf16 pairs), dP, and the
// accumulators (dV | dK for DKV, dQ for DQ)
constexpr int TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_P = 128, TM_DS = 192, TM_DP = 256, TM_A0 = 384, TM_A1 = 448;
constexpr float LOG2E = 1.4426950408889634f;

struct BwdArgs {
    void* dqkv;  // bf16 or fp16, as the operands
    const float* lse;
    const float* D;
    int T, C, NH, BH, nblk, items;
    float scale, scale_log2;
    unsigned int* err;
};

// One work item: (tile, b, h), heaviest tiles first across all heads (key
// tile 0 meets every query block, query tile nblk-1 every key block).
struct Item {
    int tile, bh, b, h, r0, n;
};
template <bool DKV> DEVI Item decode_item(const BwdArgs& a, int idx) {
    Item it;
    const int grp = idx / a.BH;
    it.bh = idx % a.BH;
    it.tile = DKV ? grp : a.nblk - 1 - grp;
    it.b = it.bh / a.NH;
    it.h = it.bh % a.NH;
    it.r0 = it.tile * BLK;
    it.n = DKV ? a.nblk - it.tile : it.tile + 1;  // column blocks visited
    return it;
}

// Persistent: each CTA takes one item per round (a snake over the CTAs);
// the ring and every barrier phase run on counters global to the CTA, so the
// next item's loads and first MMAs overlap this item's last blocks and its
// epilogue.
// KIND 0: bf16 operands, 2: fp16 (the tcgen05 kind::f16 operand type)
template <bool DKV, int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    flash_bwd_tc_k(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ BwdArgs a) {
    using H = typename std::conditional<KIND == 2, f16, bf16>::type;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + OFF_BAR;
    uint8_t* bars_ptr = base_ptr + OFF_BAR;
    auto x_full = [&](int b) { return bars + 8u * b; };
    auto x_empty = [&](int b) { return bars + 8u * (2 + b); };
    auto st_full = [&](int s) { return bars + 8u * (4 + s); };
    auto st_empty = [&](int s) { return bars + 8u * (4 + STAGES + s); };
    constexpr int B0 = 4 + 2 * STAGES;
    const uint32_t s_full = bars + 8u * B0, s_empty = bars + 8u * (B0 + 1);
    const uint32_t dp_full = bars + 8u * (B0 + 2), dp_empty = bars + 8u * (B0 + 3);
    const uint32_t p_full = bars + 8u * (B0 + 4), p_empty = bars + 8u * (B0 + 5);
    const uint32_t ds_full = bars + 8u * (B0 + 6), ds_empty = bars + 8u * (B0 + 7);
    // per accumulator buffer (DQ alternates two; DKV's dV | dK fill the rest of TMEM)
    auto acc_full = [&](int b) { return bars + 8u * (B0 + 8 + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (B0 + 10 + b); };
    const uint32_t drain = bars + 8u * (B0 + 12);
    constexpr int NBARS = B0 + 13;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);   // ring loads issued
    int* x_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 12);  // fixed-tile loads issued [2]
    static_assert(8 * NBARS + 20 <= 256, "barrier area");

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int T = a.T, C = a.C;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(x_full(b), 1);
            mbar_init(x_empty(b), 1);
        }
        for (int s = 0; s < STAGES; s++) {
            mbar_init(st_full(s), 1);
            mbar_init(st_empty(s), 2);  // released by both MMA-issuing warps
        }
        mbar_init(s_full, 1);
        mbar_init(s_empty, CW);
        mbar_init(dp_full, 1);
        mbar_init(dp_empty, CW);
        mbar_init(p_full, CW);
        mbar_init(p_empty, 1);
        mbar_init(ds_full, CW);
        mbar_init(ds_empty, 1);
        for (int b = 0; b < 2; b++) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), CW);
        }
        mbar_init(drain, 2);
        *abort_flag = 0;
        *n_issued_smem = 0;
        x_issued_smem[0] = 0;
        x_issued_smem[1] = 0;
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

    // round t of the item walk: a snake over the CTAs (forward on even
    // rounds, backward on odd ones) evens out the heavy-first item sizes
    auto item_of = [&](int t) {
        const int G = (int)gridDim.x, c = (int)blockIdx.x;
        return t * G + ((t & 1) ? G - 1 - c : c);
    };

    // warp-uniform bounded wait
    auto wait_warp = [&](uint32_t bar, uint32_t parity) {
        int w = 1;
        if (lane == 0) w = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
        return __shfl_sync(0xffffffffu, w, 0) != 0;
    };

    if (warp == 0) {
        // ---------------- loads
        int g = 0;
        bool ok = true;
        // the fixed tiles of the CTA's t-th item into buffer t & 1, once the
        // item two back has released it
        auto load_x = [&](int t, int idx) -> bool {
            const Item it = decode_item<DKV>(a, idx);
            const int xb = t & 1;
            if (!wait_warp(x_empty(xb), (uint32_t)(((t >> 1) & 1) ^ 1))) return false;
            if (lane == 0) {
                const uint32_t x = base + OFF_X + xb * 2 * TILE;
                mbar_expect_tx(x_full(xb), 2 * TILE);
                if (DKV) {
                    tma_load_3d(x, &tqkv, x_full(xb), C + it.h * HSZ, it.r0, it.b);
                    tma_load_3d(x + TILE, &tqkv, x_full(xb), 2 * C + it.h * HSZ, it.r0, it.b);
                } else {
                    tma_load_3d(x, &tqkv, x_full(xb), it.h * HSZ, it.r0, it.b);
                    tma_load_3d(x + TILE, &tdo, x_full(xb), it.h * HSZ, it.r0, it.b);
                }
                ++x_issued_smem[xb];
            }
            return true;
        };
        if (item_of(0) < a.items) ok = load_x(0, item_of(0));
        for (int t = 0, idx = item_of(0); ok && idx < a.items; idx = item_of(++t)) {
            const Item it = decode_item<DKV>(a, idx);
            const int xq = it.h * HSZ, xk = C + it.h * HSZ, xv = 2 * C + it.h * HSZ;
            for (int u = 0; u < it.n; u++, g++) {
                const int st = g % STAGES;
                if (!wait_warp(st_empty(st), (uint32_t)(((g / STAGES) & 1) ^ 1))) { ok = false; break; }
                const int c0 = (DKV ? it.tile + u : u) * BLK;
                if (DKV) {
                    // the block's LSE (as -LSE * log2 e; -inf past the sequence end,
                    // which zeroes those columns of P) and D
                    float4 nl, dd;
                    float* pn = &nl.x;
                    float* pd = &dd.x;
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int q = c0 + lane * 4 + e;
                        const bool in = q < T;
                        pn[e] = in ? -a.lse[(size_t)it.bh * T + q] * LOG2E : -INFINITY;
                        pd[e] = in ? a.D[(size_t)it.bh * T + q] : 0.f;
                    }
                    float* vec = reinterpret_cast<float*>(base_ptr + OFF_VEC + st * 1024);
                    reinterpret_cast<float4*>(vec)[lane] = nl;
                    reinterpret_cast<float4*>(vec + 128)[lane] = dd;
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t y = base + OFF_Y + st * 2 * TILE;
                    mbar_expect_tx(st_full(st), 2 * TILE);
                    if (DKV) {
                        tma_load_3d(y, &tqkv, st_full(st), xq, c0, it.b);
                        tma_load_3d(y + TILE, &tdo, st_full(st), it.h * HSZ, c0, it.b);
                    } else {
                        tma_load_3d(y, &tqkv, st_full(st), xk, c0, it.b);
                        tma_load_3d(y + TILE, &tqkv, st_full(st), xv, c0, it.b);
                    }
                    *n_issued_smem = g + 1;
                }
                // the next item's fixed tiles, right after this item's first block
                if (u == 0 && item_of(t + 1) < a.items && !load_x(t + 1, item_of(t + 1))) {
                    ok = false;
                    break;
                }
            }
        }
    } else if (warp == 1 || warp == QKW) {
        // ---------------- MMA issuers: warp QKW issues S and dP, warp 1 the
        // accumulating MMAs, so neither chain waits behind the other. Each
        // runs its loop as a whole warp; one elected lane issues.
        const uint32_t idSq = idesc<KIND>(0, 0, BLK, BLK);  // S, dP: both operands K-major
        const uint32_t idAcc = idesc<KIND>(0, 1, BLK, HSZ); // acc += (P|dS) Y: Y is MN-major
        auto ybuf = [&](int g, int which) { return base + OFF_Y + (g % STAGES) * 2 * TILE + which * TILE; };
        auto issue_qk = [&](uint32_t d, uint32_t x, uint32_t y) {
            const uint64_t dx = sdesc(x, 16, 1024), dy = sdesc(y, 16, 1024);
#pragma unroll
            for (int k = 0; k < HSZ / 16; k++)  // +32 bytes along K per step
                umma_warp<KIND, 1>(d, dx + 2 * k, dy + 2 * k, idSq, k ? 1u : 0u);
        };
        // acc += A Y, A = bf16 pairs in TMEM from column ta (16 rows of K = 8
        // columns per step), Y = 2048 bytes per step
        auto issue_acc = [&](uint32_t d, uint32_t ta, uint32_t y, bool accumulate) {
            const uint64_t dy = sdesc(y, 8192, 1024);
#pragma unroll
            for (int k = 0; k < BLK / 16; k++)
                umma_ts_warp(d, ta + (uint32_t)(k * 8), dy + 128 * k, idAcc, (accumulate || k) ? 1u : 0u);
        };
        int g = 0;
        bool ok = true;
        for (int t = 0, idx = item_of(0); ok && idx < a.items; idx = item_of(++t)) {
            const int n = decode_item<DKV>(a, idx).n;
            if (warp == QKW) {
                const int xb = t & 1;
                const uint32_t x0 = base + OFF_X + xb * 2 * TILE, x1 = x0 + TILE;
                if (!mbar_wait_warp(x_full(xb), (uint32_t)((t >> 1) & 1), abort_flag)) break;
                for (int u = 0; u < n; u++, g++) {
                    // S of block g once its ring stage landed and the previous S was read
                    if (!mbar_wait_warp(st_full(g % STAGES), (uint32_t)((g / STAGES) & 1), abort_flag) ||
                        !mbar_wait_warp(s_empty, (uint32_t)((g & 1) ^ 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(tmem_base + TM_S, x0, ybuf(g, 0));
                    umma_commit_warp<1>(s_full);
                    // dP of block g once the previous dP was read
                    if (!mbar_wait_warp(dp_empty, (uint32_t)((g & 1) ^ 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(tmem_base + TM_DP, x1, ybuf(g, 1));
                    umma_commit_warp<1>(dp_full);
                    umma_commit_warp<1>(st_empty(g % STAGES));  // this warp's reads of the stage
                }
                if (ok) umma_commit_warp<1>(x_empty(xb));  // the item's last reads of its fixed tiles
            } else {
                // DQ alternates two accumulator buffers over the items; the buffer's
                // previous item has been read out
                const int ab = DKV ? 0 : (t & 1);
                const uint32_t acc_par = DKV ? (uint32_t)(t & 1) : (uint32_t)((t >> 1) & 1);
                if (!mbar_wait_warp(acc_empty(ab), acc_par ^ 1u, abort_flag)) break;
                tc_fence_after();
                for (int u = 0; u < n; u++, g++) {
                    const uint32_t par = (uint32_t)(g & 1);
                    if (DKV) {
                        if (!mbar_wait_warp(p_full, par, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        issue_acc(tmem_base + TM_A0, tmem_base + TM_P, ybuf(g, 1), u > 0);  // dV += P^T dO
                        umma_commit_warp<1>(p_empty);
                    }
                    if (!mbar_wait_warp(ds_full, par, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    // DKV: dK += dS^T Q; DQ: dQ += dS K
                    issue_acc(tmem_base + (DKV || ab ? TM_A1 : TM_A0), tmem_base + TM_DS, ybuf(g, 0), u > 0);
                    umma_commit_warp<1>(ds_empty);
                    umma_commit_warp<1>(st_empty(g % STAGES));  // this warp's reads of the stage
                }
                if (ok) umma_commit_warp<1>(acc_full(ab));
            }
        }
    } else if (warp >= 2 && warp < 2 + CW) {
        // ---------------- P and dS: CW warps, CQ per TMEM lane quarter, each
        // on COLS consecutive columns of its row
        const int qq = warp & 3;             // TMEM lane quarter
        const int cq = (warp - 2) >> 2;      // column group
        const int r = qq * 32 + lane;        // row within the tile
        const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
        const int c_base = cq * COLS;
        const uint32_t tS = tmem_base + lane_off + TM_S + c_base;
        const uint32_t tdP = tmem_base + lane_off + TM_DP + c_base;
        const uint32_t tP = tmem_base + lane_off + TM_P + c_base / 2;   // bf16 pairs
        const uint32_t tDS = tmem_base + lane_off + TM_DS + c_base / 2;
        static_assert(COLS == 32, "one 32-column TMEM load per operand");
        int g = 0;
        bool ok = true;
        // Item t's accumulators are read out after the first block of item t + 1
        // (whose S and dP were computed under item t's last block), so the
        // wait for item t's last MMAs and the read-out overlap the tensor work
        // of item t + 1. The columns split over the column groups: DKV
        // [dV 64 | dK 64] at TM_A0; DQ dQ 64 at TM_A0 or TM_A1 (item parity).
        int pend_t = -1;
        Item pend_it{};
        auto epilogue = [&](int t, const Item& it) -> bool {
            const int ab = DKV ? 0 : (t & 1);
            const uint32_t acc_par = DKV ? (uint32_t)(t & 1) : (uint32_t)((t >> 1) & 1);
            if (!wait_warp(acc_full(ab), acc_par)) return false;
            tc_fence_after();
            constexpr int W = (DKV ? 128 : 64) / CQ;  // columns per thread
            const int a0 = cq * W;                    // first accumulator column
            const uint32_t tacc = tmem_base + lane_off + (ab ? TM_A1 : TM_A0) + (uint32_t)a0;
            float v[W];
#pragma unroll
            for (int ch = 0; ch < W; ch += 16)
                tmem_ld16(tacc + (uint32_t)ch, *reinterpret_cast<float(*)[16]>(v + ch));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(ab));  // the buffer's next item may overwrite them
            const int row = it.r0 + r;
            if (row < T) {
                const bool is_k = DKV && a0 >= 64;
                const float sc = (!DKV || is_k) ? a.scale : 1.f;
                const int col = DKV ? (is_k ? C + it.h * HSZ : 2 * C + it.h * HSZ) + (a0 % 64)
                                    : it.h * HSZ + a0;
                H* dst = (H*)a.dqkv + ((size_t)it.b * T + row) * 3 * C + col;
#pragma unroll
                for (int d = 0; d < W; d += 8) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) pk[e] = f2_h2<H>(v[d + 2 * e] * sc, v[d + 2 * e + 1] * sc);
                    *reinterpret_cast<uint4*>(dst + d) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
            return true;
        };
        for (int t = 0, idx = item_of(0); ok && idx < a.items; idx = item_of(++t)) {
            const Item it = decode_item<DKV>(a, idx);
            const int row = it.r0 + r;  // key (DKV) or query (DQ)
            // DQ: the row's LSE and D
            float nl_row = -INFINITY, d_row = 0.f;
            if (!DKV && row < T) {
                nl_row = -a.lse[(size_t)it.bh * T + row] * LOG2E;
                d_row = a.D[(size_t)it.bh * T + row];
            }
            for (int u = 0; u < it.n; u++, g++) {
                const int st = g % STAGES;
                const uint32_t par = (uint32_t)(g & 1);
                if (!wait_warp(s_full, par)) { ok = false; break; }
                tc_fence_after();
                const float* vec = reinterpret_cast<const float*>(base_ptr + OFF_VEC + st * 1024);
                // the diagonal block: DKV sees it first, DQ last
                const bool diag = DKV ? u == 0 : u == it.n - 1;
                float P[COLS];
                {
                    float v[32];
                    tmem_ld32(tS, v);
                    // S may be overwritten by the next block's MMA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_empty);
                    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int c = c_base + e;
                        float4 nl4;
                        if (DKV) nl4 = *reinterpret_cast<const float4*>(vec + c);
                        else nl4 = make_float4(nl_row, nl_row, nl_row, nl_row);
                        // exponent arguments two at a time (packed fp32 FMA)
                        const float2 x01 = ffma2(make_float2(v[e], v[e + 1]), sc2, make_float2(nl4.x, nl4.y));
                        const float2 x23 = ffma2(make_float2(v[e + 2], v[e + 3]), sc2, make_float2(nl4.z, nl4.w));
                        float p4[4] = {ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x), ex2_approx(x23.y)};
#pragma unroll
                        for (int f = 0; f < 4; f++) {
                            // causal: query >= key
                            if (diag) p4[f] = (DKV ? c + f >= r : c + f <= r) ? p4[f] : 0.f;
                            P[e + f] = p4[f];
                        }
                    }
                }
                if (DKV) {
                    // P^T as bf16 pairs into TMEM, once the previous dV MMA read it
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) pk[e] = f2_h2<H>(P[2 * e], P[2 * e + 1]);
                    if (!wait_warp(p_empty, par ^ 1u)) { ok = false; break; }
                    tc_fence_after();
                    tmem_st16_nowait(tP, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full);
                }
                if (!wait_warp(dp_full, par)) { ok = false; break; }
                tc_fence_after();
                uint32_t dsk[16];
                {
                    float v[32];
                    tmem_ld32(tdP, v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dp_empty);
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int c = c_base + e;
                        float4 d4;
                        if (DKV) d4 = *reinterpret_cast<const float4*>(vec + 128 + c);
                        else d4 = make_float4(d_row, d_row, d_row, d_row);
                        // P (dP - D), two at a time (packed fp32 add and multiply)
                        const float2 s01 = fmul2(make_float2(P[e], P[e + 1]),
                                                 fadd2(make_float2(v[e], v[e + 1]), make_float2(-d4.x, -d4.y)));
                        const float2 s23 = fmul2(make_float2(P[e + 2], P[e + 3]),
                                                 fadd2(make_float2(v[e + 2], v[e + 3]), make_float2(-d4.z, -d4.w)));
                        dsk[e >> 1] = f2_h2<H>(s01.x, s01.y);
                        dsk[(e >> 1) + 1] = f2_h2<H>(s23.x, s23.y);
                    }
                }
                if (!wait_warp(ds_empty, par ^ 1u)) { ok = false; break; }
                tc_fence_after();
                tmem_st16_nowait(tDS, dsk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
                if (u == 0 && pend_t >= 0) {
                    if (!epilogue(pend_t, pend_it)) { ok = false; break; }
                    pend_t = -1;
                }
            }
            if (!ok) break;
            pend_t = t;
            pend_it = it;
        }
        // the last item's read-out
        if (ok && pend_t >= 0) epilogue(pend_t, pend_it);
    }

    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) {
            // let every issued copy land before the shared memory is released
            for (int b = 0; b < 2; b++) {
                const int nx = x_issued_smem[b];
                if (nx > 0) mbar_wait_drain(x_full(b), (uint32_t)((nx - 1) & 1));
            }
            const int issued = *n_issued_smem;
            for (int s = 0; s < STAGES; s++) {
                if (issued > s) {
                    const int lst = s + ((issued - 1 - s) / STAGES) * STAGES;
                    mbar_wait_drain(st_full(s), (uint32_t)((lst / STAGES) & 1));
                }
            }
            atomicOr(a.err, DEVERR_TIMEOUT);
        }
        if (warp == 1 || warp == QKW) {  // each issuing lane commits (elected as when issuing)
            umma_commit_local_warp<1>(drain);
            if (lane == 0) mbar_wait_drain(drain, 0);
            __syncwarp();
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, TMEM_COLS);
    }
}

// D_i = dO_i . O_i for every (b, h, i), eight threads per row (16-byte loads)
template <typename H>
__global__ void rowdot64_k(float* __restrict__ D, const H* __restrict__ dout,
                           const H* __restrict__ out, int T, int C, int NH, int nrows) {
    pdl_enter();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    const int row = idx >> 3, part = idx & 7;
    float s = 0.f;
    if (row < nrows) {
        const int bh = row / T, t = row % T;
        const int b = bh / NH, h = bh % NH;
        const size_t off = ((size_t)b * T + t) * C + (size_t)h * HSZ + part * 8;
        const Vec16<H> g = ld16(dout + off), o = ld16(out + off);
#pragma unroll
        for (int e = 0; e < 8; e++) s = fmaf(to_f(g.v[e]), to_f(o.v[e]), s);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (row < nrows && part == 0) D[row] = s;
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

// (B, T, width) bf16 or fp16 as a 3-D tensor (width, T, B) with 64 x 128 x 1 boxes
static int make_map(CUtensorMap* tm, DType dt, const void* p, int width, int T, int B) {
    auto fn = encode_fn();
    if (!fn) return set_error(GPT2_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)T * width * 2};
    cuuint32_t box[3] = {HSZ, BLK, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(tm, dt == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
           const_cast<void*>(p), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return set_error(GPT2_ERR_CUDA, "flash backward: tensor map encoding failed");
    return GPT2_OK;
}

template <bool DKV, int KIND> static int opt_in() {
    static bool done = false;
    if (done) return GPT2_OK;
    const cudaError_t e = cudaFuncSetAttribute(flash_bwd_tc_k<DKV, KIND>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess)
        return set_error(GPT2_ERR_CUDA, "flash backward: shared-memory opt-in failed: %s", cudaGetErrorString(e));
    done = true;
    return GPT2_OK;
}

}  // namespace fabw

// D = rowsum(dO * O), then dQ (query tiles) and dK, dV (key tiles)
int launch_flash_backward_tc(DType dt, void* dqkv, const void* dout, const void* qkv, const void* out,
                             const float* lse, float* D, int B, int T, int C, int NH, cudaStream_t s,
                             unsigned int* err) {
    using namespace fabw;
    if (dt != DT_BF16 && dt != DT_F16) return set_error(GPT2_ERR_CONFIG, "flash backward: 16-bit operands only");
    const bool h16 = dt == DT_F16;
    if ((uintptr_t)qkv % 16 || (uintptr_t)dout % 16 || (uintptr_t)out % 16 || C % 64 || C / NH != HSZ)
        return set_error(GPT2_ERR_ALIGN, "flash backward: 16-byte aligned operands and head size 64 needed");
    CUtensorMap tqkv, tdo;
    int rc = make_map(&tqkv, dt, qkv, 3 * C, T, B);
    if (rc == GPT2_OK) rc = make_map(&tdo, dt, dout, C, T, B);
    if (rc == GPT2_OK) rc = h16 ? opt_in<true, 2>() : opt_in<true, 0>();
    if (rc == GPT2_OK) rc = h16 ? opt_in<false, 2>() : opt_in<false, 0>();
    if (rc != GPT2_OK) return rc;
    const int nrows = B * NH * T;
    note_launch(3);
    if (h16)
        launch_pdl(rowdot64_k<f16>, dim3((nrows * 8 + 255) / 256), dim3(256), 0, s, D, (const f16*)dout,
                   (const f16*)out, T, C, NH, nrows);
    else
        launch_pdl(rowdot64_k<bf16>, dim3((nrows * 8 + 255) / 256), dim3(256), 0, s, D, (const bf16*)dout,
                   (const bf16*)out, T, C, NH, nrows);
    BwdArgs a;
    a.dqkv = dqkv;
    a.lse = lse;
    a.D = D;
    a.T = T;
    a.C = C;
    a.NH = NH;
    a.BH = B * NH;
    a.nblk = (T + BLK - 1) / BLK;
    a.items = a.nblk * a.BH;
    a.scale = 1.f / sqrtf((float)HSZ);
    a.scale_log2 = LOG2E * a.scale;
    a.err = err;
    const int grid = a.items < num_sms() ? a.items : num_sms();  // persistent
    if (h16) {
        launch_pdl(flash_bwd_tc_k<false, 2>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, tqkv, tdo, a);
        launch_pdl(flash_bwd_tc_k<true, 2>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, tqkv, tdo, a);
    } else {
        launch_pdl(flash_bwd_tc_k<false, 0>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, tqkv, tdo, a);
        launch_pdl(flash_bwd_tc_k<true, 0>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, tqkv, tdo, a);
    }
    return GPT2_OK;
}

// the bounded-wait limit of this translation unit's kernels (0: the default)
int set_wait_limit_attn_bwd(unsigned long long ns) {
    return tc::set_tu_wait_limit(ns ? ns : tc::WAIT_LIMIT_NS) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gk
