// attention_tc.cu -- causal flash attention forward on the tcgen05 tensor
// cores (sm_103a), head size 64, bf16 in, fp32 softmax, bf16 out + fp32 LSE.
//
// Computes for every (b, h) and query i: O_i = sum_{j<=i} softmax_j(q_i.k_j /
// sqrt(64)) v_j and LSE_i (llm.c "train_gpt2.cu", attention_forward with
// softmax_forward_kernel5, in flash form: no T x T matrix is stored).
//
// Persistent: one CTA per SM. A work item is 256 consecutive queries of one
// (b, h), taken as two 128-row tiles; items are ordered longest first (the
// last queries see the most keys) and dealt to the CTAs in snake order, so
// every CTA gets a similar number of key blocks. Roles (320 threads):
//   warp 0       TMA: the two Q tiles of each item into a 2-deep buffer, the
//                K and V blocks of 128 keys into a 4-stage ring (3-D tensor map
//                over (3C, T, B): rows past the end of a sequence read as 0);
//   warp 1       issues the MMAs (the whole warp runs the loop, one elected
//                lane issues): S_t = Q_t K^T (M=128, N=128,
//                K=64, both operands in shared memory) and O_t += P_t V
//                (M=128, N=64, K=128) with P_t read from tensor memory and V
//                the MN-major operand. S_t for the next key block (or the next
//                item) is issued as soon as the softmax threads have copied
//                S_t into registers, so it overlaps their exponentials;
//   warps 2..9   two softmax warpgroups, one per query tile (one TMEM lane =
//                one query row = one thread): S row from TMEM, row max,
//                P = exp2(s - m) written back to TMEM as bf16 pairs, and the
//                item's epilogue O / l (staged per warp in shared memory and
//                written by TMA stores) and LSE. A row's reference max m moves
//                only when a block's max exceeds it by more than 8 (so p <=
//                256); the warp then rescales its O rows in TMEM after the
//                previous P.V has completed.
// TMEM, 512 columns: tile t at t*256 holds S (128 fp32 columns), O (+128, 64
// columns) and P (+192, 64 columns of bf16 pairs).
// All waits are bounded; on expiry the CTA records DEVERR_TIMEOUT, drains its
// copies and MMAs and frees TMEM.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

namespace gk {
namespace fatc {
using namespace tc;

constexpr int HSZ = 64;
constexpr int BQ = 128;          // queries per tile
constexpr int NQT = 2;           // query tiles per item
constexpr int BKV = 128;         // keys per block
constexpr int KV_STAGES = 4;
constexpr int Q_BUFS = 2;
constexpr int TILE_BYTES = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr int NUM_THREADS = 64 + NQT * 128;
constexpr int OFF_Q = 0;                                   // [buf][tile]
constexpr int OFF_KV = OFF_Q + Q_BUFS * NQT * TILE_BYTES;  // [stage]: K, then V
constexpr int STG_BYTES = 32 * 128;  // a softmax warp's output staging: 32 rows x 64 16-bit values
constexpr int OFF_STG = OFF_KV + KV_STAGES * 2 * TILE_BYTES;
constexpr int OFF_BAR = OFF_STG + NQT * 4 * STG_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
constexpr int TMEM_COLS = 512;
constexpr int TM_TILE = 256;  // columns per query tile
constexpr int TM_O = 128;
constexpr int TM_P = 192;
constexpr float LN2_F = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.f;  // lazy-rescale threshold (log2 units)

struct FwdArgs {
    void* out;  // bf16 or fp16, as the operands
    float* lse;
    int T, C, NH, BH;
    int nqb, nitems;
    float scale_log2;
    unsigned int* err;
};

// item u (longest first): its (b, h), first query and key blocks per tile
struct Item {
    int bh, q0, n[NQT], nmax;
};
DEVI Item decode_item(const FwdArgs& a, int u) {
    Item it;
    const int qblk = a.nqb - 1 - u / a.BH;
    it.bh = u % a.BH;
    it.q0 = qblk * NQT * BQ;
    it.nmax = 0;
#pragma unroll
    for (int t = 0; t < NQT; t++) {
        const int qs = it.q0 + t * BQ;
        // BQ == BKV: tile t sees key blocks 0 .. qs / BKV
        it.n[t] = qs < a.T ? qs / BKV + 1 : 0;
        it.nmax = max(it.nmax, it.n[t]);
    }
    return it;
}
// the r-th item of CTA c among G CTAs (snake order); -1 past the end
DEVI int item_of(int r, int c, int G, int nitems) {
    const int u = r * G + ((r & 1) ? G - 1 - c : c);
    return u < nitems ? u : -1;
}

// KIND 0: bf16 operands and output, 2: fp16 (the tcgen05 kind::f16 operand type)
template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    flash_fwd_tc_k(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmo,
                   const __grid_constant__ FwdArgs a) {
    using H = typename std::conditional<KIND == 2, f16, bf16>::type;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + OFF_BAR;
    uint8_t* bars_ptr = base_ptr + OFF_BAR;
    auto qfull = [&](int q) { return bars + 8u * q; };
    auto qempty = [&](int q) { return bars + 8u * (2 + q); };
    auto kvfull = [&](int s) { return bars + 8u * (4 + s); };
    auto kvempty = [&](int s) { return bars + 8u * (8 + s); };
    auto sfull = [&](int t) { return bars + 8u * (12 + t); };
    auto sfree = [&](int t) { return bars + 8u * (14 + t); };
    auto pfull = [&](int t) { return bars + 8u * (16 + t); };
    auto pempty = [&](int t) { return bars + 8u * (18 + t); };
    auto ofull = [&](int t) { return bars + 8u * (20 + t); };
    const uint32_t drain = bars + 8u * 22;
    constexpr int NBARS = 23;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* q_issued = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);    // [Q_BUFS]
    int* kv_issued = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 16);  // [KV_STAGES]
    static_assert(8 * NBARS + 16 + 4 * KV_STAGES <= 256, "barrier area");

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int C = a.C;

    if (threadIdx.x == 0) {
        for (int q = 0; q < Q_BUFS; q++) {
            mbar_init(qfull(q), 1);
            mbar_init(qempty(q), 1);
            q_issued[q] = 0;
        }
        for (int s = 0; s < KV_STAGES; s++) {
            mbar_init(kvfull(s), 1);
            mbar_init(kvempty(s), 1);
            kv_issued[s] = 0;
        }
        for (int t = 0; t < NQT; t++) {
            mbar_init(sfull(t), 1);
            mbar_init(sfree(t), 4);  // one arrival per warp of the tile's warpgroup
            mbar_init(pfull(t), 4);
            mbar_init(pempty(t), 1);
            mbar_init(ofull(t), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
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
            // copies issued per Q buffer and ring slot are counted in shared
            // memory (read when draining after an abort)
            int kb = 0;
            bool ok = true;
            for (int r = 0, u; ok && (u = item_of(r, c, G, a.nitems)) >= 0; r++) {
                const Item it = decode_item(a, u);
                const int b = it.bh / a.NH, h = it.bh % a.NH;
                const int qb = r & 1;
                if (!mbar_wait(qempty(qb), (uint32_t)(((r >> 1) & 1) ^ 1), abort_flag)) break;
                mbar_expect_tx(qfull(qb), NQT * TILE_BYTES);
                for (int t = 0; t < NQT; t++)
                    tma_load_3d(base + OFF_Q + (qb * NQT + t) * TILE_BYTES, &tm, qfull(qb), h * HSZ,
                                it.q0 + t * BQ, b);
                ++q_issued[qb];
                for (int i = 0; i < it.nmax; i++, kb++) {
                    const int st = kb % KV_STAGES;
                    if (!mbar_wait(kvempty(st), (uint32_t)(((kb / KV_STAGES) & 1) ^ 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kv = base + OFF_KV + st * 2 * TILE_BYTES;
                    mbar_expect_tx(kvfull(st), 2 * TILE_BYTES);
                    tma_load_3d(kv, &tm, kvfull(st), C + h * HSZ, i * BKV, b);
                    tma_load_3d(kv + TILE_BYTES, &tm, kvfull(st), 2 * C + h * HSZ, i * BKV, b);
                    ++kv_issued[st];
                }
            }
        }
    } else if (warp == 1) {
        {
            // ---------------- MMA issuer (the whole warp runs it, one elected lane issues)
            const uint32_t idS = idesc<KIND>(0, 0, BQ, BKV);
            const uint32_t idPV = idesc<KIND>(0, 1, BQ, HSZ);
            int ns[NQT] = {0, 0}, npv[NQT] = {0, 0};
            // bit s: the current fill of ring slot s (bit 4 + b: of Q buffer b)
            // has been waited for; cleared when the slot is handed back
            uint32_t seen = 0;
            bool ok = true;
            auto wait_once = [&](uint32_t bit, uint32_t bar, uint32_t parity) -> bool {
                if (seen & bit) return true;
                if (!mbar_wait_warp(bar, parity, abort_flag)) return false;
                seen |= bit;
                return true;
            };
            // S_t = Q_t K^T for the CTA's r-th item (Q buffer r & 1) against
            // the key block in ring position kb
            auto issue_s = [&](int t, int r, int kb) -> bool {
                if (ns[t] > 0 && !mbar_wait_warp(sfree(t), (uint32_t)((ns[t] - 1) & 1), abort_flag)) return false;
                const int st = kb % KV_STAGES;
                if (!wait_once(16u << (r & 1), qfull(r & 1), (uint32_t)((r >> 1) & 1))) return false;
                if (!wait_once(1u << st, kvfull(st), (uint32_t)((kb / KV_STAGES) & 1))) return false;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(t * TM_TILE);
                const uint64_t dq = sdesc(base + OFF_Q + ((r & 1) * NQT + t) * TILE_BYTES, 16, 1024);
                const uint64_t dk = sdesc(base + OFF_KV + st * 2 * TILE_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < HSZ / 16; kk++)  // +32 bytes along K per step
                    umma_warp<KIND, 1>(d, dq + 2 * kk, dk + 2 * kk, idS, kk ? 1u : 0u);
                umma_commit_warp<1>(sfull(t));
                ++ns[t];
                return true;
            };
            int kb0 = 0;  // ring position of the current item's key block 0
            int u = item_of(0, c, G, a.nitems);
            Item it = decode_item(a, u >= 0 ? u : 0);
            if (u >= 0) {
#pragma unroll
                for (int t = 0; t < NQT; t++)
                    if (ok && it.n[t] > 0) ok = issue_s(t, 0, 0);
            }
            for (int r = 0; ok && u >= 0; r++) {
                const int un = item_of(r + 1, c, G, a.nitems);
                const Item nx = decode_item(a, un >= 0 ? un : 0);
                for (int i = 0; ok && i < it.nmax; i++) {
#pragma unroll
                    for (int t = 0; t < NQT; t++) {
                        if (!ok) continue;
                        if (i + 1 < it.n[t]) {
                            ok = issue_s(t, r, kb0 + i + 1);
                        } else if (un >= 0 && nx.n[t] > 0 &&
                                   i == (it.n[t] > 0 ? it.n[t] - 1 : it.nmax - 1)) {
                            ok = issue_s(t, r + 1, kb0 + it.nmax);  // block 0 of the next item
                        }
                    }
                    const int st = (kb0 + i) % KV_STAGES;
                    const uint64_t dv = sdesc(base + OFF_KV + st * 2 * TILE_BYTES + TILE_BYTES, 8192, 1024);
#pragma unroll
                    for (int t = 0; t < NQT; t++) {
                        if (!ok || i >= it.n[t]) continue;
                        if (!mbar_wait_warp(pfull(t), (uint32_t)(npv[t] & 1), abort_flag)) {
                            ok = false;
                            continue;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + (uint32_t)(t * TM_TILE + TM_O);
                        const uint32_t p = tmem_base + (uint32_t)(t * TM_TILE + TM_P);
#pragma unroll
                        for (int kk = 0; kk < BKV / 16; kk++)  // 16 keys = 8 P columns, 2048 bytes of V
                            umma_ts_warp(d, p + (uint32_t)(kk * 8), dv + 128 * kk, idPV, (i | kk) ? 1u : 0u);
                        umma_commit_warp<1>(pempty(t));
                        if (i == it.n[t] - 1) umma_commit_warp<1>(ofull(t));  // O_t of this item is complete
                        ++npv[t];
                    }
                    if (ok) {
                        umma_commit_warp<1>(kvempty(st));  // K/V of this slot are no longer read
                        seen &= ~(1u << st);
                    }
                }
                if (ok) {
                    umma_commit_warp<1>(qempty(r & 1));  // every S of this item is issued
                    seen &= ~(16u << (r & 1));
                }
                kb0 += it.nmax;
                u = un;
                it = nx;
            }
        }
    } else {
        // ---------------- softmax warpgroups
        const int t = (warp - 2) >> 2;
        const int qq = warp & 3;  // TMEM lane quarter
        const int row = qq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
        const uint32_t tS = tmem_base + (uint32_t)(t * TM_TILE) + lane_off;
        const uint32_t tO = tS + TM_O;
        const uint32_t tP = tS + TM_P;
        uint8_t* stg = base_ptr + OFF_STG + (warp - 2) * STG_BYTES;
        const uint32_t stg_s = base + OFF_STG + (uint32_t)((warp - 2) * STG_BYTES);
        const float sl = a.scale_log2;
        int g = 0, nout = 0;
        bool ok = true;
        auto wait_warp = [&](uint32_t bar, uint32_t parity) {
            int w = 1;
            if (lane == 0) w = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
            w = __shfl_sync(0xffffffffu, w, 0);
            return w != 0;
        };
        for (int r = 0, u; ok && (u = item_of(r, c, G, a.nitems)) >= 0; r++) {
            const Item it = decode_item(a, u);
            const int n = t == 0 ? it.n[0] : it.n[1];
            if (n == 0) continue;
            const int query = it.q0 + t * BQ + row;
            float m = -INFINITY, l = 0.f;
            for (int i = 0; i < n; i++, g++) {
                if (!wait_warp(sfull(t), (uint32_t)(g & 1))) { ok = false; break; }
                tc_fence_after();
                float s[128];
                tmem_ld64(tS, *reinterpret_cast<float(*)[64]>(&s[0]));
                tmem_ld64(tS + 64, *reinterpret_cast<float(*)[64]>(&s[64]));
                // S_t may now be overwritten by the next Q K^T
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree(t));
                const int k0 = i * BKV;
                if (k0 + BKV - 1 > it.q0 + t * BQ) {  // diagonal block: keys after the query are masked
                    const int lim = query - k0;
#pragma unroll
                    for (int j = 0; j < 128; j++) s[j] = j <= lim ? s[j] : -INFINITY;
                }
                float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int j = 4; j < 124; j += 8) {
                    m4[0] = fmax3(m4[0], s[j], s[j + 1]);
                    m4[1] = fmax3(m4[1], s[j + 2], s[j + 3]);
                    m4[2] = fmax3(m4[2], s[j + 4], s[j + 5]);
                    m4[3] = fmax3(m4[3], s[j + 6], s[j + 7]);
                }
                m4[0] = fmax3(m4[0], s[124], s[125]);
                m4[1] = fmax3(m4[1], s[126], s[127]);
                const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]) * sl;
                // P_t (and O_t) may be written once the previous P.V is done
                if (!wait_warp(pempty(t), (uint32_t)((g & 1) ^ 1))) { ok = false; break; }
                tc_fence_after();
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
                const float2 sc2 = make_float2(sl, sl), nm2 = make_float2(-m, -m);
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int ch = 0; ch < 4; ch++) {  // 32 keys = 16 columns of bf16 pairs
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) {
                        const int j = ch * 32 + 2 * e;
                        float2 x = ffma2(make_float2(s[j], s[j + 1]), sc2, nm2);
                        x.x = ex2_approx(x.x);
                        x.y = ex2_approx(x.y);
                        acc[e & 1] = fadd2(acc[e & 1], x);
                        pk[e] = f2_h2<H>(x.x, x.y);
                    }
                    tmem_st16_nowait(tP + ch * 16, pk);
                }
                tmem_wait_st();
                l += (acc[0].x + acc[1].x) + (acc[0].y + acc[1].y);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull(t));
            }
            if (!ok) break;
            // the item's last P.V completes O_t
            if (!wait_warp(ofull(t), (uint32_t)(nout & 1))) { ok = false; break; }
            ++nout;
            tc_fence_after();
            float ov[64];
            tmem_ld64(tO, ov);
            // O_t is read: the next item's first P.V may overwrite it (it is
            // issued after this warpgroup's next pfull arrival)
            tc_fence_before();
            const int b = it.bh / a.NH, h = it.bh % a.NH;
            const float inv = 1.f / l;
            uint32_t pk[HSZ / 2];
#pragma unroll
            for (int d = 0; d < HSZ / 2; d++) pk[d] = f2_h2<H>(ov[2 * d] * inv, ov[2 * d + 1] * inv);
            // the warp's 32 output rows through its staging buffer (128-byte
            // swizzle) and one TMA store, once its previous store has read it;
            // rows past the sequence end are clipped by the store
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; k++)
                *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0 && it.q0 + t * BQ + qq * 32 < a.T) {  // (no store wholly past the end)
                tma_store_3d(&tmo, stg_s, h * HSZ, it.q0 + t * BQ + qq * 32, b);
                bulk_commit();
            }
            if (query < a.T) a.lse[(size_t)it.bh * a.T + query] = (m + log2f(l)) * LN2_F;
        }
        if (lane == 0) bulk_wait_all();  // the output stores are complete before the CTA exits
    }

    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) {
            // wait for every copy this CTA issued: the last phase of each barrier
            for (int q = 0; q < Q_BUFS; q++)
                if (q_issued[q] > 0) mbar_wait_drain(qfull(q), (uint32_t)((q_issued[q] - 1) & 1));
            for (int s = 0; s < KV_STAGES; s++)
                if (kv_issued[s] > 0) mbar_wait_drain(kvfull(s), (uint32_t)((kv_issued[s] - 1) & 1));
            atomicOr(a.err, DEVERR_TIMEOUT);
        }
        if (warp == 1) {  // the issuing lane commits (elected as when issuing)
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

// qkv (B, T, 3C) bf16 or fp16 viewed as a 3-D tensor (3C, T, B); 64 x 128 x 1 boxes
int launch_flash_forward_tc(DType dt, void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
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
    if (dt != DT_BF16 && dt != DT_F16) return set_error(GPT2_ERR_CONFIG, "flash forward: 16-bit operands only");
    if (fn(&tm, dt == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
           const_cast<void*>(qkv), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return set_error(GPT2_ERR_CUDA, "flash forward: tensor map encoding failed");
    // out (B, T, C) as a 3-D tensor (C, T, B); 64 x 32 x 1 boxes (one softmax warp's rows)
    if ((uintptr_t)out % 16) return set_error(GPT2_ERR_ALIGN, "flash forward: out must be 16-byte aligned");
    CUtensorMap tmo;
    cuuint64_t odims[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t ostrides[2] = {(cuuint64_t)C * 2, (cuuint64_t)T * C * 2};
    cuuint32_t obox[3] = {HSZ, 32, 1};
    if (fn(&tmo, dt == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, odims,
           ostrides, obox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return set_error(GPT2_ERR_CUDA, "flash forward: output tensor map encoding failed");
    auto kern = dt == DT_F16 ? flash_fwd_tc_k<2> : flash_fwd_tc_k<0>;
    static bool attr[2] = {false, false};
    if (!attr[dt == DT_F16]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return set_error(GPT2_ERR_CUDA, "flash forward: shared-memory opt-in failed: %s",
                             cudaGetErrorString(e));
        attr[dt == DT_F16] = true;
    }
    FwdArgs a;
    a.out = out;
    a.lse = lse;
    a.T = T;
    a.C = C;
    a.NH = NH;
    a.BH = B * NH;
    a.nqb = (T + NQT * BQ - 1) / (NQT * BQ);
    a.nitems = a.nqb * a.BH;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)HSZ);
    a.err = err;
    if (a.nitems == 0) return GPT2_OK;
    dim3 grid(std::min(a.nitems, num_sms()));
    note_launch(1);
    launch_pdl(kern, grid, dim3(NUM_THREADS), SMEM_BYTES, s, tm, tmo, a);
    return GPT2_OK;
}

// the bounded-wait limit of this translation unit's kernels (0: the default)
int set_wait_limit_attn_fwd(unsigned long long ns) {
    return tc::set_tu_wait_limit(ns ? ns : tc::WAIT_LIMIT_NS) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gk
