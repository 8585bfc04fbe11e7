// gemm_tc.cu -- tcgen05 tensor-core GEMM for sm_103a with fused epilogues.
//
// D[M,N] = A[M,K] . B[N,K]^T covering every matmul of the training step:
// matmul_forward (K-major A and B), and matmul_backward's dX = dY W
// (K-major A, MN-major B) and dW += dY^T X (MN-major A and B) (llm.c
// "train_gpt2.cu", matmul_forward_cublaslt / matmul_backward).
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      one elected thread issues TMA tile loads (128-byte swizzle)
//               into a STAGES-deep shared-memory ring guarded by mbarriers;
//   warp 1      allocates TMEM; one elected thread issues tcgen05.mma
//               (M=128, N=BN, fp32 accumulators in TMEM) and commits each
//               stage back to the producer;
//   warps 2..9  epilogue: tcgen05.ld the accumulator (each warp reads 32 rows
//               of its TMEM lane quarter, one row per thread, and half of the
//               columns of every sub-tile), apply
//               bias / GELU / residual / GELU-backward / += in 128-byte-wide
//               column sub-tiles staged in 128B-swizzled shared memory: the
//               residual / GELU input / += operand arrives by TMA load
//               (prefetched one sub-tile ahead) and results leave by TMA
//               store, so no thread touches global memory row by row and the
//               ragged tails are clipped by the tensor maps.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1. Every mbarrier wait is bounded in time; on expiry the CTA records
// DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <stdlib.h>

#include <mutex>
#include <type_traits>

namespace gk {
namespace tc {

constexpr int BM = 128;
constexpr int ROWB = 128;  // bytes of K held per shared-memory row (one swizzle span)
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half of a sub-tile's columns
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int NUM_THREADS = 64 + EPI_THREADS;
constexpr int GROUP_M = 16;  // m-blocks per rasterisation group (L2 locality of A and B)

constexpr int EPI_BUF_BYTES = BM * ROWB;  // one epilogue staging buffer: 128 rows x 128 bytes
// staging buffers per epilogue: the two-output and element-heavy epilogues
// take four, so that two sub-tiles' stores (and the next operand load) stay
// in flight while the next sub-tile is written; the rest keep two and one
// more pipeline stage
template <int EPI> __host__ __device__ constexpr int epi_bufs() {
    return (EPI == EPI_GELU || EPI == EPI_GELU_BWD || EPI == EPI_SPLITK) ? 4 : 2;
}

// CG = CTAs per MMA: 1 (tcgen05 cta_group::1, 128 x BN tiles) or 2 (a CTA
// pair runs cta_group::2 MMAs on 256 x BN tiles; each CTA holds 128 rows of A
// and BN/2 rows of B in its shared memory and its 128 accumulator rows in TMEM)
template <int BN, int CG, int EB> struct Cfg {
    static constexpr int A_BYTES = BM * ROWB;
    static constexpr int B_BYTES = (BN / CG) * ROWB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_BYTES = 256 + 1024;  // barriers, flags, per-row softmax partials
    static constexpr int STAGES = (224 * 1024 - EB * EPI_BUF_BYTES - BAR_BYTES - 1024) / STAGE_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + EB * EPI_BUF_BYTES + BAR_BYTES + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct Args {
    int M, N, K;
    int num_m, num_n, num_kb;
    int cg;  // CTAs per MMA (1 or 2)
    int a_mn, b_mn;
    void* D;
    long long ldd;
    const void* bias;
    const void* aux;
    long long ldaux;
    void* D2;
    float* part;
    int part_ld;
    int splits, kb_per;  // split-K: K ranges per tile and k-blocks per range
    unsigned int* err;
};

// tile order: groups of GROUP_M consecutive m-blocks (m-block pairs for
// cta_group::2) sweep all n-blocks before the next group starts
DEVI void tile_coords(int st, int num_mg, int num_n, int group, int& mg, int& nb) {
    const int per_group = group * num_n;
    const int g = st / per_group, idx = st - g * per_group;
    const int first = g * group;
    const int gm = min(group, num_mg - first);
    mg = first + idx % gm;
    nb = idx / gm;
}

// barrier 1 among the epilogue threads
DEVI void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory"); }

// ------------------------------------------------------------------ epilogue
// One 128-byte-wide column sub-tile (SUBN columns) of one row: the thread's
// accumulator values v[], its row `rl` inside the tile, and the staging
// buffers (128 rows x 128 bytes, 16-byte chunk k of row r at chunk k ^ (r & 7)).
// buf0 holds the TMA-loaded operand (residual, GELU input or the current D)
// and receives the result; buf1 receives the second output of EPI_GELU.
template <typename T, int EPI>
DEVI void epilogue_subtile(const Args& a, const float* v, uint8_t* buf0, uint8_t* buf1, int rl,
                           int row, int n0s, int kbeg, float& pmax, float& psum) {
    constexpr int VEC = Vec16<T>::N;
    const T* bias = (const T*)a.bias;
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
        const int k = kbeg + kk;  // 16-byte chunk of the 128-byte row
        const int off = rl * ROWB + ((k ^ (rl & 7)) << 4);
        const int n = n0s + k * VEC;
        const bool colok = n < a.N;
        float x[VEC];
#pragma unroll
        for (int e = 0; e < VEC; e++) x[e] = v[kk * VEC + e];
        if constexpr (EPI == EPI_STORE || EPI == EPI_GELU || EPI == EPI_RESID ||
                      EPI == EPI_GELU_PART) {
            if (bias && colok) {
                Vec16<T> bb = ld16(bias + n);
#pragma unroll
                for (int e = 0; e < VEC; e++) x[e] += to_f(bb.v[e]);
            }
        }
        Vec16<T> o;
        if constexpr (EPI == EPI_STORE) {
#pragma unroll
            for (int e = 0; e < VEC; e++) o.v[e] = from_f<T>(x[e]);
        } else if constexpr (EPI == EPI_GELU) {
            Vec16<T> g;
#pragma unroll
            for (int e = 0; e < VEC; e++) {
                o.v[e] = from_f<T>(x[e]);
                g.v[e] = from_f<T>(sizeof(T) == 2 ? gelu_fwd_fast(to_f(o.v[e])) : gelu_fwd(to_f(o.v[e])));
            }
            *reinterpret_cast<int4*>(buf1 + off) = *reinterpret_cast<const int4*>(&g);
        } else if constexpr (EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_ACCUM) {
            Vec16<T> r;
            *reinterpret_cast<int4*>(&r) = *reinterpret_cast<const int4*>(buf0 + off);
#pragma unroll
            for (int e = 0; e < VEC; e++) {
                const float rv = to_f(r.v[e]);
                if constexpr (EPI == EPI_RESID) o.v[e] = from_f<T>(x[e] + rv);
                else if constexpr (EPI == EPI_GELU_BWD)
                    o.v[e] = from_f<T>(x[e] * (sizeof(T) == 2 ? gelu_grad_fast(rv) : gelu_grad(rv)));
                else o.v[e] = from_f<T>(rv + x[e]);
            }
        } else if constexpr (EPI == EPI_GELU_PART) {
            float cm = pmax;
#pragma unroll
            for (int e = 0; e < VEC; e++) {
                x[e] = gelu_fwd(x[e]);
                cm = fmaxf(cm, x[e]);
            }
#pragma unroll
            for (int e = 0; e < VEC; e++) o.v[e] = from_f<T>(x[e]);
            if (colok && row < a.M) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; e++) s += expf(x[e] - cm);
                psum = psum * expf(pmax - cm) + s;
                pmax = cm;
            }
        }
        *reinterpret_cast<int4*>(buf0 + off) = *reinterpret_cast<const int4*>(&o);
    }
}

// ------------------------------------------------------------------ kernel
template <int BN, int KIND, int EPI, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_k(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
              const __grid_constant__ CUtensorMap tmX, const __grid_constant__ Args args) {
    constexpr int EPI_BUFS = epi_bufs<EPI>();
    using C = Cfg<BN, CG, EPI_BUFS>;
    using T = typename std::conditional<KIND == 0, bf16, float>::type;
    constexpr int KE = ROWB / (int)sizeof(T);  // K elements per stage
    constexpr int UK = KIND == 0 ? 16 : 8;     // K elements per MMA
    constexpr int KSTEPS = KE / UK;            // MMAs per stage (4)
    constexpr int SUBN = ROWB / (int)sizeof(T);  // epilogue sub-tile width (columns)
    constexpr int NSUB = BN / SUBN;
    constexpr int BNC = BN / CG;               // rows of B this CTA holds
    constexpr bool HAS_AUX = EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_ACCUM;
    // staging buffers per sub-tile: EPI_GELU's two outputs; EPI_SPLITK's fp32
    // sub-tile is 256 bytes wide (one buffer per column half)
    constexpr int OUTS = (EPI == EPI_GELU || EPI == EPI_SPLITK) ? 2 : 1;
    static_assert(EPI != EPI_SPLITK || KIND == 0, "split-K partials: bf16 operands only");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t ebuf = base + C::STAGES * C::STAGE_BYTES;
    uint8_t* ebuf_ptr = base_ptr + C::STAGES * C::STAGE_BYTES;
    const uint32_t bars = ebuf + EPI_BUFS * EPI_BUF_BYTES;
    uint8_t* bars_ptr = ebuf_ptr + EPI_BUFS * EPI_BUF_BYTES;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
    auto tfull = [&](int a) { return bars + 8u * (2 * C::STAGES + a); };
    auto tempty = [&](int a) { return bars + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t drain = bars + 8u * (2 * C::STAGES + 4);
    auto auxfull = [&](int b) { return bars + 8u * (2 * C::STAGES + 5 + b); };
    constexpr int NBARS = 2 * C::STAGES + 5 + EPI_BUFS;
    static_assert(8 * NBARS + 16 <= 256, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);
    volatile int* epi_abort = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 12);
    float2* row_part = reinterpret_cast<float2*>(bars_ptr + 256);  // [BM] softmax partials

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int rank = CG == 2 ? (int)(cluster_rank() & 1u) : 0;  // 0: pair leader (issues MMAs)
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), CG);  // one arrival from each CTA's epilogue
        }
        mbar_init(drain, 1);
        for (int b = 0; b < EPI_BUFS; b++) mbar_init(auxfull(b), 1);
        *abort_flag = 0;
        *n_issued_smem = 0;
        *epi_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (CG == 2) cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    const uint32_t tmem_base = *tmem_slot;
    pdl_enter();  // global memory is touched only from here on
    // a pair of CTAs takes an m-block pair (rows m0 .. m0+255) of one n-block
    const int num_mg = (args.num_m + CG - 1) / CG;
    const int num_super = num_mg * args.num_n;
    // work units: K range `split` of tile `st % num_super`, split-major so that
    // concurrent units share their K range of A and B in L2
    const int num_units = num_super * args.splits;
    const int group = GROUP_M / CG;
    const int cid = (int)blockIdx.x / CG, ncl = (int)gridDim.x / CG;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs of a pair)
            int stage = 0, n_issued = 0;
            uint32_t phase = 0;
            for (int st = cid; st < num_units; st += ncl) {
                int mg, nbk;
                tile_coords(st % num_super, num_mg, args.num_n, group, mg, nbk);
                const int m0 = (mg * CG + rank) * BM, n0 = nbk * BN;
                const int kb0 = (st / num_super) * args.kb_per;
                const int kb1 = min(args.num_kb, kb0 + args.kb_per);
                bool ok = true;
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t sa = base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    const int k0 = kb * KE;
                    uint32_t bar = full(stage);
                    if constexpr (CG == 2) bar = mapa_rank(bar, 0);  // completions go to the leader
                    if (rank == 0) mbar_expect_tx(full(stage), CG * C::STAGE_BYTES);
                    auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y) {
                        if constexpr (CG == 1) tma_load_2d(dst, tm, bar, x, y);
                        else tma_load_2d_pair(dst, tm, bar, x, y);
                    };
                    if (!args.a_mn) {
                        load(sa, &tmA, k0, m0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / KE; j++) load(sa + j * KE * ROWB, &tmA, m0 + j * KE, k0);
                    }
                    // this CTA's BN/CG rows of B
                    if (!args.b_mn) {
                        load(sb, &tmB, k0, n0 + rank * BNC);
                    } else {
#pragma unroll
                        for (int j = 0; j < BNC / KE; j++)
                            load(sb + j * KE * ROWB, &tmB, n0 + rank * BNC + j * KE, k0);
                    }
                    ++n_issued;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            *n_issued_smem = n_issued;
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (the pair leader)
            const uint32_t id = idesc<KIND>(args.a_mn, args.b_mn, BM * CG, BN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int st = cid; st < num_units; st += ncl) {
                if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                const int kb0 = (st / num_super) * args.kb_per;
                const int kb1 = min(args.num_kb, kb0 + args.kb_per);
                bool ok = true;
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(full(stage), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < KSTEPS; k++) {
                        const uint64_t da = args.a_mn
                                                ? sdesc(sa + k * UK * ROWB, KE * ROWB, 1024)
                                                : sdesc(sa + k * UK * (int)sizeof(T), 16, 1024);
                        const uint64_t db = args.b_mn
                                                ? sdesc(sb + k * UK * ROWB, KE * ROWB, 1024)
                                                : sdesc(sb + k * UK * (int)sizeof(T), 16, 1024);
                        umma<KIND, CG>(d, da, db, id, (kb > kb0 || k) ? 1u : 0u);
                    }
                    umma_commit<CG>(empty(stage));  // frees the stage in every CTA of the pair
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit<CG>(tfull(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue warps 2..9
        // Every epilogue thread runs every iteration (the named barriers stay
        // matched); after an expired wait the work is skipped, not the loop.
        const int q = warp & 3;         // TMEM lane quarter this warp may access
        const int hh = (warp - 2) >> 2;  // which half of each sub-tile's columns
        const int rl = q * 32 + lane;
        const bool elected = warp == 2 && lane == 0;
        constexpr int HALF = SUBN / 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        int u = 0;  // sub-tile counter: staging buffer rotation and aux barrier phases
        bool aborted = false;
        int last_aux_u[EPI_BUFS];  // latest aux load per buffer (elected thread)
        for (int b = 0; b < EPI_BUFS; b++) last_aux_u[b] = -1;
        if constexpr (HAS_AUX) {
            if (elected && cid < num_units) {
                int mg, nbk;
                tile_coords(cid % num_super, num_mg, args.num_n, group, mg, nbk);
                mbar_expect_tx(auxfull(0), EPI_BUF_BYTES);
                tma_load_2d(ebuf, &tmX, auxfull(0), nbk * BN, (mg * CG + rank) * BM);
                last_aux_u[0] = 0;
            }
        }
        for (int st = cid; st < num_units; st += ncl) {
            int mg, nb;
            tile_coords(st % num_super, num_mg, args.num_n, group, mg, nb);
            const int split = st / num_super;
            const int m0 = (mg * CG + rank) * BM, n0 = nb * BN;
            int ok = 1;
            if (lane == 0 && !aborted) ok = mbar_wait(tfull(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                aborted = true;
                *epi_abort = 1;
            }
            if (!aborted) tc_fence_after();
            const int row = m0 + rl;
            float pmax = -INFINITY, psum = 0.f;
#pragma unroll 1
            for (int j = 0; j < NSUB; j++, u++) {
                const int b0 = (u * OUTS) % EPI_BUFS;
                if (elected && !aborted) {
                    if constexpr (HAS_AUX) {
                        // prefetch the next sub-tile's operand into the next buffer
                        int nt = st, nj = j + 1;
                        if (nj == NSUB) { nt = st + ncl; nj = 0; }
                        if (nt < num_units) {
                            const int nb1 = (u + 1) % EPI_BUFS;
                            int nmg, nnb;
                            tile_coords(nt % num_super, num_mg, args.num_n, group, nmg, nnb);
                            // the store that last read buffer nb1 is done
                            bulk_wait_read<EPI_BUFS - 2>();
                            mbar_expect_tx(auxfull(nb1), EPI_BUF_BYTES);
                            tma_load_2d(ebuf + nb1 * EPI_BUF_BYTES, &tmX, auxfull(nb1),
                                        nnb * BN + nj * SUBN, (nmg * CG + rank) * BM);
                            last_aux_u[nb1] = u + 1;
                        }
                        if (!mbar_wait(auxfull(b0), (uint32_t)((u / EPI_BUFS) & 1), abort_flag)) {
                            aborted = true;
                            *epi_abort = 1;
                        }
                    } else {
                        bulk_wait_read<EPI_BUFS / OUTS - 1>();  // buffers b0.. are free again
                    }
                }
                epi_bar();  // operands landed / buffers free
                int ab = aborted || *epi_abort;
                ab = __shfl_sync(0xffffffffu, ab, 0);
                aborted = ab != 0;
                if (!aborted) {
                    float v[HALF];
                    const uint32_t taddr = tmem_base + (uint32_t)(acc * BN + j * SUBN + hh * HALF) +
                                           ((uint32_t)(q * 32) << 16);
                    if constexpr (HALF == 32) tmem_ld32(taddr, v);
                    else tmem_ld16(taddr, v);
                    if constexpr (EPI == EPI_SPLITK) {
                        // this half's 32 fp32 columns = one 128-byte staging row
                        uint8_t* bp = ebuf_ptr + (b0 + hh) * EPI_BUF_BYTES + rl * ROWB;
#pragma unroll
                        for (int k = 0; k < 8; k++)
                            *reinterpret_cast<float4*>(bp + ((k ^ (rl & 7)) << 4)) =
                                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    } else {
                        epilogue_subtile<T, EPI>(args, v, ebuf_ptr + b0 * EPI_BUF_BYTES,
                                                 ebuf_ptr + ((b0 + 1) % EPI_BUFS) * EPI_BUF_BYTES, rl,
                                                 row, n0 + j * SUBN, hh * 4, pmax, psum);
                    }
                }
                fence_async_smem();
                epi_bar();  // staging written
                if (elected && !aborted) {
                    if constexpr (EPI == EPI_SPLITK) {
                        // (N, M, splits) fp32 map: ragged rows clip inside their own slice
                        tma_store_3d(&tmD, ebuf + b0 * EPI_BUF_BYTES, n0 + j * SUBN, m0, split);
                        tma_store_3d(&tmD, ebuf + (b0 + 1) * EPI_BUF_BYTES, n0 + j * SUBN + HALF, m0, split);
                    } else {
                        tma_store_2d(&tmD, ebuf + b0 * EPI_BUF_BYTES, n0 + j * SUBN, m0);
                        if constexpr (EPI == EPI_GELU)
                            tma_store_2d(&tmD2, ebuf + (b0 + 1) * EPI_BUF_BYTES, n0 + j * SUBN, m0);
                    }
                    bulk_commit();
                }
            }
            if constexpr (EPI == EPI_GELU_PART) {
                // merge the two column halves of the row, then one partial per (row, tile)
                if (hh == 1) row_part[rl] = make_float2(pmax, psum);
                epi_bar();
                if (hh == 0 && row < args.M && !aborted) {
                    const float2 o = row_part[rl];
                    const float m = fmaxf(pmax, o.x);
                    float sum = 0.f;
                    if (pmax != -INFINITY) sum += psum * expf(pmax - m);
                    if (o.x != -INFINITY) sum += o.y * expf(o.x - m);
                    reinterpret_cast<float2*>(args.part)[(size_t)row * args.part_ld + nb] =
                        make_float2(m, sum);
                }
            }
            // this CTA's accumulator rows are read: release them to the leader's MMA
            if (!aborted) tc_fence_before();
            epi_bar();
            if (elected) {
                if constexpr (CG == 1) mbar_arrive(tempty(acc));
                else mbar_arrive_cluster(mapa_rank(tempty(acc), 0));
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (elected) {
            bulk_wait_all();
            if (aborted) {
                for (int b = 0; b < EPI_BUFS; b++)
                    if (last_aux_u[b] >= 0)
                        mbar_wait_drain(auxfull(b), (uint32_t)((last_aux_u[b] / EPI_BUFS) & 1));
            }
        }
    }

    __syncthreads();
    if (*abort_flag || *epi_abort) {
        // drain: wait for every TMA copy this CTA issued, and for all MMAs issued so far
        if (threadIdx.x == 0) {
            const int n_issued = *n_issued_smem;
            if (rank == 0) {
                for (int s = 0; s < C::STAGES; s++) {
                    if (n_issued > s) {
                        const int last = s + ((n_issued - 1 - s) / C::STAGES) * C::STAGES;
                        mbar_wait_drain(full(s), (uint32_t)((last / C::STAGES) & 1));
                    }
                }
            }
            atomicOr(args.err, DEVERR_TIMEOUT);
        }
        if (threadIdx.x == 32 && rank == 0) {
            umma_commit_local<CG>(drain);
            mbar_wait_drain(drain, 0);
        }
        __syncthreads();
    }
    if constexpr (CG == 2) cluster_sync();  // the peer's arrivals and copies are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tc

// ------------------------------------------------------------------ host side
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

// 2-D tiled map over a row-major matrix with `rows` rows of `inner` elements
// (row pitch ld elements); box = box_inner x box_outer, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* ptr, DType dt, uint64_t inner, uint64_t rows,
                     long long ld, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    const size_t esz = dt == DT_BF16 ? 2 : 4;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, dt == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// (N, M, S) fp32 map over S consecutive M x N slices (row pitch N): the
// split-K partials; box = box_inner x box_outer x 1, 128-byte swizzle
static bool make_map_3d_f32(CUtensorMap* m, void* ptr, int N, int M, int S, uint32_t box_inner,
                            uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)S};
    cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)M * N * 4};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D[m, n] += sum over s = 0..S-1 (in order) of ws[s][m][n]; 8 columns per thread
__global__ void __launch_bounds__(256) splitk_reduce_k(bf16* __restrict__ D, long long ldd,
                                                       const float* __restrict__ ws, int M, int N,
                                                       int S) {
    pdl_enter();
    const int n8 = N / 8;
    const long long total = (long long)M * n8;
    const size_t slice = (size_t)M * N;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / n8), c = (int)(i % n8) * 8;
        const float* w = ws + (size_t)m * N + c;
        float acc[8];
        {
            const float4 x0 = __ldcs(reinterpret_cast<const float4*>(w));
            const float4 x1 = __ldcs(reinterpret_cast<const float4*>(w + 4));
            acc[0] = x0.x; acc[1] = x0.y; acc[2] = x0.z; acc[3] = x0.w;
            acc[4] = x1.x; acc[5] = x1.y; acc[6] = x1.z; acc[7] = x1.w;
        }
        for (int sp = 1; sp < S; sp++) {
            const float4 x0 = __ldcs(reinterpret_cast<const float4*>(w + sp * slice));
            const float4 x1 = __ldcs(reinterpret_cast<const float4*>(w + sp * slice + 4));
            acc[0] += x0.x; acc[1] += x0.y; acc[2] += x0.z; acc[3] += x0.w;
            acc[4] += x1.x; acc[5] += x1.y; acc[6] += x1.z; acc[7] += x1.w;
        }
        bf16* d = D + (size_t)m * ldd + c;
        Vec16<bf16> o = ld16(d);
#pragma unroll
        for (int e = 0; e < 8; e++) o.v[e] = from_f<bf16>(to_f(o.v[e]) + acc[e]);
        st16(d, o);
    }
}

static int launch_splitk_reduce(bf16* D, long long ldd, const float* ws, int M, int N, int S,
                                cudaStream_t s) {
    const long long total = (long long)M * (N / 8);
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    note_launch(1);
    launch_pdl(splitk_reduce_k, dim3((unsigned)blocks), dim3(256), 0, s, D, ldd, ws, M, N, S);
    return GPT2_OK;
}

struct Maps {
    CUtensorMap a, b, d, d2, x;
};

// Persistent launch: one CTA per SM, or -- for CTA pairs -- as many 2-CTA
// clusters as can be co-resident (cudaOccupancyMaxActiveClusters).
template <int BN, int KIND, int EPI, int CG>
static int launch_tc(const Maps& mp, const tc::Args& a, cudaStream_t s) {
    using C = tc::Cfg<BN, CG, tc::epi_bufs<EPI>()>;
    auto kern = tc::gemm_tc_k<BN, KIND, EPI, CG>;
    static bool attr_done = false;
    static int max_clusters = 0;
    if (!attr_done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
            cudaSuccess)
            return GPT2_ERR_CUDA;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(tc::NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    const long long supers = (long long)((a.num_m + CG - 1) / CG) * a.num_n * a.splits;
    if constexpr (CG == 1) {
        const int sms = num_sms();
        cfg.gridDim = dim3((unsigned)(supers < sms ? supers : sms));
        cfg.attrs = attr;
        cfg.numAttrs = 0;
    } else {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (max_clusters == 0) {
            int n = 0;
            cfg.gridDim = dim3(2 * 64);
            if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess || n < 1)
                return GPT2_ERR_CUDA;
            max_clusters = n;
        }
        const long long ncl = supers < max_clusters ? supers : max_clusters;
        cfg.gridDim = dim3((unsigned)(ncl * 2));
    }
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs++;
    }
    note_launch(1);
    if (cudaLaunchKernelEx(&cfg, kern, mp.a, mp.b, mp.d, mp.d2, mp.x, a) != cudaSuccess)
        return GPT2_ERR_CUDA;
    return GPT2_OK;
}

template <int BN, int KIND, int CG>
static int dispatch_epi(int epi, const Maps& mp, const tc::Args& a, cudaStream_t s) {
    if constexpr (KIND == 0) {
        switch (epi) {
            case EPI_STORE: return launch_tc<BN, KIND, EPI_STORE, CG>(mp, a, s);
            case EPI_GELU: return launch_tc<BN, KIND, EPI_GELU, CG>(mp, a, s);
            case EPI_RESID: return launch_tc<BN, KIND, EPI_RESID, CG>(mp, a, s);
            case EPI_GELU_BWD: return launch_tc<BN, KIND, EPI_GELU_BWD, CG>(mp, a, s);
            case EPI_ACCUM: return launch_tc<BN, KIND, EPI_ACCUM, CG>(mp, a, s);
            case EPI_SPLITK: return launch_tc<BN, KIND, EPI_SPLITK, CG>(mp, a, s);
            default: return GPT2_ERR_CONFIG;
        }
    } else {
        switch (epi) {
            case EPI_STORE: return launch_tc<BN, KIND, EPI_STORE, CG>(mp, a, s);
            case EPI_GELU_PART: return launch_tc<BN, KIND, EPI_GELU_PART, CG>(mp, a, s);
            default: return GPT2_ERR_CONFIG;
        }
    }
}

int gemm_tc_part_tile_n() { return 256; }

static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int gemm_tc(const GemmParams& p, DType dt, cudaStream_t s, unsigned int* err) {
    if (p.M <= 0 || p.N <= 0 || p.K <= 0) return GPT2_ERR_ARG;
    const int esz = dt == DT_BF16 ? 2 : 4;
    const int vec = 16 / esz;
    const int KE = tc::ROWB / esz;
    // tf32 operands only in K-major form
    if (dt == DT_F32 && (!p.a_kmajor || !p.b_kmajor)) return GPT2_ERR_CONFIG;
    if (!al16(p.A) || !al16(p.B) || !al16(p.D) || (p.lda * esz) % 16 || (p.ldb * esz) % 16 ||
        (p.ldd * esz) % 16 || p.N % vec)
        return GPT2_ERR_ALIGN;
    const bool has_aux = p.epi == EPI_RESID || p.epi == EPI_GELU_BWD;
    if (has_aux && (!p.aux || !al16(p.aux) || (p.ldaux * esz) % 16)) return GPT2_ERR_ALIGN;
    if (p.bias && !al16(p.bias)) return GPT2_ERR_ALIGN;
    if (p.epi == EPI_GELU && (!p.D2 || !al16(p.D2))) return GPT2_ERR_ALIGN;

    const int sms = num_sms();
    const long long nm = (p.M + tc::BM - 1) / tc::BM;
    // CTA pairs (256-row MMAs, half of B per CTA) when the m-blocks pair up
    // without much waste; GPT2_GEMM_CG=1 forces single-CTA MMAs
    static const int force_cg = [] {
        const char* e = getenv("GPT2_GEMM_CG");
        return e ? atoi(e) : 0;
    }();
    int cg = (nm >= 2 && (nm % 2 == 0 || nm >= 8)) ? 2 : 1;
    if (force_cg == 1) cg = 1;
    // tile width: 256 (a 256 x 256 pair tile halves the operand traffic per
    // flop of a 256 x 128 one); 128 only for narrow outputs
    int BN = p.N <= 128 ? 128 : 256;
    if (p.epi != EPI_GELU_PART) {
        // GPT2_GEMM_BN=128|256 overrides the choice (tuning)
        static const int force_bn = [] {
            const char* e = getenv("GPT2_GEMM_BN");
            return e ? atoi(e) : 0;
        }();
        if (force_bn == 128 || force_bn == 256) BN = force_bn;
    } else {
        BN = 256;
    }
    tc::Args a;
    a.M = p.M; a.N = p.N; a.K = p.K;
    a.num_m = (int)nm;
    a.cg = cg;
    a.num_n = (p.N + BN - 1) / BN;
    a.num_kb = (p.K + KE - 1) / KE;
    a.a_mn = p.a_kmajor ? 0 : 1;
    a.b_mn = p.b_kmajor ? 0 : 1;
    a.D = p.D; a.ldd = p.ldd; a.bias = p.bias; a.aux = p.aux; a.ldaux = p.ldaux; a.D2 = p.D2;
    a.part = p.part; a.part_ld = p.part_ld; a.err = err;
    a.splits = 1;
    a.kb_per = a.num_kb;
    // Split-K for "+=" products with fewer tiles than CTA slots (the weight
    // grads): each K range writes fp32 partials to the scratch and a second
    // kernel adds them to D in range order (deterministic). The range count
    // minimises a cost model: waves x (k-blocks per range + 6) x 0.25 us per
    // 256-wide k-block, plus the partials' traffic at 5 TB/s.
    if (p.epi == EPI_ACCUM && dt == DT_BF16 && p.ws && p.ws_floats > 0) {
        const long long units = cg == 2 ? sms / 2 : sms;
        const long long tiles = ((nm + cg - 1) / cg) * a.num_n;
        const double t_kb = 0.25 * BN / 256.0, mn = (double)p.M * p.N;
        auto est = [&](int sp) {
            const long long kbp = (a.num_kb + sp - 1) / sp;
            const long long waves = (tiles * sp + units - 1) / units;
            double t = (double)waves * (double)(kbp + 6) * t_kb;
            if (sp > 1) t += (8.0 * sp * mn + 4.0 * mn) / 5e6;
            return t;
        };
        int best = 1;
        double best_t = est(1);
        for (int sp = 2; sp <= 16; sp++) {
            if ((a.num_kb + sp - 1) / sp < 4) break;
            if ((double)sp * mn > (double)p.ws_floats) break;
            const double t = est(sp);
            if (t < best_t * 0.97) { best = sp; best_t = t; }
        }
        if (best > 1) {
            a.kb_per = (a.num_kb + best - 1) / best;
            a.splits = (a.num_kb + a.kb_per - 1) / a.kb_per;
        }
    }

    Maps mp;
    const int SUBN = tc::ROWB / esz;
    bool ok = p.a_kmajor ? make_map(&mp.a, p.A, dt, p.K, p.M, p.lda, KE, tc::BM)
                         : make_map(&mp.a, p.A, dt, p.M, p.K, p.lda, KE, KE);
    ok = ok && (p.b_kmajor ? make_map(&mp.b, p.B, dt, p.K, p.N, p.ldb, KE, BN / cg)
                           : make_map(&mp.b, p.B, dt, p.N, p.K, p.ldb, KE, KE));
    if (a.splits > 1) {
        ok = ok && make_map_3d_f32(&mp.d, p.ws, p.N, p.M, a.splits, 32, tc::BM);
        mp.d2 = mp.d;
        mp.x = mp.d;
        if (!ok) return GPT2_ERR_CUDA;
        const int rc = cg == 2 ? dispatch_epi<256, 0, 2>(EPI_SPLITK, mp, a, s)
                               : dispatch_epi<256, 0, 1>(EPI_SPLITK, mp, a, s);
        if (rc != GPT2_OK) return rc;
        return launch_splitk_reduce((bf16*)p.D, p.ldd, p.ws, p.M, p.N, a.splits, s);
    }
    ok = ok && make_map(&mp.d, p.D, dt, p.N, p.M, p.ldd, SUBN, tc::BM);
    ok = ok && make_map(&mp.d2, p.epi == EPI_GELU ? p.D2 : p.D, dt, p.N, p.M, p.ldd, SUBN, tc::BM);
    if (has_aux) ok = ok && make_map(&mp.x, p.aux, dt, p.N, p.M, p.ldaux, SUBN, tc::BM);
    else ok = ok && make_map(&mp.x, p.D, dt, p.N, p.M, p.ldd, SUBN, tc::BM);  // += reads D itself
    if (!ok) return GPT2_ERR_CUDA;
    if (dt == DT_BF16) {
        if (cg == 2)
            return BN == 256 ? dispatch_epi<256, 0, 2>(p.epi, mp, a, s) : dispatch_epi<128, 0, 2>(p.epi, mp, a, s);
        return BN == 256 ? dispatch_epi<256, 0, 1>(p.epi, mp, a, s) : dispatch_epi<128, 0, 1>(p.epi, mp, a, s);
    }
    if (cg == 2)
        return BN == 256 ? dispatch_epi<256, 1, 2>(p.epi, mp, a, s) : dispatch_epi<128, 1, 2>(p.epi, mp, a, s);
    return BN == 256 ? dispatch_epi<256, 1, 1>(p.epi, mp, a, s) : dispatch_epi<128, 1, 1>(p.epi, mp, a, s);
}

}  // namespace gk
