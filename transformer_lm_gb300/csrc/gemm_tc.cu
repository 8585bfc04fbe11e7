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
//   warps 2..9  epilogue: each warp owns the 32 rows of its TMEM lane
//               quarter and every other 128-byte-wide column chunk of a tile
//               (one row per thread): it tcgen05.ld's the chunk, applies bias /
//               GELU / residual / GELU-backward / += (the operand row segment
//               read straight from global memory), stages the result in its own
//               4 KB 128B-swizzled buffer and writes it with its own TMA store.
//               The warps never wait for one another inside a tile; ragged
//               tails are clipped by the tensor maps.
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

constexpr int STG_BYTES = 32 * ROWB;  // an epilogue warp's staging: 32 rows x 128 bytes

// CG = CTAs per MMA: 1 (tcgen05 cta_group::1, 128 x BN tiles) or 2 (a CTA
// pair runs cta_group::2 MMAs on 256 x BN tiles; each CTA holds 128 rows of A
// and BN/2 rows of B in its shared memory and its 128 accumulator rows in TMEM)
// NSTG staging buffers per epilogue warp (two for the two-output GELU epilogue)
template <int BN, int CG, int NSTG = 1> struct Cfg {
    static constexpr int A_BYTES = BM * ROWB;
    static constexpr int B_BYTES = (BN / CG) * ROWB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BYTES = EPI_WARPS * NSTG * STG_BYTES;
    static constexpr int BAR_BYTES = 256;  // barriers and flags
    static constexpr int STAGES = (227 * 1024 - EPI_BYTES - BAR_BYTES - 1024) / STAGE_BYTES;
    static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // two accumulators, power of two
    static constexpr int USED_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
    static_assert(USED_BYTES <= 227 * 1024, "shared memory");
    // Every CTA requests the per-block maximum, whatever its layout uses: a
    // CTA then holds its SM alone, and no CTA of another kernel (one launched
    // early by programmatic dependent launch, or one of the other stream's)
    // shares the SM with the persistent tile loop. With the layout's size
    // alone, small kernels could join a GEMM CTA on its SM; the GPT-2 350M
    // step then stopped making progress now and then (not explained).
    static constexpr int SMEM_BYTES = 227 * 1024;
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
    float* cs;  // EPI_GELU_BWD, optional: column sums of the output per 32-row group
    long long ldcs;
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

// gelu(x) = 0.5 x (1 + tanh(x (K0 + K0 K1 x^2))) for two values, packed fp32
// arithmetic and the hardware tanh (used where the result is rounded to bf16)
DEVI float2 gelu_fwd_fast2(float2 x) {
    const float2 u = fmul2(x, ffma2(fmul2(x, x), make_float2(GELU_K0 * GELU_K1, GELU_K0 * GELU_K1),
                                    make_float2(GELU_K0, GELU_K0)));
    const float2 h = fmul2(x, make_float2(0.5f, 0.5f));
    return ffma2(h, make_float2(tanh_fast(u.x), tanh_fast(u.y)), h);
}
// gelu'(x) for two values with packed fp32 arithmetic and the hardware tanh
// (used where the result is rounded to bf16): with t = tanh(x (K0 + K0 K1 x^2)),
// gelu'(x) = (0.5 + 0.5 t) + x (0.5 K0 + 1.5 K0 K1 x^2) (1 - t^2)
DEVI float2 gelu_grad_fast2(float2 x) {
    const float2 x2 = fmul2(x, x);
    const float2 u = fmul2(x, ffma2(x2, make_float2(GELU_K0 * GELU_K1, GELU_K0 * GELU_K1),
                                    make_float2(GELU_K0, GELU_K0)));
    const float2 t = make_float2(tanh_fast(u.x), tanh_fast(u.y));
    const float2 a = ffma2(t, make_float2(0.5f, 0.5f), make_float2(0.5f, 0.5f));
    const float2 b = fmul2(x, ffma2(x2, make_float2(1.5f * GELU_K0 * GELU_K1, 1.5f * GELU_K0 * GELU_K1),
                                    make_float2(0.5f * GELU_K0, 0.5f * GELU_K0)));
    const float2 omt = ffma2(t, make_float2(-t.x, -t.y), make_float2(1.f, 1.f));
    return ffma2(b, omt, a);
}

// ------------------------------------------------------------------ epilogue
// One 128-byte output chunk of one row: the accumulator values v[OC], the
// chunk's first column nc, the row; the result leaves packed in o (and the
// second output of EPI_GELU in o2). Columns past N are computed but clipped
// by the store.
// The operand row segment of a chunk (residual, GELU input, or D itself for
// +=), read straight from global memory; zeros outside the matrix.
template <typename T, int EPI, int OC>
DEVI void load_operand(const Args& a, int row, int nc, Vec16<T> (&r)[OC * sizeof(T) / 16]) {
    constexpr int VEC = 16 / (int)sizeof(T);
    if constexpr (EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_ACCUM) {
        const T* src = EPI == EPI_ACCUM ? (const T*)a.D + (size_t)row * a.ldd
                                        : (const T*)a.aux + (size_t)row * a.ldaux;
#pragma unroll
        for (int k = 0; k < OC / VEC; k++) {
            if (row < a.M && nc + k * VEC < a.N)
                *reinterpret_cast<int4*>(&r[k]) = *reinterpret_cast<const int4*>(src + nc + k * VEC);
            else
                *reinterpret_cast<int4*>(&r[k]) = make_int4(0, 0, 0, 0);
        }
    }
}

// A chunk's bias (the output's element type, OC columns = 128 bytes) spread
// over the warp: lane l holds its 4-byte word l (columns 2l, 2l + 1 of a
// 16-bit output, column l of fp32); 0 past N or without a bias. Read a chunk
// ahead of its use: every lane needs every column, so the word is broadcast by
// shuffles at use instead of each thread re-reading the 128 bytes.
template <typename TO> DEVI uint32_t load_bias_word(const Args& a, int nc, int lane) {
    constexpr int PER = 4 / (int)sizeof(TO);
    const int c = nc + lane * PER;
    if (!a.bias || c >= a.N) return 0u;
    return __ldg(reinterpret_cast<const unsigned int*>(reinterpret_cast<const TO*>(a.bias) + c));
}

template <typename T, typename TO, int EPI, int OC>
DEVI void epilogue_chunk(const Args& a, float (&v)[OC], const Vec16<T> (&r)[OC * sizeof(T) / 16], int row,
                         int nc, uint32_t bw, uint32_t (&o)[32], uint32_t (&o2)[32]) {
    constexpr int VEC = 16 / (int)sizeof(T);
    if constexpr (EPI == EPI_STORE || EPI == EPI_GELU || EPI == EPI_RESID) {
        if (a.bias) {
#pragma unroll
            for (int e2 = 0; e2 < 32; e2++) {
                const uint32_t w = __shfl_sync(0xffffffffu, bw, e2);
                if constexpr (sizeof(TO) == 2) {
                    const float2 f = h2_f2<TO>(w);
                    v[2 * e2] += f.x;
                    v[2 * e2 + 1] += f.y;
                } else {
                    v[e2] += __uint_as_float(w);
                }
            }
        }
    }
    if constexpr (EPI == EPI_GELU_BWD && sizeof(T) == 2) {
#pragma unroll
        for (int k = 0; k < OC / VEC; k++)
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                const float2 g = gelu_grad_fast2(make_float2(to_f(r[k].v[e]), to_f(r[k].v[e + 1])));
                const float2 y = fmul2(make_float2(v[k * VEC + e], v[k * VEC + e + 1]), g);
                v[k * VEC + e] = y.x;
                v[k * VEC + e + 1] = y.y;
            }
    } else if constexpr (EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_ACCUM) {
#pragma unroll
        for (int k = 0; k < OC / VEC; k++)
#pragma unroll
            for (int e = 0; e < VEC; e++) {
                const float rv = to_f(r[k].v[e]);
                float& x = v[k * VEC + e];
                if constexpr (EPI == EPI_RESID) x += rv;
                else if constexpr (EPI == EPI_GELU_BWD) x *= gelu_grad(rv);
                else x = rv + x;
            }
    }
    if constexpr (sizeof(TO) == 4) {
#pragma unroll
        for (int e = 0; e < 32; e++) o[e] = __float_as_uint(v[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 32; e++) {
            o[e] = f2_h2<TO>(v[2 * e], v[2 * e + 1]);
            if constexpr (EPI == EPI_GELU) {
                // GELU of the rounded pre-activation (what the backward sees)
                const float2 g = gelu_fwd_fast2(h2_f2<TO>(o[e]));
                o2[e] = f2_h2<TO>(g.x, g.y);
            }
        }
    }
}

// a warp's 32 staged rows: row `lane`, 16-byte chunk k at k ^ (lane & 7)
DEVI void stage_row(uint8_t* stg, int lane, const uint32_t (&o)[32]) {
#pragma unroll
    for (int k = 0; k < 8; k++)
        *reinterpret_cast<uint4*>(stg + lane * ROWB + ((k ^ (lane & 7)) << 4)) =
            make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
}

// ------------------------------------------------------------------ kernel
template <int BN, int KIND, int EPI, int CG>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_k(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
              const __grid_constant__ Args args) {
    using C = Cfg<BN, CG, EPI == EPI_GELU ? 2 : 1>;
    // KIND 0: bf16 operands, 1: fp32 (tf32 MMAs), 2: fp16 operands
    using T = typename std::conditional<KIND == 1, float,
                                        typename std::conditional<KIND == 2, f16, bf16>::type>::type;
    constexpr int KE = ROWB / (int)sizeof(T);  // K elements per stage
    constexpr int UK = KIND == 1 ? 8 : 16;     // K elements per MMA
    constexpr int KSTEPS = KE / UK;            // MMAs per stage (4)
    constexpr int BNC = BN / CG;               // rows of B this CTA holds
    // epilogue output: fp32 for kind::tf32 and split-K partials
    // operator's GELU tiles, else the operands' 16-bit type;
    // a 128-byte chunk holds OC output columns
    constexpr bool OUT_F32 = KIND == 1 || EPI == EPI_SPLITK;
    using TO = typename std::conditional<OUT_F32, float, T>::type;
    constexpr int OC = OUT_F32 ? 32 : 64;
    constexpr int NCH = BN / OC;
    static_assert(EPI != EPI_SPLITK || KIND != 1, "split-K partials: 16-bit operands only");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t ebuf = base + C::STAGES * C::STAGE_BYTES;
    uint8_t* ebuf_ptr = base_ptr + C::STAGES * C::STAGE_BYTES;
    const uint32_t bars = ebuf + C::EPI_BYTES;
    uint8_t* bars_ptr = ebuf_ptr + C::EPI_BYTES;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
    auto tfull = [&](int a) { return bars + 8u * (2 * C::STAGES + a); };
    auto tempty = [&](int a) { return bars + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t drain = bars + 8u * (2 * C::STAGES + 4);
    constexpr int NBARS = 2 * C::STAGES + 5;
    static_assert(8 * NBARS + 16 <= 256, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * NBARS + 8);
    volatile int* epi_abort = reinterpret_cast<volatile int*>(bars_ptr + 8 * NBARS + 12);

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int rank = CG == 2 ? (int)(cluster_rank() & 1u) : 0;  // 0: pair leader (issues MMAs)
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), CG * EPI_WARPS);  // one arrival per epilogue warp of each CTA
        }
        mbar_init(drain, 1);
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
        if (rank == 0) {
            // ---------------- MMA issuer (the pair leader): the whole warp runs
            // the loop, one elected lane issues
            const uint32_t id = idesc<KIND>(args.a_mn, args.b_mn, BM * CG, BN);
            // descriptor advance per K step, in 16-byte units: MN-major operands
            // move by UK rows of 128 bytes, K-major ones by UK elements
            const uint32_t lbo_a = args.a_mn ? KE * ROWB : 16, lbo_b = args.b_mn ? KE * ROWB : 16;
            const uint64_t step_a = (uint64_t)((args.a_mn ? UK * ROWB : UK * (int)sizeof(T)) >> 4);
            const uint64_t step_b = (uint64_t)((args.b_mn ? UK * ROWB : UK * (int)sizeof(T)) >> 4);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ready = false;  // the current stage is known to have landed
            for (int st = cid; st < num_units; st += ncl) {
                if (!mbar_wait_warp(tempty(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                const int kb0 = (st / num_super) * args.kb_per;
                const int kb1 = min(args.num_kb, kb0 + args.kb_per);
                bool ok = true;
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!ready && !mbar_wait_warp(full(stage), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = base + stage * C::STAGE_BYTES;
                    const uint64_t da = sdesc(sa, lbo_a, 1024), db = sdesc(sa + C::A_BYTES, lbo_b, 1024);
                    const int nst = stage + 1 == C::STAGES ? 0 : stage + 1;
                    const uint32_t nph = stage + 1 == C::STAGES ? phase ^ 1u : phase;
#pragma unroll
                    for (int k = 0; k < KSTEPS; k++) {
                        // test the next stage while this stage's MMAs are queued,
                        // so a landed stage costs no wait between the groups
                        if (k == KSTEPS - 1) ready = __all_sync(0xffffffffu, mbar_test(full(nst), nph));
                        umma_warp<KIND, CG>(d, da + k * step_a, db + k * step_b, id, (kb > kb0 || k) ? 1u : 0u);
                    }
                    umma_commit_warp<CG>(empty(stage));  // frees the stage in every CTA of the pair
                    stage = nst;
                    phase = nph;
                }
                if (!ok) break;
                umma_commit_warp<CG>(tfull(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue warps 2..9: a warp owns its TMEM lane
        // quarter's 32 rows and the column chunks j = hh, hh + 2, ... of each
        // tile; it stages a chunk in its own buffer and stores it itself.
        // After an expired wait the work is skipped.
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int hh = (warp - 2) >> 2;  // chunk parity
        const int rl = q * 32 + lane;    // row within the tile
        constexpr int NSTG = EPI == EPI_GELU ? 2 : 1;
        uint8_t* stg = ebuf_ptr + (warp - 2) * NSTG * STG_BYTES;
        const uint32_t stg_s = ebuf + (uint32_t)((warp - 2) * NSTG * STG_BYTES);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool aborted = false;
        const uint32_t tempty_leader = CG == 2 ? mapa_rank(tempty(0), 0) : 0u;
        for (int st = cid; st < num_units; st += ncl) {
            int mg, nb;
            tile_coords(st % num_super, num_mg, args.num_n, group, mg, nb);
            const int split = st / num_super;
            const int m0 = (mg * CG + rank) * BM, n0 = nb * BN;
            const int row = m0 + rl;
            // the first chunk's operand is read while the MMAs run
            constexpr int NV = OC * (int)sizeof(T) / 16;
            Vec16<T> r[NV];
            load_operand<T, EPI, OC>(args, row, n0 + hh * OC, r);
            uint32_t bw = load_bias_word<TO>(args, n0 + hh * OC, lane);
            int ok = 1;
            if (lane == 0 && !aborted) ok = mbar_wait(tfull(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || *epi_abort) {
                aborted = true;
                *epi_abort = 1;
            }
            if (!aborted) tc_fence_after();
#pragma unroll 1
            for (int j = hh; j < NCH && !aborted; j += 2) {
                const int nc = n0 + j * OC;
                float v[OC];
                const uint32_t taddr = tmem_base + (uint32_t)(acc * BN + j * OC) + ((uint32_t)(q * 32) << 16);
                if constexpr (OC == 64) tmem_ld64(taddr, v);
                else tmem_ld32(taddr, v);
                Vec16<T> rn[NV];  // the next chunk's operand, in flight during this one
                if (j + 2 < NCH) load_operand<T, EPI, OC>(args, row, nc + 2 * OC, rn);
                const uint32_t bwn = j + 2 < NCH ? load_bias_word<TO>(args, nc + 2 * OC, lane) : 0u;
                uint32_t o[32], o2[32];
                epilogue_chunk<T, TO, EPI, OC>(args, v, r, row, nc, bw, o, o2);
                bw = bwn;
#pragma unroll
                for (int k = 0; k < NV; k++) r[k] = rn[k];
                // this warp's previous stores have read the staging buffer(s)
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                stage_row(stg, lane, o);
                if constexpr (EPI == EPI_GELU) stage_row(stg + STG_BYTES, lane, o2);  // its own buffer
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (EPI == EPI_SPLITK) tma_store_3d(&tmD, stg_s, nc, m0 + q * 32, split);
                    else tma_store_2d(&tmD, stg_s, nc, m0 + q * 32);
                    if constexpr (EPI == EPI_GELU) tma_store_2d(&tmD2, stg_s + STG_BYTES, nc, m0 + q * 32);
                    bulk_commit();
                }
                if constexpr (EPI == EPI_GELU_BWD && sizeof(TO) == 2) {
                    if (args.cs) {
                        // column sums of the staged (rounded) chunk over the warp's
                        // rows, read back from the staging buffer (which the store
                        // only reads too): lane l adds the column pair 2l, 2l + 1
                        const int rows = min(32, args.M - (m0 + q * 32));
                        const int wofs = ((lane >> 2) << 4) | ((lane & 3) << 2);
                        float2 cs2 = make_float2(0.f, 0.f);
#pragma unroll 8
                        for (int rr = 0; rr < rows; rr++) {
                            const uint32_t u = *reinterpret_cast<const uint32_t*>(
                                stg + rr * ROWB + (wofs ^ ((rr & 7) << 4)));
                            cs2 = fadd2(cs2, h2_f2<TO>(u));
                        }
                        if (rows > 0 && nc + 2 * lane < args.N)
                            *reinterpret_cast<float2*>(args.cs + (size_t)((m0 + q * 32) / 32) * args.ldcs + nc +
                                                       2 * lane) = cs2;
                    }
                }
            }
            // this warp's accumulator rows are read: release them to the leader's MMA
            if (!aborted) tc_fence_before();
            __syncwarp();
            if (lane == 0 && !aborted) {
                if constexpr (CG == 1) mbar_arrive(tempty(acc));
                else mbar_arrive_cluster_relaxed(tempty_leader + 8u * (uint32_t)acc);
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_all();
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
        if (CG == 2 && rank == 1 && threadIdx.x == 0) {
            // this CTA's loads complete on the leader's barriers, which it cannot
            // wait on: give any still in flight a bounded time (100 us) to land
            const unsigned long long t0 = globaltimer();
            while (globaltimer() - t0 < 100000ull) {
            }
        }
        if (warp == 1 && rank == 0) {  // the issuing lane commits (elected as when issuing)
            umma_commit_local_warp<CG>(drain);
            if (lane == 0) mbar_wait_drain(drain, 0);
            __syncwarp();
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
    const size_t esz = dtype_size(dt);
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType ty = dt == DT_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dt == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = fn(m, ty,
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

// D[m, n] (+)= sum over s = 0..S-1 (in order) of ws[s][m][n]; 8 columns per thread
template <typename H>
__global__ void __launch_bounds__(256) splitk_reduce_k(H* __restrict__ D, long long ldd,
                                                       const float* __restrict__ ws, int M, int N,
                                                       int S, int accumulate) {
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
        H* d = D + (size_t)m * ldd + c;
        Vec16<H> o;
        if (accumulate) o = ld16(d);  // in flight with the partials
        // four ranges' loads in flight at a time, added in range order
        int sp = 1;
        for (; sp + 3 < S; sp += 4) {
            float4 x[4][2];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                x[j][0] = __ldcs(reinterpret_cast<const float4*>(w + (sp + j) * slice));
                x[j][1] = __ldcs(reinterpret_cast<const float4*>(w + (sp + j) * slice + 4));
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                acc[0] += x[j][0].x; acc[1] += x[j][0].y; acc[2] += x[j][0].z; acc[3] += x[j][0].w;
                acc[4] += x[j][1].x; acc[5] += x[j][1].y; acc[6] += x[j][1].z; acc[7] += x[j][1].w;
            }
        }
        for (; sp < S; sp++) {
            const float4 x0 = __ldcs(reinterpret_cast<const float4*>(w + sp * slice));
            const float4 x1 = __ldcs(reinterpret_cast<const float4*>(w + sp * slice + 4));
            acc[0] += x0.x; acc[1] += x0.y; acc[2] += x0.z; acc[3] += x0.w;
            acc[4] += x1.x; acc[5] += x1.y; acc[6] += x1.z; acc[7] += x1.w;
        }
        if (accumulate) {
#pragma unroll
            for (int e = 0; e < 8; e++) o.v[e] = from_f<H>(to_f(o.v[e]) + acc[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) o.v[e] = from_f<H>(acc[e]);
        }
        st16(d, o);
    }
}

static int launch_splitk_reduce(DType dt, void* D, long long ldd, const float* ws, int M, int N, int S,
                                int accumulate, cudaStream_t s) {
    const long long total = (long long)M * (N / 8);
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    note_launch(1);
    if (dt == DT_F16)
        launch_pdl(splitk_reduce_k<f16>, dim3((unsigned)blocks), dim3(256), 0, s, (f16*)D, ldd, ws, M, N, S,
                   accumulate);
    else
        launch_pdl(splitk_reduce_k<bf16>, dim3((unsigned)blocks), dim3(256), 0, s, (bf16*)D, ldd, ws, M, N, S,
                   accumulate);
    return GPT2_OK;
}

struct Maps {
    CUtensorMap a, b, d, d2;
};

// Persistent launch: one CTA per SM, or -- for CTA pairs -- as many 2-CTA
// clusters as can be co-resident (cudaOccupancyMaxActiveClusters).
template <int BN, int KIND, int EPI, int CG>
static int launch_tc(const Maps& mp, const tc::Args& a, cudaStream_t s) {
    using C = tc::Cfg<BN, CG, EPI == EPI_GELU ? 2 : 1>;
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
    cudaLaunchAttribute attr[3];
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
    cfg.numAttrs += launch_attrs(attr + cfg.numAttrs);
    note_launch(1);
    if (cudaLaunchKernelEx(&cfg, kern, mp.a, mp.b, mp.d, mp.d2, a) != cudaSuccess)
        return GPT2_ERR_CUDA;
    return GPT2_OK;
}

template <int BN, int KIND, int CG>
static int dispatch_epi(int epi, const Maps& mp, const tc::Args& a, cudaStream_t s) {
    if constexpr (KIND != 1) {
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
            default: return GPT2_ERR_CONFIG;
        }
    }
}

static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int gemm_tc(const GemmParams& p, DType dt, cudaStream_t s, unsigned int* err) {
    if (p.M <= 0 || p.N <= 0 || p.K <= 0) return GPT2_ERR_ARG;
    const int esz = (int)dtype_size(dt);
    const int vec = 16 / esz;
    const int KE = tc::ROWB / esz;
    // tf32 operands only in K-major form
    if (dt == DT_F32 && (!p.a_kmajor || !p.b_kmajor)) return GPT2_ERR_CONFIG;
    // the fused operator's GELU tiles (and bias) are fp32 whatever the operands
    const DType out_dt = dt;
    const int osz = (int)dtype_size(out_dt);
    if (!al16(p.A) || !al16(p.B) || !al16(p.D) || (p.lda * esz) % 16 || (p.ldb * esz) % 16 ||
        (p.ldd * osz) % 16 || p.N % (16 / osz) || (dt != DT_F32 && p.N % vec))
        return GPT2_ERR_ALIGN;
    const bool has_aux = p.epi == EPI_RESID || p.epi == EPI_GELU_BWD;
    if (has_aux && (!p.aux || !al16(p.aux) || (p.ldaux * esz) % 16)) return GPT2_ERR_ALIGN;
    if (p.bias && !al16(p.bias)) return GPT2_ERR_ALIGN;
    if (p.epi == EPI_GELU && (!p.D2 || !al16(p.D2))) return GPT2_ERR_ALIGN;
    // column sums: the GELU-backward epilogue of 16-bit outputs only
    if (p.cs && (p.epi != EPI_GELU_BWD || dt == DT_F32 || ((uintptr_t)p.cs & 7u) || (p.ldcs & 1) ||
                 p.ldcs < p.N))
        return GPT2_ERR_CONFIG;

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
    // 192-wide tiles (B K-major only: a CTA's 96 rows of B are one TMA box) when
    // they fill the last wave of CTA pairs markedly better than 256-wide ones
    if (BN == 256 && p.b_kmajor && dt != DT_F32 &&
        (p.epi == EPI_STORE || p.epi == EPI_GELU || p.epi == EPI_RESID || p.epi == EPI_GELU_BWD)) {
        const long long units = cg == 2 ? sms / 2 : sms, mg = (nm + cg - 1) / cg;
        // time ~ waves x tile width
        auto cost = [&](int bn) {
            const long long tiles = mg * ((p.N + bn - 1) / bn);
            return (double)((tiles + units - 1) / units) * bn;
        };
        if (cost(192) < 0.92 * cost(256)) BN = 192;
    }
    {
        // GPT2_GEMM_BN=128|192|256 overrides the choice (tuning; 192 with K-major B only)
        static const int force_bn = [] {
            const char* e = getenv("GPT2_GEMM_BN");
            return e ? atoi(e) : 0;
        }();
        if (force_bn == 128 || force_bn == 256 || (force_bn == 192 && p.b_kmajor && p.epi != EPI_ACCUM))
            BN = force_bn;
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
    a.cs = p.cs; a.ldcs = p.ldcs;
    a.err = err;
    a.splits = 1;
    a.kb_per = a.num_kb;
    // Split-K for "+=" products with fewer tiles than CTA slots (the weight
    // grads) and for long-K plain stores without bias whose tiles fill the last
    // wave of CTA pairs poorly: each K range writes fp32 partials to the
    // scratch and a second kernel adds them (to D, or into D) in range order
    // (deterministic). The range count minimises a cost model: waves x
    // (k-blocks per range + 6) x 0.25 us per 256-wide k-block, plus the
    // partials' traffic at 5 TB/s.
    const bool split_ok = p.epi == EPI_ACCUM || (p.epi == EPI_STORE && !p.bias && BN == 256);
    if (split_ok && dt != DT_F32 && p.ws && p.ws_floats > 0) {
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
    bool ok = p.a_kmajor ? make_map(&mp.a, p.A, dt, p.K, p.M, p.lda, KE, tc::BM)
                         : make_map(&mp.a, p.A, dt, p.M, p.K, p.lda, KE, KE);
    ok = ok && (p.b_kmajor ? make_map(&mp.b, p.B, dt, p.K, p.N, p.ldb, KE, BN / cg)
                           : make_map(&mp.b, p.B, dt, p.N, p.K, p.ldb, KE, KE));
    if (a.splits > 1) {
        // fp32 partials: 32-column x 32-row boxes, one per epilogue warp and chunk
        ok = ok && make_map_3d_f32(&mp.d, p.ws, p.N, p.M, a.splits, 32, 32);
        mp.d2 = mp.d;
        if (!ok) return GPT2_ERR_CUDA;
        const int rc = dt == DT_F16 ? (cg == 2 ? dispatch_epi<256, 2, 2>(EPI_SPLITK, mp, a, s)
                                               : dispatch_epi<256, 2, 1>(EPI_SPLITK, mp, a, s))
                                    : (cg == 2 ? dispatch_epi<256, 0, 2>(EPI_SPLITK, mp, a, s)
                                               : dispatch_epi<256, 0, 1>(EPI_SPLITK, mp, a, s));
        if (rc != GPT2_OK) return rc;
        return launch_splitk_reduce(dt, p.D, p.ldd, p.ws, p.M, p.N, a.splits, p.epi == EPI_ACCUM ? 1 : 0, s);
    }
    // output boxes: one 128-byte chunk x 32 rows (an epilogue warp's store)
    const int OCO = tc::ROWB / osz;
    ok = ok && make_map(&mp.d, p.D, out_dt, p.N, p.M, p.ldd, OCO, 32);
    ok = ok && make_map(&mp.d2, p.epi == EPI_GELU ? p.D2 : p.D, out_dt, p.N, p.M, p.ldd, OCO, 32);
    if (!ok) return GPT2_ERR_CUDA;
    if (dt == DT_BF16) {
        if (BN == 192)
            return cg == 2 ? dispatch_epi<192, 0, 2>(p.epi, mp, a, s) : dispatch_epi<192, 0, 1>(p.epi, mp, a, s);
        if (cg == 2)
            return BN == 256 ? dispatch_epi<256, 0, 2>(p.epi, mp, a, s) : dispatch_epi<128, 0, 2>(p.epi, mp, a, s);
        return BN == 256 ? dispatch_epi<256, 0, 1>(p.epi, mp, a, s) : dispatch_epi<128, 0, 1>(p.epi, mp, a, s);
    }
    if (dt == DT_F16) {
        if (BN == 192)
            return cg == 2 ? dispatch_epi<192, 2, 2>(p.epi, mp, a, s) : dispatch_epi<192, 2, 1>(p.epi, mp, a, s);
        if (cg == 2)
            return BN == 256 ? dispatch_epi<256, 2, 2>(p.epi, mp, a, s) : dispatch_epi<128, 2, 2>(p.epi, mp, a, s);
        return BN == 256 ? dispatch_epi<256, 2, 1>(p.epi, mp, a, s) : dispatch_epi<128, 2, 1>(p.epi, mp, a, s);
    }
    if (cg == 2)
        return BN == 256 ? dispatch_epi<256, 1, 2>(p.epi, mp, a, s) : dispatch_epi<128, 1, 2>(p.epi, mp, a, s);
    return BN == 256 ? dispatch_epi<256, 1, 1>(p.epi, mp, a, s) : dispatch_epi<128, 1, 1>(p.epi, mp, a, s);
}

// the bounded-wait limit of this translation unit's kernels (0: the default)
int set_wait_limit_gemm(unsigned long long ns) {
    return tc::set_tu_wait_limit(ns ? ns : tc::WAIT_LIMIT_NS) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gk
