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
//   warps 2..5  epilogue: tcgen05.ld the accumulator (each warp owns its
//               32-lane TMEM quarter = 32 rows, one row per thread), apply
//               bias / GELU / residual / GELU-backward / += and store.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1. Every mbarrier wait is bounded in time; on expiry the CTA records
// DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"

#include "gpt2.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

namespace gk {
namespace tc {

constexpr int BM = 128;
constexpr int ROWB = 128;  // bytes of K held per shared-memory row (one swizzle span)
constexpr int NUM_THREADS = 192;
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s per wait

template <int BN> struct Cfg {
    static constexpr int A_BYTES = BM * ROWB;
    static constexpr int B_BYTES = BN * ROWB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
};

struct Args {
    int M, N, K;
    int num_m, num_n, num_kb;
    int a_mn, b_mn;
    void* D;
    long long ldd;
    const void* bias;
    const void* aux;
    long long ldaux;
    void* D2;
    float* part;
    int part_ld;
    unsigned int* err;
};

// ------------------------------------------------------------------ PTX wrappers
DEVI uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DEVI void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
DEVI void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
DEVI void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
DEVI unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase with the given parity to complete. Returns false when
// the time limit passes (and raises the CTA's abort flag) or when another
// role has already aborted.
DEVI bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// bounded wait that ignores the abort flag (used while draining)
DEVI bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
    return true;
}

DEVI void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

DEVI void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
}
DEVI void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DEVI void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// KIND 0: kind::f16 with bf16 operands; KIND 1: kind::tf32
template <int KIND>
DEVI void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    if constexpr (KIND == 0) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
            : "memory");
    }
}

// 32 lanes x 32 consecutive fp32 columns; the wait is inside the same asm
// statement so no use of the registers can be scheduled before it.
DEVI void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
          "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]),
          "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]),
          "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), the fixed 0b001 at bits 46-48, and
// the 128-byte swizzle mode (2) at bits 61-63. Tiles are 1024-byte aligned,
// so the base-offset field stays 0.
DEVI uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: D fp32 (bits 4-5 = 1), A/B format (bits 7-9,
// 10-12: bf16 = 1 for kind::f16, tf32 = 2 for kind::tf32), A/B major
// (bits 15/16: 1 = MN-major), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int KIND>
DEVI uint32_t idesc(int a_mn, int b_mn, int M, int N) {
    uint32_t fmt = KIND == 0 ? 1u : 2u;
    uint32_t d = 0;
    d |= 1u << 4;
    d |= fmt << 7;
    d |= fmt << 10;
    d |= (uint32_t)a_mn << 15;
    d |= (uint32_t)b_mn << 16;
    d |= (uint32_t)(N >> 3) << 17;
    d |= (uint32_t)(M >> 4) << 24;
    return d;
}

// ------------------------------------------------------------------ epilogue
template <typename T, int EPI>
DEVI void epilogue_chunk(const Args& a, int row, int n0, const float (&v)[32], float& pmax,
                         float& psum) {
    constexpr int VEC = Vec16<T>::N;
    T* D = (T*)a.D + (size_t)row * a.ldd;
    const T* bias = (const T*)a.bias;
#pragma unroll
    for (int j = 0; j < 32; j += VEC) {
        const int n = n0 + j;
        if (n >= a.N) break;
        float x[VEC];
#pragma unroll
        for (int k = 0; k < VEC; k++) x[k] = v[j + k];
        if constexpr (EPI == EPI_STORE || EPI == EPI_GELU || EPI == EPI_RESID ||
                      EPI == EPI_GELU_PART) {
            if (bias) {
                Vec16<T> b = ld16(bias + n);
#pragma unroll
                for (int k = 0; k < VEC; k++) x[k] += to_f(b.v[k]);
            }
        }
        Vec16<T> o;
        if constexpr (EPI == EPI_STORE) {
#pragma unroll
            for (int k = 0; k < VEC; k++) o.v[k] = from_f<T>(x[k]);
            st16(D + n, o);
        } else if constexpr (EPI == EPI_GELU) {
            Vec16<T> g;
#pragma unroll
            for (int k = 0; k < VEC; k++) {
                o.v[k] = from_f<T>(x[k]);
                g.v[k] = from_f<T>(gelu_fwd(to_f(o.v[k])));
            }
            st16(D + n, o);
            st16((T*)a.D2 + (size_t)row * a.ldd + n, g);
        } else if constexpr (EPI == EPI_RESID) {
            Vec16<T> r = ld16((const T*)a.aux + (size_t)row * a.ldaux + n);
#pragma unroll
            for (int k = 0; k < VEC; k++) o.v[k] = from_f<T>(x[k] + to_f(r.v[k]));
            st16(D + n, o);
        } else if constexpr (EPI == EPI_GELU_BWD) {
            Vec16<T> r = ld16((const T*)a.aux + (size_t)row * a.ldaux + n);
#pragma unroll
            for (int k = 0; k < VEC; k++) o.v[k] = from_f<T>(x[k] * gelu_grad(to_f(r.v[k])));
            st16(D + n, o);
        } else if constexpr (EPI == EPI_ACCUM) {
            Vec16<T> r = ld16(D + n);
#pragma unroll
            for (int k = 0; k < VEC; k++) o.v[k] = from_f<T>(to_f(r.v[k]) + x[k]);
            st16(D + n, o);
        } else if constexpr (EPI == EPI_GELU_PART) {
            float cm = pmax;
#pragma unroll
            for (int k = 0; k < VEC; k++) {
                x[k] = gelu_fwd(x[k]);
                cm = fmaxf(cm, x[k]);
            }
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < VEC; k++) {
                o.v[k] = from_f<T>(x[k]);
                s += expf(x[k] - cm);
            }
            psum = psum * expf(pmax - cm) + s;
            pmax = cm;
            st16(D + n, o);
        }
    }
}

// ------------------------------------------------------------------ kernel
template <int BN, int KIND, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_k(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ Args args) {
    using C = Cfg<BN>;
    using T = typename std::conditional<KIND == 0, bf16, float>::type;
    constexpr int KE = ROWB / (int)sizeof(T);  // K elements per stage
    constexpr int UK = KIND == 0 ? 16 : 8;     // K elements per MMA
    constexpr int KSTEPS = KE / UK;            // MMAs per stage (4)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + C::STAGES * C::STAGE_BYTES;
    uint8_t* bars_ptr = base_ptr + C::STAGES * C::STAGE_BYTES;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
    auto tfull = [&](int a) { return bars + 8u * (2 * C::STAGES + a); };
    auto tempty = [&](int a) { return bars + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t drain = bars + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + 8 * (2 * C::STAGES + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars_ptr + 8 * (2 * C::STAGES + 5) + 4);
    int* n_issued_smem = reinterpret_cast<int*>(bars_ptr + 8 * (2 * C::STAGES + 6));

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *n_issued_smem = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = args.num_m * args.num_n;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0, n_issued = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile % args.num_m) * BM, n0 = (tile / args.num_m) * BN;
                bool ok = true;
                for (int kb = 0; kb < args.num_kb; kb++) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t sa = base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    mbar_expect_tx(full(stage), C::STAGE_BYTES);
                    const int k0 = kb * KE;
                    if (!args.a_mn) {
                        tma_load_2d(sa, &tmA, full(stage), k0, m0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / KE; j++)
                            tma_load_2d(sa + j * KE * ROWB, &tmA, full(stage), m0 + j * KE, k0);
                    }
                    if (!args.b_mn) {
                        tma_load_2d(sb, &tmB, full(stage), k0, n0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / KE; j++)
                            tma_load_2d(sb + j * KE * ROWB, &tmB, full(stage), n0 + j * KE, k0);
                    }
                    ++n_issued;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            *n_issued_smem = n_issued;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t id = idesc<KIND>(args.a_mn, args.b_mn, BM, BN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < args.num_kb; kb++) {
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
                        umma<KIND>(d, da, db, id, (kb | k) ? 1u : 0u);
                    }
                    umma_commit(empty(stage));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(tfull(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue warps 2..5
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int mb = tile % args.num_m, nb = tile / args.num_m;
            const int m0 = mb * BM, n0 = nb * BN;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(tfull(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            float pmax = -INFINITY, psum = 0.f;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                float v[32];
                tmem_ld32(tmem_base + (uint32_t)(acc * BN + c) + ((uint32_t)(q * 32) << 16), v);
                if (row < args.M && n0 + c < args.N)
                    epilogue_chunk<T, EPI>(args, row, n0 + c, v, pmax, psum);
            }
            if constexpr (EPI == EPI_GELU_PART) {
                if (row < args.M)
                    reinterpret_cast<float2*>(args.part)[(size_t)row * args.part_ld + nb] =
                        make_float2(pmax, psum);
            }
            tc_fence_before();
            mbar_arrive(tempty(acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // drain: wait for every TMA copy this CTA issued, and for all MMAs issued so far
        if (threadIdx.x == 0) {
            const int n_issued = *n_issued_smem;
            for (int s = 0; s < C::STAGES; s++) {
                if (n_issued > s) {
                    const int last = s + ((n_issued - 1 - s) / C::STAGES) * C::STAGES;
                    mbar_wait_drain(full(s), (uint32_t)((last / C::STAGES) & 1));
                }
            }
            atomicOr(args.err, DEVERR_TIMEOUT);
        }
        if (threadIdx.x == 32) {
            umma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
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

template <int BN, int KIND, int EPI>
static int launch_tc(const CUtensorMap& ta, const CUtensorMap& tb, const tc::Args& a, int grid,
                     cudaStream_t s) {
    using C = tc::Cfg<BN>;
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(tc::gemm_tc_k<BN, KIND, EPI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess)
            return GPT2_ERR_CUDA;
        attr_done = true;
    }
    note_launch(1);
    tc::gemm_tc_k<BN, KIND, EPI><<<grid, tc::NUM_THREADS, C::SMEM_BYTES, s>>>(ta, tb, a);
    return GPT2_OK;
}

template <int BN, int KIND>
static int dispatch_epi(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const tc::Args& a,
                        int grid, cudaStream_t s) {
    if constexpr (KIND == 0) {
        switch (epi) {
            case EPI_STORE: return launch_tc<BN, KIND, EPI_STORE>(ta, tb, a, grid, s);
            case EPI_GELU: return launch_tc<BN, KIND, EPI_GELU>(ta, tb, a, grid, s);
            case EPI_RESID: return launch_tc<BN, KIND, EPI_RESID>(ta, tb, a, grid, s);
            case EPI_GELU_BWD: return launch_tc<BN, KIND, EPI_GELU_BWD>(ta, tb, a, grid, s);
            case EPI_ACCUM: return launch_tc<BN, KIND, EPI_ACCUM>(ta, tb, a, grid, s);
            default: return GPT2_ERR_CONFIG;
        }
    } else {
        switch (epi) {
            case EPI_STORE: return launch_tc<BN, KIND, EPI_STORE>(ta, tb, a, grid, s);
            case EPI_GELU_PART: return launch_tc<BN, KIND, EPI_GELU_PART>(ta, tb, a, grid, s);
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
    if ((p.epi == EPI_RESID || p.epi == EPI_GELU_BWD) && (!al16(p.aux) || (p.ldaux * esz) % 16))
        return GPT2_ERR_ALIGN;
    if (p.bias && !al16(p.bias)) return GPT2_ERR_ALIGN;
    if (p.epi == EPI_GELU && !al16(p.D2)) return GPT2_ERR_ALIGN;

    const int sms = num_sms();
    // tile width: fewer waves x narrower tiles wins; EPI_GELU_PART fixes 256
    int BN = 256;
    if (p.epi != EPI_GELU_PART) {
        const long long nm = (p.M + tc::BM - 1) / tc::BM;
        const long long t256 = nm * ((p.N + 255) / 256), t128 = nm * ((p.N + 127) / 128);
        const long long c256 = ((t256 + sms - 1) / sms) * 256, c128 = ((t128 + sms - 1) / sms) * 128;
        if (c128 < c256) BN = 128;
    }
    tc::Args a;
    a.M = p.M; a.N = p.N; a.K = p.K;
    a.num_m = (p.M + tc::BM - 1) / tc::BM;
    a.num_n = (p.N + BN - 1) / BN;
    a.num_kb = (p.K + KE - 1) / KE;
    a.a_mn = p.a_kmajor ? 0 : 1;
    a.b_mn = p.b_kmajor ? 0 : 1;
    a.D = p.D; a.ldd = p.ldd; a.bias = p.bias; a.aux = p.aux; a.ldaux = p.ldaux; a.D2 = p.D2;
    a.part = p.part; a.part_ld = p.part_ld; a.err = err;

    CUtensorMap ta, tb;
    bool ok = p.a_kmajor ? make_map(&ta, p.A, dt, p.K, p.M, p.lda, KE, tc::BM)
                         : make_map(&ta, p.A, dt, p.M, p.K, p.lda, KE, KE);
    ok = ok && (p.b_kmajor ? make_map(&tb, p.B, dt, p.K, p.N, p.ldb, KE, BN)
                           : make_map(&tb, p.B, dt, p.N, p.K, p.ldb, KE, KE));
    if (!ok) return GPT2_ERR_CUDA;
    const long long tiles = (long long)a.num_m * a.num_n;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (dt == DT_BF16)
        return BN == 256 ? dispatch_epi<256, 0>(p.epi, ta, tb, a, grid, s)
                         : dispatch_epi<128, 0>(p.epi, ta, tb, a, grid, s);
    return BN == 256 ? dispatch_epi<256, 1>(p.epi, ta, tb, a, grid, s)
                     : dispatch_epi<128, 1>(p.epi, ta, tb, a, grid, s);
}

}  // namespace gk
