// kernels.cu -- memory-bound kernels of the GPT-2 training step (sm_103a).
//
// Each kernel streams its tensors with 16-byte vector accesses, keeps
// reductions deterministic (fixed-order two-stage sums instead of float
// atomics), and sizes its grid from the SM count.
//
// Page references are to llm.c "train_gpt2.cu" (the mixed-precision CUDA
// training step) unless stated otherwise.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include "gpt2.h"

#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <type_traits>

namespace gk {

bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("GPT2_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

namespace {
thread_local int t_launch_priority = 0;
}
int launch_priority() { return t_launch_priority; }
void set_launch_priority(int priority) { t_launch_priority = priority; }

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

static std::atomic<long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

// runs the statement with E = the element type of dt (bf16, fp16 or fp32)
#define DISPATCH_E(dt, ...)                \
    do {                                   \
        if ((dt) == DT_BF16) {             \
            using E = bf16;                \
            __VA_ARGS__;                   \
        } else if ((dt) == DT_F16) {       \
            using E = f16;                 \
            __VA_ARGS__;                   \
        } else {                           \
            using E = float;               \
            __VA_ARGS__;                   \
        }                                  \
    } while (0)

static inline unsigned int grid_for(size_t work, int block, int per_sm = 8) {
    size_t g = (work + block - 1) / block;
    size_t cap = (size_t)num_sms() * per_sm;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (unsigned int)g;
}

// ------------------------------------------------------------------ tokens
// Copies device token ids into the model's buffer; ids outside [0, V) are
// replaced by 0 (so no later gather leaves its table) and flagged.
__global__ void copy_tokens_k(const int* __restrict__ src, int* __restrict__ dst, int n, int V,
                              unsigned int* err) {
    pdl_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        int t = src[i];
        if (t < 0 || t >= V) {
            atomicOr(err, DEVERR_TOKEN);
            t = 0;
        }
        dst[i] = t;
    }
}

void launch_copy_tokens(const int* src, int* dst, int n, int V, unsigned int* err, cudaStream_t s) {
    note_launch(1);
    launch_pdl(copy_tokens_k, grid_for(n, 256), 256, 0, s, src, dst, n, V, err);
}

// ------------------------------------------------------------------ encoder
// encoder_forward_kernel2/3: out[b,t,:] = wte[tok[b,t],:] + wpe[t,:]
template <typename T>
__global__ void encoder_forward_k(T* __restrict__ out, const int* __restrict__ tok,
                                  const T* __restrict__ wte, const T* __restrict__ wpe, int BT,
                                  int Tn, int C) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    const int cv = C / VEC;
    const size_t nvec = (size_t)BT * cv;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
         i += (size_t)gridDim.x * blockDim.x) {
        int bt = (int)(i / cv);
        int c = (int)(i % cv) * VEC;
        int t = bt % Tn;
        Vec16<T> a = ld16(wte + (size_t)tok[bt] * C + c);
        Vec16<T> p = ld16(wpe + (size_t)t * C + c);
        Vec16<T> o;
#pragma unroll
        for (int k = 0; k < VEC; k++) o.v[k] = from_f<T>(to_f(a.v[k]) + to_f(p.v[k]));
        st16(out + (size_t)bt * C + c, o);
    }
}

void launch_encoder_forward(DType dt, void* out, const int* tok, const void* wte, const void* wpe,
                            int B, int T, int C, cudaStream_t s) {
    note_launch(1);
    size_t work = (size_t)B * T * C / dtype_vec(dt);
    unsigned g = grid_for(work, 256);
    DISPATCH_E(dt, launch_pdl(encoder_forward_k<E>, g, 256, 0, s, (E*)out, tok, (const E*)wte,
                              (const E*)wpe, B * T, T, C));
}

// encoder_backward_kernel, made deterministic.
// dwpe[t,:] += sum over b of dout[b,t,:] (fixed b order).
template <typename T>
__global__ void encoder_backward_wpe_k(T* __restrict__ dwpe, const T* __restrict__ dout, int B,
                                       int Tn, int C) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    const int cv = C / VEC;
    const int nvec = Tn * cv;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += gridDim.x * blockDim.x) {
        int t = i / cv, c = (i % cv) * VEC;
        float acc[VEC];
#pragma unroll
        for (int k = 0; k < VEC; k++) acc[k] = 0.f;
        for (int b = 0; b < B; b++) {
            Vec16<T> d = ld16(dout + ((size_t)b * Tn + t) * C + c);
#pragma unroll
            for (int k = 0; k < VEC; k++) acc[k] += to_f(d.v[k]);
        }
        T* dst = dwpe + (size_t)t * C + c;
        Vec16<T> w = ld16(dst);
#pragma unroll
        for (int k = 0; k < VEC; k++) w.v[k] = from_f<T>(to_f(w.v[k]) + acc[k]);
        st16(dst, w);
    }
}

// token histogram (integer atomics: the counts are exact whatever the order)
__global__ void token_count_k(const int* __restrict__ tok, int n, int* counts) {
    pdl_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        atomicAdd(&counts[tok[i]], 1);
}

// single-block exclusive scan: offsets[v] = sum_{u<v} counts[u], offsets[Vp] = total;
// cursor[v] = offsets[v]
__global__ void __launch_bounds__(1024) token_scan_k(const int* __restrict__ counts, int Vp,
                                                     int* __restrict__ offsets,
                                                     int* __restrict__ cursor) {
    pdl_enter();
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (Vp + nt - 1) / nt;
    const int lo = min(Vp, tid * per), hi = min(Vp, lo + per);
    int local = 0;
    for (int v = lo; v < hi; v++) local += counts[v];
    // inclusive scan of `local` across the block
    int lane = tid & 31, warp = tid >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < nt / 32) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    int base = (warp > 0 ? warp_tot[warp - 1] : 0) + x - local;  // exclusive prefix of this thread
    for (int v = lo; v < hi; v++) {
        offsets[v] = base;
        cursor[v] = base;
        base += counts[v];
    }
    if (tid == nt - 1) offsets[Vp] = base;
}

// the same scan with the counts staged in shared memory: the global reads and
// writes are coalesced, and each thread scans a contiguous run from shared memory
// (Vp ints of dynamic shared memory)
__global__ void __launch_bounds__(1024) token_scan_smem_k(const int* __restrict__ counts, int Vp,
                                                          int* __restrict__ offsets,
                                                          int* __restrict__ cursor) {
    pdl_enter();
    extern __shared__ int tsm[];
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    // eight loads in flight per thread
    int v0 = tid;
    for (; v0 + 7 * nt < Vp; v0 += 8 * nt) {
        int c[8];
#pragma unroll
        for (int u = 0; u < 8; u++) c[u] = counts[v0 + u * nt];
#pragma unroll
        for (int u = 0; u < 8; u++) tsm[v0 + u * nt] = c[u];
    }
    for (; v0 < Vp; v0 += nt) tsm[v0] = counts[v0];
    __syncthreads();
    const int per = (Vp + nt - 1) / nt;
    const int lo = min(Vp, tid * per), hi = min(Vp, lo + per);
    int local = 0;
    for (int v = lo; v < hi; v++) local += tsm[v];
    const int lane = tid & 31, warp = tid >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < nt / 32) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    int base = (warp > 0 ? warp_tot[warp - 1] : 0) + x - local;
    for (int v = lo; v < hi; v++) {
        const int c = tsm[v];
        tsm[v] = base;
        base += c;
    }
    if (tid == nt - 1) offsets[Vp] = base;
    __syncthreads();
    for (int v = tid; v < Vp; v += nt) {
        const int o = tsm[v];
        offsets[v] = o;
        cursor[v] = o;
    }
}

__global__ void token_scatter_k(const int* __restrict__ tok, int n, int* cursor,
                                int* __restrict__ order) {
    pdl_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        int slot = atomicAdd(&cursor[tok[i]], 1);
        order[slot] = i;
    }
}

// place each position at its rank (ascending position) inside its token's bucket
__global__ void token_rank_k(const int* __restrict__ tok, const int* __restrict__ offsets,
                             const int* __restrict__ order, int n, int* __restrict__ sorted) {
    pdl_enter();
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < n; s += gridDim.x * blockDim.x) {
        int pos = order[s];
        int v = tok[pos];
        int lo = offsets[v], hi = offsets[v + 1];
        int rank = 0;
        for (int j = lo; j < hi; j++) rank += (order[j] < pos);
        sorted[lo + rank] = pos;
    }
}

// one warp per vocabulary row: dwte[v,:] += sum of dout rows of its positions, ascending
template <typename T>
__global__ void encoder_backward_wte_k(T* __restrict__ dwte, const T* __restrict__ dout,
                                       const int* __restrict__ offsets,
                                       const int* __restrict__ sorted, int Vp, int C) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    constexpr int CH = 4;  // vectors per lane per pass
    const int warps = blockDim.x / 32;
    const int v = blockIdx.x * warps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (v >= Vp) return;
    const int lo = offsets[v], hi = offsets[v + 1];
    if (lo == hi) return;
    const int cv = C / VEC;
    for (int c0 = 0; c0 < cv; c0 += 32 * CH) {
        float acc[CH][VEC];
#pragma unroll
        for (int j = 0; j < CH; j++)
#pragma unroll
            for (int k = 0; k < VEC; k++) acc[j][k] = 0.f;
        for (int s = lo; s < hi; s++) {
            const T* row = dout + (size_t)sorted[s] * C;
#pragma unroll
            for (int j = 0; j < CH; j++) {
                int vi = c0 + lane + 32 * j;
                if (vi < cv) {
                    Vec16<T> d = ld16(row + vi * VEC);
#pragma unroll
                    for (int k = 0; k < VEC; k++) acc[j][k] += to_f(d.v[k]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < CH; j++) {
            int vi = c0 + lane + 32 * j;
            if (vi < cv) {
                T* dst = dwte + (size_t)v * C + vi * VEC;
                Vec16<T> w = ld16(dst);
#pragma unroll
                for (int k = 0; k < VEC; k++) w.v[k] = from_f<T>(to_f(w.v[k]) + acc[j][k]);
                st16(dst, w);
            }
        }
    }
}

void launch_zero(void* p, size_t bytes, cudaStream_t s);

void launch_encoder_backward(DType dt, void* dwte, void* dwpe, const void* dout, const int* tok,
                             int B, int T, int C, int Vp, int* ws_counts, int* ws_offsets,
                             int* ws_cursor, int* ws_order, int* ws_sorted, cudaStream_t s) {
    note_launch(6);
    const int n = B * T;
    const int VEC = dtype_vec(dt);
    unsigned g = grid_for((size_t)T * C / VEC, 256);
    DISPATCH_E(dt, launch_pdl(encoder_backward_wpe_k<E>, g, 256, 0, s, (E*)dwpe, (const E*)dout, B, T, C));
    launch_zero(ws_counts, sizeof(int) * (size_t)Vp, s);
    launch_pdl(token_count_k, grid_for(n, 256), 256, 0, s, tok, n, ws_counts);
    const size_t scan_smem = sizeof(int) * (size_t)Vp;
    if (scan_smem <= 200 * 1024) {
        static size_t done = 0;
        if (scan_smem > done) {
            cudaFuncSetAttribute(token_scan_smem_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem);
            done = scan_smem;
        }
        launch_pdl(token_scan_smem_k, 1, 1024, scan_smem, s, ws_counts, Vp, ws_offsets, ws_cursor);
    } else {
        launch_pdl(token_scan_k, 1, 1024, 0, s, ws_counts, Vp, ws_offsets, ws_cursor);
    }
    launch_pdl(token_scatter_k, grid_for(n, 256), 256, 0, s, tok, n, ws_cursor, ws_order);
    launch_pdl(token_rank_k, grid_for(n, 256), 256, 0, s, tok, ws_offsets, ws_order, n, ws_sorted);
    unsigned gw = (unsigned)((Vp + 7) / 8);
    DISPATCH_E(dt, launch_pdl(encoder_backward_wte_k<E>, gw, 256, 0, s, (E*)dwte, (const E*)dout, ws_offsets,
                              ws_sorted, Vp, C));
}

// ------------------------------------------------------------------ LayerNorm
using tc::fadd2;
using tc::ffma2;
using tc::fmul2;
// two bf16 (one 32-bit word, low half first) widened to fp32, and back (rounded)
DEVI float2 bf2_f2(uint32_t u) { return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)); }
// the same widening, opaque to the compiler: recomputed at every use rather
// than kept live in registers between a kernel's passes over a row
DEVI float2 bf2_f2_v(uint32_t u) {
    uint32_t lo, hi;
    asm volatile("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;" : "=r"(lo), "=r"(hi) : "r"(u));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
DEVI uint32_t f2_bf2(float2 v) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t*>(&b);
}
// the same for either 16-bit type (fp16 widens with two conversions)
template <typename H> DEVI float2 h2_f2_v(uint32_t u);
template <> DEVI float2 h2_f2_v<bf16>(uint32_t u) { return bf2_f2_v(u); }
template <> DEVI float2 h2_f2_v<f16>(uint32_t u) {
    float lo, hi;
    asm volatile("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                 : "=f"(lo), "=f"(hi)
                 : "r"(u));
    return make_float2(lo, hi);
}
template <typename H> DEVI uint32_t f2_h2v(float2 v) { return f2_h2<H>(v.x, v.y); }
// plain widening (the compiler may keep the result live)
template <typename H> DEVI float2 h2_f2w(uint32_t u);
template <> DEVI float2 h2_f2w<bf16>(uint32_t u) { return bf2_f2(u); }
template <> DEVI float2 h2_f2w<f16>(uint32_t u) { return h2_f2<f16>(u); }
// layernorm_forward_kernel3: one warp per row, the row held in registers;
// mean, biased variance, rstd = 1/sqrt(var + 1e-5), y = (x - mean) rstd w + b.
// mean/rstd are kept in fp32.
template <typename T, int MAXV>
__global__ void layernorm_forward_k(T* __restrict__ out, float* __restrict__ mean,
                                    float* __restrict__ rstd, const T* __restrict__ inp,
                                    const T* __restrict__ w, const T* __restrict__ b, int N,
                                    int C) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    const int warps = blockDim.x / 32;
    const int row = blockIdx.x * warps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const int cv = C / VEC;
    const T* x = inp + (size_t)row * C;
    float xs[MAXV][VEC];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; j++) {
        int vi = lane + 32 * j;
        if (vi < cv) {
            Vec16<T> a = ld16(x + vi * VEC);
#pragma unroll
            for (int k = 0; k < VEC; k++) {
                xs[j][k] = to_f(a.v[k]);
                s += xs[j][k];
            }
        }
    }
    const float m = warp_sum(s) / C;
    float var = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; j++) {
        int vi = lane + 32 * j;
        if (vi < cv) {
#pragma unroll
            for (int k = 0; k < VEC; k++) {
                float d = xs[j][k] - m;
                var += d * d;
            }
        }
    }
    var = warp_sum(var) / C;
    const float r = rsqrtf(var + 1e-5f);
    T* y = out + (size_t)row * C;
#pragma unroll
    for (int j = 0; j < MAXV; j++) {
        int vi = lane + 32 * j;
        if (vi < cv) {
            Vec16<T> wv = ld16(w + vi * VEC), bv = ld16(b + vi * VEC), o;
#pragma unroll
            for (int k = 0; k < VEC; k++)
                o.v[k] = from_f<T>((xs[j][k] - m) * r * to_f(wv.v[k]) + to_f(bv.v[k]));
            st16(y + vi * VEC, o);
        }
    }
    if (lane == 0) {
        mean[row] = m;
        rstd[row] = r;
    }
}

// 16-bit rows (bf16 or fp16, H) with C = 256 NV (NV <= 4): lane l keeps the
// row's 16-byte vectors l, l + 32, ... as packed 16-bit words (4 NV registers)
// and widens them anew in each pass, so the kernel fits in 40 registers and 48
// one-row warps are resident per SM; the statistics and the affine map use
// packed fp32 arithmetic.
template <typename H, int NV, int RW>
__global__ void __launch_bounds__(256, RW == 1 ? (NV <= 3 ? 6 : 4) : (NV <= 3 ? 4 : 3)) layernorm_forward_bf16_k(H* __restrict__ out, float* __restrict__ mean,
                                                                   float* __restrict__ rstd,
                                                                   const H* __restrict__ inp,
                                                                   const H* __restrict__ w,
                                                                   const H* __restrict__ b, int N) {
    constexpr int C = 256 * NV;
    pdl_enter();
    // RW rows per warp, rows row0, row0 + 8, ... of the block's 8 RW rows: all
    // of the warp's loads are issued before the first row's arithmetic
    const int row0 = blockIdx.x * 8 * RW + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row0 >= N) return;
    uint4 xv[RW][NV];
#pragma unroll
    for (int q = 0; q < RW; q++) {
        const int row = row0 + 8 * q;
        const uint4* x = reinterpret_cast<const uint4*>(inp + (size_t)row * C) + lane;
#pragma unroll
        for (int j = 0; j < NV; j++) xv[q][j] = row < N ? x[32 * j] : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint4* wp = reinterpret_cast<const uint4*>(w) + lane;
    const uint4* bp = reinterpret_cast<const uint4*>(b) + lane;
#pragma unroll
    for (int q = 0; q < RW; q++) {
        const int row = row0 + 8 * q;
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NV; j++) {
            s2 = fadd2(s2, fadd2(h2_f2_v<H>(xv[q][j].x), h2_f2_v<H>(xv[q][j].y)));
            s2 = fadd2(s2, fadd2(h2_f2_v<H>(xv[q][j].z), h2_f2_v<H>(xv[q][j].w)));
        }
        const float m = warp_sum(s2.x + s2.y) / C;
        const float2 nm = make_float2(-m, -m);
        float2 v2 = make_float2(0.f, 0.f);
        auto sq = [&](uint32_t u) {
            const float2 d = fadd2(h2_f2_v<H>(u), nm);
            v2 = ffma2(d, d, v2);
        };
#pragma unroll
        for (int j = 0; j < NV; j++) {
            sq(xv[q][j].x); sq(xv[q][j].y); sq(xv[q][j].z); sq(xv[q][j].w);
        }
        const float var = warp_sum(v2.x + v2.y) / C;
        const float r = rsqrtf(var + 1e-5f);
        if (row >= N) break;
        // y = (x r - m r) w + b
        const float2 r2 = make_float2(r, r), nmr = make_float2(-m * r, -m * r);
        uint4* y = reinterpret_cast<uint4*>(out + (size_t)row * C) + lane;
        auto aff = [&](uint32_t xu, uint32_t wu, uint32_t bu) {
            return f2_h2v<H>(ffma2(ffma2(h2_f2_v<H>(xu), r2, nmr), h2_f2_v<H>(wu), h2_f2_v<H>(bu)));
        };
#pragma unroll
        for (int j = 0; j < NV; j++) {
            const uint4 wu = __ldg(wp + 32 * j), bu = __ldg(bp + 32 * j);
            y[32 * j] = make_uint4(aff(xv[q][j].x, wu.x, bu.x), aff(xv[q][j].y, wu.y, bu.y),
                                   aff(xv[q][j].z, wu.z, bu.z), aff(xv[q][j].w, wu.w, bu.w));
        }
        if (lane == 0) {
            mean[row] = m;
            rstd[row] = r;
        }
    }
}

static int maxv_for(int cv) {
    int per = (cv + 31) / 32;
    return per <= 1 ? 1 : per <= 2 ? 2 : per <= 4 ? 4 : 8;
}

void launch_layernorm_forward(DType dt, void* out, float* mean, float* rstd, const void* inp,
                              const void* w, const void* b, int N, int C, cudaStream_t s) {
    note_launch(1);
    const int VEC = dtype_vec(dt);
    const int mv = maxv_for(C / VEC);
    const int block = 256, rows = block / 32;
    unsigned g = (unsigned)((N + rows - 1) / rows);
    if (dt != DT_F32 && C % 256 == 0 && C <= 1024) {
        const int nv = C / 256;
        // two rows per warp while the rows still fill a wave of resident warps
        // at two per warp, else one
        static const int rw_env = [] {
            const char* e = getenv("GPT2_LN_ROWS");
            return e ? atoi(e) : 0;
        }();
        const int rw = rw_env == 1 || rw_env == 2 ? rw_env : 2;
        const unsigned g2 = (unsigned)((N + rows * rw - 1) / (rows * rw));
#define LNF2(H, NVV)                                                                                       \
    do {                                                                                                   \
        if (rw == 2)                                                                                       \
            launch_pdl(layernorm_forward_bf16_k<H, NVV, 2>, g2, block, 0, s, (H*)out, mean, rstd,           \
                       (const H*)inp, (const H*)w, (const H*)b, N);                                        \
        else                                                                                               \
            launch_pdl(layernorm_forward_bf16_k<H, NVV, 1>, g2, block, 0, s, (H*)out, mean, rstd,           \
                       (const H*)inp, (const H*)w, (const H*)b, N);                                        \
    } while (0)
        if (dt == DT_BF16) {
            if (nv == 1) LNF2(bf16, 1); else if (nv == 2) LNF2(bf16, 2); else if (nv == 3) LNF2(bf16, 3);
            else LNF2(bf16, 4);
        } else {
            if (nv == 1) LNF2(f16, 1); else if (nv == 2) LNF2(f16, 2); else if (nv == 3) LNF2(f16, 3);
            else LNF2(f16, 4);
        }
#undef LNF2
        return;
    }
#define LNF(TT, MV)                                                                            \
    launch_pdl(layernorm_forward_k<TT, MV>, g, block, 0, s, (TT*)out, mean, rstd, (const TT*)inp,        \
                                                    (const TT*)w, (const TT*)b, N, C)
    DISPATCH_E(dt, if (mv == 1) LNF(E, 1); else if (mv == 2) LNF(E, 2); else if (mv == 4) LNF(E, 4);
                   else LNF(E, 8));
#undef LNF
}

// layernorm_backward_kernel6, deterministic and with += for every output:
//   nhat = (x - mean) rstd, g = w * dy,
//   dx (+)= rstd (g - mean_c(g) - nhat mean_c(g nhat)),
//   dw += sum_rows nhat dy, db += sum_rows dy.
// Stage 1: one warp per row (a row lives in registers, NV 16-byte vectors per
// lane); per-column partial sums stay in registers across the warp's rows,
// the block folds its warps in a fixed order and writes one partial row to ws.
// Stage 2 (reduce_partials_k) sums the partial rows in block order.
constexpr int LNB_BLOCK = 256;

template <typename T, int NV>
__global__ void __launch_bounds__(LNB_BLOCK) layernorm_backward_k(
    T* __restrict__ dinp, float* __restrict__ ws, const T* __restrict__ dout,
    const T* __restrict__ inp, const T* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int accumulate) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    // per-warp partial sums, [warp][dw | db][k][vector]: lane-consecutive addresses
    extern __shared__ float sm[];
    const int warps = blockDim.x / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int cv = C / VEC;
    float* mine = sm + (size_t)warp * 2 * C;
    for (int c = lane; c < 2 * C; c += 32) mine[c] = 0.f;
    __syncwarp();
    for (int row = blockIdx.x * warps + warp; row < N; row += gridDim.x * warps) {
        const T* x = inp + (size_t)row * C;
        const T* dy = dout + (size_t)row * C;
        const float mu = mean[row], rs = rstd[row];
        // pass 1: the two row reductions (the row stays in L1 for pass 2)
        float gsum = 0.f, gnsum = 0.f;
#pragma unroll
        for (int j = 0; j < NV; j++) {
            const int vi = lane + 32 * j;
            if (vi < cv) {
                Vec16<T> xv = ld16(x + vi * VEC), dv = ld16(dy + vi * VEC), wv = ld16(w + vi * VEC);
#pragma unroll
                for (int k = 0; k < VEC; k++) {
                    const float g = to_f(wv.v[k]) * to_f(dv.v[k]);
                    gsum += g;
                    gnsum += g * (to_f(xv.v[k]) - mu) * rs;
                }
            }
        }
        gsum = warp_sum(gsum) / C;
        gnsum = warp_sum(gnsum) / C;
        // pass 2: outputs and the parameter partials
        T* dx = dinp + (size_t)row * C;
#pragma unroll
        for (int j = 0; j < NV; j++) {
            const int vi = lane + 32 * j;
            if (vi < cv) {
                Vec16<T> xv = ld16_cs(x + vi * VEC), dv = ld16_cs(dy + vi * VEC), wv = ld16(w + vi * VEC);
                Vec16<T> o;
                if (accumulate) o = ld16(dx + vi * VEC);
#pragma unroll
                for (int k = 0; k < VEC; k++) {
                    const float d = to_f(dv.v[k]);
                    const float nh = (to_f(xv.v[k]) - mu) * rs;
                    const float g = to_f(wv.v[k]) * d;
                    const float val = rs * (g - gsum - nh * gnsum);
                    o.v[k] = from_f<T>(accumulate ? to_f(o.v[k]) + val : val);
                    mine[k * cv + vi] += nh * d;
                    mine[C + k * cv + vi] += d;
                }
                st16(dx + vi * VEC, o);
            }
        }
    }
    __syncthreads();
    // fold the warps' slices in warp order and write this block's partial row
    // in column order (column vi*VEC + k)
    float* dst = ws + (size_t)blockIdx.x * 2 * C;
    for (int c = threadIdx.x; c < 2 * C; c += blockDim.x) {
        const int half = c >= C, cc = c - half * C;
        const int vi = cc / VEC, k = cc % VEC;
        float t = 0.f;
        for (int wi = 0; wi < warps; wi++) t += sm[(size_t)wi * 2 * C + half * C + k * cv + vi];
        dst[c] = t;
    }
}

// The same operation (bf16, C <= 768) as a persistent kernel fed by bulk
// copies: one producer thread streams each of the CTA's rows (x, dy and, for
// +=, the current dx) from HBM into a ring of LNQ_RING shared-memory slots with
// cp.async.bulk, so up to LNQ_RING rows per SM are in flight. A row is taken
// by a group of NV warps, each lane holding one 16-byte vector (8 columns) of
// it; the groups take the slots in turn, combine the two row sums through
// shared memory under a named barrier, write dx, and keep the dw / db partials
// (and, with `with_colsum`, the column sums of the written dx: the bias
// gradient of the matmul that produced this residual-stream gradient) in
// registers. The CTA folds its warps in order into one partial row
// [dw | db | colsum] of G*C floats at part[blockIdx.x].
constexpr int LNQ_RING = 10;  // ring slots
constexpr int LNQ_SR = 4;     // consecutive rows per slot (one bulk copy per array)
constexpr int LNQ_THREADS = 512;  // 15 consumer warps + the producer warp
constexpr int LNQ_XCH = 16 * 2 * 4;  // exchange entries: groups x parity x warps in a group

// bytes of the ring or of the fold [groups][3][C] fp32, whichever is larger
__host__ __device__ inline size_t lnq_body_bytes(int C, int groups) {
    const size_t ring = (size_t)LNQ_RING * LNQ_SR * 3 * C * 2, fold = (size_t)groups * 3 * C * 4;
    return ((ring > fold ? ring : fold) + 15) / 16 * 16;
}

template <typename H, int NV>
__global__ void __launch_bounds__(LNQ_THREADS, 1) layernorm_backward_bulk_k(
    H* __restrict__ dinp, float* __restrict__ part, const H* __restrict__ dout,
    const H* __restrict__ inp, const H* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int accumulate, int with_colsum,
    unsigned int* __restrict__ err) {
    constexpr int VEC = 8;
    constexpr int GROUPS = (LNQ_THREADS / 32 - 1) / NV;  // row groups of NV warps
    constexpr int CWARPS = GROUPS * NV;                    // consumer warps
    static_assert(GROUPS <= 15 && NV <= 4, "named barriers and the exchange area");
    extern __shared__ __align__(128) uint8_t lnq_sm[];
    const int rowb = C * 2, arrb = LNQ_SR * rowb, slotb = 3 * arrb;  // a slot: [x | dy | dx] x SR rows
    uint8_t* ring = lnq_sm;
    const uint32_t ring_s = tc::smem_u32(ring);
    // the ring, later reused by the fold of the groups' partial sums
    uint8_t* tail = lnq_sm + lnq_body_bytes(C, GROUPS);
    const uint32_t bars = tc::smem_u32(tail);
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (LNQ_RING + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 16 * LNQ_RING);
    int* issued_s = reinterpret_cast<int*>(tail + 16 * LNQ_RING + 4);
    // [group][row-pair parity][warp in group]: the two rows' (sum of w dy, sum
    // of w dy nhat), and whether that warp's wait for the slot succeeded
    float2* xch = reinterpret_cast<float2*>(tail + 16 * LNQ_RING + 16);
    int* xok = reinterpret_cast<int*>(tail + 16 * LNQ_RING + 16 + LNQ_XCH * 16);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int producer = LNQ_THREADS / 32 - 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < LNQ_RING; s++) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), NV);  // one arrival per warp of the group
        }
        *abort_flag = 0;
        *issued_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_enter();
    // this CTA's rows: a contiguous range, in slots of LNQ_SR rows
    const int per = (N + (int)gridDim.x - 1) / (int)gridDim.x;
    const int r_begin = min(N, (int)blockIdx.x * per), r_end = min(N, r_begin + per);
    const int nk = (r_end - r_begin + LNQ_SR - 1) / LNQ_SR;  // slots of this CTA
    const int cv = C / VEC;
    const int G = with_colsum ? 3 : 2;
    const int grp = warp / NV, wig = warp % NV;  // row group, warp in group
    const int vi = wig * 32 + lane;              // this lane's vector of the row
    const bool has = warp < CWARPS && vi < cv;
    float adw[VEC], adb[VEC], acs[VEC];
#pragma unroll
    for (int e = 0; e < VEC; e++) adw[e] = adb[e] = acs[e] = 0.f;
    if (warp == producer) {
        if (lane == 0) {
            int issued = 0;
            for (int k = 0; k < nk; k++) {
                const int s = k % LNQ_RING;
                if (!tc::mbar_wait(empty(s), (uint32_t)(((k / LNQ_RING) & 1) ^ 1), abort_flag)) break;
                const size_t r = (size_t)r_begin + (size_t)k * LNQ_SR;
                const uint32_t nb = (uint32_t)(min(LNQ_SR, r_end - (int)r) * rowb);
                const uint32_t dst = ring_s + (uint32_t)(s * slotb);
                tc::mbar_expect_tx(full(s), (accumulate ? 3u : 2u) * nb);
                tc::bulk_load(dst, inp + r * C, nb, full(s));
                tc::bulk_load(dst + arrb, dout + r * C, nb, full(s));
                if (accumulate) tc::bulk_load(dst + 2 * arrb, dinp + r * C, nb, full(s));
                ++issued;
            }
            *issued_s = issued;
        }
    } else if (warp < CWARPS) {
        Vec16<H> wv;
        if (has) wv = ld16(w + vi * VEC);
        int par = 0;
        bool ok_all = true;
        for (int k = grp; ok_all && k < nk; k += GROUPS) {
            const int s = k % LNQ_RING;
            int ok = 1;
            if (lane == 0) ok = tc::mbar_wait(full(s), (uint32_t)((k / LNQ_RING) & 1), abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // a failed wait is acted on only after the group's barrier below, so
            // that all of the group's warps leave together
            if (NV == 1 && !ok) break;
            const uint8_t* slot = ring + (size_t)s * slotb;
            const int r0 = r_begin + k * LNQ_SR;
            const int nrows = min(LNQ_SR, r_end - r0);
            // two rows at a time: their loads, sums and exchanges overlap
            for (int i = 0; i < nrows; i += 2, par ^= 1) {
                const int nr = min(2, nrows - i);
                float mu[2], rs[2], g[2][VEC], nh[2][VEC];
                Vec16<H> dvv[2], ovv[2];
                float gs[2] = {0.f, 0.f}, gns[2] = {0.f, 0.f};
                const bool use = has && ok;
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const size_t r = (size_t)r0 + i + (q < nr ? q : 0);
                    mu[q] = mean[r];
                    rs[q] = rstd[r];
                    const uint8_t* rowp = slot + (size_t)(i + (q < nr ? q : 0)) * rowb;
                    Vec16<H> xv;
                    if (use) {
                        xv = *reinterpret_cast<const Vec16<H>*>(rowp + vi * 16);
                        dvv[q] = *reinterpret_cast<const Vec16<H>*>(rowp + arrb + vi * 16);
                        if (accumulate) ovv[q] = *reinterpret_cast<const Vec16<H>*>(rowp + 2 * arrb + vi * 16);
                    }
#pragma unroll
                    for (int e = 0; e < VEC; e++) {
                        g[q][e] = use ? to_f(wv.v[e]) * to_f(dvv[q].v[e]) : 0.f;
                        nh[q][e] = use ? (to_f(xv.v[e]) - mu[q]) * rs[q] : 0.f;
                        gs[q] += g[q][e];
                        gns[q] += g[q][e] * nh[q][e];
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        gs[q] += __shfl_xor_sync(0xffffffffu, gs[q], o);
                        gns[q] += __shfl_xor_sync(0xffffffffu, gns[q], o);
                    }
                }
                if (NV > 1) {
                    // the group's warps exchange their sums and wait results
                    // (double-buffered by row-pair parity)
                    float4* x4 = reinterpret_cast<float4*>(xch) + ((size_t)grp * 2 + par) * NV;
                    int* o2 = xok + ((size_t)grp * 2 + par) * NV;
                    if (lane == 0) {
                        x4[wig] = make_float4(gs[0], gns[0], gs[1], gns[1]);
                        o2[wig] = ok;
                    }
                    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(NV * 32) : "memory");
                    gs[0] = gns[0] = gs[1] = gns[1] = 0.f;
#pragma unroll
                    for (int j2 = 0; j2 < NV; j2++) {
                        const float4 t = x4[j2];
                        ok_all = ok_all && o2[j2] != 0;
                        gs[0] += t.x;
                        gns[0] += t.y;
                        gs[1] += t.z;
                        gns[1] += t.w;
                    }
                    if (!ok_all) break;
                }
                if (use) {
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        if (q >= nr) break;
                        const float gm = gs[q] / C, gnm = gns[q] / C;
                        Vec16<H> o;
#pragma unroll
                        for (int e = 0; e < VEC; e++) {
                            const float val = rs[q] * (g[q][e] - gm - nh[q][e] * gnm);
                            const float d = to_f(dvv[q].v[e]);
                            o.v[e] = from_f<H>(accumulate ? to_f(ovv[q].v[e]) + val : val);
                            adw[e] += nh[q][e] * d;
                            adb[e] += d;
                            acs[e] += to_f(o.v[e]);
                        }
                        st16(dinp + ((size_t)r0 + i + q) * C + vi * VEC, o);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && ok) tc::mbar_arrive(empty(s));  // this warp is done with the slot
        }
    }
    __syncthreads();
    if (*abort_flag) {
        // let every issued copy land before the ring is reused or released
        if (threadIdx.x == 32 * producer) {
            const int issued = *issued_s;
            for (int s = 0; s < LNQ_RING && s < issued; s++) {
                const int lst = s + ((issued - 1 - s) / LNQ_RING) * LNQ_RING;
                tc::mbar_wait_drain(full(s), (uint32_t)((lst / LNQ_RING) & 1));
            }
            atomicOr(err, DEVERR_TIMEOUT);
        }
        __syncthreads();
    }
    // fold the row groups in order through the (now idle) ring memory:
    // fold[group][dw | db | colsum][column]
    float* fold = reinterpret_cast<float*>(lnq_sm);
    if (has) {
        float* mine = fold + (size_t)grp * G * C;
#pragma unroll
        for (int e = 0; e < VEC; e++) {
            mine[vi * VEC + e] = adw[e];
            mine[C + vi * VEC + e] = adb[e];
            if (with_colsum) mine[2 * C + vi * VEC + e] = acs[e];
        }
    }
    __syncthreads();
    float* dst = part + (size_t)blockIdx.x * G * C;
    for (int c = threadIdx.x; c < G * C; c += blockDim.x) {
        float t = 0.f;
        for (int gi = 0; gi < GROUPS; gi++) t += fold[(size_t)gi * G * C + c];
        dst[c] = t;
    }
}

// The same operation (bf16, C = 256 NV) with one warp per row: lane l holds
// the row's 16-byte vectors l, l + 32, ... (8 columns each), so every access
// of a warp covers 512 contiguous bytes, and the row sums are warp shuffles.
// Each warp streams its rows (x, dy and, for +=, the current dx) through its
// own ring of LNW_BUF row slots in shared memory with cp.async, so LNW_BUF - 1
// rows per warp are in flight while one is computed without holding them in
// registers. The dw / db / colsum partials of the lane's columns stay in
// registers across the warp's rows. The CTA's rows are a contiguous range,
// taken by its warps in turn; the warps' partials are folded in warp order
// into part[blockIdx.x] = [dw | db (| colsum)] (G*C floats).
constexpr int LNW_WARPS = 8;
constexpr int LNW_BUF = 4;

DEVI void lnw_cp16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <typename H, int NV>
__global__ void __launch_bounds__(32 * LNW_WARPS, 1) layernorm_backward_warp_k(
    H* __restrict__ dinp, float* __restrict__ part, const H* __restrict__ dout,
    const H* __restrict__ inp, const H* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int accumulate, int with_colsum) {
    constexpr int VEC = 8;
    constexpr int ROWB = 256 * NV * 2;  // bytes of one row of one array
    // [warp][slot][x | dy | dx] rows; reused at the end for the fold [warp][G][C]
    extern __shared__ __align__(16) uint8_t lnw_sm[];
    pdl_enter();
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int per = (N + (int)gridDim.x - 1) / (int)gridDim.x;
    const int r_begin = min(N, (int)blockIdx.x * per), r_end = min(N, r_begin + per);
    const int G = with_colsum ? 3 : 2;
    uint8_t* ring = lnw_sm + (size_t)warp * LNW_BUF * 3 * ROWB;
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    // packed fp32 arithmetic on column pairs: lane l's vector j holds columns
    // (l + 32 j) * 8 + 2 e, + 1 in pair e
    float2 wf[NV][VEC / 2];
#pragma unroll
    for (int j = 0; j < NV; j++) {
        const uint4 u = *reinterpret_cast<const uint4*>(w + (lane + 32 * j) * VEC);
        wf[j][0] = h2_f2w<H>(u.x); wf[j][1] = h2_f2w<H>(u.y); wf[j][2] = h2_f2w<H>(u.z); wf[j][3] = h2_f2w<H>(u.w);
    }
    float2 adw[NV][VEC / 2], adb[NV][VEC / 2], acs[NV][VEC / 2];
#pragma unroll
    for (int j = 0; j < NV; j++)
#pragma unroll
        for (int e = 0; e < VEC / 2; e++) adw[j][e] = adb[j][e] = acs[j][e] = make_float2(0.f, 0.f);
    // the warp's k-th row is r_begin + warp + k * LNW_WARPS, in slot k % LNW_BUF;
    // one commit group per row (empty groups past the end keep the count)
    auto issue = [&](int k) {
        const int r = r_begin + warp + k * LNW_WARPS;
        if (r < r_end) {
            const uint32_t slot = ring_s + (uint32_t)((k % LNW_BUF) * 3 * ROWB);
            const size_t off = (size_t)r * C + lane * VEC;
#pragma unroll
            for (int j = 0; j < NV; j++) {
                const uint32_t o = (uint32_t)((lane + 32 * j) * 16);
                lnw_cp16(slot + o, inp + off + 32 * j * VEC);
                lnw_cp16(slot + ROWB + o, dout + off + 32 * j * VEC);
                if (accumulate) lnw_cp16(slot + 2 * ROWB + o, dinp + off + 32 * j * VEC);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int k = 0; k < LNW_BUF - 1; k++) issue(k);
    // lane l holds the mean and rstd of the warp's row k0 + l (k0 = k rounded
    // down to a multiple of 32), read a batch at a time ahead of their rows
    float mu_l = 0.f, rs_l = 0.f;
    for (int k = 0;; k++) {
        const int r = r_begin + warp + k * LNW_WARPS;
        if (r >= r_end) break;
        if ((k & 31) == 0) {
            const int rr = r + lane * LNW_WARPS;
            mu_l = rr < r_end ? mean[rr] : 0.f;
            rs_l = rr < r_end ? rstd[rr] : 0.f;
        }
        issue(k + LNW_BUF - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(LNW_BUF - 1) : "memory");
        __syncwarp();
        const uint8_t* slot = ring + (size_t)(k % LNW_BUF) * 3 * ROWB;
        const float mu = __shfl_sync(0xffffffffu, mu_l, k & 31), rs = __shfl_sync(0xffffffffu, rs_l, k & 31);
        const float2 rs2 = make_float2(rs, rs), nmr = make_float2(-mu * rs, -mu * rs);
        // g = w dy and nhat = (x - mean) rstd per column; the row sums of g and
        // g nhat; the dw, db column partials
        float2 g[NV][VEC / 2], nh[NV][VEC / 2];
        float2 gs2 = make_float2(0.f, 0.f), gns2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NV; j++) {
            const uint4 xu = *reinterpret_cast<const uint4*>(slot + (lane + 32 * j) * 16);
            const uint4 du = *reinterpret_cast<const uint4*>(slot + ROWB + (lane + 32 * j) * 16);
            const uint32_t xw[4] = {xu.x, xu.y, xu.z, xu.w}, dw[4] = {du.x, du.y, du.z, du.w};
#pragma unroll
            for (int e = 0; e < VEC / 2; e++) {
                const float2 d = h2_f2w<H>(dw[e]);
                g[j][e] = fmul2(wf[j][e], d);
                nh[j][e] = ffma2(h2_f2w<H>(xw[e]), rs2, nmr);
                gs2 = fadd2(gs2, g[j][e]);
                gns2 = ffma2(g[j][e], nh[j][e], gns2);
                adw[j][e] = ffma2(nh[j][e], d, adw[j][e]);
                adb[j][e] = fadd2(adb[j][e], d);
            }
        }
        float gs = gs2.x + gs2.y, gns = gns2.x + gns2.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            gs += __shfl_xor_sync(0xffffffffu, gs, o);
            gns += __shfl_xor_sync(0xffffffffu, gns, o);
        }
        // dx = rstd (g - mean(g) - nhat mean(g nhat)) = rstd g + c0 + c1 nhat
        const float c0 = -rs * (gs / C), c1 = -rs * (gns / C);
        const float2 c02 = make_float2(c0, c0), c12 = make_float2(c1, c1);
        H* dx = dinp + (size_t)r * C + lane * VEC;
#pragma unroll
        for (int j = 0; j < NV; j++) {
            uint32_t ow[4] = {0u, 0u, 0u, 0u};
            if (accumulate) {
                const uint4 ou = *reinterpret_cast<const uint4*>(slot + 2 * ROWB + (lane + 32 * j) * 16);
                ow[0] = ou.x; ow[1] = ou.y; ow[2] = ou.z; ow[3] = ou.w;
            }
            uint32_t res[4];
#pragma unroll
            for (int e = 0; e < VEC / 2; e++) {
                float2 v = ffma2(nh[j][e], c12, ffma2(g[j][e], rs2, c02));
                if (accumulate) v = fadd2(h2_f2w<H>(ow[e]), v);
                res[e] = f2_h2v<H>(v);
                acs[j][e] = fadd2(acs[j][e], h2_f2w<H>(res[e]));
            }
            *reinterpret_cast<uint4*>(dx + 32 * j * VEC) = make_uint4(res[0], res[1], res[2], res[3]);
        }
        __syncwarp();  // every lane has read the slot before it is refilled
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // fold the warps in order through the (now idle) rings: [warp][G][C]
    float* fold = reinterpret_cast<float*>(lnw_sm);
    float* mine = fold + (size_t)warp * G * C;
#pragma unroll
    for (int j = 0; j < NV; j++)
#pragma unroll
        for (int e = 0; e < VEC / 2; e++) {
            const int c = (lane + 32 * j) * VEC + 2 * e;
            *reinterpret_cast<float2*>(mine + c) = adw[j][e];
            *reinterpret_cast<float2*>(mine + C + c) = adb[j][e];
            if (with_colsum) *reinterpret_cast<float2*>(mine + 2 * C + c) = acs[j][e];
        }
    __syncthreads();
    float* dst = part + (size_t)blockIdx.x * G * C;
    for (int c = threadIdx.x; c < G * C; c += blockDim.x) {
        float t = 0.f;
#pragma unroll
        for (int wi = 0; wi < LNW_WARPS; wi++) t += fold[(size_t)wi * G * C + c];
        dst[c] = t;
    }
}

// dst[c] (+)= sum over p of part[p * pstride + c] for every descriptor, summed in
// increasing p (one launch for many parameter tensors)
template <typename T>
__global__ void __launch_bounds__(256) reduce_partials_multi_k(const PartialDesc* __restrict__ d) {
    pdl_enter();
    const PartialDesc pd = d[blockIdx.y];
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= pd.width) return;
    const float* p = pd.part + c;
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < pd.P; i++) acc += p[(size_t)i * pd.pstride];
    T* o = (T*)pd.dst + c;
    *o = from_f<T>(to_f(*o) + acc);
}

// dst[c] += sum over p of ws[p][c] for c in [0, W), summed in increasing p;
// columns [split, W) go to dst2[c - split]. One warp per (32-column group,
// p residue mod 8), folded across the 8 warps in order.
template <typename T>
__global__ void __launch_bounds__(256) reduce_partials_k(T* __restrict__ dst, T* __restrict__ dst2,
                                                         int split, const float* __restrict__ ws,
                                                         int P, int W) {
    pdl_enter();
    __shared__ float part[8][33];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (c < W) {
#pragma unroll 8
        for (int p = warp; p < P; p += 8) acc += ws[(size_t)p * W + c];
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c < W) {
        float t = 0.f;
#pragma unroll
        for (int wi = 0; wi < 8; wi++) t += part[wi][lane];
        T* o = c < split ? dst + c : dst2 + (c - split);
        *o = from_f<T>(to_f(*o) + t);
    }
}

// one wave: as many blocks as are resident at once (at most 4 per SM), each
// walking rows with its warps
template <typename T, int NV>
static int lnb_blocks(int N, size_t smem) {
    static int per_sm = 0;
    if (per_sm == 0) {
        cudaFuncSetAttribute(layernorm_backward_k<T, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(float) * 2 * 2048 * (LNB_BLOCK / 32)));
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layernorm_backward_k<T, NV>, LNB_BLOCK,
                                                          smem) != cudaSuccess || n < 1)
            n = 1;
        per_sm = n < 4 ? n : 4;
    }
    const int rows_per_block = LNB_BLOCK / 32;
    const int g = (N + rows_per_block - 1) / rows_per_block;
    const int cap = per_sm * num_sms();
    return g < cap ? (g < 1 ? 1 : g) : cap;
}

size_t layernorm_backward_ws_floats(int C) { return (size_t)4 * num_sms() * 2 * C; }

void launch_layernorm_backward(DType dt, void* dinp, void* dw, void* db, const void* dout,
                               const void* inp, const void* w, const float* mean,
                               const float* rstd, int N, int C, int accumulate, float* ws,
                               unsigned int* err, cudaStream_t s) {
    // partial rows [P][dw | db], then their in-order sum into dw and db
    const int P = launch_layernorm_backward_part(dt, dinp, ws, dout, inp, w, mean, rstd, N, C,
                                                 accumulate, 0, err, s);
    note_launch(1);
    const unsigned rg = (unsigned)((2 * C + 31) / 32);
    DISPATCH_E(dt, launch_pdl(reduce_partials_k<E>, rg, 256, 0, s, (E*)dw, (E*)db, C, ws, P, 2 * C));
}

// ------------------------------------------------------------------ partial-row form
bool layernorm_backward_fuses_colsum(DType dt, int C) {
    // the bulk-copy kernel up to 768 columns, the warp-per-row kernel also at 1024
    return dt != DT_F32 && (C * 2) % 16 == 0 && ((C / 8 + 31) / 32 <= 3 || C == 1024);
}

int layernorm_backward_part_rows(DType dt, int N, int C) {
    if (layernorm_backward_fuses_colsum(dt, C)) return N < num_sms() ? N : num_sms();
    const size_t smem = sizeof(float) * 2 * C * (LNB_BLOCK / 32);
    const int nv = (C / dtype_vec(dt) + 31) / 32;
    if (dt == DT_BF16) {
        switch (nv) {
            case 4: return lnb_blocks<bf16, 4>(N, smem); case 5: return lnb_blocks<bf16, 5>(N, smem);
            case 6: return lnb_blocks<bf16, 6>(N, smem); case 7: return lnb_blocks<bf16, 7>(N, smem);
            default: return lnb_blocks<bf16, 8>(N, smem);
        }
    }
    if (dt == DT_F16) {  // (each instantiation opts in to its shared memory itself)
        switch (nv) {
            case 4: return lnb_blocks<f16, 4>(N, smem); case 5: return lnb_blocks<f16, 5>(N, smem);
            case 6: return lnb_blocks<f16, 6>(N, smem); case 7: return lnb_blocks<f16, 7>(N, smem);
            default: return lnb_blocks<f16, 8>(N, smem);
        }
    }
    switch (nv) {
        case 1: return lnb_blocks<float, 1>(N, smem); case 2: return lnb_blocks<float, 2>(N, smem);
        case 3: return lnb_blocks<float, 3>(N, smem); case 4: return lnb_blocks<float, 4>(N, smem);
        case 5: return lnb_blocks<float, 5>(N, smem); case 6: return lnb_blocks<float, 6>(N, smem);
        case 7: return lnb_blocks<float, 7>(N, smem); default: return lnb_blocks<float, 8>(N, smem);
    }
}

template <typename H, int NV> static size_t lnq_opt_in(int C) {
    const size_t smem = lnq_body_bytes(C, (LNQ_THREADS / 32 - 1) / NV) + 16 * LNQ_RING + 16 + LNQ_XCH * 20;
    static size_t done = 0;
    if (smem > done) {
        cudaFuncSetAttribute(layernorm_backward_bulk_k<H, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        done = smem;
    }
    return smem;
}

int launch_layernorm_backward_part(DType dt, void* dinp, float* part, const void* dout,
                                   const void* inp, const void* w, const float* mean,
                                   const float* rstd, int N, int C, int accumulate, int with_colsum,
                                   unsigned int* err, cudaStream_t s) {
    const int P = layernorm_backward_part_rows(dt, N, C);
    if (layernorm_backward_fuses_colsum(dt, C) && C % 256 == 0) {
        const int nv = C / 256;
        // the warps' row rings, later reused by the fold [warp][3][C] fp32
        const size_t ring = (size_t)LNW_WARPS * LNW_BUF * 3 * C * 2, fold = sizeof(float) * LNW_WARPS * 3 * C;
        const size_t smem = ring > fold ? ring : fold;
        note_launch(1);
#define LNW(H, NVV)                                                                                    \
    do {                                                                                               \
        static size_t done = 0;                                                                        \
        if (smem > done) {                                                                             \
            cudaFuncSetAttribute(layernorm_backward_warp_k<H, NVV>,                                    \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);              \
            done = smem;                                                                               \
        }                                                                                              \
        launch_pdl(layernorm_backward_warp_k<H, NVV>, dim3(P), dim3(32 * LNW_WARPS), smem, s,          \
                   (H*)dinp, part, (const H*)dout, (const H*)inp, (const H*)w, mean, rstd,             \
                   N, C, accumulate, with_colsum);                                                     \
    } while (0)
        if (dt == DT_BF16) {
            if (nv == 1) LNW(bf16, 1); else if (nv == 2) LNW(bf16, 2); else if (nv == 3) LNW(bf16, 3);
            else LNW(bf16, 4);
        } else {
            if (nv == 1) LNW(f16, 1); else if (nv == 2) LNW(f16, 2); else if (nv == 3) LNW(f16, 3);
            else LNW(f16, 4);
        }
#undef LNW
        return P;
    }
    if (layernorm_backward_fuses_colsum(dt, C)) {
        const int nv = (C / 8 + 31) / 32;
        note_launch(1);
#define LNQ(H, NVV)                                                                              \
    launch_pdl(layernorm_backward_bulk_k<H, NVV>, dim3(P), dim3(LNQ_THREADS),                    \
               lnq_opt_in<H, NVV>(C), s, (H*)dinp, part, (const H*)dout, (const H*)inp,          \
               (const H*)w, mean, rstd, N, C, accumulate, with_colsum, err)
        if (dt == DT_BF16) {
            if (nv == 1) LNQ(bf16, 1); else if (nv == 2) LNQ(bf16, 2); else LNQ(bf16, 3);
        } else {
            if (nv == 1) LNQ(f16, 1); else if (nv == 2) LNQ(f16, 2); else LNQ(f16, 3);
        }
#undef LNQ
        return P;
    }
    note_launch(1);
    const size_t smem = sizeof(float) * 2 * C * (LNB_BLOCK / 32);
    const int nv = (C / dtype_vec(dt) + 31) / 32;
#define LNB2(TT, NVV)                                                                            \
    launch_pdl(layernorm_backward_k<TT, NVV>, dim3(P), dim3(LNB_BLOCK), smem, s, (TT*)dinp, part,  \
               (const TT*)dout, (const TT*)inp, (const TT*)w, mean, rstd, N, C, accumulate)
    if (dt == DT_BF16) {
        switch (nv) {
            case 4: LNB2(bf16, 4); break; case 5: LNB2(bf16, 5); break; case 6: LNB2(bf16, 6); break;
            case 7: LNB2(bf16, 7); break; default: LNB2(bf16, 8); break;
        }
    } else if (dt == DT_F16) {
        switch (nv) {
            case 4: LNB2(f16, 4); break; case 5: LNB2(f16, 5); break; case 6: LNB2(f16, 6); break;
            case 7: LNB2(f16, 7); break; default: LNB2(f16, 8); break;
        }
    } else {
        switch (nv) {
            case 1: LNB2(float, 1); break; case 2: LNB2(float, 2); break; case 3: LNB2(float, 3); break;
            case 4: LNB2(float, 4); break; case 5: LNB2(float, 5); break; case 6: LNB2(float, 6); break;
            case 7: LNB2(float, 7); break; default: LNB2(float, 8); break;
        }
    }
#undef LNB2
    return P;
}

void launch_reduce_partials_multi(DType dt, const PartialDesc* d_desc, int ndesc, int maxwidth,
                                  cudaStream_t s) {
    if (ndesc <= 0) return;
    note_launch(1);
    const dim3 grid((unsigned)((maxwidth + 255) / 256), (unsigned)ndesc);
    DISPATCH_E(dt, launch_pdl(reduce_partials_multi_k<E>, grid, dim3(256), 0, s, d_desc));
}

// ------------------------------------------------------------------ bias gradient
// matmul_backward_bias_kernel4 read with +=: dbias[n] += sum over rows of dout[:, n].
// Stage 1: block (x: 32*VEC columns, y: a slab of rows), 8 warps stride the
// slab, warps folded in order; stage 2 (reduce_partials_k) sums the slabs in order.
constexpr int CS_SLABS = 128;

template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_k(float* __restrict__ ws,
                                                        const T* __restrict__ dout, int M, int N,
                                                        int rows_per_slab) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    __shared__ float sm[8][32 * VEC];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int col = (blockIdx.x * 32 + lane) * VEC;
    const int r0 = blockIdx.y * rows_per_slab;
    const int r1 = min(M, r0 + rows_per_slab);
    float acc[VEC];
#pragma unroll
    for (int k = 0; k < VEC; k++) acc[k] = 0.f;
    if (col < N) {
        const T* p = dout + col;
        int r = r0 + warp;
        // four independent rows per iteration keep four loads in flight per lane
        for (; r + 24 < r1; r += 32) {
            const Vec16<T> a = ld16_cs(p + (size_t)r * N), b = ld16_cs(p + (size_t)(r + 8) * N);
            const Vec16<T> c = ld16_cs(p + (size_t)(r + 16) * N), d = ld16_cs(p + (size_t)(r + 24) * N);
#pragma unroll
            for (int k = 0; k < VEC; k++)
                acc[k] += (to_f(a.v[k]) + to_f(b.v[k])) + (to_f(c.v[k]) + to_f(d.v[k]));
        }
        for (; r < r1; r += 8) {
            const Vec16<T> a = ld16_cs(p + (size_t)r * N);
#pragma unroll
            for (int k = 0; k < VEC; k++) acc[k] += to_f(a.v[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < VEC; k++) sm[warp][lane * VEC + k] = acc[k];
    __syncthreads();
    for (int c = threadIdx.x; c < 32 * VEC; c += blockDim.x) {
        float sacc = 0.f;
        for (int wi = 0; wi < 8; wi++) sacc += sm[wi][c];
        int gc = blockIdx.x * 32 * VEC + c;
        if (gc < N) ws[(size_t)blockIdx.y * N + gc] = sacc;
    }
}

size_t colsum_ws_floats(int N) { return (size_t)CS_SLABS * N; }

int colsum_part_rows(int M) {
    int R = (M + 31) / 32;
    if (R > CS_SLABS) R = CS_SLABS;
    if (R < 1) R = 1;
    const int rps = (M + R - 1) / R;
    return (M + rps - 1) / rps;
}

int launch_colsum_part(DType dt, float* part, const void* dout, int M, int N, cudaStream_t s) {
    const int R = colsum_part_rows(M);
    const int rps = (M + R - 1) / R;
    const int VEC = dtype_vec(dt);
    const dim3 grid((N + 32 * VEC - 1) / (32 * VEC), R);
    note_launch(1);
    DISPATCH_E(dt, launch_pdl(colsum_partial_k<E>, grid, dim3(256), 0, s, part, (const E*)dout, M, N, rps));
    return R;
}

void launch_colsum_accum(DType dt, void* dbias, const void* dout, int M, int N, float* ws,
                         cudaStream_t s) {
    note_launch(2);
    const int VEC = dtype_vec(dt);
    int R = (M + 31) / 32;
    if (R > CS_SLABS) R = CS_SLABS;
    if (R < 1) R = 1;
    int rps = (M + R - 1) / R;
    R = (M + rps - 1) / rps;
    dim3 grid((N + 32 * VEC - 1) / (32 * VEC), R);
    const unsigned rg = (unsigned)((N + 31) / 32);
    DISPATCH_E(dt, launch_pdl(colsum_partial_k<E>, grid, 256, 0, s, ws, (const E*)dout, M, N, rps);
                   launch_pdl(reduce_partials_k<E>, rg, 256, 0, s, (E*)dbias, (E*)dbias, N, ws, R, N));
}

// ------------------------------------------------------------------ classifier
// fused_classifier_kernel3: per row, softmax over the first V logits,
// loss = log(sum exp(l - max)) + max - l[target], and the logits are replaced
// by dlogits = (p - 1[i == target]) * dloss; the padded columns [V, Vp) get 0.
// Pass 1 reads the row once (online max/sum per 16-byte vector); pass 2
// re-reads it (an L2 hit: each block's row is only ~100 KB) and writes. Both
// passes issue CLS_UNROLL independent 16-byte loads per thread before using
// them, so enough bytes are in flight to cover the memory latency.
// exp(x - m) is taken as 2^(x log2(e) - m log2(e)): one FMA and the hardware
// ex2 per element (relative error ~2^-22).
constexpr int CLS_BLOCK = 512;
constexpr int CLS_UNROLL = 4;
constexpr float CLS_LOG2E = 1.4426950408889634f;

DEVI float cls_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
__global__ void __launch_bounds__(CLS_BLOCK, 3) classifier_k(T* __restrict__ logits,
                                                          float* __restrict__ losses,
                                                          const int* __restrict__ targets, int V,
                                                          int Vp, float dloss,
                                                          const float* __restrict__ dloss_scale) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    if (dloss_scale) dloss *= *dloss_scale;  // loss scaling (fp16 training)
    __shared__ float s_max[32], s_sum[32];
    __shared__ float s_tlogit;
    const int row = blockIdx.x;
    T* x = logits + (size_t)row * Vp;
    const int tgt = targets[row];
    if (threadIdx.x == 0) s_tlogit = to_f(x[tgt]);
    const int nvec = Vp / VEC;
    float m = -INFINITY, sum = 0.f;
    auto update = [&](const Vec16<T>& a, int vi) {
        float f[VEC];
        float lm = -INFINITY;
#pragma unroll
        for (int k = 0; k < VEC; k++) {
            f[k] = (vi * VEC + k < V) ? to_f(a.v[k]) : -INFINITY;
            lm = fmaxf(lm, f[k]);
        }
        if (lm == -INFINITY) return;
        const float nm = fmaxf(m, lm), nl = -nm * CLS_LOG2E;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < VEC; k++) acc += cls_exp2(fmaf(f[k], CLS_LOG2E, nl));
        sum = sum * cls_exp2((m - nm) * CLS_LOG2E) + acc;
        m = nm;
    };
    int vi = threadIdx.x;
    for (; vi + (CLS_UNROLL - 1) * CLS_BLOCK < nvec; vi += CLS_UNROLL * CLS_BLOCK) {
        Vec16<T> a[CLS_UNROLL];
#pragma unroll
        for (int u = 0; u < CLS_UNROLL; u++) a[u] = ld16(x + (size_t)(vi + u * CLS_BLOCK) * VEC);
#pragma unroll
        for (int u = 0; u < CLS_UNROLL; u++) update(a[u], vi + u * CLS_BLOCK);
    }
    for (; vi < nvec; vi += CLS_BLOCK) update(ld16(x + (size_t)vi * VEC), vi);
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32, nw = blockDim.x / 32;
    float wm = warp_max(m);
    if (lane == 0) s_max[warp] = wm;
    __syncthreads();
    float bm = warp_max(lane < nw ? s_max[lane] : -INFINITY);
    float ws = warp_sum(m == -INFINITY ? 0.f : sum * cls_exp2((m - bm) * CLS_LOG2E));
    if (lane == 0) s_sum[warp] = ws;
    __syncthreads();
    const float bs = warp_sum(lane < nw ? s_sum[lane] : 0.f);
    if (threadIdx.x == 0) losses[row] = logf(bs) + bm - s_tlogit;
    const float inv = 1.f / bs, bl = -bm * CLS_LOG2E;
    auto grad = [&](const Vec16<T>& a, int vi) {
        Vec16<T> o;
#pragma unroll
        for (int k = 0; k < VEC; k++) {
            const int i = vi * VEC + k;
            float d = 0.f;
            if (i < V) {
                const float p = cls_exp2(fmaf(to_f(a.v[k]), CLS_LOG2E, bl)) * inv;
                d = (p - (i == tgt ? 1.f : 0.f)) * dloss;
            }
            o.v[k] = from_f<T>(d);
        }
        st16_cs(x + (size_t)vi * VEC, o);
    };
    vi = threadIdx.x;
    for (; vi + (CLS_UNROLL - 1) * CLS_BLOCK < nvec; vi += CLS_UNROLL * CLS_BLOCK) {
        Vec16<T> a[CLS_UNROLL];
#pragma unroll
        for (int u = 0; u < CLS_UNROLL; u++) a[u] = ld16(x + (size_t)(vi + u * CLS_BLOCK) * VEC);
#pragma unroll
        for (int u = 0; u < CLS_UNROLL; u++) grad(a[u], vi + u * CLS_BLOCK);
    }
    for (; vi < nvec; vi += CLS_BLOCK) grad(ld16(x + (size_t)vi * VEC), vi);
}

void launch_classifier(DType dt, void* logits, float* losses, const int* targets, int BT, int V,
                       int Vp, float dloss, cudaStream_t s, const float* dloss_scale) {
    note_launch(1);
    DISPATCH_E(dt, launch_pdl(classifier_k<E>, BT, CLS_BLOCK, 0, s, (E*)logits, losses, targets, V, Vp, dloss,
                              dloss_scale));
}

// ------------------------------------------------------------------ inference
// Probabilities of the tied classifier (fused_classifier_kernel3's probs
// output, for a forward without targets): probs[r][i] = softmax over i < V of
// logits[r][:], 0 on the padding [V, Vp). One block per row.
template <typename T>
__global__ void __launch_bounds__(512) probs_k(float* __restrict__ probs, const T* __restrict__ logits,
                                               int V, int Vp) {
    pdl_enter();
    __shared__ float s_red[32];
    const T* x = logits + (size_t)blockIdx.x * Vp;
    float* y = probs + (size_t)blockIdx.x * Vp;
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32, nw = blockDim.x / 32;
    float m = -INFINITY;
    for (int i = threadIdx.x; i < V; i += blockDim.x) m = fmaxf(m, to_f(x[i]));
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    m = warp_max(lane < nw ? s_red[lane] : -INFINITY);
    __syncthreads();
    float sum = 0.f;
    for (int i = threadIdx.x; i < V; i += blockDim.x) sum += expf(to_f(x[i]) - m);
    sum = warp_sum(sum);
    if (lane == 0) s_red[warp] = sum;
    __syncthreads();
    sum = warp_sum(lane < nw ? s_red[lane] : 0.f);
    const float inv = 1.f / sum;
    for (int i = threadIdx.x; i < Vp; i += blockDim.x) y[i] = i < V ? expf(to_f(x[i]) - m) * inv : 0.f;
}

void launch_probs(DType dt, float* probs, const void* logits, int rows, int V, int Vp, cudaStream_t s) {
    note_launch(1);
    DISPATCH_E(dt, launch_pdl(probs_k<E>, rows, 512, 0, s, probs, (const E*)logits, V, Vp));
}

// sample_softmax on the device: one block per row r, logits row at
// logits + r * row_stride; with p = softmax over i < V and the coin c in
// [0, 1), the sample is the first i whose cumulative probability exceeds c
// (V - 1 if rounding leaves none). The row max is subtracted before
// exponentiating (same probabilities, no overflow). Thread j owns the
// contiguous index range [j*chunk, (j+1)*chunk); the block scans the range
// sums, and the thread whose range holds c * sum walks it in index order.
// The index goes to out[r * out_stride].
constexpr int SAMPLE_BLOCK = 1024;

template <typename T>
__global__ void __launch_bounds__(SAMPLE_BLOCK) sample_k(const T* __restrict__ logits, long long row_stride,
                                                         int V, const float* __restrict__ coins,
                                                         int* __restrict__ out, long long out_stride) {
    pdl_enter();
    __shared__ float s_red[32];
    __shared__ int s_idx;
    const T* x = logits + (size_t)blockIdx.x * row_stride;
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
    constexpr int NW = SAMPLE_BLOCK / 32;
    float m = -INFINITY;
    for (int i = threadIdx.x; i < V; i += SAMPLE_BLOCK) m = fmaxf(m, to_f(x[i]));
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    if (threadIdx.x == 0) s_idx = V - 1;
    __syncthreads();
    m = warp_max(s_red[lane]);
    __syncthreads();
    const int chunk = (V + SAMPLE_BLOCK - 1) / SAMPLE_BLOCK;
    const int i0 = min(V, (int)threadIdx.x * chunk), i1 = min(V, i0 + chunk);
    float own = 0.f;
    for (int i = i0; i < i1; i++) own += expf(to_f(x[i]) - m);
    // inclusive scan of the range sums: within the warp, then over warps
    float inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        float w = s_red[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        s_red[lane] = w;
    }
    __syncthreads();
    const float before = warp > 0 ? s_red[warp - 1] : 0.f;
    inc += before;
    const float excl = inc - own;
    const float target = coins[blockIdx.x] * s_red[NW - 1];
    if (target < inc && i1 > i0) {
        // this range or an earlier one holds the sample: the first such range wins
        float cdf = excl;
        int idx = i1 - 1;
        for (int i = i0; i < i1; i++) {
            cdf += expf(to_f(x[i]) - m);
            if (target < cdf) {
                idx = i;
                break;
            }
        }
        atomicMin(&s_idx, idx);
    }
    __syncthreads();
    if (threadIdx.x == 0) out[(size_t)blockIdx.x * out_stride] = s_idx;
}

void launch_sample(DType dt, const void* logits, long long row_stride, int rows, int V, const float* coins,
                   int* out, long long out_stride, cudaStream_t s) {
    note_launch(1);
    DISPATCH_E(dt, launch_pdl(sample_k<E>, rows, SAMPLE_BLOCK, 0, s, (const E*)logits, row_stride, V, coins,
                              out, out_stride));
}

// mean of n floats in a fixed order (single block)
__global__ void __launch_bounds__(1024) mean_k(const float* __restrict__ x, int n,
                                               float* __restrict__ out) {
    pdl_enter();
    __shared__ float sw[32];
    float s = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += x[i];
    s = warp_sum(s);
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
    if (lane == 0) sw[warp] = s;
    __syncthreads();
    if (warp == 0) {
        float t = lane < (int)(blockDim.x / 32) ? sw[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) out[0] = t / (float)n;
    }
}

void launch_mean(const float* x, int n, float* out, cudaStream_t s) {
    note_launch(1);
    launch_pdl(mean_k, 1, 1024, 0, s, x, n, out);
}

// ------------------------------------------------------------------ AdamW
// adamw_kernel3 (master-weight path) / train_gpt2_fp32.cu adamw_kernel2:
// m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2, theta -= lr (mhat/(sqrt(vhat)+eps) + wd theta).
template <typename T>
DEVI float adamw_one(float g, float& m, float& v, float theta, float lr, float b1, float b2,
                     float c1, float c2, float eps, float wd) {
    m = fmaf(b1, m - g, g);          // b1 m + (1 - b1) g
    v = fmaf(b2, v - g * g, g * g);  // b2 v + (1 - b2) g^2
    float mh = m / c1, vh = v / c2;
    return theta - lr * (mh / (sqrtf(vh) + eps) + wd * theta);
}

// adamw_kernel3 without master weights: the update in fp32, operation by
// operation as the page writes it (lerp as two FMAs; the rn intrinsics keep
// the compiler from contracting or reordering), then stochastic rounding of
// the result to bf16. Element `idx` of the flat buffer is the page's thread
// idx % 512 of block idx / 512; its random word is the SquirrelNoise5 hash of
// that position under the step's seed, hashed once more with the same
// position by the page's bf16 rounding routine.
DEVI uint32_t squirrel_noise5(uint32_t pos, uint32_t seed) {
    uint32_t b = pos * 0xd2a80a3fu;
    b += seed;
    b ^= b >> 9;
    b += 0xa884f197u;
    b ^= b >> 11;
    b *= 0x6C736F4Bu;
    b ^= b >> 13;
    b += 0xB79F3ABBu;
    b ^= b >> 15;
    b *= 0x1b56c4f5u;
    b ^= b >> 17;
    return b;
}
DEVI uint32_t noise_2d(uint32_t x, uint32_t y, uint32_t seed) {
    return squirrel_noise5(x + 198491317u * y, seed);
}
DEVI bf16 round_bf16_stochastic(float p, size_t idx, uint32_t seed) {
    const uint32_t x = (uint32_t)(idx & 511), y = (uint32_t)(idx >> 9);
    const uint32_t rnd = noise_2d(x, y, noise_2d(x, y, seed));
    uint32_t bits = __float_as_uint(p);
    bits = (bits & 0xFFFFu) > (rnd & 0xFFFFu) ? (bits | 0xFFFFu) : (bits & ~0xFFFFu);
    return __float2bfloat16_rn(__uint_as_float(bits));
}
DEVI float adamw_one_sr(float g, float& m, float& v, float old, float lr, float b1, float b2,
                        float c1, float c2, float eps, float wd) {
    m = __fmaf_rn(b1, m, __fmaf_rn(-b1, g, g));
    const float gg = __fmul_rn(g, g);
    v = __fmaf_rn(b2, v, __fmaf_rn(-b2, gg, gg));
    const float mh = __fdiv_rn(m, c1), vh = __fdiv_rn(v, c2);
    const float den = __fadd_rn(__fsqrt_rn(vh), eps);
    const float upd = __fadd_rn(__fdiv_rn(mh, den), __fmul_rn(wd, old));
    return __fsub_rn(old, __fmul_rn(lr, upd));
}

// SR: bf16 parameters without a master copy, updated in place with
// stochastic rounding (seed: this step's, or hyper[7] in graph replays).
// scaler (fp16 training): the gradients hold loss-scale times the gradient;
// a step whose gradients overflowed is skipped, the others are unscaled
// (multiplied by 1/scale, a power of two: exact).
template <typename T, bool SR>
__global__ void adamw_k(T* __restrict__ params, float* __restrict__ master,
                        const T* __restrict__ grads, float* __restrict__ mst,
                        float* __restrict__ vst, const AdamRanges r, float lr, float b1, float b2,
                        float c1, float c2, float eps, float wd, uint32_t seed,
                        const float* __restrict__ hyper, const LossScaler* __restrict__ scaler) {
    pdl_enter();
    if (hyper) {  // hyperparameters from device memory (graph replays)
        lr = hyper[0]; b1 = hyper[1]; b2 = hyper[2]; c1 = hyper[3]; c2 = hyper[4];
        eps = hyper[5]; wd = hyper[6];
        seed = __float_as_uint(hyper[7]);
    }
    float inv_scale = 1.f;
    if (scaler) {
        if (scaler->found_inf) return;  // the whole update is skipped
        inv_scale = 1.f / scaler->scale;
    }
    // this block row's range of the flat parameter buffers
    const size_t off = r.off[blockIdx.y], n = r.n[blockIdx.y];
    params += off;
    grads += off;
    mst += off;
    vst += off;
    if (master) master += off;
    const size_t stride = (size_t)gridDim.x * blockDim.x * 4;
    for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
        if (i + 4 <= n) {
            float4 m4 = __ldcs(reinterpret_cast<const float4*>(mst + i));
            float4 v4 = __ldcs(reinterpret_cast<const float4*>(vst + i));
            float g[4], th[4];
            if constexpr (sizeof(T) == 2) {
                uint2 graw = __ldcs(reinterpret_cast<const uint2*>(grads + i));
                const T* gb = reinterpret_cast<const T*>(&graw);
#pragma unroll
                for (int k = 0; k < 4; k++) g[k] = to_f(gb[k]) * inv_scale;
            } else {
                float4 g4 = __ldcs(reinterpret_cast<const float4*>(grads + i));
                g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
            }
            if (!SR && master) {
                float4 t4 = __ldcs(reinterpret_cast<const float4*>(master + i));
                th[0] = t4.x; th[1] = t4.y; th[2] = t4.z; th[3] = t4.w;
            } else {
#pragma unroll
                for (int k = 0; k < 4; k++) th[k] = to_f(params[i + k]);
            }
            float mm[4] = {m4.x, m4.y, m4.z, m4.w}, vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                if constexpr (SR) th[k] = adamw_one_sr(g[k], mm[k], vv[k], th[k], lr, b1, b2, c1, c2, eps, wd);
                else th[k] = adamw_one<T>(g[k], mm[k], vv[k], th[k], lr, b1, b2, c1, c2, eps, wd);
            }
            __stcs(reinterpret_cast<float4*>(mst + i), make_float4(mm[0], mm[1], mm[2], mm[3]));
            __stcs(reinterpret_cast<float4*>(vst + i), make_float4(vv[0], vv[1], vv[2], vv[3]));
            if (!SR && master)
                __stcs(reinterpret_cast<float4*>(master + i), make_float4(th[0], th[1], th[2], th[3]));
            if constexpr (sizeof(T) == 2) {
                uint2 praw;
                T* pb = reinterpret_cast<T*>(&praw);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    if constexpr (SR) pb[k] = round_bf16_stochastic(th[k], off + i + k, seed);
                    else pb[k] = from_f<T>(th[k]);
                }
                __stcs(reinterpret_cast<uint2*>(params + i), praw);
            } else {
                __stcs(reinterpret_cast<float4*>(params + i), make_float4(th[0], th[1], th[2], th[3]));
            }
        } else {
            for (size_t j = i; j < n; j++) {
                float mm = mst[j], vv = vst[j];
                if constexpr (SR) {
                    const float th = adamw_one_sr(to_f(grads[j]), mm, vv, to_f(params[j]), lr, b1, b2, c1,
                                                  c2, eps, wd);
                    if constexpr (sizeof(T) == 2) params[j] = round_bf16_stochastic(th, off + j, seed);
                } else {
                    float th = master ? master[j] : to_f(params[j]);
                    th = adamw_one<T>(to_f(grads[j]) * inv_scale, mm, vv, th, lr, b1, b2, c1, c2, eps, wd);
                    if (master) master[j] = th;
                    params[j] = from_f<T>(th);
                }
                mst[j] = mm;
                vst[j] = vv;
            }
        }
    }
}

void launch_adamw(DType dt, void* params, float* master, const void* grads, float* m, float* v,
                  size_t n, float lr, float b1, float b2, float c1, float c2, float eps, float wd,
                  const float* hyper, cudaStream_t s, bool stochastic, uint32_t seed,
                  const LossScaler* scaler) {
    AdamRanges r = {};
    r.off[0] = 0;
    r.n[0] = n;
    launch_adamw_ranges(dt, params, master, grads, m, v, r, 1, lr, b1, b2, c1, c2, eps, wd, hyper, s,
                        stochastic, seed, scaler);
}

void launch_adamw_ranges(DType dt, void* params, float* master, const void* grads, float* m,
                         float* v, const AdamRanges& r, int nranges, float lr, float b1, float b2,
                         float c1, float c2, float eps, float wd, const float* hyper, cudaStream_t s,
                         bool stochastic, uint32_t seed, const LossScaler* scaler) {
    if (nranges <= 0) return;
    size_t nmax = 0;
    for (int i = 0; i < nranges; i++) nmax = r.n[i] > nmax ? r.n[i] : nmax;
    note_launch(1);
    const dim3 grid(grid_for((nmax + 3) / 4, 256, 8), (unsigned)nranges);
    if (dt == DT_BF16 && stochastic)
        launch_pdl(adamw_k<bf16, true>, grid, dim3(256), 0, s, (bf16*)params, (float*)nullptr,
                   (const bf16*)grads, m, v, r, lr, b1, b2, c1, c2, eps, wd, seed, hyper, scaler);
    else
        DISPATCH_E(dt, launch_pdl(adamw_k<E, false>, grid, dim3(256), 0, s, (E*)params, master,
                                  (const E*)grads, m, v, r, lr, b1, b2, c1, c2, eps, wd, seed, hyper,
                                  scaler));
}

// ------------------------------------------------------------------ loss scaling (fp16)
// found_inf = 1 if any gradient is inf or NaN (its exponent bits all ones)
template <typename T>
__global__ void nonfinite_k(const T* __restrict__ g, size_t n, LossScaler* __restrict__ sc) {
    pdl_enter();
    constexpr int VEC = Vec16<T>::N;
    bool bad = false;
    const size_t nv = n / VEC;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(g) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if constexpr (sizeof(T) == 2) {
                constexpr uint32_t E = std::is_same<T, f16>::value ? 0x7C007C00u : 0x7F807F80u;
                bad |= (w[k] & 0xFFFFu & E) == (E & 0xFFFFu) || (w[k] & 0xFFFF0000u & E) == (E & 0xFFFF0000u);
            } else {
                bad |= (w[k] & 0x7F800000u) == 0x7F800000u;
            }
        }
    }
    for (size_t j = nv * VEC + (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < n;
         j += (size_t)gridDim.x * blockDim.x)
        bad |= !isfinite(to_f(g[j]));
    if (__syncthreads_or(bad) && threadIdx.x == 0) sc->found_inf = 1;
}

void launch_nonfinite(DType dt, const void* grads, size_t n, LossScaler* sc, cudaStream_t s) {
    note_launch(1);
    const unsigned g = grid_for(n / 8 + 1, 256, 8);
    DISPATCH_E(dt, launch_pdl(nonfinite_k<E>, g, 256, 0, s, (const E*)grads, n, sc));
}

// after the update: an overflowed step halves the scale and restarts the count
// of good steps; growth_interval good steps in a row double it
__global__ void scaler_update_k(LossScaler* __restrict__ sc) {
    pdl_enter();
    if (sc->found_inf) {
        sc->scale *= 0.5f;
        sc->good_steps = 0;
        sc->skipped += 1;
    } else if (++sc->good_steps >= sc->growth_interval) {
        sc->scale *= 2.0f;
        sc->good_steps = 0;
    }
    sc->found_inf = 0;
}

void launch_scaler_update(LossScaler* sc, cudaStream_t s) {
    note_launch(1);
    launch_pdl(scaler_update_k, 1, 1, 0, s, sc);
}

__global__ void set_hyper_k(float* h, float lr, float b1, float b2, float c1, float c2, float eps,
                            float wd, uint32_t seed) {
    pdl_enter();
    h[0] = lr; h[1] = b1; h[2] = b2; h[3] = c1; h[4] = c2; h[5] = eps; h[6] = wd;
    h[7] = __uint_as_float(seed);
}

void launch_set_hyper(float* h, float lr, float b1, float b2, float c1, float c2, float eps, float wd,
                      uint32_t seed, cudaStream_t s) {
    note_launch(1);
    launch_pdl(set_hyper_k, 1, 1, 0, s, h, lr, b1, b2, c1, c2, eps, wd, seed);
}

// ------------------------------------------------------------------ utilities
__global__ void zero_k(int4* __restrict__ p, size_t n16, char* __restrict__ tail, size_t ntail) {
    pdl_enter();
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i < n16; i += (size_t)gridDim.x * blockDim.x) p[i] = make_int4(0, 0, 0, 0);
    if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = 0;
}

void launch_zero(void* p, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return;
    note_launch(1);
    // p is at least 256-byte aligned (every buffer comes from cudaMalloc offsets of 256)
    size_t n16 = bytes / 16, ntail = bytes % 16;
    launch_pdl(zero_k, grid_for(n16 ? n16 : 1, 256, 8), 256, 0, s, (int4*)p, n16, (char*)p + n16 * 16, ntail);
}

// counter-based normal generator for the initial weights: SplitMix64 output
// function over (seed, stream, index), Box-Muller on two 32-bit halves.
DEVI unsigned long long splitmix64(unsigned long long z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <typename T>
__global__ void init_normal_k(T* __restrict__ p, size_t n, float stddev, unsigned long long seed,
                              unsigned long long stream_id) {
    const unsigned long long base = seed * 0x9E3779B97F4A7C15ull + (stream_id << 40);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        unsigned long long z = splitmix64(base + i);
        float u1 = ((float)(unsigned)(z >> 40) + 0.5f) * (1.0f / 16777216.0f);
        float u2 = ((float)(unsigned)((z >> 8) & 0xFFFFFFu) + 0.5f) * (1.0f / 16777216.0f);
        float r = sqrtf(-2.0f * logf(u1));
        p[i] = from_f<T>(stddev * r * cospif(2.0f * u2));
    }
}

template <typename T>
__global__ void fill_k(T* __restrict__ p, size_t n, float value) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = from_f<T>(value);
}

void launch_init_normal(DType dt, void* p, size_t n, float stddev, unsigned long long seed,
                        unsigned long long stream_id, cudaStream_t s) {
    note_launch(1);
    unsigned g = grid_for(n, 256, 16);
    DISPATCH_E(dt, init_normal_k<E><<<g, 256, 0, s>>>((E*)p, n, stddev, seed, stream_id));
}

void launch_fill(DType dt, void* p, size_t n, float value, cudaStream_t s) {
    note_launch(1);
    unsigned g = grid_for(n, 256, 16);
    DISPATCH_E(dt, fill_k<E><<<g, 256, 0, s>>>((E*)p, n, value));
}

template <typename T>
__global__ void to_f32_k(float* __restrict__ dst, const T* __restrict__ src, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = to_f(src[i]);
}
template <typename T>
__global__ void from_f32_k(T* __restrict__ dst, const float* __restrict__ src, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = from_f<T>(src[i]);
}

void launch_to_f32(DType dt, float* dst, const void* src, size_t n, cudaStream_t s) {
    note_launch(1);
    unsigned g = grid_for(n, 256, 16);
    DISPATCH_E(dt, to_f32_k<E><<<g, 256, 0, s>>>(dst, (const E*)src, n));
}
void launch_from_f32(DType dt, void* dst, const float* src, size_t n, cudaStream_t s) {
    note_launch(1);
    unsigned g = grid_for(n, 256, 16);
    DISPATCH_E(dt, from_f32_k<E><<<g, 256, 0, s>>>((E*)dst, src, n));
}

// ------------------------------------------------------------------ fused operator, pass 2
// Each row of y holds gelu(x W^T + b); part[row][t] = (max, sum exp(y - max)) of
// column tile t. Combine the tile partials, then y <- exp(y - max) / sum in place.
__global__ void __launch_bounds__(256) softmax_finish_k(float* __restrict__ y,
                                                        const float2* __restrict__ part, int N,
                                                        int tiles) {
    __shared__ float s_m, s_inv;
    const int row = blockIdx.x;
    if (threadIdx.x < 32) {
        float m = -INFINITY;
        for (int t = threadIdx.x; t < tiles; t += 32) m = fmaxf(m, part[(size_t)row * tiles + t].x);
        m = warp_max(m);
        float s = 0.f;
        for (int t = threadIdx.x; t < tiles; t += 32) {
            float2 p = part[(size_t)row * tiles + t];
            s += p.y * expf(p.x - m);
        }
        s = warp_sum(s);
        if (threadIdx.x == 0) {
            s_m = m;
            s_inv = 1.f / s;
        }
    }
    __syncthreads();
    const float m = s_m, inv = s_inv;
    float* yr = y + (size_t)row * N;
    const int nv = N / 4;
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        float4 v = reinterpret_cast<float4*>(yr)[i];
        v.x = expf(v.x - m) * inv;
        v.y = expf(v.y - m) * inv;
        v.z = expf(v.z - m) * inv;
        v.w = expf(v.w - m) * inv;
        __stcs(reinterpret_cast<float4*>(yr) + i, v);
    }
}

void launch_softmax_finish(float* y, const float* part, int M, int N, int tiles, cudaStream_t s) {
    note_launch(1);
    softmax_finish_k<<<M, 256, 0, s>>>(y, (const float2*)part, N, tiles);
}

// the bounded-wait limit of this translation unit's kernels (0: the default)
int set_wait_limit_kernels(unsigned long long ns) {
    return tc::set_tu_wait_limit(ns ? ns : tc::WAIT_LIMIT_NS) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace gk
