// internal.h -- launchers shared between the translation units of libgpt2.so.
// Host-side declarations only; no torch types anywhere.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

// device-side error bits, read by the host after a synchronisation
#define DEVERR_TIMEOUT 1u
#define DEVERR_TOKEN 2u

namespace gk {

// element type of parameters/activations
enum DType { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
inline size_t dtype_size(DType dt) { return dt == DT_F32 ? 4 : 2; }
// elements in a 16-byte vector
inline int dtype_vec(DType dt) { return dt == DT_F32 ? 4 : 8; }

// GEMM epilogues, applied to the fp32 accumulator acc[m][n]:
//  EPI_STORE     D = acc (+ bias[n])
//  EPI_GELU      D = acc + bias[n] (pre-activation), D2 = gelu(D)
//  EPI_RESID     D = acc + bias[n] + aux[m][n]           (residual add)
//  EPI_GELU_BWD  D = acc * gelu'(aux[m][n])                (GELU backward)
//  EPI_ACCUM     D = D + acc                               (parameter-gradient +=)
enum Epi { EPI_STORE = 0, EPI_GELU = 1, EPI_RESID = 2, EPI_GELU_BWD = 3, EPI_ACCUM = 4,
           EPI_SPLITK = 6 };  // internal to gemm_tc: fp32 partial sums of one K range

// D[M,N] = A[M,K] . B[N,K]^T with operands given by their storage order:
//  a_kmajor: A(m,k) = A[m*lda + k], else A(m,k) = A[k*lda + m]
//  b_kmajor: B(n,k) = B[n*ldb + k], else B(n,k) = B[k*ldb + n]
//  D(m,n) = D[m*ldd + n]; aux(m,n) = aux[m*ldaux + n]
struct GemmParams {
    const void* A; long long lda; int a_kmajor;
    const void* B; long long ldb; int b_kmajor;
    void* D; long long ldd;
    const void* bias;
    const void* aux; long long ldaux;
    void* D2;
    float* ws; size_t ws_floats;  // optional fp32 scratch: lets EPI_ACCUM split K (0 = never)
    // optional (EPI_GELU_BWD on the tensor cores only): the column sums of the
    // rounded output over each 32-row group, cs[(row / 32) * ldcs + col]
    float* cs; long long ldcs;
    int M, N, K;
    int epi;
};

// fp32 split-K scratch the model gives its GEMMs: four (4C x C) slices
inline size_t gemm_ws_floats(int C) { return (size_t)16 * C * C; }
// the main stream's split-K scratch: three K ranges of a (B*T) x C product
inline size_t gemm_ws_main_floats(size_t BT, int C) { return (size_t)3 * BT * C; }

// SIMT (FP32 FMA) GEMM, dtype = element type of A, B, D, bias, aux.
int gemm_simt(const GemmParams& p, DType dt, cudaStream_t s);

// tcgen05 tensor-core GEMM: DT_BF16 -> kind::f16 (bf16 in, fp32 accumulate);
// DT_F32 -> kind::tf32. err: device error word (bounded waits).
// Returns 0, or a negative GPT2_ERR_* code for unsupported shapes/alignment.
int gemm_tc(const GemmParams& p, DType dt, cudaStream_t s, unsigned int* err);

// ---- memory-bound kernels (kernels.cu) ----
void launch_copy_tokens(const int* src, int* dst, int n, int V, unsigned int* err, cudaStream_t s);
void launch_encoder_forward(DType dt, void* out, const int* tok, const void* wte, const void* wpe,
                            int B, int T, int C, cudaStream_t s);
// deterministic: dwpe[t] += sum_b dout[b,t]; dwte[tok] += sum over positions in position order
void launch_encoder_backward(DType dt, void* dwte, void* dwpe, const void* dout, const int* tok,
                             int B, int T, int C, int Vp, int* ws_counts, int* ws_offsets,
                             int* ws_cursor, int* ws_order, int* ws_sorted, cudaStream_t s);
void launch_layernorm_forward(DType dt, void* out, float* mean, float* rstd, const void* inp,
                              const void* w, const void* b, int N, int C, cudaStream_t s);
// dinp (+= if accumulate else =), dw += sum, db += sum (two-stage, deterministic).
// ws: fp32 scratch of at least layernorm_backward_ws_floats(C) floats.
// err: device error word of the bounded waits
void launch_layernorm_backward(DType dt, void* dinp, void* dw, void* db, const void* dout,
                               const void* inp, const void* w, const float* mean,
                               const float* rstd, int N, int C, int accumulate, float* ws,
                               unsigned int* err, cudaStream_t s);
size_t layernorm_backward_ws_floats(int C);
// dbias[n] += sum_m dout[m][n] (two-stage, deterministic)
void launch_colsum_accum(DType dt, void* dbias, const void* dout, int M, int N, float* ws,
                         cudaStream_t s);
size_t colsum_ws_floats(int N);

// ---- partial sums reduced once per backward ----
// dst[c] += sum over p < P (in order) of part[p * pstride + c], c < width;
// dst has the model's element type
struct PartialDesc {
    const float* part;
    long long pstride;
    int P, width;
    void* dst;
};
// LayerNorm backward that leaves its parameter sums as partial rows
// part[p][G*C] = [dw | db | colsum of the written dinp rows (G = 3)];
// returns the row count P. The column sums are fused only where
// layernorm_backward_fuses_colsum(dt, C); otherwise G = 2.
bool layernorm_backward_fuses_colsum(DType dt, int C);
int layernorm_backward_part_rows(DType dt, int N, int C);
int launch_layernorm_backward_part(DType dt, void* dinp, float* part, const void* dout,
                                   const void* inp, const void* w, const float* mean,
                                   const float* rstd, int N, int C, int accumulate, int with_colsum,
                                   unsigned int* err, cudaStream_t s);
// column sums of dout (M, N) as partial rows part[R][N]; returns R
int colsum_part_rows(int M);
int launch_colsum_part(DType dt, float* part, const void* dout, int M, int N, cudaStream_t s);
// one launch over a device table of descriptors
void launch_reduce_partials_multi(DType dt, const PartialDesc* d_desc, int ndesc, int maxwidth,
                                  cudaStream_t s);
// logits (BT, Vp) -> dlogits in place; losses[BT] fp32. dloss_scale: NULL, or
// a device float the seed dloss is multiplied by (the loss scale of fp16 training)
void launch_classifier(DType dt, void* logits, float* losses, const int* targets, int BT, int V,
                       int Vp, float dloss, cudaStream_t s, const float* dloss_scale = nullptr);
void launch_mean(const float* x, int n, float* out, cudaStream_t s);
// probs (rows, Vp) fp32 = softmax over the first V columns of logits (rows, Vp); 0 on the padding
void launch_probs(DType dt, float* probs, const void* logits, int rows, int V, int Vp, cudaStream_t s);
// per row r: the index sampled from softmax(logits[r*row_stride + 0 .. V)) with coins[r]
// (llm.c sample_softmax), written to out[r * out_stride]
void launch_sample(DType dt, const void* logits, long long row_stride, int rows, int V, const float* coins,
                   int* out, long long out_stride, cudaStream_t s);
// ranges of the flat parameter buffers one AdamW launch updates (offsets and
// counts are multiples of 4)
struct AdamRanges {
    size_t off[8], n[8];
};
// dynamic loss scaling of fp16 training, in device memory (graph replays keep
// it current): the backward is seeded with scale / (k B T); a step whose
// gradients hold an inf or NaN is skipped and halves the scale; growth_interval
// good steps in a row double it
struct LossScaler {
    float scale;
    int good_steps;
    int found_inf;
    int growth_interval;
    long long skipped;
};
// found_inf |= any gradient is inf or NaN
void launch_nonfinite(DType dt, const void* grads, size_t n, LossScaler* sc, cudaStream_t s);
// the scale's update after an AdamW launch (which skipped the step on found_inf)
void launch_scaler_update(LossScaler* sc, cudaStream_t s);
void launch_adamw_ranges(DType dt, void* params, float* master, const void* grads, float* m,
                         float* v, const AdamRanges& r, int nranges, float lr, float b1, float b2,
                         float c1, float c2, float eps, float wd, const float* hyper, cudaStream_t s,
                         bool stochastic = false, uint32_t seed = 0, const LossScaler* scaler = nullptr);
// hyper: NULL, or device floats {lr, b1, b2, c1, c2, eps, wd, seed bits} that
// replace the by-value ones (a CUDA graph replays the launch with new values
// there). stochastic (bf16 only): no master copy; the fp32 update is rounded
// to the bf16 parameter stochastically with this step's seed.
void launch_adamw(DType dt, void* params, float* master, const void* grads, float* m, float* v,
                  size_t n, float lr, float b1, float b2, float c1, float c2, float eps, float wd,
                  const float* hyper, cudaStream_t s, bool stochastic = false, uint32_t seed = 0,
                  const LossScaler* scaler = nullptr);
// writes {lr, b1, b2, c1, c2, eps, wd, seed bits} to h with a one-thread kernel
void launch_set_hyper(float* h, float lr, float b1, float b2, float c1, float c2, float eps, float wd,
                      uint32_t seed, cudaStream_t s);
void launch_zero(void* p, size_t bytes, cudaStream_t s);
void launch_init_normal(DType dt, void* p, size_t n, float stddev, unsigned long long seed,
                        unsigned long long stream_id, cudaStream_t s);
void launch_fill(DType dt, void* p, size_t n, float value, cudaStream_t s);
void launch_to_f32(DType dt, float* dst, const void* src, size_t n, cudaStream_t s);
void launch_from_f32(DType dt, void* dst, const float* src, size_t n, cudaStream_t s);
// out = softmax over each row of a (M,N) fp32 tile-partial GELU output (fused operator pass 2)
void launch_softmax_finish(float* y, const float* part, int M, int N, int tiles, cudaStream_t s);

// ---- fused operator (fused_tc.cu) ----
// y = gelu(x W^T + b) (fp32 x (M,K), W (N,K), b (N), y (M,N), all 16-byte
// aligned, K % 4 == 0 == N % 4) with the bf16 hi/lo split of x and W done in
// the kernel; part[row * part_ld + t] = (max, sum exp(y - max)) over the row's
// column tile t of tile_n (256 or 224) columns (float2; part_ld >= the tile
// count). err: device error word of the bounded waits.
int launch_fused_split_gemm(const float* x, const float* W, const float* b, float* y, float* part,
                            int part_ld, int M, int K, int N, int tile_n, cudaStream_t s, unsigned int* err);
// the tile width the fused product takes for an (M, N) output: 224 where it
// needs fewer rounds of the CTA pairs and M * ceil(N / 224) <= max_partials, else 256
int fused_split_tile_n(int M, int N, long long max_partials);

// ---- attention (attention.cu) ----
// qkv (B,T,3C) -> out (B,T,C), lse (B,NH,T) fp32 natural-log sum of exp of the scaled scores
// returns 0 or a GPT2_ERR_* code; err: device error word of the bounded waits
int launch_attention_forward(DType dt, int tensor_cores, void* out, float* lse, const void* qkv,
                             int B, int T, int C, int NH, cudaStream_t s, unsigned int* err);
// tcgen05 flash forward (bf16 or fp16, head size 64)
int launch_flash_forward_tc(DType dt, void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
                            cudaStream_t s, unsigned int* err);
// dqkv (B,T,3C) written; D scratch (B,NH,T) fp32; returns 0 or a GPT2_ERR_* code
int launch_attention_backward(DType dt, int tensor_cores, void* dqkv, const void* dout,
                              const void* qkv, const void* out, const float* lse, float* D,
                              int B, int T, int C, int NH, cudaStream_t s, unsigned int* err);
// tcgen05 flash backward (bf16 or fp16, head size 64): D = rowsum(dO * O), then dQ, dK, dV
int launch_flash_backward_tc(DType dt, void* dqkv, const void* dout, const void* qkv, const void* out,
                             const float* lse, float* D, int B, int T, int C, int NH, cudaStream_t s,
                             unsigned int* err);

int num_sms();

// the limit of the bounded in-kernel waits of each translation unit's kernels
// (ns; 0 restores the default of 2 s); drain waits after an abort keep 2 s
int set_wait_limit_gemm(unsigned long long ns);
int set_wait_limit_attn_fwd(unsigned long long ns);
int set_wait_limit_attn_bwd(unsigned long long ns);
int set_wait_limit_kernels(unsigned long long ns);
int set_wait_limit_fused(unsigned long long ns);

// Programmatic dependent launch for the step's kernels (GPT2_PDL=0 turns it
// off): the kernel may be scheduled while the previous one drains, and waits
// for it in pdl_enter().
bool pdl_enabled();
// Scheduling priority of the launches issued from now on by this thread (0:
// the stream's own). The backward raises it for its main-stream chain, so
// that SMs freed by a finishing kernel go to the critical path first.
int launch_priority();
void set_launch_priority(int priority);
// the attributes every launch of the library carries: programmatic stream
// serialization (unless turned off) and the current priority; returns the count
inline unsigned launch_attrs(cudaLaunchAttribute* attr) {
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        n++;
    }
    if (const int pr = launch_priority()) {
        attr[n].id = cudaLaunchAttributePriority;
        attr[n].val.priority = pr;
        n++;
    }
    return n;
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = launch_attrs(attr);
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
// records the library's last error (text and GPT2_ERR_* code); returns code
int set_error(int code, const char* fmt, ...);
// number of errors recorded so far (tells whether a callee described its failure)
unsigned long long error_serial();
// host-side count of kernel launches made by this library (for benchmark reporting)
void note_launch(int n);
long long launch_count();

}  // namespace gk
