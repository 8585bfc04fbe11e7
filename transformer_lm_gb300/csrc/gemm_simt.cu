// gemm_simt.cu -- SIMT FP32-FMA GEMM with the fused epilogues.
//
// The fp32 training path with the tensor cores off (llm.c "train_gpt2.cu",
// main: "-f 0" disables TF32; train_gpt2_fp32.cu runs plain fp32 cuBLAS)
// computes every matmul here: 64x64 output tile per 256-thread block, 4x4
// outputs per thread, K staged through shared memory 16 at a time. Operands
// may be K-major or MN-major (the forward, dX and dW products of
// matmul_forward / matmul_backward all map onto D = A . B^T).
#include "common.cuh"
#include "internal.h"

#include "gpt2.h"

namespace gk {

template <typename T>
DEVI void epi_scalar(const GemmParams& p, int m, int n, float acc) {
    T* D = (T*)p.D;
    const T* bias = (const T*)p.bias;
    const T* aux = (const T*)p.aux;
    const size_t idx = (size_t)m * p.ldd + n;
    switch (p.epi) {
        case EPI_STORE:
            if (bias) acc += to_f(bias[n]);
            D[idx] = from_f<T>(acc);
            break;
        case EPI_GELU: {
            if (bias) acc += to_f(bias[n]);
            T pre = from_f<T>(acc);
            D[idx] = pre;
            ((T*)p.D2)[idx] = from_f<T>(gelu_fwd(to_f(pre)));
            break;
        }
        case EPI_RESID:
            if (bias) acc += to_f(bias[n]);
            D[idx] = from_f<T>(acc + to_f(aux[(size_t)m * p.ldaux + n]));
            break;
        case EPI_GELU_BWD:
            D[idx] = from_f<T>(acc * gelu_grad(to_f(aux[(size_t)m * p.ldaux + n])));
            break;
        case EPI_ACCUM:
            D[idx] = from_f<T>(to_f(D[idx]) + acc);
            break;
        default:
            break;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_k(const GemmParams p) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const T* A = (const T*)p.A;
    const T* B = (const T*)p.B;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < p.K; k0 += 16) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int e = tid + r * 256;
            int mm, kk;
            if (p.a_kmajor) { mm = e / 16; kk = e % 16; } else { kk = e / 64; mm = e % 64; }
            const int gm = m0 + mm, gkk = k0 + kk;
            float v = 0.f;
            if (gm < p.M && gkk < p.K)
                v = to_f(p.a_kmajor ? A[(size_t)gm * p.lda + gkk] : A[(size_t)gkk * p.lda + gm]);
            As[kk][mm] = v;
            int nn;
            if (p.b_kmajor) { nn = e / 16; kk = e % 16; } else { kk = e / 64; nn = e % 64; }
            const int gn = n0 + nn, gk2 = k0 + kk;
            float w = 0.f;
            if (gn < p.N && gk2 < p.K)
                w = to_f(p.b_kmajor ? B[(size_t)gn * p.ldb + gk2] : B[(size_t)gk2 * p.ldb + gn]);
            Bs[kk][nn] = w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int m = m0 + ty * 4 + i;
        if (m >= p.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int n = n0 + tx * 4 + j;
            if (n < p.N) epi_scalar<T>(p, m, n, acc[i][j]);
        }
    }
}

int gemm_simt(const GemmParams& p, DType dt, cudaStream_t s) {
    if (p.M <= 0 || p.N <= 0 || p.K <= 0) return GPT2_ERR_ARG;
    if (p.cs) return GPT2_ERR_CONFIG;  // column sums come with the tensor-core epilogue only
    dim3 grid((p.N + 63) / 64, (p.M + 63) / 64);
    if (grid.y > 65535) return GPT2_ERR_CONFIG;
    note_launch(1);
    if (dt == DT_BF16) gemm_simt_k<bf16><<<grid, 256, 0, s>>>(p);
    else if (dt == DT_F16) gemm_simt_k<f16><<<grid, 256, 0, s>>>(p);
    else gemm_simt_k<float><<<grid, 256, 0, s>>>(p);
    return GPT2_OK;
}

}  // namespace gk
