// ops.cu -- stand-alone operator entry points of libgpt2.so (device pointers).
//
//  * fused_linear_bias_gelu_softmax: y = softmax_row(gelu_tanh(x W^T + b))
//    (POPCORNBENCH "fused Linear + GELU + Softmax" problem: nn.Linear, GELU,
//    softmax over dim 1). Pass 1 is the tcgen05 TF32 GEMM whose epilogue adds
//    the bias, applies GELU, stores the row tile and records, per row and
//    256-column tile, (max, sum exp(v - max)). Pass 2 merges the tile
//    partials of each row and rewrites the row as exp(v - max) / sum.
//  * gpt2_gemm / gpt2_attention_forward / gpt2_attention_backward: the
//    training step's kernels exposed one at a time.
#include "gpt2.h"
#include "common.cuh"
#include "internal.h"

#include <cuda_runtime.h>

#include <mutex>

using namespace gk;

namespace {

constexpr int kMaxDevices = 64;
std::mutex ops_mu;
unsigned int* dev_err[kMaxDevices] = {nullptr};
float* dev_part[kMaxDevices] = {nullptr};
size_t dev_part_bytes[kMaxDevices] = {0};

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return GPT2_ERR_CUDA;
    return GPT2_OK;
}

// device error word shared by the stand-alone entry points of this device
unsigned int* err_word(int dev) {
    std::lock_guard<std::mutex> lk(ops_mu);
    if (!dev_err[dev]) {
        unsigned int* p = nullptr;
        if (cudaMalloc(&p, 256) != cudaSuccess) return nullptr;
        if (cudaMemset(p, 0, 256) != cudaSuccess) return nullptr;
        dev_err[dev] = p;
    }
    return dev_err[dev];
}

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int fused_linear_bias_gelu_softmax(const float* x, const float* W, const float* b, float* out,
                                   int M, int K, int N, void* stream) {
    if (!x || !W || !b || !out) return GPT2_ERR_ARG;
    if (M < 1 || K < 1 || N < 1) return GPT2_ERR_ARG;
    if (!al16(x) || !al16(W) || !al16(b) || !al16(out) || K % 4 || N % 4) return GPT2_ERR_ALIGN;
    int dev;
    if (current_device(&dev) != GPT2_OK) return GPT2_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (!err) return GPT2_ERR_NOMEM;
    const int tile_n = gemm_tc_part_tile_n();
    const int tiles = (N + tile_n - 1) / tile_n;
    const size_t need = (size_t)M * tiles * 2 * sizeof(float);
    float* part;
    {
        std::lock_guard<std::mutex> lk(ops_mu);
        if (dev_part_bytes[dev] < need) {
            if (dev_part[dev]) cudaFree(dev_part[dev]);
            dev_part[dev] = nullptr;
            dev_part_bytes[dev] = 0;
            if (cudaMalloc(&dev_part[dev], need) != cudaSuccess) return GPT2_ERR_NOMEM;
            dev_part_bytes[dev] = need;
        }
        part = dev_part[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    GemmParams p = {};
    p.A = x; p.lda = K; p.a_kmajor = 1;
    p.B = W; p.ldb = K; p.b_kmajor = 1;
    p.D = out; p.ldd = N; p.bias = b;
    p.part = part; p.part_ld = tiles;
    p.M = M; p.N = N; p.K = K; p.epi = EPI_GELU_PART;
    int rc = gemm_tc(p, DT_F32, s, err);
    if (rc != GPT2_OK) return rc;
    launch_softmax_finish(out, part, M, N, tiles, s);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int gpt2_gemm(int dtype, int tensor_cores, int epilogue, const void* A, long long lda, int a_kmajor,
              const void* B, long long ldb, int b_kmajor, void* D, long long ldd, const void* bias,
              const void* aux, long long ldaux, void* D2, int M, int N, int K, void* stream) {
    if (!A || !B || !D) return GPT2_ERR_ARG;
    if (dtype != GPT2_FP32 && dtype != GPT2_BF16) return GPT2_ERR_CONFIG;
    if (epilogue < EPI_STORE || epilogue > EPI_ACCUM) return GPT2_ERR_ARG;
    if ((epilogue == EPI_RESID || epilogue == EPI_GELU_BWD) && !aux) return GPT2_ERR_ARG;
    if (epilogue == EPI_GELU && !D2) return GPT2_ERR_ARG;
    GemmParams p = {};
    p.A = A; p.lda = lda; p.a_kmajor = a_kmajor ? 1 : 0;
    p.B = B; p.ldb = ldb; p.b_kmajor = b_kmajor ? 1 : 0;
    p.D = D; p.ldd = ldd; p.bias = bias; p.aux = aux; p.ldaux = ldaux; p.D2 = D2;
    p.M = M; p.N = N; p.K = K; p.epi = epilogue;
    const DType dt = dtype == GPT2_BF16 ? DT_BF16 : DT_F32;
    int rc;
    if (tensor_cores) {
        int dev;
        if (current_device(&dev) != GPT2_OK) return GPT2_ERR_CUDA;
        unsigned int* err = err_word(dev);
        if (!err) return GPT2_ERR_NOMEM;
        rc = gemm_tc(p, dt, (cudaStream_t)stream, err);
    } else {
        rc = gemm_simt(p, dt, (cudaStream_t)stream);
    }
    if (rc != GPT2_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int gpt2_attention_forward(int dtype, int tensor_cores, const void* qkv, void* out, float* lse,
                           int B, int T, int C, int NH, void* stream) {
    if (!qkv || !out || !lse) return GPT2_ERR_ARG;
    if (B < 1 || T < 1 || NH < 1 || C % NH) return GPT2_ERR_ARG;
    const int HS = C / NH;
    if (HS != 16 && HS != 32 && HS != 64 && HS != 128) return GPT2_ERR_CONFIG;
    if (dtype != GPT2_FP32 && dtype != GPT2_BF16) return GPT2_ERR_CONFIG;
    launch_attention_forward(dtype == GPT2_BF16 ? DT_BF16 : DT_F32, tensor_cores, out, lse, qkv, B,
                             T, C, NH, (cudaStream_t)stream);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int gpt2_attention_backward(int dtype, int tensor_cores, const void* dout, const void* qkv,
                            const void* out, const float* lse, void* dqkv, float* scratch_D, int B,
                            int T, int C, int NH, void* stream) {
    if (!dout || !qkv || !out || !lse || !dqkv || !scratch_D) return GPT2_ERR_ARG;
    if (B < 1 || T < 1 || NH < 1 || C % NH) return GPT2_ERR_ARG;
    const int HS = C / NH;
    if (HS != 16 && HS != 32 && HS != 64 && HS != 128) return GPT2_ERR_CONFIG;
    if (dtype != GPT2_FP32 && dtype != GPT2_BF16) return GPT2_ERR_CONFIG;
    launch_attention_backward(dtype == GPT2_BF16 ? DT_BF16 : DT_F32, tensor_cores, dqkv, dout, qkv,
                              out, lse, scratch_D, B, T, C, NH, (cudaStream_t)stream);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

int gpt2_device_status(void) {
    int dev;
    if (current_device(&dev) != GPT2_OK) return GPT2_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (!err) return GPT2_ERR_NOMEM;
    unsigned int h = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return GPT2_ERR_CUDA;
    if (cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return GPT2_ERR_CUDA;
    if (h) {
        cudaMemset(err, 0, 4);
        if (h & DEVERR_TIMEOUT) return GPT2_ERR_DEVICE_TIMEOUT;
    }
    return GPT2_OK;
}

}  // extern "C"
