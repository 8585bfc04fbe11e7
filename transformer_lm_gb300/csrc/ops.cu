// ops.cu -- stand-alone operator entry points of libgpt2.so (device pointers).
//
//  * fused_linear_bias_gelu_softmax: y = softmax_row(gelu_tanh(x W^T + b))
//    (POPCORNBENCH "fused Linear + GELU + Softmax" problem: nn.Linear, GELU,
//    softmax over dim 1). The product kernel (fused_tc.cu) splits x and W into
//    bf16 halves (hi, lo) in shared memory as their fp32 tiles arrive and runs
//    x W^T as hi.hi + hi.lo + lo.hi on the bf16 tensor cores (about 2^-16
//    relative per product, fp32 accumulation); its epilogue adds the bias,
//    applies GELU, stores the row tile and records, per row and column tile
//    (256 or 224 columns), (max, sum exp(v - max)). The last pass merges the tile partials of
//    each row and rewrites the row as exp(v - max) / sum. The allocation-free
//    variant runs the same two kernels with its partials in a static array.
//  * gpt2_gemm / gpt2_attention_forward / gpt2_attention_backward: the
//    training step's kernels exposed one at a time.
#include "gpt2.h"
#include "common.cuh"
#include "internal.h"

#include <cuda_runtime.h>

#include <mutex>

using namespace gk;

// partials the fused operator's 224-column tiles may need at most: the
// allocation-free entry point's static array (131072 float2), so that both
// entry points choose the same tiles for every shape either accepts
#define FUSED_NARROW_MAX_PARTIALS (1LL << 17)

namespace {

constexpr int kMaxDevices = 64;
std::mutex ops_mu;
unsigned int* dev_err[kMaxDevices] = {nullptr};
float* dev_part[kMaxDevices] = {nullptr};
size_t dev_part_bytes[kMaxDevices] = {0};

// status of the launches just issued, with CUDA's message kept for gpt2_last_error
int launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GPT2_OK : set_error(GPT2_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
}

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

bool known_dtype(int dtype) { return dtype == GPT2_FP32 || dtype == GPT2_BF16 || dtype == GPT2_FP16; }
DType to_dt(int dtype) { return dtype == GPT2_BF16 ? DT_BF16 : dtype == GPT2_FP16 ? DT_F16 : DT_F32; }

const char* code_text(int rc) {
    switch (rc) {
        case GPT2_ERR_CONFIG: return "unsupported dtype, epilogue, head size or tile configuration";
        case GPT2_ERR_ALIGN: return "a pointer, leading dimension or size is not aligned as required";
        case GPT2_ERR_CUDA: return "a CUDA call failed";
        case GPT2_ERR_NOMEM: return "a device allocation failed";
        case GPT2_ERR_ARG: return "NULL pointer or size out of range";
        case GPT2_ERR_DEVICE_TIMEOUT:
            return "a bounded in-kernel wait expired; the results of the calls since the last check are invalid";
        default: return "failed";
    }
}

// Every entry point below returns through one of these, so that each failed
// call leaves a description in gpt2_last_error: a callee's own message
// stands; an error no callee described gets its code's text, prefixed with
// the entry point's name.
struct ErrScope {
    const char* op;
    unsigned long long serial;
    explicit ErrScope(const char* name) : op(name), serial(error_serial()) {}
    int operator()(int rc) const {
        if (rc != GPT2_OK && error_serial() == serial) set_error(rc, "%s: %s", op, code_text(rc));
        return rc;
    }
};

}  // namespace

static int noalloc_err_of(int dev, unsigned int* bits);

extern "C" {

int fused_linear_bias_gelu_softmax(const float* x, const float* W, const float* b, float* out,
                                   int M, int K, int N, void* stream) {
    const ErrScope ret("fused_linear_bias_gelu_softmax");
    if (!x || !W || !b || !out) return ret(GPT2_ERR_ARG);
    if (M < 1 || K < 1 || N < 1) return ret(GPT2_ERR_ARG);
    if (!al16(x) || !al16(W) || !al16(b) || !al16(out) || K % 4 || N % 4) return ret(GPT2_ERR_ALIGN);
    int dev;
    if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    unsigned int* err = err_word(dev);
    if (!err) return ret(GPT2_ERR_NOMEM);
    // the same tile choice as the allocation-free entry point (whose static
    // partials bound the narrower tiles), so the two give identical results
    const int tile_n = fused_split_tile_n(M, N, FUSED_NARROW_MAX_PARTIALS);
    const int tiles = (int)(((long long)N + tile_n - 1) / tile_n);
    // scratch: the row-tile softmax partials
    const size_t need = ((size_t)M * tiles * 2 * sizeof(float) + 255) / 256 * 256;
    char* scratch;
    {
        std::lock_guard<std::mutex> lk(ops_mu);
        if (dev_part_bytes[dev] < need) {
            if (dev_part[dev]) cudaFree(dev_part[dev]);
            dev_part[dev] = nullptr;
            dev_part_bytes[dev] = 0;
            if (cudaMalloc(&dev_part[dev], need) != cudaSuccess) return ret(GPT2_ERR_NOMEM);
            dev_part_bytes[dev] = need;
        }
        scratch = (char*)dev_part[dev];
    }
    float* part = (float*)scratch;
    cudaStream_t s = (cudaStream_t)stream;
    const int rc = launch_fused_split_gemm(x, W, b, out, part, tiles, M, K, N, tile_n, s, err);
    if (rc != GPT2_OK) return ret(rc);
    launch_softmax_finish(out, part, M, N, tiles, s);
    return ret(launch_status());
}

int gpt2_gemm(int dtype, int tensor_cores, int epilogue, const void* A, long long lda, int a_kmajor,
              const void* B, long long ldb, int b_kmajor, void* D, long long ldd, const void* bias,
              const void* aux, long long ldaux, void* D2, int M, int N, int K, float* ws,
              size_t ws_floats, void* stream) {
    const ErrScope ret("gpt2_gemm");
    if (!A || !B || !D) return ret(GPT2_ERR_ARG);
    if (!known_dtype(dtype)) return ret(GPT2_ERR_CONFIG);
    if (epilogue < EPI_STORE || epilogue > EPI_ACCUM) return ret(GPT2_ERR_ARG);
    if ((epilogue == EPI_RESID || epilogue == EPI_GELU_BWD) && !aux) return ret(GPT2_ERR_ARG);
    if (epilogue == EPI_GELU && !D2) return ret(GPT2_ERR_ARG);
    GemmParams p = {};
    p.A = A; p.lda = lda; p.a_kmajor = a_kmajor ? 1 : 0;
    p.B = B; p.ldb = ldb; p.b_kmajor = b_kmajor ? 1 : 0;
    p.D = D; p.ldd = ldd; p.bias = bias; p.aux = aux; p.ldaux = ldaux; p.D2 = D2;
    p.M = M; p.N = N; p.K = K; p.epi = epilogue;
    if (ws && ((uintptr_t)ws & 15u)) return ret(GPT2_ERR_ALIGN);
    p.ws = ws; p.ws_floats = ws ? ws_floats : 0;
    const DType dt = to_dt(dtype);
    int rc;
    if (tensor_cores) {
        int dev;
        if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
        unsigned int* err = err_word(dev);
        if (!err) return ret(GPT2_ERR_NOMEM);
        rc = gemm_tc(p, dt, (cudaStream_t)stream, err);
    } else {
        rc = gemm_simt(p, dt, (cudaStream_t)stream);
    }
    if (rc != GPT2_OK) return ret(rc);
    return ret(launch_status());
}

int gpt2_attention_forward(int dtype, int tensor_cores, const void* qkv, void* out, float* lse,
                           int B, int T, int C, int NH, void* stream) {
    const ErrScope ret("gpt2_attention_forward");
    if (!qkv || !out || !lse) return ret(GPT2_ERR_ARG);
    if (B < 1 || T < 1 || NH < 1 || C % NH) return ret(GPT2_ERR_ARG);
    const int HS = C / NH;
    if (HS != 16 && HS != 32 && HS != 64 && HS != 128) return ret(GPT2_ERR_CONFIG);
    if (!known_dtype(dtype)) return ret(GPT2_ERR_CONFIG);
    int dev;
    if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    unsigned int* err = err_word(dev);
    if (!err) return ret(GPT2_ERR_NOMEM);
    const int rc = launch_attention_forward(to_dt(dtype), tensor_cores, out,
                                            lse, qkv, B, T, C, NH, (cudaStream_t)stream, err);
    if (rc != GPT2_OK) return ret(rc);
    return ret(launch_status());
}

int gpt2_attention_backward(int dtype, int tensor_cores, const void* dout, const void* qkv,
                            const void* out, const float* lse, void* dqkv, float* scratch_D, int B,
                            int T, int C, int NH, void* stream) {
    const ErrScope ret("gpt2_attention_backward");
    if (!dout || !qkv || !out || !lse || !dqkv || !scratch_D) return ret(GPT2_ERR_ARG);
    if (B < 1 || T < 1 || NH < 1 || C % NH) return ret(GPT2_ERR_ARG);
    const int HS = C / NH;
    if (HS != 16 && HS != 32 && HS != 64 && HS != 128) return ret(GPT2_ERR_CONFIG);
    if (!known_dtype(dtype)) return ret(GPT2_ERR_CONFIG);
    int dev;
    if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    unsigned int* err = err_word(dev);
    if (!err) return ret(GPT2_ERR_NOMEM);
    const int rc = launch_attention_backward(to_dt(dtype), tensor_cores, dqkv,
                                             dout, qkv, out, lse, scratch_D, B, T, C, NH,
                                             (cudaStream_t)stream, err);
    if (rc != GPT2_OK) return ret(rc);
    return ret(launch_status());
}

int gpt2_layernorm_forward(int dtype, void* out, float* mean, float* rstd, const void* inp,
                           const void* w, const void* b, int N, int C, void* stream) {
    const ErrScope ret("gpt2_layernorm_forward");
    if (!out || !mean || !rstd || !inp || !w || !b) return ret(GPT2_ERR_ARG);
    if (!known_dtype(dtype)) return ret(GPT2_ERR_CONFIG);
    if (N < 1 || C < 8 || C % 8 || C > (dtype == GPT2_FP32 ? 1024 : 2048)) return ret(GPT2_ERR_ARG);
    launch_layernorm_forward(to_dt(dtype), out, mean, rstd, inp, w, b, N,
                             C, (cudaStream_t)stream);
    return ret(launch_status());
}

size_t gpt2_layernorm_backward_scratch_floats(int C) { return layernorm_backward_ws_floats(C); }

int gpt2_layernorm_backward(int dtype, void* dinp, void* dw, void* db, const void* dout,
                            const void* inp, const void* w, const float* mean, const float* rstd,
                            int N, int C, int accumulate, float* scratch, void* stream) {
    const ErrScope ret("gpt2_layernorm_backward");
    if (!dinp || !dw || !db || !dout || !inp || !w || !mean || !rstd || !scratch) return ret(GPT2_ERR_ARG);
    if (!known_dtype(dtype)) return ret(GPT2_ERR_CONFIG);
    if (N < 1 || C < 8 || C % 8 || C > (dtype == GPT2_FP32 ? 1024 : 2048)) return ret(GPT2_ERR_ARG);
    int dev;
    if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    unsigned int* err = err_word(dev);
    if (!err) return ret(GPT2_ERR_NOMEM);
    launch_layernorm_backward(to_dt(dtype), dinp, dw, db, dout, inp, w, mean,
                              rstd, N, C, accumulate, scratch, err, (cudaStream_t)stream);
    return ret(launch_status());
}

int gpt2_device_status(void) {
    const ErrScope ret("gpt2_device_status");
    int dev;
    if (current_device(&dev) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    if (cudaDeviceSynchronize() != cudaSuccess) return ret(GPT2_ERR_CUDA);
    unsigned int h = 0;
    // the allocation-free variant's word (only once it has been set up here)
    if (noalloc_err_of(dev, &h) != GPT2_OK) return ret(GPT2_ERR_CUDA);
    // the shared word of the allocating entry points; none exists until one of
    // them ran on this device, and then nothing can have been recorded
    unsigned int* err = nullptr;
    {
        std::lock_guard<std::mutex> lk(ops_mu);
        err = dev_err[dev];
    }
    if (err) {
        unsigned int h2 = 0;
        if (cudaMemcpy(&h2, err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ret(GPT2_ERR_CUDA);
        if (h2) cudaMemset(err, 0, 4);
        h |= h2;
    }
    if (h & DEVERR_TIMEOUT) return ret(GPT2_ERR_DEVICE_TIMEOUT);
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of fused_linear_bias_gelu_softmax.
//
// Some callers cannot let a library call cudaMalloc: processes that hand all
// device memory to their own pool allocator up front (a cudaMalloc behind the
// pool's back can fail or fragment that memory), and loops that cannot take
// the device-wide synchronisation cudaMalloc may imply. For them the per-row
// softmax partials live in the file-scope device array below, reserved when
// the library is loaded and held by every device that loads it until exit.
//
// Limits and sharing: at most NOALLOC_MAX_PARTIALS (row, column tile) pairs:
// calls with M * ceil(N / 256) <= 131072 are accepted (1 MiB of float2), and
// the product takes its narrower 224-column tiles only where their partials
// fit the array as well. Every call uses
// the same array and leaves the previous call's partials in it; nothing needs
// clearing because the GEMM epilogue writes every partial a call reads.
// Calls whose GPU work overlaps (different streams, no ordering between them)
// race on the array and give wrong results.
// Set-up: the first call on a device, with that device current, looks up the
// array's device address (cudaGetSymbolAddress); that first call should come
// before any stream capture.
// ---------------------------------------------------------------------------

}  // extern "C"

#define NOALLOC_MAX_PARTIALS (1 << 17)
static_assert(FUSED_NARROW_MAX_PARTIALS <= NOALLOC_MAX_PARTIALS, "224-column tiles fit the static partials");

static __device__ __align__(256) float2 g_noalloc_part[NOALLOC_MAX_PARTIALS];
// bounded-wait timeout bits of the allocation-free variant (starts at zero)
static __device__ __align__(256) unsigned int g_noalloc_err[64];

namespace {
struct NoAllocDevice {
    bool ready = false;
    float* part = nullptr;
    unsigned int* err = nullptr;
};
NoAllocDevice noalloc_dev[kMaxDevices];
}  // namespace

// Host code cannot use the arrays' names as device addresses: look the
// addresses up once per device (with that device current) and pass them on.
static int noalloc_setup(int dev, NoAllocDevice* out) {
    std::lock_guard<std::mutex> lk(ops_mu);
    if (!noalloc_dev[dev].ready) {
        void* part = nullptr;
        void* err = nullptr;
        if (cudaGetSymbolAddress(&part, g_noalloc_part) != cudaSuccess) return GPT2_ERR_CUDA;
        if (cudaGetSymbolAddress(&err, g_noalloc_err) != cudaSuccess) return GPT2_ERR_CUDA;
        noalloc_dev[dev].part = (float*)part;
        noalloc_dev[dev].err = (unsigned int*)err;
        noalloc_dev[dev].ready = true;
    }
    *out = noalloc_dev[dev];
    return GPT2_OK;
}

// reads (and clears) the variant's timeout bits; 0 if it was never set up on dev
static int noalloc_err_of(int dev, unsigned int* bits) {
    *bits = 0;
    bool ready;
    {
        std::lock_guard<std::mutex> lk(ops_mu);
        ready = noalloc_dev[dev].ready;
    }
    if (!ready) return GPT2_OK;
    if (cudaMemcpyFromSymbol(bits, g_noalloc_err, sizeof(unsigned int)) != cudaSuccess)
        return GPT2_ERR_CUDA;
    if (*bits) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_noalloc_err, &zero, sizeof(unsigned int)) != cudaSuccess)
            return GPT2_ERR_CUDA;
    }
    return GPT2_OK;
}

extern "C" int fused_linear_bias_gelu_softmax_noalloc(const float* x, const float* W,
                                                      const float* b, float* out, int M, int K,
                                                      int N, void* stream) {
    const ErrScope ret("fused_linear_bias_gelu_softmax_noalloc");
    if (!x || !W || !b || !out) return gk::set_error(GPT2_ERR_ARG, "fused op (no-alloc): NULL pointer");
    if (M < 1 || K < 1 || N < 1)
        return gk::set_error(GPT2_ERR_ARG, "fused op (no-alloc): M, K, N must be >= 1");
    if (!al16(x) || !al16(W) || !al16(b) || !al16(out) || K % 4 || N % 4)
        return gk::set_error(GPT2_ERR_ALIGN,
                             "fused op (no-alloc): pointers must be 16-byte aligned, K and N multiples of 4");
    const long long tiles256 = ((long long)N + 255) / 256;
    if ((long long)M * tiles256 > NOALLOC_MAX_PARTIALS)
        return gk::set_error(GPT2_ERR_ARG,
                             "fused op (no-alloc): M * ceil(N/256) = %lld exceeds the static scratch "
                             "limit of %d",
                             (long long)M * tiles256, NOALLOC_MAX_PARTIALS);
    // 224-column tiles only where their partials fit the array too
    const int tile_n = fused_split_tile_n(M, N, FUSED_NARROW_MAX_PARTIALS);
    const long long tiles = ((long long)N + tile_n - 1) / tile_n;
    int dev;
    if (current_device(&dev) != GPT2_OK) return gk::set_error(GPT2_ERR_CUDA, "no current device");
    NoAllocDevice d;
    if (noalloc_setup(dev, &d) != GPT2_OK)
        return gk::set_error(GPT2_ERR_CUDA, "fused op (no-alloc): cudaGetSymbolAddress failed");
    cudaStream_t s = (cudaStream_t)stream;
    const int rc = launch_fused_split_gemm(x, W, b, out, d.part, (int)tiles, M, K, N, tile_n, s, d.err);
    if (rc != GPT2_OK) return ret(rc);
    launch_softmax_finish(out, d.part, M, N, (int)tiles, s);
    if (cudaGetLastError() != cudaSuccess)
        return gk::set_error(GPT2_ERR_CUDA, "fused op (no-alloc): launch failed");
    return GPT2_OK;
}
