// common.cuh -- shared device helpers for the GB300 GPT-2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DEVI __device__ __forceinline__

typedef __nv_bfloat16 bf16;
typedef __half f16;

// ---------------------------------------------------------------- conversions
DEVI float to_f(float x) { return x; }
DEVI float to_f(bf16 x) { return __bfloat162float(x); }
DEVI float to_f(f16 x) { return __half2float(x); }
template <typename T> DEVI T from_f(float x);
template <> DEVI float from_f<float>(float x) { return x; }
template <> DEVI bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }
template <> DEVI f16 from_f<f16>(float x) { return __float2half_rn(x); }

// two 16-bit values in one 32-bit word (low half first) widened to fp32, and
// two fp32 values rounded (nearest even) into one such word
template <typename H> DEVI float2 h2_f2(uint32_t u);
template <> DEVI float2 h2_f2<bf16>(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
template <> DEVI float2 h2_f2<f16>(uint32_t u) { return __half22float2(*reinterpret_cast<const __half2*>(&u)); }
template <typename H> DEVI uint32_t f2_h2(float a, float b);
template <> DEVI uint32_t f2_h2<bf16>(float a, float b) {
    __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&r);
}
template <> DEVI uint32_t f2_h2<f16>(float a, float b) {
    __half2 r = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&r);
}

// 16-byte vector of T (4 floats or 8 bf16)
template <typename T> struct alignas(16) Vec16 {
    static constexpr int N = 16 / sizeof(T);
    T v[N];
};

template <typename T> DEVI Vec16<T> ld16(const T* p) {
    Vec16<T> r;
    *reinterpret_cast<int4*>(&r) = *reinterpret_cast<const int4*>(p);
    return r;
}
// streaming load (evict-first), for data that is read once
template <typename T> DEVI Vec16<T> ld16_cs(const T* p) {
    Vec16<T> r;
    *reinterpret_cast<int4*>(&r) = __ldcs(reinterpret_cast<const int4*>(p));
    return r;
}
template <typename T> DEVI void st16(T* p, const Vec16<T>& v) {
    *reinterpret_cast<int4*>(p) = *reinterpret_cast<const int4*>(&v);
}
template <typename T> DEVI void st16_cs(T* p, const Vec16<T>& v) {
    __stcs(reinterpret_cast<int4*>(p), *reinterpret_cast<const int4*>(&v));
}

// ---------------------------------------------------------------- reductions
// Programmatic dependent launch: allow the next kernel of the stream to be
// scheduled (its prologue overlaps this kernel's tail), then wait until every
// kernel this one depends on has finished and its writes are visible. Every
// kernel launched through launch_pdl calls it before its first global memory
// access; without the launch attribute both instructions do nothing.
DEVI void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

DEVI float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
DEVI float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------- GELU (tanh form)
// gelu(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
#define GELU_K0 0.7978845608028654f  // sqrt(2/pi)
#define GELU_K1 0.044715f
DEVI float gelu_fwd(float x) {
    float u = GELU_K0 * (x + GELU_K1 * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}
// hardware tanh (tanh.approx.f32, max relative error about 2^-11): used where the
// result is rounded to bf16 right away, so its error is below the rounding
DEVI float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// d gelu / dx = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3 * 0.044715 x^2)
DEVI float gelu_grad(float x) {
    float u = GELU_K0 * (x + GELU_K1 * x * x * x);
    float t = tanhf(u);
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * GELU_K0 * (1.0f + 3.0f * GELU_K1 * x * x);
}

