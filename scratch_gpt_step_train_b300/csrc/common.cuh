// common.cuh -- small device helpers shared by the kernels of libgpt2b300.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;


__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// Butterfly reductions over the 32 lanes of a warp (__shfl_xor_sync), the
// primitive named in "Karpathy's llm.c ...", section "Code anatomy", item 2.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Programmatic dependent launch: every kernel of the library is launched
// allowed to start before the kernel ahead of it in the stream has finished
// (launch_pdl); gdc_wait() blocks until that kernel has completed and its
// memory is visible, and must come before the first global-memory access.
// gdc_launch_dependents() then lets the next kernel's blocks be scheduled as
// this grid's blocks finish, so its launch and setup overlap this grid's tail.
__device__ __forceinline__ void gdc_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void gdc_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Vector of N elements of T moved as one 16-byte (or smaller) access.
template <typename T, int N>
struct alignas(sizeof(T) * N) Vec {
    T v[N];
};

template <typename T, int N>
__device__ __forceinline__ void load_vec_f(float* dst, const T* src) {
    Vec<T, N> x = *reinterpret_cast<const Vec<T, N>*>(src);
#pragma unroll
    for (int i = 0; i < N; i++) dst[i] = to_f(x.v[i]);
}
template <typename T, int N>
__device__ __forceinline__ void store_vec_f(T* dst, const float* src) {
    Vec<T, N> x;
#pragma unroll
    for (int i = 0; i < N; i++) x.v[i] = from_f<T>(src[i]);
    *reinterpret_cast<Vec<T, N>*>(dst) = x;
}

// tanh-form GELU (Hendrycks & Gimpel 2016), 0.5 x (1 + tanh(u)) with
// u = sqrt(2/pi) (x + 0.044715 x^3), and its analytic derivative.  Both are
// evaluated through the exact identity 0.5 (1 + tanh(u)) = 1 / (1 + e^{-2u}),
// which keeps full relative precision in the negative tail where 1 + tanh(u)
// would cancel in fp32 (and 1 - tanh(u)^2 = 4 s (1 - s) with s that sigmoid).
// gelu(x) and gelu'(x) together, sharing the sigmoid.  Every operation is an
// explicitly rounded intrinsic (never contracted into an FMA differently by
// the compiler), so all kernels that call it get the same bits for the same x.
__device__ __forceinline__ void gelu_and_grad_f(float x, float& g, float& dg) {
    const float k = 0.7978845608028654f;
    const float x2 = __fmul_rn(x, x);
    const float u = __fmul_rn(k, __fmaf_rn(__fmul_rn(0.044715f, x2), x, x));
    const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(__fmul_rn(-2.0f, u))));
    const float du = __fmul_rn(k, __fmaf_rn(3.0f * 0.044715f, x2, 1.0f));
    g = __fmul_rn(x, sg);
    dg = __fmaf_rn(__fmul_rn(__fmul_rn(__fmul_rn(2.0f, x), sg), __fsub_rn(1.0f, sg)), du, sg);
}
__device__ __forceinline__ float gelu_f(float x) {
    float g, dg;
    gelu_and_grad_f(x, g, dg);
    return g;
}
__device__ __forceinline__ float gelu_grad_f(float x) {
    float g, dg;
    gelu_and_grad_f(x, g, dg);
    return dg;
}
