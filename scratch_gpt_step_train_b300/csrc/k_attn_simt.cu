// k_attn_simt.cu -- causal multi-head attention, forward and backward, with
// fp32 FFMA arithmetic (parity mode).
//
// Definition ("Getting started with LLMs from Andrej Karpathy's talk",
// self-attention section): O = softmax(Q K^T / sqrt(d_k)) V per head, with the
// causal mask of GPT-2 (query t sees keys 0..t; later keys are left out of the
// softmax).  The forward is flash-style: keys are visited in tiles with an
// online (max, sum) softmax, so the T x T matrix is never stored; the row
// log-sum-exp is kept for the backward pass, which recomputes P from it:
//   P = exp(S - lse), dV = P^T dO, dP = dO V^T, D = rowsum(dO o O),
//   dS = P o (dP - D), dQ = dS K / sqrt(hd), dK = dS^T Q / sqrt(hd).
// dQ and (dK, dV) are produced by two kernels that each own their outputs,
// so no atomics are needed and the result is deterministic.
//
// Layout: qkv [B,T,3C] = Q | K | V, head h at columns h*hd.. of each block;
// out [B,T,C]; lse [B,H,T] fp32.
#include "common.cuh"
#include "kernels.h"

namespace gk {

#define AT_TILE 64

template <typename T, int HD>
__global__ void __launch_bounds__(AT_TILE) k_attn_fwd(T* out, float* lse, const T* qkv, int T_,
                                                      int C, int H) {
    gdc_wait();
    gdc_launch_dependents();
    extern __shared__ float sm[];
    float* Ks = sm;                      // [AT_TILE][HD]
    float* Vs = sm + AT_TILE * HD;       // [AT_TILE][HD]
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int t = blockIdx.x * AT_TILE + threadIdx.x;
    size_t C3 = 3 * (size_t)C;
    const T* base = qkv + (size_t)b * T_ * C3 + (size_t)h * HD;
    float scale = rsqrtf((float)HD);
    float q[HD], o[HD];
    bool live = t < T_;
    if (live) {
#pragma unroll
        for (int i = 0; i < HD; i++) q[i] = to_f(base[(size_t)t * C3 + i]);
    }
#pragma unroll
    for (int i = 0; i < HD; i++) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    int tmax = min(T_ - 1, (int)(blockIdx.x * AT_TILE + AT_TILE - 1));
    for (int k0 = 0; k0 <= tmax; k0 += AT_TILE) {
        __syncthreads();
        for (int e = threadIdx.x; e < AT_TILE * HD; e += AT_TILE) {
            int j = e / HD, i = e % HD, key = k0 + j;
            float kv = 0.f, vv = 0.f;
            if (key < T_) {
                kv = to_f(base[(size_t)key * C3 + C + i]);
                vv = to_f(base[(size_t)key * C3 + 2 * C + i]);
            }
            Ks[e] = kv;
            Vs[e] = vv;
        }
        __syncthreads();
        if (!live) continue;
        int jmax = min(AT_TILE - 1, t - k0);
        for (int j = 0; j <= jmax; j++) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < HD; i++) s = fmaf(q[i], Ks[j * HD + i], s);
            s *= scale;
            if (s > m) {
                float corr = __expf(m - s);
                l *= corr;
#pragma unroll
                for (int i = 0; i < HD; i++) o[i] *= corr;
                m = s;
            }
            float p = __expf(s - m);
            l += p;
#pragma unroll
            for (int i = 0; i < HD; i++) o[i] = fmaf(p, Vs[j * HD + i], o[i]);
        }
    }
    if (!live) return;
    float inv = 1.f / l;
    T* orow = out + ((size_t)b * T_ + t) * C + (size_t)h * HD;
#pragma unroll
    for (int i = 0; i < HD; i++) orow[i] = from_f<T>(o[i] * inv);
    lse[((size_t)b * H + h) * T_ + t] = m + logf(l);
}

// D[b,h,t] = sum_i dO[b,t,h,i] * O[b,t,h,i]
template <typename T>
__global__ void k_attn_D(float* Dv, const T* dout, const T* out, int B, int T_, int C, int H,
                         int hd) {
    gdc_wait();
    gdc_launch_dependents();
    long idx = blockIdx.x * (long)blockDim.x + threadIdx.x;
    if (idx >= (long)B * H * T_) return;
    int t = (int)(idx % T_);
    int bh = (int)(idx / T_), b = bh / H, h = bh % H;
    const T* a = dout + ((size_t)b * T_ + t) * C + (size_t)h * hd;
    const T* o = out + ((size_t)b * T_ + t) * C + (size_t)h * hd;
    float s = 0.f;
    for (int i = 0; i < hd; i++) s = fmaf(to_f(a[i]), to_f(o[i]), s);
    Dv[idx] = s;
}


// dQ: one thread per query.
template <typename T, int HD>
__global__ void __launch_bounds__(AT_TILE) k_attn_dq(T* dqkv, const T* dout, const T* qkv,
                                                     const float* lse, const float* Dv, int T_,
                                                     int C, int H) {
    gdc_wait();
    gdc_launch_dependents();
    extern __shared__ float sm[];
    const int P = HD + 1;
    float* Ks = sm;                    // [AT_TILE][HD]
    float* Vs = Ks + AT_TILE * HD;     // [AT_TILE][HD]
    float* Qs = Vs + AT_TILE * HD;     // [AT_TILE][P]
    float* dOs = Qs + AT_TILE * P;     // [AT_TILE][P]
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int tl = threadIdx.x, t = blockIdx.x * AT_TILE + tl;
    size_t C3 = 3 * (size_t)C;
    const T* base = qkv + (size_t)b * T_ * C3 + (size_t)h * HD;
    bool live = t < T_;
    for (int i = 0; i < HD; i++) {
        Qs[tl * P + i] = live ? to_f(base[(size_t)t * C3 + i]) : 0.f;
        dOs[tl * P + i] = live ? to_f(dout[((size_t)b * T_ + t) * C + (size_t)h * HD + i]) : 0.f;
    }
    float L = live ? lse[(size_t)bh * T_ + t] : 0.f;
    float Dt = live ? Dv[(size_t)bh * T_ + t] : 0.f;
    float scale = rsqrtf((float)HD);
    float dq[HD];
#pragma unroll
    for (int i = 0; i < HD; i++) dq[i] = 0.f;
    int tmax = min(T_ - 1, (int)(blockIdx.x * AT_TILE + AT_TILE - 1));
    for (int k0 = 0; k0 <= tmax; k0 += AT_TILE) {
        __syncthreads();
        for (int e = threadIdx.x; e < AT_TILE * HD; e += AT_TILE) {
            int j = e / HD, i = e % HD, key = k0 + j;
            Ks[e] = key < T_ ? to_f(base[(size_t)key * C3 + C + i]) : 0.f;
            Vs[e] = key < T_ ? to_f(base[(size_t)key * C3 + 2 * C + i]) : 0.f;
        }
        __syncthreads();
        if (!live) continue;
        int jmax = min(AT_TILE - 1, t - k0);
        for (int j = 0; j <= jmax; j++) {
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int i = 0; i < HD; i++) {
                s = fmaf(Qs[tl * P + i], Ks[j * HD + i], s);
                dp = fmaf(dOs[tl * P + i], Vs[j * HD + i], dp);
            }
            float p = __expf(s * scale - L);
            float ds = p * (dp - Dt);
#pragma unroll
            for (int i = 0; i < HD; i++) dq[i] = fmaf(ds, Ks[j * HD + i], dq[i]);
        }
    }
    if (!live) return;
    T* dst = dqkv + ((size_t)b * T_ + t) * C3 + (size_t)h * HD;
#pragma unroll
    for (int i = 0; i < HD; i++) dst[i] = from_f<T>(dq[i] * scale);
}

// dK, dV: one thread per key.
template <typename T, int HD>
__global__ void __launch_bounds__(AT_TILE) k_attn_dkv(T* dqkv, const T* dout, const T* qkv,
                                                      const float* lse, const float* Dv, int T_,
                                                      int C, int H) {
    gdc_wait();
    gdc_launch_dependents();
    extern __shared__ float sm[];
    const int P = HD + 1;
    float* Ks = sm;                    // [AT_TILE][P]  this block's keys
    float* Vs = Ks + AT_TILE * P;      // [AT_TILE][P]
    float* Qs = Vs + AT_TILE * P;      // [AT_TILE][HD] query tile
    float* dOs = Qs + AT_TILE * HD;    // [AT_TILE][HD]
    float* Ls = dOs + AT_TILE * HD;    // [AT_TILE]
    float* Ds = Ls + AT_TILE;          // [AT_TILE]
    int bh = blockIdx.y, b = bh / H, h = bh % H;
    int jl = threadIdx.x, j = blockIdx.x * AT_TILE + jl;
    size_t C3 = 3 * (size_t)C;
    const T* base = qkv + (size_t)b * T_ * C3 + (size_t)h * HD;
    bool live = j < T_;
    for (int i = 0; i < HD; i++) {
        Ks[jl * P + i] = live ? to_f(base[(size_t)j * C3 + C + i]) : 0.f;
        Vs[jl * P + i] = live ? to_f(base[(size_t)j * C3 + 2 * C + i]) : 0.f;
    }
    float scale = rsqrtf((float)HD);
    float dk[HD], dv[HD];
#pragma unroll
    for (int i = 0; i < HD; i++) dk[i] = dv[i] = 0.f;
    for (int q0 = blockIdx.x * AT_TILE; q0 < T_; q0 += AT_TILE) {
        __syncthreads();
        for (int e = threadIdx.x; e < AT_TILE * HD; e += AT_TILE) {
            int r = e / HD, i = e % HD, t = q0 + r;
            Qs[e] = t < T_ ? to_f(base[(size_t)t * C3 + i]) : 0.f;
            dOs[e] = t < T_ ? to_f(dout[((size_t)b * T_ + t) * C + (size_t)h * HD + i]) : 0.f;
        }
        {
            int t = q0 + threadIdx.x;
            Ls[threadIdx.x] = t < T_ ? lse[(size_t)bh * T_ + t] : 0.f;
            Ds[threadIdx.x] = t < T_ ? Dv[(size_t)bh * T_ + t] : 0.f;
        }
        __syncthreads();
        if (!live) continue;
        int rmax = min(AT_TILE - 1, T_ - 1 - q0);
        int rmin = max(0, j - q0);
        for (int r = rmin; r <= rmax; r++) {
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int i = 0; i < HD; i++) {
                s = fmaf(Qs[r * HD + i], Ks[jl * P + i], s);
                dp = fmaf(dOs[r * HD + i], Vs[jl * P + i], dp);
            }
            float p = __expf(s * scale - Ls[r]);
            float ds = p * (dp - Ds[r]);
#pragma unroll
            for (int i = 0; i < HD; i++) {
                dv[i] = fmaf(p, dOs[r * HD + i], dv[i]);
                dk[i] = fmaf(ds, Qs[r * HD + i], dk[i]);
            }
        }
    }
    if (!live) return;
    T* dst = dqkv + ((size_t)b * T_ + j) * C3 + (size_t)h * HD;
#pragma unroll
    for (int i = 0; i < HD; i++) {
        dst[C + i] = from_f<T>(dk[i] * scale);
        dst[2 * C + i] = from_f<T>(dv[i]);
    }
}

template <typename T, int HD>
static cudaError_t attn_fwd_hd(void* out, float* lse, const void* qkv, int B, int T_, int C,
                               int H, cudaStream_t s) {
    dim3 grid((T_ + AT_TILE - 1) / AT_TILE, B * H);
    size_t smem = 2 * AT_TILE * HD * sizeof(float);
    auto kf = k_attn_fwd<T, HD>;
    cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(kf, grid, AT_TILE, smem, s, (T*)out, lse, (const T*)qkv, T_, C, H);
    return cudaGetLastError();
}

template <typename T, int HD>
static cudaError_t attn_bwd_hd(void* dqkv, const void* dout, const void* qkv, const void* out,
                               const float* lse, int B, int T_, int C, int H, float* Dv,
                               cudaStream_t s) {
    long n = (long)B * H * T_;
    launch_pdl(k_attn_D<T>, (int)((n + 255) / 256), 256, 0, s, Dv, (const T*)dout, (const T*)out, B, T_,
                                                       C, H, HD);
    dim3 grid((T_ + AT_TILE - 1) / AT_TILE, B * H);
    const int P = HD + 1;
    size_t smq = (2 * AT_TILE * HD + 2 * AT_TILE * P) * sizeof(float);
    auto kq = k_attn_dq<T, HD>;
    cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
    launch_pdl(kq, grid, AT_TILE, smq, s, (T*)dqkv, (const T*)dout, (const T*)qkv, lse, Dv, T_, C, H);
    size_t smk = (2 * AT_TILE * P + 2 * AT_TILE * HD + 2 * AT_TILE) * sizeof(float);
    auto kk = k_attn_dkv<T, HD>;
    cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
    launch_pdl(kk, grid, AT_TILE, smk, s, (T*)dqkv, (const T*)dout, (const T*)qkv, lse, Dv, T_, C, H);
    return cudaGetLastError();
}

#define HD_DISPATCH(FN, T, ...)                       \
    switch (C / H) {                                  \
        case 8: return FN<T, 8>(__VA_ARGS__);         \
        case 16: return FN<T, 16>(__VA_ARGS__);       \
        case 32: return FN<T, 32>(__VA_ARGS__);       \
        case 64: return FN<T, 64>(__VA_ARGS__);       \
        case 128: return FN<T, 128>(__VA_ARGS__);     \
        default: return cudaErrorInvalidValue;        \
    }

cudaError_t attention_forward(int act, void* out, float* lse, const void* qkv, int B, int T_,
                              int C, int H, unsigned* err, cudaStream_t s) {
    if (attention_tc_supported(act, B, T_, C, H, qkv))
        return attention_forward_tc(out, lse, qkv, B, T_, C, H, err, s);
    if (act == ACT_BF16) {
        HD_DISPATCH(attn_fwd_hd, bf16, out, lse, qkv, B, T_, C, H, s)
    } else {
        HD_DISPATCH(attn_fwd_hd, float, out, lse, qkv, B, T_, C, H, s)
    }
}

size_t attention_backward_scratch(int B, int T_, int H) {
    return (size_t)B * H * T_ * sizeof(float);
}

cudaError_t attention_backward(int act, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T_, int C, int H,
                               void* scratch, unsigned* err, cudaStream_t s) {
    float* Dv = (float*)scratch;
    if (attention_tc_supported(act, B, T_, C, H, qkv))
        return attention_backward_tc(dqkv, dout, qkv, out, lse, Dv, B, T_, C, H, err, s);
    if (act == ACT_BF16) {
        HD_DISPATCH(attn_bwd_hd, bf16, dqkv, dout, qkv, out, lse, B, T_, C, H, Dv, s)
    } else {
        HD_DISPATCH(attn_bwd_hd, float, dqkv, dout, qkv, out, lse, B, T_, C, H, Dv, s)
    }
}

}  // namespace gk
