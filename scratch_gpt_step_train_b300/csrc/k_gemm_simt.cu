// k_gemm_simt.cu -- D[M,N] = A[M,K] . B[N,K]^T with fp32 FFMA accumulation and
// the fused epilogues of the GPT-2 step (bias, bias+GELU keeping the
// pre-activation, bias+residual, fp32 gradient accumulation, GELU backward).
//
// This is the parity-mode contraction (no TF32, no tensor cores): the linear
// layers of "Karpathy's llm.c: understanding LLM training from scratch in
// C/CUDA", "Code anatomy" (QKV, attention projection, MLP fc / fc-proj,
// tied classifier), forward and backward.  A and B may each be K-major or
// M/N-major, so the backward products dX = dY W and dW = dY^T X need no
// transposed copies.
#include "common.cuh"
#include "kernels.h"

namespace gk {

#define SG_BM 64
#define SG_BN 64
#define SG_BK 16

template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simt(GemmDesc d) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ float As[SG_BK][SG_BM + 4];
    __shared__ float Bs[SG_BK][SG_BN + 4];
    const T* A = (const T*)d.A;
    const T* B = (const T*)d.B;
    int tid = threadIdx.x;
    int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
    int tx = tid % 16, ty = tid / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d.K; k0 += SG_BK) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int m, k;
            if (d.a_kmajor) { k = tid % 16; m = tid / 16 + 16 * i; }
            else { m = tid % 64; k = tid / 64 + 4 * i; }
            int gm = m0 + m, gk_ = k0 + k;
            float v = 0.f;
            if (gm < d.M && gk_ < d.K)
                v = to_f(d.a_kmajor ? A[(size_t)gm * d.lda + gk_] : A[(size_t)gk_ * d.lda + gm]);
            As[k][m] = v;
            int n;
            if (d.b_kmajor) { k = tid % 16; n = tid / 16 + 16 * i; }
            else { n = tid % 64; k = tid / 64 + 4 * i; }
            int gn = n0 + n;
            gk_ = k0 + k;
            v = 0.f;
            if (gn < d.N && gk_ < d.K)
                v = to_f(d.b_kmajor ? B[(size_t)gn * d.ldb + gk_] : B[(size_t)gk_ * d.ldb + gn]);
            Bs[k][n] = v;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < SG_BK; k++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

    const T* bias = (const T*)d.bias;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int m = m0 + ty * 4 + i;
        if (m >= d.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int n = n0 + tx * 4 + j;
            if (n >= d.N) continue;
            float v = acc[i][j];
            switch (d.epi) {
                case EPI_ACCUM_F32: {
                    float* D = (float*)d.D + (size_t)m * d.ldd + n;
                    *D += v;
                    break;
                }
                case EPI_GELU_BWD: {
                    float pre = to_f(((const T*)d.aux)[(size_t)m * d.ldx + n]);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(v * gelu_grad_f(pre));
                    break;
                }
                case EPI_MUL_AUX: {
                    float dg = to_f(((const T*)d.aux)[(size_t)m * d.ldx + n]);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(v * dg);
                    break;
                }
                case EPI_GELU_D: {
                    if (bias) v += to_f(bias[n]);
                    float g, dg;
                    gelu_and_grad_f(v, g, dg);
                    ((T*)d.aux)[(size_t)m * d.ldx + n] = from_f<T>(dg);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(g);
                    break;
                }
                case EPI_GELU: {
                    if (bias) v += to_f(bias[n]);
                    ((T*)d.aux)[(size_t)m * d.ldx + n] = from_f<T>(v);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(gelu_f(v));
                    break;
                }
                case EPI_RESID: {
                    if (bias) v += to_f(bias[n]);
                    v += to_f(((const T*)d.resid)[(size_t)m * d.ldr + n]);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(v);
                    break;
                }
                default: {
                    if (bias) v += to_f(bias[n]);
                    ((T*)d.D)[(size_t)m * d.ldd + n] = from_f<T>(v);
                }
            }
        }
    }
}

cudaError_t gemm_simt(const GemmDesc& d, cudaStream_t s) {
    if (d.M <= 0 || d.N <= 0) return cudaSuccess;
    dim3 grid((d.N + SG_BN - 1) / SG_BN, (d.M + SG_BM - 1) / SG_BM);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    if (d.act == ACT_BF16) launch_pdl(k_gemm_simt<bf16>, grid, 256, 0, s, d);
    else launch_pdl(k_gemm_simt<float>, grid, 256, 0, s, d);
    return cudaGetLastError();
}

}  // namespace gk
