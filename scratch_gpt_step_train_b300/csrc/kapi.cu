// kapi.cu -- the kernel-level C-ABI (include/gpt2_kernels.h): thin wrappers
// that validate arguments and launch the same kernels the model path uses.
#include "../../include/gpt2.h"
#include "../../include/gpt2_kernels.h"
#include "gemm_tc.h"
#include "kernels.h"

#include <cstring>

using namespace gk;

static int rc_of(cudaError_t e) {
    if (e == cudaSuccess) return GPT2_OK;
    if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
        cudaGetLastError();
        return GPT2_ERR_ARG;
    }
    return GPT2_ERR_CUDA;
}
static bool dt_ok(int dtype) { return dtype == ACT_F32 || dtype == ACT_BF16; }

extern "C" size_t gpt2k_matmul_scratch_bytes(void) { return gemm_tc_scratch_bytes(); }

extern "C" int gpt2k_binary_arch(void) {
    const int v = gemm_tc_binary_version();
    return v < 0 ? GPT2_ERR_CUDA : v;
}

extern "C" int gpt2k_matmul(int dtype, int impl, int M, int N, int K, const void* A, long lda,
                            int a_kmajor, const void* B, long ldb, int b_kmajor, void* D,
                            long ldd, const void* bias, const void* resid, long ldr, void* aux,
                            long ldx, int epi, void* scratch, size_t scratch_bytes,
                            unsigned* err, void* stream) {
    if (!dt_ok(dtype) || M < 1 || N < 1 || K < 1 || !A || !B || !D) return GPT2_ERR_ARG;
    if (epi < EPI_STORE || epi > EPI_MUL_AUX) return GPT2_ERR_ARG;
    if (epi == EPI_RESID && !resid) return GPT2_ERR_ARG;
    if ((epi == EPI_GELU || epi == EPI_GELU_BWD || epi == EPI_GELU_D || epi == EPI_MUL_AUX) &&
        !aux)
        return GPT2_ERR_ARG;
    GemmDesc d;
    d.M = M; d.N = N; d.K = K;
    d.A = A; d.lda = lda; d.a_kmajor = a_kmajor;
    d.B = B; d.ldb = ldb; d.b_kmajor = b_kmajor;
    d.D = D; d.ldd = ldd;
    d.bias = bias; d.resid = resid; d.ldr = ldr; d.aux = aux; d.ldx = ldx;
    d.epi = epi; d.act = dtype;
    d.dbias = nullptr;
    d.colpart = nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    bool tc = dtype == ACT_BF16 && gemm_tc_available() && gemm_tc_supported(d);
    if (impl == 2 && !tc) return GPT2_ERR_ARG;
    if (impl == 1 || !tc) return rc_of(gemm_simt(d, s));
    int nl;
    return rc_of(gemm_tc(d, scratch, scratch_bytes, err, s, &nl));
}

extern "C" int gpt2k_matmul_bias_grad(int M, int N, int K, const void* A, long lda,
                                      int a_kmajor, const void* B, long ldb, int b_kmajor,
                                      void* D, long ldd, void* aux, long ldx, int epi,
                                      float* dbias, void* scratch, size_t scratch_bytes,
                                      unsigned* err, void* stream) {
    if (M < 1 || N < 1 || K < 1 || !A || !B || !D || !aux || !dbias || !scratch)
        return GPT2_ERR_ARG;
    if (epi != EPI_MUL_AUX && epi != EPI_GELU_BWD) return GPT2_ERR_ARG;
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.M = M; d.N = N; d.K = K;
    d.A = A; d.lda = lda; d.a_kmajor = a_kmajor;
    d.B = B; d.ldb = ldb; d.b_kmajor = b_kmajor;
    d.D = D; d.ldd = ldd;
    d.aux = aux; d.ldx = ldx;
    d.epi = epi; d.act = ACT_BF16;
    d.dbias = dbias;
    if (!gemm_tc_available() || !gemm_tc_supported(d)) return GPT2_ERR_ARG;
    int nl;
    return rc_of(gemm_tc(d, scratch, scratch_bytes, err, (cudaStream_t)stream, &nl));
}

extern "C" int gpt2k_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B,
                                       int T, int C, int H, void* stream) {
    if (!dt_ok(dtype) || B < 1 || T < 1 || H < 1 || C % H) return GPT2_ERR_ARG;
    return rc_of(attention_forward(dtype, out, lse, qkv, B, T, C, H, nullptr, (cudaStream_t)stream));
}

extern "C" size_t gpt2k_attention_backward_scratch_bytes(int B, int T, int C, int H) {
    (void)C;
    return attention_backward_scratch(B, T, H);
}

extern "C" int gpt2k_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv,
                                        const void* out, const float* lse, int B, int T, int C,
                                        int H, void* scratch, void* stream) {
    if (!dt_ok(dtype) || B < 1 || T < 1 || H < 1 || C % H || !scratch) return GPT2_ERR_ARG;
    return rc_of(attention_backward(dtype, dqkv, dout, qkv, out, lse, B, T, C, H, scratch,
                                    nullptr, (cudaStream_t)stream));
}

extern "C" int gpt2k_layernorm_forward(int dtype, void* out, float* mean, float* rstd,
                                       const void* x, const void* w, const void* b, int N, int C,
                                       void* stream) {
    if (!dt_ok(dtype) || N < 1 || C < 1) return GPT2_ERR_ARG;
    return rc_of(layernorm_forward(dtype, out, mean, rstd, x, w, b, N, C, (cudaStream_t)stream));
}

extern "C" size_t gpt2k_layernorm_backward_scratch_bytes(int N, int C) {
    return layernorm_backward_scratch(N, C, true);
}

extern "C" int gpt2k_layernorm_backward(int dtype, void* dx, float* dw, float* db, float* dxsum,
                                        const void* dout, const void* x, const void* w,
                                        const float* mean, const float* rstd, int N, int C,
                                        int accumulate, void* scratch, void* stream) {
    if (!dt_ok(dtype) || N < 1 || C < 1 || !scratch) return GPT2_ERR_ARG;
    return rc_of(layernorm_backward(dtype, dx, dw, db, dxsum, dout, x, w, mean, rstd, N, C,
                                    accumulate != 0, scratch, (cudaStream_t)stream));
}

extern "C" int gpt2k_encoder_forward(int dtype, void* out, const int32_t* tok, const void* wte,
                                     const void* wpe, int B, int T, int C, int V, unsigned* err,
                                     void* stream) {
    if (!dt_ok(dtype) || B < 1 || T < 1 || C < 1 || V < 1 || !err) return GPT2_ERR_ARG;
    return rc_of(encoder_forward(dtype, out, tok, wte, wpe, B, T, C, V, err,
                                 (cudaStream_t)stream));
}

extern "C" size_t gpt2k_encoder_backward_scratch_bytes(int B, int T, int C, int Vp) {
    return encoder_backward_scratch(B, T, C, Vp);
}

extern "C" int gpt2k_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx,
                                      const int32_t* tok, int B, int T, int C, int Vp,
                                      void* scratch, void* stream) {
    if (!dt_ok(dtype) || B < 1 || T < 1 || C < 1 || Vp < 1 || !scratch) return GPT2_ERR_ARG;
    return rc_of(encoder_backward(dtype, dwte, dwpe, dx, tok, B, T, C, Vp, scratch,
                                  (cudaStream_t)stream));
}

extern "C" int gpt2k_crossentropy(int dtype, void* logits, float* losses, const int32_t* tgt,
                                  int N, int V, int Vp, float dloss, unsigned* err,
                                  void* stream) {
    if (!dt_ok(dtype) || N < 1 || V < 1 || Vp < V || !err) return GPT2_ERR_ARG;
    return rc_of(crossentropy_fused(dtype, logits, losses, tgt, N, V, Vp, dloss, err,
                                    (cudaStream_t)stream));
}

extern "C" int gpt2k_stochastic_round_bf16(void* out, const float* in, size_t n, uint64_t seed,
                                           uint64_t k0, void* stream) {
    if (!out || !in) return GPT2_ERR_ARG;
    if (n == 0) return GPT2_OK;
    return rc_of(stochastic_round_bf16(out, in, n, seed, k0, (cudaStream_t)stream));
}

extern "C" int gpt2k_gelu_forward(int dtype, void* out, const void* in, size_t n, void* stream) {
    if (!dt_ok(dtype) || !out || !in) return GPT2_ERR_ARG;
    if (n == 0) return GPT2_OK;
    return rc_of(gelu_forward(dtype, out, in, n, (cudaStream_t)stream));
}

extern "C" size_t gpt2k_bias_grad_scratch_bytes(int N, int OC) { return bias_grad_scratch(N, OC); }

extern "C" int gpt2k_bias_grad(int dtype, float* db, const void* dout, int N, int OC,
                               void* scratch, void* stream) {
    if (!dt_ok(dtype) || N < 1 || OC < 1 || !scratch) return GPT2_ERR_ARG;
    return rc_of(bias_grad(dtype, db, dout, N, OC, scratch, (cudaStream_t)stream));
}
