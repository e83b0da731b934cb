/*
 * gpt2_kernels.h -- kernel-level C-ABI of libgpt2b300: each hot-path
 * operation of the GPT-2 training step as one call on caller-owned device
 * buffers, so that every operation can be checked on its own (at full size)
 * against an independent reference.  The model-level calls in gpt2.h run
 * exactly these kernels.
 *
 * Common rules
 *  - dtype: 0 = fp32 elements, 1 = bf16 elements, for every activation /
 *    weight buffer of the call (statistics, lse and losses are always fp32).
 *  - All pointers are device pointers on the current device; all work is
 *    enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *    the call returns without waiting.  Buffers are owned by the caller and
 *    must not overlap unless stated.
 *  - `scratch` is caller-owned device memory of at least the size the
 *    matching *_scratch_bytes call returns (256-byte aligned).
 *  - `err` (where present) is a device unsigned word the kernels OR error
 *    bits into: 1 = an id outside [0, V), 2 = a bounded wait ran out.
 *  - Return: 0 on success, -1 (GPT2_ERR_ARG) for a shape / alignment the
 *    kernels do not take, -2 (GPT2_ERR_CUDA) if a launch failed.
 */
#ifndef GPT2_B300_KERNELS_H
#define GPT2_B300_KERNELS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The architecture the library's kernels were built for, as the CUDA runtime
 * reports it for the loaded tensor-core matmul kernel on the current device
 * (cudaFuncAttributes.binaryVersion: major*10 + minor, 103 for sm_103a), or
 * -2 (GPT2_ERR_CUDA) if the kernel cannot be loaded on this device.  Needs a
 * GPU; it launches nothing. */
int gpt2k_binary_arch(void);

/* Linear layer, forward and backward ("Karpathy's llm.c: understanding LLM
 * training from scratch in C/CUDA", "Code anatomy": the QKV / projection /
 * MLP / classifier matmuls):  D[M,N] = epi(sum_k A[m,k] B[n,k]).
 *   A[m,k] is at A[m*lda + k] if a_kmajor else A[k*lda + m]; same for B with n.
 *   epi 0: D = acc (+ bias[n])                      (bias may be NULL)
 *   epi 1: aux = acc + bias[n]; D = gelu_tanh(aux)
 *   epi 2: D = resid[m,n] + acc (+ bias[n])
 *   epi 3: D (fp32) += acc                          (weight-gradient accumulate)
 *   epi 4: D = acc * gelu_tanh'(aux[m,n])           (MLP backward)
 *   epi 5: x = acc + bias[n]; D = gelu_tanh(x), aux = gelu_tanh'(x)
 *          (MLP forward keeping the derivative instead of x)
 *   epi 6: D = acc * aux[m,n]                        (MLP backward with epi 5's aux)
 * impl: 0 = automatic (tensor cores for bf16 when the shape fits, else the
 * fp32-FFMA kernel), 1 = fp32-FFMA kernel, 2 = tensor cores (bf16 only;
 * returns -1 if the shape does not fit: N % 8, 16-byte aligned bases,
 * leading dimensions % 8). */
size_t gpt2k_matmul_scratch_bytes(void);
int gpt2k_matmul(int dtype, int impl, int M, int N, int K, const void* A, long lda, int a_kmajor,
                 const void* B, long ldb, int b_kmajor, void* D, long ldd, const void* bias,
                 const void* resid, long ldr, void* aux, long ldx, int epi, void* scratch,
                 size_t scratch_bytes, unsigned* err, void* stream);
/* The MLP input gradient with the fc bias gradient of the same product (the
 * bias gradient is the column sum of the pre-activation gradient, "Karpathy's
 * llm.c: understanding LLM training from scratch in C/CUDA", "Code anatomy",
 * the matmul backward): bf16 on the tensor cores, epi 6 (D = acc * aux) or
 * epi 4 (D = acc * gelu_tanh'(aux)) as in gpt2k_matmul, and
 *   dbias[n] += sum_m D[m,n]
 * summed in fp32 over D's bf16 values, in a fixed order (32-row blocks, then
 * the blocks in order).  dbias: N floats, device.
 * scratch: at least ceil(M/32) * N * 4 bytes (gpt2k_matmul_scratch_bytes()
 * covers M * N <= 512 Mi), owned by the caller and overwritten.  Returns -1
 * for another epi, NULL pointers or a shape the tensor cores do not take
 * (as impl 2 of gpt2k_matmul). */
int gpt2k_matmul_bias_grad(int M, int N, int K, const void* A, long lda, int a_kmajor,
                           const void* B, long ldb, int b_kmajor, void* D, long ldd, void* aux,
                           long ldx, int epi, float* dbias, void* scratch, size_t scratch_bytes,
                           unsigned* err, void* stream);

/* Causal self-attention ("Getting started with LLMs from Andrej Karpathy's
 * talk", self-attention: softmax(Q K^T / sqrt(d_k)) V), query t attending to
 * keys 0..t.  qkv [B,T,3C] = Q | K | V with head h at columns h*hd.. of each
 * C block; out [B,T,C]; lse [B,H,T] = log-sum-exp of each score row. */
int gpt2k_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B, int T,
                            int C, int H, void* stream);
size_t gpt2k_attention_backward_scratch_bytes(int B, int T, int C, int H);
/* dqkv [B,T,3C] (overwritten) from dout [B,T,C], qkv, out and lse of the forward. */
int gpt2k_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv,
                             const void* out, const float* lse, int B, int T, int C, int H,
                             void* scratch, void* stream);

/* LayerNorm over rows of C (eps 1e-5, biased variance): out = (x-mean)*rstd*w + b,
 * mean/rstd [N] fp32 saved.  Backward: dx [N,C] (dtype) receives the input
 * gradient -- added to its contents if `accumulate` is nonzero, else written
 * over them; dw, db [C] (fp32) ACCUMULATE sum_n dy*xhat and sum_n dy; if dxsum
 * [C] (fp32) is not NULL it ACCUMULATES the column sums of the dx rows as
 * written (the bias gradient of a linear layer whose output gradient is dx).
 * Scratch from gpt2k_layernorm_backward_scratch_bytes covers the dxsum case. */
int gpt2k_layernorm_forward(int dtype, void* out, float* mean, float* rstd, const void* x,
                            const void* w, const void* b, int N, int C, void* stream);
size_t gpt2k_layernorm_backward_scratch_bytes(int N, int C);
int gpt2k_layernorm_backward(int dtype, void* dx, float* dw, float* db, float* dxsum,
                             const void* dout, const void* x, const void* w, const float* mean,
                             const float* rstd, int N, int C, int accumulate, void* scratch,
                             void* stream);

/* Allocation-free LayerNorm backward.  The pages have no counterpart: this
 * is the same computation as gpt2k_layernorm_backward (accumulating into dx,
 * no dxsum) for callers that cannot
 * allocate device memory -- their memory belongs to another allocator that
 * gives them only the operation's tensors, or they run where cudaMalloc /
 * cudaFree must not be called (both may synchronise the device).  Instead of
 * caller scratch it uses a fixed array in device global memory (4.6 MiB,
 * enough for rows of C <= 2048) that every GPU which loads the library holds
 * until the process exits.  It allocates nothing and calls no allocating
 * routine.
 *  - Returns -1 (GPT2_ERR_ARG) for C > 2048 (beyond the fixed scratch) or a bad
 *    shape, -2 if the array's device address cannot be found or a launch fails.
 *  - The first call on each device looks up the array's address with that
 *    device current and keeps it for the process: it assumes one primary
 *    context per device for the process's life (after cudaDeviceReset the
 *    kept address is stale).  Make that first call before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU (on
 *    different streams) race.  Each call fully overwrites the part it uses, so
 *    contents left by an earlier call are harmless. */
int gpt2k_layernorm_backward_noalloc(int dtype, void* dx, float* dw, float* db,
                                     const void* dout, const void* x, const void* w,
                                     const float* mean, const float* rstd, int N, int C,
                                     void* stream);

/* Token + position embedding: out[b,t,:] = wte[tok[b,t],:] + wpe[t,:].
 * Backward ACCUMULATES dwte[tok[b,t],:] += dx[b,t,:] (each row's sum taken
 * in position order, no atomics) and dwpe[t,:] += sum_b dx[b,t,:].  Vp (the
 * rows of dwte) must be a multiple of 4, else GPT2_ERR_ARG; scratch holds
 * gpt2k_encoder_backward_scratch_bytes(B, T, C, Vp) bytes, owned by the
 * caller, not read before it is written. */
int gpt2k_encoder_forward(int dtype, void* out, const int32_t* tok, const void* wte,
                          const void* wpe, int B, int T, int C, int V, unsigned* err,
                          void* stream);
size_t gpt2k_encoder_backward_scratch_bytes(int B, int T, int C, int Vp);
int gpt2k_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx,
                           const int32_t* tok, int B, int T, int C, int Vp, void* scratch,
                           void* stream);

/* Softmax cross-entropy over the first V of Vp columns of logits [N,Vp]:
 * losses[n] = logsumexp(logits[n,:V]) - logits[n,tgt[n]]; if dloss != 0 the
 * row is overwritten in place by (softmax - onehot(tgt)) * dloss, pad
 * columns set to 0 ("Karpathy reproduces GPT-2 (1.6B) in llm.c", "PyTorch
 * comparison": the fused classifier). */
int gpt2k_crossentropy(int dtype, void* logits, float* losses, const int32_t* tgt, int N, int V,
                       int Vp, float dloss, unsigned* err, void* stream);

/* Elementwise tanh-form GELU, out[i] = gelu(in[i]) for i < n, the formula of
 * the fp32 fused epilogue (sigmoid form, see epi 5): the recompute path of the
 * MLP ("Karpathy reproduces GPT-2 (1.6B) in llm.c", "Parameter guide" -r 1)
 * runs it in the forward and again in the backward on the same stored input,
 * so both results are identical.  out and in may be the same buffer. */
int gpt2k_gelu_forward(int dtype, void* out, const void* in, size_t n, void* stream);

/* Stochastic rounding fp32 -> bf16 (the parameter update without fp32 master
 * weights, "Karpathy reproduces GPT-2 (1.6B) in llm.c", "Parameter guide"
 * -w 0): out[i] (bf16 bits) = (bits(in[i]) + r) >> 16 with r the top 16 bits
 * of output number k0 + i (0-based) of the SplitMix64 stream of `seed`
 * (Steele, Lea & Flood 2014: output k = mix(seed + (k+1) * 0x9E3779B97F4A7C15));
 * |x| is rounded up with probability (low 16 bits of x)/65536.  NaN -> NaN. */
int gpt2k_stochastic_round_bf16(void* out, const float* in, size_t n, uint64_t seed, uint64_t k0,
                                void* stream);

/* Bias gradient: db[o] += sum_n dout[n,o] (fixed summation order). */
size_t gpt2k_bias_grad_scratch_bytes(int N, int OC);
int gpt2k_bias_grad(int dtype, float* db, const void* dout, int N, int OC, void* scratch,
                    void* stream);

#ifdef __cplusplus
}
#endif
#endif
