// kernels.h -- host-side launchers of the libgpt2b300 kernels (internal).
//
// Every launcher enqueues on the given stream and returns the launch status.
// `act` selects the activation / compute-copy element type: ACT_F32 (fp32)
// or ACT_BF16 (bf16).  Gradients of parameters are always fp32.
#pragma once
#include <cuda_runtime.h>
#include <utility>
#include <stddef.h>
#include <stdint.h>

// Device error word bits (OR-ed by kernels, read by the host at sync points).
#define GPT2_DEVERR_TOKEN 1u    // a token/target id outside [0, V)
#define GPT2_DEVERR_TIMEOUT 2u  // a bounded wait in a pipelined kernel ran out
#define GPT2_DEVERR_SHAPE 4u    // a kernel was launched with a shape it cannot do

namespace gk {

// Launches kernel k with programmatic stream serialization allowed: it may
// begin while the previous kernel in the stream drains; every kernel of the
// library calls gdc_wait() before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

enum { ACT_F32 = 0, ACT_BF16 = 1 };
inline size_t act_size(int act) { return act == ACT_BF16 ? 2 : 4; }

// Canonical tensor indices (weights are out x in, row-major).
enum {
    P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_PROJW, P_PROJB,
    P_LN2W, P_LN2B, P_FCW, P_FCB, P_FCPROJW, P_FCPROJB, P_LNFW, P_LNFB, P_NUM
};

struct ParamLayout {
    size_t off[P_NUM + 1];  // element offsets; off[P_NUM] = total
    int L, C, V, Vp, T;
};
void make_layout(ParamLayout* lay, int L, int C, int V, int T);

// ---- parameters -----------------------------------------------------------
cudaError_t init_params(float* master, const ParamLayout& lay, uint64_t seed, cudaStream_t s);
cudaError_t cast_to_bf16(void* dst, const float* src, size_t n, cudaStream_t s);

// ---- embedding ------------------------------------------------------------
// out[b,t,:] = wte[tok[b,t],:] + wpe[t,:]; ids outside [0,V) set err bit.
cudaError_t encoder_forward(int act, void* out, const int* tok, const void* wte, const void* wpe,
                            int B, int T, int C, int V, unsigned* err, cudaStream_t s);
// Scratch for the deterministic embedding backward (bytes).
size_t encoder_backward_scratch(int B, int T, int C, int Vp);
// dwte[tok] += dx rows (each row sum taken in position order), dwpe[t] += sum_b dx[b,t].
cudaError_t encoder_backward(int act, float* dwte, float* dwpe, const void* dx, const int* tok,
                             int B, int T, int C, int Vp, void* scratch, cudaStream_t s);

// ---- layernorm ------------------------------------------------------------
cudaError_t layernorm_forward(int act, void* out, float* mean, float* rstd, const void* x,
                              const void* w, const void* b, int N, int C, cudaStream_t s);
// scratch for the partial column sums (dxsum != NULL needs the larger size)
size_t layernorm_backward_scratch(int N, int C, bool dxsum);
// dx += (accum_dx) or = the LayerNorm input gradient; dw += sum dy*xhat,
// db += sum dy; dxsum (if not NULL) += the column sums of the dx rows written.
cudaError_t layernorm_backward(int act, void* dx, float* dw, float* db, float* dxsum,
                               const void* dout, const void* x, const void* w, const float* mean,
                               const float* rstd, int N, int C, bool accum_dx, void* scratch,
                               cudaStream_t s);
// its row kernel alone: partials [nparts][(dxsum ? 3 : 2) * C] (dw | db |
// dxsum columns) into part (layernorm_backward_scratch bytes)
cudaError_t layernorm_backward_rows(int act, void* dx, bool dxsum, const void* dout,
                                    const void* x, const void* w, const float* mean,
                                    const float* rstd, int N, int C, bool accum_dx, float* part,
                                    int* nparts, cudaStream_t s);

// ---- bias gradient: db[o] += sum_n dout[n,o] (deterministic, two stage) ---
size_t bias_grad_scratch(int N, int OC);
// db[c] += sum_{i < nparts} part[i * ncols + c], rows in order (one launch)
cudaError_t colsum_add(float* db, const float* part, int nparts, int ncols, cudaStream_t s);
// Deferred column sums.  The *_rows producers write their per-block column
// partials [nparts][ncols] into a caller's region and report nparts; one
// colsum_batch call then adds every task's sums into its outputs: out[k][c]
// += sum_i part[i * ncols + k * n0 + c] (k < ncols / n0), the same order of
// additions as the immediate forms.
struct ColsumTask {
    const float* part;
    float* out[3];
    int nparts, ncols, n0;
};
cudaError_t colsum_batch(const ColsumTask* tasks, int n, cudaStream_t s, int* nlaunch);
// the bias gradient's row kernel alone: partials [nparts][OC], nparts <= ceil(N / 64)
cudaError_t bias_grad_rows(int act, float* part, const void* dout, int N, int OC, int* nparts,
                           cudaStream_t s);
cudaError_t bias_grad(int act, float* db, const void* dout, int N, int OC, void* scratch,
                      cudaStream_t s);

// ---- classifier: loss per row + dlogits in place ----------------------------
// logits [N,Vp]; losses[n] = lse(logits[n,:V]) - logits[n,tgt]; if dloss != 0
// the row is overwritten by (softmax - onehot)*dloss (pad columns -> 0).
cudaError_t crossentropy_fused(int act, void* logits, float* losses, const int* tgt, int N,
                               int V, int Vp, float dloss, unsigned* err, cudaStream_t s);
// out[0] = mean(x[0..n)) in a fixed summation order (one block).
cudaError_t mean_reduce(float* out, const float* x, int n, cudaStream_t s);

// ---- AdamW ------------------------------------------------------------------
struct AdamArgs {
    float lr, b1, b2, eps, wd;
    float bc1, bc2;          // 1 - b1^t, 1 - b2^t
    float inv_accum, clip;
    const int* d_count;           // if not NULL: the divisor is *d_count (on the device)
    size_t dec_lo[5], dec_hi[5];  // decayed index ranges [lo, hi)
    int t;                        // this update's step count (1-based)
    uint64_t sr_seed;             // stochastic-rounding stream (bf16-only parameters)
    size_t base;                  // canonical index of the first element updated (a shard)
    size_t n_total;               // length of the whole canonical vector
};
size_t adamw_scratch();
// state[0] = norm, state[1] = total gradient scale, state[2] = finite flag
cudaError_t adamw_step(float* w, float* m, float* v, const float* g, void* wbf16, size_t n,
                       const AdamArgs& a, float* state, void* scratch, cudaStream_t s);
// the two halves of adamw_step: the norm pass (fills state) and the update
cudaError_t adamw_norm(const float* g, size_t n, const AdamArgs& a, float* state, void* scratch,
                       cudaStream_t s);
cudaError_t adamw_update(float* w, float* m, float* v, const float* g, void* wbf16, size_t n,
                         const AdamArgs& a, const float* state, cudaStream_t s);
// the whole AdamW step in one cooperative launch: the global norm and clip
// scale over g[0, n_total), the update of the n_upd elements at w, m, v (g
// read from g + lo; a.base = the canonical index of the first), the bf16 copy
// refreshed (sr: parameters only in bf16, stochastic rounding at wbf16).
// Results are bit for bit those of adamw_norm + adamw_update.  scratch: at
// least adamw_fused_scratch() bytes; bar: two words that are zero before the
// first launch (the kernel leaves them so).
size_t adamw_fused_scratch();
cudaError_t adamw_fused(float* w, float* m, float* v, const float* g, void* wbf16,
                        size_t n_total, size_t lo, size_t n_upd, bool sr, const AdamArgs& a,
                        float* state, void* scratch, unsigned* bar, unsigned* err,
                        cudaStream_t s);
// out[i] = gelu(in[i]) for i < n (dtype act), the fused epilogue's formula
cudaError_t gelu_forward(int act, void* out, const void* in, size_t n, cudaStream_t s);
// parameters held only in bf16: AdamW in fp32, stochastic rounding back
cudaError_t adamw_update_bf16_sr(void* wbf16, float* m, float* v, const float* g, size_t n,
                                 const AdamArgs& a, const float* state, cudaStream_t s);
// out[i] = stochastic rounding of in[i] to bf16 with counter k0 + i of `seed`
cudaError_t stochastic_round_bf16(void* out, const float* in, size_t n, uint64_t seed,
                                  uint64_t k0, cudaStream_t s);
// acc[0] += x[0] on the device
cudaError_t accumulate_scalar(float* acc, const float* x, cudaStream_t s);

// ---- SIMT matmul (fp32 FFMA) ----------------------------------------------
enum Epi {
    EPI_STORE = 0,      // D = acc (+ bias)
    EPI_GELU = 1,       // aux = acc + bias; D = gelu(aux)
    EPI_RESID = 2,      // D = resid + acc + bias
    EPI_ACCUM_F32 = 3,  // D(fp32) += acc
    EPI_GELU_BWD = 4,   // D = acc * gelu'(aux)
    EPI_GELU_D = 5,     // x = acc + bias; D = gelu(x), aux = gelu'(x)
    EPI_MUL_AUX = 6     // D = acc * aux  (aux holding gelu' from EPI_GELU_D)
};
struct GemmDesc {
    int M, N, K;
    const void* A; long lda; int a_kmajor;  // A[m,k] at m*lda+k (K-major) or k*lda+m
    const void* B; long ldb; int b_kmajor;  // B[n,k] at n*ldb+k (K-major) or k*ldb+n
    void* D; long ldd;                      // D[m,n] at m*ldd+n
    const void* bias;                       // [N] act type, or NULL
    const void* resid; long ldr;            // EPI_RESID
    void* aux; long ldx;  // out: EPI_GELU, EPI_GELU_D; in: EPI_GELU_BWD, EPI_MUL_AUX
    int epi;
    int act;                                // element type of A, B, bias, resid, aux, D (non-accum)
    // EPI_MUL_AUX / EPI_GELU_BWD on the tensor cores only, else NULL:
    // dbias[n] += sum_m D[m,n] (D's bf16 values, summed in fp32)
    float* dbias;
    // instead of dbias (same modes): the column sums of each 32-row block,
    // [ceil(M/32)][N], written here for a later colsum_batch
    float* colpart;
};
cudaError_t gemm_simt(const GemmDesc& d, cudaStream_t s);

// ---- attention (causal, softmax(Q K^T / sqrt(hd)) V) --------------------------
// qkv [B,T,3C]; out [B,T,C]; lse [B,H,T] fp32.  bf16 with head size 64 runs
// on the tensor cores (k_attn_tc.cu), everything else on the FFMA kernels.
// err (may be NULL) receives GPT2_DEVERR_TIMEOUT from a bounded wait.
cudaError_t attention_forward(int act, void* out, float* lse, const void* qkv, int B, int T,
                              int C, int H, unsigned* err, cudaStream_t s);
bool attention_tc_supported(int act, int B, int T, int C, int H, const void* qkv);
cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C,
                                 int H, unsigned* err, cudaStream_t s);
cudaError_t attention_backward_tc(void* dqkv, const void* dout, const void* qkv, const void* out,
                                  const float* lse, float* Dv, int B, int T, int C, int H,
                                  unsigned* err, cudaStream_t s);
void* tc_encode_fn();
size_t attention_backward_scratch(int B, int T, int H);
// dqkv [B,T,3C] is overwritten
cudaError_t attention_backward(int act, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T, int C, int H,
                               void* scratch, unsigned* err, cudaStream_t s);

}  // namespace gk
