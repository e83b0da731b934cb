/*
 * gpt2.h -- C-ABI of libgpt2b300, one GPT-2 training step on one B300 (sm_103a).
 *
 * The step is the one described on "Karpathy's llm.c: understanding LLM
 * training from scratch in C/CUDA", section "Code anatomy": token+position
 * embedding, pre-LN transformer blocks (LayerNorm, fused QKV projection,
 * causal multi-head softmax attention, output projection + residual, 4C MLP
 * with tanh-GELU + residual), final LayerNorm, a classifier tied to the token
 * embedding with softmax cross-entropy, the hand-derived backward pass in
 * reverse graph order, and one AdamW update over fp32 master weights
 * ("Karpathy reproduces GPT-2 (1.6B) in llm.c", section "Training" and its
 * flag guide: AdamW, weight decay 0.1 on 2-D weights, gradient clipping,
 * gradient accumulation, vocabulary padded 50257 -> 50304).
 *
 * Conventions shared by every call
 *  - Every call takes the handle made by gpt2_create and returns an int status
 *    (GPT2_OK or a negative GPT2_ERR_*); gpt2_last_error() gives a sentence.
 *  - All GPU work is enqueued on the handle's CUDA stream (the `stream`
 *    argument of gpt2_create, a cudaStream_t; NULL = the legacy default
 *    stream).  Calls return without waiting unless stated otherwise.
 *  - Device pointers ("d_" prefix) must point to memory on the handle's
 *    device; host pointers ("h_" prefix) to ordinary or pinned host memory.
 *  - A handle is not thread-safe: one host thread at a time.
 *  - The handle owns all model state: parameters, gradients, optimizer state
 *    and activations live in one device workspace, either allocated once by
 *    gpt2_create or supplied by the caller.  Token buffers stay the caller's.
 *
 * Canonical parameter order (weights out x in, row-major), used by every
 * get/set call:  wte[Vp,C] wpe[T,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C]
 * qkvb[L,3C] projw[L,C,C] projb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C]
 * fcb[L,4C] fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C],
 * where Vp = V rounded up to a multiple of 128 (padded rows are 0 and stay 0).
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gpt2 gpt2_t;

/* Arithmetic modes.
 *  GPT2_FP32: parameters, activations and gradients in fp32, every matmul and
 *             attention product with fp32 FFMA (no TF32).  This is the parity
 *             mode, checked against the CPU oracle.
 *  GPT2_BF16: fp32 master weights, AdamW state and gradients; bf16 compute
 *             copies of the weights and bf16 activations; tensor-core
 *             contractions with fp32 accumulation; fp32 LayerNorm statistics,
 *             softmax, loss.  This is the mixed-precision training mode of
 *             "Karpathy's llm.c ...", section "Code anatomy", item 3. */
enum { GPT2_FP32 = 0, GPT2_BF16 = 1 };
/* Activation recompute, OR-ed into `mode` ("Karpathy reproduces GPT-2 (1.6B)
 * in llm.c", "Parameter guide" -r 1 / -r 2: recompute in the backward to save
 * memory).
 *  GPT2_RECOMPUTE_GELU: the MLP keeps only x = ln2 Wfc^T + b per layer; gelu(x)
 *    lives in one buffer shared by all layers, filled by an elementwise GELU
 *    kernel in the forward and refilled by the same kernel in the backward
 *    (bit-identical), and the fcproj input gradient takes gelu'(x) from x.
 *    Saves L-1 activations of B*T*4C.
 *  GPT2_RECOMPUTE_LN (implies the above): the two LayerNorm outputs of each
 *    layer are not kept either; the backward reruns the LayerNorm forward on
 *    the kept residual stream (bit-identical).  Saves 2(L-1) of B*T*C more.
 * In fp32 mode a recompute run is bit for bit the same as a run without. */
enum { GPT2_RECOMPUTE_GELU = 0x10, GPT2_RECOMPUTE_LN = 0x20 };
/* Parameters without fp32 master weights, OR-ed into GPT2_BF16 ("Karpathy
 * reproduces GPT-2 (1.6B) in llm.c", "Parameter guide" -w 0): the parameters
 * exist only in bf16 (4 bytes/parameter less); AdamW (moments fp32) computes
 * each new value in fp32 from the widened bf16 value and rounds it back
 * stochastically: update t rounds parameter i with counter (t-1)*N + i of the
 * SplitMix64 stream of seed ^ 0x5352000000000000 (the rounding rule of
 * gpt2k_stochastic_round_bf16).  get/set_params widen exactly / round to
 * nearest even; checkpoints hold the widened values. */
enum { GPT2_NO_MASTER = 0x40 };

enum {
    GPT2_OK = 0,
    GPT2_ERR_ARG = -1,          /* bad argument or unsupported shape            */
    GPT2_ERR_CUDA = -2,         /* a CUDA runtime/driver call failed            */
    GPT2_ERR_OOM = -3,          /* device allocation failed                     */
    GPT2_ERR_STATE = -4,        /* call out of order (e.g. backward w/o forward)*/
    GPT2_ERR_TOKEN_RANGE = -5,  /* a token or target id outside [0, V)          */
    GPT2_ERR_NONFINITE = -6,    /* gradient norm not finite: update skipped     */
    GPT2_ERR_TIMEOUT = -7,      /* a bounded device-side wait ran out           */
    GPT2_ERR_IO = -8            /* a checkpoint file could not be read/written  */
};

/* Bytes of device workspace a handle of this shape needs (0 if the shape is
 * rejected).  Shape limits: C % H == 0; in GPT2_BF16 mode C % 8 == 0; the
 * attention head size C/H is at most 128. */
size_t gpt2_workspace_bytes(int L, int H, int C, int V, int T, int B, int mode);

/* Make a model with L layers, H heads, width C, vocabulary V (padded
 * internally to Vp), context T and micro-batch B.  Parameters are initialised
 * from `seed`: matrices and both embeddings ~ N(0, 0.02), the two residual
 * projections (projw, fcprojw) ~ N(0, 0.02/sqrt(2L)), biases 0, LayerNorm
 * gains 1; element i of the canonical vector uses SplitMix64 outputs 2i and
 * 2i+1 for a Box-Muller normal.
 *   workspace: NULL -> the library cudaMallocs gpt2_workspace_bytes() once and
 *              frees it in gpt2_destroy; else a device buffer of ws_bytes
 *              (>= gpt2_workspace_bytes, 256-byte aligned) that the caller
 *              keeps alive until gpt2_destroy.
 *   stream:    cudaStream_t to enqueue on.
 * Synchronises the stream once (initialisation).  On failure *out = NULL. */
int gpt2_create(gpt2_t** out, int L, int H, int C, int V, int T, int B, uint64_t seed,
                int mode, void* workspace, size_t ws_bytes, void* stream);

void gpt2_destroy(gpt2_t* g);
const char* gpt2_last_error(gpt2_t* g);

/* Change the stream later calls enqueue on. */
int gpt2_set_stream(gpt2_t* g, void* stream);

/* Forward pass over one micro-batch: d_tokens and d_targets are int32 [B,T]
 * on the device.  d_targets NULL: logits only (readable by gpt2_get_logits),
 * no loss, and gpt2_backward is refused.  With targets the mean
 * cross-entropy over the B*T positions is computed and the logits buffer is
 * overwritten in place by d(loss)/d(logits) for the backward pass (the
 * probabilities are never stored).  h_loss NULL: stay asynchronous (the loss
 * stays on the device, gpt2_get_loss reads it); else synchronise and write
 * the loss.  Out-of-range ids are flagged on the device and reported as
 * GPT2_ERR_TOKEN_RANGE at the next synchronising call. */
int gpt2_forward(gpt2_t* g, const int32_t* d_tokens, const int32_t* d_targets, float* h_loss);

/* As gpt2_forward, with tokens/targets in host memory: copies them into the
 * handle's own device buffers (cudaMemcpyAsync on the handle's stream), then
 * runs the same forward pass. h_targets may be NULL. */
int gpt2_forward_host(gpt2_t* g, const int32_t* h_tokens, const int32_t* h_targets,
                      float* h_loss);

/* Backward pass of the last forward (which must have had targets):
 * gradients += d(mean micro-batch loss)/d(params); the micro-batch counter
 * n_accum is incremented.  Asynchronous. */
int gpt2_backward(gpt2_t* g);

/* One AdamW step on the accumulated gradients.  The gradient used is the mean
 * over the n_accum micro-batches, g/n_accum; its global L2 norm n over all
 * parameters is computed; if clip > 0 and n > clip every gradient is scaled
 * by clip/n.  Then m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2, and
 * w -= lr (m_hat / (sqrt(v_hat) + eps) + wd w [w is a 2-D weight: wte, wpe,
 * qkvw, projw, fcw, fcprojw]), with bias corrections 1-b1^t, 1-b2^t and t the
 * 1-based step count.  In GPT2_BF16 mode the bf16 compute copy is refreshed
 * (round to nearest even).  Synchronises.  A non-finite n leaves every state
 * unchanged and returns GPT2_ERR_NONFINITE.  h_grad_norm (optional) gets n.
 * Gradients are left as they are (call gpt2_zero_grad). */
int gpt2_adamw_step(gpt2_t* g, float lr, float b1, float b2, float eps, float wd, float clip,
                    float* h_grad_norm);

/* gradients = 0, n_accum = 0.  Asynchronous. */
int gpt2_zero_grad(gpt2_t* g);

/* Wait for the stream, then report any error flagged on the device. */
int gpt2_sync(gpt2_t* g);

/* ---- inspection (synchronise; fp32 host buffers, canonical order) ---- */
size_t gpt2_num_params(gpt2_t* g);      /* stored count, padded vocabulary */
int gpt2_padded_vocab(gpt2_t* g);
int gpt2_get_params(gpt2_t* g, float* h_buf);       /* master weights        */
int gpt2_set_params(gpt2_t* g, const float* h_buf); /* also refreshes bf16   */
int gpt2_get_grads(gpt2_t* g, float* h_buf);        /* accumulated, not /n   */
int gpt2_set_grads(gpt2_t* g, const float* h_buf);
int gpt2_get_opt_state(gpt2_t* g, float* h_m, float* h_v, int* h_step);
/* AdamW first/second moments and the step count t (m, v: fp32, canonical
 * order, either may be NULL to leave it unchanged; step >= 0). */
int gpt2_set_opt_state(gpt2_t* g, const float* h_m, const float* h_v, int step);
/* ---- update skipping on loss / gradient-norm spikes ("Karpathy reproduces
 * GPT-2 (1.6B) in llm.c", "Training": the flags -sl 5.0 -sg 5.0 skip the
 * update on transient instabilities).  With the detector on, gpt2_adamw_step
 * computes the step's mean micro-batch loss (the losses of the forwards
 * followed by gpt2_backward since the last gpt2_zero_grad) and the gradient
 * norm, their z-scores against the previous `window` steps ((x - mean)/std,
 * population std; no z until `window` steps are recorded), and skips the
 * update -- parameters, moments and step count unchanged -- when a z-score
 * exceeds its threshold.  Every step's values are recorded, skipped or not.
 * loss_z, grad_z <= 0 switch a criterion off; window 0 switches the detector
 * off (the default); window 1 is rejected (GPT2_ERR_ARG).  Setting it clears
 * the recorded window. */
int gpt2_set_spike_skip(gpt2_t* g, float loss_z, float grad_z, int window);
/* outcome of the last gpt2_adamw_step: skipped (0/1) and the two z-scores
 * (NaN when the detector is off or its window is not yet full) */
int gpt2_last_step_info(gpt2_t* g, int* skipped, float* z_loss, float* z_grad);

/* ---- data parallelism ("Karpathy reproduces GPT-2 (1.6B) in llm.c",
 * "Training": one process per GPU, gradients averaged over the ranks, the
 * optimizer state sharded ZeRO-1 style, -z 1).  One step on R ranks: every
 * rank runs its micro-batches (forward + backward), sums the gradient vectors
 * of all ranks into each (an all-reduce over gpt2_grads_buffer), sets the
 * divisor to the micro-batch count summed over the ranks (gpt2_set_grad_count
 * from the host, or gpt2_set_grad_count_device from a device word that a
 * collective summed), applies gpt2_adamw_step_shard to its own slice [lo, hi)
 * of the canonical vector -- the global norm and clip come from the whole
 * summed gradient, so every rank takes the same decision -- and the ranks then
 * gather the updated slices of the parameters the forward reads (the bf16
 * copy in GPT2_BF16 mode, the fp32 parameters in GPT2_FP32 mode: the d_bf16 or
 * d_master pointer of gpt2_params_buffer).  The collectives are the caller's
 * (NCCL through torch.distributed in the binding's DataParallel).  Device
 * pointers stay valid for the handle's life. */
int gpt2_grads_buffer(gpt2_t* g, float** d_grads, size_t* n);
/* d_master: the fp32 parameters -- NULL without master weights and on a
 * sharded bf16 handle (which holds only its slice of them); d_bf16: NULL in
 * GPT2_FP32 mode.  *n = the number of parameters N. */
int gpt2_params_buffer(gpt2_t* g, float** d_master, void** d_bf16, size_t* n);
int gpt2_get_grad_count(gpt2_t* g, int* count);
int gpt2_set_grad_count(gpt2_t* g, int count);  /* count >= 1 */
/* The next update (gpt2_adamw_step or gpt2_adamw_step_shard) divides by the
 * int32 at d_count (device memory of the handle's device, 4-byte aligned),
 * read by the update's kernels in stream order -- so a count summed over the
 * ranks by a collective never has to come back to the host.  The setting
 * serves that one update, which clears it whatever its outcome; the host
 * count (gpt2_get_grad_count) is left as it was.  A count of 0 on the device
 * makes the norm non-finite: the update is skipped with GPT2_ERR_NONFINITE. */
int gpt2_set_grad_count_device(gpt2_t* g, const int* d_count);
/* AdamW on [lo, hi) of the canonical vector (lo a multiple of 4, hi a
 * multiple of 4 or N); the step count advances.  On a sharded handle [lo, hi)
 * must be its own slice.  GPT2_ERR_STATE with the spike detector on (its
 * decision needs every rank's loss).  After a failed update (a non-finite
 * norm) the gradient buffer still holds what the caller put there (after an
 * all-reduce: the sum over the ranks): call gpt2_zero_grad before the next
 * micro-batches. */
int gpt2_adamw_step_shard(gpt2_t* g, size_t lo, size_t hi, float lr, float b1, float b2,
                          float eps, float wd, float clip, float* h_grad_norm);
/* ZeRO-1 handles.  gpt2_create_shard is gpt2_create for a rank that owns the
 * canonical slice [lo, hi) (lo a multiple of 4, hi a multiple of 4 or N): the
 * handle holds the AdamW moments m, v of the slice alone and, in GPT2_BF16
 * mode with master weights, the fp32 master of the slice alone (the forward
 * reads the full bf16 copy; in GPT2_FP32 mode the fp32 parameters are what the
 * forward reads, so they stay whole).  Per rank that saves 8 (N - (hi - lo))
 * bytes of moments, plus 4 (N - (hi - lo)) of master in GPT2_BF16 mode, against
 * gpt2_workspace_bytes (the pages' 1558M run keeps 1/8 of m, v and the master
 * on each of 8 GPUs).  On such a handle: gpt2_adamw_step returns
 * GPT2_ERR_STATE (use gpt2_adamw_step_shard on [lo, hi)); gpt2_get_params
 * returns the parameters the forward reads (in GPT2_BF16 mode the bf16 copy,
 * widened); gpt2_set_params sets the bf16 copy (rounded to nearest even) and
 * the slice's master; gpt2_get/set_opt_state move hi - lo moments each;
 * checkpoints return GPT2_ERR_STATE (a rank holds only its slice).
 * gpt2_workspace_bytes_shard returns 0 for a shape or slice it rejects. */
size_t gpt2_workspace_bytes_shard(int L, int H, int C, int V, int T, int B, int mode, size_t lo,
                                  size_t hi);
int gpt2_create_shard(gpt2_t** out, int L, int H, int C, int V, int T, int B, uint64_t seed,
                      int mode, size_t lo, size_t hi, void* workspace, size_t ws_bytes,
                      void* stream);
/* [lo, hi) of a sharded handle; [0, N) otherwise */
int gpt2_shard_bounds(gpt2_t* g, size_t* lo, size_t* hi);
/* the fp32 master of the handle's slice (hi - lo values; the whole vector on
 * an unsharded handle); GPT2_ERR_STATE without master weights */
int gpt2_get_shard_master(gpt2_t* g, float* h);

/* ---- checkpoints: a file with the fp32 parameters, the AdamW moments and
 * step count, and the spike detector's settings and window (this library's
 * own format: an 88-byte header "GPT2B3CK", version 1, L H C V T mode,
 * nparams, t, detector state, the handle's seed (the stochastic-rounding
 * stream of GPT2_NO_MASTER continues from it); then params, m, v as fp32 in
 * canonical order and
 * the detector's two windows as float64).  A handle of the same L, H, C, V and
 * T (any B, any mode) that loads it continues training bit for bit as the
 * saving handle would have ("Karpathy reproduces GPT-2 (1.6B) in llm.c",
 * "Training": -n saves checkpoints, -y 1 resumes bit-exactly).  Errors:
 * GPT2_ERR_IO (open/read/write, not a checkpoint, truncated), GPT2_ERR_ARG (the
 * checkpoint's shapes differ from the handle's). */
int gpt2_save_checkpoint(gpt2_t* g, const char* path);
int gpt2_load_checkpoint(gpt2_t* g, const char* path);

/* logits [B,T,V] of the last forward WITHOUT targets (real columns only) */
int gpt2_get_logits(gpt2_t* g, float* h_buf);
int gpt2_get_loss(gpt2_t* g, float* h_loss);        /* mean loss, last fwd  */
int gpt2_get_losses(gpt2_t* g, float* h_buf);       /* per position [B,T]   */

/* ---- per-kernel timing (CUDA events on the handle's stream) ----
 * gpt2_prof_enable(g, mask): bit c of mask turns on timing of class c (0 turns
 * all timing off).  Every launch of an enabled class is bracketed by events;
 * gpt2_prof_read sums the elapsed times since the last reset.  Classes are
 * numbered 0..gpt2_prof_num_classes()-1 and named by gpt2_prof_name().
 * flops / bytes are the ALGORITHMIC work of the counted launches (model
 * flops for contractions; compulsory HBM bytes for the rest). */
int gpt2_prof_enable(gpt2_t* g, unsigned class_mask);
int gpt2_prof_reset(gpt2_t* g);
int gpt2_prof_num_classes(void);
const char* gpt2_prof_name(int cls);
int gpt2_prof_read(gpt2_t* g, int cls, double* ms, long long* launches, double* flops,
                   double* bytes);

/* Number of CUDA kernels this handle has launched since gpt2_create
 * (memsets and copies are not counted). */
long long gpt2_launch_count(gpt2_t* g);

#ifdef __cplusplus
}
#endif
#endif
