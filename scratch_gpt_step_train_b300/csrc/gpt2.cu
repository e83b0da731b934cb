// gpt2.cu -- host orchestration of the GPT-2 training step behind the C-ABI
// declared in include/gpt2.h: workspace planning (one allocation), the launch
// sequence of the forward pass, the backward pass in reverse graph order,
// the AdamW step, error reporting and per-kernel event timing.
//
// The order of operations follows "Karpathy's llm.c: understanding LLM
// training from scratch in C/CUDA", "Code anatomy" (encoder -> per-layer
// layernorm / attention / MLP -> classifier; backward from d(loss)/d(logits)
// back through every layer; one parameter-update kernel), and the gradient
// accumulation / AdamW / clipping of "Karpathy reproduces GPT-2 (1.6B) in
// llm.c", "Training".
#include "../../include/gpt2.h"
#include "kernels.h"
#include "gemm_tc.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

using namespace gk;

// ---------------------------------------------------------------------------
// kernel classes for event timing
// ---------------------------------------------------------------------------
enum {
    // linear layers, one class per (layer, direction)
    K_QKV_FWD, K_PROJ_FWD, K_FC_FWD, K_FCPROJ_FWD, K_CLS_FWD,
    K_QKV_DX, K_PROJ_DX, K_FC_DX, K_FCPROJ_DX, K_CLS_DX,
    K_QKV_DW, K_PROJ_DW, K_FC_DW, K_FCPROJ_DW, K_CLS_DW,
    K_ATTN_FWD, K_ATTN_BWD, K_LN_FWD, K_LN_BWD, K_XENT, K_EMB_FWD, K_EMB_BWD, K_BIAS, K_ADAM,
    K_ZERO, K_RECOMP, K_COLSUM, K_NCLASS
};
static const char* kClassNames[K_NCLASS] = {
    "matmul_qkv_fwd", "matmul_proj_fwd", "matmul_fc_fwd", "matmul_fcproj_fwd",
    "matmul_classifier_fwd", "matmul_qkv_dx", "matmul_proj_dx", "matmul_fc_dx",
    "matmul_fcproj_dx", "matmul_classifier_dx", "matmul_qkv_dw", "matmul_proj_dw",
    "matmul_fc_dw", "matmul_fcproj_dw", "matmul_classifier_dw", "attention_fwd",
    "attention_bwd", "layernorm_fwd", "layernorm_bwd", "crossentropy", "embedding_fwd",
    "embedding_bwd", "bias_grad", "adamw", "zero_grad", "recompute", "grad_colsum"};

struct ProfRec {
    int cls;
    cudaEvent_t a, b;
    double flops, bytes;
};

struct gpt2 {
    int L, H, C, V, Vp, T, B, mode, act;
    int recompute;  // 0: keep all activations; 1: GELU output recomputed; 2: and LN outputs
    bool no_master;  // parameters only in bf16, updated with stochastic rounding
    uint64_t seed;
    size_t BT;
    ParamLayout lay;
    size_t nparams;
    cudaStream_t stream;
    void* ws;
    bool own_ws;
    size_t ws_bytes;
    bool use_tc;  // tensor-core GEMMs (bf16 mode)
    int device;   // CUDA device of the workspace

    float *master, *grads, *m, *v;
    void* pc;  // compute copy of the parameters (== master in fp32 mode)
    // ZeRO-1 shard: the handle holds the AdamW moments (and, in bf16 mode,
    // the fp32 master) of the canonical slice [sh_lo, sh_hi) only
    bool sharded = false;
    size_t sh_lo = 0, sh_hi = 0;
    // the micro-batch count of the next update, read on the device (NULL: n_accum)
    const int* d_count = nullptr;
    // elements of the moment buffers, and of the master buffer
    size_t n_state() const { return sharded ? sh_hi - sh_lo : nparams; }
    bool master_sliced() const { return sharded && act == ACT_BF16 && !no_master; }
    // activations
    void *encoded, *ln1, *qkv, *atty, *x1, *ln2, *fch, *fchg, *x2, *lnf, *logits;
    float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lnf_mean, *lnf_rstd, *lse, *losses;
    float* loss;
    // backward buffers
    void *dres, *dbig, *dln, *datty, *dqkv;
    void* scratch;
    size_t scratch_bytes;
    // column partials of the LayerNorm-weight and bias gradients of one
    // backward pass, one region per producer, summed by one batched launch
    // at its end: (2L+1) LayerNorm regions, then L qkv-bias, then L fc-bias
    float* dpart;
    size_t ln_part_bytes, qkvb_part_bytes, fcb_part_bytes;
    std::vector<ColsumTask> ctasks;
    int32_t *tok, *tgt;
    unsigned* err;
    float* adam_state;
    unsigned* adam_bar;  // grid-barrier words of the single-launch AdamW (zero between launches)

    int n_accum, t, have_targets, logits_valid, have_fwd;
    std::string last_err;

    // update skipping on loss / gradient-norm spikes: z-scores of this step's
    // mean loss and gradient norm against the previous sk_window steps
    float sk_loss_z = 0.f, sk_grad_z = 0.f;  // thresholds (<= 0: criterion off)
    int sk_window = 0;                       // 0: detector off
    int sk_count = 0, sk_pos = 0;            // values recorded (<= window), ring position
    std::vector<double> sk_loss_hist, sk_grad_hist;
    int last_skipped = 0;
    float last_zl = NAN, last_zg = NAN;

    long long launches;  // kernels launched by this handle
    unsigned prof_mask;  // classes timed with events
    bool prof_on, prof_cur;
    std::vector<ProfRec> prof;
    size_t prof_used;
    double prof_ms[K_NCLASS], prof_flops[K_NCLASS], prof_bytes[K_NCLASS];
    long long prof_n[K_NCLASS];
};

static int fail(gpt2* g, int code, const char* fmt, ...) {
    if (g) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        g->last_err = buf;
    }
    return code;
}

#define CK(expr)                                                                         \
    do {                                                                                 \
        cudaError_t e_ = (expr);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return fail(g, GPT2_ERR_CUDA, "%s: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                             \
    } while (0)

// ---------------------------------------------------------------------------
// event timing around one launch group
// ---------------------------------------------------------------------------
static void prof_begin(gpt2* g, int cls, double flops, double bytes) {
    g->prof_cur = g->prof_on && ((g->prof_mask >> cls) & 1u);
    if (!g->prof_cur) return;
    if (g->prof_used == g->prof.size()) {
        ProfRec r;
        cudaEventCreate(&r.a);
        cudaEventCreate(&r.b);
        g->prof.push_back(r);
    }
    ProfRec& r = g->prof[g->prof_used];
    r.cls = cls;
    r.flops = flops;
    r.bytes = bytes;
    cudaEventRecord(r.a, g->stream);
}
static void prof_end(gpt2* g) {
    if (!g->prof_cur) return;
    cudaEventRecord(g->prof[g->prof_used].b, g->stream);
    g->prof_used++;
}
static void prof_collect(gpt2* g) {
    if (g->prof_used == 0) return;
    cudaEventSynchronize(g->prof[g->prof_used - 1].b);
    for (size_t i = 0; i < g->prof_used; i++) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, g->prof[i].a, g->prof[i].b);
        int c = g->prof[i].cls;
        g->prof_ms[c] += ms;
        g->prof_flops[c] += g->prof[i].flops;
        g->prof_bytes[c] += g->prof[i].bytes;
        g->prof_n[c] += 1;
    }
    g->prof_used = 0;
}

// ---------------------------------------------------------------------------
// workspace plan
// ---------------------------------------------------------------------------
struct Planner {
    char* base;
    size_t off;
    void* take(size_t bytes) {
        void* p = base ? base + off : nullptr;
        off += (bytes + 255) & ~(size_t)255;
        return p;
    }
};

static size_t scratch_need(int L, int H, int C, int Vp, int T, int B) {
    size_t BT = (size_t)B * T;
    size_t s = layernorm_backward_scratch((int)BT, C, true);
    size_t x;
    if ((x = bias_grad_scratch((int)BT, 4 * C)) > s) s = x;
    if ((x = encoder_backward_scratch(B, T, C, Vp)) > s) s = x;
    if ((x = attention_backward_scratch(B, T, H)) > s) s = x;
    if ((x = adamw_scratch()) > s) s = x;
    if ((x = adamw_fused_scratch()) > s) s = x;
    if ((x = gemm_tc_scratch_bytes()) > s) s = x;
    return s;
}

static void plan(gpt2* g, char* base, size_t* total) {
    Planner p{base, 0};
    size_t N = g->nparams, BT = g->BT, C = g->C, L = g->L;
    size_t as = act_size(g->act);
    const size_t S = g->n_state();
    g->master = g->no_master ? nullptr : (float*)p.take((g->master_sliced() ? S : N) * 4);
    g->grads = (float*)p.take(N * 4);
    g->m = (float*)p.take(S * 4);
    g->v = (float*)p.take(S * 4);
    g->pc = g->act == ACT_BF16 ? p.take(N * 2) : (void*)g->master;
    g->encoded = p.take(BT * C * as);
    // with recompute, one layer's buffer serves every layer (refilled when needed)
    const size_t Lln = g->recompute >= 2 ? 1 : L, Lg = g->recompute >= 1 ? 1 : L;
    g->ln1 = p.take(Lln * BT * C * as);
    g->qkv = p.take(L * BT * 3 * C * as);
    g->atty = p.take(L * BT * C * as);
    g->x1 = p.take(L * BT * C * as);
    g->ln2 = p.take(Lln * BT * C * as);
    g->fch = p.take(L * BT * 4 * C * as);
    g->fchg = p.take(Lg * BT * 4 * C * as);
    g->x2 = p.take(L * BT * C * as);
    g->lnf = p.take(BT * C * as);
    g->logits = p.take(BT * (size_t)g->Vp * as);
    g->ln1_mean = (float*)p.take(L * BT * 4);
    g->ln1_rstd = (float*)p.take(L * BT * 4);
    g->ln2_mean = (float*)p.take(L * BT * 4);
    g->ln2_rstd = (float*)p.take(L * BT * 4);
    g->lnf_mean = (float*)p.take(BT * 4);
    g->lnf_rstd = (float*)p.take(BT * 4);
    g->lse = (float*)p.take(L * (size_t)g->B * g->H * g->T * 4);
    g->losses = (float*)p.take(BT * 4);
    g->loss = (float*)p.take(16);
    g->dres = p.take(BT * C * as);
    g->dbig = p.take(BT * 4 * C * as);
    g->dln = p.take(BT * C * as);
    g->datty = p.take(BT * C * as);
    g->dqkv = p.take(BT * 3 * C * as);
    g->scratch_bytes = scratch_need(g->L, g->H, g->C, g->Vp, g->T, g->B);
    g->scratch = p.take(g->scratch_bytes);
    auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
    g->ln_part_bytes = al(layernorm_backward_scratch((int)BT, (int)C, true));
    g->qkvb_part_bytes = al(bias_grad_scratch((int)BT, (int)(3 * C)));
    g->fcb_part_bytes = al(std::max((BT + 31) / 32 * 4 * C * 4,
                                    bias_grad_scratch((int)BT, (int)(4 * C))));
    g->dpart = (float*)p.take((2 * L + 1) * g->ln_part_bytes +
                              L * (g->qkvb_part_bytes + g->fcb_part_bytes));
    g->tok = (int32_t*)p.take(BT * 4);
    g->tgt = (int32_t*)p.take(BT * 4);
    g->err = (unsigned*)p.take(16);
    g->adam_state = (float*)p.take(16);
    g->adam_bar = (unsigned*)p.take(16);
    *total = p.off;
}

static bool shape_ok(int L, int H, int C, int V, int T, int B, int mode) {
    if (L < 1 || H < 1 || C < 1 || V < 1 || T < 1 || B < 1) return false;
    if (C % H) return false;
    int hd = C / H;
    if (hd != 8 && hd != 16 && hd != 32 && hd != 64 && hd != 128) return false;
    if (mode & ~(0xF | GPT2_RECOMPUTE_GELU | GPT2_RECOMPUTE_LN | GPT2_NO_MASTER)) return false;
    if ((mode & GPT2_NO_MASTER) && (mode & 0xF) != GPT2_BF16) return false;
    mode &= 0xF;
    if (mode != GPT2_FP32 && mode != GPT2_BF16) return false;
    if (mode == GPT2_BF16 && C % 8) return false;
    if ((long)B * T > (1L << 30) / 4) return false;
    if (V >= (1 << 21) - 128) return false;
    if (C > 2048 || (C % 4 && C > 512)) return false;  // LayerNorm register tiling
    return true;
}

static bool shard_ok(size_t n, size_t lo, size_t hi) {
    return lo <= hi && hi <= n && lo % 4 == 0 && (hi % 4 == 0 || hi == n);
}

static size_t workspace_bytes(int L, int H, int C, int V, int T, int B, int mode, bool sharded,
                              size_t lo, size_t hi) {
    if (!shape_ok(L, H, C, V, T, B, mode)) return 0;
    gpt2 tmp;
    tmp.L = L; tmp.H = H; tmp.C = C; tmp.V = V; tmp.T = T; tmp.B = B; tmp.mode = mode;
    tmp.act = (mode & 0xF) == GPT2_BF16 ? ACT_BF16 : ACT_F32;
    tmp.recompute = (mode & GPT2_RECOMPUTE_LN) ? 2 : ((mode & GPT2_RECOMPUTE_GELU) ? 1 : 0);
    tmp.no_master = (mode & GPT2_NO_MASTER) != 0;
    tmp.Vp = ((V + 127) / 128) * 128;
    tmp.BT = (size_t)B * T;
    make_layout(&tmp.lay, L, C, V, T);
    tmp.nparams = tmp.lay.off[P_NUM];
    if (sharded && !shard_ok(tmp.nparams, lo, hi)) return 0;
    tmp.sharded = sharded;
    tmp.sh_lo = lo;
    tmp.sh_hi = hi;
    size_t total;
    plan(&tmp, nullptr, &total);
    return total;
}

extern "C" size_t gpt2_workspace_bytes(int L, int H, int C, int V, int T, int B, int mode) {
    return workspace_bytes(L, H, C, V, T, B, mode, false, 0, 0);
}
extern "C" size_t gpt2_workspace_bytes_shard(int L, int H, int C, int V, int T, int B, int mode,
                                             size_t lo, size_t hi) {
    return workspace_bytes(L, H, C, V, T, B, mode, true, lo, hi);
}

// ---------------------------------------------------------------------------
// create / destroy
// ---------------------------------------------------------------------------
static int create(gpt2_t** out, int L, int H, int C, int V, int T, int B, uint64_t seed, int mode,
                  bool sharded, size_t lo, size_t hi, void* workspace, size_t ws_bytes,
                  void* stream) {
    if (!out) return GPT2_ERR_ARG;
    *out = nullptr;
    if (!shape_ok(L, H, C, V, T, B, mode)) return GPT2_ERR_ARG;
    gpt2* g = new gpt2();
    g->L = L; g->H = H; g->C = C; g->V = V; g->T = T; g->B = B; g->mode = mode;
    g->act = (mode & 0xF) == GPT2_BF16 ? ACT_BF16 : ACT_F32;
    g->recompute = (mode & GPT2_RECOMPUTE_LN) ? 2 : ((mode & GPT2_RECOMPUTE_GELU) ? 1 : 0);
    g->no_master = (mode & GPT2_NO_MASTER) != 0;
    g->seed = seed;
    g->Vp = ((V + 127) / 128) * 128;
    g->BT = (size_t)B * T;
    make_layout(&g->lay, L, C, V, T);
    g->nparams = g->lay.off[P_NUM];
    if (sharded && !shard_ok(g->nparams, lo, hi)) {
        delete g;
        return GPT2_ERR_ARG;
    }
    g->sharded = sharded;
    g->sh_lo = lo;
    g->sh_hi = hi;
    g->stream = (cudaStream_t)stream;
    g->prof_on = false;
    g->prof_cur = false;
    g->prof_mask = 0;
    g->prof_used = 0;
    g->launches = 0;
    size_t need;
    plan(g, nullptr, &need);
    g->device = 0;
    if (workspace) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, workspace) != cudaSuccess ||
            pa.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            delete g;
            return GPT2_ERR_ARG;
        }
        g->device = pa.device;
    } else {
        cudaGetDevice(&g->device);
    }
    cudaSetDevice(g->device);
    if (workspace) {
        if (ws_bytes < need || ((uintptr_t)workspace & 255)) {
            delete g;
            return GPT2_ERR_ARG;
        }
        g->ws = workspace;
        g->own_ws = false;
    } else {
        if (cudaMalloc(&g->ws, need) != cudaSuccess) {
            cudaGetLastError();
            delete g;
            return GPT2_ERR_OOM;
        }
        g->own_ws = true;
    }
    g->ws_bytes = need;
    plan(g, (char*)g->ws, &need);
    g->use_tc = (g->act == ACT_BF16) && gemm_tc_available();
    cudaError_t e;
    do {
        if ((e = cudaMemsetAsync(g->grads, 0, g->nparams * 4, g->stream))) break;
        if ((e = cudaMemsetAsync(g->m, 0, g->n_state() * 4, g->stream))) break;
        if ((e = cudaMemsetAsync(g->v, 0, g->n_state() * 4, g->stream))) break;
        if ((e = cudaMemsetAsync(g->err, 0, 16, g->stream))) break;
        if ((e = cudaMemsetAsync(g->adam_bar, 0, 16, g->stream))) break;
        if (g->no_master || g->master_sliced()) {
            // the fp32 init passes through the gradient buffer: rounded to
            // bf16 for the compute copy, and its slice kept as the master
            if ((e = init_params(g->grads, g->lay, seed, g->stream))) break;
            if ((e = cast_to_bf16(g->pc, g->grads, g->nparams, g->stream))) break;
            if (g->master_sliced() && g->n_state() &&
                (e = cudaMemcpyAsync(g->master, g->grads + lo, g->n_state() * 4,
                                     cudaMemcpyDeviceToDevice, g->stream)))
                break;
            if ((e = cudaMemsetAsync(g->grads, 0, g->nparams * 4, g->stream))) break;
        } else {
            if ((e = init_params(g->master, g->lay, seed, g->stream))) break;
            if (g->act == ACT_BF16 && (e = cast_to_bf16(g->pc, g->master, g->nparams, g->stream)))
                break;
        }
        e = cudaStreamSynchronize(g->stream);
    } while (0);
    if (e != cudaSuccess) {
        if (g->own_ws) cudaFree(g->ws);
        delete g;
        return GPT2_ERR_CUDA;
    }
    *out = g;
    return GPT2_OK;
}

extern "C" int gpt2_create(gpt2_t** out, int L, int H, int C, int V, int T, int B, uint64_t seed,
                           int mode, void* workspace, size_t ws_bytes, void* stream) {
    return create(out, L, H, C, V, T, B, seed, mode, false, 0, 0, workspace, ws_bytes, stream);
}
extern "C" int gpt2_create_shard(gpt2_t** out, int L, int H, int C, int V, int T, int B,
                                 uint64_t seed, int mode, size_t lo, size_t hi, void* workspace,
                                 size_t ws_bytes, void* stream) {
    return create(out, L, H, C, V, T, B, seed, mode, true, lo, hi, workspace, ws_bytes, stream);
}

extern "C" void gpt2_destroy(gpt2_t* g) {
    if (!g) return;
    cudaStreamSynchronize(g->stream);
    for (auto& r : g->prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    if (g->own_ws) cudaFree(g->ws);
    delete g;
}

extern "C" const char* gpt2_last_error(gpt2_t* g) { return g ? g->last_err.c_str() : "null handle"; }

extern "C" int gpt2_set_stream(gpt2_t* g, void* stream) {
    if (!g) return GPT2_ERR_ARG;
    g->stream = (cudaStream_t)stream;
    return GPT2_OK;
}

// Read and clear the device error word (synchronises).
static int check_dev_err(gpt2* g) {
    unsigned e = 0;
    CK(cudaMemcpyAsync(&e, g->err, 4, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    if (e) {
        CK(cudaMemsetAsync(g->err, 0, 4, g->stream));
        if (e & GPT2_DEVERR_TOKEN)
            return fail(g, GPT2_ERR_TOKEN_RANGE, "a token or target id is outside [0, V)");
        if (e & GPT2_DEVERR_TIMEOUT) {
            // a barrier left half-way must start from zero again
            CK(cudaMemsetAsync(g->adam_bar, 0, 16, g->stream));
            return fail(g, GPT2_ERR_TIMEOUT, "a bounded device wait ran out");
        }
        return fail(g, GPT2_ERR_CUDA, "device error word 0x%x", e);
    }
    return GPT2_OK;
}

extern "C" int gpt2_sync(gpt2_t* g) {
    if (!g) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    return check_dev_err(g);
}

// ---------------------------------------------------------------------------
// building blocks
// ---------------------------------------------------------------------------
static void* pc_tensor(gpt2* g, int k, int l) {
    size_t per = g->lay.off[k + 1] - g->lay.off[k];
    if (k >= P_LN1W && k <= P_FCPROJB) per /= g->L;
    return (char*)g->pc + (g->lay.off[k] + (size_t)l * per) * act_size(g->act);
}
static float* grad_tensor(gpt2* g, int k, int l) {
    size_t per = g->lay.off[k + 1] - g->lay.off[k];
    if (k >= P_LN1W && k <= P_FCPROJB) per /= g->L;
    return g->grads + g->lay.off[k] + (size_t)l * per;
}
static void* act_at(gpt2* g, void* base, size_t elems_per_layer, int l) {
    return (char*)base + (size_t)l * elems_per_layer * act_size(g->act);
}

// D[M,N] (epilogue) A[M,K] . B[N,K]^T
static int mm(gpt2* g, int cls, GemmDesc d) {
    d.act = g->act;
    double fl = 2.0 * d.M * d.N * d.K;
    double as = (double)act_size(g->act);
    double by = as * ((double)d.M * d.K + (double)d.N * d.K) +
                (d.epi == EPI_ACCUM_F32 ? 8.0 : as) * d.M * d.N;
    prof_begin(g, cls, fl, by);
    cudaError_t e;
    if (g->use_tc && gemm_tc_supported(d)) {
        int nl = 0;
        e = gemm_tc(d, g->scratch, g->scratch_bytes, g->err, g->stream, &nl);
        g->launches += nl;
    } else {
        e = gemm_simt(d, g->stream);
        g->launches += 1;
    }
    prof_end(g);
    if (e != cudaSuccess)
        return fail(g, GPT2_ERR_CUDA, "matmul M=%d N=%d K=%d epi=%d: %s", d.M, d.N, d.K, d.epi,
                    cudaGetErrorString(e));
    return GPT2_OK;
}

static GemmDesc gd(int M, int N, int K, const void* A, long lda, int akm, const void* Bm, long ldb,
                   int bkm, void* D, long ldd, int epi) {
    GemmDesc d;
    memset(&d, 0, sizeof d);
    d.M = M; d.N = N; d.K = K;
    d.A = A; d.lda = lda; d.a_kmajor = akm;
    d.B = Bm; d.ldb = ldb; d.b_kmajor = bkm;
    d.D = D; d.ldd = ldd; d.epi = epi;
    return d;
}

#define RUN(expr)                      \
    do {                               \
        int rc_ = (expr);              \
        if (rc_ != GPT2_OK) return rc_; \
    } while (0)

#define LAUNCH(cls, nk, fl, by, expr)                                                        \
    do {                                                                                     \
        g->launches += (nk);                                                                 \
        prof_begin(g, cls, fl, by);                                                          \
        cudaError_t e_ = (expr);                                                             \
        prof_end(g);                                                                         \
        if (e_ != cudaSuccess)                                                               \
            return fail(g, GPT2_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));           \
    } while (0)

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
static int forward_impl(gpt2* g, bool with_targets, float* h_loss) {
    int B = g->B, T = g->T, C = g->C, L = g->L, H = g->H, Vp = g->Vp;
    int BT = (int)g->BT;
    size_t as = act_size(g->act);
    size_t c = C, bt = g->BT;
    LAUNCH(K_EMB_FWD, 1, 0, as * 3.0 * bt * c,
           encoder_forward(g->act, g->encoded, g->tok, pc_tensor(g, P_WTE, 0),
                           pc_tensor(g, P_WPE, 0), B, T, C, g->V, g->err, g->stream));
    const void* resid = g->encoded;
    double ln_bytes = as * 2.0 * bt * c + 8.0 * bt;
    const int lln = g->recompute >= 2 ? 0 : 1, lg = g->recompute >= 1 ? 0 : 1;
    for (int l = 0; l < L; l++) {
        void* ln1 = act_at(g, g->ln1, bt * c, l * lln);
        void* qkv = act_at(g, g->qkv, bt * 3 * c, l);
        void* atty = act_at(g, g->atty, bt * c, l);
        void* x1 = act_at(g, g->x1, bt * c, l);
        void* ln2 = act_at(g, g->ln2, bt * c, l * lln);
        void* fch = act_at(g, g->fch, bt * 4 * c, l);
        void* fchg = act_at(g, g->fchg, bt * 4 * c, l * lg);
        void* x2 = act_at(g, g->x2, bt * c, l);
        float* lse = g->lse + (size_t)l * B * H * T;
        LAUNCH(K_LN_FWD, 1, 0, ln_bytes,
               layernorm_forward(g->act, ln1, g->ln1_mean + l * bt, g->ln1_rstd + l * bt, resid,
                                 pc_tensor(g, P_LN1W, l), pc_tensor(g, P_LN1B, l), BT, C,
                                 g->stream));
        GemmDesc d = gd(BT, 3 * C, C, ln1, C, 1, pc_tensor(g, P_QKVW, l), C, 1, qkv, 3 * C,
                        EPI_STORE);
        d.bias = pc_tensor(g, P_QKVB, l);
        RUN(mm(g, K_QKV_FWD, d));
        // causal attention flops: QK^T and PV over the lower triangle
        double afl = 2.0 * 2.0 * B * H * ((double)T * (T + 1) / 2) * (C / H);
        LAUNCH(K_ATTN_FWD, 1, afl, as * 4.0 * bt * c + 4.0 * B * H * T,
               attention_forward(g->act, atty, lse, qkv, B, T, C, H, g->err, g->stream));
        d = gd(BT, C, C, atty, C, 1, pc_tensor(g, P_PROJW, l), C, 1, x1, C, EPI_RESID);
        d.bias = pc_tensor(g, P_PROJB, l);
        d.resid = resid;
        d.ldr = C;
        RUN(mm(g, K_PROJ_FWD, d));
        LAUNCH(K_LN_FWD, 1, 0, ln_bytes,
               layernorm_forward(g->act, ln2, g->ln2_mean + l * bt, g->ln2_rstd + l * bt, x1,
                                 pc_tensor(g, P_LN2W, l), pc_tensor(g, P_LN2B, l), BT, C,
                                 g->stream));
        if (g->recompute >= 1) {
            // keep x = ln2 Wfc^T + b; gelu(x) goes to the shared buffer and is
            // recomputed from x by the same kernel in the backward
            d = gd(BT, 4 * C, C, ln2, C, 1, pc_tensor(g, P_FCW, l), C, 1, fch, 4 * C, EPI_STORE);
            d.bias = pc_tensor(g, P_FCB, l);
            RUN(mm(g, K_FC_FWD, d));
            LAUNCH(K_RECOMP, 1, 0, as * 8.0 * bt * c,
                   gelu_forward(g->act, fchg, fch, bt * 4 * c, g->stream));
        } else {
            d = gd(BT, 4 * C, C, ln2, C, 1, pc_tensor(g, P_FCW, l), C, 1, fchg, 4 * C,
                   EPI_GELU_D);
            d.bias = pc_tensor(g, P_FCB, l);
            d.aux = fch;
            d.ldx = 4 * C;
            RUN(mm(g, K_FC_FWD, d));
        }
        d = gd(BT, C, 4 * C, fchg, 4 * C, 1, pc_tensor(g, P_FCPROJW, l), 4 * C, 1, x2, C,
               EPI_RESID);
        d.bias = pc_tensor(g, P_FCPROJB, l);
        d.resid = x1;
        d.ldr = C;
        RUN(mm(g, K_FCPROJ_FWD, d));
        resid = x2;
    }
    LAUNCH(K_LN_FWD, 1, 0, ln_bytes,
           layernorm_forward(g->act, g->lnf, g->lnf_mean, g->lnf_rstd, resid,
                             pc_tensor(g, P_LNFW, 0), pc_tensor(g, P_LNFB, 0), BT, C, g->stream));
    GemmDesc d = gd(BT, Vp, C, g->lnf, C, 1, pc_tensor(g, P_WTE, 0), C, 1, g->logits, Vp,
                    EPI_STORE);
    RUN(mm(g, K_CLS_FWD, d));
    g->have_targets = with_targets ? 1 : 0;
    g->logits_valid = with_targets ? 0 : 1;
    g->have_fwd = 1;
    if (with_targets) {
        LAUNCH(K_XENT, 1, 0, as * 2.0 * bt * Vp,
               crossentropy_fused(g->act, g->logits, g->losses, g->tgt, BT, g->V, Vp,
                                  1.0f / (float)BT, g->err, g->stream));
        LAUNCH(K_XENT, 1, 0, 4.0 * bt, mean_reduce(g->loss, g->losses, BT, g->stream));
        if (h_loss) {
            RUN(check_dev_err(g));
            CK(cudaMemcpy(h_loss, g->loss, 4, cudaMemcpyDeviceToHost));
        }
    } else if (h_loss) {
        *h_loss = NAN;
        RUN(check_dev_err(g));
    }
    return GPT2_OK;
}

extern "C" int gpt2_forward(gpt2_t* g, const int32_t* d_tokens, const int32_t* d_targets,
                            float* h_loss) {
    if (!g || !d_tokens) return fail(g, GPT2_ERR_ARG, "null handle or tokens");
    cudaSetDevice(g->device);
    CK(cudaMemcpyAsync(g->tok, d_tokens, g->BT * 4, cudaMemcpyDeviceToDevice, g->stream));
    if (d_targets)
        CK(cudaMemcpyAsync(g->tgt, d_targets, g->BT * 4, cudaMemcpyDeviceToDevice, g->stream));
    return forward_impl(g, d_targets != nullptr, h_loss);
}

extern "C" int gpt2_forward_host(gpt2_t* g, const int32_t* h_tokens, const int32_t* h_targets,
                                 float* h_loss) {
    if (!g || !h_tokens) return fail(g, GPT2_ERR_ARG, "null handle or tokens");
    cudaSetDevice(g->device);
    CK(cudaMemcpyAsync(g->tok, h_tokens, g->BT * 4, cudaMemcpyHostToDevice, g->stream));
    if (h_targets)
        CK(cudaMemcpyAsync(g->tgt, h_targets, g->BT * 4, cudaMemcpyHostToDevice, g->stream));
    return forward_impl(g, h_targets != nullptr, h_loss);
}

// ---------------------------------------------------------------------------
// backward (reverse graph order)
// ---------------------------------------------------------------------------
extern "C" int gpt2_backward(gpt2_t* g) {
    if (!g) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    if (!g->have_fwd || !g->have_targets)
        return fail(g, GPT2_ERR_STATE, "backward needs a preceding forward with targets");
    int B = g->B, T = g->T, C = g->C, L = g->L, H = g->H, Vp = g->Vp;
    int BT = (int)g->BT;
    size_t as = act_size(g->act);
    size_t c = C, bt = g->BT;
    void* dres = g->dres;
    // classifier: dlogits sit in the logits buffer
    GemmDesc d = gd(BT, C, Vp, g->logits, Vp, 1, pc_tensor(g, P_WTE, 0), C, 0, g->dln, C,
                    EPI_STORE);
    RUN(mm(g, K_CLS_DX, d));
    d = gd(Vp, C, BT, g->logits, Vp, 0, g->lnf, C, 0, grad_tensor(g, P_WTE, 0), C,
           EPI_ACCUM_F32);
    RUN(mm(g, K_CLS_DW, d));
    const void* xL = L > 0 ? act_at(g, g->x2, bt * c, L - 1) : g->encoded;
    // the residual-stream gradient dres is written (not accumulated) by the
    // final LayerNorm's backward; each LayerNorm backward that feeds a
    // projection's output gradient also yields that projection's bias
    // gradient as the column sums of dres
    double lnb_bytes = as * 4.0 * bt * c + 8.0 * bt;
    // the column sums (LayerNorm weights, biases) of the whole pass are
    // gathered as tasks and summed by one batched launch at its end
    g->ctasks.clear();
    int np = 0;
    auto ln_task = [&](int idx, float* dw, float* db, float* dxsum) {
        float* part = (float*)((char*)g->dpart + (size_t)idx * g->ln_part_bytes);
        g->ctasks.push_back(ColsumTask{part, {dw, db, dxsum}, np, (dxsum ? 3 : 2) * C, C});
        return part;
    };
    char* const qkvb_base = (char*)g->dpart + (size_t)(2 * L + 1) * g->ln_part_bytes;
    char* const fcb_base = qkvb_base + (size_t)L * g->qkvb_part_bytes;
    {
        float* dxs = L > 0 ? grad_tensor(g, P_FCPROJB, L - 1) : nullptr;
        float* part = (float*)g->dpart;
        LAUNCH(K_LN_BWD, 1, 0, as * 3.0 * bt * c + 8.0 * bt,
               layernorm_backward_rows(g->act, dres, dxs != nullptr, g->dln, xL,
                                       pc_tensor(g, P_LNFW, 0), g->lnf_mean, g->lnf_rstd, BT, C,
                                       false, part, &np, g->stream));
        ln_task(0, grad_tensor(g, P_LNFW, 0), grad_tensor(g, P_LNFB, 0), dxs);
    }
    const int lln = g->recompute >= 2 ? 0 : 1, lg = g->recompute >= 1 ? 0 : 1;
    const double ln_bytes = as * 2.0 * bt * c + 8.0 * bt;
    for (int l = L - 1; l >= 0; l--) {
        const void* rin = l == 0 ? g->encoded : act_at(g, g->x2, bt * c, l - 1);
        void* ln1 = act_at(g, g->ln1, bt * c, l * lln);
        void* qkv = act_at(g, g->qkv, bt * 3 * c, l);
        void* atty = act_at(g, g->atty, bt * c, l);
        void* x1 = act_at(g, g->x1, bt * c, l);
        void* ln2 = act_at(g, g->ln2, bt * c, l * lln);
        void* fch = act_at(g, g->fch, bt * 4 * c, l);
        void* fchg = act_at(g, g->fchg, bt * 4 * c, l * lg);
        float* lse = g->lse + (size_t)l * B * H * T;
        // MLP: x2 = x1 + fcproj(gelu(fc(ln2(x1))))
        if (g->recompute >= 1)  // gelu(x) again, by the forward's kernel, from the kept x
            LAUNCH(K_RECOMP, 1, 0, as * 8.0 * bt * c,
                   gelu_forward(g->act, fchg, fch, bt * 4 * c, g->stream));
        d = gd(C, 4 * C, BT, dres, C, 0, fchg, 4 * C, 0, grad_tensor(g, P_FCPROJW, l), 4 * C,
               EPI_ACCUM_F32);
        RUN(mm(g, K_FCPROJ_DW, d));
        // dx of fcproj times gelu'(x): kept by the forward (epilogue MUL_AUX), or
        // evaluated from the kept x (GELU_BWD) when the GELU output is recomputed
        d = gd(BT, 4 * C, C, dres, C, 1, pc_tensor(g, P_FCPROJW, l), 4 * C, 0, g->dbig, 4 * C,
               g->recompute >= 1 ? EPI_GELU_BWD : EPI_MUL_AUX);
        d.aux = fch;
        d.ldx = 4 * C;
        // the fc bias gradient (column sums of this product's output): its
        // partials come out of the same kernel on the tensor cores
        d.act = g->act;
        float* fcb_part = (float*)(fcb_base + (size_t)l * g->fcb_part_bytes);
        const bool fused_fcb = g->use_tc && gemm_tc_supported(d);
        if (fused_fcb) {
            d.colpart = fcb_part;
            g->ctasks.push_back(ColsumTask{fcb_part, {grad_tensor(g, P_FCB, l), nullptr, nullptr},
                                           (BT + 31) / 32, 4 * C, 4 * C});
        }
        RUN(mm(g, K_FCPROJ_DX, d));
        if (g->recompute >= 2)  // ln2(x1) again (the same kernel on the same input)
            LAUNCH(K_RECOMP, 1, 0, ln_bytes,
                   layernorm_forward(g->act, ln2, g->ln2_mean + l * bt, g->ln2_rstd + l * bt, x1,
                                     pc_tensor(g, P_LN2W, l), pc_tensor(g, P_LN2B, l), BT, C,
                                     g->stream));
        d = gd(4 * C, C, BT, g->dbig, 4 * C, 0, ln2, C, 0, grad_tensor(g, P_FCW, l), C,
               EPI_ACCUM_F32);
        RUN(mm(g, K_FC_DW, d));
        if (!fused_fcb) {
            LAUNCH(K_BIAS, 1, 0, as * bt * 4 * c,
                   bias_grad_rows(g->act, fcb_part, g->dbig, BT, 4 * C, &np, g->stream));
            g->ctasks.push_back(ColsumTask{fcb_part, {grad_tensor(g, P_FCB, l), nullptr, nullptr},
                                           np, 4 * C, 4 * C});
        }
        d = gd(BT, C, 4 * C, g->dbig, 4 * C, 1, pc_tensor(g, P_FCW, l), C, 0, g->dln, C,
               EPI_STORE);
        RUN(mm(g, K_FC_DX, d));
        {
            float* part = (float*)((char*)g->dpart + (size_t)(1 + 2 * l) * g->ln_part_bytes);
            LAUNCH(K_LN_BWD, 1, 0, lnb_bytes,
                   layernorm_backward_rows(g->act, dres, true, g->dln, x1,
                                           pc_tensor(g, P_LN2W, l), g->ln2_mean + l * bt,
                                           g->ln2_rstd + l * bt, BT, C, true, part, &np,
                                           g->stream));
            ln_task(1 + 2 * l, grad_tensor(g, P_LN2W, l), grad_tensor(g, P_LN2B, l),
                    grad_tensor(g, P_PROJB, l));
        }
        // attention: x1 = rin + proj(attn(qkv(ln1(rin))))
        d = gd(C, C, BT, dres, C, 0, atty, C, 0, grad_tensor(g, P_PROJW, l), C, EPI_ACCUM_F32);
        RUN(mm(g, K_PROJ_DW, d));
        d = gd(BT, C, C, dres, C, 1, pc_tensor(g, P_PROJW, l), C, 0, g->datty, C, EPI_STORE);
        RUN(mm(g, K_PROJ_DX, d));
        double afl = 2.5 * 2.0 * 2.0 * B * H * ((double)T * (T + 1) / 2) * (C / H);
        const int attn_bwd_kernels = attention_tc_supported(g->act, B, T, C, H, qkv) ? 2 : 3;
        LAUNCH(K_ATTN_BWD, attn_bwd_kernels, afl, as * 8.0 * bt * c,
               attention_backward(g->act, g->dqkv, g->datty, qkv, atty, lse, B, T, C, H,
                                  g->scratch, g->err, g->stream));
        if (g->recompute >= 2)  // ln1(rin) again
            LAUNCH(K_RECOMP, 1, 0, ln_bytes,
                   layernorm_forward(g->act, ln1, g->ln1_mean + l * bt, g->ln1_rstd + l * bt, rin,
                                     pc_tensor(g, P_LN1W, l), pc_tensor(g, P_LN1B, l), BT, C,
                                     g->stream));
        d = gd(3 * C, C, BT, g->dqkv, 3 * C, 0, ln1, C, 0, grad_tensor(g, P_QKVW, l), C,
               EPI_ACCUM_F32);
        RUN(mm(g, K_QKV_DW, d));
        {
            float* part = (float*)(qkvb_base + (size_t)l * g->qkvb_part_bytes);
            LAUNCH(K_BIAS, 1, 0, as * bt * 3 * c,
                   bias_grad_rows(g->act, part, g->dqkv, BT, 3 * C, &np, g->stream));
            g->ctasks.push_back(ColsumTask{part, {grad_tensor(g, P_QKVB, l), nullptr, nullptr},
                                           np, 3 * C, 3 * C});
        }
        d = gd(BT, C, 3 * C, g->dqkv, 3 * C, 1, pc_tensor(g, P_QKVW, l), C, 0, g->dln, C,
               EPI_STORE);
        RUN(mm(g, K_QKV_DX, d));
        {
            float* dxs = l > 0 ? grad_tensor(g, P_FCPROJB, l - 1) : nullptr;
            float* part = (float*)((char*)g->dpart + (size_t)(2 + 2 * l) * g->ln_part_bytes);
            LAUNCH(K_LN_BWD, 1, 0, lnb_bytes,
                   layernorm_backward_rows(g->act, dres, dxs != nullptr, g->dln, rin,
                                           pc_tensor(g, P_LN1W, l), g->ln1_mean + l * bt,
                                           g->ln1_rstd + l * bt, BT, C, true, part, &np,
                                           g->stream));
            ln_task(2 + 2 * l, grad_tensor(g, P_LN1W, l), grad_tensor(g, P_LN1B, l), dxs);
        }
    }
    {
        double cby = 0;
        for (const ColsumTask& t : g->ctasks) cby += 4.0 * t.ncols * (t.nparts + 2.0);
        const int nk = ((int)g->ctasks.size() + 95) / 96;
        int nl = 0;
        LAUNCH(K_COLSUM, nk, 0, cby,
               colsum_batch(g->ctasks.data(), (int)g->ctasks.size(), g->stream, &nl));
    }
    LAUNCH(K_EMB_BWD, 9, 0, as * bt * c + 8.0 * T * c,
           encoder_backward(g->act, grad_tensor(g, P_WTE, 0), grad_tensor(g, P_WPE, 0), dres,
                            g->tok, B, T, C, Vp, g->scratch, g->stream));
    if (g->sk_window > 0) {
        // running sum of the micro-batch losses (loss[1]) for the spike detector
        g->launches += 1;
        CK(accumulate_scalar(g->loss + 1, g->loss, g->stream));
    }
    g->n_accum++;
    g->have_fwd = 0;
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// optimizer
// ---------------------------------------------------------------------------
extern "C" int gpt2_zero_grad(gpt2_t* g) {
    if (!g) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    prof_begin(g, K_ZERO, 0, 4.0 * g->nparams);
    cudaError_t e = cudaMemsetAsync(g->grads, 0, g->nparams * 4, g->stream);
    if (e == cudaSuccess && g->sk_window > 0) e = cudaMemsetAsync(g->loss + 1, 0, 4, g->stream);
    prof_end(g);
    if (e) return fail(g, GPT2_ERR_CUDA, "zero_grad: %s", cudaGetErrorString(e));
    g->n_accum = 0;
    return GPT2_OK;
}

// z-score of x against the recorded window: (x - mean) / std with the
// population std of the window's values; NaN until the window is full; with a
// zero std, 0 for x == mean and +-infinity otherwise
static float spike_z(const gpt2* g, const std::vector<double>& hist, double x) {
    if (g->sk_count < g->sk_window) return NAN;
    double mean = 0.0;
    for (int i = 0; i < g->sk_window; i++) mean += hist[i];
    mean /= g->sk_window;
    double var = 0.0;
    for (int i = 0; i < g->sk_window; i++) var += (hist[i] - mean) * (hist[i] - mean);
    const double sd = sqrt(var / g->sk_window);
    if (sd == 0.0) return x == mean ? 0.f : (x > mean ? INFINITY : -INFINITY);
    return (float)((x - mean) / sd);
}

// norm pass, then the update of bf16-only parameters with stochastic rounding
// AdamW arguments of step t (1-based): bias corrections, the 1/count of the
// accumulated micro-batches, the weight-decayed ranges (the weight matrices and
// both embedding tables: decay on 2-D tensors only), and the stochastic-rounding stream.  base is the
// canonical index of the first element the update launch sees.
static AdamArgs adam_args(const gpt2* g, int t, float lr, float b1, float b2, float eps, float wd,
                          float clip, size_t base) {
    AdamArgs a;
    a.lr = lr; a.b1 = b1; a.b2 = b2; a.eps = eps; a.wd = wd;
    a.bc1 = (float)(1.0 - pow((double)b1, t));
    a.bc2 = (float)(1.0 - pow((double)b2, t));
    a.inv_accum = g->n_accum > 0 ? 1.0f / (float)g->n_accum : 0.f;
    a.d_count = nullptr;
    a.clip = clip;
    const size_t* o = g->lay.off;
    a.dec_lo[0] = o[P_WTE];     a.dec_hi[0] = o[P_LN1W];
    a.dec_lo[1] = o[P_QKVW];    a.dec_hi[1] = o[P_QKVB];
    a.dec_lo[2] = o[P_PROJW];   a.dec_hi[2] = o[P_PROJB];
    a.dec_lo[3] = o[P_FCW];     a.dec_hi[3] = o[P_FCB];
    a.dec_lo[4] = o[P_FCPROJW]; a.dec_hi[4] = o[P_FCPROJB];
    a.t = t;
    a.sr_seed = g->seed ^ 0x5352000000000000ull;  // "SR": the stochastic-rounding stream
    a.base = base;
    a.n_total = g->nparams;
    return a;
}

extern "C" int gpt2_adamw_step(gpt2_t* g, float lr, float b1, float b2, float eps, float wd,
                               float clip, float* h_grad_norm) {
    if (!g) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    // the device-side count (if any) serves this one update, whatever its outcome
    const int* dc = g->d_count;
    g->d_count = nullptr;
    if (g->sharded)
        return fail(g, GPT2_ERR_STATE, "a sharded handle updates its slice (gpt2_adamw_step_shard)");
    if (!dc && g->n_accum < 1) return fail(g, GPT2_ERR_STATE, "adamw_step without accumulated grads");
    const int t = g->t + 1;
    AdamArgs a = adam_args(g, t, lr, b1, b2, eps, wd, clip, 0);
    a.d_count = dc;
    void* wb = g->act == ACT_BF16 ? g->pc : nullptr;
    const double ad_bytes = 34.0 * g->nparams + (g->act == ACT_BF16 ? 2.0 * g->nparams : 0.0);
    g->last_skipped = 0;
    g->last_zl = g->last_zg = NAN;
    if (g->sk_window <= 0) {
        // norm, clip and update in one cooperative launch
        if (g->no_master) {
            LAUNCH(K_ADAM, 1, 0, ad_bytes - 6.0 * g->nparams,
                   adamw_fused(nullptr, g->m, g->v, g->grads, g->pc, g->nparams, 0, g->nparams,
                               true, a, g->adam_state, g->scratch, g->adam_bar, g->err,
                               g->stream));
        } else {
            LAUNCH(K_ADAM, 1, 0, ad_bytes,
                   adamw_fused(g->master, g->m, g->v, g->grads, wb, g->nparams, 0, g->nparams,
                               false, a, g->adam_state, g->scratch, g->adam_bar, g->err,
                               g->stream));
        }
        float st[3];
        CK(cudaMemcpyAsync(st, g->adam_state, 12, cudaMemcpyDeviceToHost, g->stream));
        RUN(check_dev_err(g));
        if (h_grad_norm) *h_grad_norm = st[0];
        if (st[2] == 0.f)
            return fail(g, GPT2_ERR_NONFINITE, "gradient norm is not finite (%g)", st[0]);
        g->t = t;
        return GPT2_OK;
    }
    // spike detector on: the norm pass, then the decision on the host, then
    // the update (or not)
    LAUNCH(K_ADAM, 2, 0, 4.0 * g->nparams,
           adamw_norm(g->grads, g->nparams, a, g->adam_state, g->scratch, g->stream));
    float st[3], lsum = 0.f;
    CK(cudaMemcpyAsync(st, g->adam_state, 12, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaMemcpyAsync(&lsum, g->loss + 1, 4, cudaMemcpyDeviceToHost, g->stream));
    RUN(check_dev_err(g));  // synchronises the stream
    if (h_grad_norm) *h_grad_norm = st[0];
    const double step_loss = (double)lsum / (g->n_accum > 0 ? g->n_accum : 1), norm = st[0];
    g->last_zl = spike_z(g, g->sk_loss_hist, step_loss);
    g->last_zg = spike_z(g, g->sk_grad_hist, norm);
    const bool spike = (g->sk_loss_z > 0.f && g->last_zl > g->sk_loss_z) ||
                       (g->sk_grad_z > 0.f && g->last_zg > g->sk_grad_z);
    // every step's values enter the window, skipped or not
    g->sk_loss_hist[g->sk_pos] = step_loss;
    g->sk_grad_hist[g->sk_pos] = norm;
    g->sk_pos = (g->sk_pos + 1) % g->sk_window;
    if (g->sk_count < g->sk_window) g->sk_count++;
    if (st[2] == 0.f) return fail(g, GPT2_ERR_NONFINITE, "gradient norm is not finite (%g)", st[0]);
    if (spike) {
        g->last_skipped = 1;  // parameters, moments and the step count unchanged
        return GPT2_OK;
    }
    if (g->no_master)
        LAUNCH(K_ADAM, 1, 0, ad_bytes - 10.0 * g->nparams,
               adamw_update_bf16_sr(g->pc, g->m, g->v, g->grads, g->nparams, a, g->adam_state,
                                    g->stream));
    else
        LAUNCH(K_ADAM, 1, 0, ad_bytes - 4.0 * g->nparams,
               adamw_update(g->master, g->m, g->v, g->grads, wb, g->nparams, a, g->adam_state,
                            g->stream));
    g->t = t;
    return GPT2_OK;
}

extern "C" int gpt2_set_spike_skip(gpt2_t* g, float loss_z, float grad_z, int window) {
    if (!g || window < 0 || window == 1 || window > (1 << 20)) return GPT2_ERR_ARG;
    g->sk_loss_z = loss_z;
    g->sk_grad_z = grad_z;
    g->sk_window = window;
    g->sk_count = g->sk_pos = 0;
    g->sk_loss_hist.assign(window, 0.0);
    g->sk_grad_hist.assign(window, 0.0);
    if (window > 0) {
        cudaSetDevice(g->device);
        CK(cudaMemsetAsync(g->loss + 1, 0, 4, g->stream));  // no partial sum carried in
    }
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// data parallelism: buffers for an external all-reduce / all-gather, the
// gradient divisor, and the AdamW update of one shard of the parameters
// ---------------------------------------------------------------------------
extern "C" int gpt2_grads_buffer(gpt2_t* g, float** d_grads, size_t* n) {
    if (!g) return GPT2_ERR_ARG;
    if (d_grads) *d_grads = g->grads;
    if (n) *n = g->nparams;
    return GPT2_OK;
}
extern "C" int gpt2_params_buffer(gpt2_t* g, float** d_master, void** d_bf16, size_t* n) {
    if (!g) return GPT2_ERR_ARG;
    // NULL without master weights, or when the handle holds only its slice
    if (d_master) *d_master = g->master_sliced() ? nullptr : g->master;
    if (d_bf16) *d_bf16 = g->act == ACT_BF16 ? g->pc : nullptr;
    if (n) *n = g->nparams;
    return GPT2_OK;
}
extern "C" int gpt2_get_grad_count(gpt2_t* g, int* count) {
    if (!g || !count) return GPT2_ERR_ARG;
    *count = g->n_accum;
    return GPT2_OK;
}
extern "C" int gpt2_set_grad_count(gpt2_t* g, int count) {
    if (!g || count < 1) return GPT2_ERR_ARG;
    g->n_accum = count;
    return GPT2_OK;
}
extern "C" int gpt2_set_grad_count_device(gpt2_t* g, const int* d_count) {
    if (!g || !d_count || ((uintptr_t)d_count & 3)) return GPT2_ERR_ARG;
    g->d_count = d_count;
    return GPT2_OK;
}
extern "C" int gpt2_shard_bounds(gpt2_t* g, size_t* lo, size_t* hi) {
    if (!g) return GPT2_ERR_ARG;
    if (lo) *lo = g->sharded ? g->sh_lo : 0;
    if (hi) *hi = g->sharded ? g->sh_hi : g->nparams;
    return GPT2_OK;
}
extern "C" int gpt2_get_shard_master(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    if (!g->master) return fail(g, GPT2_ERR_STATE, "no fp32 master weights (GPT2_NO_MASTER)");
    cudaSetDevice(g->device);
    const float* src = g->master_sliced() ? g->master : g->master + (g->sharded ? g->sh_lo : 0);
    CK(cudaMemcpyAsync(h, src, g->n_state() * 4, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    return GPT2_OK;
}

extern "C" int gpt2_adamw_step_shard(gpt2_t* g, size_t lo, size_t hi, float lr, float b1, float b2,
                                     float eps, float wd, float clip, float* h_grad_norm) {
    if (!g || !shard_ok(g->nparams, lo, hi)) return GPT2_ERR_ARG;
    if (g->sharded && (lo != g->sh_lo || hi != g->sh_hi)) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    // the device-side count (if any) serves this one update, whatever its outcome
    const int* dc = g->d_count;
    g->d_count = nullptr;
    if (!dc && g->n_accum < 1)
        return fail(g, GPT2_ERR_STATE, "adamw_step_shard without accumulated grads");
    if (g->sk_window > 0)
        return fail(g, GPT2_ERR_STATE, "the spike detector needs the whole update (not a shard)");
    const int t = g->t + 1;
    AdamArgs a = adam_args(g, t, lr, b1, b2, eps, wd, clip, lo);
    a.d_count = dc;
    const size_t n = hi - lo;
    // the slice's moments (and master): the whole buffers' [lo, hi), or all of
    // a sharded handle's
    float* ms = g->sharded ? g->m : g->m + lo;
    float* vs = g->sharded ? g->v : g->v + lo;
    float* ws = g->master_sliced() ? g->master : (g->master ? g->master + lo : nullptr);
    // the norm (and the clip scale) over every gradient, the update on [lo, hi),
    // in one cooperative launch
    {
        const size_t as = act_size(g->act);
        void* wb = g->act == ACT_BF16 ? (void*)((char*)g->pc + lo * as) : nullptr;
        if (g->no_master)
            LAUNCH(K_ADAM, 1, 0, 4.0 * g->nparams + 26.0 * n,
                   adamw_fused(nullptr, ms, vs, g->grads, wb, g->nparams, lo, n, true, a,
                               g->adam_state, g->scratch, g->adam_bar, g->err, g->stream));
        else
            LAUNCH(K_ADAM, 1, 0, 4.0 * g->nparams + 30.0 * n,
                   adamw_fused(ws, ms, vs, g->grads, wb, g->nparams, lo, n, false, a,
                               g->adam_state, g->scratch, g->adam_bar, g->err, g->stream));
    }
    float st[3];
    CK(cudaMemcpyAsync(st, g->adam_state, 12, cudaMemcpyDeviceToHost, g->stream));
    RUN(check_dev_err(g));
    if (h_grad_norm) *h_grad_norm = st[0];
    if (st[2] == 0.f) return fail(g, GPT2_ERR_NONFINITE, "gradient norm is not finite (%g)", st[0]);
    g->t = t;
    return GPT2_OK;
}

extern "C" int gpt2_last_step_info(gpt2_t* g, int* skipped, float* z_loss, float* z_grad) {
    if (!g) return GPT2_ERR_ARG;
    if (skipped) *skipped = g->last_skipped;
    if (z_loss) *z_loss = g->last_zl;
    if (z_grad) *z_grad = g->last_zg;
    return GPT2_OK;
}

// fp32 <-> the parameters: the master copy, or (no master) the bf16 values
// widened exactly / rounded to nearest even, converted on the host
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
    return (uint16_t)((b + 0x7fffu + ((b >> 16) & 1u)) >> 16);
}
static int params_to_host(gpt2* g, float* h) {
    if (!g->no_master && !g->master_sliced()) {
        CK(cudaMemcpyAsync(h, g->master, g->nparams * 4, cudaMemcpyDeviceToHost, g->stream));
        CK(cudaStreamSynchronize(g->stream));
        return GPT2_OK;
    }
    std::vector<uint16_t> tmp(g->nparams);
    CK(cudaMemcpyAsync(tmp.data(), g->pc, g->nparams * 2, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    for (size_t i = 0; i < g->nparams; i++) {
        const uint32_t u = (uint32_t)tmp[i] << 16;
        memcpy(&h[i], &u, 4);
    }
    return GPT2_OK;
}
static int params_from_host(gpt2* g, const float* h) {
    if (g->master_sliced() && g->n_state())
        CK(cudaMemcpyAsync(g->master, h + g->sh_lo, g->n_state() * 4, cudaMemcpyHostToDevice,
                           g->stream));
    if (!g->no_master && !g->master_sliced()) {
        CK(cudaMemcpyAsync(g->master, h, g->nparams * 4, cudaMemcpyHostToDevice, g->stream));
        if (g->act == ACT_BF16) CK(cast_to_bf16(g->pc, g->master, g->nparams, g->stream));
        CK(cudaStreamSynchronize(g->stream));
        return GPT2_OK;
    }
    std::vector<uint16_t> tmp(g->nparams);
    for (size_t i = 0; i < g->nparams; i++) tmp[i] = f32_to_bf16_rne(h[i]);
    CK(cudaMemcpyAsync(g->pc, tmp.data(), g->nparams * 2, cudaMemcpyHostToDevice, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// checkpoints: fp32 parameters, AdamW moments and step count, and the spike
// detector's window, so that a run resumed from a checkpoint continues bit for
// bit as if it had not stopped
// ---------------------------------------------------------------------------
struct CkptHeader {  // 88 bytes, little-endian, no implicit padding
    char magic[8];  // "GPT2B3CK"
    uint32_t version;
    int32_t L, H, C, V, T, mode;
    uint32_t pad0;
    uint64_t nparams;
    int32_t t;
    int32_t sk_window, sk_count, sk_pos;
    float sk_loss_z, sk_grad_z;
    uint64_t seed;  // the handle's seed: the stochastic-rounding stream continues from it
    uint32_t reserved[2];
};
static_assert(sizeof(CkptHeader) == 88, "checkpoint header layout");
static const char kCkptMagic[8] = {'G', 'P', 'T', '2', 'B', '3', 'C', 'K'};

extern "C" int gpt2_save_checkpoint(gpt2_t* g, const char* path) {
    if (!g || !path) return GPT2_ERR_ARG;
    if (g->sharded)
        return fail(g, GPT2_ERR_STATE, "a sharded handle holds only its slice of the state");
    cudaSetDevice(g->device);
    CkptHeader hd;
    memset(&hd, 0, sizeof hd);
    memcpy(hd.magic, kCkptMagic, 8);
    hd.version = 1;
    hd.L = g->L; hd.H = g->H; hd.C = g->C; hd.V = g->V; hd.T = g->T; hd.mode = g->mode;
    hd.nparams = g->nparams;
    hd.t = g->t;
    hd.sk_window = g->sk_window; hd.sk_count = g->sk_count; hd.sk_pos = g->sk_pos;
    hd.sk_loss_z = g->sk_loss_z; hd.sk_grad_z = g->sk_grad_z;
    hd.seed = g->seed;
    FILE* f = fopen(path, "wb");
    if (!f) return fail(g, GPT2_ERR_IO, "cannot open %s for writing", path);
    bool ok = fwrite(&hd, sizeof hd, 1, f) == 1;
    std::vector<float> buf(ok ? g->nparams : 0);
    const float* src[3] = {nullptr, g->m, g->v};  // params through params_to_host
    for (int k = 0; ok && k < 3; k++) {
        if (k == 0) {
            const int rc = params_to_host(g, buf.data());
            if (rc != GPT2_OK) {
                fclose(f);
                return rc;
            }
        } else if (cudaMemcpy(buf.data(), src[k], g->nparams * 4, cudaMemcpyDeviceToHost) !=
                   cudaSuccess) {
            fclose(f);
            return fail(g, GPT2_ERR_CUDA, "checkpoint: device read failed");
        }
        ok = fwrite(buf.data(), 4, g->nparams, f) == g->nparams;
    }
    if (ok && g->sk_window > 0)
        ok = fwrite(g->sk_loss_hist.data(), 8, g->sk_window, f) == (size_t)g->sk_window &&
             fwrite(g->sk_grad_hist.data(), 8, g->sk_window, f) == (size_t)g->sk_window;
    if (fclose(f) != 0) ok = false;
    return ok ? GPT2_OK : fail(g, GPT2_ERR_IO, "write to %s failed", path);
}

extern "C" int gpt2_load_checkpoint(gpt2_t* g, const char* path) {
    if (!g || !path) return GPT2_ERR_ARG;
    if (g->sharded)
        return fail(g, GPT2_ERR_STATE, "a sharded handle holds only its slice of the state");
    cudaSetDevice(g->device);
    FILE* f = fopen(path, "rb");
    if (!f) return fail(g, GPT2_ERR_IO, "cannot open %s", path);
    CkptHeader hd;
    if (fread(&hd, sizeof hd, 1, f) != 1 || memcmp(hd.magic, kCkptMagic, 8) != 0 ||
        hd.version != 1) {
        fclose(f);
        return fail(g, GPT2_ERR_IO, "%s is not a checkpoint of this library", path);
    }
    if (hd.L != g->L || hd.H != g->H || hd.C != g->C || hd.V != g->V || hd.T != g->T ||
        hd.nparams != g->nparams || hd.t < 0 || hd.sk_window < 0 || hd.sk_window == 1 ||
        hd.sk_window > (1 << 20) || hd.sk_count < 0 || hd.sk_count > hd.sk_window ||
        hd.sk_pos < 0 || (hd.sk_window > 0 && hd.sk_pos >= hd.sk_window)) {
        fclose(f);
        return fail(g, GPT2_ERR_ARG, "checkpoint %s (L=%d H=%d C=%d V=%d T=%d) does not fit this model",
                    path, hd.L, hd.H, hd.C, hd.V, hd.T);
    }
    std::vector<float> buf(g->nparams);
    float* dst[3] = {nullptr, g->m, g->v};  // params through params_from_host
    bool ok = true;
    for (int k = 0; ok && k < 3; k++) {
        ok = fread(buf.data(), 4, g->nparams, f) == g->nparams;
        if (!ok) break;
        if (k == 0) {
            const int rc = params_from_host(g, buf.data());
            if (rc != GPT2_OK) {
                fclose(f);
                return rc;
            }
        } else if (cudaMemcpy(dst[k], buf.data(), g->nparams * 4, cudaMemcpyHostToDevice) !=
                   cudaSuccess) {
            fclose(f);
            return fail(g, GPT2_ERR_CUDA, "checkpoint: device write failed");
        }
    }
    std::vector<double> lh(hd.sk_window), gh(hd.sk_window);
    if (ok && hd.sk_window > 0)
        ok = fread(lh.data(), 8, hd.sk_window, f) == (size_t)hd.sk_window &&
             fread(gh.data(), 8, hd.sk_window, f) == (size_t)hd.sk_window;
    fclose(f);
    if (!ok) return fail(g, GPT2_ERR_IO, "%s is truncated", path);
    CK(cudaStreamSynchronize(g->stream));
    g->t = hd.t;
    g->sk_window = hd.sk_window; g->sk_count = hd.sk_count; g->sk_pos = hd.sk_pos;
    g->sk_loss_z = hd.sk_loss_z; g->sk_grad_z = hd.sk_grad_z;
    g->sk_loss_hist = lh;
    g->sk_grad_hist = gh;
    g->seed = hd.seed;
    g->last_skipped = 0;
    g->last_zl = g->last_zg = NAN;
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// inspection
// ---------------------------------------------------------------------------
extern "C" size_t gpt2_num_params(gpt2_t* g) { return g ? g->nparams : 0; }
extern "C" int gpt2_padded_vocab(gpt2_t* g) { return g ? g->Vp : 0; }

extern "C" int gpt2_get_params(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    return params_to_host(g, h);
}
extern "C" int gpt2_set_params(gpt2_t* g, const float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    return params_from_host(g, h);
}
extern "C" int gpt2_get_grads(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    CK(cudaMemcpyAsync(h, g->grads, g->nparams * 4, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    return GPT2_OK;
}
extern "C" int gpt2_set_grads(gpt2_t* g, const float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    CK(cudaMemcpyAsync(g->grads, h, g->nparams * 4, cudaMemcpyHostToDevice, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    if (g->n_accum < 1) g->n_accum = 1;
    return GPT2_OK;
}
extern "C" int gpt2_get_opt_state(gpt2_t* g, float* hm, float* hv, int* step) {
    if (!g) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    if (hm) CK(cudaMemcpyAsync(hm, g->m, g->n_state() * 4, cudaMemcpyDeviceToHost, g->stream));
    if (hv) CK(cudaMemcpyAsync(hv, g->v, g->n_state() * 4, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    if (step) *step = g->t;
    return GPT2_OK;
}

extern "C" int gpt2_set_opt_state(gpt2_t* g, const float* hm, const float* hv, int step) {
    if (!g || step < 0) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    if (hm) CK(cudaMemcpyAsync(g->m, hm, g->n_state() * 4, cudaMemcpyHostToDevice, g->stream));
    if (hv) CK(cudaMemcpyAsync(g->v, hv, g->n_state() * 4, cudaMemcpyHostToDevice, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    g->t = step;
    return GPT2_OK;
}

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

extern "C" int gpt2_get_logits(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    if (!g->logits_valid)
        return fail(g, GPT2_ERR_STATE, "logits are kept only after a forward without targets");
    size_t as = act_size(g->act);
    std::vector<char> tmp(g->BT * g->V * as);
    CK(cudaMemcpy2DAsync(tmp.data(), g->V * as, g->logits, (size_t)g->Vp * as, g->V * as, g->BT,
                         cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    size_t n = g->BT * g->V;
    if (g->act == ACT_BF16) {
        const uint16_t* s = (const uint16_t*)tmp.data();
        for (size_t i = 0; i < n; i++) h[i] = bf16_bits_to_float(s[i]);
    } else {
        memcpy(h, tmp.data(), n * 4);
    }
    return GPT2_OK;
}
extern "C" int gpt2_get_loss(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    RUN(check_dev_err(g));
    CK(cudaMemcpy(h, g->loss, 4, cudaMemcpyDeviceToHost));
    return GPT2_OK;
}
extern "C" int gpt2_get_losses(gpt2_t* g, float* h) {
    if (!g || !h) return GPT2_ERR_ARG;
    cudaSetDevice(g->device);
    CK(cudaMemcpyAsync(h, g->losses, g->BT * 4, cudaMemcpyDeviceToHost, g->stream));
    CK(cudaStreamSynchronize(g->stream));
    return GPT2_OK;
}

// ---------------------------------------------------------------------------
// profiling
// ---------------------------------------------------------------------------
extern "C" int gpt2_prof_enable(gpt2_t* g, unsigned class_mask) {
    if (!g) return GPT2_ERR_ARG;
    if (!class_mask) prof_collect(g);
    g->prof_on = class_mask != 0;
    g->prof_mask = class_mask;
    return GPT2_OK;
}
extern "C" long long gpt2_launch_count(gpt2_t* g) { return g ? g->launches : -1; }
extern "C" int gpt2_prof_reset(gpt2_t* g) {
    if (!g) return GPT2_ERR_ARG;
    prof_collect(g);
    for (int i = 0; i < K_NCLASS; i++) {
        g->prof_ms[i] = g->prof_flops[i] = g->prof_bytes[i] = 0;
        g->prof_n[i] = 0;
    }
    return GPT2_OK;
}
extern "C" int gpt2_prof_num_classes(void) { return K_NCLASS; }
extern "C" const char* gpt2_prof_name(int c) {
    return (c >= 0 && c < K_NCLASS) ? kClassNames[c] : "";
}
extern "C" int gpt2_prof_read(gpt2_t* g, int c, double* ms, long long* n, double* fl,
                              double* by) {
    if (!g || c < 0 || c >= K_NCLASS) return GPT2_ERR_ARG;
    prof_collect(g);
    if (ms) *ms = g->prof_ms[c];
    if (n) *n = g->prof_n[c];
    if (fl) *fl = g->prof_flops[c];
    if (by) *by = g->prof_bytes[c];
    return GPT2_OK;
}
