/*
 * gpt2_oracle.c -- a plain, slow, CPU reference of one GPT-2 training step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only at the canonical parameter order
 * (described below in prose, restated independently on each side) and at the
 * seeded input generators, which hold none of the method's arithmetic.
 *
 * What it computes (sources, by page title and section):
 *  - "Karpathy's llm.c: understanding LLM training from scratch in C/CUDA",
 *    section "Code anatomy -- CPU version train_gpt2.c": the step is the
 *    chain encoder_forward -> layernorm_forward -> attention ... -> backward
 *    in reverse graph order -> parameter update, written as plain loops.
 *  - "Karpathy reproduces GPT-2 (1.6B) in llm.c", section "Parameter guide":
 *    AdamW with weight decay on 2-D weights only (-c 0.1), global gradient
 *    norm, gradient accumulation over micro-batches (-d), vocabulary padded
 *    from 50257 to 50304 (section "PyTorch comparison").
 *  - "Getting started with LLMs from Andrej Karpathy's talk", section on
 *    self-attention: Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - LayerNorm eps = 1e-5, biased variance (divide by C).
 *  - GELU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))).
 *  - Causal mask: query t attends to keys 0..t; masked keys are left out of
 *    the softmax (not set to a large negative number).
 *  - Q, K, V are consecutive C-wide blocks of the 3C QKV output; head h uses
 *    columns h*hd .. (h+1)*hd - 1 of each block.
 *  - Vocabulary rows are padded up to a multiple of 128 (50257 -> 50304,
 *    2 -> 128); padded rows start at 0 and their logits are left out of the
 *    softmax, so their gradient is exactly 0 and they stay 0.
 *  - Loss = mean over all B*T positions of -log softmax(logits)[target].
 *  - Gradients accumulate (+=) over micro-batches; the update divides by the
 *    number of micro-batches, clips by the global L2 norm (clip <= 0: off),
 *    then applies AdamW with bias correction, eps outside the sqrt, and
 *    decoupled decay lr*wd*w on the 2-D tensors {wte, wpe, qkvw, projw, fcw,
 *    fcprojw}.  A non-finite norm skips the update and leaves every state
 *    untouched.
 *  - Init: matrices and both embeddings ~ N(0, 0.02); projw and fcprojw
 *    ~ N(0, 0.02/sqrt(2L)); biases 0; LayerNorm gain 1, bias 0; padded wte
 *    rows 0.  Element i of the canonical vector draws outputs 2i and 2i+1 of
 *    the SplitMix64 generator (Steele, Lea & Flood, OOPSLA 2014) seeded with
 *    `seed`, maps each to a uniform in (0,1) with 53 bits, and applies the
 *    Box-Muller transform (Box & Muller 1958) in double, then rounds the
 *    scaled value to fp32.
 *
 * Canonical parameter order (weights are out x in, row-major):
 *   wte[Vp,C] wpe[T,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C] qkvb[L,3C]
 *   projw[L,C,C] projb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C] fcb[L,4C]
 *   fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C]
 *
 * The arithmetic type is `real` (double unless built with -DREAL=float).
 * OpenMP pragmas sit only on loops whose iterations write disjoint outputs,
 * so every output is summed in the same sequential order at any thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL double
#endif
typedef REAL real;

#define OG_LN_EPS 1e-5
#define OG_PI 3.14159265358979323846

/* ------------------------------------------------------------------ */
/* Random init: SplitMix64 stream + Box-Muller                         */
/* ------------------------------------------------------------------ */

/* Output number j (0-based) of SplitMix64 seeded with `seed`: the state
 * advances by the golden-ratio increment before each output, and each output
 * is the state passed through the generator's 64-bit finaliser. */
static uint64_t og_splitmix64(uint64_t seed, uint64_t j) {
    uint64_t z = seed + (j + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static double og_uniform_open(uint64_t x) {
    /* top 53 bits, centred in their cell: strictly inside (0, 1) */
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* fp32-rounded N(0, std^2) sample for canonical element i */
float og_normal_sample(uint64_t seed, uint64_t i, double std) {
    double u1 = og_uniform_open(og_splitmix64(seed, 2 * i));
    double u2 = og_uniform_open(og_splitmix64(seed, 2 * i + 1));
    double z = sqrt(-2.0 * log(u1)) * cos(2.0 * OG_PI * u2);
    return (float)(z * std);
}

/* Stochastic rounding of fp32 to bf16 (the parameter update without fp32
 * master weights, "Karpathy reproduces GPT-2 (1.6B) in llm.c", "Parameter
 * guide" -w 0).  The bf16 value is the top half of the fp32 bit pattern; the
 * bottom half (the fraction f / 65536 of the way from |x| truncated to the next
 * bf16 magnitude) decides: round |x| up iff r < f, with r the top 16 bits of
 * SplitMix64 output k0 + i -- i.e. with probability f / 65536.  Written as:
 * up iff f + r >= 65536 (a carry out of the bottom half).  NaN gives the quiet
 * NaN 0x7fc0. */
void og_stochastic_round_bf16(uint16_t* out, const float* in, size_t n, uint64_t seed,
                              uint64_t k0) {
    for (size_t i = 0; i < n; i++) {
        uint32_t b;
        memcpy(&b, &in[i], 4);
        if ((b & 0x7fffffffu) > 0x7f800000u) {
            out[i] = 0x7fc0;
            continue;
        }
        uint32_t r = (uint32_t)(og_splitmix64(seed, k0 + i) >> 48);
        uint32_t top = b >> 16, f = b & 0xffffu;
        out[i] = (uint16_t)(f + r >= 65536u ? top + 1u : top);
    }
}

/* ------------------------------------------------------------------ */
/* Parameter layout                                                    */
/* ------------------------------------------------------------------ */

enum {
    P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_PROJW, P_PROJB,
    P_LN2W, P_LN2B, P_FCW, P_FCB, P_FCPROJW, P_FCPROJB, P_LNFW, P_LNFB,
    P_COUNT
};

int og_padded_vocab(int V) { return ((V + 127) / 128) * 128; }

static void og_param_sizes(size_t sz[P_COUNT], int L, int C, int Vp, int T) {
    size_t c = (size_t)C, l = (size_t)L;
    sz[P_WTE] = (size_t)Vp * c;
    sz[P_WPE] = (size_t)T * c;
    sz[P_LN1W] = l * c;
    sz[P_LN1B] = l * c;
    sz[P_QKVW] = l * 3 * c * c;
    sz[P_QKVB] = l * 3 * c;
    sz[P_PROJW] = l * c * c;
    sz[P_PROJB] = l * c;
    sz[P_LN2W] = l * c;
    sz[P_LN2B] = l * c;
    sz[P_FCW] = l * 4 * c * c;
    sz[P_FCB] = l * 4 * c;
    sz[P_FCPROJW] = l * c * 4 * c;
    sz[P_FCPROJB] = l * c;
    sz[P_LNFW] = c;
    sz[P_LNFB] = c;
}

/* number of stored parameters for padded vocabulary Vp */
size_t og_param_count(int L, int C, int Vp, int T) {
    size_t sz[P_COUNT], n = 0;
    og_param_sizes(sz, L, C, Vp, T);
    for (int i = 0; i < P_COUNT; i++) n += sz[i];
    return n;
}

/* ------------------------------------------------------------------ */
/* Layer operations (plain loops)                                      */
/* ------------------------------------------------------------------ */

/* out[b,t,:] = wte[tok[b,t],:] + wpe[t,:] */
void og_encoder_forward(real* out, const int* tok, const real* wte,
                        const real* wpe, int B, int T, int C) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            real* o = out + ((size_t)b * T + t) * C;
            const real* e = wte + (size_t)tok[b * T + t] * C;
            const real* p = wpe + (size_t)t * C;
            for (int c = 0; c < C; c++) o[c] = e[c] + p[c];
        }
}

/* dwte[tok[b,t],:] += dout[b,t,:];  dwpe[t,:] += dout[b,t,:]
 * (positions visited in order b = 0.., t = 0..) */
void og_encoder_backward(real* dwte, real* dwpe, const real* dout,
                         const int* tok, int B, int T, int C) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            const real* d = dout + ((size_t)b * T + t) * C;
            real* e = dwte + (size_t)tok[b * T + t] * C;
            real* p = dwpe + (size_t)t * C;
            for (int c = 0; c < C; c++) {
                e[c] += d[c];
                p[c] += d[c];
            }
        }
}

/* y = (x - mean) * rstd * w + b over each row of C; saves mean, rstd */
void og_layernorm_forward(real* out, real* mean, real* rstd, const real* inp,
                          const real* w, const real* b, int N, int C) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* x = inp + (size_t)n * C;
        real m = 0;
        for (int c = 0; c < C; c++) m += x[c];
        m = m / C;
        real v = 0;
        for (int c = 0; c < C; c++) v += (x[c] - m) * (x[c] - m);
        v = v / C;
        real s = 1 / sqrt(v + (real)OG_LN_EPS);
        real* y = out + (size_t)n * C;
        for (int c = 0; c < C; c++) y[c] = (x[c] - m) * s * w[c] + b[c];
        mean[n] = m;
        rstd[n] = s;
    }
}

/* Backward of the row normalisation.  dinp is ACCUMULATED into; dw, db too.
 * xhat = (x-mean)*rstd, g = dout*w:
 *   dinp += rstd * (g - mean(g) - xhat * mean(g*xhat)),
 *   dw += dout*xhat, db += dout (summed over rows in order). */
void og_layernorm_backward(real* dinp, real* dw, real* db, const real* dout,
                           const real* inp, const real* w, const real* mean,
                           const real* rstd, int N, int C) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* x = inp + (size_t)n * C;
        const real* dy = dout + (size_t)n * C;
        real m = mean[n], s = rstd[n];
        real g_mean = 0, gx_mean = 0;
        for (int c = 0; c < C; c++) {
            real xhat = (x[c] - m) * s;
            real g = dy[c] * w[c];
            g_mean += g;
            gx_mean += g * xhat;
        }
        g_mean = g_mean / C;
        gx_mean = gx_mean / C;
        real* dx = dinp + (size_t)n * C;
        for (int c = 0; c < C; c++) {
            real xhat = (x[c] - m) * s;
            real g = dy[c] * w[c];
            dx[c] += s * (g - g_mean - xhat * gx_mean);
        }
    }
    /* parameter gradients: each column summed over rows n = 0.. in order */
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        real aw = 0, ab = 0;
        for (int n = 0; n < N; n++) {
            real xhat = (inp[(size_t)n * C + c] - mean[n]) * rstd[n];
            aw += dout[(size_t)n * C + c] * xhat;
            ab += dout[(size_t)n * C + c];
        }
        dw[c] += aw;
        db[c] += ab;
    }
}

/* out[n,o] = bias[o] + sum_c inp[n,c] * w[o,c]   (w is OC x C; bias may be NULL) */
void og_matmul_forward(real* out, const real* inp, const real* w,
                       const real* bias, int N, int C, int OC) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* x = inp + (size_t)n * C;
        for (int o = 0; o < OC; o++) {
            const real* wr = w + (size_t)o * C;
            real acc = bias ? bias[o] : 0;
            for (int c = 0; c < C; c++) acc += x[c] * wr[c];
            out[(size_t)n * OC + o] = acc;
        }
    }
}

/* Backward of out = inp w^T + b.  All three outputs are ACCUMULATED into:
 *   dinp[n,c] += sum_o dout[n,o] w[o,c]
 *   dw[o,c]   += sum_n dout[n,o] inp[n,c]
 *   dbias[o]  += sum_n dout[n,o]           (dbias may be NULL) */
void og_matmul_backward(real* dinp, real* dw, real* dbias, const real* dout,
                        const real* inp, const real* w, int N, int C, int OC) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        real* dx = dinp + (size_t)n * C;
        for (int o = 0; o < OC; o++) {
            real d = dout[(size_t)n * OC + o];
            const real* wr = w + (size_t)o * C;
            for (int c = 0; c < C; c++) dx[c] += d * wr[c];
        }
    }
#pragma omp parallel for schedule(static)
    for (int o = 0; o < OC; o++) {
        real* dwr = dw + (size_t)o * C;
        real db = 0;
        for (int n = 0; n < N; n++) {
            real d = dout[(size_t)n * OC + o];
            const real* x = inp + (size_t)n * C;
            for (int c = 0; c < C; c++) dwr[c] += d * x[c];
            db += d;
        }
        if (dbias) dbias[o] += db;
    }
}

/* Causal multi-head attention.  qkv[b,t,:] = [q | k | v], each C wide,
 * head h at columns h*hd.. of each block.  For query t the scores over keys
 * t2 <= t are s = q.k / sqrt(hd); att = softmax(s) over those keys only;
 * out[b,t,h*hd+i] = sum_{t2<=t} att * v[t2, i].  att is [B,H,T,T] with
 * zeros above the diagonal (kept for the backward pass). */
void og_attention_forward(real* out, real* att, const real* qkv, int B, int T,
                          int C, int H) {
    int hd = C / H;
    real scale = 1 / sqrt((real)hd);
    size_t C3 = (size_t)3 * C;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++)
            for (int t = 0; t < T; t++) {
                const real* q = qkv + ((size_t)b * T + t) * C3 + (size_t)h * hd;
                real* a = att + (((size_t)b * H + h) * T + t) * T;
                real mx = -INFINITY;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* k = qkv + ((size_t)b * T + t2) * C3 + C + (size_t)h * hd;
                    real s = 0;
                    for (int i = 0; i < hd; i++) s += q[i] * k[i];
                    s = s * scale;
                    a[t2] = s;
                    if (s > mx) mx = s;
                }
                real sum = 0;
                for (int t2 = 0; t2 <= t; t2++) {
                    a[t2] = exp(a[t2] - mx);
                    sum += a[t2];
                }
                for (int t2 = 0; t2 <= t; t2++) a[t2] = a[t2] / sum;
                for (int t2 = t + 1; t2 < T; t2++) a[t2] = 0;
                real* o = out + ((size_t)b * T + t) * C + (size_t)h * hd;
                for (int i = 0; i < hd; i++) o[i] = 0;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* v = qkv + ((size_t)b * T + t2) * C3 + 2 * (size_t)C + (size_t)h * hd;
                    for (int i = 0; i < hd; i++) o[i] += a[t2] * v[i];
                }
            }
}

/* Backward of og_attention_forward; dqkv is ACCUMULATED into.
 * With dA[t2] = dout_t . v[t2]:  dv[t2] += att[t2] dout_t;
 * dS[t2] = att[t2] (dA[t2] - sum_t3 att[t3] dA[t3]);
 * dq_t += scale sum dS[t2] k[t2];  dk[t2] += scale dS[t2] q_t. */
void og_attention_backward(real* dqkv, const real* dout, const real* qkv,
                           const real* att, int B, int T, int C, int H) {
    int hd = C / H;
    real scale = 1 / sqrt((real)hd);
    size_t C3 = (size_t)3 * C;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            real* dA = (real*)malloc(sizeof(real) * (size_t)T);
            for (int t = 0; t < T; t++) {
                const real* a = att + (((size_t)b * H + h) * T + t) * T;
                const real* dy = dout + ((size_t)b * T + t) * C + (size_t)h * hd;
                const real* q = qkv + ((size_t)b * T + t) * C3 + (size_t)h * hd;
                real* dq = dqkv + ((size_t)b * T + t) * C3 + (size_t)h * hd;
                real dot = 0;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* v = qkv + ((size_t)b * T + t2) * C3 + 2 * (size_t)C + (size_t)h * hd;
                    real* dv = dqkv + ((size_t)b * T + t2) * C3 + 2 * (size_t)C + (size_t)h * hd;
                    real s = 0;
                    for (int i = 0; i < hd; i++) {
                        s += dy[i] * v[i];
                        dv[i] += a[t2] * dy[i];
                    }
                    dA[t2] = s;
                    dot += a[t2] * s;
                }
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* k = qkv + ((size_t)b * T + t2) * C3 + C + (size_t)h * hd;
                    real* dk = dqkv + ((size_t)b * T + t2) * C3 + C + (size_t)h * hd;
                    real ds = a[t2] * (dA[t2] - dot) * scale;
                    for (int i = 0; i < hd; i++) {
                        dq[i] += ds * k[i];
                        dk[i] += ds * q[i];
                    }
                }
            }
            free(dA);
        }
}

/* GELU, tanh form (Hendrycks & Gimpel 2016) */
static real og_gelu_scalar(real x) {
    real k = sqrt(2 / (real)OG_PI);
    real u = k * (x + (real)0.044715 * x * x * x);
    return (real)0.5 * x * (1 + tanh(u));
}

/* derivative of og_gelu_scalar, taken analytically */
static real og_gelu_grad_scalar(real x) {
    real k = sqrt(2 / (real)OG_PI);
    real u = k * (x + (real)0.044715 * x * x * x);
    real th = tanh(u);
    real du = k * (1 + 3 * (real)0.044715 * x * x);
    return (real)0.5 * (1 + th) + (real)0.5 * x * (1 - th * th) * du;
}

void og_gelu_forward(real* out, const real* inp, size_t n) {
    for (size_t i = 0; i < n; i++) out[i] = og_gelu_scalar(inp[i]);
}

/* dinp = gelu'(inp) * dout  (overwrites dinp) */
void og_gelu_backward(real* dinp, const real* inp, const real* dout, size_t n) {
    for (size_t i = 0; i < n; i++) dinp[i] = og_gelu_grad_scalar(inp[i]) * dout[i];
}

/* out = a + b */
void og_residual_forward(real* out, const real* a, const real* b, size_t n) {
    for (size_t i = 0; i < n; i++) out[i] = a[i] + b[i];
}

/* Softmax over the first V of Vp columns and cross-entropy per row.
 * probs pad columns are set to 0.  losses[n] = lse_n - logits[n, tgt[n]]. */
void og_crossentropy_forward(real* probs, real* losses, const real* logits,
                             const int* tgt, int N, int V, int Vp) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* z = logits + (size_t)n * Vp;
        real* p = probs + (size_t)n * Vp;
        real mx = -INFINITY;
        for (int j = 0; j < V; j++)
            if (z[j] > mx) mx = z[j];
        real sum = 0;
        for (int j = 0; j < V; j++) sum += exp(z[j] - mx);
        for (int j = 0; j < V; j++) p[j] = exp(z[j] - mx) / sum;
        for (int j = V; j < Vp; j++) p[j] = 0;
        real lse = mx + log(sum);
        losses[n] = lse - z[tgt[n]];
    }
}

/* dlogits[n,j] = (probs[n,j] - [j == tgt[n]]) * dloss for j < V; 0 for pads.
 * (overwrites dlogits) */
void og_crossentropy_backward(real* dlogits, const real* probs, const int* tgt,
                              real dloss, int N, int V, int Vp) {
    for (int n = 0; n < N; n++) {
        for (int j = 0; j < Vp; j++) {
            real ind = (j == tgt[n]) ? 1 : 0;
            dlogits[(size_t)n * Vp + j] = (j < V) ? (probs[(size_t)n * Vp + j] - ind) * dloss : 0;
        }
    }
}

/* sum of squares of g (in index order), accumulated in double in either
 * build: the global gradient norm sums ~10^8 squares, and a float running sum
 * of that many terms drops most of the later ones once the total is large
 * (4.5% low at the 124M size), which is no evaluation of the definition */
real og_sumsq(const real* g, size_t n) {
    double s = 0;
    for (size_t i = 0; i < n; i++) s += (double)g[i] * (double)g[i];
    return (real)s;
}

/* One AdamW update of n elements at step t (t >= 1), on gradient g*gscale.
 * decay != 0 applies the decoupled term lr*wd*w.  */
void og_adamw(real* w, real* m, real* v, const real* g, size_t n, real gscale,
              real lr, real b1, real b2, real eps, real wd, int decay, int t) {
    real bc1 = 1 - pow(b1, t), bc2 = 1 - pow(b2, t);
    for (size_t i = 0; i < n; i++) {
        real gi = g[i] * gscale;
        m[i] = b1 * m[i] + (1 - b1) * gi;
        v[i] = b2 * v[i] + (1 - b2) * gi * gi;
        real mhat = m[i] / bc1;
        real vhat = v[i] / bc2;
        w[i] = w[i] - lr * (mhat / (sqrt(vhat) + eps) + (decay ? wd * w[i] : 0));
    }
}

/* ------------------------------------------------------------------ */
/* Whole model                                                         */
/* ------------------------------------------------------------------ */

typedef struct {
    int L, H, C, V, Vp, T, B;
    size_t sizes[P_COUNT], offs[P_COUNT], nparams;
    real *params, *grads, *m, *v;
    int t, n_accum, have_fwd;
    int *tokens, *targets;
    /* activations (per layer where indexed by l) */
    real *encoded;                          /* [BT,C] */
    real *ln1, *ln1_mean, *ln1_rstd;        /* [L,BT,C], [L,BT] */
    real *qkv;                              /* [L,BT,3C] */
    real *atty;                             /* [L,BT,C] */
    real *att;                              /* [L,B,H,T,T] */
    real *attproj, *resid2;                 /* [L,BT,C] */
    real *ln2, *ln2_mean, *ln2_rstd;        /* [L,BT,C], [L,BT] */
    real *fch, *fch_gelu;                   /* [L,BT,4C] */
    real *fcproj, *resid3;                  /* [L,BT,C] */
    real *lnf, *lnf_mean, *lnf_rstd;        /* [BT,C], [BT] */
    real *logits, *probs, *losses;          /* [BT,Vp], [BT,Vp], [BT] */
    real mean_loss;
} og_model;

static real* og_zalloc(size_t n) {
    real* p = (real*)calloc(n ? n : 1, sizeof(real));
    if (!p) {
        fprintf(stderr, "gpt2_oracle: out of memory (%zu elements)\n", n);
        abort();
    }
    return p;
}

static real* P(og_model* g, int which, int l) {
    size_t per = g->sizes[which];
    if (which >= P_LN1W && which <= P_FCPROJB) per /= (size_t)g->L;
    return g->params + g->offs[which] + (size_t)l * per;
}

static real* G(og_model* g, int which, int l) {
    size_t per = g->sizes[which];
    if (which >= P_LN1W && which <= P_FCPROJB) per /= (size_t)g->L;
    return g->grads + g->offs[which] + (size_t)l * per;
}

/* Fill params with the seeded init (see header). */
static void og_init_params(og_model* g, uint64_t seed) {
    double std = 0.02, std_res = 0.02 / sqrt(2.0 * g->L);
    for (int k = 0; k < P_COUNT; k++) {
        /* each element depends only on (seed, its index): iterations are independent */
#pragma omp parallel for schedule(static)
        for (size_t j = 0; j < g->sizes[k]; j++) {
            size_t i = g->offs[k] + j;
            real val;
            switch (k) {
                case P_WTE:
                    val = ((int)(j / g->C) < g->V) ? (real)og_normal_sample(seed, i, std) : 0;
                    break;
                case P_WPE: case P_QKVW: case P_FCW:
                    val = (real)og_normal_sample(seed, i, std);
                    break;
                case P_PROJW: case P_FCPROJW:
                    val = (real)og_normal_sample(seed, i, std_res);
                    break;
                case P_LN1W: case P_LN2W: case P_LNFW:
                    val = 1;
                    break;
                default:
                    val = 0;
            }
            g->params[i] = val;
        }
    }
}

og_model* og_create(int L, int H, int C, int V, int T, int B, uint64_t seed) {
    if (L < 1 || H < 1 || C < 1 || C % H || V < 1 || T < 1 || B < 1) return NULL;
    og_model* g = (og_model*)calloc(1, sizeof(og_model));
    g->L = L; g->H = H; g->C = C; g->V = V; g->Vp = og_padded_vocab(V);
    g->T = T; g->B = B;
    og_param_sizes(g->sizes, L, C, g->Vp, T);
    size_t off = 0;
    for (int k = 0; k < P_COUNT; k++) { g->offs[k] = off; off += g->sizes[k]; }
    g->nparams = off;
    g->params = og_zalloc(off);
    g->grads = og_zalloc(off);
    g->m = og_zalloc(off);
    g->v = og_zalloc(off);
    og_init_params(g, seed);
    size_t BT = (size_t)B * T, c = (size_t)C, l = (size_t)L;
    g->tokens = (int*)calloc(BT, sizeof(int));
    g->targets = (int*)calloc(BT, sizeof(int));
    g->encoded = og_zalloc(BT * c);
    g->ln1 = og_zalloc(l * BT * c);
    g->ln1_mean = og_zalloc(l * BT);
    g->ln1_rstd = og_zalloc(l * BT);
    g->qkv = og_zalloc(l * BT * 3 * c);
    g->atty = og_zalloc(l * BT * c);
    g->att = og_zalloc(l * (size_t)B * H * T * T);
    g->attproj = og_zalloc(l * BT * c);
    g->resid2 = og_zalloc(l * BT * c);
    g->ln2 = og_zalloc(l * BT * c);
    g->ln2_mean = og_zalloc(l * BT);
    g->ln2_rstd = og_zalloc(l * BT);
    g->fch = og_zalloc(l * BT * 4 * c);
    g->fch_gelu = og_zalloc(l * BT * 4 * c);
    g->fcproj = og_zalloc(l * BT * c);
    g->resid3 = og_zalloc(l * BT * c);
    g->lnf = og_zalloc(BT * c);
    g->lnf_mean = og_zalloc(BT);
    g->lnf_rstd = og_zalloc(BT);
    g->logits = og_zalloc(BT * g->Vp);
    g->probs = og_zalloc(BT * g->Vp);
    g->losses = og_zalloc(BT);
    return g;
}

void og_destroy(og_model* g) {
    if (!g) return;
    real* bufs[] = {g->params, g->grads, g->m, g->v, g->encoded, g->ln1, g->ln1_mean,
                    g->ln1_rstd, g->qkv, g->atty, g->att, g->attproj, g->resid2, g->ln2,
                    g->ln2_mean, g->ln2_rstd, g->fch, g->fch_gelu, g->fcproj, g->resid3,
                    g->lnf, g->lnf_mean, g->lnf_rstd, g->logits, g->probs, g->losses};
    for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); i++) free(bufs[i]);
    free(g->tokens);
    free(g->targets);
    free(g);
}

size_t og_num_params(og_model* g) { return g->nparams; }
int og_padded_V(og_model* g) { return g->Vp; }

/* Forward pass.  targets may be NULL (then no loss; returns NaN).
 * Returns -1e30 if a token or target is outside [0, V). */
double og_forward(og_model* g, const int* tokens, const int* targets) {
    int B = g->B, T = g->T, C = g->C, L = g->L, H = g->H, V = g->V, Vp = g->Vp;
    size_t BT = (size_t)B * T, c = (size_t)C;
    for (size_t i = 0; i < BT; i++) {
        if (tokens[i] < 0 || tokens[i] >= V) return -1e30;
        if (targets && (targets[i] < 0 || targets[i] >= V)) return -1e30;
    }
    memcpy(g->tokens, tokens, BT * sizeof(int));
    og_encoder_forward(g->encoded, tokens, P(g, P_WTE, 0), P(g, P_WPE, 0), B, T, C);
    const real* resid = g->encoded;
    for (int l = 0; l < L; l++) {
        real* ln1 = g->ln1 + l * BT * c;
        real* qkv = g->qkv + l * BT * 3 * c;
        real* atty = g->atty + l * BT * c;
        real* att = g->att + l * (size_t)B * H * T * T;
        real* attproj = g->attproj + l * BT * c;
        real* resid2 = g->resid2 + l * BT * c;
        real* ln2 = g->ln2 + l * BT * c;
        real* fch = g->fch + l * BT * 4 * c;
        real* fch_gelu = g->fch_gelu + l * BT * 4 * c;
        real* fcproj = g->fcproj + l * BT * c;
        real* resid3 = g->resid3 + l * BT * c;
        og_layernorm_forward(ln1, g->ln1_mean + l * BT, g->ln1_rstd + l * BT, resid,
                             P(g, P_LN1W, l), P(g, P_LN1B, l), (int)BT, C);
        og_matmul_forward(qkv, ln1, P(g, P_QKVW, l), P(g, P_QKVB, l), (int)BT, C, 3 * C);
        og_attention_forward(atty, att, qkv, B, T, C, H);
        og_matmul_forward(attproj, atty, P(g, P_PROJW, l), P(g, P_PROJB, l), (int)BT, C, C);
        og_residual_forward(resid2, resid, attproj, BT * c);
        og_layernorm_forward(ln2, g->ln2_mean + l * BT, g->ln2_rstd + l * BT, resid2,
                             P(g, P_LN2W, l), P(g, P_LN2B, l), (int)BT, C);
        og_matmul_forward(fch, ln2, P(g, P_FCW, l), P(g, P_FCB, l), (int)BT, C, 4 * C);
        og_gelu_forward(fch_gelu, fch, BT * 4 * c);
        og_matmul_forward(fcproj, fch_gelu, P(g, P_FCPROJW, l), P(g, P_FCPROJB, l), (int)BT,
                          4 * C, C);
        og_residual_forward(resid3, resid2, fcproj, BT * c);
        resid = resid3;
    }
    og_layernorm_forward(g->lnf, g->lnf_mean, g->lnf_rstd, resid, P(g, P_LNFW, 0),
                         P(g, P_LNFB, 0), (int)BT, C);
    og_matmul_forward(g->logits, g->lnf, P(g, P_WTE, 0), NULL, (int)BT, C, Vp);
    g->have_fwd = 0;
    if (!targets) return NAN;
    memcpy(g->targets, targets, BT * sizeof(int));
    og_crossentropy_forward(g->probs, g->losses, g->logits, targets, (int)BT, V, Vp);
    real s = 0;
    for (size_t i = 0; i < BT; i++) s += g->losses[i];
    g->mean_loss = s / (real)BT;
    g->have_fwd = 1;
    return (double)g->mean_loss;
}

/* Backward of the last forward (which must have had targets); gradients
 * are accumulated into grads.  Returns 0, or -1 without a forward. */
int og_backward(og_model* g) {
    if (!g->have_fwd) return -1;
    int B = g->B, T = g->T, C = g->C, L = g->L, H = g->H, V = g->V, Vp = g->Vp;
    size_t BT = (size_t)B * T, c = (size_t)C;
    real* dlogits = og_zalloc(BT * Vp);
    real* dlnf = og_zalloc(BT * c);
    real* dresid = og_zalloc(BT * c);
    real* dfch_gelu = og_zalloc(BT * 4 * c);
    real* dfch = og_zalloc(BT * 4 * c);
    real* dln2 = og_zalloc(BT * c);
    real* datty = og_zalloc(BT * c);
    real* dqkv = og_zalloc(BT * 3 * c);
    real* dln1 = og_zalloc(BT * c);

    og_crossentropy_backward(dlogits, g->probs, g->targets, 1 / (real)BT, (int)BT, V, Vp);
    og_matmul_backward(dlnf, G(g, P_WTE, 0), NULL, dlogits, g->lnf, P(g, P_WTE, 0), (int)BT, C, Vp);
    const real* residL = L > 0 ? g->resid3 + (size_t)(L - 1) * BT * c : g->encoded;
    og_layernorm_backward(dresid, G(g, P_LNFW, 0), G(g, P_LNFB, 0), dlnf, residL,
                          P(g, P_LNFW, 0), g->lnf_mean, g->lnf_rstd, (int)BT, C);
    for (int l = L - 1; l >= 0; l--) {
        const real* resid_in = l == 0 ? g->encoded : g->resid3 + (size_t)(l - 1) * BT * c;
        real* ln1 = g->ln1 + l * BT * c;
        real* qkv = g->qkv + l * BT * 3 * c;
        real* atty = g->atty + l * BT * c;
        real* att = g->att + l * (size_t)B * H * T * T;
        real* resid2 = g->resid2 + l * BT * c;
        real* ln2 = g->ln2 + l * BT * c;
        real* fch = g->fch + l * BT * 4 * c;
        real* fch_gelu = g->fch_gelu + l * BT * 4 * c;
        memset(dfch_gelu, 0, sizeof(real) * BT * 4 * c);
        memset(dln2, 0, sizeof(real) * BT * c);
        memset(datty, 0, sizeof(real) * BT * c);
        memset(dqkv, 0, sizeof(real) * BT * 3 * c);
        memset(dln1, 0, sizeof(real) * BT * c);
        /* MLP branch: resid3 = resid2 + fcproj(gelu(fc(ln2(resid2)))) */
        og_matmul_backward(dfch_gelu, G(g, P_FCPROJW, l), G(g, P_FCPROJB, l), dresid, fch_gelu,
                           P(g, P_FCPROJW, l), (int)BT, 4 * C, C);
        og_gelu_backward(dfch, fch, dfch_gelu, BT * 4 * c);
        og_matmul_backward(dln2, G(g, P_FCW, l), G(g, P_FCB, l), dfch, ln2, P(g, P_FCW, l),
                           (int)BT, C, 4 * C);
        og_layernorm_backward(dresid, G(g, P_LN2W, l), G(g, P_LN2B, l), dln2, resid2,
                              P(g, P_LN2W, l), g->ln2_mean + l * BT, g->ln2_rstd + l * BT,
                              (int)BT, C);
        /* attention branch: resid2 = resid_in + proj(attn(qkv(ln1(resid_in)))) */
        og_matmul_backward(datty, G(g, P_PROJW, l), G(g, P_PROJB, l), dresid, atty,
                           P(g, P_PROJW, l), (int)BT, C, C);
        og_attention_backward(dqkv, datty, qkv, att, B, T, C, H);
        og_matmul_backward(dln1, G(g, P_QKVW, l), G(g, P_QKVB, l), dqkv, ln1, P(g, P_QKVW, l),
                           (int)BT, C, 3 * C);
        og_layernorm_backward(dresid, G(g, P_LN1W, l), G(g, P_LN1B, l), dln1, resid_in,
                              P(g, P_LN1W, l), g->ln1_mean + l * BT, g->ln1_rstd + l * BT,
                              (int)BT, C);
    }
    og_encoder_backward(G(g, P_WTE, 0), G(g, P_WPE, 0), dresid, g->tokens, B, T, C);
    free(dlogits); free(dlnf); free(dresid); free(dfch_gelu); free(dfch);
    free(dln2); free(datty); free(dqkv); free(dln1);
    g->n_accum++;
    return 0;
}

void og_zero_grad(og_model* g) {
    memset(g->grads, 0, sizeof(real) * g->nparams);
    g->n_accum = 0;
}

static int og_decayed(int k) {
    return k == P_WTE || k == P_WPE || k == P_QKVW || k == P_PROJW || k == P_FCW ||
           k == P_FCPROJW;
}

/* Optimizer step over all parameters.  Returns 0 on success, -1 if no
 * backward was accumulated, -6 (and changes nothing) if the norm of the
 * averaged gradient is not finite.  *norm_out gets that norm. */
int og_adamw_step(og_model* g, double lr, double b1, double b2, double eps,
                  double wd, double clip, double* norm_out) {
    if (g->n_accum < 1) return -1;
    real inv_accum = 1 / (real)g->n_accum;
    real norm = sqrt(og_sumsq(g->grads, g->nparams)) * inv_accum;
    if (norm_out) *norm_out = (double)norm;
    if (!isfinite(norm)) return -6;
    real s = (clip > 0 && norm > clip) ? (real)clip / norm : 1;
    g->t += 1;
    for (int k = 0; k < P_COUNT; k++) {
        size_t o = g->offs[k];
        og_adamw(g->params + o, g->m + o, g->v + o, g->grads + o, g->sizes[k], inv_accum * s,
                 (real)lr, (real)b1, (real)b2, (real)eps, (real)wd, og_decayed(k), g->t);
    }
    return 0;
}

/* ---- accessors (copy in/out as double regardless of `real`) ---- */

static void og_copy_out(double* dst, const real* src, size_t n) {
    for (size_t i = 0; i < n; i++) dst[i] = (double)src[i];
}
static void og_copy_in(real* dst, const double* src, size_t n) {
    for (size_t i = 0; i < n; i++) dst[i] = (real)src[i];
}

void og_get_params(og_model* g, double* out) { og_copy_out(out, g->params, g->nparams); }
void og_set_params(og_model* g, const double* in) { og_copy_in(g->params, in, g->nparams); }
void og_get_grads(og_model* g, double* out) { og_copy_out(out, g->grads, g->nparams); }
void og_set_grads(og_model* g, const double* in) { og_copy_in(g->grads, in, g->nparams); }
void og_get_m(og_model* g, double* out) { og_copy_out(out, g->m, g->nparams); }
void og_get_v(og_model* g, double* out) { og_copy_out(out, g->v, g->nparams); }
double og_get_param(og_model* g, size_t i) { return (double)g->params[i]; }
void og_set_param(og_model* g, size_t i, double x) { g->params[i] = (real)x; }
void og_set_n_accum(og_model* g, int n) { g->n_accum = n; }
int og_get_step(og_model* g) { return g->t; }

/* logits [B*T, V] (real vocabulary columns only) */
void og_get_logits(og_model* g, double* out) {
    size_t BT = (size_t)g->B * g->T;
    for (size_t n = 0; n < BT; n++)
        for (int j = 0; j < g->V; j++) out[n * g->V + j] = (double)g->logits[n * g->Vp + j];
}
/* softmax probabilities [B*T, V] of the last forward with targets */
void og_get_probs(og_model* g, double* out) {
    size_t BT = (size_t)g->B * g->T;
    for (size_t n = 0; n < BT; n++)
        for (int j = 0; j < g->V; j++) out[n * g->V + j] = (double)g->probs[n * g->Vp + j];
}
void og_get_losses(og_model* g, double* out) {
    og_copy_out(out, g->losses, (size_t)g->B * g->T);
}
/* final LayerNorm output [B*T, C] */
void og_get_lnf(og_model* g, double* out) {
    og_copy_out(out, g->lnf, (size_t)g->B * g->T * g->C);
}
/* offset and size of canonical tensor k (0..15), for tests */
size_t og_tensor_offset(og_model* g, int k) { return g->offs[k]; }
size_t og_tensor_size(og_model* g, int k) { return g->sizes[k]; }
