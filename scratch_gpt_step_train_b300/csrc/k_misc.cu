// k_misc.cu -- the memory-bound kernels of the GPT-2 step: parameter init,
// embedding forward/backward, LayerNorm forward/backward, bias gradients,
// fused softmax cross-entropy, and the AdamW update with global-norm clipping.
//
// Sources (page title, section):
//  * "Karpathy's llm.c: understanding LLM training from scratch in C/CUDA",
//    "Code anatomy": encoder_forward / encoder_backward, layernorm_forward,
//    warp_reduce_max / warp_reduce_sum shuffle reductions, the single-kernel
//    update_params, explicit bf16 compute copies of fp32 master weights.
//  * "Karpathy reproduces GPT-2 (1.6B) in llm.c", "Training" and the flag
//    guide: AdamW with weight decay on 2-D weights only, gradient-norm clip,
//    gradient accumulation; "PyTorch comparison": the fused classifier that
//    never materialises the probabilities, vocabulary padded to 50304.
// Every reduction below runs in a fixed order (no float atomics), so a rerun
// on the same inputs gives the same bits.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <algorithm>
#include <math.h>
#include <type_traits>

namespace gk {

static inline int cdiv(long a, long b) { return (int)((a + b - 1) / b); }

void make_layout(ParamLayout* lay, int L, int C, int V, int T) {
    size_t c = (size_t)C, l = (size_t)L;
    int Vp = ((V + 127) / 128) * 128;
    size_t sz[P_NUM] = {(size_t)Vp * c, (size_t)T * c, l * c, l * c, l * 3 * c * c, l * 3 * c,
                        l * c * c, l * c, l * c, l * c, l * 4 * c * c, l * 4 * c,
                        l * 4 * c * c, l * c, c, c};
    size_t o = 0;
    for (int k = 0; k < P_NUM; k++) {
        lay->off[k] = o;
        o += sz[k];
    }
    lay->off[P_NUM] = o;
    lay->L = L; lay->C = C; lay->V = V; lay->Vp = Vp; lay->T = T;
}

// ===========================================================================
// Parameter init: SplitMix64 (Steele, Lea & Flood 2014) counter stream and the
// Box-Muller transform (Box & Muller 1958) in double, rounded to fp32.
// ===========================================================================
__device__ __forceinline__ uint64_t sm64_at(uint64_t seed, uint64_t j) {
    // state after j+1 increments of the Weyl sequence, then the output mix
    uint64_t z = seed + (j + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
__device__ __forceinline__ double unit_open(uint64_t x) {
    return ((double)(x >> 11) + 0.5) * 0x1.0p-53;
}

__global__ void k_init_params(float* p, ParamLayout lay, uint64_t seed, double sd, double sd_res) {
    gdc_wait();
    gdc_launch_dependents();
    size_t n = lay.off[P_NUM];
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        int k = 0;
        while (k + 1 < P_NUM && lay.off[k + 1] <= i) k++;
        double std = 0.0;
        float fixed = 0.0f;
        switch (k) {
            case P_WTE:
                if ((i - lay.off[P_WTE]) / (size_t)lay.C < (size_t)lay.V) std = sd;
                break;
            case P_WPE: case P_QKVW: case P_FCW: std = sd; break;
            case P_PROJW: case P_FCPROJW: std = sd_res; break;
            case P_LN1W: case P_LN2W: case P_LNFW: fixed = 1.0f; break;
            default: break;
        }
        if (std > 0.0) {
            double u1 = unit_open(sm64_at(seed, 2 * (uint64_t)i));
            double u2 = unit_open(sm64_at(seed, 2 * (uint64_t)i + 1));
            double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
            p[i] = (float)(z * std);
        } else {
            p[i] = fixed;
        }
    }
}

cudaError_t init_params(float* master, const ParamLayout& lay, uint64_t seed, cudaStream_t s) {
    launch_pdl(k_init_params, 148 * 8, 256, 0, s, master, lay, seed, 0.02, 0.02 / sqrt(2.0 * lay.L));
    return cudaGetLastError();
}

// ===========================================================================
// Stochastic rounding fp32 -> bf16 with a counter-based random stream: the
// element rounded with counter value k takes the top 16 bits r of the k-th
// SplitMix64 output of seed s and becomes (bits(x) + r) >> 16.  Since the
// formats are sign-magnitude, that rounds |x| up with probability
// (low 16 bits of x) / 65536, down otherwise: unbiased.  NaN stays NaN.
// ===========================================================================
__device__ __forceinline__ uint16_t sround_bf16(float x, uint64_t word) {
    const uint32_t b = __float_as_uint(x);
    if ((b & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;  // NaN
    return (uint16_t)((b + (uint32_t)(word >> 48)) >> 16);
}
__global__ void k_sround(uint16_t* out, const float* in, size_t n, uint64_t seed, uint64_t k0) {
    gdc_wait();
    gdc_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        out[i] = sround_bf16(in[i], sm64_at(seed, k0 + i));
}
cudaError_t stochastic_round_bf16(void* out, const float* in, size_t n, uint64_t seed,
                                  uint64_t k0, cudaStream_t s) {
    launch_pdl(k_sround, 148 * 8, 256, 0, s, (uint16_t*)out, in, n, seed, k0);
    return cudaGetLastError();
}

__global__ void k_cast_bf16(bf16* dst, const float* src, size_t n) {
    gdc_wait();
    gdc_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __float2bfloat16_rn(src[i]);
}
cudaError_t cast_to_bf16(void* dst, const float* src, size_t n, cudaStream_t s) {
    launch_pdl(k_cast_bf16, 148 * 8, 256, 0, s, (bf16*)dst, src, n);
    return cudaGetLastError();
}

// ===========================================================================
// Embedding forward: one thread per VEC-wide chunk of a row.
// ===========================================================================
template <typename T, int VEC>
__global__ void k_encoder_fwd(T* out, const int* tok, const T* wte, const T* wpe, int BT, int T_,
                              int C, int V, unsigned* err) {
    gdc_wait();
    gdc_launch_dependents();
    int cv = C / VEC;
    long total = (long)BT * cv;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total;
         idx += (long)gridDim.x * blockDim.x) {
        int row = (int)(idx / cv), c = (int)(idx % cv) * VEC;
        int id = tok[row];
        if (id < 0 || id >= V) {
            if (c == 0) atomicOr(err, GPT2_DEVERR_TOKEN);
            id = 0;
        }
        int t = row % T_;
        float a[VEC], b[VEC];
        load_vec_f<T, VEC>(a, wte + (size_t)id * C + c);
        load_vec_f<T, VEC>(b, wpe + (size_t)t * C + c);
#pragma unroll
        for (int j = 0; j < VEC; j++) a[j] += b[j];
        store_vec_f<T, VEC>(out + (size_t)row * C + c, a);
    }
}

template <typename T>
static cudaError_t enc_fwd_t(void* out, const int* tok, const void* wte, const void* wpe, int B,
                             int T_, int C, int V, unsigned* err, cudaStream_t s) {
    int BT = B * T_;
    constexpr int VM = 16 / sizeof(T);
    if (C % VM == 0) {
        long total = (long)BT * (C / VM);
        launch_pdl(k_encoder_fwd<T, VM>, cdiv(total, 256) < 148 * 16 ? cdiv(total, 256) : 148 * 16, 256, 0, s, (T*)out, tok, (const T*)wte, (const T*)wpe, BT, T_, C, V, err);
    } else {
        long total = (long)BT * C;
        launch_pdl(k_encoder_fwd<T, 1>, cdiv(total, 256) < 148 * 16 ? cdiv(total, 256) : 148 * 16, 256, 0, s, (T*)out, tok, (const T*)wte, (const T*)wpe, BT, T_, C, V, err);
    }
    return cudaGetLastError();
}
cudaError_t encoder_forward(int act, void* out, const int* tok, const void* wte, const void* wpe,
                            int B, int T_, int C, int V, unsigned* err, cudaStream_t s) {
    if (act == ACT_BF16) return enc_fwd_t<bf16>(out, tok, wte, wpe, B, T_, C, V, err, s);
    return enc_fwd_t<float>(out, tok, wte, wpe, B, T_, C, V, err, s);
}

// ===========================================================================
// Elementwise GELU, out = gelu(in), with the same device function
// (gelu_and_grad_f) as the fp32 fused epilogue, so that an output recomputed
// later from the same input is bit for bit the one computed first.
// ===========================================================================
template <typename T, int VEC>
__global__ void __launch_bounds__(256) k_gelu_fwd(T* out, const T* in, size_t n) {
    gdc_wait();
    gdc_launch_dependents();
    const size_t nv = n / VEC;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nv;
         i += (size_t)gridDim.x * blockDim.x) {
        float x[VEC], y[VEC];
        load_vec_f<T, VEC>(x, in + i * VEC);
#pragma unroll
        for (int j = 0; j < VEC; j++) {
            float dg;
            gelu_and_grad_f(x[j], y[j], dg);
        }
        store_vec_f<T, VEC>(out + i * VEC, y);
    }
    for (size_t e = nv * VEC + blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
         e += (size_t)gridDim.x * blockDim.x) {
        float y, dg;
        gelu_and_grad_f(to_f(in[e]), y, dg);
        out[e] = from_f<T>(y);
    }
}
cudaError_t gelu_forward(int act, void* out, const void* in, size_t n, cudaStream_t s) {
    if (act == ACT_BF16) {
        if (((uintptr_t)out | (uintptr_t)in) & 15)
            launch_pdl(k_gelu_fwd<bf16, 1>, 148 * 8, 256, 0, s, (bf16*)out, (const bf16*)in, n);
        else
            launch_pdl(k_gelu_fwd<bf16, 8>, 148 * 8, 256, 0, s, (bf16*)out, (const bf16*)in, n);
    } else {
        if (((uintptr_t)out | (uintptr_t)in) & 15)
            launch_pdl(k_gelu_fwd<float, 1>, 148 * 8, 256, 0, s, (float*)out, (const float*)in, n);
        else
            launch_pdl(k_gelu_fwd<float, 4>, 148 * 8, 256, 0, s, (float*)out, (const float*)in, n);
    }
    return cudaGetLastError();
}

// ===========================================================================
// LayerNorm forward: one warp per row, mean, rstd = 1/sqrt(var + 1e-5) with
// the biased variance.  Persistent warps walk the rows with a stride; the next
// row's data (packed, VEC-wide loads) is in flight while the current row is
// normalised.
// ===========================================================================
template <typename T, int VEC, int IT>
__global__ void __launch_bounds__(256) k_ln_fwd(T* out, float* mean, float* rstd, const T* x,
                                                const T* w, const T* b, int N, int C) {
    gdc_wait();
    gdc_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x / 32);
    int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    Vec<T, VEC> cur[IT], nxt[IT];
    auto load = [&](int r, Vec<T, VEC>* v) {
        if (r < N) {
#pragma unroll
            for (int it = 0; it < IT; it++) {
                const int c = (it * 32 + lane) * VEC;
                if (c < C) v[it] = *reinterpret_cast<const Vec<T, VEC>*>(x + (size_t)r * C + c);
            }
        }
    };
    load(row, cur);
    for (; row < N; row += nw) {
        load(row + nw, nxt);
        float s = 0.f;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            if ((it * 32 + lane) * VEC < C) {
#pragma unroll
                for (int j = 0; j < VEC; j++) s += to_f(cur[it].v[j]);
            }
        }
        const float m = warp_sum(s) / C;
        float ss = 0.f;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            if ((it * 32 + lane) * VEC < C) {
#pragma unroll
                for (int j = 0; j < VEC; j++) {
                    const float d = to_f(cur[it].v[j]) - m;
                    ss += d * d;
                }
            }
        }
        const float r = rsqrtf(warp_sum(ss) / C + 1e-5f);
        T* yr = out + (size_t)row * C;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            const int c = (it * 32 + lane) * VEC;
            if (c < C) {
                float wv[VEC], bv[VEC], y[VEC];
                load_vec_f<T, VEC>(wv, w + c);
                load_vec_f<T, VEC>(bv, b + c);
#pragma unroll
                for (int j = 0; j < VEC; j++) y[j] = (to_f(cur[it].v[j]) - m) * r * wv[j] + bv[j];
                store_vec_f<T, VEC>(yr + c, y);
            }
        }
        if (lane == 0) {
            mean[row] = m;
            rstd[row] = r;
        }
#pragma unroll
        for (int it = 0; it < IT; it++) cur[it] = nxt[it];
    }
}

template <typename T, int VEC, int IT>
static cudaError_t ln_fwd_launch(void* out, float* mean, float* rstd, const void* x,
                                 const void* w, const void* b, int N, int C, cudaStream_t s) {
    auto kern = k_ln_fwd<T, VEC, IT>;
    static int occ = 0;  // resident blocks per SM (the same on every device it runs on)
    if (!occ && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 256, 0) != cudaSuccess ||
                 occ < 1))
        occ = 1;
    int dev = 0, nsm = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int nb = std::min(cdiv(N, 8), nsm * occ);
    launch_pdl(kern, nb, 256, 0, s, (T*)out, mean, rstd, (const T*)x, (const T*)w, (const T*)b, N,
               C);
    return cudaGetLastError();
}

template <typename T, int VEC>
static cudaError_t ln_fwd_vec(void* out, float* mean, float* rstd, const void* x, const void* w,
                              const void* b, int N, int C, cudaStream_t s) {
    const int it = cdiv(C, 32 * VEC);
#define LNF(I) return ln_fwd_launch<T, VEC, I>(out, mean, rstd, x, w, b, N, C, s)
    switch (it) {
        case 1: LNF(1);
        case 2: LNF(2);
        case 3: LNF(3);
        case 4: LNF(4);
        case 5: LNF(5);
        case 6: LNF(6);
        case 7: LNF(7);
        case 8: LNF(8);
        default:
            if (it <= 12) LNF(12);
            if (it <= 16) LNF(16);
            return cudaErrorInvalidValue;
    }
#undef LNF
}
template <typename T>
static cudaError_t ln_fwd_t(void* out, float* mean, float* rstd, const void* x, const void* w,
                            const void* b, int N, int C, cudaStream_t s) {
    constexpr int VM = 16 / sizeof(T);
    if (C % VM == 0) return ln_fwd_vec<T, VM>(out, mean, rstd, x, w, b, N, C, s);
    return ln_fwd_vec<T, 1>(out, mean, rstd, x, w, b, N, C, s);
}
cudaError_t layernorm_forward(int act, void* out, float* mean, float* rstd, const void* x,
                              const void* w, const void* b, int N, int C, cudaStream_t s) {
    if (act == ACT_BF16) return ln_fwd_t<bf16>(out, mean, rstd, x, w, b, N, C, s);
    return ln_fwd_t<float>(out, mean, rstd, x, w, b, N, C, s);
}

// ===========================================================================
// LayerNorm backward.  Per row (xhat = (x-mean)*rstd, g = dy*w):
//   dx (+)= rstd * (g - mean(g) - xhat * mean(g*xhat))
// One warp per row.  The column sums dw = sum dy*xhat, db = sum dy (and, when
// asked, dxsum = sum of the written dx rows) are accumulated per lane in shared
// memory: accumulator slot (it*VEC + j)*32 + lane of a warp's slice holds the
// partial of column (it*32 + lane)*VEC + j, so each lane only ever touches its
// own slots and the registers stay free for the row data.  At the end the
// block folds its warps' slices in warp order into one partial row per
// accumulator, and k_colsum adds the block partials in block order.
// ===========================================================================
#define LNB_MAX_BLOCKS 296

// Makes the compiler treat the vector's contents as changed here, so that it
// recomputes what it derived from them before instead of keeping those values
// live in registers (the row data packed as T is the cheaper thing to keep).
template <typename T, int VEC>
__device__ __forceinline__ void opaque(Vec<T, VEC>& v) {
    if constexpr (sizeof(Vec<T, VEC>) % 4 == 0) {
        uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int k = 0; k < (int)(sizeof(Vec<T, VEC>) / 4); k++) asm volatile("" : "+r"(u[k]));
    }
}

template <int VEC, int IT, int NACC>
struct LnbCfg {
    static constexpr int S = IT * VEC * 32;  // accumulator slots per warp
    // 8 warps a block while two blocks' slices fit in shared memory, else 4
    static constexpr int W = (2 * 8 * NACC * S * 4 <= 220 * 1024) ? 8 : 4;
};

template <typename T, int VEC, int IT, int NACC>
__global__ void __launch_bounds__(LnbCfg<VEC, IT, NACC>::W * 32, 2)
    k_ln_bwd(T* dx, float* part, const T* dout, const T* x, const T* w, const float* mean,
             const float* rstd, int N, int C, int accum_dx) {
    gdc_wait();
    gdc_launch_dependents();
    extern __shared__ float lsm[];  // [warps][NACC][S]
    constexpr int S = LnbCfg<VEC, IT, NACC>::S;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x / 32;
    float* acc = lsm + (size_t)warp * NACC * S + lane;
#pragma unroll
    for (int k = 0; k < NACC * IT * VEC; k++) acc[k * 32] = 0.f;
    for (int row = blockIdx.x * nwarps + warp; row < N; row += gridDim.x * nwarps) {
        const T* xr = x + (size_t)row * C;
        const T* dyr = dout + (size_t)row * C;
        T* dxr = dx + (size_t)row * C;
        const float m = mean[row], r = rstd[row];
        // x, dy and the incoming dx of the row are independent loads: issue
        // them together so that the row costs one memory latency
        Vec<T, VEC> xv[IT], dv[IT], ov[IT];
#pragma unroll
        for (int it = 0; it < IT; it++) {
            const int c = (it * 32 + lane) * VEC;
            if (c < C) {
                xv[it] = *reinterpret_cast<const Vec<T, VEC>*>(xr + c);
                dv[it] = *reinterpret_cast<const Vec<T, VEC>*>(dyr + c);
                if (accum_dx) ov[it] = *reinterpret_cast<const Vec<T, VEC>*>(dxr + c);
            }
        }
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            const int c = (it * 32 + lane) * VEC;
            if (c < C) {
                float wv[VEC];
                load_vec_f<T, VEC>(wv, w + c);
#pragma unroll
                for (int j = 0; j < VEC; j++) {
                    const float xh = (to_f(xv[it].v[j]) - m) * r;
                    const float dy = to_f(dv[it].v[j]);
                    const float g = dy * wv[j];
                    sg += g;
                    sgx += g * xh;
                    float* a = acc + (it * VEC + j) * 32;
                    a[0] += dy * xh;
                    a[S] += dy;
                }
            }
        }
        sg = warp_sum(sg) / C;
        sgx = warp_sum(sgx) / C;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            opaque(xv[it]);
            opaque(dv[it]);
        }
        asm volatile("" ::: "memory");  // reload w rather than hold it
#pragma unroll
        for (int it = 0; it < IT; it++) {
            const int c = (it * 32 + lane) * VEC;
            if (c < C) {
                float wv[VEC];
                load_vec_f<T, VEC>(wv, w + c);
                Vec<T, VEC> o;
#pragma unroll
                for (int j = 0; j < VEC; j++) {
                    const float xh = (to_f(xv[it].v[j]) - m) * r;
                    const float g = to_f(dv[it].v[j]) * wv[j];
                    float d = r * (g - sg - xh * sgx);
                    if (accum_dx) d += to_f(ov[it].v[j]);
                    o.v[j] = from_f<T>(d);
                    // the column sum is of the value as stored
                    if (NACC == 3) acc[(2 * IT * VEC + it * VEC + j) * 32] += to_f(o.v[j]);
                }
                *reinterpret_cast<Vec<T, VEC>*>(dxr + c) = o;
            }
        }
    }
    __syncthreads();
    // fold the warps' slices in warp order into this block's partial rows
    for (int s = threadIdx.x; s < NACC * S; s += blockDim.x) {
        const int k = s / S, q = s - k * S;
        const int ln = q & 31, jj = (q >> 5) % VEC, itq = (q >> 5) / VEC;
        const int c = (itq * 32 + ln) * VEC + jj;
        if (c < C) {
            float t = 0.f;
            for (int wi = 0; wi < nwarps; wi++) t += lsm[(size_t)wi * NACC * S + s];
            part[((size_t)blockIdx.x * NACC + k) * C + c] = t;
        }
    }
}

// bf16 rows with C % 8 == 0: the same computation with the column sums in
// registers and the row data staged through shared memory by cp.async.  A row
// is handled by a team of RS warps, each owning a contiguous part of its
// 16-byte column vectors (IT per lane); the team adds its parts' row sums in
// part order through shared memory.  Each lane copies exactly the vectors it
// later reads, into a two-slot ring of its warp, so the copy of the team's next
// row is in flight while it works on the current one, and a lane only ever
// waits for its own copies (cp.async.wait_group).  Registers hold no row data.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int NPEND>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(NPEND) : "memory");
}
__device__ __forceinline__ void bf16x8_to_f(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
// element h (0 = low half) of a packed bf16 pair, widened to fp32
__device__ __forceinline__ float bf_half(uint32_t u, int h) {
    return __uint_as_float(h ? (u & 0xffff0000u) : (u << 16));
}
__device__ __forceinline__ uint32_t pack2_bf16_rn(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int IT, int NACC, int RS>
__global__ void __launch_bounds__(256, 2)
    k_ln_bwd_ring(bf16* dx, float* part, const bf16* dout, const bf16* x, const bf16* w,
                  const float* mean, const float* rstd, int N, int C, int accum_dx) {
    gdc_wait();
    gdc_launch_dependents();
    // ring: [warp][slot 0/1][x | dy | dx][IT*32 vectors]; reused for the fold
    extern __shared__ __align__(16) unsigned char rsm[];
    __shared__ float xch[2][8][2];          // [row parity][warp] partial (sum g, sum g*xhat)
    constexpr int ROWV = IT * 32;           // vectors per row part and array (max)
    constexpr int SLOT = 3 * ROWV * 16;     // bytes per slot
    constexpr bool WREG = IT * (NACC + 1) <= 9;  // w of the lane's columns kept in registers
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x / 32;
    const int teams = nwarps / RS, team = warp / RS, pix = warp % RS;
    const int nvec = C / 8, vpp = (nvec + RS - 1) / RS;
    const int v0 = pix * vpp;
    const int lim = min(nvec, v0 + vpp) - v0;  // vectors of this part: it*32 + lane < lim
    const uint32_t ring = tc::smem_u32(rsm) + (uint32_t)warp * 2 * SLOT;
    float wr[WREG ? IT : 1][8];
    float acc[NACC][IT][8];
    const bf16* wl = w + (v0 + lane) * 8;  // this lane's first vector of w
#pragma unroll
    for (int it = 0; it < IT; it++) {
        const bool ok = it * 32 + lane < lim;
        if (WREG && ok) bf16x8_to_f(*reinterpret_cast<const uint4*>(wl + it * 256), wr[it]);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            if (WREG && !ok) wr[it][j] = 0.f;
#pragma unroll
            for (int a = 0; a < NACC; a++) acc[a][it][j] = 0.f;
        }
    }
    auto wpacked = [&](int it) -> uint4 {  // w of vector it, when not held in registers
        if constexpr (WREG) return make_uint4(0u, 0u, 0u, 0u);
        else return *reinterpret_cast<const uint4*>(wl + it * 256);
    };
    const int stride = gridDim.x * teams;
    auto issue = [&](int row, int slot) {
        if (row < N) {
            const uint32_t base = ring + slot * SLOT + lane * 16;
            const size_t g = (size_t)row * C + (v0 + lane) * 8;
#pragma unroll
            for (int it = 0; it < IT; it++) {
                if (it * 32 + lane < lim) {
                    const uint32_t o = it * 512;
                    cp_async16(base + o, x + g + it * 256);
                    cp_async16(base + ROWV * 16 + o, dout + g + it * 256);
                    if (accum_dx) cp_async16(base + 2 * ROWV * 16 + o, dx + g + it * 256);
                }
            }
        }
        cp_async_commit();  // an empty group past the last row keeps the count uniform
    };
    int row = blockIdx.x * teams + team;
    issue(row, 0);
    for (int k = 0; row < N; row += stride, k++) {
        issue(row + stride, (k + 1) & 1);
        cp_async_wait<1>();  // this lane's copies of `row` have landed
        const unsigned char* sl = rsm + (size_t)warp * 2 * SLOT + (size_t)(k & 1) * SLOT;
        const float m = mean[row], r = rstd[row], mr = -m * r;
        float sg = 0.f, sgx = 0.f;
        // packed bf16 pairs are widened one 32-bit word at a time
#pragma unroll
        for (int it = 0; it < IT; it++) {
            if (it * 32 + lane < lim) {
                const uint4 ux = *reinterpret_cast<const uint4*>(sl + (it * 32 + lane) * 16);
                const uint4 ud =
                    *reinterpret_cast<const uint4*>(sl + ROWV * 16 + (it * 32 + lane) * 16);
                const uint4 uw = wpacked(it);
                const uint32_t xw[4] = {ux.x, ux.y, ux.z, ux.w}, dw4[4] = {ud.x, ud.y, ud.z, ud.w};
                const uint32_t ww[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float xv = bf_half(xw[j >> 1], j & 1), dv = bf_half(dw4[j >> 1], j & 1);
                    const float xh = fmaf(xv, r, mr);
                    const float g = dv * (WREG ? wr[WREG ? it : 0][j] : bf_half(ww[j >> 1], j & 1));
                    sg += g;
                    sgx = fmaf(g, xh, sgx);
                    acc[0][it][j] = fmaf(dv, xh, acc[0][it][j]);
                    acc[1][it][j] += dv;
                }
            }
        }
        sg = warp_sum(sg);
        sgx = warp_sum(sgx);
        if (RS > 1) {
            // the row's sums: the team's parts added in part order
            if (lane == 0) {
                xch[k & 1][warp][0] = sg;
                xch[k & 1][warp][1] = sgx;
            }
            named_bar_sync(1 + team, RS * 32);
            sg = sgx = 0.f;
#pragma unroll
            for (int q = 0; q < RS; q++) {
                sg += xch[k & 1][team * RS + q][0];
                sgx += xch[k & 1][team * RS + q][1];
            }
        }
        sg /= C;
        sgx /= C;
        bf16* dxr = dx + (size_t)row * C + (v0 + lane) * 8;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            if (it * 32 + lane < lim) {
                const uint4 ux = *reinterpret_cast<const uint4*>(sl + (it * 32 + lane) * 16);
                const uint4 ud =
                    *reinterpret_cast<const uint4*>(sl + ROWV * 16 + (it * 32 + lane) * 16);
                uint4 uo = make_uint4(0u, 0u, 0u, 0u);
                if (accum_dx)
                    uo = *reinterpret_cast<const uint4*>(sl + 2 * ROWV * 16 + (it * 32 + lane) * 16);
                const uint4 uw = wpacked(it);
                const uint32_t xw[4] = {ux.x, ux.y, ux.z, ux.w}, dw4[4] = {ud.x, ud.y, ud.z, ud.w};
                const uint32_t ow[4] = {uo.x, uo.y, uo.z, uo.w}, ww[4] = {uw.x, uw.y, uw.z, uw.w};
                uint32_t res[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float d2[2];
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int j = 2 * q + h;
                        const float xh = fmaf(bf_half(xw[q], h), r, mr);
                        const float g = bf_half(dw4[q], h) *
                                        (WREG ? wr[WREG ? it : 0][j] : bf_half(ww[q], h));
                        // bf_half of a zero word is 0 when there is no incoming dx
                        d2[h] = fmaf(r, fmaf(-xh, sgx, g - sg), bf_half(ow[q], h));
                    }
                    res[q] = pack2_bf16_rn(d2[0], d2[1]);
                    if (NACC == 3) {
                        // the column sum is of the value as stored
                        acc[NACC - 1][it][2 * q] += bf_half(res[q], 0);
                        acc[NACC - 1][it][2 * q + 1] += bf_half(res[q], 1);
                    }
                }
                *reinterpret_cast<uint4*>(dxr + it * 256) = make_uint4(res[0], res[1], res[2], res[3]);
            }
        }
    }
    cp_async_wait<0>();  // nothing may still be landing in the ring
    __syncthreads();
    // fold: slot (a, it, j, lane) of warp w at ((w*NACC + a)*IT*8 + it*8 + j)*32 + lane;
    // column vector v0(part) + it*32 + lane is owned by one warp of every team
    constexpr int S = IT * 8 * 32;
    float* fs = reinterpret_cast<float*>(rsm);
#pragma unroll
    for (int a = 0; a < NACC; a++)
#pragma unroll
        for (int it = 0; it < IT; it++)
#pragma unroll
            for (int j = 0; j < 8; j++)
                fs[((size_t)warp * NACC + a) * S + (it * 8 + j) * 32 + lane] = acc[a][it][j];
    __syncthreads();
    for (int q = threadIdx.x; q < NACC * RS * S; q += blockDim.x) {
        const int a = q / (RS * S), rem = q - a * (RS * S);
        const int pq = rem / S, sq = rem - pq * S;
        const int ln = sq & 31, jj = (sq >> 5) & 7, itq = sq >> 8;
        const int vi = pq * vpp + itq * 32 + ln;
        if (itq * 32 + ln < vpp && vi < nvec) {
            float t = 0.f;
            for (int tt = 0; tt < teams; tt++)
                t += fs[((size_t)(tt * RS + pq) * NACC + a) * S + sq];
            part[((size_t)blockIdx.x * NACC + a) * C + vi * 8 + jj] = t;
        }
    }
}

// outs[k][c] += sum_i part[i*ld + k*n0 + c] for column k*n0 + c < ncols, in a
// fixed order: thread row ty (of 8) sums the rows i = ty (mod 8) in four
// interleaved chains (i = ty + 32q + {0, 8, 16, 24}) whose loads are in flight
// together, adds the chains in order, then row 0 adds the 8 row sums in order.
// 32 consecutive columns per block (coalesced).
struct ColsumOut {
    float* p[3];
};
__device__ __forceinline__ void colsum_cols(const ColsumOut& outs, int n0, int ncols,
                                            const float* part, int nparts, long ld, int cblock) {
    __shared__ float sh[8][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int c = cblock * 32 + tx;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < ncols) {
        // 16 independent loads in flight per thread: the partial rows are few
        // (one per producer block), so latency, not bandwidth, sets the time
        for (int i = ty; i < nparts; i += 128) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 16; q++)
                v[q] = i + 8 * q < nparts ? part[(size_t)(i + 8 * q) * ld + c] : 0.f;
#pragma unroll
            for (int q = 0; q < 16; q++) a[q & 3] += v[q];
        }
    }
    sh[ty][tx] = (a[0] + a[1]) + (a[2] + a[3]);
    __syncthreads();
    if (ty == 0 && c < ncols) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; k++) t += sh[k][tx];
        const int k = c / n0;
        outs.p[k][c - k * n0] += t;
    }
}
__global__ void __launch_bounds__(256) k_colsum(ColsumOut outs, int n0, int ncols,
                                                const float* part, int nparts, long ld) {
    gdc_wait();
    gdc_launch_dependents();
    colsum_cols(outs, n0, ncols, part, nparts, ld, blockIdx.x);
}

// Many column sums in one launch: task i owns blocks [blk0[i], blk0[i+1]),
// each summing 32 columns exactly as k_colsum does.
#define COLSUM_MAX_TASKS 96
struct ColsumBatch {
    ColsumTask t[COLSUM_MAX_TASKS];
    int blk0[COLSUM_MAX_TASKS + 1];
    int ntasks;
};
__global__ void __launch_bounds__(256) k_colsum_batch(const __grid_constant__ ColsumBatch b) {
    gdc_wait();
    gdc_launch_dependents();
    int lo = 0, hi = b.ntasks - 1;  // the last task whose first block <= blockIdx.x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (b.blk0[mid] <= (int)blockIdx.x) lo = mid;
        else hi = mid - 1;
    }
    const ColsumTask& t = b.t[lo];
    ColsumOut o{{t.out[0], t.out[1], t.out[2]}};
    colsum_cols(o, t.n0, t.ncols, t.part, t.nparts, (long)t.ncols, (int)blockIdx.x - b.blk0[lo]);
}
cudaError_t colsum_batch(const ColsumTask* tasks, int n, cudaStream_t s, int* nlaunch) {
    if (nlaunch) *nlaunch = 0;
    for (int i0 = 0; i0 < n; i0 += COLSUM_MAX_TASKS) {
        ColsumBatch b;
        b.ntasks = std::min(COLSUM_MAX_TASKS, n - i0);
        int nb = 0;
        for (int i = 0; i < b.ntasks; i++) {
            b.t[i] = tasks[i0 + i];
            b.blk0[i] = nb;
            nb += cdiv(b.t[i].ncols, 32);
        }
        b.blk0[b.ntasks] = nb;
        launch_pdl(k_colsum_batch, nb, 256, 0, s, b);
        if (nlaunch) ++*nlaunch;
    }
    return cudaGetLastError();
}

cudaError_t colsum_add(float* db, const float* part, int nparts, int ncols, cudaStream_t s) {
    ColsumOut o{{db, nullptr, nullptr}};
    launch_pdl(k_colsum, cdiv(ncols, 32), 256, 0, s, o, ncols, ncols, part, nparts, (long)ncols);
    return cudaGetLastError();
}

size_t layernorm_backward_scratch(int N, int C, bool dxsum) {
    return (size_t)LNB_MAX_BLOCKS * (dxsum ? 3 : 2) * C * sizeof(float);
}

template <int IT, int NACC, int RS>
static cudaError_t ln_bwd_ring_launch(bf16* dx, float* part, const bf16* dout, const bf16* x,
                                      const bf16* w, const float* mean, const float* rstd, int N,
                                      int C, int accum, int* nb_out, cudaStream_t s) {
    constexpr size_t smem = (size_t)8 * 2 * 3 * IT * 32 * 16;
    static_assert(smem >= (size_t)8 * NACC * IT * 256 * 4, "fold does not fit the ring");
    auto kern = k_ln_bwd_ring<IT, NACC, RS>;
    // the opt-in always: with the kernel's static shared memory, a ring of
    // exactly 48 KB (C = 1024 with the dxsum column) is already over the default
    {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int nb = cdiv(N, (8 / RS) * 4);
    if (nb > LNB_MAX_BLOCKS) nb = LNB_MAX_BLOCKS;
    *nb_out = nb;
    launch_pdl(kern, nb, 256, smem, s, dx, part, dout, x, w, mean, rstd, N, C, accum);
    return cudaGetLastError();
}

template <typename T, int VEC, int IT, int NACC>
static cudaError_t ln_bwd_launch(T* dx, float* part, const T* dout, const T* x, const T* w,
                                 const float* mean, const float* rstd, int N, int C, int accum,
                                 int* nb_out, cudaStream_t s) {
    if constexpr (std::is_same<T, bf16>::value && VEC == 8) {
        // register column sums, cp.async-staged rows: one warp per row while a
        // lane's column sums fit in registers, else two warps per row
        const int nvec = C / 8;
        if constexpr (IT * NACC <= 9)
            return ln_bwd_ring_launch<IT, NACC, 1>(dx, part, dout, x, w, mean, rstd, N, C, accum,
                                                   nb_out, s);
        const int it2 = cdiv(cdiv(nvec, 2), 32);
        switch (it2) {
            case 2: return ln_bwd_ring_launch<2, NACC, 2>(dx, part, dout, x, w, mean, rstd, N, C,
                                                         accum, nb_out, s);
            case 3: return ln_bwd_ring_launch<3, NACC, 2>(dx, part, dout, x, w, mean, rstd, N, C,
                                                         accum, nb_out, s);
            case 4: return ln_bwd_ring_launch<4, NACC, 2>(dx, part, dout, x, w, mean, rstd, N, C,
                                                         accum, nb_out, s);
            default: break;  // wider rows: shared-memory column sums below
        }
    }
    constexpr int S = LnbCfg<VEC, IT, NACC>::S, W = LnbCfg<VEC, IT, NACC>::W;
    constexpr size_t smem = (size_t)W * NACC * S * sizeof(float);
    static_assert(smem <= 227 * 1024, "LayerNorm backward slices exceed shared memory");
    auto kern = k_ln_bwd<T, VEC, IT, NACC>;
    {  // the opt-in always (dynamic plus static shared memory may pass 48 KB)
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int nb = cdiv(N, W * 4);
    if (nb > LNB_MAX_BLOCKS) nb = LNB_MAX_BLOCKS;
    *nb_out = nb;
    launch_pdl(kern, nb, W * 32, smem, s, dx, part, dout, x, w, mean, rstd, N, C, accum);
    return cudaGetLastError();
}

template <typename T, int VEC, int NACC>
static cudaError_t ln_bwd_vec(T* dx, float* part, const T* dout, const T* x, const T* w,
                              const float* mean, const float* rstd, int N, int C, int accum,
                              int* nb, cudaStream_t s) {
    const int it = cdiv(C, 32 * VEC);
#define LNB(I)                                                                                   \
    return ln_bwd_launch<T, VEC, I, NACC>(dx, part, dout, x, w, mean, rstd, N, C, accum, nb, s)
    switch (it) {
        case 1: LNB(1);
        case 2: LNB(2);
        case 3: LNB(3);
        case 4: LNB(4);
        case 5: LNB(5);
        case 6: LNB(6);
        case 7: LNB(7);
        case 8: LNB(8);
        default:
            if (it <= 12) LNB(12);
            if (it <= 16) LNB(16);
            return cudaErrorInvalidValue;
    }
#undef LNB
}

// the row kernel alone: per-block column partials [nb][nacc * C] into part
template <typename T>
static cudaError_t ln_bwd_rows(void* dx, bool dxsum, const void* dout, const void* x,
                               const void* w, const float* mean, const float* rstd, int N, int C,
                               int accum, float* part, int* nb, cudaStream_t s) {
    constexpr int VM = 16 / sizeof(T);
    *nb = 0;
#define LNV(V, A)                                                                                \
    ln_bwd_vec<T, V, A>((T*)dx, part, (const T*)dout, (const T*)x, (const T*)w, mean, rstd, N,  \
                        C, accum, nb, s)
    if (C % VM == 0) return dxsum ? LNV(VM, 3) : LNV(VM, 2);
    return dxsum ? LNV(1, 3) : LNV(1, 2);
#undef LNV
}
cudaError_t layernorm_backward_rows(int act, void* dx, bool dxsum, const void* dout,
                                    const void* x, const void* w, const float* mean,
                                    const float* rstd, int N, int C, bool accum_dx, float* part,
                                    int* nparts, cudaStream_t s) {
    if (C > 2048) return cudaErrorInvalidValue;
    if (act == ACT_BF16)
        return ln_bwd_rows<bf16>(dx, dxsum, dout, x, w, mean, rstd, N, C, accum_dx, part, nparts,
                                 s);
    return ln_bwd_rows<float>(dx, dxsum, dout, x, w, mean, rstd, N, C, accum_dx, part, nparts,
                              s);
}
cudaError_t layernorm_backward(int act, void* dx, float* dw, float* db, float* dxsum,
                               const void* dout, const void* x, const void* w, const float* mean,
                               const float* rstd, int N, int C, bool accum_dx, void* scratch,
                               cudaStream_t s) {
    float* part = (float*)scratch;
    int nb = 0;
    cudaError_t e = layernorm_backward_rows(act, dx, dxsum != nullptr, dout, x, w, mean, rstd, N,
                                            C, accum_dx, part, &nb, s);
    if (e != cudaSuccess) return e;
    const int nacc = dxsum ? 3 : 2;
    ColsumOut o{{dw, db, dxsum}};
    launch_pdl(k_colsum, cdiv(nacc * C, 32), 256, 0, s, o, C, nacc * C, part, nb, (long)nacc * C);
    return cudaGetLastError();
}

// ===========================================================================
// Bias gradient: db[o] += sum_n dout[n,o].  Rows are cut into chunks of
// BG_ROWS; block (x, p) sums the chunks p, p + P, p + 2P, ... (P = gridDim.y)
// for 32 column vectors into partial row p, and k_colsum adds the P partial
// rows in order -- a fixed summation order whatever the grid's timing.  P is
// chosen so that the grid fills the GPU about four blocks deep.
// ===========================================================================
#define BG_ROWS 64

// block (32 x 8 threads): thread row ty sums rows ty, ty+8, ... of each chunk
// (the chunk's 8 loads issued together), then the 8 row sums are added in order
template <typename T, int VEC>
__global__ void __launch_bounds__(256) k_bias_part(float* part, const T* dout, int N, int OC,
                                                   int nch) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ float sh[8][32 * VEC + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int c = (blockIdx.x * 32 + tx) * VEC;
    float a[VEC];
#pragma unroll
    for (int j = 0; j < VEC; j++) a[j] = 0.f;
    if (c < OC) {
        for (int q = blockIdx.y; q < nch; q += gridDim.y) {
            const int r0 = q * BG_ROWS + ty;
            Vec<T, VEC> v[BG_ROWS / 8];
#pragma unroll
            for (int k = 0; k < BG_ROWS / 8; k++) {
                const int r = r0 + 8 * k;
                if (r < N) {
                    v[k] = *reinterpret_cast<const Vec<T, VEC>*>(dout + (size_t)r * OC + c);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; j++) v[k].v[j] = from_f<T>(0.f);
                }
            }
#pragma unroll
            for (int k = 0; k < BG_ROWS / 8; k++)
#pragma unroll
                for (int j = 0; j < VEC; j++) a[j] += to_f(v[k].v[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < VEC; j++) sh[ty][tx * VEC + j] = a[j];
    __syncthreads();
    if (ty == 0 && c < OC) {
#pragma unroll
        for (int j = 0; j < VEC; j++) {
            float t = 0.f;
#pragma unroll
            for (int k = 0; k < 8; k++) t += sh[k][tx * VEC + j];
            part[(size_t)blockIdx.y * OC + c + j] = t;
        }
    }
}
size_t bias_grad_scratch(int N, int OC) { return (size_t)cdiv(N, BG_ROWS) * OC * sizeof(float); }

template <typename T>
static cudaError_t bias_grad_rows_t(float* part, const void* dout, int N, int OC, int* nparts,
                                    cudaStream_t s) {
    constexpr int VM = 16 / sizeof(T);
    const int nch = cdiv(N, BG_ROWS);
    const int vec = OC % VM == 0 ? VM : 1;
    const int gx = cdiv(OC / vec, 32);
    // P partial rows: as many as keep the whole grid resident (8 blocks of 256
    // threads per SM), preferring a P that divides the chunk count so that
    // every block sums the same number of chunks
    const int pmax = std::max(1, std::min(nch, 148 * 8 / gx));
    int P = pmax;
    for (int q = pmax; q >= 1; q--)
        if (nch % q == 0) {
            if (2 * q >= pmax) P = q;
            break;
        }
    dim3 grid(gx, P);
    if (vec == VM) launch_pdl(k_bias_part<T, VM>, grid, 256, 0, s, part, (const T*)dout, N, OC, nch);
    else launch_pdl(k_bias_part<T, 1>, grid, 256, 0, s, part, (const T*)dout, N, OC, nch);
    *nparts = P;
    return cudaGetLastError();
}
cudaError_t bias_grad_rows(int act, float* part, const void* dout, int N, int OC, int* nparts,
                           cudaStream_t s) {
    if (act == ACT_BF16) return bias_grad_rows_t<bf16>(part, dout, N, OC, nparts, s);
    return bias_grad_rows_t<float>(part, dout, N, OC, nparts, s);
}
cudaError_t bias_grad(int act, float* db, const void* dout, int N, int OC, void* scratch,
                      cudaStream_t s) {
    float* part = (float*)scratch;
    int P = 0;
    cudaError_t e = bias_grad_rows(act, part, dout, N, OC, &P, s);
    if (e != cudaSuccess) return e;
    ColsumOut o{{db, nullptr, nullptr}};
    launch_pdl(k_colsum, cdiv(OC, 32), 256, 0, s, o, OC, OC, part, P, OC);
    return cudaGetLastError();
}

// ===========================================================================
// Fused classifier loss.  One block per row: an online (max, sum-exp) pass over
// the V real columns, lse = max + log(sum); loss = lse - z[target]; then, when
// dloss != 0, the row is overwritten in place by (softmax - onehot) * dloss
// with the padded columns set to 0.  The probabilities are never stored.
// ===========================================================================
__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
    float M = fmaxf(m, m2);
    float a = (m == -INFINITY) ? 0.f : s * __expf(m - M);
    float b = (m2 == -INFINITY) ? 0.f : s2 * __expf(m2 - M);
    m = M;
    s = a + b;
}

template <typename T, int VEC>
__global__ void __launch_bounds__(512) k_xent(T* logits, float* losses, const int* tgt, int V,
                                              int Vp, float dloss, unsigned* err) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ float sm_m[32], sm_s[32];
    __shared__ float sh_lse;
    int row = blockIdx.x;
    T* z = logits + (size_t)row * Vp;
    int y = tgt[row];
    if (y < 0 || y >= V) {
        if (threadIdx.x == 0) atomicOr(err, GPT2_DEVERR_TOKEN);
        y = 0;
    }
    float zy = to_f(z[y]);
    float m = -INFINITY, s = 0.f;
    for (int j = threadIdx.x * VEC; j < V; j += blockDim.x * VEC) {
        float v[VEC];
        load_vec_f<T, VEC>(v, z + j);
#pragma unroll
        for (int e = 0; e < VEC; e++) {
            if (j + e < V) {
                float x = v[e];
                if (x > m) {
                    s = s * __expf(m - x) + 1.f;
                    m = x;
                } else {
                    s += __expf(x - m);
                }
            }
        }
    }
    // warp then block combine of (m, s) pairs
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_combine(m, s, m2, s2);
    }
    int warp = threadIdx.x / 32, lane = threadIdx.x & 31, nw = blockDim.x / 32;
    if (lane == 0) {
        sm_m[warp] = m;
        sm_s[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
        m = lane < nw ? sm_m[lane] : -INFINITY;
        s = lane < nw ? sm_s[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            ms_combine(m, s, m2, s2);
        }
        if (lane == 0) {
            float lse = m + logf(s);
            sh_lse = lse;
            losses[row] = lse - zy;
        }
    }
    __syncthreads();
    if (dloss == 0.f) return;
    float lse = sh_lse;
    for (int j = threadIdx.x * VEC; j < Vp; j += blockDim.x * VEC) {
        float v[VEC];
        load_vec_f<T, VEC>(v, z + j);
#pragma unroll
        for (int e = 0; e < VEC; e++) {
            int col = j + e;
            float p = __expf(v[e] - lse);
            v[e] = col < V ? (p - (col == y ? 1.f : 0.f)) * dloss : 0.f;
        }
        store_vec_f<T, VEC>(z + j, v);
    }
}

// ---------------------------------------------------------------------------
// bf16 rows staged whole in shared memory.  One persistent block per SM walks
// the rows blockIdx.x, blockIdx.x + gridDim.x, ...; while it works on one row,
// a bulk copy (cp.async.bulk, completion counted on an mbarrier) brings the
// next row into the other half of the double buffer, so each row is read from
// HBM once and the next read is always in flight.  Per row: max over the V
// real columns, sum of exp(z - max), lse = max + log(sum), loss, then the
// in-place write of (softmax - onehot) * dloss with the pad columns zeroed.
// ---------------------------------------------------------------------------
#define XS_THREADS 1024
// a packed bf16 pair reinterpreted (register to register)
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t x) {
    __nv_bfloat162 r;
    memcpy(&r, &x, sizeof r);
    return r;
}
#define XS_CHUNK 32768u  // bytes per bulk copy

__device__ __forceinline__ float ex2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// block-wide reduction (op 0 = max, 1 = sum) of one value per thread
__device__ __forceinline__ float block_reduce(float v, int op, float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = op ? warp_sum(v) : warp_max(v);
    __syncthreads();  // red[] may still be read by the previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[lane];  // blockDim.x == 1024: 32 warps
    return op ? warp_sum(v) : warp_max(v);
}

__global__ void __launch_bounds__(XS_THREADS, 1)
    k_xent_staged(bf16* logits, float* losses, const int* tgt, int N, int V, int Vp, float dloss,
                  unsigned* err) {
    gdc_wait();
    gdc_launch_dependents();
    extern __shared__ __align__(128) unsigned char xsm[];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ float red[32];
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const uint32_t rowb = (uint32_t)Vp * 2u;
    const uint32_t buf0 = tc::smem_u32(xsm);
    const uint32_t bar0 = tc::smem_u32(&bars[0]);
    auto issue = [&](int row, int b) {  // thread 0: bring `row` into half b
        const uint32_t bar = bar0 + 8u * b, dst = buf0 + rowb * b;
        const char* src = reinterpret_cast<const char*>(logits + (size_t)row * Vp);
        tc::mbar_expect_tx(bar, rowb);
        for (uint32_t o = 0; o < rowb; o += XS_CHUNK)
            bulk_g2s(dst + o, src + o, rowb - o < XS_CHUNK ? rowb - o : XS_CHUNK, bar);
    };
    if (tid == 0) {
        tc::mbar_init(bar0, 1);
        tc::mbar_init(bar0 + 8, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if ((int)blockIdx.x < N) issue(blockIdx.x, 0);
    }
    __syncthreads();
    int k = 0, row = blockIdx.x;
    for (; row < N; row += gridDim.x, k++) {
        const int b = k & 1;
        const int nrow = row + gridDim.x;
        if (tid == 0 && nrow < N) {
            // half b^1 was last read in the previous iteration, which ended
            // with a block barrier; order those reads before the async write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(nrow, b ^ 1);
        }
        tc::mbar_wait(bar0 + 8u * b, (uint32_t)(k >> 1) & 1u, &abort_flag, err);
        __syncthreads();
        if (abort_flag) break;
        const bf16* z = reinterpret_cast<const bf16*>(xsm + (size_t)rowb * b);
        int y = tgt[row];
        if (y < 0 || y >= V) {
            if (tid == 0) atomicOr(err, GPT2_DEVERR_TOKEN);
            y = 0;
        }
        // vectors of 8: [0, nfull) hold only real columns; the rest (the one
        // straddling V, then pure padding) take per-element checks
        const int nfull = V / 8, nvec = Vp / 8;
        const float L2E = 1.4426950408889634f;
        // pass 1: row max over the real columns (packed bf16 pairs)
        __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
        for (int j = tid; j < nfull; j += XS_THREADS) {
            const uint4 u = *reinterpret_cast<const uint4*>(z + 8 * j);
            m2 = __hmax2(m2, __hmax2(__hmax2(as_bf2(u.x), as_bf2(u.y)),
                                     __hmax2(as_bf2(u.z), as_bf2(u.w))));
        }
        float m = fmaxf(__low2float(m2), __high2float(m2));
        for (int c = 8 * nfull + tid; c < V; c += XS_THREADS) m = fmaxf(m, to_f(z[c]));
        m = block_reduce(m, 0, red);
        // pass 2: sum of exp(z - max)
        const float nm = -m * L2E;
        float sum = 0.f;
        for (int j = tid; j < nfull; j += XS_THREADS) {
            const uint4 u = *reinterpret_cast<const uint4*>(z + 8 * j);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 8; e++) sum += ex2f_approx(fmaf(bf_half(w4[e >> 1], e & 1), L2E, nm));
        }
        for (int c = 8 * nfull + tid; c < V; c += XS_THREADS)
            sum += ex2f_approx(fmaf(to_f(z[c]), L2E, nm));
        sum = block_reduce(sum, 1, red);
        const float lse = m + logf(sum);
        if (tid == 0) losses[row] = lse - to_f(z[y]);
        if (dloss != 0.f) {
            // pass 3: dlogits = softmax * dloss over the row, then the target
            // column minus dloss; written over the row in global memory
            bf16* zo = logits + (size_t)row * Vp;
            const float nl = -lse * L2E;
            for (int j = tid; j < nfull; j += XS_THREADS) {
                const uint4 u = *reinterpret_cast<const uint4*>(z + 8 * j);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; q++)
                    o[q] = pack2_bf16_rn(ex2f_approx(fmaf(bf_half(w4[q], 0), L2E, nl)) * dloss,
                                         ex2f_approx(fmaf(bf_half(w4[q], 1), L2E, nl)) * dloss);
                *reinterpret_cast<uint4*>(zo + 8 * j) = make_uint4(o[0], o[1], o[2], o[3]);
                if (y >> 3 == j)  // the target column: rewritten by the same thread
                    zo[y] = from_f<bf16>((ex2f_approx(fmaf(to_f(z[y]), L2E, nl)) - 1.f) * dloss);
            }
            for (int j = nfull + tid; j < nvec; j += XS_THREADS) {
                Vec<bf16, 8> v = *reinterpret_cast<const Vec<bf16, 8>*>(z + 8 * j);
                Vec<bf16, 8> o;
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int col = 8 * j + e;
                    const float pv = ex2f_approx(fmaf(to_f(v.v[e]), L2E, nl));
                    o.v[e] = from_f<bf16>(col < V ? (pv - (col == y ? 1.f : 0.f)) * dloss : 0.f);
                }
                *reinterpret_cast<Vec<bf16, 8>*>(zo + 8 * j) = o;
            }
        }
        __syncthreads();  // half b is free for the copy issued next iteration
    }
    if (abort_flag && tid == 0) {
        // a wait ran out in iteration k: let this block's copies still in
        // flight (row k's, and the prefetch of the next row if one was
        // issued) land, within the same bound, before its shared memory is
        // released
        volatile int own = 0;
        tc::mbar_wait(bar0 + 8u * (k & 1), (uint32_t)(k >> 1) & 1u, &own, nullptr);
        own = 0;
        if (row + (int)gridDim.x < N)
            tc::mbar_wait(bar0 + 8u * ((k + 1) & 1), (uint32_t)((k + 1) >> 1) & 1u, &own,
                          nullptr);
    }
}

cudaError_t crossentropy_fused(int act, void* logits, float* losses, const int* tgt, int N,
                               int V, int Vp, float dloss, unsigned* err, cudaStream_t s) {
    if (Vp % 8) return cudaErrorInvalidValue;
    if (act == ACT_BF16) {
        const size_t smem = (size_t)4 * Vp;  // two bf16 rows
        if (smem <= 200 * 1024 && ((uintptr_t)logits & 15) == 0) {
            static_assert(XS_THREADS == 1024, "block_reduce assumes 32 warps");
            int dev = 0, nsm = 148;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
            cudaError_t e = cudaFuncSetAttribute(
                k_xent_staged, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            const int grid = N < nsm ? N : nsm;
            launch_pdl(k_xent_staged, grid, XS_THREADS, smem, s, (bf16*)logits, losses, tgt, N, V, Vp,
                                                        dloss, err);
        } else {
            launch_pdl(k_xent<bf16, 8>, N, 512, 0, s, (bf16*)logits, losses, tgt, V, Vp, dloss, err);
        }
    } else {
        launch_pdl(k_xent<float, 4>, N, 512, 0, s, (float*)logits, losses, tgt, V, Vp, dloss, err);
    }
    return cudaGetLastError();
}

__global__ void k_mean(float* out, const float* x, int n) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ double sh[32];
    double a = 0.0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) a += (double)x[i];
    a = warp_sum_d(a);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x / 32] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        a = threadIdx.x < blockDim.x / 32 ? sh[threadIdx.x] : 0.0;
        a = warp_sum_d(a);
        if (threadIdx.x == 0) out[0] = (float)(a / n);
    }
}
cudaError_t mean_reduce(float* out, const float* x, int n, cudaStream_t s) {
    launch_pdl(k_mean, 1, 1024, 0, s, out, x, n);
    return cudaGetLastError();
}

// ===========================================================================
// Embedding backward without float atomics.
//  1. k_emb_rank: each 1024-position block sorts its (token, position) keys in
//     shared memory (bitonic), giving each position its rank among equal
//     tokens of the block and the block's count per token.
//  2. k_emb_blockprefix: per token, exclusive prefix of the block counts.
//  3. k_emb_scan: exclusive scans of the per-token totals -> bucket starts,
//     and of the chunk counts (buckets split in chunks of EMB_R rows); the
//     list of tokens with more than one chunk.
//  4. k_emb_place: stable placement -> positions sorted by (token, position).
//  5. k_emb_items: list the (token, chunk) work items.
//  6. k_emb_reduce: one warp per item sums its <= EMB_R rows in position
//     order; single-chunk tokens add into dwte directly, the others write a
//     partial row; k_emb_fold adds those partials to dwte in chunk order.
//  7. k_wpe_bwd: dwpe[t] += sum over b (in order).
// ===========================================================================
#define EMB_BLK 1024
#define EMB_R 32

struct EmbScratch {
    int* blkcnt;   // [nb][Vp]
    int* cnt;      // [Vp]
    int* start;    // [Vp+1]
    int* itemoff;  // [Vp+1]
    int* poff;     // [Vp+1]
    int* lrank;    // [BT]
    int* sorted;   // [BT]
    int2* items;   // [max_items]
    float* part;   // [max_part][C]
    int* mlist;    // [1 + max_multi]: the count of tokens with more than one chunk, then they
    int nb, max_items, max_part, max_multi;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static EmbScratch emb_carve(void* base, int BT, int C, int Vp, size_t* total) {
    EmbScratch e;
    e.nb = cdiv(BT, EMB_BLK);
    e.max_items = cdiv(BT, EMB_R) + (BT < Vp ? BT : Vp);
    e.max_part = 2 * cdiv(BT, EMB_R) + 1;
    e.max_multi = cdiv(BT, EMB_R + 1);  // a multi-chunk token holds > EMB_R positions
    char* p = (char*)base;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        char* r = p ? p + o : nullptr;
        o += align256(bytes);
        return r;
    };
    e.blkcnt = (int*)take((size_t)e.nb * Vp * 4);
    e.cnt = (int*)take((size_t)Vp * 4);
    e.start = (int*)take((size_t)(Vp + 1) * 4);
    e.itemoff = (int*)take((size_t)(Vp + 1) * 4);
    e.poff = (int*)take((size_t)(Vp + 1) * 4);
    e.lrank = (int*)take((size_t)BT * 4);
    e.sorted = (int*)take((size_t)BT * 4);
    e.items = (int2*)take((size_t)e.max_items * 8);
    e.part = (float*)take((size_t)e.max_part * C * 4);
    e.mlist = (int*)take((size_t)(e.max_multi + 1) * 4);
    if (total) *total = o;
    return e;
}

size_t encoder_backward_scratch(int B, int T_, int C, int Vp) {
    size_t t;
    emb_carve(nullptr, B * T_, C, Vp, &t);
    return t;
}

__global__ void __launch_bounds__(EMB_BLK) k_emb_rank(const int* tok, int BT, int Vp, int* lrank,
                                                      int* blkcnt) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ unsigned key[EMB_BLK];
    __shared__ int rs[EMB_BLK];
    int i = threadIdx.x, pos = blockIdx.x * EMB_BLK + i;
    unsigned k = 0xffffffffu;
    if (pos < BT) {
        int t = tok[pos];
        if (t < 0 || t >= Vp) t = 0;
        k = ((unsigned)t << 11) | (unsigned)i;
    }
    key[i] = k;
    __syncthreads();
    // bitonic sort, ascending
    for (int size = 2; size <= EMB_BLK; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            int j = i ^ stride;
            if (j > i) {
                unsigned a = key[i], b = key[j];
                bool up = (i & size) == 0;
                if ((a > b) == up) {
                    key[i] = b;
                    key[j] = a;
                }
            }
            __syncthreads();
        }
    }
    unsigned ki = key[i];
    bool valid = ki != 0xffffffffu;
    unsigned ti = ki >> 11;
    bool head = valid && (i == 0 || (key[i - 1] >> 11) != ti);
    rs[i] = head ? i : 0;
    __syncthreads();
    // inclusive max-scan: start index of each run
    for (int off = 1; off < EMB_BLK; off <<= 1) {
        int v = rs[i];
        if (i >= off) v = max(v, rs[i - off]);
        __syncthreads();
        rs[i] = v;
        __syncthreads();
    }
    if (valid) {
        int st = rs[i];
        int li = (int)(ki & 2047u);
        lrank[blockIdx.x * EMB_BLK + li] = i - st;
        bool tail = (i == EMB_BLK - 1) || (key[i + 1] >> 11) != ti;
        if (tail) blkcnt[(size_t)blockIdx.x * Vp + ti] = i - st + 1;
    }
}

__global__ void k_emb_blockprefix(int* blkcnt, int* cnt, int nb, int Vp) {
    gdc_wait();
    gdc_launch_dependents();
    int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= Vp) return;
    int run = 0;
    // 16 block counts at a time: independent loads in flight together, then
    // the prefix over them in block order
    for (int b0 = 0; b0 < nb; b0 += 16) {
        int c[16];
#pragma unroll
        for (int k = 0; k < 16; k++) c[k] = b0 + k < nb ? blkcnt[(size_t)(b0 + k) * Vp + v] : 0;
#pragma unroll
        for (int k = 0; k < 16; k++) {
            if (b0 + k < nb) blkcnt[(size_t)(b0 + k) * Vp + v] = run;
            run += c[k];
        }
    }
    cnt[v] = run;
}

// Exclusive scans over v in [0, Vp) of n_v (bucket starts), chunks_v (work
// item offsets), chunks_v of the multi-chunk tokens (partial-row offsets) and
// [chunks_v > 1] (their place in mlist).  Block b scans v in [1024 b, 1024 b +
// 1024) after summing every count below its range itself (at most Vp ints,
// read as int4 from L2), so the blocks need no communication and the result
// does not depend on their order.  Vp is a multiple of 4.
__global__ void __launch_bounds__(1024) k_emb_scan(const int* cnt, int* start, int* itemoff,
                                                   int* poff, int* mlist, int Vp) {
    gdc_wait();
    gdc_launch_dependents();
    constexpr int Q = 4;
    __shared__ int wpre[Q][32], wloc[Q][32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int base = blockIdx.x * 1024;
    auto terms = [](int n, int* q) {
        const int ch = (n + EMB_R - 1) / EMB_R;
        q[0] = n;
        q[1] = ch;
        q[2] = ch > 1 ? ch : 0;
        q[3] = ch > 1 ? 1 : 0;
    };
    // 1. this thread's share of the sums below `base` (v, v+1, v+2, v+3 < base
    //    whenever v < base: both are multiples of 4)
    int pre[Q] = {0, 0, 0, 0};
    for (int v0 = 0; v0 < base; v0 += 4 * 4096) {
        int4 c[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int v = v0 + 4096 * k + 4 * t;
            c[k] = v < base ? *reinterpret_cast<const int4*>(cnt + v) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int n4[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                int q[Q];
                terms(n4[j], q);
#pragma unroll
                for (int i = 0; i < Q; i++) pre[i] += q[i];
            }
        }
    }
    // 2. this block's own range: one token per thread
    const int v = base + t;
    int own[Q];
    terms(v < Vp ? cnt[v] : 0, own);
    int inc[Q];
#pragma unroll
    for (int i = 0; i < Q; i++) inc[i] = own[i];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int i = 0; i < Q; i++) {
            const int y = __shfl_up_sync(0xffffffffu, inc[i], off);
            if (lane >= off) inc[i] += y;
            pre[i] += __shfl_xor_sync(0xffffffffu, pre[i], off);
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < Q; i++) {
            wloc[i][warp] = inc[i];
            wpre[i][warp] = pre[i];
        }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < Q; i++) {
            int x = wloc[i][lane], y = wpre[i][lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += u;
                y += __shfl_xor_sync(0xffffffffu, y, off);
            }
            wloc[i][lane] = x;  // inclusive over the warps
            wpre[i][lane] = y;  // every lane: the block's total below `base`
        }
    }
    __syncthreads();
    int ex[Q];
#pragma unroll
    for (int i = 0; i < Q; i++) ex[i] = wpre[i][0] + (warp ? wloc[i][warp - 1] : 0) + inc[i] - own[i];
    if (v < Vp) {
        start[v] = ex[0];
        itemoff[v] = ex[1];
        poff[v] = ex[2];
        if (own[3]) mlist[1 + ex[3]] = v;
    }
    if (base + 1024 >= Vp && t == 0) {
        start[Vp] = wpre[0][0] + wloc[0][31];
        itemoff[Vp] = wpre[1][0] + wloc[1][31];
        poff[Vp] = wpre[2][0] + wloc[2][31];
        mlist[0] = wpre[3][0] + wloc[3][31];
    }
}

__global__ void k_emb_place(const int* tok, int BT, int Vp, const int* start, const int* blkcnt,
                            const int* lrank, int* sorted) {
    gdc_wait();
    gdc_launch_dependents();
    int pos = blockIdx.x * blockDim.x + threadIdx.x;
    if (pos >= BT) return;
    int t = tok[pos];
    if (t < 0 || t >= Vp) t = 0;
    int b = pos / EMB_BLK;
    sorted[start[t] + blkcnt[(size_t)b * Vp + t] + lrank[pos]] = pos;
}

__global__ void k_emb_items(const int* cnt, const int* itemoff, int2* items, int Vp) {
    gdc_wait();
    gdc_launch_dependents();
    int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= Vp) return;
    int n = cnt[v];
    int ch = (n + EMB_R - 1) / EMB_R, o = itemoff[v];
    for (int c = 0; c < ch; c++) items[o + c] = make_int2(v, c);
}

template <typename T, int VEC, int IT>
__global__ void k_emb_reduce2(float* dwte, float* part, const T* dx, const int* sorted,
                              const int* cnt, const int* start, const int* n_items,
                              const int* poff, const int2* items, int C) {
    gdc_wait();
    gdc_launch_dependents();
    int item = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x & 31;
    if (item >= *n_items) return;
    int2 vc = items[item];
    int v = vc.x, c = vc.y;
    int n = cnt[v];
    int r0 = c * EMB_R, r1 = min(n, r0 + EMB_R);
    float acc[IT][VEC];
#pragma unroll
    for (int it = 0; it < IT; it++)
#pragma unroll
        for (int j = 0; j < VEC; j++) acc[it][j] = 0.f;
    const int* rows = sorted + start[v];
    for (int r = r0; r < r1; r++) {
        const T* src = dx + (size_t)rows[r] * C;
#pragma unroll
        for (int it = 0; it < IT; it++) {
            int col = (it * 32 + lane) * VEC;
            if (col < C) {
                float x[VEC];
                load_vec_f<T, VEC>(x, src + col);
#pragma unroll
                for (int j = 0; j < VEC; j++) acc[it][j] += x[j];
            }
        }
    }
    bool single = n <= EMB_R;
    float* dst = single ? dwte + (size_t)v * C : part + (size_t)(poff[v] + c) * C;
#pragma unroll
    for (int it = 0; it < IT; it++) {
        int col = (it * 32 + lane) * VEC;
        if (col < C) {
#pragma unroll
            for (int j = 0; j < VEC; j++) {
                if (single) dst[col + j] += acc[it][j];
                else dst[col + j] = acc[it][j];
            }
        }
    }
}

// block (x, y): multi-chunk token x, columns [256 y, 256 y + 256): dwte[v] +=
// its partial rows added in chunk order (eight loads in flight at a time)
__global__ void k_emb_fold(float* dwte, const float* part, const int* cnt, const int* poff,
                           const int* mlist, int C) {
    gdc_wait();
    gdc_launch_dependents();
    if ((int)blockIdx.x >= mlist[0]) return;
    const int v = mlist[1 + blockIdx.x], n = cnt[v];
    const int ch = (n + EMB_R - 1) / EMB_R;
    const float* p = part + (size_t)poff[v] * C;
    const int col = blockIdx.y * 256 + threadIdx.x;
    if (col >= C) return;
    float a = 0.f;
    for (int k0 = 0; k0 < ch; k0 += 8) {
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; k++) x[k] = k0 + k < ch ? p[(size_t)(k0 + k) * C + col] : 0.f;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (k0 + k < ch) a += x[k];
    }
    dwte[(size_t)v * C + col] += a;
}

template <typename T, int VEC>
__global__ void k_wpe_bwd(float* dwpe, const T* dx, int B, int T_, int C) {
    gdc_wait();
    gdc_launch_dependents();
    long idx = blockIdx.x * (long)blockDim.x + threadIdx.x;
    int cv = C / VEC;
    if (idx >= (long)T_ * cv) return;
    int t = (int)(idx / cv), c = (int)(idx % cv) * VEC;
    float a[VEC];
#pragma unroll
    for (int j = 0; j < VEC; j++) a[j] = 0.f;
    for (int b = 0; b < B; b++) {
        float x[VEC];
        load_vec_f<T, VEC>(x, dx + ((size_t)b * T_ + t) * C + c);
#pragma unroll
        for (int j = 0; j < VEC; j++) a[j] += x[j];
    }
#pragma unroll
    for (int j = 0; j < VEC; j++) dwpe[(size_t)t * C + c + j] += a[j];
}

template <typename T, int VEC>
static cudaError_t emb_bwd_vec(float* dwte, float* dwpe, const void* dx, const int* tok, int B,
                               int T_, int C, int Vp, void* scratch, cudaStream_t s) {
    int BT = B * T_;
    EmbScratch e = emb_carve(scratch, BT, C, Vp, nullptr);
    cudaMemsetAsync(e.blkcnt, 0, (size_t)e.nb * Vp * 4, s);
    launch_pdl(k_emb_rank, e.nb, EMB_BLK, 0, s, tok, BT, Vp, e.lrank, e.blkcnt);
    launch_pdl(k_emb_blockprefix, cdiv(Vp, 256), 256, 0, s, e.blkcnt, e.cnt, e.nb, Vp);
    if (Vp % 4) return cudaErrorInvalidValue;
    launch_pdl(k_emb_scan, cdiv(Vp, 1024), 1024, 0, s, e.cnt, e.start, e.itemoff, e.poff, e.mlist,
               Vp);
    launch_pdl(k_emb_place, cdiv(BT, 256), 256, 0, s, tok, BT, Vp, e.start, e.blkcnt, e.lrank, e.sorted);
    launch_pdl(k_emb_items, cdiv(Vp, 256), 256, 0, s, e.cnt, e.itemoff, e.items, Vp);
    int it = cdiv(C, 32 * VEC);
    const int* n_items = e.itemoff + Vp;
    dim3 g(cdiv(e.max_items, 8));
#define EMR(I)                                                                                   \
    launch_pdl(k_emb_reduce2<T, VEC, I>, g, 256, 0, s, dwte, e.part, (const T*)dx, e.sorted, e.cnt,      \
                                               e.start, n_items, e.poff, e.items, C)
    if (it <= 1) EMR(1);
    else if (it <= 2) EMR(2);
    else if (it <= 4) EMR(4);
    else if (it <= 8) EMR(8);
    else if (it <= 16) EMR(16);
    else return cudaErrorInvalidValue;
#undef EMR
    launch_pdl(k_emb_fold, dim3(e.max_multi, cdiv(C, 256)), 256, 0, s, dwte, e.part, e.cnt, e.poff,
               e.mlist, C);
    launch_pdl(k_wpe_bwd<T, VEC>, cdiv((long)T_ * (C / VEC), 256), 256, 0, s, dwpe, (const T*)dx, B, T_,
                                                                       C);
    return cudaGetLastError();
}
template <typename T>
static cudaError_t emb_bwd_t(float* dwte, float* dwpe, const void* dx, const int* tok, int B,
                             int T_, int C, int Vp, void* scratch, cudaStream_t s) {
    constexpr int VM = 16 / sizeof(T);
    if (C % VM == 0) return emb_bwd_vec<T, VM>(dwte, dwpe, dx, tok, B, T_, C, Vp, scratch, s);
    return emb_bwd_vec<T, 1>(dwte, dwpe, dx, tok, B, T_, C, Vp, scratch, s);
}
cudaError_t encoder_backward(int act, float* dwte, float* dwpe, const void* dx, const int* tok,
                             int B, int T_, int C, int Vp, void* scratch, cudaStream_t s) {
    if (Vp >= (1 << 21)) return cudaErrorInvalidValue;
    if (act == ACT_BF16) return emb_bwd_t<bf16>(dwte, dwpe, dx, tok, B, T_, C, Vp, scratch, s);
    return emb_bwd_t<float>(dwte, dwpe, dx, tok, B, T_, C, Vp, scratch, s);
}

// ===========================================================================
// AdamW with global-norm clipping ("update_params" in one pass over the
// parameters after a norm pass).
//  k_sumsq:     fixed grid; block b sums squares of its contiguous range.
//  k_adam_norm: one block folds the block partials in order (fp64),
//               n = sqrt(S)/n_accum, scale = (1/n_accum) * min(1, clip/n).
//  k_adam:      per element update; skipped entirely if n is not finite.
// ===========================================================================
#define ADAM_NB 1184

__global__ void __launch_bounds__(256) k_sumsq(const float* g, size_t n, double* part) {
    gdc_wait();
    gdc_launch_dependents();
    __shared__ double sh[8];
    size_t chunk = ((n + ADAM_NB - 1) / ADAM_NB + 3) & ~(size_t)3;
    size_t lo = (size_t)blockIdx.x * chunk, hi = lo + chunk < n ? lo + chunk : n;
    float a = 0.f;
    if (lo < hi) {
        size_t nv = (hi - lo) / 4;
        const float4* g4 = reinterpret_cast<const float4*>(g + lo);
        for (size_t i = threadIdx.x; i < nv; i += blockDim.x) {
            float4 x = g4[i];
            a += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
        }
        for (size_t i = lo + nv * 4 + threadIdx.x; i < hi; i += blockDim.x) a += g[i] * g[i];
    }
    double d = warp_sum_d((double)a);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x / 32] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < 8; w++) t += sh[w];
        part[blockIdx.x] = t;
    }
}

__global__ void k_adam_norm(const double* part, float* state, float inv_accum, float clip,
                            const int* d_count) {
    gdc_wait();
    gdc_launch_dependents();
    // the same correctly rounded quotient the host forms from its own count
    if (d_count) inv_accum = __fdiv_rn(1.0f, (float)*d_count);
    __shared__ double sh[32];
    double a = 0.0;
    for (int i = threadIdx.x; i < ADAM_NB; i += blockDim.x) a += part[i];
    a = warp_sum_d(a);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x / 32] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < (int)(blockDim.x / 32); w++) t += sh[w];
        float norm = (float)(sqrt(t) * (double)inv_accum);
        int finite = isfinite(norm) ? 1 : 0;
        float sc = inv_accum;
        if (finite && clip > 0.f && norm > clip) sc = inv_accum * (clip / norm);
        state[0] = norm;
        state[1] = sc;
        state[2] = (float)finite;
    }
}

// element i of the launch is canonical element a.base + i
__device__ __forceinline__ bool decayed(size_t i, const AdamArgs& a) {
    i += a.base;
#pragma unroll
    for (int k = 0; k < 5; k++)
        if (i >= a.dec_lo[k] && i < a.dec_hi[k]) return true;
    return false;
}

__device__ __forceinline__ float adam_one(float& w, float& m, float& v, float g, float sc,
                                          const AdamArgs& a, bool dec) {
    float gi = g * sc;
    m = a.b1 * m + (1.f - a.b1) * gi;
    v = a.b2 * v + (1.f - a.b2) * gi * gi;
    float mh = m / a.bc1, vh = v / a.bc2;
    w = w - a.lr * (mh / (sqrtf(vh) + a.eps) + (dec ? a.wd * w : 0.f));
    return w;
}

__global__ void __launch_bounds__(256) k_adam(float* w, float* m, float* v, const float* g,
                                              bf16* wb, size_t n, AdamArgs a,
                                              const float* state) {
    gdc_wait();
    gdc_launch_dependents();
    if (state[2] == 0.f) return;
    float sc = state[1];
    size_t nv = n / 4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nv;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 W = reinterpret_cast<float4*>(w)[i];
        float4 M = reinterpret_cast<float4*>(m)[i];
        float4 Vv = reinterpret_cast<float4*>(v)[i];
        float4 G = reinterpret_cast<const float4*>(g)[i];
        size_t e = i * 4;
        adam_one(W.x, M.x, Vv.x, G.x, sc, a, decayed(e, a));
        adam_one(W.y, M.y, Vv.y, G.y, sc, a, decayed(e + 1, a));
        adam_one(W.z, M.z, Vv.z, G.z, sc, a, decayed(e + 2, a));
        adam_one(W.w, M.w, Vv.w, G.w, sc, a, decayed(e + 3, a));
        reinterpret_cast<float4*>(w)[i] = W;
        reinterpret_cast<float4*>(m)[i] = M;
        reinterpret_cast<float4*>(v)[i] = Vv;
        if (wb) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(W.x, W.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(W.z, W.w);
            uint2 pk;
            pk.x = *reinterpret_cast<unsigned*>(&lo);
            pk.y = *reinterpret_cast<unsigned*>(&hi);
            reinterpret_cast<uint2*>(wb)[i] = pk;
        }
    }
    for (size_t e = nv * 4 + blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
         e += (size_t)gridDim.x * blockDim.x) {
        float W = w[e], M = m[e], Vv = v[e];
        adam_one(W, M, Vv, g[e], sc, a, decayed(e, a));
        w[e] = W;
        m[e] = M;
        v[e] = Vv;
        if (wb) wb[e] = __float2bfloat16_rn(W);
    }
}

// AdamW for parameters held only in bf16: the update in fp32 from the widened
// bf16 value, then stochastic rounding back to bf16 with counter (t-1)*n + i
// of the stream a.sr_seed (t = this update's step count).
__global__ void __launch_bounds__(256) k_adam_bf16_sr(bf16* wb, float* m, float* v,
                                                      const float* g, size_t n, AdamArgs a,
                                                      const float* state) {
    gdc_wait();
    gdc_launch_dependents();
    if (state[2] == 0.f) return;
    const float sc = state[1];
    const uint64_t k0 = (uint64_t)(a.t - 1) * (uint64_t)a.n_total + a.base;
    uint16_t* wu = reinterpret_cast<uint16_t*>(wb);
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
         e += (size_t)gridDim.x * blockDim.x) {
        float W = __uint_as_float((uint32_t)wu[e] << 16), M = m[e], Vv = v[e];
        adam_one(W, M, Vv, g[e], sc, a, decayed(e, a));
        m[e] = M;
        v[e] = Vv;
        wu[e] = sround_bf16(W, sm64_at(a.sr_seed, k0 + e));
    }
}
cudaError_t adamw_update_bf16_sr(void* wbf16, float* m, float* v, const float* g, size_t n,
                                 const AdamArgs& a, const float* state, cudaStream_t s) {
    launch_pdl(k_adam_bf16_sr, 148 * 8, 256, 0, s, (bf16*)wbf16, m, v, g, n, a, state);
    return cudaGetLastError();
}

size_t adamw_scratch() { return ADAM_NB * sizeof(double); }

// ---------------------------------------------------------------------------
// AdamW with the global norm and clip in one launch ("update_params" of
// "Karpathy's llm.c ...", "Performance comparison": one kernel for the whole
// parameter update).  A cooperative launch (every block resident at once):
//   1. the blocks compute the square sums of the ADAM_NB chunks that k_sumsq
//      would (virtual block b = blockIdx.x, blockIdx.x + gridDim.x, ...), in
//      the same order, into part[];
//   2. a grid barrier (a counter and a generation word in device memory; each
//      waiting thread spins a bounded number of clock cycles, then sets
//      GPT2_DEVERR_TIMEOUT and the flag that skips the update);
//   3. every block folds part[] exactly as k_adam_norm does (1024 virtual
//      threads, butterfly warp sums, warps in order), so every block holds the
//      same norm and scale, bit for bit the three-kernel result; block 0
//      writes state[];
//   4. the update of [0, n_upd) as k_adam / k_adam_bf16_sr (element-wise).
// ---------------------------------------------------------------------------
constexpr long long ADAM_BAR_LIMIT = 4000000000LL;  // ~2 s of SM clock

__device__ bool adam_grid_barrier(unsigned* bar, unsigned nblocks, unsigned* err) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned* gen = bar + 1;
        const unsigned g0 = *gen;
        __threadfence();
        const unsigned arrived = atomicAdd(bar, 1u) + 1u;
        int ok = 1;
        if (arrived == nblocks) {
            bar[0] = 0u;  // reset for the next barrier, before releasing the others
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const long long t0 = clock64();
            while (*gen == g0) {
                if (clock64() - t0 > ADAM_BAR_LIMIT) {
                    ok = 0;
                    if (err) atomicOr(err, GPT2_DEVERR_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

template <bool SR>
__global__ void __launch_bounds__(256) k_adam_fused(float* w, float* m, float* v, const float* g,
                                                    void* wb, size_t n_total, size_t lo,
                                                    size_t n_upd, AdamArgs a, float* state,
                                                    double* part, unsigned* bar, unsigned* err) {
    __shared__ double sh[32];
    __shared__ float sc_s;
    __shared__ int fin_s;
    // 1. square sums of the ADAM_NB chunks of the whole gradient
    const size_t chunk = ((n_total + ADAM_NB - 1) / ADAM_NB + 3) & ~(size_t)3;
    for (int vb = blockIdx.x; vb < ADAM_NB; vb += gridDim.x) {
        const size_t b0 = (size_t)vb * chunk, b1 = b0 + chunk < n_total ? b0 + chunk : n_total;
        float acc = 0.f;
        if (b0 < b1) {
            const size_t nv = (b1 - b0) / 4;
            const float4* g4 = reinterpret_cast<const float4*>(g + b0);
            for (size_t i = threadIdx.x; i < nv; i += blockDim.x) {
                const float4 x = g4[i];
                acc += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
            }
            for (size_t i = b0 + nv * 4 + threadIdx.x; i < b1; i += blockDim.x) acc += g[i] * g[i];
        }
        const double d = warp_sum_d((double)acc);
        if ((threadIdx.x & 31) == 0) sh[threadIdx.x / 32] = d;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int k = 0; k < 8; k++) t += sh[k];
            part[vb] = t;
        }
        __syncthreads();
    }
    // 2. every partial written
    const bool ok = adam_grid_barrier(bar, gridDim.x, err);
    // 3. the fold of k_adam_norm, 1024 virtual threads over 256
    for (int k = 0; k < 4; k++) {
        const int vt = threadIdx.x + 256 * k;
        double x = 0.0;
        for (int i = vt; i < ADAM_NB; i += 1024) x += __ldcg(part + i);  // L2: other blocks' writes
        x = warp_sum_d(x);
        if ((threadIdx.x & 31) == 0) sh[vt / 32] = x;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int k = 0; k < 32; k++) t += sh[k];
        float inv = a.d_count ? __fdiv_rn(1.0f, (float)*a.d_count) : a.inv_accum;
        const float norm = (float)(sqrt(t) * (double)inv);
        const int finite = isfinite(norm) ? 1 : 0;
        float sc = inv;
        if (finite && a.clip > 0.f && norm > a.clip) sc = inv * (a.clip / norm);
        sc_s = sc;
        fin_s = finite && ok;
        if (blockIdx.x == 0) {
            state[0] = norm;
            state[1] = sc;
            state[2] = (float)finite;
        }
    }
    __syncthreads();
    if (!fin_s) return;
    const float sc = sc_s;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    if (!SR) {
        // 4. the update of [lo, lo + n_upd): w, m, v at their offsets, the
        // bf16 copy (if any) refreshed
        float* W = w;
        const float* G = g + lo;
        bf16* WB = reinterpret_cast<bf16*>(wb);
        const size_t nv = n_upd / 4;
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nv; i += stride) {
            float4 X = reinterpret_cast<float4*>(W)[i];
            float4 M = reinterpret_cast<float4*>(m)[i];
            float4 Vv = reinterpret_cast<float4*>(v)[i];
            const float4 Gr = reinterpret_cast<const float4*>(G)[i];
            const size_t e = i * 4;
            adam_one(X.x, M.x, Vv.x, Gr.x, sc, a, decayed(e, a));
            adam_one(X.y, M.y, Vv.y, Gr.y, sc, a, decayed(e + 1, a));
            adam_one(X.z, M.z, Vv.z, Gr.z, sc, a, decayed(e + 2, a));
            adam_one(X.w, M.w, Vv.w, Gr.w, sc, a, decayed(e + 3, a));
            reinterpret_cast<float4*>(W)[i] = X;
            reinterpret_cast<float4*>(m)[i] = M;
            reinterpret_cast<float4*>(v)[i] = Vv;
            if (WB) {
                __nv_bfloat162 l2 = __floats2bfloat162_rn(X.x, X.y);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(X.z, X.w);
                uint2 pk;
                pk.x = *reinterpret_cast<unsigned*>(&l2);
                pk.y = *reinterpret_cast<unsigned*>(&h2);
                reinterpret_cast<uint2*>(WB)[i] = pk;
            }
        }
        for (size_t e = nv * 4 + blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n_upd;
             e += stride) {
            float X = W[e], M = m[e], Vv = v[e];
            adam_one(X, M, Vv, G[e], sc, a, decayed(e, a));
            W[e] = X;
            m[e] = M;
            v[e] = Vv;
            if (WB) WB[e] = __float2bfloat16_rn(X);
        }
    } else {
        const uint64_t k0 = (uint64_t)(a.t - 1) * (uint64_t)a.n_total + a.base;
        uint16_t* wu = reinterpret_cast<uint16_t*>(wb);
        const float* G = g + lo;
        for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n_upd; e += stride) {
            float X = __uint_as_float((uint32_t)wu[e] << 16), M = m[e], Vv = v[e];
            adam_one(X, M, Vv, G[e], sc, a, decayed(e, a));
            m[e] = M;
            v[e] = Vv;
            wu[e] = sround_bf16(X, sm64_at(a.sr_seed, k0 + e));
        }
    }
}

size_t adamw_fused_scratch() { return ADAM_NB * sizeof(double) + 256; }

template <bool SR>
static int fused_grid() {
    static int grid = 0;
    if (grid == 0) {
        int dev = 0, nsm = 148, per = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_adam_fused<SR>, 256, 0) !=
                cudaSuccess ||
            per < 1) {
            cudaGetLastError();
            per = 1;
        }
        grid = nsm * (per < 8 ? per : 8);
    }
    return grid;
}

cudaError_t adamw_fused(float* w, float* m, float* v, const float* g, void* wbf16,
                        size_t n_total, size_t lo, size_t n_upd, bool sr, const AdamArgs& a,
                        float* state, void* scratch, unsigned* bar, unsigned* err,
                        cudaStream_t s) {
    double* part = (double*)scratch;
    const int grid = sr ? fused_grid<true>() : fused_grid<false>();
    void* args[] = {&w, &m, &v, (void*)&g, &wbf16, &n_total, &lo, &n_upd, (void*)&a, &state,
                    &part, &bar, &err};
    return cudaLaunchCooperativeKernel(
        sr ? (const void*)k_adam_fused<true> : (const void*)k_adam_fused<false>, dim3(grid),
        dim3(256), args, 0, s);
}

cudaError_t adamw_norm(const float* g, size_t n, const AdamArgs& a, float* state, void* scratch,
                       cudaStream_t s) {
    double* part = (double*)scratch;
    launch_pdl(k_sumsq, ADAM_NB, 256, 0, s, g, n, part);
    launch_pdl(k_adam_norm, 1, 1024, 0, s, part, state, a.inv_accum, a.clip, a.d_count);
    return cudaGetLastError();
}
cudaError_t adamw_update(float* w, float* m, float* v, const float* g, void* wbf16, size_t n,
                         const AdamArgs& a, const float* state, cudaStream_t s) {
    launch_pdl(k_adam, 148 * 8, 256, 0, s, w, m, v, g, (bf16*)wbf16, n, a, state);
    return cudaGetLastError();
}
cudaError_t adamw_step(float* w, float* m, float* v, const float* g, void* wbf16, size_t n,
                       const AdamArgs& a, float* state, void* scratch, cudaStream_t s) {
    cudaError_t e = adamw_norm(g, n, a, state, scratch, s);
    if (e != cudaSuccess) return e;
    return adamw_update(w, m, v, g, wbf16, n, a, state, s);
}

// acc[0] += x[0] (the running sum of the micro-batch losses of a step)
__global__ void k_accum1(float* acc, const float* x) {
    gdc_wait();
    gdc_launch_dependents();
    if (threadIdx.x == 0) acc[0] += x[0];
}
cudaError_t accumulate_scalar(float* acc, const float* x, cudaStream_t s) {
    launch_pdl(k_accum1, 1, 32, 0, s, acc, x);
    return cudaGetLastError();
}

}  // namespace gk
