// k_attn_tc.cu -- causal multi-head attention on the sm_103a tensor cores
// (tcgen05.mma with accumulators in tensor memory, TMA tile loads), head size 64.
//
// Definition ("Getting started with LLMs from Andrej Karpathy's talk",
// self-attention section): O = softmax(Q K^T / sqrt(d_k)) V per head, causal
// (query t sees keys 0..t; later keys are left out of the softmax).  The
// pages run attention as cuDNN FlashAttention or as two llm.c kernels
// ("Karpathy's llm.c: understanding LLM training from scratch in C/CUDA",
// "Code anatomy" item 2 and "Performance comparison"); here it is one fused
// kernel per direction, written for tcgen05.
//
// Forward (one CTA per 128-query tile of one (batch, head); 320 threads):
//   warp 0, lane 0  TMA: the Q tile once, then K_j, V_j tiles (128 keys x 64)
//                   through a ring of five shared-memory slots
//   warp 1, lane 0  tcgen05.mma issue, TMEM (256 columns):
//                     S_j = Q K_j^T   M=128 N=128 K=64   -> fp32 cols [0,128)
//                     O  += P_j V_j   M=128 N=64  K=128  -> fp32 cols [128,192)
//                   with P_j (bf16, two per column) read from cols [192,256);
//                   S_{j+1} is issued as soon as the softmax warps hold S_j
//   warps 2-9       two warps per TMEM lane quarter, each one half of the
//                   keys of 32 rows: tcgen05.ld of S_j, row max (exchanged
//                   between the halves), P_j = exp2(S_j c - m) in base 2,
//                   tcgen05.st of P_j; the running max m is raised (and O, the
//                   row sum rescaled in TMEM) only when a row max exceeds it
//                   by more than 2^8.
// Keys are visited in tiles 0..q (q = the query tile); only the diagonal tile
// needs the causal mask.  The TMA producer and the MMA issuer sit in warps of
// their own: a thread issuing tcgen05.mma back to back is held for about a
// hundred cycles per instruction, and sharing a warp with the producer's
// waits costs a few percent more.  Two CTAs share an SM (~100 KB smem, 256 TMEM
// columns and 96 registers a thread each), so one CTA's softmax overlaps the
// other's products.
// Outputs: O [B,T,C] (bf16) and the row log-sum-exp [B,H,T] (fp32, natural
// log), which the backward pass uses to recompute P.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace gk {

namespace {

using namespace tc;

constexpr int HD = 64;
constexpr int TILE = 128;               // queries per CTA = keys per tile
constexpr int TILE_BYTES = TILE * 128;  // 128 rows of 64 bf16
// forward smem: Q, a ring of F_NRING K/V slots (K_0 V_0 K_1 V_1 ... in order),
// then the row-max exchange, the final row-sum exchange and the barriers (P
// lives in TMEM)
constexpr int F_NRING = 5;
constexpr int F_Q = 0, F_RING = 16384, F_RED = F_RING + F_NRING * 16384, F_LS = F_RED + 2048,
              F_BAR = F_LS + 1024;
// the barriers sit below the TMEM address slot and the abort flag (offset 128)
static_assert(16 * F_NRING + 40 <= 128, "forward barriers overlap the TMEM slot");
constexpr int F_SMEM = F_BAR + 256 + 1024;

struct AttnParams {
    int B, T, C, H, nqt;
    bf16* out;
    float* lse;
    unsigned* err;
    float scale_log2;  // log2(e) / sqrt(hd)
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x with one MUFU instruction (ex2.approx: ~2 ulp; P is rounded to bf16 next)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// every lane of the warp waits (suspended in the barrier's try_wait until the
// phase completes: no divergent polling loop); the warp goes on only if all
// lanes saw the phase complete
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err, int lane) {
    (void)lane;
    const bool ok = mbar_wait(bar, parity, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// the 8 softmax warps (256 threads) synchronise among themselves
__device__ __forceinline__ void named_sync_softmax() {
    asm volatile("bar.sync 1, 256;" ::: "memory");
}
// the two softmax warps that share TMEM lane quarter q (warps w and w + 4 with
// w % 4 == q, among warps 2-9) synchronise: named barrier 2 + q, 64 threads
__device__ __forceinline__ void pair_sync(int q) {
    asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory");
}

constexpr int FWD_THREADS = 320;  // warp 0: TMA (lane 0); warp 1: MMA (lane 0); 8 softmax warps
constexpr float RESCALE_SLACK = 8.0f;  // log2 units: P stays <= 2^8 between rescales

__global__ void __launch_bounds__(FWD_THREADS, 2) k_attn_fwd_tc(const __grid_constant__ CUtensorMap map,
                                                                AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t sQ = base + F_Q, sRing = base + F_RING;
    float* red = (float*)(base_gen + F_RED);  // [2 buffers][2 halves][128 rows]
    float* lsum = (float*)(base_gen + F_LS);  // [2 halves][128 rows]
    const uint32_t bar = base + F_BAR;
    // full[F_NRING], empty[F_NRING] for the ring; q; s (S ready); pf (P ready);
    // o (P.V done); sfree (S copied to registers: the next S may overwrite it)
    const uint32_t b_full = bar, b_empty = bar + 8 * F_NRING, b_q = bar + 16 * F_NRING,
                   b_sfull = b_q + 8, b_pfull = b_q + 16, b_ofull = b_q + 24, b_sfree = b_q + 32;
    uint32_t* tmem_slot = (uint32_t*)(base_gen + F_BAR + 128);
    volatile int* abort_flag = (volatile int*)(base_gen + F_BAR + 132);

    // blocks launch in linear order, x fastest: every head's longest rows
    // first, so that the short tiles fill in the tail
    const int qt = p.nqt - 1 - (int)blockIdx.y;
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int nkt = qt + 1;
    const int row0 = b * p.T;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < F_NRING; i++) {
            mbar_init(b_full + 8 * i, 1);
            mbar_init(b_empty + 8 * i, 1);
        }
        mbar_init(b_q, 1);
        mbar_init(b_sfull, 1);
        mbar_init(b_pfull, 8);
        mbar_init(b_ofull, 1);
        mbar_init(b_sfree, 8);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map) : "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    gdc_wait();  // setup above touches no global memory
    gdc_launch_dependents();
    // S [128 x 128] fp32, O [128 x 64] fp32, P [128 x 128] bf16 (64 columns)
    const uint32_t tS = tmem, tO = tmem + 128, tP = tmem + 192;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ producer
            const int ck = p.C + h * HD, cv = 2 * p.C + h * HD;
            mbar_expect_tx(b_q, TILE_BYTES);
            tma_load_2d(sQ, &map, b_q, h * HD, row0 + qt * TILE);
            int last[F_NRING];  // use count of each slot's last load
            for (int s = 0; s < F_NRING; s++) last[s] = -1;
            for (int it = 0; it < 2 * nkt; it++) {
                const int s = it % F_NRING, u = it / F_NRING;
                if (!mbar_wait(b_empty + 8 * s, (u & 1) ^ 1, abort_flag, p.err)) break;
                mbar_expect_tx(b_full + 8 * s, TILE_BYTES);
                tma_load_2d(sRing + s * TILE_BYTES, &map, b_full + 8 * s, (it & 1) ? cv : ck,
                            row0 + (it >> 1) * TILE);
                last[s] = u;
            }
            if (*abort_flag) {
                for (int s = 0; s < F_NRING; s++) {
                    const int ls = last[s];
                    if (ls < 0) continue;
                    long long t0 = clock64();
                    while (!mbar_try(b_full + 8 * s, ls & 1) && clock64() - t0 < WAIT_LIMIT) {
                    }
                }
                long long t0 = clock64();
                while (!mbar_try(b_q, 0) && clock64() - t0 < WAIT_LIMIT) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ----------------------------------------------------------- MMA
            constexpr uint32_t ID_S = make_idesc(128, 128, false, false);
            constexpr uint32_t ID_O = make_idesc(128, 64, false, true);
            // descriptors are built once; a K step advances the start address
            // field (bits 0..13, in 16-byte units) by a constant
            const uint64_t dQ = sdesc(sQ, 0, 1024);
            const uint64_t dRingK = sdesc(sRing, 0, 1024), dRingV = sdesc(sRing, 8192, 1024);
            auto issue_s = [&](int j) -> bool {
                const int it = 2 * j, s = it % F_NRING;
                if (!mbar_wait(b_full + 8 * s, (it / F_NRING) & 1, abort_flag, p.err))
                    return false;
                tc_fence_after();
                const uint64_t dK = dRingK + (uint64_t)((s * TILE_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < HD / 16; k++)
                    umma_bf16(tS, dQ + (uint64_t)(k * 2), dK + (uint64_t)(k * 2), ID_S, k > 0);
                umma_commit(b_sfull);
                umma_commit(b_empty + 8 * s);
                return true;
            };
            bool ok = mbar_wait(b_q, 0, abort_flag, p.err) && issue_s(0);
            for (int j = 0; ok && j < nkt; j++) {
                // S_{j+1} as soon as the softmax warps hold S_j in registers,
                // so that it overlaps their work on tile j
                if (j + 1 < nkt) {
                    if (!mbar_wait(b_sfree, j & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    if (!issue_s(j + 1)) break;
                }
                if (!mbar_wait(b_pfull, j & 1, abort_flag, p.err)) break;
                tc_fence_after();
                const int it = 2 * j + 1, s = it % F_NRING;
                if (!mbar_wait(b_full + 8 * s, (it / F_NRING) & 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint64_t dV = dRingV + (uint64_t)((s * TILE_BYTES) >> 4);
                // O += P_j V_j (O starts at the first tile); P is read from TMEM,
                // 16 keys (8 columns) per instruction
#pragma unroll
                for (int k = 0; k < TILE / 16; k++)
                    umma_bf16_tmem_a(tO, tP + (uint32_t)(8 * k), dV + (uint64_t)(k * 128), ID_O,
                                     (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(b_ofull);
                umma_commit(b_empty + 8 * s);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        // warp pair (w, w+4) shares TMEM lane quarter w & 3: half 0 takes keys
        // [0,64) of each tile and output columns [0,32), half 1 the rest.
        // O accumulates in TMEM; the running max m used for P is raised (and O,
        // l rescaled) only when the row max exceeds it by more than 2^8, so P
        // stays <= 256 and most tiles need no rescale.
        const int q = warp & 3, hf = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const int qi = qt * TILE + r;
        const uint32_t loff = (uint32_t)(q * 32) << 16;
        const int kb = hf * 64;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        // After a failed wait a warp keeps going round the loop without work,
        // so that its partner warp still meets it at each barrier.
        for (int j = 0; j < nkt; j++) {
            if (!ok || !warp_wait(b_sfull, j & 1, abort_flag, p.err, lane)) {
                ok = false;
                pair_sync(q);
                continue;
            }
            tc_fence_after();
            uint32_t sv[2][32];
            tmem_ld32_async(tS + loff + kb, sv[0]);
            tmem_ld32_async(tS + loff + kb + 32, sv[1]);
            tmem_wait32(sv[0]);
            tmem_wait32(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_sfree);
            if (j == qt) {  // causal mask of the diagonal tile: keys > row
#pragma unroll
                for (int c = 0; c < 2; c++)
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (kb + 32 * c + i > r) sv[c][i] = __float_as_uint(-INFINITY);
            }
            // row max over the 64 columns as a tree (8 independent chains),
            // exchanged with the partner warp that holds the other 64
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) m8[i] = __uint_as_float(sv[0][i]);
#pragma unroll
            for (int i = 8; i < 64; i++) m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(sv[i >> 5][i & 31]));
#pragma unroll
            for (int w = 4; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; i++) m8[i] = fmaxf(m8[i], m8[i + w]);
            const float mx = m8[0];
            float* rb = red + (j & 1) * 256;
            rb[hf * 128 + r] = mx;
            pair_sync(q);
            const float mrow = fmaxf(rb[r], rb[128 + r]) * p.scale_log2;
            const bool need = mrow > m_used + RESCALE_SLACK;
            const float m_new = need ? mrow : m_used;
            // P_j in registers first (exponentials relative to m_new)
            uint32_t pk[32];
            float l4[4] = {0.f, 0.f, 0.f, 0.f};  // the tile's row sum in 4 chains
#pragma unroll
            for (int i = 0; i < 32; i++) {
                const float a =
                    ex2(fmaf(__uint_as_float(sv[i >> 4][(2 * i) & 31]), p.scale_log2, -m_new));
                const float e =
                    ex2(fmaf(__uint_as_float(sv[i >> 4][(2 * i + 1) & 31]), p.scale_log2, -m_new));
                l4[i & 3] += a + e;
                pk[i] = pack_bf16x2(a, e);
            }
            // P.V of the previous tile must be done: it reads the P columns of
            // TMEM and writes O, which a rescale rewrites
            if (j > 0 && !warp_wait(b_ofull, (j - 1) & 1, abort_flag, p.err, lane)) {
                ok = false;
                continue;
            }
            tc_fence_after();
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                const float corr = need ? ex2(m_used - m_new) : 1.f;
                uint32_t t[32];
                tmem_ld32_async(tO + loff + hf * 32, t);
                tmem_wait32(t);
#pragma unroll
                for (int i = 0; i < 32; i++) t[i] = __float_as_uint(__uint_as_float(t[i]) * corr);
                tmem_st32(tO + loff + hf * 32, t);
                l *= corr;
            }
            m_used = m_new;
            l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            // keys [kb, kb+64) of each row: 32 packed columns of P
            tmem_st32(tP + loff + hf * 32, pk);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pfull);
        }
        bool fin = ok && warp_wait(b_ofull, (nkt - 1) & 1, abort_flag, p.err, lane);
        uint32_t t[32];
        if (fin) {
            tc_fence_after();
            tmem_ld32_async(tO + loff + hf * 32, t);
            tmem_wait32(t);
        }
        // fold the two halves' row sums (every softmax thread reaches this)
        lsum[hf * 128 + r] = l;
        pair_sync(q);
        if (fin && qi < p.T) {
            const float lt = lsum[r] + lsum[128 + r];
            const float inv = 1.f / lt;
            bf16* dst = p.out + ((size_t)(row0 + qi)) * p.C + h * HD + hf * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint4 u;
                u.x = pack_bf16x2(__uint_as_float(t[i]) * inv, __uint_as_float(t[i + 1]) * inv);
                u.y = pack_bf16x2(__uint_as_float(t[i + 2]) * inv, __uint_as_float(t[i + 3]) * inv);
                u.z = pack_bf16x2(__uint_as_float(t[i + 4]) * inv, __uint_as_float(t[i + 5]) * inv);
                u.w = pack_bf16x2(__uint_as_float(t[i + 6]) * inv, __uint_as_float(t[i + 7]) * inv);
                *reinterpret_cast<uint4*>(dst + i) = u;
            }
            if (hf == 0) p.lse[(size_t)bh * p.T + qi] = (m_used + log2f(lt)) * 0.6931471805599453f;
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ---------------------------------------------------------------------------
// Backward.  With P = exp(S/sqrt(hd) - lse) recomputed from the saved lse and
// D = rowsum(dO o O):  dP = dO V^T, dS = P o (dP - D),
//   dV = P^T dO,  dK = dS^T Q / sqrt(hd),  dQ = dS K / sqrt(hd).
// k_attn_dkv_tc: one CTA per (128-key tile, batch, head), visiting query tiles
//   i >= key tile.  S^T = K Q_i^T and dP^T = V dO_i^T land in TMEM; one thread
//   per key row forms P^T and dS^T (bf16, swizzled smem), then
//   dV += P^T dO_i and dK += dS^T Q_i accumulate in TMEM (Q_i and dO_i tiles
//   are read K-major for the first products and MN-major for the second).
// k_attn_dq_tc (launched first): one CTA per (128-query tile, batch, head); it
//   forms D of its queries from its dO and O tiles and writes it, then visits
//   key tiles j <= query tile: S = Q K_j^T, dP = dO V_j^T, dS -> TMEM,
//   dQ += dS K_j (dS read from TMEM as the A operand).
// Each CTA owns its outputs: no atomics, deterministic.
// The 128-row side of each kernel (keys in k_attn_dkv_tc, queries in
// k_attn_dq_tc) is visited in steps of 64 on the other side, so every CTA
// holds at most 256 TMEM columns and ~100 KB of shared memory: two CTAs share
// an SM, and one CTA's softmax phase overlaps the other's products.
constexpr int BWD_THREADS = 320;  // warp 0: TMA (lane 0); warp 1: MMA (lane 0); 8 softmax warps
constexpr int SUB = 64;           // rows of the 64-wide side
constexpr int SUB_BYTES = SUB * 128;

struct AttnBwdParams {
    int B, T, C, H, nqt, nsub;  // nsub = ceil(T / 64)
    const float* lse;  // [B,H,T] natural log
    float* Dv;         // [B,H,T] rowsum(dO o O): written by the dQ kernel, read by dK/dV
    bf16* dqkv;
    unsigned* err;
    float scale_log2;  // log2(e)/sqrt(hd)
    float scale;       // 1/sqrt(hd)
};

// row r, columns [c0, c0+32) of a 128 x 64 bf16 K-major tile (one 128-byte
// swizzle atom column)
__device__ __forceinline__ void st_row32_64(uint32_t tile, int r, int c0, const uint32_t* pk) {
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
        const int chunk = (c0 >> 3) + cc;
        st_shared_v4(tile + r * 128 + ((uint32_t)(chunk ^ (r & 7)) << 4), pk[4 * cc],
                     pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
    }
}

struct BwdMaps {
    CUtensorMap qkv128, qkv64, do128, do64, o128;  // boxes 64 x 128 rows / 64 x 64 rows
};

// dK, dV: CTA = (128-key tile kt, batch, head); query steps of 64.
constexpr int D_K = 0, D_V = 16384, D_Q0 = 32768, D_Q1 = 40960, D_DO0 = 49152, D_DO1 = 57344,
              D_PT = 65536, D_DST = 81920, D_LSE = 98304, D_D = 98560, D_BAR = 98816;
constexpr int D_SMEM = D_BAR + 256 + 1024;

__global__ void __launch_bounds__(BWD_THREADS, 2)
    k_attn_dkv_tc(const __grid_constant__ BwdMaps maps, AttnBwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t sK = base + D_K, sV = base + D_V, sPT = base + D_PT, sDST = base + D_DST;
    float* lse_s = (float*)(base_gen + D_LSE);
    float* d_s = (float*)(base_gen + D_D);
    const uint32_t bar = base + D_BAR;
    const uint32_t b_kv = bar, b_qdf0 = bar + 8, b_qdf1 = bar + 16, b_qde0 = bar + 24,
                   b_qde1 = bar + 32, b_sfull = bar + 40, b_psfull = bar + 48,
                   b_psfree = bar + 56, b_acc = bar + 64, b_sfree = bar + 72;
    uint32_t* tmem_slot = (uint32_t*)(base_gen + D_BAR + 128);
    volatile int* abort_flag = (volatile int*)(base_gen + D_BAR + 132);

    const int kt = (int)blockIdx.y;  // most query steps first (x fastest: all heads)
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int i0 = 2 * kt;       // first 64-query step that sees these keys
    const int nq = p.nsub - i0;  // query steps
    const int row0 = b * p.T;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        mbar_init(b_qdf0, 1);
        mbar_init(b_qdf1, 1);
        mbar_init(b_qde0, 1);
        mbar_init(b_qde1, 1);
        mbar_init(b_sfull, 1);
        mbar_init(b_psfull, 8);
        mbar_init(b_psfree, 1);
        mbar_init(b_acc, 1);
        mbar_init(b_sfree, 8);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    gdc_wait();  // setup above touches no global memory
    gdc_launch_dependents();
    const uint32_t tST = tmem, tDPT = tmem + 64, tDV = tmem + 128, tDK = tmem + 192;

    if (warp == 0) {
        if (lane == 0) {
            const int ck = p.C + h * HD, cv = 2 * p.C + h * HD;
            mbar_expect_tx(b_kv, 2 * TILE_BYTES);
            tma_load_2d(sK, &maps.qkv128, b_kv, ck, row0 + kt * TILE);
            tma_load_2d(sV, &maps.qkv128, b_kv, cv, row0 + kt * TILE);
            int issued0 = -1, issued1 = -1;
            for (int n = 0; n < nq; n++) {
                const int s = n & 1, u = n >> 1;
                if (!mbar_wait(s ? b_qde1 : b_qde0, (u & 1) ^ 1, abort_flag, p.err)) break;
                const uint32_t ff = s ? b_qdf1 : b_qdf0;
                const int qrow = row0 + (i0 + n) * SUB;
                mbar_expect_tx(ff, 2 * SUB_BYTES);
                tma_load_2d(base + (s ? D_Q1 : D_Q0), &maps.qkv64, ff, h * HD, qrow);
                tma_load_2d(base + (s ? D_DO1 : D_DO0), &maps.do64, ff, h * HD, qrow);
                if (s) issued1 = u;
                else issued0 = u;
            }
            if (*abort_flag) {
                for (int s = 0; s < 2; s++) {
                    const int is = s ? issued1 : issued0;
                    if (is < 0) continue;
                    long long t0 = clock64();
                    while (!mbar_try(s ? b_qdf1 : b_qdf0, is & 1) && clock64() - t0 < WAIT_LIMIT) {
                    }
                }
                long long t0 = clock64();
                while (!mbar_try(b_kv, 0) && clock64() - t0 < WAIT_LIMIT) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = make_idesc(128, SUB, false, false);
            constexpr uint32_t ID_O = make_idesc(128, 64, false, true);
            const uint64_t dK = sdesc(sK, 0, 1024), dV = sdesc(sV, 0, 1024);
            const uint64_t dPT = sdesc(sPT, 0, 1024), dDST = sdesc(sDST, 0, 1024);
            // S^T = K Q_n^T and dP^T = V dO_n^T (128 keys x 64 queries)
            auto issue_s = [&](int n) -> bool {
                const int s = n & 1, u = n >> 1;
                if (!mbar_wait(s ? b_qdf1 : b_qdf0, u & 1, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t sq = base + (s ? D_Q1 : D_Q0), sd = base + (s ? D_DO1 : D_DO0);
                const uint64_t dq_k = sdesc(sq, 0, 1024), dd_k = sdesc(sd, 0, 1024);
#pragma unroll
                for (int k = 0; k < HD / 16; k++)
                    umma_bf16(tST, dK + (uint64_t)(2 * k), dq_k + (uint64_t)(2 * k), ID_S, k > 0);
#pragma unroll
                for (int k = 0; k < HD / 16; k++)
                    umma_bf16(tDPT, dV + (uint64_t)(2 * k), dd_k + (uint64_t)(2 * k), ID_S, k > 0);
                umma_commit(b_sfull);
                return true;
            };
            bool ok = mbar_wait(b_kv, 0, abort_flag, p.err) && issue_s(0);
            for (int n = 0; ok && n < nq; n++) {
                const int s = n & 1;
                const uint32_t sq = base + (s ? D_Q1 : D_Q0), sd = base + (s ? D_DO1 : D_DO0);
                const uint64_t dq_m = sdesc(sq, 8192, 1024), dd_m = sdesc(sd, 8192, 1024);
                // the next step's products as soon as the softmax warps hold
                // this step's S^T and dP^T in registers
                if (n + 1 < nq) {
                    if (!mbar_wait(b_sfree, n & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    if (!issue_s(n + 1)) break;
                }
                if (!mbar_wait(b_psfull, n & 1, abort_flag, p.err)) break;
                tc_fence_after();
                // dV += P^T dO, dK += dS^T Q (K = the 64 queries)
#pragma unroll
                for (int k = 0; k < SUB / 16; k++) {
                    umma_bf16(tDV, dPT + (uint64_t)(2 * k), dd_m + (uint64_t)(128 * k), ID_O,
                              (n > 0 || k > 0));
                    umma_bf16(tDK, dDST + (uint64_t)(2 * k), dq_m + (uint64_t)(128 * k), ID_O,
                              (n > 0 || k > 0));
                }
                umma_commit(s ? b_qde1 : b_qde0);
                umma_commit(b_psfree);
            }
            if (ok) umma_commit(b_acc);
        }
    } else {
        // warp pair (w, w+4) shares TMEM lane quarter w & 3; half hf takes query
        // columns [32 hf, 32 hf + 32) of each step and output columns [32 hf, +32)
        const int q = warp & 3, hf = (warp - 2) >> 2;
        const int r = q * 32 + lane;   // key row within the tile
        const int kj = kt * TILE + r;  // key index in the sequence
        const int tid = threadIdx.x - 64;
        const uint32_t loff = (uint32_t)(q * 32) << 16;
        const int c0 = hf * 32;
        bool ok = true;
        for (int n = 0; n < nq; n++) {
            const int qbase = (i0 + n) * SUB;
            named_sync_softmax();  // everyone is done with the previous lse/D
            if (tid < SUB) {
                const int qi = qbase + tid;
                lse_s[tid] = qi < p.T ? p.lse[(size_t)bh * p.T + qi] * 1.4426950408889634f : 0.f;
                d_s[tid] = qi < p.T ? p.Dv[(size_t)bh * p.T + qi] : 0.f;
            }
            named_sync_softmax();
            // after a failed wait a warp goes on round the loop without work,
            // so that every softmax thread still meets each named barrier
            if (!ok) continue;
            if (!warp_wait(b_sfull, n & 1, abort_flag, p.err, lane)) {
                ok = false;
                continue;
            }
            tc_fence_after();
            uint32_t sv[32], dp[32];
            tmem_ld32_async(tST + loff + c0, sv);
            tmem_ld32_async(tDPT + loff + c0, dp);
            tmem_wait32(sv);
            tmem_wait32(dp);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_sfree);  // the next S^T, dP^T may land
            // the whole step lies after this key tile and inside the sequence
            const bool full = qbase >= kt * TILE + TILE && qbase + SUB <= p.T;
            uint32_t pp[16], dd[16];
            if (full) {
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    const int c = c0 + 2 * e;
                    const float p0 = ex2(fmaf(__uint_as_float(sv[2 * e]), p.scale_log2, -lse_s[c]));
                    const float p1 =
                        ex2(fmaf(__uint_as_float(sv[2 * e + 1]), p.scale_log2, -lse_s[c + 1]));
                    pp[e] = pack_bf16x2(p0, p1);
                    dd[e] = pack_bf16x2(p0 * (__uint_as_float(dp[2 * e]) - d_s[c]),
                                        p1 * (__uint_as_float(dp[2 * e + 1]) - d_s[c + 1]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int z = 0; z < 2; z++) {
                        const int c = c0 + 2 * e + z;
                        const int qi = qbase + c;
                        const bool live = qi < p.T && kj <= qi;
                        const float pr = live ? ex2(fmaf(__uint_as_float(sv[2 * e + z]),
                                                         p.scale_log2, -lse_s[c]))
                                              : 0.f;
                        pv[z] = pr;
                        dv[z] = live ? pr * (__uint_as_float(dp[2 * e + z]) - d_s[c]) : 0.f;
                    }
                    pp[e] = pack_bf16x2(pv[0], pv[1]);
                    dd[e] = pack_bf16x2(dv[0], dv[1]);
                }
            }
            // the previous step's products must be done reading the P^T, dS^T tiles
            if (n > 0 && !warp_wait(b_psfree, (n - 1) & 1, abort_flag, p.err, lane)) {
                ok = false;
                continue;
            }
            st_row32_64(sPT, r, c0, pp);
            st_row32_64(sDST, r, c0, dd);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_psfull);
        }
        if (ok && warp_wait(b_acc, 0, abort_flag, p.err, lane)) {
            tc_fence_after();
            bf16* dst = p.dqkv + (size_t)(row0 + kj) * 3 * p.C + h * HD + hf * 32;
            uint32_t v[32], k[32];
            tmem_ld32_async(tDV + loff + hf * 32, v);
            tmem_ld32_async(tDK + loff + hf * 32, k);
            tmem_wait32(v);
            tmem_wait32(k);
            if (kj < p.T) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 uv, uk;
                    uv.x = pack_bf16x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
                    uv.y = pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                    uv.z = pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
                    uv.w = pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
                    uk.x = pack_bf16x2(__uint_as_float(k[e]) * p.scale, __uint_as_float(k[e + 1]) * p.scale);
                    uk.y = pack_bf16x2(__uint_as_float(k[e + 2]) * p.scale, __uint_as_float(k[e + 3]) * p.scale);
                    uk.z = pack_bf16x2(__uint_as_float(k[e + 4]) * p.scale, __uint_as_float(k[e + 5]) * p.scale);
                    uk.w = pack_bf16x2(__uint_as_float(k[e + 6]) * p.scale, __uint_as_float(k[e + 7]) * p.scale);
                    *reinterpret_cast<uint4*>(dst + 2 * p.C + e) = uv;
                    *reinterpret_cast<uint4*>(dst + p.C + e) = uk;
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// dQ: CTA = (128-query tile qt, batch, head); key steps of 64 through a ring of
// E_NRING (K_j, V_j) slots; dS lives in TMEM.  The CTA also forms D =
// rowsum(dO o O) of its queries (from its dO and O tiles) and writes it for
// the dK/dV kernel, which runs after it.
constexpr int E_NRING = 3;
constexpr int E_Q = 0, E_DO = 16384, E_O = 32768, E_KV = 49152,
              E_BAR = E_KV + E_NRING * 2 * SUB_BYTES, E_DX = E_BAR + 256;
constexpr int E_SMEM = E_DX + 1024 + 1024;

__global__ void __launch_bounds__(BWD_THREADS, 2)
    k_attn_dq_tc(const __grid_constant__ BwdMaps maps, AttnBwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t sQ = base + E_Q, sDO = base + E_DO, sKV = base + E_KV;
    const uint32_t bar = base + E_BAR;
    // q; kv full[E_NRING]; kv empty[E_NRING]; s, ds full / free, acc, s consumed
    const uint32_t b_q = bar, b_kvf = bar + 8, b_kve = bar + 8 + 8 * E_NRING,
                   b_sfull = bar + 8 + 16 * E_NRING, b_dsfull = b_sfull + 8,
                   b_dsfree = b_sfull + 16, b_acc = b_sfull + 24, b_sfree = b_sfull + 32;
    uint32_t* tmem_slot = (uint32_t*)(base_gen + E_BAR + 128);
    volatile int* abort_flag = (volatile int*)(base_gen + E_BAR + 132);

    const int qt = p.nqt - 1 - (int)blockIdx.y;  // most key steps first
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int nk = min(2 * qt + 2, p.nsub);  // 64-key steps 0..nk-1
    const int row0 = b * p.T;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int i = 0; i < E_NRING; i++) {
            mbar_init(b_kvf + 8 * i, 1);
            mbar_init(b_kve + 8 * i, 1);
        }
        mbar_init(b_sfull, 1);
        mbar_init(b_dsfull, 8);
        mbar_init(b_dsfree, 1);
        mbar_init(b_acc, 1);
        mbar_init(b_sfree, 8);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    gdc_wait();  // setup above touches no global memory
    gdc_launch_dependents();
    // S, dP, dQ [128 x 64] fp32; dS [128 x 64] bf16 (32 columns)
    const uint32_t tS = tmem, tDP = tmem + 64, tDQ = tmem + 128, tDS = tmem + 192;

    if (warp == 0) {
        if (lane == 0) {
            const int ck = p.C + h * HD, cv = 2 * p.C + h * HD;
            mbar_expect_tx(b_q, 3 * TILE_BYTES);
            tma_load_2d(sQ, &maps.qkv128, b_q, h * HD, row0 + qt * TILE);
            tma_load_2d(sDO, &maps.do128, b_q, h * HD, row0 + qt * TILE);
            tma_load_2d(base + E_O, &maps.o128, b_q, h * HD, row0 + qt * TILE);
            int issued[E_NRING];
            for (int s = 0; s < E_NRING; s++) issued[s] = -1;
            for (int j = 0; j < nk; j++) {
                const int s = j % E_NRING, u = j / E_NRING;
                if (!mbar_wait(b_kve + 8 * s, (u & 1) ^ 1, abort_flag, p.err)) break;
                const uint32_t ff = b_kvf + 8 * s;
                mbar_expect_tx(ff, 2 * SUB_BYTES);
                tma_load_2d(sKV + s * 2 * SUB_BYTES, &maps.qkv64, ff, ck, row0 + j * SUB);
                tma_load_2d(sKV + s * 2 * SUB_BYTES + SUB_BYTES, &maps.qkv64, ff, cv,
                            row0 + j * SUB);
                issued[s] = u;
            }
            if (*abort_flag) {
                for (int s = 0; s < E_NRING; s++) {
                    const int is = issued[s];
                    if (is < 0) continue;
                    long long t0 = clock64();
                    while (!mbar_try(b_kvf + 8 * s, is & 1) && clock64() - t0 < WAIT_LIMIT) {
                    }
                }
                long long t0 = clock64();
                while (!mbar_try(b_q, 0) && clock64() - t0 < WAIT_LIMIT) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = make_idesc(128, SUB, false, false);
            constexpr uint32_t ID_O = make_idesc(128, 64, false, true);
            const uint64_t dQ = sdesc(sQ, 0, 1024), dDO = sdesc(sDO, 0, 1024);
            // S = Q K_j^T, dP = dO V_j^T (128 queries x 64 keys)
            auto issue_s = [&](int j) -> bool {
                const int s = j % E_NRING, u = j / E_NRING;
                if (!mbar_wait(b_kvf + 8 * s, u & 1, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t sk = sKV + s * 2 * SUB_BYTES, sv = sk + SUB_BYTES;
                const uint64_t dk_k = sdesc(sk, 0, 1024), dv_k = sdesc(sv, 0, 1024);
#pragma unroll
                for (int k = 0; k < HD / 16; k++)
                    umma_bf16(tS, dQ + (uint64_t)(2 * k), dk_k + (uint64_t)(2 * k), ID_S, k > 0);
#pragma unroll
                for (int k = 0; k < HD / 16; k++)
                    umma_bf16(tDP, dDO + (uint64_t)(2 * k), dv_k + (uint64_t)(2 * k), ID_S, k > 0);
                umma_commit(b_sfull);
                return true;
            };
            bool ok = mbar_wait(b_q, 0, abort_flag, p.err) && issue_s(0);
            for (int j = 0; ok && j < nk; j++) {
                const int s = j % E_NRING;
                const uint32_t sk = sKV + s * 2 * SUB_BYTES;
                const uint64_t dk_m = sdesc(sk, 8192, 1024);
                // the next step's products as soon as the softmax warps hold
                // this step's S and dP in registers
                if (j + 1 < nk) {
                    if (!mbar_wait(b_sfree, j & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    if (!issue_s(j + 1)) break;
                }
                if (!mbar_wait(b_dsfull, j & 1, abort_flag, p.err)) break;
                tc_fence_after();
                // dQ += dS K_j (K = the 64 keys; dS read from TMEM, 8 columns
                // = 16 keys per instruction)
#pragma unroll
                for (int k = 0; k < SUB / 16; k++)
                    umma_bf16_tmem_a(tDQ, tDS + (uint32_t)(8 * k), dk_m + (uint64_t)(128 * k),
                                     ID_O, (j > 0 || k > 0));
                umma_commit(b_kve + 8 * s);
                umma_commit(b_dsfree);
            }
            if (ok) umma_commit(b_acc);
        }
    } else {
        const int q = warp & 3, hf = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const int qi = qt * TILE + r;
        const uint32_t loff = (uint32_t)(q * 32) << 16;
        const int c0 = hf * 32;
        const bool qlive = qi < p.T;
        const float lse2 = qlive ? p.lse[(size_t)bh * p.T + qi] * 1.4426950408889634f : 0.f;
        bool ok = warp_wait(b_q, 0, abort_flag, p.err, lane);
        // D of this row: the half's 32 products from the swizzled dO and O
        // tiles, then the two halves added in half order
        float dpart = 0.f;
        if (ok) {
            const uint8_t* rdo = base_gen + E_DO + r * 128;
            const uint8_t* ro = base_gen + E_O + r * 128;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int off = ((hf * 4 + c) ^ (r & 7)) << 4;
                const uint4 a = *reinterpret_cast<const uint4*>(rdo + off);
                const uint4 o = *reinterpret_cast<const uint4*>(ro + off);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const float av = __uint_as_float((e & 1) ? (aw[e >> 1] & 0xffff0000u) : (aw[e >> 1] << 16));
                    const float ov = __uint_as_float((e & 1) ? (ow[e >> 1] & 0xffff0000u) : (ow[e >> 1] << 16));
                    dpart = fmaf(av, ov, dpart);
                }
            }
        }
        float* dx_s = reinterpret_cast<float*>(base_gen + E_DX);  // [2 halves][128 rows]
        dx_s[hf * 128 + r] = dpart;
        named_sync_softmax();
        const float Dq = qlive ? dx_s[r] + dx_s[128 + r] : 0.f;
        if (ok && hf == 0 && qlive) p.Dv[(size_t)bh * p.T + qi] = Dq;
        for (int j = 0; j < nk; j++) {
            if (!warp_wait(b_sfull, j & 1, abort_flag, p.err, lane)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[32], dp[32];
            tmem_ld32_async(tS + loff + c0, sv);
            tmem_ld32_async(tDP + loff + c0, dp);
            tmem_wait32(sv);
            tmem_wait32(dp);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_sfree);  // the next S, dP may land
            const int kbase = j * SUB;
            uint32_t dd[16];
            if (kbase + SUB <= qt * TILE) {  // every key of the step precedes every query
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    const float p0 = ex2(fmaf(__uint_as_float(sv[2 * e]), p.scale_log2, -lse2));
                    const float p1 = ex2(fmaf(__uint_as_float(sv[2 * e + 1]), p.scale_log2, -lse2));
                    dd[e] = pack_bf16x2(p0 * (__uint_as_float(dp[2 * e]) - Dq),
                                        p1 * (__uint_as_float(dp[2 * e + 1]) - Dq));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    float dv[2];
#pragma unroll
                    for (int z = 0; z < 2; z++) {
                        const int kk = kbase + c0 + 2 * e + z;
                        const bool live = qlive && kk <= qi;
                        const float pr =
                            live ? ex2(fmaf(__uint_as_float(sv[2 * e + z]), p.scale_log2, -lse2))
                                 : 0.f;
                        dv[z] = live ? pr * (__uint_as_float(dp[2 * e + z]) - Dq) : 0.f;
                    }
                    dd[e] = pack_bf16x2(dv[0], dv[1]);
                }
            }
            // the previous step's product must be done reading the dS columns
            if (j > 0 && !warp_wait(b_dsfree, (j - 1) & 1, abort_flag, p.err, lane)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st16(tDS + loff + (uint32_t)(c0 >> 1), dd);  // keys c0.. of the step
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_dsfull);
        }
        const bool fin = ok && warp_wait(b_acc, 0, abort_flag, p.err, lane);
        uint32_t v[32];
        if (fin) {
            tc_fence_after();
            bf16* dst = p.dqkv + (size_t)(row0 + qi) * 3 * p.C + h * HD + hf * 32;
            tmem_ld32_async(tDQ + loff + hf * 32, v);
            tmem_wait32(v);
            if (qlive) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 u;
                    u.x = pack_bf16x2(__uint_as_float(v[e]) * p.scale, __uint_as_float(v[e + 1]) * p.scale);
                    u.y = pack_bf16x2(__uint_as_float(v[e + 2]) * p.scale, __uint_as_float(v[e + 3]) * p.scale);
                    u.z = pack_bf16x2(__uint_as_float(v[e + 4]) * p.scale, __uint_as_float(v[e + 5]) * p.scale);
                    u.w = pack_bf16x2(__uint_as_float(v[e + 6]) * p.scale, __uint_as_float(v[e + 7]) * p.scale);
                    *reinterpret_cast<uint4*>(dst + e) = u;
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

bool attention_tc_supported(int act, int B, int T, int C, int H, const void* qkv) {
    if (act != ACT_BF16 || H < 1 || C % H || C / H != HD || C % 8) return false;
    if (((uintptr_t)qkv & 15) != 0) return false;
    if ((long)B * T >= (1L << 31) - 256) return false;
    return tc_encode_fn() != nullptr;
}

static bool map_rows(CUtensorMap* m, const void* base, long width, long rows, int box_rows) {
    EncodeTiledFn enc = (EncodeTiledFn)tc_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)width * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t attention_backward_tc(void* dqkv, const void* dout, const void* qkv, const void* out,
                                  const float* lse, float* Dv, int B, int T, int C, int H,
                                  unsigned* err, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_dkv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, D_SMEM);
        cudaFuncSetAttribute(k_attn_dq_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, E_SMEM);
        attr = true;
    }
    if (((uintptr_t)dout & 15) || ((uintptr_t)dqkv & 15) || ((uintptr_t)out & 15))
        return cudaErrorInvalidValue;
    BwdMaps maps;
    const long rows = (long)B * T;
    if (!map_rows(&maps.qkv128, qkv, 3L * C, rows, 128) ||
        !map_rows(&maps.qkv64, qkv, 3L * C, rows, 64) ||
        !map_rows(&maps.do128, dout, C, rows, 128) || !map_rows(&maps.do64, dout, C, rows, 64) ||
        !map_rows(&maps.o128, out, C, rows, 128))
        return cudaErrorInvalidValue;
    AttnBwdParams p;
    p.B = B; p.T = T; p.C = C; p.H = H;
    p.nqt = (T + TILE - 1) / TILE;
    p.nsub = (T + SUB - 1) / SUB;
    p.lse = lse;
    p.Dv = Dv;
    p.dqkv = (bf16*)dqkv;
    p.err = err;
    p.scale = 1.0f / sqrtf((float)HD);
    p.scale_log2 = 1.4426950408889634f * p.scale;
    dim3 grid(B * H, p.nqt);
    // dQ first: it also writes D, which dK/dV reads
    launch_pdl(k_attn_dq_tc, grid, BWD_THREADS, E_SMEM, s, maps, p);
    launch_pdl(k_attn_dkv_tc, grid, BWD_THREADS, D_SMEM, s, maps, p);
    return cudaGetLastError();
}

cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C,
                                 int H, unsigned* err, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM);
        attr = true;
    }
    EncodeTiledFn enc = (EncodeTiledFn)tc_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)3 * C, (cuuint64_t)B * T};
    cuuint64_t strides[1] = {(cuuint64_t)3 * C * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    AttnParams p;
    p.B = B; p.T = T; p.C = C; p.H = H;
    p.nqt = (T + TILE - 1) / TILE;
    p.out = (bf16*)out;
    p.lse = lse;
    p.err = err;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
    dim3 grid(B * H, p.nqt);
    launch_pdl(k_attn_fwd_tc, grid, FWD_THREADS, F_SMEM, s, map, p);
    return cudaGetLastError();
}

}  // namespace gk
