// gemm_tc_kernel.cuh -- bf16 x bf16 -> fp32 matmul on the 5th-generation tensor cores
// of sm_103a (tcgen05.mma, accumulator in tensor memory), operands staged in
// shared memory by TMA, with the fused epilogues of the GPT-2 step.
//
// These are the dense contractions of the step -- the QKV, attention-output,
// MLP and tied-classifier linear layers of "Karpathy's llm.c: understanding
// LLM training from scratch in C/CUDA", "Code anatomy", forward and backward
// (the pages run them through cuBLAS/cuBLASLt with a GELU epilogue,
// "Karpathy reproduces GPT-2 (1.6B) in llm.c", flag guide; here they are
// written directly for the B300).
//
// D[M,N] = A[M,K] . B[N,K]^T.  Each operand is either K-major (rows of K
// contiguous) or M/N-major (the transpose is stored); the instruction
// descriptor's transpose bits select the smem layout, so dX = dY W and
// dW = dY^T X run without transposed copies.
//
// Kernel organisation (one persistent CTA per SM, 320 threads):
//   warp 0    TMA producer: 2-D tiled loads, 128-byte swizzle, STAGES-deep
//             ring of (A, B) stages guarded by full/empty mbarriers
//   warp 1    allocates 2*BN TMEM columns; lane 0 issues tcgen05.mma
//             (M=128, N=BN, K=16) and tcgen05.commit to free stages and to
//             publish a finished accumulator
//   warps 2-9 epilogue: warp w takes TMEM lane quarter w % 4 and one half of
//             the tile's columns: tcgen05.ld in 32-column chunks, bias / GELU
//             / residual / fp32 accumulate, staged in shared memory and
//             written by TMA bulk stores
// Two TMEM accumulators let the epilogue of tile i overlap the mainloop of
// tile i+1.  Every mbarrier wait is bounded (clock64 budget): on expiry the
// CTA raises an abort flag, sets GPT2_DEVERR_TIMEOUT in the device error
// word, lets every role leave its loop, waits for its own TMA loads, frees
// its TMEM and returns.
//
// Weight-gradient products have K = B*T (16384) and few output tiles; they
// are split along K into fp32 partial tiles summed in a fixed order by a
// second kernel (deterministic; no float atomics).
// This header holds the kernel template (the epilogue mode is a template
// parameter, so each mode's code is compiled on its own: smaller, and without
// runtime branches on the mode) and its launchers; k_gemm_tc_epi_*.cu
// instantiate the launchers two modes per file, k_gemm_tc.cu holds the host
// logic (tile choice, split-K model, the shared state).
#pragma once
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace gk {
namespace tcg {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int NUM_THREADS = 320;  // producer, MMA, 8 epilogue warps

// BN = 256 tiles run on CTA pairs (tcgen05 cta_group::2): the pair computes a
// 256 x 256 tile, each CTA holding 128 rows of A and 128 rows (of N) of B, so
// a stage is 32 KB per CTA and six fit; BN = 128 tiles run on single CTAs.
template <int BN, int KB>
struct Cfg {
    static constexpr bool PAIR = BN == 256;
    // KB k-blocks (64 deep) per pipeline stage: two halve the stage barriers
    // and commits per instruction, which pays on the long-K products
    static constexpr int KB2 = KB;
    static constexpr int STAGES = 6 / KB2;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
    static constexpr int HALF_BYTES = A_BYTES + B_BYTES;  // one k-block
    static constexpr int STAGE_BYTES = KB2 * HALF_BYTES;
    static constexpr int STG_BYTES = 8 * 4096;  // epilogue staging: 4 KB per epilogue warp
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = STAGES * STAGE_BYTES + STG_BYTES + 1024 + BAR_BYTES;
};

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, splits, k_per_split, num_tiles;
    int n_fastest;  // work-unit order: 1 = output-column tiles vary fastest
    int epi;
    void* D;
    long ldd;
    const bf16* bias;
    const bf16* resid;
    long ldr;
    bf16* aux;
    long ldx;
    float* part;
    // EPI_MUL_AUX / EPI_GELU_BWD: column sums of each 32-row block of D (its
    // bf16 values, summed in fp32), [ceil(M/32)][N], or NULL
    float* colpart;
    unsigned* err;
};

enum { EPI_PART_F32 = 100 };

// ------------------------------------------------------------------ epilogue
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void ld8_bf16(float* f, const bf16* p) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ void st8_bf16(bf16* p, const float* f) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}

// GELU and GELU' for the bf16 epilogues: the same sigmoid form as gelu_f /
// gelu_grad_f with the fast exp and divide intrinsics (a few fp32 ulp, far
// below the bf16 rounding of the stored result); u is clamped at -40 so the
// divisor stays finite.
__device__ __forceinline__ float gelu_fast(float x) {
    const float k = 0.7978845608028654f;
    float u = fmaxf(k * (x + 0.044715f * x * x * x), -40.0f);
    return __fdividef(x, 1.0f + __expf(-2.0f * u));
}
// gelu(x) and gelu'(x) sharing one sigmoid s = 1/(1 + e^{-2u}) (two MUFU
// operations).  With u = k (x + c x^3), the derivative term 2 x du/dx equals
// 6u - 4kx exactly, so gelu' = s + (s - s^2)(6u - 4kx) costs three FMAs.
__device__ __forceinline__ void gelu_and_grad_fast(float x, float& g, float& dg) {
    const float k = 0.7978845608028654f;
    const float u = k * fmaf(0.044715f * x, x * x, x);
    const float s = __fdividef(1.0f, 1.0f + __expf(-2.0f * fmaxf(u, -40.0f)));
    g = x * s;
    dg = fmaf(fmaf(-s, s, s), fmaf(-4.0f * k, x, 6.0f * u), s);
}
__device__ __forceinline__ float gelu_grad_fast(float x) {
    const float k = 0.7978845608028654f;
    float x2 = x * x;
    float u = fmaxf(k * (x + 0.044715f * x2 * x), -40.0f);
    float sg = __fdividef(1.0f, 1.0f + __expf(-2.0f * u));
    float du = k * (1.0f + 3.0f * 0.044715f * x2);
    return sg + 2.0f * x * sg * (1.0f - sg) * du;
}

// TMA bulk-store helpers (smem -> global through a tensor map)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"((uint64_t)map), "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"((uint64_t)map), "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
        ::"l"((uint64_t)map), "r"(src), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// row r of a 32 x 32 bf16 staging tile (64-byte rows, 64-byte swizzle)
__device__ __forceinline__ void stage_bf16_row(uint32_t stg, int r, const float* x) {
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float* f = x + 8 * k;
        st_shared_v4(stg + r * 64 + ((uint32_t)(k ^ ((r >> 1) & 3)) << 4),
                     pack2_bf16(f[0], f[1]), pack2_bf16(f[2], f[3]), pack2_bf16(f[4], f[5]),
                     pack2_bf16(f[6], f[7]));
    }
}
// row r of a 32 x 32 fp32 staging tile (128-byte rows, 128-byte swizzle)
__device__ __forceinline__ void stage_f32_row(uint32_t stg, int r, const float* x) {
#pragma unroll
    for (int k = 0; k < 8; k++)
        st_shared_v4(stg + r * 128 + ((uint32_t)(k ^ (r & 7)) << 4), __float_as_uint(x[4 * k]),
                     __float_as_uint(x[4 * k + 1]), __float_as_uint(x[4 * k + 2]),
                     __float_as_uint(x[4 * k + 3]));
}

struct EpiMaps {
    CUtensorMap d;    // bf16 [M,N] box 32x32 SW64, or fp32 [M,N] box 32x32 SW128 (accumulate)
    CUtensorMap aux;  // bf16 [M,N] box 32x32 SW64 (GELU pre-activation, or gelu')
    CUtensorMap part; // fp32 [splits,M,N] box 32x32x1 SW128 (split-K partials)
};

// ------------------------------------------------------- CTA-pair helpers
// (tcgen05 cta_group::2: the pair's MMAs are issued by the leader, rank 0;
// every load and every signal goes to one CTA's own barrier, one copy per
// destination)
__device__ __forceinline__ uint32_t pair_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t pair_mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void pair_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// TMA 2-D load into this CTA's shared memory whose completion is counted on
// the mbarrier at cluster address `bar` (the leader's)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}
// arrive (once the pair's MMAs issued so far complete) on the mbarrier at
// cluster address `bar`
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

// Row-wise operand of a chunk that comes from global memory (the residual for
// EPI_RESID, the pre-activation for EPI_GELU_BWD): 32 bf16 of this lane's row,
// loaded one chunk ahead so the load latency hides behind the previous chunk.
template <int EPI>
__device__ __forceinline__ void epi_prefetch(const TcParams& p, int row, int col, uint4 (&pf)[4]) {
    const bf16* src = nullptr;
    if (EPI == EPI_RESID) src = p.resid + (size_t)row * p.ldr + col;
    else if (EPI == EPI_GELU_BWD || EPI == EPI_MUL_AUX) src = p.aux + (size_t)row * p.ldx + col;
    const int nv = min(32, p.N - col);
#pragma unroll
    for (int k = 0; k < 4; k++)
        pf[k] = (src && row < p.M && 8 * k < nv) ? *reinterpret_cast<const uint4*>(src + 8 * k)
                                                  : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void unpack8_bf16(float* f, uint4 u) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// One warp: the 32 x 32 chunk at rows [row0, row0+32), columns [col, col+32);
// lane = row within the chunk; v = this lane's 32 accumulator values; pf =
// this lane's prefetched row operand (see epi_prefetch).
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const EpiMaps& m, int row0,
                                               int col, int lane, float* v, int split,
                                               uint32_t stg, const uint4 (&pf)[4]) {
    const int nv = min(32, p.N - col);  // multiple of 8
    if (EPI == EPI_GELU_BWD) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            float pre[8];
            unpack8_bf16(pre, pf[k]);
#pragma unroll
            for (int i = 0; i < 8; i++) v[8 * k + i] *= gelu_grad_fast(pre[i]);
        }
    } else if (EPI == EPI_MUL_AUX) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            float dg[8];
            unpack8_bf16(dg, pf[k]);
#pragma unroll
            for (int i = 0; i < 8; i++) v[8 * k + i] *= dg[i];
        }
    } else if (EPI != EPI_ACCUM_F32 && EPI != EPI_PART_F32) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (p.bias && 8 * k < nv) {
                float b[8];
                ld8_bf16(b, p.bias + col + 8 * k);
#pragma unroll
                for (int i = 0; i < 8; i++) v[8 * k + i] += b[i];
            }
            if (EPI == EPI_RESID) {
                float r8[8];
                unpack8_bf16(r8, pf[k]);
#pragma unroll
                for (int i = 0; i < 8; i++) v[8 * k + i] += r8[i];
            }
        }
    }
    // the previous chunk's bulk stores must have finished reading the staging tile
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    if (EPI == EPI_ACCUM_F32 || EPI == EPI_PART_F32) {
        stage_f32_row(stg, lane, v);
    } else if (EPI == EPI_GELU_D) {
        float dg[32];
#pragma unroll
        for (int i = 0; i < 32; i++) gelu_and_grad_fast(v[i], v[i], dg[i]);
        stage_bf16_row(stg + 2048, lane, dg);  // gelu'
        stage_bf16_row(stg, lane, v);
    } else if (EPI == EPI_GELU) {
        stage_bf16_row(stg + 2048, lane, v);  // pre-activation
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = gelu_fast(v[i]);
        stage_bf16_row(stg, lane, v);
    } else {
        stage_bf16_row(stg, lane, v);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (EPI == EPI_ACCUM_F32) tma_reduce_add_2d(&m.d, stg, col, row0);
        else if (EPI == EPI_PART_F32) tma_store_3d(&m.part, stg, col, row0, split);
        else {
            tma_store_2d(&m.d, stg, col, row0);
            if (EPI == EPI_GELU || EPI == EPI_GELU_D)
                tma_store_2d(&m.aux, stg + 2048, col, row0);
        }
        bulk_commit();
    }
    if ((EPI == EPI_MUL_AUX || EPI == EPI_GELU_BWD) && p.colpart) {
        // column sums of the staged (bf16) piece, read back from shared memory
        // beside the bulk store: lane l takes columns 2(l & 15), 2(l & 15) + 1
        // over rows 16(l >> 4) .. +15 in order, then the two row halves are
        // added (a fixed order); rows past M hold zeros
        const int cp = lane & 15, rh = lane >> 4;
        const uint32_t unit = (uint32_t)(cp >> 2), wb = (uint32_t)(cp & 3) * 4u;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int r = 16 * rh + i;
            const uint32_t u =
                ld_shared_u32(stg + (uint32_t)(r * 64) + ((unit ^ (uint32_t)((r >> 1) & 3)) << 4) + wb);
            s0 += __uint_as_float(u << 16);
            s1 += __uint_as_float(u & 0xffff0000u);
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        if (rh == 0 && row0 < p.M && 2 * cp < nv)
            *reinterpret_cast<float2*>(p.colpart + (size_t)(row0 >> 5) * p.N + col + 2 * cp) =
                make_float2(s0, s1);
    }
}

// ------------------------------------------------------------------- kernel
template <int BN, bool A_MN, bool B_MN, int EPI, int KB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
              const __grid_constant__ EpiMaps maps, TcParams p) {
    using CF = Cfg<BN, KB>;
    constexpr bool PAIR = CF::PAIR;
    constexpr int S = CF::STAGES;
    constexpr uint32_t IDESC = make_idesc(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t tiles = (raw + 1023u) & ~1023u;
    uint8_t* tiles_gen = smem_raw + (tiles - raw);
    const uint32_t stg_base = tiles + S * CF::STAGE_BYTES;  // 1024-aligned
    const uint32_t bars = stg_base + CF::STG_BYTES;
    const uint32_t full = bars, empty = bars + 8 * S, tfull = bars + 16 * S,
                   tempty = tfull + 16;
    uint32_t* tmem_slot = (uint32_t*)(tiles_gen + S * CF::STAGE_BYTES + CF::STG_BYTES + 16 * S + 32);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(tfull + 8 * b, 1);
            mbar_init(tempty + 8 * b, PAIR ? 16 : 8);  // both CTAs' epilogue warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&mapA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&mapB) : "memory");
    }
    if (warp == 1) {
        // a pair allocates together: one warp of each CTA
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(2 * BN)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            tmem_alloc(smem_u32(tmem_slot), 2 * BN);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if (PAIR) pair_sync();  // the peer's barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    gdc_wait();  // setup above touches no global memory
    gdc_launch_dependents();
    // work units: output tiles (times K splits), strided over the CTAs; a pair
    // takes two vertically adjacent 128-row tiles, rank r the rows 128 r ..
    const uint32_t rank = PAIR ? pair_rank() : 0u;
    const bool leader = rank == 0;
    const int units_m = PAIR ? (p.tiles_m + 1) / 2 : p.tiles_m;
    const int units_mn = units_m * p.tiles_n;
    const int num_units = units_mn * p.splits;
    const int unit0 = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
    const int ustep = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- producer
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;  // bit s: stage s has a load in flight or landed
            bool ok = true;
            for (int u = unit0; ok && u < num_units; u += ustep) {
                const int split = u / units_mn, r = u % units_mn;
                const int um = p.n_fastest ? r / p.tiles_n : r % units_m;
                const int tn = p.n_fastest ? r % p.tiles_n : r / units_m;
                const int tm = PAIR ? 2 * um + (int)rank : um;
                const int k0 = split * p.k_per_split;
                const int k1 = min(p.K, k0 + p.k_per_split);
                const int nkb = (k1 - k0 + BK - 1) / BK;
                // a pair CTA loads its own rows of A and its half (of N) of B
                const int bn0 = tn * BN + (PAIR ? (int)rank * (BN / 2) : 0);
                for (int kb2 = 0; kb2 < nkb; kb2 += CF::KB2) {
                    if (!mbar_wait(empty + 8 * s, ph ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const int nh = min(CF::KB2, nkb - kb2);
                    const uint32_t fb = full + 8 * s;
                    if (PAIR) {
                        if (leader) mbar_expect_tx(fb, 2 * nh * CF::HALF_BYTES);
                    } else {
                        mbar_expect_tx(fb, nh * CF::HALF_BYTES);
                    }
                    for (int hh = 0; hh < nh; hh++) {
                        const uint32_t sa = tiles + s * CF::STAGE_BYTES + hh * CF::HALF_BYTES,
                                       sb = sa + CF::A_BYTES;
                        const int kk = k0 + (kb2 + hh) * BK;
                        if (PAIR) {
                            // both CTAs' bytes are counted on the leader's barrier
                            const uint32_t fl = pair_mapa(fb, 0);
                            if (!A_MN) {
                                tma_load_2d_pair(sa, &mapA, fl, kk, tm * BM);
                            } else {
                                tma_load_2d_pair(sa, &mapA, fl, tm * BM, kk);
                                tma_load_2d_pair(sa + 8192, &mapA, fl, tm * BM + 64, kk);
                            }
                            if (!B_MN) {
                                tma_load_2d_pair(sb, &mapB, fl, kk, bn0);
                            } else {
#pragma unroll
                                for (int j = 0; j < BN / 128; j++)
                                    tma_load_2d_pair(sb + j * 8192, &mapB, fl, bn0 + 64 * j, kk);
                            }
                        } else {
                            if (!A_MN) {
                                tma_load_2d(sa, &mapA, fb, kk, tm * BM);
                            } else {
                                tma_load_2d(sa, &mapA, fb, tm * BM, kk);
                                tma_load_2d(sa + 8192, &mapA, fb, tm * BM + 64, kk);
                            }
                            if (!B_MN) {
                                tma_load_2d(sb, &mapB, fb, kk, bn0);
                            } else {
#pragma unroll
                                for (int j = 0; j < BN / 64; j++)
                                    tma_load_2d(sb + j * 8192, &mapB, fb, bn0 + 64 * j, kk);
                            }
                        }
                    }
                    issued |= 1u << s;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // drain: wait (bounded, ignoring the abort flag) for every
                // stage's most recent load so no copy lands after exit (a
                // pair's loads all complete on the leader's barriers; the
                // pair synchronises before either CTA exits)
                for (int i = 0; i < S; i++) {
                    if (!((issued >> i) & 1u)) continue;
                    // the last issue of stage i used parity (ph if i < s else ph^1)
                    uint32_t par = i < s ? ph : ph ^ 1u;
                    long long t0 = clock64();
                    while (!mbar_try(full + 8 * i, par) && clock64() - t0 < WAIT_LIMIT) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // --------------------------------------------------------- MMA
            // (a pair's products are issued by its leader: M = 256, each CTA's
            // TMEM receiving its 128 rows)
            int s = 0;
            uint32_t ph = 0;
            int lt = 0;
            bool ok = true;
            // stage-0 descriptors; stages and K steps add start-address offsets
            const uint64_t dA0 = A_MN ? sdesc(tiles, 8192, 1024) : sdesc(tiles, 0, 1024);
            const uint64_t dB0 = B_MN ? sdesc(tiles + CF::A_BYTES, 8192, 1024)
                                      : sdesc(tiles + CF::A_BYTES, 0, 1024);
            for (int u = unit0; ok && u < num_units; u += ustep, lt++) {
                const int split = u / units_mn;
                const int k0 = split * p.k_per_split;
                const int k1 = min(p.K, k0 + p.k_per_split);
                const int nkb = (k1 - k0 + BK - 1) / BK;
                const int b = lt & 1;
                const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
                if (!mbar_wait(tempty + 8 * b, aph ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(b * BN);
                for (int kb2 = 0; kb2 < nkb; kb2 += CF::KB2) {
                    if (!mbar_wait(full + 8 * s, ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nh = min(CF::KB2, nkb - kb2);
                    for (int hh = 0; hh < nh; hh++) {
                        const int kb = kb2 + hh;
                        const uint64_t ad0 =
                            dA0 + (uint64_t)((s * CF::STAGE_BYTES + hh * CF::HALF_BYTES) >> 4);
                        const uint64_t bd0 =
                            dB0 + (uint64_t)((s * CF::STAGE_BYTES + hh * CF::HALF_BYTES) >> 4);
#pragma unroll
                        for (int k = 0; k < BK / 16; k++) {
                            if (PAIR)
                                umma_bf16_pair(dt, ad0 + (uint64_t)(k * (A_MN ? 128 : 2)),
                                               bd0 + (uint64_t)(k * (B_MN ? 128 : 2)), IDESC,
                                               (kb > 0 || k > 0) ? 1u : 0u);
                            else
                                umma_bf16(dt, ad0 + (uint64_t)(k * (A_MN ? 128 : 2)),
                                          bd0 + (uint64_t)(k * (B_MN ? 128 : 2)), IDESC,
                                          (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    if (PAIR) {  // the stage is free in both CTAs
                        umma_commit_pair(pair_mapa(empty + 8 * s, 0));
                        umma_commit_pair(pair_mapa(empty + 8 * s, 1));
                    } else {
                        umma_commit(empty + 8 * s);
                    }
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if (PAIR) {  // the accumulator is ready in both CTAs
                    umma_commit_pair(pair_mapa(tfull + 8 * b, 0));
                    umma_commit_pair(pair_mapa(tfull + 8 * b, 1));
                } else {
                    umma_commit(tfull + 8 * b);
                }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        // warps 2..9: TMEM lane quarter (warp % 4) x column half
        const int q = warp & 3;
        const int cbeg = ((warp - 2) >> 2) * (BN / 2);
        constexpr int NCH = BN / 64;  // 32-column chunks per half
        const uint32_t stg = stg_base + (uint32_t)(warp - 2) * 4096u;
        const bool has_pf = EPI == EPI_RESID || EPI == EPI_GELU_BWD || EPI == EPI_MUL_AUX;
        int lt = 0;
        for (int u = unit0; u < num_units; u += ustep, lt++) {
            const int split = u / units_mn, r = u % units_mn;
            const int um = p.n_fastest ? r / p.tiles_n : r % units_m;
            const int tn = p.n_fastest ? r % p.tiles_n : r / units_m;
            const int tm = PAIR ? 2 * um + (int)rank : um;
            const int b = lt & 1;
            const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
            const int row = tm * BM + q * 32 + lane;
            uint4 pf[2][4];
            // the first chunk's row operand does not depend on the accumulator:
            // fetch it before waiting for the tile
            if (has_pf) epi_prefetch<EPI>(p, row, tn * BN + cbeg, pf[0]);
            // every lane waits (suspended in the barrier's try_wait until the
            // phase completes); the warp goes on only if all saw it complete
            const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull + 8 * b, aph, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + cbeg);
            uint32_t buf[2][32];
            tmem_ld32_async(taddr, buf[0]);
            tmem_wait32(buf[0]);
#pragma unroll
            for (int c = 0; c < NCH; c++) {
                if (c + 1 < NCH) {
                    tmem_ld32_async(taddr + (uint32_t)(32 * (c + 1)), buf[(c + 1) & 1]);
                    if (has_pf) epi_prefetch<EPI>(p, row, tn * BN + cbeg + 32 * (c + 1), pf[(c + 1) & 1]);
                }
                const int col = tn * BN + cbeg + 32 * c;
                if (col < p.N) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(buf[c & 1][i]);
                    epilogue_chunk<EPI>(p, maps, tm * BM + q * 32, col, lane, v, split, stg, pf[c & 1]);
                }
                if (c + 1 < NCH) tmem_wait32(buf[(c + 1) & 1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {  // the accumulator buffer is free (on the leader's barrier)
                if (PAIR && !leader) mbar_arrive_cluster(pair_mapa(tempty + 8 * b, 0));
                else mbar_arrive(tempty + 8 * b);
            }
        }
        if (lane == 0) bulk_wait0();  // all bulk stores of this warp complete
        __syncwarp();
    }
    __syncthreads();
    // a pair: no signal of either CTA may target a CTA that has exited, and
    // the pair deallocates its TMEM together
    if (PAIR) pair_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(2 * BN)
                         : "memory");
        else
            tmem_dealloc(tmem_base, 2 * BN);
    }
}


// ----------------------------------------------------------------- launchers
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// shared state and tensor-map helpers (defined in k_gemm_tc.cu)
extern int g_num_sms;
bool make_map(CUtensorMap* m, const void* base, long inner, long outer, long ld, int box_outer);
bool make_epi_maps(EpiMaps* em, const GemmDesc& d, const TcParams& tp);

template <int BN, bool AM, bool BMN, int EPI, int KB>
cudaError_t launch_one(const GemmDesc& d, const TcParams& tp, cudaStream_t s) {
    static bool attr = false;  // the dynamic shared-memory size, set once per kernel
    if (!attr) {
        if (cudaFuncSetAttribute(k_gemm_tc<BN, AM, BMN, EPI, KB>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BN, KB>::SMEM) != cudaSuccess)
            return cudaGetLastError();
        attr = true;
    }
    CUtensorMap ma, mb;
    EpiMaps em;
    if (!make_epi_maps(&em, d, tp)) return cudaErrorInvalidValue;
    // A: K-major -> [M rows][K], box 64(K) x 128(M);  MN-major -> [K rows][M], box 64(M) x 64(K)
    bool ok = AM ? make_map(&ma, d.A, d.M, d.K, d.lda, 64)
                 : make_map(&ma, d.A, d.K, d.M, d.lda, BM);
    // B: K-major box 64(K) x BN rows (a pair CTA: its BN/2);  N-major box 64(N) x 64(K)
    constexpr bool PAIR = Cfg<BN, KB>::PAIR;
    ok = ok && (BMN ? make_map(&mb, d.B, d.N, d.K, d.ldb, 64)
                    : make_map(&mb, d.B, d.K, d.N, d.ldb, PAIR ? BN / 2 : BN));
    if (!ok) return cudaErrorInvalidValue;
    if (!PAIR) {
        const int grid = tp.num_tiles < g_num_sms ? tp.num_tiles : g_num_sms;
        launch_pdl(k_gemm_tc<BN, AM, BMN, EPI, KB>, grid, NUM_THREADS, Cfg<BN, KB>::SMEM, s, ma, mb, em, tp);
        return cudaGetLastError();
    }
    // CTA pairs: clusters of 2, as many as can be resident at once
    static int resident = 0;
    if (resident == 0) {
        cudaLaunchConfig_t oc;
        memset(&oc, 0, sizeof oc);
        oc.gridDim = dim3(g_num_sms);
        oc.blockDim = dim3(NUM_THREADS);
        oc.dynamicSmemBytes = Cfg<BN, KB>::SMEM;
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeClusterDimension;
        ca[0].val.clusterDim.x = 2;
        ca[0].val.clusterDim.y = 1;
        ca[0].val.clusterDim.z = 1;
        oc.attrs = ca;
        oc.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<BN, AM, BMN, EPI, KB>, &oc) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = g_num_sms / 2;
        }
        resident = n < g_num_sms / 2 ? n : g_num_sms / 2;
    }
    const int units = ((tp.tiles_m + 1) / 2) * tp.tiles_n * tp.splits;
    int pairs = resident;
    if (units < pairs) pairs = units;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Cfg<BN, KB>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute la[2];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 2;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    la[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, AM, BMN, EPI, KB>, ma, mb, em, tp);
}

// the launch for epilogue mode EPI, tile width bn and operand layouts am, bm
// modes whose 256-wide products take two k-blocks per stage when K is long
// (measured: 2-6% faster there; the multiply-by-aux epilogue and the split
// partials were not)
constexpr bool kb2_mode(int epi) {
    return epi == EPI_STORE || epi == EPI_RESID || epi == EPI_GELU || epi == EPI_GELU_D ||
           epi == EPI_ACCUM_F32;
}
template <int EPI>
cudaError_t launch_epi(int bn, bool am, bool bm, bool kb2, const GemmDesc& d, const TcParams& tp,
                       cudaStream_t s) {
    if (bn == 256) {
        if constexpr (kb2_mode(EPI)) {
            if (kb2) {
                if (!am && !bm) return launch_one<256, false, false, EPI, 2>(d, tp, s);
                if (!am && bm) return launch_one<256, false, true, EPI, 2>(d, tp, s);
                if (am && !bm) return launch_one<256, true, false, EPI, 2>(d, tp, s);
                return launch_one<256, true, true, EPI, 2>(d, tp, s);
            }
        }
        if (!am && !bm) return launch_one<256, false, false, EPI, 1>(d, tp, s);
        if (!am && bm) return launch_one<256, false, true, EPI, 1>(d, tp, s);
        if (am && !bm) return launch_one<256, true, false, EPI, 1>(d, tp, s);
        return launch_one<256, true, true, EPI, 1>(d, tp, s);
    }
    if (!am && !bm) return launch_one<128, false, false, EPI, 1>(d, tp, s);
    if (!am && bm) return launch_one<128, false, true, EPI, 1>(d, tp, s);
    if (am && !bm) return launch_one<128, true, false, EPI, 1>(d, tp, s);
    return launch_one<128, true, true, EPI, 1>(d, tp, s);
}

#define GK_GEMM_EPI_EXTERN(E)                                                                 \
    extern template cudaError_t launch_epi<E>(int, bool, bool, bool, const GemmDesc&,              \
                                              const TcParams&, cudaStream_t);
#define GK_GEMM_EPI_INSTANTIATE(E)                                                          \
    template cudaError_t launch_epi<E>(int, bool, bool, bool, const GemmDesc&, const TcParams&, \
                                       cudaStream_t);

}  // namespace tcg
}  // namespace gk
