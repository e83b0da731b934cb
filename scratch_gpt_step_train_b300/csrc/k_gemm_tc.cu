// k_gemm_tc.cu -- bf16 x bf16 -> fp32 matmul on the 5th-generation tensor cores
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
#include "gemm_tc_kernel.cuh"

namespace gk {
namespace tcg {

GK_GEMM_EPI_EXTERN(EPI_STORE)
GK_GEMM_EPI_EXTERN(EPI_RESID)
GK_GEMM_EPI_EXTERN(EPI_GELU)
GK_GEMM_EPI_EXTERN(EPI_GELU_D)
GK_GEMM_EPI_EXTERN(EPI_GELU_BWD)
GK_GEMM_EPI_EXTERN(EPI_MUL_AUX)
GK_GEMM_EPI_EXTERN(EPI_ACCUM_F32)
GK_GEMM_EPI_EXTERN(EPI_PART_F32)

// split-K: D[m,n] += sum_s part[s][m][n], s in order
__global__ void k_splitk_reduce(float* D, long ldd, const float* part, int M, int N, int splits) {
    gdc_wait();
    gdc_launch_dependents();
    long idx = blockIdx.x * (long)blockDim.x + threadIdx.x;
    long nv = (long)M * (N / 4);
    if (idx >= nv) return;
    int m = (int)(idx / (N / 4)), n = (int)(idx % (N / 4)) * 4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; s++) {
        float4 x = *reinterpret_cast<const float4*>(part + ((size_t)s * M + m) * N + n);
        a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    }
    float4* d = reinterpret_cast<float4*>(D + (size_t)m * ldd + n);
    float4 o = *d;
    o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
    *d = o;
}


// ----------------------------------------------------------------- host side
EncodeTiledFn g_encode = nullptr;
int g_num_sms = 148;
int g_state = -1;  // -1 unknown, 0 unavailable, 1 ready


// 2-D bf16 tensor map: inner extent `inner` (contiguous), `outer` rows of
// `ld` elements; box = 64 x box_outer; 128-byte swizzle; OOB reads give 0.
bool make_map(CUtensorMap* m, const void* base, long inner, long outer, long ld, int box_outer) {
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_epi(CUtensorMap* m, void* base, CUtensorMapDataType dt, int esz, int rank,
                  const cuuint64_t* dims, const cuuint64_t* strides_bytes) {
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, rank, base, dims, strides_bytes, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          esz == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_epi_maps(EpiMaps* em, const GemmDesc& d, const TcParams& tp) {
    memset(em, 0, sizeof(*em));
    bool ok = true;
    if (tp.epi == EPI_ACCUM_F32) {
        cuuint64_t dims[2] = {(cuuint64_t)d.N, (cuuint64_t)d.M};
        cuuint64_t st[1] = {(cuuint64_t)d.ldd * 4};
        ok = make_map_epi(&em->d, d.D, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, dims, st);
    } else if (tp.epi == EPI_PART_F32) {
        cuuint64_t dims[3] = {(cuuint64_t)d.N, (cuuint64_t)d.M, (cuuint64_t)tp.splits};
        cuuint64_t st[2] = {(cuuint64_t)d.N * 4, (cuuint64_t)d.N * d.M * 4};
        ok = make_map_epi(&em->part, tp.part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, dims, st);
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)d.N, (cuuint64_t)d.M};
        cuuint64_t st[1] = {(cuuint64_t)d.ldd * 2};
        ok = make_map_epi(&em->d, d.D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, dims, st);
        if (ok && (tp.epi == EPI_GELU || tp.epi == EPI_GELU_D)) {
            cuuint64_t sx[1] = {(cuuint64_t)d.ldx * 2};
            ok = make_map_epi(&em->aux, d.aux, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, dims, sx);
        }
    }
    return ok;
}



}  // namespace tcg

using namespace tcg;

bool gemm_tc_available() {
    if (g_state >= 0) return g_state == 1;
    g_state = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return false;
    if (prop.major != 10 || prop.minor != 3) return false;
    g_num_sms = prop.multiProcessorCount;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return false;
    }
    g_encode = (EncodeTiledFn)fn;
    if (cudaGetLastError() != cudaSuccess) return false;
    g_state = 1;
    return true;
}

int gemm_tc_binary_version() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, k_splitk_reduce) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return a.binaryVersion;
}

void* tc_encode_fn() { return gemm_tc_available() ? (void*)g_encode : nullptr; }

static bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

bool gemm_tc_supported(const GemmDesc& d) {
    if (d.act != ACT_BF16 || d.M < 1 || d.N < 1 || d.K < 1) return false;
    if (d.N % 8) return false;
    if (!al16(d.A) || !al16(d.B) || !al16(d.D)) return false;
    if ((d.lda % 8) || (d.ldb % 8) || (d.ldd % 8)) return false;
    if (d.a_kmajor ? d.lda < d.K : d.lda < d.M) return false;
    if (d.b_kmajor ? d.ldb < d.K : d.ldb < d.N) return false;
    if (d.epi == EPI_RESID && (!d.resid || !al16(d.resid) || d.ldr % 8)) return false;
    if ((d.epi == EPI_GELU || d.epi == EPI_GELU_BWD || d.epi == EPI_GELU_D ||
         d.epi == EPI_MUL_AUX) &&
        (!d.aux || !al16(d.aux) || d.ldx % 8))
        return false;
    if (d.bias && !al16(d.bias)) return false;
    return true;
}

size_t gemm_tc_scratch_bytes() { return (size_t)64 << 20; }

cudaError_t gemm_tc(const GemmDesc& d, void* scratch, size_t scratch_bytes, unsigned* err,
                    cudaStream_t s, int* nlaunch) {
    if (nlaunch) *nlaunch = 0;
    if (!gemm_tc_available()) return cudaErrorNotSupported;
    if (!gemm_tc_supported(d)) return cudaErrorInvalidValue;
    const int tiles_m = (d.M + BM - 1) / BM;
    // 128 x 256 tiles halve the operand traffic per flop against 128 x 128
    const bool can_split = d.epi == EPI_ACCUM_F32 && d.K >= 8 * BK && scratch;
    const int kb = (d.K + BK - 1) / BK;
    int BN = 256, splits = 1;
    if (can_split) {
        // Weight-gradient products (long K, few output tiles): pick the tile
        // width and the K split from a time model -- whole waves of work units
        // over the SMs, each unit's k-blocks at the tile width's rate, plus the
        // fp32 traffic of the output (read-modify-write) and of the split's
        // partial sums (written, then read back by the ordered reduction).
        // The k-block rates are measured ones (128 x 256 and 128 x 128 tiles,
        // each CTA loading its whole A and B tiles).
        const double kblock_us[2] = {0.30, 0.31};  // 128x256 / 128x128
        const double bytes_per_us = 5.0e6;
        const double mn4 = 4.0 * d.M * d.N;
        double best = 1e30;
        for (int w = 0; w < 2; w++) {
            const int bn = w ? 128 : 256;
            const long t = (long)tiles_m * ((d.N + bn - 1) / bn);
            for (int sp = 1; sp <= 16 && (sp == 1 || sp <= kb / 4); sp++) {
                if (sp > 1 && (size_t)sp * d.M * d.N * 4 > scratch_bytes) break;
                const int kbs = (kb + sp - 1) / sp, sps = (kb + kbs - 1) / kbs;
                if (sp > 1 && sps != sp) continue;
                const long waves = (t * sps + g_num_sms - 1) / g_num_sms;
                const double us = waves * kbs * kblock_us[w] +
                                  (sps > 1 ? 2.0 * sps + 2.0 : 2.0) * mn4 / bytes_per_us;
                if (us < best - 1e-9) {
                    best = us;
                    BN = bn;
                    splits = sps;
                }
            }
        }
    } else if (d.N <= 128 || (long)tiles_m * ((d.N + 255) / 256) < g_num_sms) {
        // narrow outputs, and products with too few 128 x 256 tiles
        BN = 128;
    }
    const int tiles_n = (d.N + BN - 1) / BN;
    TcParams tp;
    tp.M = d.M; tp.N = d.N; tp.K = d.K;
    tp.tiles_m = tiles_m;
    tp.tiles_n = tiles_n;
    tp.splits = 1;
    tp.k_per_split = ((d.K + BK - 1) / BK) * BK;
    // the larger operand is streamed once when the tiles that share it run
    // side by side: output-column tiles fastest when A (M x K) is the larger
    tp.n_fastest = d.M > d.N ? 1 : 0;
    tp.epi = d.epi;
    tp.D = d.D; tp.ldd = d.ldd;
    tp.bias = (const bf16*)d.bias;
    tp.resid = (const bf16*)d.resid; tp.ldr = d.ldr;
    tp.aux = (bf16*)d.aux; tp.ldx = d.ldx;
    tp.part = (float*)scratch;
    tp.colpart = nullptr;
    tp.err = err;
    const int row_blocks = (d.M + 31) / 32;
    if (d.dbias || d.colpart) {
        // column partial sums (in scratch, then one ordered sum into dbias;
        // or in the caller's region, summed later)
        if (d.epi != EPI_MUL_AUX && d.epi != EPI_GELU_BWD) return cudaErrorInvalidValue;
        if (d.dbias && (!scratch || (size_t)row_blocks * d.N * 4 > scratch_bytes))
            return cudaErrorInvalidValue;
        tp.colpart = d.dbias ? (float*)scratch : d.colpart;
    }
    const long tiles = (long)tiles_m * tiles_n;
    if (splits > 1) {
        const int kbs = (kb + splits - 1) / splits;
        tp.k_per_split = kbs * BK;
        tp.splits = (kb + kbs - 1) / kbs;
        tp.epi = EPI_PART_F32;
    }
    tp.num_tiles = (int)(tiles * tp.splits);
    const bool am = !d.a_kmajor, bm = !d.b_kmajor;
    // two k-blocks per pipeline stage for the long-K products, and for the
    // GELU forward already at K = 768 (measured: -2.5% there, +1% for the
    // other K = 768 modes)
    const bool kb2 = tp.splits == 1 && (d.K >= 1536 || (d.epi == EPI_GELU_D && d.K >= 512));
    cudaError_t e;
    switch (tp.epi) {  // one kernel per epilogue mode
        case EPI_STORE: e = launch_epi<EPI_STORE>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_RESID: e = launch_epi<EPI_RESID>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_GELU: e = launch_epi<EPI_GELU>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_GELU_D: e = launch_epi<EPI_GELU_D>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_GELU_BWD: e = launch_epi<EPI_GELU_BWD>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_MUL_AUX: e = launch_epi<EPI_MUL_AUX>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_ACCUM_F32: e = launch_epi<EPI_ACCUM_F32>(BN, am, bm, kb2, d, tp, s); break;
        case EPI_PART_F32: e = launch_epi<EPI_PART_F32>(BN, am, bm, kb2, d, tp, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if (nlaunch) *nlaunch = 1;
    if (d.dbias) {
        if (nlaunch) *nlaunch = 2;
        return colsum_add(d.dbias, tp.colpart, row_blocks, d.N, s);
    }
    if (tp.splits > 1) {
        if (nlaunch) *nlaunch = 2;
        long nv = (long)d.M * (d.N / 4);
        launch_pdl(k_splitk_reduce, (int)((nv + 255) / 256), 256, 0, s, (float*)d.D, d.ldd, tp.part, d.M,
                                                                d.N, tp.splits);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace gk
