// gemm_tc.h -- tensor-core (tcgen05 / TMEM / TMA) matmul for bf16 operands.
#pragma once
#include "kernels.h"

namespace gk {
// true if this process can run the tcgen05 path (device is sm_103 and the
// driver entry point for tensor-map encoding was found)
bool gemm_tc_available();
// true if this descriptor's shape, strides and alignment fit the kernel:
// bf16, N % 8 == 0, 16-byte aligned bases, leading dimensions % 8 == 0
bool gemm_tc_supported(const GemmDesc& d);
// binaryVersion of the loaded tensor-core GEMM kernel (major*10+minor), or -1
int gemm_tc_binary_version();
// bytes of scratch the split-K weight-gradient products may use
size_t gemm_tc_scratch_bytes();
// D = epilogue(A . B^T).  scratch: split-K partials (may be NULL: no split);
// err: device error word (timeouts); *nlaunch: kernels launched (1 or 2).
cudaError_t gemm_tc(const GemmDesc& d, void* scratch, size_t scratch_bytes, unsigned* err,
                    cudaStream_t s, int* nlaunch);
}  // namespace gk
