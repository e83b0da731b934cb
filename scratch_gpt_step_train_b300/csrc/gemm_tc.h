// gemm_tc.h -- tensor-core (tcgen05 / TMEM / TMA) matmul for bf16 operands.
#pragma once
#include "kernels.h"

namespace gk {
// true if this process can run the tcgen05 path (device is sm_103 and the
// driver entry point for tensor-map encoding was found)
bool gemm_tc_available();
// true if this descriptor's shape, strides and alignment fit the kernel
bool gemm_tc_supported(const GemmDesc& d);
cudaError_t gemm_tc(const GemmDesc& d, cudaStream_t s);
}  // namespace gk
