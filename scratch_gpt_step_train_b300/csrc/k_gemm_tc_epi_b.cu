// k_gemm_tc_epi_b.cu -- the tensor-core matmul kernels of two epilogue modes
// (EPI_GELU, EPI_GELU_D): every tile width and operand layout of each (the kernel
// template and its launchers are in gemm_tc_kernel.cuh).
#include "gemm_tc_kernel.cuh"

namespace gk {
namespace tcg {
GK_GEMM_EPI_INSTANTIATE(EPI_GELU)
GK_GEMM_EPI_INSTANTIATE(EPI_GELU_D)
}  // namespace tcg
}  // namespace gk
