// k_gemm_tc_epi_c.cu -- the tensor-core matmul kernels of two epilogue modes
// (EPI_GELU_BWD, EPI_MUL_AUX): every tile width and operand layout of each (the kernel
// template and its launchers are in gemm_tc_kernel.cuh).
#include "gemm_tc_kernel.cuh"

namespace gk {
namespace tcg {
GK_GEMM_EPI_INSTANTIATE(EPI_GELU_BWD)
GK_GEMM_EPI_INSTANTIATE(EPI_MUL_AUX)
}  // namespace tcg
}  // namespace gk
