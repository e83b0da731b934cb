// k_gemm_tc_epi_a.cu -- the tensor-core matmul kernels of two epilogue modes
// (EPI_STORE, EPI_RESID): every tile width and operand layout of each (the kernel
// template and its launchers are in gemm_tc_kernel.cuh).
#include "gemm_tc_kernel.cuh"

namespace gk {
namespace tcg {
GK_GEMM_EPI_INSTANTIATE(EPI_STORE)
GK_GEMM_EPI_INSTANTIATE(EPI_RESID)
}  // namespace tcg
}  // namespace gk
