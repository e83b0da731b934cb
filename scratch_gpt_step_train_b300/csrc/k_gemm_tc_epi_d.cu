// k_gemm_tc_epi_d.cu -- the tensor-core matmul kernels of two epilogue modes
// (EPI_ACCUM_F32, EPI_PART_F32): every tile width and operand layout of each (the kernel
// template and its launchers are in gemm_tc_kernel.cuh).
#include "gemm_tc_kernel.cuh"

namespace gk {
namespace tcg {
GK_GEMM_EPI_INSTANTIATE(EPI_ACCUM_F32)
GK_GEMM_EPI_INSTANTIATE(EPI_PART_F32)
}  // namespace tcg
}  // namespace gk
