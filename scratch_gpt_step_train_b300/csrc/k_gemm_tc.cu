// k_gemm_tc.cu -- placeholder until the tcgen05 kernel lands.
#include "gemm_tc.h"
namespace gk {
bool gemm_tc_available() { return false; }
bool gemm_tc_supported(const GemmDesc&) { return false; }
cudaError_t gemm_tc(const GemmDesc&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gk
