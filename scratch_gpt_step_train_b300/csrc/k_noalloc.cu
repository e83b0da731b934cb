// k_noalloc.cu -- LayerNorm backward for callers that cannot allocate device
// memory.
//
// gpt2k_layernorm_backward needs caller-provided scratch for its per-block
// partial dgamma/dbeta sums.  Some callers cannot make that allocation: their
// device memory is owned by another allocator that hands them only the
// operation's own tensors, or they run in a loop that must never call
// cudaMalloc/cudaFree (each may synchronise the device).  This file gives them
// one entry point that allocates nothing: the scratch is a fixed array in
// device global memory, reserved when the library's module is loaded on a
// device and kept until the process exits.
#include <mutex>

#include "../../include/gpt2.h"
#include "../../include/gpt2_kernels.h"
#include "kernels.h"

namespace {

// Largest row width the array serves, and its size: one row of C partial
// dgamma and one of C partial dbeta per block, for the kernel's maximum block
// count (296) -- 296 * 2 * 2048 * 4 bytes = 4.6 MiB per device.
constexpr int kMaxC = 2048;
constexpr size_t kScratchBytes = (size_t)296 * 2 * kMaxC * sizeof(float);
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address is taken per device with
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ln_bwd_scratch[kScratchBytes];

static std::mutex g_mu;
static void* g_addr[kMaxDevices];

// Device address of the array on the current device (set up once per device,
// with that device current).  NULL if the symbol cannot be resolved.
static void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ln_bwd_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

extern "C" int gpt2k_layernorm_backward_noalloc(int dtype, void* dx, float* dw, float* db,
                                                const void* dout, const void* x, const void* w,
                                                const float* mean, const float* rstd, int N,
                                                int C, void* stream) {
    if ((dtype != gk::ACT_F32 && dtype != gk::ACT_BF16) || N < 1 || C < 1) return GPT2_ERR_ARG;
    if (C > kMaxC || gk::layernorm_backward_scratch(N, C, false) > kScratchBytes)
        return GPT2_ERR_ARG;  // wider than the fixed scratch serves
    void* scratch = scratch_on_current_device();
    if (!scratch) return GPT2_ERR_CUDA;
    // every block overwrites its own partial rows before they are summed, so
    // nothing left in the array by an earlier call needs clearing
    cudaError_t e = gk::layernorm_backward(dtype, dx, dw, db, nullptr, dout, x, w, mean, rstd, N,
                                           C, true, scratch, (cudaStream_t)stream);
    if (e == cudaSuccess) return GPT2_OK;
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? GPT2_ERR_ARG : GPT2_ERR_CUDA;
}
