// ttt_no_alloc.cu -- ttt_linear_bwd_static: the TTT-Linear backward pass on the library's
// own static device scratch instead of a caller-provided workspace.
//
// The scratch is a file-scope __device__ array in this translation unit (its own module):
// no cudaMalloc, cudaFree or allocating library routine is involved.  The first call on a
// device, with that device current, resolves the array's device address with
// cudaGetSymbolAddress (which may load this module) and caches it per device; later calls
// reuse it.  Nothing in the scratch has to start at zero: the backward kernels write every
// byte they read (state checkpoints, per-row partial gradients) earlier in the same call.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "ttt_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::atomic<void *> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device (resolved once per device).
cudaError_t scratch_on_current_device(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t ttt_linear_bwd_static_scratch_bytes(void) { return kScratchBytes; }

ttt_status ttt_linear_bwd_static(const ttt_desc *desc, const void *Q, const void *K, const void *V,
                                 const float *eta, const float *W0, const float *b0, const float *gamma,
                                 const float *beta, const void *dZ, const float *dW_final,
                                 const float *db_final, void *dQ, void *dK, void *dV, float *deta,
                                 float *dW0, float *db0, float *dgamma, float *dbeta, ttt_stream_t stream)
{
    const size_t need = ttt_linear_bwd_workspace_size(desc);
    if (need > kScratchBytes) {
        // a valid, supported call that needs more than the static scratch holds
        return ttt::fail_static_scratch(need, kScratchBytes);
    }
    void *scratch = nullptr;
    if (need > 0) {
        cudaError_t e = scratch_on_current_device(&scratch);
        if (e != cudaSuccess) return ttt::fail_cuda("static scratch address", e);
    }
    // need == 0 (invalid or unsupported descriptor): ttt_linear_bwd reports the reason
    return ttt_linear_bwd(desc, Q, K, V, eta, W0, b0, gamma, beta, dZ, dW_final, db_final, dQ, dK, dV,
                          deta, dW0, db0, dgamma, dbeta, scratch, kScratchBytes, stream);
}

}  // extern "C"
