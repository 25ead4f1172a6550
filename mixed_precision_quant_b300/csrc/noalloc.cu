// noalloc.cu -- the fixed scratch area of fp8_grouped_gemm_fused_quant_noalloc.
//
// The allocation-free form of the fused grouped GEMM keeps the quantized activations in a
// file-scope device array instead of a caller-provided workspace, so a call needs no
// memory from anyone.  The array's address is looked up once per device, with that device
// current, on the first call (cudaGetSymbolAddress); later calls reuse it.
#include <mutex>

#include "mpq_internal.h"

namespace mpq {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];   // per device, filled on first use
std::mutex g_scratch_mu;

} // namespace

cudaError_t noalloc_scratch(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

} // namespace mpq
