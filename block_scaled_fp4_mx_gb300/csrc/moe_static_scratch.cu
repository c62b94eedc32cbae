// moe_static_scratch.cu -- a fixed device scratch area for the MoE layer, so that a
// caller without an allocator (or one that must not allocate on the hot path) can
// run it: a static __device__ array in its own translation unit (its own module).
// Nothing here calls cudaMalloc.
//
// The array's device address belongs to the module as loaded in the current
// context. It is looked up again on every call (cudaGetSymbolAddress is a host
// lookup once the module is loaded), so a context that was destroyed and created
// again (cudaDeviceReset, a new primary context) hands out the address in the new
// context, never a stale one from the old.
#include <cuda_runtime.h>

#include "launch.h"

namespace fp4mx {
namespace {

constexpr uint64_t kScratchBytes = 288ull << 20;  // the 4096-token top-4 2880 x 2880 layer fits
__device__ __align__(256) uint8_t g_moe_scratch[kScratchBytes];

}  // namespace

uint64_t moe_static_scratch_bytes() { return kScratchBytes; }

cudaError_t moe_static_scratch(void **address) {
    void *ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_moe_scratch);
    if (err != cudaSuccess) return err;
    *address = ptr;
    return cudaSuccess;
}

}  // namespace fp4mx
