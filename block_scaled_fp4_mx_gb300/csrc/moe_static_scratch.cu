// moe_static_scratch.cu -- a fixed device scratch area for the MoE layer, so that a
// caller without an allocator (or one that must not allocate on the hot path) can
// run it: a static __device__ array in its own translation unit (its own module,
// loaded the first time it is used), whose address is looked up once per device.
// Nothing here calls cudaMalloc.
#include <mutex>

#include <cuda_runtime.h>

#include "launch.h"

namespace fp4mx {
namespace {

constexpr uint64_t kScratchBytes = 288ull << 20;  // the 4096-token top-4 2880 x 2880 layer fits
__device__ __align__(256) uint8_t g_moe_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_address[kMaxDevices] = {};

}  // namespace

uint64_t moe_static_scratch_bytes() { return kScratchBytes; }

cudaError_t moe_static_scratch(void **address) {
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_address[device] == nullptr) {
        err = cudaGetSymbolAddress(&g_address[device], g_moe_scratch);
        if (err != cudaSuccess) {
            g_address[device] = nullptr;
            return err;
        }
    }
    *address = g_address[device];
    return cudaSuccess;
}

}  // namespace fp4mx
