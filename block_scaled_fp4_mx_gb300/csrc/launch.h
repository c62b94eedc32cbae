// launch.h -- internal kernel launchers behind the C ABI (not exported).
// Arguments reaching these have been validated by api.cu: sizes are positive,
// pointers are device-accessible and outputs do not overlap inputs.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace fp4mx {

// Launch `kernel`; with `after_kernel` it may start while the kernel before it in the
// stream is still finishing (programmatic dependent launch): it must then wait
// (grid_dependency_wait) before it touches anything that kernel writes or reads.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool after_kernel, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_kernel ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// In a kernel launched with after_kernel: returns once the kernel before it in the
// stream has completed and its memory operations are visible (at once otherwise).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Decode n_elems (a positive multiple of 32) MXFP4 codes.
cudaError_t launch_mx_unpack(const uint8_t *packed, const uint8_t *scales, uint16_t *out,
                             int64_t n_elems, cudaStream_t stream);

// Gather-dequant num_ids (> 0) rows of `hidden` (a positive multiple of 16) codes.
cudaError_t launch_nv_gather(const int64_t *ids, int64_t num_ids, const uint8_t *weight,
                             const uint8_t *scales, const float *global_scale, int64_t vocab,
                             int64_t hidden, uint16_t *out, int32_t *err_flag,
                             cudaStream_t stream);

// Dequantise every row of a [rows, hidden] NVFP4 table (rows > 0).
cudaError_t launch_nv_dequant(const uint8_t *weight, const uint8_t *scales,
                              const float *global_scale, int64_t rows, int64_t hidden,
                              uint16_t *out, cudaStream_t stream);

// Quantise n_elems (a positive multiple of 32) bf16 values to MXFP4.
cudaError_t launch_mx_quantize(const uint16_t *in, uint8_t *packed, uint8_t *scales,
                               int64_t n_elems, cudaStream_t stream);

// Grouped MoE GEMM with MXFP4 weights decoded into the tensor-core A operand in
// tensor memory (any shape the entry point accepts; 16-byte aligned weights).
// With after_kernel (inside the MoE layer) it may start while the kernel before it
// finishes: only its activation loads wait for that kernel, so the activations must
// be that kernel's output or older, and everything else it reads must be older.
cudaError_t launch_mx_moe_gemm(const uint16_t *a, const int64_t *expert_offsets, int64_t experts,
                               int64_t max_rows, int64_t total_rows, const uint8_t *w_packed,
                               const uint8_t *w_scales, int64_t n, int64_t k, uint16_t *out,
                               int32_t *status, cudaStream_t stream, bool after_kernel = false);

// The MoE layer's gate/up GEMM: x [total_rows, k] against w1 [experts, 2n, k/2]
// (gate rows 0..n-1, up rows n..2n-1 of each expert) -> act [total_rows, n] =
// bf16(silu(gate) * up).
cudaError_t launch_mx_moe_gate_up(const uint16_t *x, const int64_t *expert_offsets, int64_t experts,
                                  int64_t max_rows, int64_t total_rows, const uint8_t *w1_packed,
                                  const uint8_t *w1_scales, int64_t n, int64_t k, uint16_t *act,
                                  int32_t *status, cudaStream_t stream, bool after_kernel = false);

// The MoE layer: routing, gate/up GEMM with silu(gate) * up, down GEMM, top-k
// weighted sum. Byte offsets of its scratch arrays in the caller's workspace.
struct MoeWorkspace {
    uint64_t counts, ticket, cursors, offsets, pos, xg, act, y, total;
};
MoeWorkspace moe_workspace_layout(int64_t tokens, int64_t topk, int64_t experts, int64_t n,
                                  int64_t k);
cudaError_t launch_mx_moe_forward(const uint16_t *a, const int32_t *topk_ids,
                                  const float *topk_weights, int64_t tokens, int64_t topk,
                                  int64_t experts, int64_t max_rows, const uint8_t *w1_packed,
                                  const uint8_t *w1_scales, const uint8_t *w2_packed,
                                  const uint8_t *w2_scales, int64_t n, int64_t k, void *workspace,
                                  uint16_t *out, int32_t *status, cudaStream_t stream);

// The MoE layer's static device scratch (fp4_mx_moe_forward_noalloc): its size,
// and its address in the current context (looked up on every call).
uint64_t moe_static_scratch_bytes();
cudaError_t moe_static_scratch(void **address);

// Bounded-wait check (wait_selftest.cu): mode 0 spinning wait, 1 sleeping wait,
// 2 a wait whose phase completes.
cudaError_t launch_wait_selftest(int32_t mode, int32_t *status, cudaStream_t stream);

// Paged MXFP4 dequant: num_pages (> 0) pages of page_elems (a positive multiple of
// 32) codes gathered from a pool by id.
cudaError_t launch_mx_unpack_pages(const int64_t *page_ids, int64_t num_pages,
                                   const uint8_t *packed, const uint8_t *scales,
                                   int64_t pool_pages, int64_t page_elems, uint16_t *out,
                                   int32_t *err_flag, cudaStream_t stream);

// Resident CTAs per SM x SM count for `kernel` at `threads` threads, cached per
// device; a grid no larger than this runs in one wave.
int max_resident_ctas(const void *kernel, int threads, int slot);

}  // namespace fp4mx
