// api.cu -- the exported C ABI (include/fp4mx.h): host-side argument checks,
// then one kernel launch on the caller's stream. No allocation, no
// synchronisation, no host<->device copies.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "fp4mx.h"
#include "launch.h"

#define FP4_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_last_error[256] = "";

void clear_error() { g_last_error[0] = '\0'; }

fp4_status cuda_failure(cudaError_t err, const char *where) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where,
                  cudaGetErrorString(err), cudaGetErrorName(err));
    return FP4_ERR_CUDA;
}

bool overlaps(const void *a, uint64_t a_bytes, const void *b, uint64_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// The pointer must be memory the current device can address: device or
// managed memory of this device, or mapped pinned host memory.
fp4_status check_device_pointer(const void *p, int device) {
    cudaPointerAttributes attr;
    const cudaError_t err = cudaPointerGetAttributes(&attr, p);
    if (err != cudaSuccess) return cuda_failure(err, "cudaPointerGetAttributes");
    switch (attr.type) {
    case cudaMemoryTypeDevice:
        if (attr.device != device) {
            std::snprintf(g_last_error, sizeof g_last_error,
                          "pointer %p belongs to device %d, current device is %d", p,
                          attr.device, device);
            return FP4_ERR_POINTER;
        }
        return FP4_OK;
    case cudaMemoryTypeManaged:
        return FP4_OK;
    case cudaMemoryTypeHost:
        if (attr.devicePointer == p) return FP4_OK;
        break;
    default:
        break;
    }
    std::snprintf(g_last_error, sizeof g_last_error,
                  "pointer %p is not device-accessible CUDA memory", p);
    return FP4_ERR_POINTER;
}

bool misaligned(const void *p, uintptr_t alignment) {
    return p != nullptr && reinterpret_cast<uintptr_t>(p) % alignment != 0;
}

fp4_status check_pointers(const void *const *ptrs, int n) {
    int device = 0;
    const cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return cuda_failure(err, "cudaGetDevice");
    for (int i = 0; i < n; ++i) {
        if (ptrs[i] == nullptr) continue;
        const fp4_status s = check_device_pointer(ptrs[i], device);
        if (s != FP4_OK) return s;
    }
    return FP4_OK;
}

// Largest NVFP4 row (hidden) and paged-unpack page (page_elems), in codes: the row
// and page kernels count a row's words and 128-word segments in 32 bits.
constexpr int64_t kMaxRowCodes = (int64_t)1 << 31;

constexpr int kMaxDevices = 64;
constexpr int kSlots = 8;
std::atomic<int> g_resident[kMaxDevices][kSlots];

}  // namespace

namespace fp4mx {

int max_resident_ctas(const void *kernel, int threads, int slot) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return 1024;
    int cached = g_resident[device][slot].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) !=
            cudaSuccess ||
        sms <= 0 || per_sm <= 0) {
        cudaGetLastError();
        return 1024;
    }
    cached = sms * per_sm;
    g_resident[device][slot].store(cached, std::memory_order_relaxed);
    return cached;
}

}  // namespace fp4mx

FP4_EXPORT fp4_status fp4_mx_unpack(const uint8_t *packed, const uint8_t *scales_e8m0,
                                    uint16_t *out_bf16, int64_t rows, int64_t k,
                                    fp4_stream_t stream) {
    clear_error();
    if (rows < 0 || k < 0 || k % 32 != 0) return FP4_ERR_SHAPE;
    if (rows == 0 || k == 0) return FP4_OK;
    if (rows > INT64_MAX / 2 / k) return FP4_ERR_SHAPE;  // rows * k * 2 bytes must fit
    if (packed == nullptr || scales_e8m0 == nullptr || out_bf16 == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(out_bf16, 2)) return FP4_ERR_ALIGN;
    const int64_t n = rows * k;
    const uint64_t out_bytes = (uint64_t)n * 2;
    if (overlaps(out_bf16, out_bytes, packed, (uint64_t)n / 2) ||
        overlaps(out_bf16, out_bytes, scales_e8m0, (uint64_t)n / 32))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {packed, scales_e8m0, out_bf16};
    const fp4_status s = check_pointers(ptrs, 3);
    if (s != FP4_OK) return s;
    const cudaError_t err =
        fp4mx::launch_mx_unpack(packed, scales_e8m0, out_bf16, n, (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_mx_unpack launch");
}

FP4_EXPORT fp4_status fp4_nv_embedding_gather(const int64_t *ids, int64_t num_ids,
                                              const uint8_t *weight,
                                              const uint8_t *block_scale_e4m3,
                                              const float *global_scale, int64_t vocab,
                                              int64_t hidden, int64_t group_size,
                                              uint16_t *out_bf16, int32_t *err_flag,
                                              fp4_stream_t stream) {
    clear_error();
    if (num_ids < 0 || vocab < 0 || hidden <= 0 || group_size <= 0) return FP4_ERR_SHAPE;
    if (hidden % group_size != 0) return FP4_ERR_GROUP;
    if (group_size != 16) return FP4_ERR_UNSUPPORTED;
    if (hidden > kMaxRowCodes) return FP4_ERR_SHAPE;
    if (num_ids == 0) return FP4_OK;
    if (vocab == 0) return FP4_ERR_SHAPE;
    if (num_ids > INT64_MAX / 2 / hidden || vocab > INT64_MAX / hidden) return FP4_ERR_SHAPE;
    if (ids == nullptr || weight == nullptr || block_scale_e4m3 == nullptr ||
        global_scale == nullptr || out_bf16 == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(ids, 8) || misaligned(global_scale, 4) || misaligned(out_bf16, 2) ||
        misaligned(err_flag, 4))
        return FP4_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)num_ids * (uint64_t)hidden * 2;
    const uint64_t w_bytes = (uint64_t)vocab * (uint64_t)hidden / 2;
    const uint64_t s_bytes = (uint64_t)vocab * (uint64_t)hidden / 16;
    if (overlaps(out_bf16, out_bytes, ids, (uint64_t)num_ids * 8) ||
        overlaps(out_bf16, out_bytes, weight, w_bytes) ||
        overlaps(out_bf16, out_bytes, block_scale_e4m3, s_bytes) ||
        overlaps(out_bf16, out_bytes, global_scale, 4) ||
        (err_flag != nullptr &&
         (overlaps(err_flag, 4, out_bf16, out_bytes) || overlaps(err_flag, 4, ids, num_ids * 8) ||
          overlaps(err_flag, 4, weight, w_bytes) ||
          overlaps(err_flag, 4, block_scale_e4m3, s_bytes) ||
          overlaps(err_flag, 4, global_scale, 4))))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {ids, weight, block_scale_e4m3, global_scale, out_bf16, err_flag};
    const fp4_status s = check_pointers(ptrs, 6);
    if (s != FP4_OK) return s;
    const cudaError_t err =
        fp4mx::launch_nv_gather(ids, num_ids, weight, block_scale_e4m3, global_scale, vocab,
                                hidden, out_bf16, err_flag, (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_nv_embedding_gather launch");
}

FP4_EXPORT fp4_status fp4_mx_quantize(const uint16_t *in_bf16, uint8_t *packed_out,
                                      uint8_t *scales_e8m0_out, int64_t rows, int64_t k,
                                      fp4_stream_t stream) {
    clear_error();
    if (rows < 0 || k < 0 || k % 32 != 0) return FP4_ERR_SHAPE;
    if (rows == 0 || k == 0) return FP4_OK;
    if (rows > INT64_MAX / 2 / k) return FP4_ERR_SHAPE;
    if (in_bf16 == nullptr || packed_out == nullptr || scales_e8m0_out == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(in_bf16, 2)) return FP4_ERR_ALIGN;
    const int64_t n = rows * k;
    const uint64_t in_bytes = (uint64_t)n * 2;
    if (overlaps(packed_out, (uint64_t)n / 2, in_bf16, in_bytes) ||
        overlaps(scales_e8m0_out, (uint64_t)n / 32, in_bf16, in_bytes) ||
        overlaps(packed_out, (uint64_t)n / 2, scales_e8m0_out, (uint64_t)n / 32))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {in_bf16, packed_out, scales_e8m0_out};
    const fp4_status s = check_pointers(ptrs, 3);
    if (s != FP4_OK) return s;
    const cudaError_t err = fp4mx::launch_mx_quantize(in_bf16, packed_out, scales_e8m0_out, n,
                                                      (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_mx_quantize launch");
}

FP4_EXPORT fp4_status fp4_mx_moe_gemm(const uint16_t *a_bf16, const int64_t *expert_offsets,
                                      int64_t experts, int64_t max_rows_per_expert,
                                      const uint8_t *w_packed, const uint8_t *w_scales_e8m0,
                                      int64_t n, int64_t k, int64_t total_rows,
                                      uint16_t *out_bf16, int32_t *status,
                                      fp4_stream_t stream) {
    clear_error();
    if (experts < 0 || max_rows_per_expert < 0 || n < 0 || k < 0 || total_rows < 0)
        return FP4_ERR_SHAPE;
    if (k % 32 != 0 || n % 32 != 0) return FP4_ERR_SHAPE;
    if (experts > 65535 || max_rows_per_expert > 65535ll * 128 || n > (1ll << 30) ||
        k > (1ll << 30) || total_rows > (1ll << 31) - 1024 ||  // 32-bit TMA row coordinates
        experts * n > (1ll << 31) - 1024)                      // of activations and weights
        return FP4_ERR_SHAPE;
    if (experts == 0 || max_rows_per_expert == 0 || n == 0) return FP4_OK;
    if (a_bf16 == nullptr || expert_offsets == nullptr || w_packed == nullptr ||
        w_scales_e8m0 == nullptr || out_bf16 == nullptr || status == nullptr)
        return FP4_ERR_NULL_PTR;
    if (k == 0) return FP4_ERR_SHAPE;  // an empty reduction: nothing to multiply
    if (misaligned(a_bf16, 16) || misaligned(w_packed, 16) || misaligned(out_bf16, 16) ||
        misaligned(expert_offsets, 8) || misaligned(status, 4))
        return FP4_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)total_rows * (uint64_t)n * 2;
    const uint64_t w_bytes = (uint64_t)experts * (uint64_t)n * (uint64_t)k / 2;
    if (overlaps(out_bf16, out_bytes, a_bf16, (uint64_t)total_rows * (uint64_t)k * 2) ||
        overlaps(out_bf16, out_bytes, w_packed, w_bytes) ||
        overlaps(out_bf16, out_bytes, w_scales_e8m0, w_bytes / 16) ||
        overlaps(out_bf16, out_bytes, expert_offsets, (uint64_t)(experts + 1) * 8) ||
        overlaps(out_bf16, out_bytes, status, 4))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {a_bf16, expert_offsets, w_packed, w_scales_e8m0, out_bf16, status};
    const fp4_status s = check_pointers(ptrs, 6);
    if (s != FP4_OK) return s;
    const cudaError_t err = fp4mx::launch_mx_moe_gemm(a_bf16, expert_offsets, experts,
                                                      max_rows_per_expert, total_rows, w_packed,
                                                      w_scales_e8m0, n, k, out_bf16, status,
                                                      (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_mx_moe_gemm launch");
}

namespace {

// Shape rules of the MoE layer entry points (see include/fp4mx.h).
bool moe_shape_ok(int64_t tokens, int64_t topk, int64_t experts, int64_t n, int64_t k) {
    if (tokens < 0 || topk < 1 || topk > 1024 || experts < 1 || experts > 65535 || n < 32 ||
        k < 32 || n % 32 != 0 || k % 32 != 0 || n > (1ll << 20) || k > (1ll << 20))
        return false;
    // slot and row indices are int32, and the GEMMs' TMA row coordinates reach
    // 320 rows past a slab's start (activations) or a box past a tile (weights)
    constexpr int64_t kMaxRows = (1ll << 31) - 1024;
    return tokens * topk <= kMaxRows && experts * 2 * n <= kMaxRows && experts * k <= kMaxRows;
}

}  // namespace

FP4_EXPORT int64_t fp4_mx_moe_workspace_bytes(int64_t tokens, int64_t topk, int64_t experts,
                                              int64_t n, int64_t k) {
    if (!moe_shape_ok(tokens, topk, experts, n, k)) return -1;
    return (int64_t)fp4mx::moe_workspace_layout(tokens, topk, experts, n, k).total;
}

FP4_EXPORT fp4_status fp4_mx_moe_forward(const uint16_t *a_bf16, const int32_t *topk_ids,
                                         const float *topk_weights, int64_t tokens, int64_t topk,
                                         int64_t experts, int64_t max_rows_per_expert,
                                         const uint8_t *w1_packed, const uint8_t *w1_scales_e8m0,
                                         const uint8_t *w2_packed, const uint8_t *w2_scales_e8m0,
                                         int64_t n, int64_t k, void *workspace,
                                         int64_t workspace_bytes, uint16_t *out_bf16,
                                         int32_t *status, fp4_stream_t stream) {
    clear_error();
    if (!moe_shape_ok(tokens, topk, experts, n, k) || max_rows_per_expert < 0) return FP4_ERR_SHAPE;
    if (tokens == 0) return FP4_OK;
    const int64_t pairs = tokens * topk;
    const int64_t max_rows = max_rows_per_expert < pairs ? max_rows_per_expert : pairs;
    if (a_bf16 == nullptr || topk_ids == nullptr || topk_weights == nullptr || w1_packed == nullptr ||
        w1_scales_e8m0 == nullptr || w2_packed == nullptr || w2_scales_e8m0 == nullptr ||
        workspace == nullptr || out_bf16 == nullptr || status == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(a_bf16, 16) || misaligned(w1_packed, 16) || misaligned(w2_packed, 16) ||
        misaligned(out_bf16, 16) || misaligned(workspace, 256) || misaligned(topk_ids, 4) ||
        misaligned(topk_weights, 4) || misaligned(status, 4))
        return FP4_ERR_ALIGN;
    const uint64_t need = fp4mx::moe_workspace_layout(tokens, topk, experts, n, k).total;
    if (workspace_bytes < 0 || (uint64_t)workspace_bytes < need) {
        std::snprintf(g_last_error, sizeof g_last_error,
                      "workspace of %lld bytes, the layer needs %llu", (long long)workspace_bytes,
                      (unsigned long long)need);
        return FP4_ERR_SHAPE;
    }
    const uint64_t out_bytes = (uint64_t)tokens * (uint64_t)k * 2;
    const uint64_t w1_bytes = (uint64_t)experts * 2 * (uint64_t)n * (uint64_t)k / 2;
    const uint64_t w2_bytes = (uint64_t)experts * (uint64_t)k * (uint64_t)n / 2;
    const void *inputs[] = {a_bf16, topk_ids, topk_weights, w1_packed, w1_scales_e8m0, w2_packed,
                            w2_scales_e8m0, status};
    const uint64_t in_bytes[] = {out_bytes, (uint64_t)pairs * 4, (uint64_t)pairs * 4, w1_bytes,
                                 w1_bytes / 16, w2_bytes, w2_bytes / 16, 4};
    for (int i = 0; i < 8; ++i)
        if (overlaps(out_bf16, out_bytes, inputs[i], in_bytes[i]) ||
            overlaps(workspace, need, inputs[i], in_bytes[i]))
            return FP4_ERR_ALIAS;
    if (overlaps(out_bf16, out_bytes, workspace, need)) return FP4_ERR_ALIAS;
    const void *ptrs[] = {a_bf16, topk_ids, topk_weights, w1_packed, w1_scales_e8m0, w2_packed,
                          w2_scales_e8m0, workspace, out_bf16, status};
    const fp4_status s = check_pointers(ptrs, 10);
    if (s != FP4_OK) return s;
    const cudaError_t err = fp4mx::launch_mx_moe_forward(
        a_bf16, topk_ids, topk_weights, tokens, topk, experts, max_rows, w1_packed, w1_scales_e8m0,
        w2_packed, w2_scales_e8m0, n, k, workspace, out_bf16, status, (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_mx_moe_forward launch");
}

FP4_EXPORT int64_t fp4_mx_moe_static_scratch_bytes(void) {
    return (int64_t)fp4mx::moe_static_scratch_bytes();
}

FP4_EXPORT fp4_status fp4_wait_selftest(int32_t mode, int32_t *status, fp4_stream_t stream) {
    clear_error();
    if (mode < 0 || mode > 2) return FP4_ERR_SHAPE;
    if (status == nullptr) return FP4_ERR_NULL_PTR;
    if (misaligned(status, 4)) return FP4_ERR_ALIGN;
    const void *ptrs[] = {status};
    const fp4_status s = check_pointers(ptrs, 1);
    if (s != FP4_OK) return s;
    const cudaError_t err = fp4mx::launch_wait_selftest(mode, status, (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_wait_selftest launch");
}

FP4_EXPORT fp4_status fp4_mx_moe_forward_noalloc(
    const uint16_t *a_bf16, const int32_t *topk_ids, const float *topk_weights, int64_t tokens,
    int64_t topk, int64_t experts, int64_t max_rows_per_expert, const uint8_t *w1_packed,
    const uint8_t *w1_scales_e8m0, const uint8_t *w2_packed, const uint8_t *w2_scales_e8m0,
    int64_t n, int64_t k, uint16_t *out_bf16, int32_t *status, fp4_stream_t stream) {
    clear_error();
    if (!moe_shape_ok(tokens, topk, experts, n, k) || max_rows_per_expert < 0) return FP4_ERR_SHAPE;
    if (tokens == 0) return FP4_OK;
    const uint64_t need = fp4mx::moe_workspace_layout(tokens, topk, experts, n, k).total;
    if (need > fp4mx::moe_static_scratch_bytes()) {  // size rejection: nothing is launched
        std::snprintf(g_last_error, sizeof g_last_error,
                      "the layer needs %llu bytes of scratch, the static area holds %llu",
                      (unsigned long long)need,
                      (unsigned long long)fp4mx::moe_static_scratch_bytes());
        return FP4_ERR_SHAPE;
    }
    void *scratch = nullptr;
    const cudaError_t err = fp4mx::moe_static_scratch(&scratch);
    if (err != cudaSuccess) return cuda_failure(err, "static scratch address");
    return fp4_mx_moe_forward(a_bf16, topk_ids, topk_weights, tokens, topk, experts,
                              max_rows_per_expert, w1_packed, w1_scales_e8m0, w2_packed,
                              w2_scales_e8m0, n, k, scratch, (int64_t)need, out_bf16, status,
                              stream);
}

FP4_EXPORT fp4_status fp4_mx_unpack_pages(const int64_t *page_ids, int64_t num_pages,
                                          const uint8_t *packed_pool,
                                          const uint8_t *scales_pool_e8m0, int64_t pool_pages,
                                          int64_t page_elems, uint16_t *out_bf16,
                                          int32_t *err_flag, fp4_stream_t stream) {
    clear_error();
    if (num_pages < 0 || pool_pages < 0 || page_elems <= 0 || page_elems % 32 != 0 ||
        page_elems > kMaxRowCodes)
        return FP4_ERR_SHAPE;
    if (num_pages == 0) return FP4_OK;
    if (pool_pages == 0) return FP4_ERR_SHAPE;
    if (num_pages > INT64_MAX / 2 / page_elems || pool_pages > INT64_MAX / page_elems)
        return FP4_ERR_SHAPE;
    if (page_ids == nullptr || packed_pool == nullptr || scales_pool_e8m0 == nullptr ||
        out_bf16 == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(page_ids, 8) || misaligned(out_bf16, 2) || misaligned(err_flag, 4))
        return FP4_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)num_pages * (uint64_t)page_elems * 2;
    const uint64_t pool_bytes = (uint64_t)pool_pages * (uint64_t)page_elems / 2;
    if (overlaps(out_bf16, out_bytes, page_ids, (uint64_t)num_pages * 8) ||
        overlaps(out_bf16, out_bytes, packed_pool, pool_bytes) ||
        overlaps(out_bf16, out_bytes, scales_pool_e8m0, pool_bytes / 16) ||
        (err_flag != nullptr &&
         (overlaps(err_flag, 4, out_bf16, out_bytes) ||
          overlaps(err_flag, 4, page_ids, (uint64_t)num_pages * 8) ||
          overlaps(err_flag, 4, packed_pool, pool_bytes) ||
          overlaps(err_flag, 4, scales_pool_e8m0, pool_bytes / 16))))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {page_ids, packed_pool, scales_pool_e8m0, out_bf16, err_flag};
    const fp4_status s = check_pointers(ptrs, 5);
    if (s != FP4_OK) return s;
    const cudaError_t err =
        fp4mx::launch_mx_unpack_pages(page_ids, num_pages, packed_pool, scales_pool_e8m0,
                                      pool_pages, page_elems, out_bf16, err_flag,
                                      (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_mx_unpack_pages launch");
}

FP4_EXPORT fp4_status fp4_nv_dequant(const uint8_t *weight, const uint8_t *block_scale_e4m3,
                                     const float *global_scale, int64_t rows, int64_t hidden,
                                     int64_t group_size, uint16_t *out_bf16,
                                     fp4_stream_t stream) {
    clear_error();
    if (rows < 0 || hidden <= 0 || group_size <= 0) return FP4_ERR_SHAPE;
    if (hidden % group_size != 0) return FP4_ERR_GROUP;
    if (group_size != 16) return FP4_ERR_UNSUPPORTED;
    if (hidden > kMaxRowCodes) return FP4_ERR_SHAPE;
    if (rows == 0) return FP4_OK;
    if (rows > INT64_MAX / 2 / hidden) return FP4_ERR_SHAPE;
    if (weight == nullptr || block_scale_e4m3 == nullptr || global_scale == nullptr ||
        out_bf16 == nullptr)
        return FP4_ERR_NULL_PTR;
    if (misaligned(global_scale, 4) || misaligned(out_bf16, 2)) return FP4_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)rows * (uint64_t)hidden * 2;
    if (overlaps(out_bf16, out_bytes, weight, (uint64_t)rows * (uint64_t)hidden / 2) ||
        overlaps(out_bf16, out_bytes, block_scale_e4m3, (uint64_t)rows * (uint64_t)hidden / 16) ||
        overlaps(out_bf16, out_bytes, global_scale, 4))
        return FP4_ERR_ALIAS;
    const void *ptrs[] = {weight, block_scale_e4m3, global_scale, out_bf16};
    const fp4_status s = check_pointers(ptrs, 4);
    if (s != FP4_OK) return s;
    const cudaError_t err = fp4mx::launch_nv_dequant(weight, block_scale_e4m3, global_scale, rows,
                                                     hidden, out_bf16, (cudaStream_t)stream);
    return err == cudaSuccess ? FP4_OK : cuda_failure(err, "fp4_nv_dequant launch");
}

FP4_EXPORT const char *fp4_status_string(fp4_status status) {
    switch (status) {
    case FP4_OK: return "ok";
    case FP4_ERR_NULL_PTR: return "a required pointer is NULL";
    case FP4_ERR_SHAPE: return "invalid shape (negative size, k % 32 != 0, or size overflow)";
    case FP4_ERR_GROUP: return "hidden size is not a multiple of group_size";
    case FP4_ERR_UNSUPPORTED: return "unsupported group_size (NVFP4 uses 16)";
    case FP4_ERR_INDEX: return "token id outside [0, vocab)";
    case FP4_ERR_CUDA: return "CUDA runtime error";
    case FP4_ERR_POINTER: return "pointer is not device-accessible CUDA memory";
    case FP4_ERR_ALIAS: return "output overlaps an input";
    case FP4_ERR_ALIGN: return "pointer not aligned to its element type";
    case FP4_ERR_TIMEOUT: return "a bounded wait on the tensor core ran out (reported in status)";
    }
    return "unknown status";
}

FP4_EXPORT const char *fp4_last_error(void) { return g_last_error; }

FP4_EXPORT int fp4_abi_version(void) { return 108; }
