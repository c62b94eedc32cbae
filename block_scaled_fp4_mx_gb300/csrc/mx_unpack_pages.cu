// mx_unpack_pages.cu -- batched (paged) MXFP4 dequant of a KV cache on sm_103a.
//
// "sgl-project/sglang pull 34222", "Risks" item 3: the KV-cache path scales its
// FP4 codes by E8M0 powers of two (kvfp4 batched_dequantize), unlike the NVFP4
// embedding. Here a page table picks pages of an MXFP4 KV pool ([pool_pages,
// page_elems/2] codes, [pool_pages, page_elems/32] E8M0 bytes) and each page is
// decoded exactly as fp4_mx_unpack decodes it. Layout of the work as in the NVFP4
// gather: a warp owns one 128-word segment of one output page (coalesced 128-byte
// warp loads, 512-byte warp stores, 4 loads in flight per lane), one-shot grid;
// pages narrower than 32 words take a flat thread-per-word kernel. An id outside
// [0, pool_pages) never faults: its row is +0.0 and the caller's flag is set.
#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr uint32_t kSegWords = 32 * kUnroll;

__global__ void __launch_bounds__(kThreads)
mx_pages_rows_kernel(const int64_t *__restrict__ page_ids, uint32_t n_units,
                     const uint32_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                     int64_t pool_pages, uint32_t words_per_page, uint32_t segs_per_page,
                     uint4 *__restrict__ out, int32_t *__restrict__ err_flag) {
    const uint32_t unit = blockIdx.x * (uint32_t)kWarps + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    const int lane = threadIdx.x & 31;
    const uint32_t t = unit / segs_per_page;
    const uint32_t w0 = (unit - t * segs_per_page) * kSegWords;
    const int64_t id = __ldg(page_ids + t);
    uint4 *out_row = out + (int64_t)t * words_per_page;
    if (id < 0 || id >= pool_pages) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t i = w0 + u * 32 + lane;
            if (i < words_per_page) st_stream(out_row + i, make_uint4(0, 0, 0, 0));
        }
        if (w0 == 0 && lane == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
        return;
    }
    const uint32_t *page = packed + id * words_per_page;
    const uint8_t *page_scales = scales + id * (words_per_page / 4);  // 4 words per block
    uint32_t w[kUnroll], e[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = w0 + u * 32 + lane;
        if (i < words_per_page) {
            w[u] = __ldg(page + i);
            e[u] = __ldg(page_scales + (i >> 2));
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = w0 + u * 32 + lane;
        if (i < words_per_page) st_stream(out_row + i, mx_decode_word(w[u], mx_scaled_table(e[u])));
    }
}

// Thread per word of the flattened [num_pages, words_per_page] output.
__global__ void __launch_bounds__(kThreads)
mx_pages_flat_kernel(const int64_t *__restrict__ page_ids, int64_t n_words,
                     const uint32_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                     int64_t pool_pages, uint32_t words_per_page, uint4 *__restrict__ out,
                     int32_t *__restrict__ err_flag) {
    const int64_t base = (int64_t)blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t f = base + u * kThreads;
        if (f >= n_words) continue;
        const int64_t t = f / words_per_page;
        const uint32_t i = (uint32_t)(f - t * words_per_page);
        const int64_t id = __ldg(page_ids + t);
        if (id < 0 || id >= pool_pages) {
            st_stream(out + f, make_uint4(0, 0, 0, 0));
            if (i == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
            continue;
        }
        const uint32_t w = __ldg(packed + id * words_per_page + i);
        const uint32_t e = __ldg(scales + id * (words_per_page / 4) + (i >> 2));
        st_stream(out + f, mx_decode_word(w, mx_scaled_table(e)));
    }
}

// Any alignment: one thread per packed byte, the independent per-code formula.
__global__ void __launch_bounds__(kThreads)
mx_pages_bytes_kernel(const int64_t *__restrict__ page_ids, int64_t num_pages,
                      const uint8_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                      int64_t pool_pages, int64_t page_elems, uint16_t *__restrict__ out,
                      int32_t *__restrict__ err_flag) {
    const int64_t half = page_elems / 2;
    const int64_t n = num_pages * half;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kThreads) {
        const int64_t t = i / half;
        const int64_t b = i - t * half;
        const int64_t id = page_ids[t];
        uint16_t *o = out + t * page_elems + 2 * b;
        if (id < 0 || id >= pool_pages) {
            o[0] = 0;
            o[1] = 0;
            if (b == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
            continue;
        }
        const uint32_t byte = packed[id * half + b];
        const uint32_t e8m0 = scales[id * (page_elems / 32) + b / 16];
        o[0] = mx_decode_code(byte & 0x0Fu, e8m0);
        o[1] = mx_decode_code(byte >> 4, e8m0);
    }
}

}  // namespace

cudaError_t launch_mx_unpack_pages(const int64_t *page_ids, int64_t num_pages,
                                   const uint8_t *packed, const uint8_t *scales,
                                   int64_t pool_pages, int64_t page_elems, uint16_t *out,
                                   int32_t *err_flag, cudaStream_t stream) {
    const bool vector_ok = (reinterpret_cast<uintptr_t>(packed) % 4 == 0) &&
                           (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    if (vector_ok) {
        const int64_t words_per_page = page_elems / 8;
        if (words_per_page >= 32) {
            const int64_t segs = (words_per_page + kSegWords - 1) / kSegWords;
            const int64_t rows_per_launch = ((int64_t)1 << 31) / segs;
            for (int64_t r0 = 0; r0 < num_pages; r0 += rows_per_launch) {
                const int64_t rows = num_pages - r0 < rows_per_launch ? num_pages - r0 : rows_per_launch;
                const int64_t units = rows * segs;
                const int grid = (int)((units + kWarps - 1) / kWarps);
                mx_pages_rows_kernel<<<grid, kThreads, 0, stream>>>(
                    page_ids + r0, (uint32_t)units, reinterpret_cast<const uint32_t *>(packed),
                    scales, pool_pages, (uint32_t)words_per_page, (uint32_t)segs,
                    reinterpret_cast<uint4 *>(out) + r0 * words_per_page, err_flag);
            }
        } else {
            constexpr int64_t kChunk = (int64_t)kThreads * kUnroll;
            const int64_t rows_per_launch = ((int64_t)1 << 40) / words_per_page;
            for (int64_t r0 = 0; r0 < num_pages; r0 += rows_per_launch) {
                const int64_t rows = num_pages - r0 < rows_per_launch ? num_pages - r0 : rows_per_launch;
                const int64_t n_words = rows * words_per_page;
                const int grid = (int)((n_words + kChunk - 1) / kChunk);
                mx_pages_flat_kernel<<<grid, kThreads, 0, stream>>>(
                    page_ids + r0, n_words, reinterpret_cast<const uint32_t *>(packed), scales,
                    pool_pages, (uint32_t)words_per_page,
                    reinterpret_cast<uint4 *>(out) + r0 * words_per_page, err_flag);
            }
        }
    } else {
        const int64_t n = num_pages * (page_elems / 2);
        const int64_t blocks = (n + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)mx_pages_bytes_kernel, kThreads, 6);
        const int grid = (int)(blocks < cap ? blocks : cap);
        mx_pages_bytes_kernel<<<grid, kThreads, 0, stream>>>(page_ids, num_pages, packed, scales,
                                                             pool_pages, page_elems, out, err_flag);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
