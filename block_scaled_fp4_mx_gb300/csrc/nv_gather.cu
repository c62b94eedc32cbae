// nv_gather.cu -- NVFP4 token-embedding gather-dequant to bf16 on sm_103a.
//
// The method ("sgl-project/sglang pull 34222", sections "Implementation
// breakdown" and "Key source snippets"): token ids pick rows of packed E2M1
// codes and of e4m3 block scales (one per 16 codes); each code's value times
// (block scale * global scale), in fp32, is rounded to bf16.
//
// A warp owns one segment of one output row (up to 32 * kUnroll words = 256 *
// kUnroll codes), so each row is read with coalesced 128-byte warp loads and
// written with 512-byte warp stores, with kUnroll loads in flight per lane.
// The grid is one-shot (one warp per segment): the block scheduler keeps the
// CTAs in flight on a compact, advancing window of the output, which measured
// faster on GB300 than a persistent grid-stride loop. Rows narrower than 32
// words take a flat kernel (one thread per word of the [num_ids, hidden]
// output) so that lanes are not left idle.
// An id outside [0, vocab) never faults: its row is written as +0.0 and the
// caller's error flag is set.
#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr uint32_t kSegWords = 32 * kUnroll;

// Warp per (row, segment). Rows are [0, num_rows) of this launch; unit = row *
// segs_per_row + segment fits in 32 bits (the launcher splits larger calls).
// kGather: the source row is ids[t] (embedding lookup); otherwise it is
// row0 + t (dense dequant of a table, ids unused).
template <bool kGather>
__global__ void __launch_bounds__(kThreads)
nv_gather_rows_kernel(const int64_t *__restrict__ ids, uint32_t n_units,
                      const uint32_t *__restrict__ weight, const uint8_t *__restrict__ scales,
                      const float *__restrict__ global_scale, int64_t vocab,
                      uint32_t words_per_row, uint32_t segs_per_row, uint4 *__restrict__ out,
                      int32_t *__restrict__ err_flag, int64_t row0) {
    const uint32_t unit = blockIdx.x * (uint32_t)kWarps + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    const int lane = threadIdx.x & 31;
    const uint32_t t = unit / segs_per_row;
    const uint32_t w0 = (unit - t * segs_per_row) * kSegWords;
    const int64_t id = kGather ? __ldg(ids + t) : row0 + t;
    uint4 *out_row = out + (int64_t)t * words_per_row;
    if (id < 0 || id >= vocab) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t i = w0 + u * 32 + lane;
            if (i < words_per_row) st_stream(out_row + i, make_uint4(0, 0, 0, 0));
        }
        if (w0 == 0 && lane == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
        return;
    }
    const float gs = __ldg(global_scale);
    const uint32_t *w_row = weight + id * words_per_row;
    const uint8_t *s_row = scales + id * (words_per_row / 2);  // 2 words per 16-code group
    uint32_t w[kUnroll], s[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = w0 + u * 32 + lane;
        if (i < words_per_row) {
            w[u] = __ldg(w_row + i);
            s[u] = __ldg(s_row + (i >> 1));
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = w0 + u * 32 + lane;
        if (i < words_per_row)
            st_stream(out_row + i, nv_decode_word(w[u], __fmul_rn(e4m3_to_f32(s[u]), gs)));
    }
}

// Thread per word of the flattened [num_rows, words_per_row] output, kUnroll
// words per thread strided by kThreads (for rows narrower than a warp's loads).
template <bool kGather>
__global__ void __launch_bounds__(kThreads)
nv_gather_flat_kernel(const int64_t *__restrict__ ids, int64_t n_words,
                      const uint32_t *__restrict__ weight, const uint8_t *__restrict__ scales,
                      const float *__restrict__ global_scale, int64_t vocab,
                      uint32_t words_per_row, uint4 *__restrict__ out,
                      int32_t *__restrict__ err_flag, int64_t row0) {
    const int64_t base = (int64_t)blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
    const float gs = __ldg(global_scale);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t f = base + u * kThreads;
        if (f >= n_words) continue;
        const int64_t t = f / words_per_row;
        const uint32_t i = (uint32_t)(f - t * words_per_row);
        const int64_t id = kGather ? __ldg(ids + t) : row0 + t;
        if (id < 0 || id >= vocab) {
            st_stream(out + f, make_uint4(0, 0, 0, 0));
            if (i == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
            continue;
        }
        const uint32_t w = __ldg(weight + id * words_per_row + i);
        const uint32_t sc = __ldg(scales + id * (words_per_row / 2) + (i >> 1));
        st_stream(out + f, nv_decode_word(w, __fmul_rn(e4m3_to_f32(sc), gs)));
    }
}

// Any alignment: one thread per packed byte of the output (two codes).
template <bool kGather>
__global__ void __launch_bounds__(kThreads)
nv_gather_bytes_kernel(const int64_t *__restrict__ ids, int64_t num_ids,
                       const uint8_t *__restrict__ weight, const uint8_t *__restrict__ scales,
                       const float *__restrict__ global_scale, int64_t vocab, int64_t hidden,
                       uint16_t *__restrict__ out, int32_t *__restrict__ err_flag) {
    const int64_t half = hidden / 2;
    const int64_t groups = hidden / 16;
    const int64_t n = num_ids * half;
    const float gs = *global_scale;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kThreads) {
        const int64_t t = i / half;
        const int64_t b = i - t * half;
        const int64_t id = kGather ? ids[t] : t;
        uint16_t *o = out + t * hidden + 2 * b;
        if (id < 0 || id >= vocab) {
            o[0] = 0;
            o[1] = 0;
            if (b == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
            continue;
        }
        const uint32_t byte = weight[id * half + b];
        const float eff = __fmul_rn(e4m3_to_f32(scales[id * groups + (2 * b) / 16]), gs);
        o[0] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(nv_code_value(byte & 0x0Fu), eff)));
        o[1] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(nv_code_value(byte >> 4), eff)));
    }
}

// Vectorised path shared by the gather and the dense dequant: row-segment
// kernel for rows of at least 32 words, flat kernel below that.
template <bool kGather>
void launch_nv_words(const int64_t *ids, int64_t num_rows, const uint8_t *weight,
                     const uint8_t *scales, const float *global_scale, int64_t vocab,
                     int64_t hidden, uint16_t *out, int32_t *err_flag, cudaStream_t stream) {
    const int64_t words_per_row = hidden / 8;
    if (words_per_row >= 32) {
        // rows in pieces so that row * segments stays below 2^31
        const int64_t segs = (words_per_row + kSegWords - 1) / kSegWords;
        const int64_t rows_per_launch = ((int64_t)1 << 31) / segs;
        for (int64_t r0 = 0; r0 < num_rows; r0 += rows_per_launch) {
            const int64_t rows = num_rows - r0 < rows_per_launch ? num_rows - r0 : rows_per_launch;
            const int64_t units = rows * segs;
            const int grid = (int)((units + kWarps - 1) / kWarps);
            nv_gather_rows_kernel<kGather><<<grid, kThreads, 0, stream>>>(
                kGather ? ids + r0 : nullptr, (uint32_t)units,
                reinterpret_cast<const uint32_t *>(weight), scales, global_scale, vocab,
                (uint32_t)words_per_row, (uint32_t)segs,
                reinterpret_cast<uint4 *>(out) + r0 * words_per_row, err_flag, r0);
        }
    } else {
        constexpr int64_t kChunk = (int64_t)kThreads * kUnroll;
        const int64_t rows_per_launch = ((int64_t)1 << 40) / words_per_row;
        for (int64_t r0 = 0; r0 < num_rows; r0 += rows_per_launch) {
            const int64_t rows = num_rows - r0 < rows_per_launch ? num_rows - r0 : rows_per_launch;
            const int64_t n_words = rows * words_per_row;
            const int grid = (int)((n_words + kChunk - 1) / kChunk);
            nv_gather_flat_kernel<kGather><<<grid, kThreads, 0, stream>>>(
                kGather ? ids + r0 : nullptr, n_words, reinterpret_cast<const uint32_t *>(weight),
                scales, global_scale, vocab, (uint32_t)words_per_row,
                reinterpret_cast<uint4 *>(out) + r0 * words_per_row, err_flag, r0);
        }
    }
}

bool vectorisable(const uint8_t *weight, const uint16_t *out) {
    return (reinterpret_cast<uintptr_t>(weight) % 4 == 0) &&
           (reinterpret_cast<uintptr_t>(out) % 16 == 0);
}

}  // namespace

cudaError_t launch_nv_gather(const int64_t *ids, int64_t num_ids, const uint8_t *weight,
                             const uint8_t *scales, const float *global_scale, int64_t vocab,
                             int64_t hidden, uint16_t *out, int32_t *err_flag,
                             cudaStream_t stream) {
    if (vectorisable(weight, out)) {
        launch_nv_words<true>(ids, num_ids, weight, scales, global_scale, vocab, hidden, out,
                              err_flag, stream);
    } else {
        const int64_t n = num_ids * (hidden / 2);
        const int64_t blocks = (n + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)nv_gather_bytes_kernel<true>, kThreads, 3);
        const int grid = (int)(blocks < cap ? blocks : cap);
        nv_gather_bytes_kernel<true><<<grid, kThreads, 0, stream>>>(
            ids, num_ids, weight, scales, global_scale, vocab, hidden, out, err_flag);
    }
    return cudaGetLastError();
}

cudaError_t launch_nv_dequant(const uint8_t *weight, const uint8_t *scales,
                              const float *global_scale, int64_t rows, int64_t hidden,
                              uint16_t *out, cudaStream_t stream) {
    if (vectorisable(weight, out)) {
        launch_nv_words<false>(nullptr, rows, weight, scales, global_scale, rows, hidden, out,
                               nullptr, stream);
    } else {
        const int64_t n = rows * (hidden / 2);
        const int64_t blocks = (n + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)nv_gather_bytes_kernel<false>, kThreads, 4);
        const int grid = (int)(blocks < cap ? blocks : cap);
        nv_gather_bytes_kernel<false><<<grid, kThreads, 0, stream>>>(
            nullptr, rows, weight, scales, global_scale, rows, hidden, out, nullptr);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
