// nv_gather.cu -- NVFP4 token-embedding gather-dequant to bf16 on sm_103a.
//
// The method ("sgl-project/sglang pull 34222", sections "Implementation
// breakdown" and "Key source snippets"): token ids pick rows of packed E2M1
// codes and of e4m3 block scales (one per 16 codes); each code's value times
// (block scale * global scale), in fp32, is rounded to bf16.
//
// A warp owns one segment of one output row (up to 32 * kUnroll words = 256 *
// kUnroll codes), so each row is read with coalesced 128-byte warp loads and
// written with 512-byte warp stores; rows are cut into segments so that a
// persistent grid of warps balances even when there are fewer rows than warps.
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
constexpr int64_t kSegWords = 32 * kUnroll;

__global__ void __launch_bounds__(kThreads)
nv_gather_words_kernel(const int64_t *__restrict__ ids, int64_t num_ids,
                       const uint32_t *__restrict__ weight, const uint8_t *__restrict__ scales,
                       const float *__restrict__ global_scale, int64_t vocab,
                       int64_t words_per_row, int64_t segs_per_row, uint4 *__restrict__ out,
                       int32_t *__restrict__ err_flag) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t n_units = num_ids * segs_per_row;
    const int64_t groups_per_row = words_per_row / 2;  // 2 words per 16-code group
    const float gs = __ldg(global_scale);
    for (int64_t unit = warp; unit < n_units; unit += n_warps) {
        const int64_t t = unit / segs_per_row;
        const int64_t w0 = (unit - t * segs_per_row) * kSegWords;
        const int64_t id = __ldg(ids + t);
        uint4 *out_row = out + t * words_per_row;
        if (id < 0 || id >= vocab) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t i = w0 + u * 32 + lane;
                if (i < words_per_row) st_stream(out_row + i, make_uint4(0, 0, 0, 0));
            }
            if (w0 == 0 && lane == 0 && err_flag != nullptr) atomicExch(err_flag, FP4_ERR_INDEX);
            continue;
        }
        const uint32_t *w_row = weight + id * words_per_row;
        const uint8_t *s_row = scales + id * groups_per_row;
        uint32_t w[kUnroll], s[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = w0 + u * 32 + lane;
            if (i < words_per_row) {
                w[u] = __ldg(w_row + i);
                s[u] = __ldg(s_row + (i >> 1));
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = w0 + u * 32 + lane;
            if (i < words_per_row) {
                const float eff = __fmul_rn(e4m3_to_f32(s[u]), gs);
                st_stream(out_row + i, nv_decode_word(w[u], eff));
            }
        }
    }
}

// Any alignment: one thread per packed byte of the output (two codes).
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
        const int64_t id = ids[t];
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

}  // namespace

cudaError_t launch_nv_gather(const int64_t *ids, int64_t num_ids, const uint8_t *weight,
                             const uint8_t *scales, const float *global_scale, int64_t vocab,
                             int64_t hidden, uint16_t *out, int32_t *err_flag,
                             cudaStream_t stream) {
    const bool vector_ok = (reinterpret_cast<uintptr_t>(weight) % 4 == 0) &&
                           (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    if (vector_ok) {
        const int64_t words_per_row = hidden / 8;
        const int64_t segs = (words_per_row + kSegWords - 1) / kSegWords;
        const int64_t units = num_ids * segs;
        const int64_t blocks = (units + kWarps - 1) / kWarps;
        const int cap = max_resident_ctas((const void *)nv_gather_words_kernel, kThreads, 2);
        const int grid = (int)(blocks < cap ? blocks : cap);
        nv_gather_words_kernel<<<grid, kThreads, 0, stream>>>(
            ids, num_ids, reinterpret_cast<const uint32_t *>(weight), scales, global_scale, vocab,
            words_per_row, segs, reinterpret_cast<uint4 *>(out), err_flag);
    } else {
        const int64_t n = num_ids * (hidden / 2);
        const int64_t blocks = (n + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)nv_gather_bytes_kernel, kThreads, 3);
        const int grid = (int)(blocks < cap ? blocks : cap);
        nv_gather_bytes_kernel<<<grid, kThreads, 0, stream>>>(ids, num_ids, weight, scales,
                                                              global_scale, vocab, hidden, out,
                                                              err_flag);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
