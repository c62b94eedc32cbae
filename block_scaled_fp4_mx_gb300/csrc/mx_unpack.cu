// mx_unpack.cu -- MXFP4 (E2M1 + E8M0 per 32) to bf16 on sm_103a.
//
// The method ("vllm-project/vllm pull 51583", sections "Motivation" and
// "Implementation breakdown"): each code's bf16 pattern gets (E - 127) << 7
// added into its exponent field with a wrapping 16-bit add, and the two zero
// codes become +0.0 lane by lane.
//
// The work is a stream: per 32-element block, 16 packed bytes and 1 scale byte
// in, 64 bytes out (2.53 bytes per element, 79% of them writes), so the kernel
// is bound by HBM bandwidth. Layout of the work: a warp instruction covers 32
// consecutive words (128 packed bytes in, 512 contiguous output bytes), so loads
// and stores are fully coalesced; each thread keeps kUnroll independent loads
// in flight before decoding. The grid is one-shot (one chunk of kThreads *
// kUnroll words per CTA, as many CTAs as chunks): the block scheduler then keeps
// the CTAs in flight on a compact, advancing window of memory, which measured
// ~15% faster on GB300 than a persistent grid-stride loop whose CTAs drift apart.
#include "fp4_decode.cuh"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
mx_unpack_words_kernel(const uint32_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                       uint4 *__restrict__ out, int64_t n_words) {
    const int64_t base = (int64_t)blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
    uint32_t w[kUnroll], e[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads;
        if (i < n_words) {
            w[u] = ld_stream(packed + i);
            e[u] = __ldg(scales + (i >> 2));  // 4 words per 32-element block
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads;
        if (i < n_words) st_stream(out + i, mx_decode_word(w[u], mx_scaled_table(e[u])));
    }
}

// Any alignment: one thread per packed byte (two outputs).
__global__ void __launch_bounds__(kThreads)
mx_unpack_bytes_kernel(const uint8_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                       uint16_t *__restrict__ out, int64_t n_bytes) {
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n_bytes;
         i += (int64_t)gridDim.x * kThreads) {
        const uint32_t byte = packed[i];
        const uint32_t e8m0 = scales[i >> 4];  // 16 bytes per 32-element block
        out[2 * i] = mx_decode_code(byte & 0x0Fu, e8m0);
        out[2 * i + 1] = mx_decode_code(byte >> 4, e8m0);
    }
}

}  // namespace

cudaError_t launch_mx_unpack(const uint8_t *packed, const uint8_t *scales, uint16_t *out,
                             int64_t n_elems, cudaStream_t stream) {
    const bool vector_ok = (reinterpret_cast<uintptr_t>(packed) % 4 == 0) &&
                           (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    if (vector_ok) {
        // One chunk per CTA; launches of at most kMaxGrid CTAs (a limit no tensor
        // that fits in memory reaches in practice).
        constexpr int64_t kChunk = (int64_t)kThreads * kUnroll;
        constexpr int64_t kMaxGrid = 1ll << 30;
        const int64_t n_words = n_elems / 8;
        for (int64_t w0 = 0; w0 < n_words; w0 += kMaxGrid * kChunk) {
            const int64_t n = (n_words - w0 < kMaxGrid * kChunk) ? n_words - w0 : kMaxGrid * kChunk;
            const int grid = (int)((n + kChunk - 1) / kChunk);
            mx_unpack_words_kernel<<<grid, kThreads, 0, stream>>>(
                reinterpret_cast<const uint32_t *>(packed) + w0, scales + w0 / 4,
                reinterpret_cast<uint4 *>(out) + w0, n);
        }
    } else {
        const int64_t n_bytes = n_elems / 2;
        const int64_t blocks = (n_bytes + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)mx_unpack_bytes_kernel, kThreads, 1);
        const int grid = (int)(blocks < cap ? blocks : cap);
        mx_unpack_bytes_kernel<<<grid, kThreads, 0, stream>>>(packed, scales, out, n_bytes);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
