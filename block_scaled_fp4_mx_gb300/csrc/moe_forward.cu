// moe_forward.cu -- the MoE layer around the MXFP4 expert GEMMs (sm_103a).
//
// The consumer of the unpack on the pages is a whole MoE layer ("vllm-project/vllm
// pull 51583": the CPU test runs ops.fused_experts_cpu with MXFP4 experts):
// tokens pick top-k experts, each expert runs gate/up GEMM -> silu(gate) * up ->
// down GEMM, and a token's output is the weighted sum over its slots. Here:
//   1. moe_count_kernel   histogram of the slots' expert ids (bad ids flagged);
//   2. moe_scan_kernel    exclusive prefix -> per-expert row offsets, cursors;
//   3. moe_scatter_kernel each valid slot takes a row of its expert's segment and
//                         copies its token's activations there (one warp per slot);
//   4. gate/up GEMM       the tensor-memory GEMM in gate/up mode: act = bf16(silu(g) * u);
//   5. down GEMM          the same kernel: y = bf16(act @ W2_e^T);
//   6. moe_combine_kernel out[m] = bf16(sum_j w[m, j] * y[row of slot j]) in fp32,
//                         slots in order j = 0, 1, ... (one warp per token).
// The order of rows inside an expert's segment follows atomic arrival and is not
// fixed, but every row is computed on its own (no value depends on its position)
// and the combine sums slots in a fixed order, so the output is deterministic.
// All scratch lives in the caller's workspace (fp4_mx_moe_workspace_bytes).
#include <cstddef>
#include <cstdint>

#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads)
moe_count_kernel(const int32_t *__restrict__ ids, int64_t pairs, int32_t experts,
                 int32_t *__restrict__ counts, int32_t *__restrict__ status) {
    for (int64_t p = (int64_t)blockIdx.x * kThreads + threadIdx.x; p < pairs;
         p += (int64_t)gridDim.x * kThreads) {
        const int32_t e = ids[p];
        if (e < 0 || e >= experts)
            atomicExch(status, FP4_ERR_INDEX);
        else
            atomicAdd(counts + e, 1);
    }
}

// One block of 1024 threads: thread t sums a contiguous run of experts, the block
// scans the run sums, and each thread writes its run's offsets. An expert with
// more rows than the capacity is flagged; the scatter then drops its slots.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
moe_scan_kernel(const int32_t *__restrict__ counts, int32_t experts, int64_t max_rows,
                int64_t *__restrict__ offsets, int32_t *__restrict__ cursors,
                int32_t *__restrict__ status) {
    __shared__ int64_t part[kScanThreads];
    const int t = threadIdx.x;
    const int per = (experts + kScanThreads - 1) / kScanThreads;
    const int e0 = t * per;
    const int e1 = e0 + per < experts ? e0 + per : experts;
    int64_t sum = 0;
    for (int e = e0; e < e1; ++e) sum += counts[e];
    part[t] = sum;
    __syncthreads();
    for (int d = 1; d < kScanThreads; d <<= 1) {  // inclusive Hillis-Steele scan
        const int64_t v = t >= d ? part[t - d] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int64_t run = part[t] - sum;  // exclusive prefix of this thread's run
    for (int e = e0; e < e1; ++e) {
        offsets[e] = run;
        cursors[e] = (int32_t)run;
        if (counts[e] > max_rows) atomicExch(status, FP4_ERR_SHAPE);
        run += counts[e];
    }
    if (t == kScanThreads - 1) offsets[experts] = part[t];
}

// One warp per slot p = m * topk + j.
__global__ void __launch_bounds__(kThreads)
moe_scatter_kernel(const int32_t *__restrict__ ids, int64_t pairs, int32_t topk, int32_t experts,
                   int64_t max_rows, const int32_t *__restrict__ counts,
                   const uint4 *__restrict__ a, int32_t row_vecs, int32_t *__restrict__ cursors,
                   int32_t *__restrict__ pos, uint4 *__restrict__ xg) {
    const int64_t p = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (p >= pairs) return;
    const int lane = threadIdx.x & 31;
    int32_t slot = -1;
    if (lane == 0) {
        const int32_t e = ids[p];
        if (e >= 0 && e < experts && counts[e] <= max_rows) slot = atomicAdd(cursors + e, 1);
        pos[p] = slot;
    }
    slot = __shfl_sync(0xFFFFFFFFu, slot, 0);
    if (slot < 0) return;
    const uint4 *src = a + (p / topk) * row_vecs;
    uint4 *dst = xg + (int64_t)slot * row_vecs;
    for (int v = lane; v < row_vecs; v += 32) dst[v] = __ldg(src + v);
}

// One warp per token: 8 output columns (one 16-byte vector) per lane per step.
__global__ void __launch_bounds__(kThreads)
moe_combine_kernel(const int32_t *__restrict__ pos, const float *__restrict__ weights,
                   int32_t topk, int64_t tokens, const uint4 *__restrict__ y, int32_t row_vecs,
                   uint4 *__restrict__ out) {
    const int64_t m = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (m >= tokens) return;
    const int lane = threadIdx.x & 31;
    for (int v = lane; v < row_vecs; v += 32) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < topk; ++j) {
            const int32_t s = __ldg(pos + m * topk + j);
            if (s < 0) continue;
            const float w = __ldg(weights + m * topk + j);
            const uint4 q = __ldg(y + (int64_t)s * row_vecs + v);
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, __uint_as_float(words[i] << 16)));
                acc[2 * i + 1] =
                    __fadd_rn(acc[2 * i + 1], __fmul_rn(w, __uint_as_float(words[i] & 0xFFFF0000u)));
            }
        }
        uint4 o;
        o.x = pack_bf16x2_rn(acc[0], acc[1]);
        o.y = pack_bf16x2_rn(acc[2], acc[3]);
        o.z = pack_bf16x2_rn(acc[4], acc[5]);
        o.w = pack_bf16x2_rn(acc[6], acc[7]);
        out[m * row_vecs + v] = o;
    }
}

}  // namespace

MoeWorkspace moe_workspace_layout(int64_t tokens, int64_t topk, int64_t experts, int64_t n,
                                  int64_t k) {
    auto up = [](uint64_t x) { return (x + 255u) & ~(uint64_t)255u; };
    const uint64_t pairs = (uint64_t)tokens * (uint64_t)topk;
    MoeWorkspace w;
    w.counts = 0;
    w.cursors = up(w.counts + 4u * (uint64_t)experts);
    w.offsets = up(w.cursors + 4u * (uint64_t)experts);
    w.pos = up(w.offsets + 8u * (uint64_t)(experts + 1));
    w.xg = up(w.pos + 4u * pairs);
    w.act = up(w.xg + 2u * pairs * (uint64_t)k);
    w.y = up(w.act + 2u * pairs * (uint64_t)n);
    w.total = up(w.y + 2u * pairs * (uint64_t)k);
    return w;
}

cudaError_t launch_mx_moe_forward(const uint16_t *a, const int32_t *topk_ids,
                                  const float *topk_weights, int64_t tokens, int64_t topk,
                                  int64_t experts, int64_t max_rows, const uint8_t *w1_packed,
                                  const uint8_t *w1_scales, const uint8_t *w2_packed,
                                  const uint8_t *w2_scales, int64_t n, int64_t k, void *workspace,
                                  uint16_t *out, int32_t *status, cudaStream_t stream) {
    const MoeWorkspace L = moe_workspace_layout(tokens, topk, experts, n, k);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *cursors = reinterpret_cast<int32_t *>(ws + L.cursors);
    int64_t *offsets = reinterpret_cast<int64_t *>(ws + L.offsets);
    int32_t *pos = reinterpret_cast<int32_t *>(ws + L.pos);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + L.act);
    uint16_t *y = reinterpret_cast<uint16_t *>(ws + L.y);
    const int64_t pairs = tokens * topk;
    cudaError_t err = cudaMemsetAsync(counts, 0, (size_t)experts * 4, stream);
    if (err != cudaSuccess) return err;
    {
        const int64_t blocks = (pairs + kThreads - 1) / kThreads;
        const int grid = (int)(blocks < 4096 ? blocks : 4096);
        moe_count_kernel<<<grid, kThreads, 0, stream>>>(topk_ids, pairs, (int32_t)experts, counts,
                                                         status);
    }
    moe_scan_kernel<<<1, kScanThreads, 0, stream>>>(counts, (int32_t)experts, max_rows, offsets,
                                                    cursors, status);
    const int32_t k_vecs = (int32_t)(k / 8);
    moe_scatter_kernel<<<(unsigned)((pairs + kWarps - 1) / kWarps), kThreads, 0, stream>>>(
        topk_ids, pairs, (int32_t)topk, (int32_t)experts, max_rows, counts,
        reinterpret_cast<const uint4 *>(a), k_vecs, cursors, pos, reinterpret_cast<uint4 *>(xg));
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    err = launch_mx_moe_gate_up(xg, offsets, experts, max_rows, pairs, w1_packed, w1_scales, n, k,
                                act, status, stream);
    if (err != cudaSuccess) return err;
    err = launch_mx_moe_gemm(act, offsets, experts, max_rows, pairs, w2_packed, w2_scales, k, n, y,
                             status, stream);
    if (err != cudaSuccess) return err;
    moe_combine_kernel<<<(unsigned)((tokens + kWarps - 1) / kWarps), kThreads, 0, stream>>>(
        pos, topk_weights, (int32_t)topk, tokens, reinterpret_cast<const uint4 *>(y), k_vecs,
        reinterpret_cast<uint4 *>(out));
    return cudaGetLastError();
}

}  // namespace fp4mx
