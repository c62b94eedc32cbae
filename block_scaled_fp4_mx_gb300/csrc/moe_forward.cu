// moe_forward.cu -- the MoE layer around the MXFP4 expert GEMMs (sm_103a).
//
// The consumer of the unpack on the pages is a whole MoE layer ("vllm-project/vllm
// pull 51583": the CPU test runs ops.fused_experts_cpu with MXFP4 experts):
// tokens pick top-k experts, each expert runs gate/up GEMM -> silu(gate) * up ->
// down GEMM, and a token's output is the weighted sum over its slots. Here:
//   1. moe_route_kernel   histogram of the slots' expert ids (bad ids flagged), and
//                         in the last block to finish the exclusive prefix ->
//                         per-expert row offsets and cursors;
//   2. moe_scatter_kernel each valid slot takes a row of its expert's segment and
//                         copies its token's activations there (one warp per slot);
//   3. gate/up GEMM       the tensor-memory GEMM in gate/up mode: act = bf16(silu(g) * u);
//   4. down GEMM          the same kernel: y = bf16(act @ W2_e^T);
//   5. moe_combine_kernel out[m] = bf16(sum_j w[m, j] * y[row of slot j]) in fp32,
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

// Histogram of the slots' expert ids, then (in the last block to finish) the
// exclusive prefix -> per-expert row offsets and scatter cursors. Each block counts
// into shared memory first (one global atomic per expert and block); the block
// that takes the last ticket scans. No block waits for another: the ticket only
// decides which one scans. An expert with more rows than the capacity is flagged;
// the scatter then drops its slots. counts[] and *ticket are zero on entry.
constexpr int kLocalExperts = 4096;  // shared-memory histogram up to this many experts
__global__ void __launch_bounds__(kThreads)
moe_route_kernel(const int32_t *__restrict__ ids, int64_t pairs, int32_t experts, int64_t max_rows,
                 int32_t *__restrict__ counts, uint32_t *__restrict__ ticket,
                 int64_t *__restrict__ offsets, int32_t *__restrict__ cursors,
                 int32_t *__restrict__ status) {
    extern __shared__ int32_t hist[];  // experts entries when experts <= kLocalExperts
    __shared__ int64_t part[kThreads];
    __shared__ bool last;
    const int t = threadIdx.x;
    const bool local = experts <= kLocalExperts;
    if (local)
        for (int e = t; e < experts; e += kThreads) hist[e] = 0;
    __syncthreads();
    for (int64_t p = (int64_t)blockIdx.x * kThreads + t; p < pairs; p += (int64_t)gridDim.x * kThreads) {
        const int32_t e = ids[p];
        if (e < 0 || e >= experts)
            atomicExch(status, FP4_ERR_INDEX);
        else if (local)
            atomicAdd(hist + e, 1);
        else
            atomicAdd(counts + e, 1);
    }
    __syncthreads();
    // one block (a decode-sized batch): its shared histogram is the whole count, so it
    // stores the counts and scans them itself, with no global atomics, fence or ticket
    const bool single = gridDim.x == 1 && local;
    if (single) {
        for (int e = t; e < experts; e += kThreads) counts[e] = hist[e];
    } else {
        if (local)
            for (int e = t; e < experts; e += kThreads)
                if (hist[e] != 0) atomicAdd(counts + e, hist[e]);
        __threadfence();  // this block's counts are visible before its ticket
        __syncthreads();
        if (t == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
        __syncthreads();
        if (!last) return;
        __threadfence();
    }
    // thread t sums a contiguous run of experts, the block scans the run sums
    const int per = (experts + kThreads - 1) / kThreads;
    const int e0 = t * per;
    const int e1 = e0 + per < experts ? e0 + per : experts;
    auto count_of = [&](int e) -> int32_t { return single ? hist[e] : __ldcg(counts + e); };
    int64_t sum = 0;
    for (int e = e0; e < e1; ++e) sum += count_of(e);
    part[t] = sum;
    __syncthreads();
    for (int d = 1; d < kThreads; d <<= 1) {  // inclusive Hillis-Steele scan
        const int64_t v = t >= d ? part[t - d] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int64_t run = part[t] - sum;  // exclusive prefix of this thread's run
    for (int e = e0; e < e1; ++e) {
        const int32_t c = count_of(e);
        offsets[e] = run;
        cursors[e] = (int32_t)run;
        if (c > max_rows) atomicExch(status, FP4_ERR_SHAPE);
        run += c;
    }
    if (t == kThreads - 1) offsets[experts] = part[t];
}

// One warp per slot p = m * topk + j.
constexpr int kScatterVecs = 12;
__global__ void __launch_bounds__(kThreads)
moe_scatter_kernel(const int32_t *__restrict__ ids, int64_t pairs, int32_t topk, int32_t experts,
                   int64_t max_rows, const int32_t *__restrict__ counts,
                   const uint4 *__restrict__ a, int32_t row_vecs, int32_t *__restrict__ cursors,
                   int32_t *__restrict__ pos, uint4 *__restrict__ xg) {
    grid_dependency_wait();  // the route kernel's counts and cursors
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
    // up to twelve 16-byte loads in flight per lane: a whole row of k = 2880 in one
    // memory latency, which is what a decode-sized batch (few slots) waits for
    for (int v0 = lane; v0 < row_vecs; v0 += kScatterVecs * 32) {
        uint4 r[kScatterVecs];
#pragma unroll
        for (int i = 0; i < kScatterVecs; ++i)
            if (v0 + 32 * i < row_vecs) r[i] = __ldg(src + v0 + 32 * i);
#pragma unroll
        for (int i = 0; i < kScatterVecs; ++i)
            if (v0 + 32 * i < row_vecs) dst[v0 + 32 * i] = r[i];
    }
}

// One warp per (token, chunk of chunk_vecs 16-byte vectors of its row): 8 output
// columns (one vector) per lane per step. With many tokens a chunk is the whole row
// (a warp per token); with few, the row is split so that enough warps are in flight
// (each step's loads wait a memory latency). The token's slot rows and weights are
// read by every warp of the token; up to kCombineSlots slots all vectors of a step
// are loaded before the sum, which still adds slot 0, 1, ... in that order (a slot
// dropped by the scatter is skipped, not added as zero).
constexpr int kCombineSlots = 8;
__device__ __forceinline__ void combine_add(float (&acc)[8], float w, const uint4 &q) {
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, __uint_as_float(words[i] << 16)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, __uint_as_float(words[i] & 0xFFFF0000u)));
    }
}

__device__ __forceinline__ uint4 combine_pack(const float (&acc)[8]) {
    uint4 o;
    o.x = pack_bf16x2_rn(acc[0], acc[1]);
    o.y = pack_bf16x2_rn(acc[2], acc[3]);
    o.z = pack_bf16x2_rn(acc[4], acc[5]);
    o.w = pack_bf16x2_rn(acc[6], acc[7]);
    return o;
}

__global__ void __launch_bounds__(kThreads)
moe_combine_kernel(const int32_t *__restrict__ pos, const float *__restrict__ weights,
                   int32_t topk, int64_t tokens, const uint4 *__restrict__ y, int32_t row_vecs,
                   int32_t chunk_vecs, int32_t chunks, uint4 *__restrict__ out) {
    grid_dependency_wait();  // the down GEMM's rows
    const int64_t wid = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t m = wid / chunks;
    if (m >= tokens) return;
    const int v0 = (int)(wid - m * chunks) * chunk_vecs;
    const int v1 = v0 + chunk_vecs < row_vecs ? v0 + chunk_vecs : row_vecs;
    const int lane = threadIdx.x & 31;
    if (topk > kCombineSlots) {
        for (int v = v0 + lane; v < v1; v += 32) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < topk; ++j) {
                const int32_t s = __ldg(pos + m * topk + j);
                if (s >= 0) combine_add(acc, __ldg(weights + m * topk + j), __ldg(y + (int64_t)s * row_vecs + v));
            }
            out[m * row_vecs + v] = combine_pack(acc);
        }
        return;
    }
    // lane j < topk reads slot j's row and weight; every lane takes them by shuffle
    int32_t s_lane = -1;
    float w_lane = 0.f;
    if (lane < topk) {
        s_lane = __ldg(pos + m * topk + lane);
        w_lane = __ldg(weights + m * topk + lane);
    }
    const uint4 *rows[kCombineSlots];
    float w[kCombineSlots];
#pragma unroll
    for (int j = 0; j < kCombineSlots; ++j) {
        const int32_t s = __shfl_sync(0xFFFFFFFFu, s_lane, j);
        w[j] = __shfl_sync(0xFFFFFFFFu, w_lane, j);
        rows[j] = (j < topk && s >= 0) ? y + (int64_t)s * row_vecs : nullptr;
    }
    for (int v = v0 + lane; v < v1; v += 32) {
        uint4 q[kCombineSlots];
#pragma unroll
        for (int j = 0; j < kCombineSlots; ++j)
            if (rows[j] != nullptr) q[j] = __ldg(rows[j] + v);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kCombineSlots; ++j)
            if (rows[j] != nullptr) combine_add(acc, w[j], q[j]);
        out[m * row_vecs + v] = combine_pack(acc);
    }
}

}  // namespace

MoeWorkspace moe_workspace_layout(int64_t tokens, int64_t topk, int64_t experts, int64_t n,
                                  int64_t k) {
    auto up = [](uint64_t x) { return (x + 255u) & ~(uint64_t)255u; };
    const uint64_t pairs = (uint64_t)tokens * (uint64_t)topk;
    MoeWorkspace w;
    w.counts = 0;
    w.ticket = w.counts + 4u * (uint64_t)experts;  // zeroed together with the counts
    w.cursors = up(w.ticket + 4u);
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
    uint32_t *ticket = reinterpret_cast<uint32_t *>(ws + L.ticket);
    int32_t *cursors = reinterpret_cast<int32_t *>(ws + L.cursors);
    int64_t *offsets = reinterpret_cast<int64_t *>(ws + L.offsets);
    int32_t *pos = reinterpret_cast<int32_t *>(ws + L.pos);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + L.act);
    uint16_t *y = reinterpret_cast<uint16_t *>(ws + L.y);
    const int64_t pairs = tokens * topk;
    const int64_t blocks = (pairs + kThreads - 1) / kThreads;
    cudaError_t err = cudaSuccess;
    // the counters and the ticket start at zero when several blocks add into them; a
    // single block (a decode-sized batch) stores its counts and takes no ticket
    if (blocks > 1 || experts > kLocalExperts) {
        err = cudaMemsetAsync(counts, 0, (size_t)(experts + 1) * 4, stream);  // + ticket
        if (err != cudaSuccess) return err;
    }
    {
        const int grid = (int)(blocks < 1024 ? blocks : 1024);
        const size_t hist_bytes = experts <= kLocalExperts ? (size_t)experts * 4 : 0;
        moe_route_kernel<<<grid, kThreads, hist_bytes, stream>>>(
            topk_ids, pairs, (int32_t)experts, max_rows, counts, ticket, offsets, cursors, status);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    // The kernels after the route kernel start while the one before them finishes
    // (programmatic dependent launch) and wait for it where they read its output:
    // scatter and combine on entry, the GEMMs in their activation loads. Everything
    // else they read is older than the route kernel, which starts only after all
    // earlier work in the stream, and so are the last readers of what they write.
    const int32_t k_vecs = (int32_t)(k / 8);
    err = launch_kernel(moe_scatter_kernel, dim3((unsigned)((pairs + kWarps - 1) / kWarps)),
                        dim3(kThreads), 0, stream, true, topk_ids, pairs, (int32_t)topk,
                        (int32_t)experts, max_rows, (const int32_t *)counts,
                        reinterpret_cast<const uint4 *>(a), k_vecs, cursors, pos,
                        reinterpret_cast<uint4 *>(xg));
    if (err != cudaSuccess) return err;
    err = launch_mx_moe_gate_up(xg, offsets, experts, max_rows, pairs, w1_packed, w1_scales, n, k,
                                act, status, stream, true);
    if (err != cudaSuccess) return err;
    err = launch_mx_moe_gemm(act, offsets, experts, max_rows, pairs, w2_packed, w2_scales, k, n, y,
                             status, stream, true);
    if (err != cudaSuccess) return err;
    // warps per token: enough to keep ~16 warps per SM in flight, at least 32 vectors
    // (one per lane) per warp; a warp per token once tokens alone fill the GPU
    int sms = 0, device = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        sms = 0;
    const int64_t want = (int64_t)(sms > 0 ? sms : 148) * 16;
    const int32_t max_chunks = (k_vecs + 31) / 32;
    int32_t chunks = (int32_t)((want + tokens - 1) / tokens);
    chunks = chunks < 1 ? 1 : (chunks > max_chunks ? max_chunks : chunks);
    const int32_t chunk_vecs = ((k_vecs + chunks - 1) / chunks + 31) / 32 * 32;
    chunks = (k_vecs + chunk_vecs - 1) / chunk_vecs;
    const int64_t combine_warps = tokens * chunks;
    return launch_kernel(moe_combine_kernel, dim3((unsigned)((combine_warps + kWarps - 1) / kWarps)),
                         dim3(kThreads), 0, stream, true, (const int32_t *)pos, topk_weights,
                         (int32_t)topk, tokens, reinterpret_cast<const uint4 *>(y), k_vecs,
                         chunk_vecs, chunks, reinterpret_cast<uint4 *>(out));
}

}  // namespace fp4mx
