// mx_moe_gemm.cu -- grouped MoE GEMM with MXFP4 expert weights (sm_103a): a
// persistent tcgen05 kernel whose decoded weight operand lives in tensor memory.
//
// The consumer the pages' unpack serves: "vllm-project/vllm pull 51583",
// "Motivation" and the comments on the unpack_B loop -- the CPU MoE GEMM
// (ops.fused_experts_cpu with CPUQuantMethod.MXFP4) unpacks a tile of MXFP4
// weights to bf16 and multiplies it with bf16 activations. Here the bf16 weights
// never reach HBM (0.53 bytes per weight are read instead of 2 + 2 for unpack,
// store and reload) and never touch shared memory either: bf16 activations x
// MXFP4 weights decoded to the values fp4_mx_unpack gives them, fp32 accumulation
// in tensor memory, bf16 out. (A zero code with the sign bit set stays -0.0 here:
// as a factor it adds nothing to a sum either way, and skipping the +0.0 fix saves
// two of the decode's ~15 integer operations per 8 codes, 5-8% of the decode-time
// GEMM's time on GB300.) The operands are swapped so that the decoded weights
// can be the tensor core's A operand, which tcgen05.mma reads from tensor memory:
//     D[weight row][token] = sum_k W[weight row][k] * X[token][k],
// 128 weight rows per M tile (one per TMEM lane), the expert's tokens as N. A
// decoder thread owns one weight row of a K slice (64 wide, or 128 = two 64-wide
// sub-slices in the configurations for up to 128 tokens): it decodes the row's 64
// codes of a sub-slice (two E8M0 blocks) in registers and writes them with one
// tcgen05.st into its own TMEM lane, 32 columns of bf16 pairs. There is no
// shared-memory copy of the decoded tile, no generic-to-async proxy fence, and the
// ring of decoded slices can be deep because tensor memory is otherwise idle.
//
// One CTA per SM walks a static list of work items (expert, token slab, tile of
// weight rows; consecutive items share the expert's activation rows in L2). With
// 256-token slabs an expert's last slab may hold up to 64 more tokens: each K
// step then issues a second MMA (N = 16..64) on the same decoded weights into
// accumulator columns 256.., so an expert of 257..320 rows (or 513..576, ...)
// needs no extra item and no extra decode of its weights. A
// stage of the operand ring holds one K slice: its activation tile(s) in shared
// memory and its decoded weights in tensor memory, under one "full" barrier (the
// TMA bytes plus one arrival per decoder warp) and one "empty" barrier (the MMA
// commit):
//   - one TMA thread streams the activation tiles (kTok tokens x 64 bf16 per
//     sub-slice, 128-byte swizzle, the MMA's B operand); inside the MoE layer the
//     kernel is a dependent launch that may start while the kernel writing the
//     activations finishes, and this thread alone waits for that kernel;
//   - another streams the packed codes of the weight slices (rows x 32 bytes, or
//     x 64 bytes with the 64-byte swizzle for slices of 128, of a 2-D uint8 tensor
//     map) through a ring of its own;
//   - 16 decoder warps: warp w writes TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31,
//     so 4 warps cover one 128-row M tile; the kMTw tiles of a slice take 4 kMTw
//     warps and the remaining warps form further groups that own every kGroups-th
//     slice; each thread loads its row's E8M0 bytes from global memory one slice
//     ahead and takes the packed codes from shared memory;
//   - MMA issuers: tcgen05.mma kind::f16 (M = 128, N = kTok, K = 16, A from TMEM),
//     one asm block per slice that also probes the next stage's barrier ahead of
//     the MMAs. A thread gets one tcgen05.mma issued per ~120-200 SM cycles,
//     whatever N is (measured on GB300), and issuers in different warps overlap:
//     one thread per item with one 256-token tile, one per 128-row tile with two
//     tiles, and four (each summing a quarter of the K slices into a partial
//     accumulator) for decode-time batches;
//   - an epilogue warpgroup reads finished accumulators with tcgen05.ld (a thread
//     holds one weight row, i.e. one output column, for 32 tokens), rounds to
//     bf16, pairs neighbouring columns with one lane exchange and stores 4-byte
//     words: the 32 lanes of a warp write two 64-byte runs of two output rows.
//     In the gate/up "halves" layout a warp's lanes i and 16 + i hold the gate
//     and up rows of one output column, so silu(gate) * up needs one xor-16 lane
//     exchange per pair of tokens and no shared memory.
//
// Every mbarrier wait is bounded: a wait that runs out sets an abort flag that
// every role polls, and the launch reports FP4_ERR_TIMEOUT in the status word
// after the MMA issuers have drained their tensor-core work and TMEM is freed. The
// decoders, the epilogue and the TMA threads wait with a suspend-time hint
// (they sleep instead of spinning, which leaves the issue slots to the MMA
// thread and the decoders that work: 5-8% faster); the MMA thread of the
// 256-token configurations polls, the issuers of the others sleep too.
#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"
#include "moe_act.cuh"
#include "tc_sm103.cuh"

namespace fp4mx {
namespace {

constexpr int kWM = 128;  // weight rows per M tile (TMEM lanes)
constexpr int kK = 64;    // K per slice
constexpr uint32_t kTmemCols = 512;
constexpr int kXBox = 128;                   // activation rows per TMA box
constexpr int kPrefixExperts = 1024;         // largest expert count of the compact item list
constexpr int kXBoxBytes = kXBox * kK * 2;  // 16 KiB
constexpr int kXExtBox = 64;                // activation rows per box of a slab's extension
constexpr int kXExtBytes = kXExtBox * kK * 2;  // 8 KiB

template <int kTok_, int kMTw_, int kAccBufs_, int kStages_, int kStagesRaw_, bool kGateUp_ = false,
          int kExt_ = 0, int kDecodeWarps_ = 16, int kEpiWarps_ = 4, bool kMmaSleep_ = false,
          int kIssuers_ = 1, int kKS_ = kK>
struct TmemCfg {
    // K per slice: 64, or 128 = two 64-wide sub-slices per stage (two activation boxes,
    // 128 codes per decoder thread, eight MMAs per commit) where a slice's handshakes
    // cost more than its work: with decode-time batches the pipeline spends ~2,000
    // cycles per slice and decoder group even with no decode or MMA (measured on GB300)
    static constexpr int kKS = kKS_;
    static constexpr int kSub = kKS_ / kK;
    // MMA issuing threads. One thread issues tcgen05.mma at a fixed rate per
    // instruction whatever N is (measured on GB300: ~145 cycles per 128 x 16 x 16
    // MMA, ~190 with 16 busy warps beside it, and the rate scales with the number
    // of issuing threads in different warps), so with few tokens per expert one
    // issuer cannot keep up with the decoders. With kIssuers = 4 the four epilogue
    // warps (one per SM sub-partition) issue too: issuer i takes the K slices of
    // decoder group i into a partial accumulator of its own, and at the end of an item
    // each of the four warps sums the four partials (in a fixed order) for its TMEM
    // lane quarter. (Issuers in warps of their own, with the epilogue apart and two
    // sets of partials, measured slower: 26 warps leave 72 registers a thread.)
    static constexpr int kIssuers = kIssuers_;
    // the MMA thread waits for full stages asleep (suspend-time hint) instead of
    // polling: where a slice holds little MMA work, a polling MMA thread takes the
    // issue slots of the decoder warps that share its SM sub-partition
    static constexpr bool kMmaSleep = kMmaSleep_;
    // warp roles: decoders, epilogue (a multiple of 4: kEpiWarps / 4 warps share
    // each TMEM lane quarter and take its chunks in turn), the activation TMA
    // thread, the weight TMA thread and the MMA thread
    static constexpr int kDecodeWarps = kDecodeWarps_;
    static constexpr int kEpiWarp0 = kDecodeWarps;
    static constexpr int kEpiWarps = kEpiWarps_;
    static constexpr int kTmaXWarp = kEpiWarp0 + kEpiWarps;
    static constexpr int kTmaWWarp = kTmaXWarp + 1;
    // with one accumulator per item, one MMA warp per 128-row weight tile: each issues
    // its tile's MMAs into its own accumulator columns, so two tiles take two issuers
    static constexpr int kTileIssuers = kIssuers == 1 ? kMTw_ : 1;
    static constexpr int kMmaWarp = kIssuers == 1 ? kTmaWWarp + 1 : -1;
    static constexpr int kThreads = (kIssuers == 1 ? kMmaWarp + kTileIssuers : kTmaWWarp + 1) * 32;
    static constexpr int kTok = kTok_;        // tokens per item (MMA N)
    // an expert's last slab may take up to kExt more tokens (a second MMA per K step
    // into accumulator columns kTok.., same decoded weights), so that rows just past
    // a multiple of kTok need no extra item
    static constexpr int kExt = kExt_;
    static constexpr int kMTw = kMTw_;        // 128-row weight tiles per item
    static constexpr int kAccBufs = kAccBufs_;  // accumulator buffers
    // gate/up mode: the epilogue writes silu(gate) * up. With two weight tiles
    // (kMTw = 2) they are gate rows n0.. and up rows n_out + n0..; with one tile
    // ("halves") it holds 64 gate rows and the 64 matching up rows, interleaved
    // by 16 so that every warp's 32 TMEM lanes hold a gate row and its up row 16
    // lanes apart: lanes 32q + i and 32q + 16 + i (i < 16) are gate and up rows
    // n0 + 16q + i, and the epilogue pairs them with one lane exchange
    static constexpr bool kGateUp = kGateUp_;
    static constexpr bool kHalves = kGateUp && kMTw_ == 1;
    // a stage of the operand ring holds one slice's activation tile (shared memory)
    // and its decoded weights (tensor memory) under one full and one empty barrier
    static constexpr int S = kStages_, SR = kStagesRaw_;
    static constexpr int kWRows = kWM * kMTw;
    static constexpr int kTileCols = kHalves ? kWM / 2 : kGateUp ? kWM : kWRows;  // output columns per item
    static constexpr int kBoxRows = kHalves ? kWM / 2 : kGateUp ? kWM : kWRows;  // rows per weight TMA box
    static constexpr int kWarpsPerSlice = 4 * kMTw;
    static constexpr int kGroups = kDecodeWarps / kWarpsPerSlice;
    // tensor memory: accumulator buffers (kIssuers partials each), then the ring of
    // decoded slices
    static constexpr int kAccCols = kMTw * (kTok + kExt);
    static constexpr int kAColBase = kAccBufs * kIssuers * kAccCols;
    static constexpr int kAStageCols = kMTw * (kKS / 2);
    // shared memory from a 1024-byte aligned base
    static constexpr int kXSubBytes = (kTok + kExt) * kK * 2;  // one 64-wide sub-slice
    static constexpr int kXBytes = kSub * kXSubBytes;
    static constexpr int kRawBytes = kWRows * (kKS / 2);
    static constexpr int kOffX = 0;
    static constexpr int kOffRaw = kOffX + S * kXBytes;
    static constexpr int kOffBar = kOffRaw + SR * kRawBytes;
    static constexpr int kNumBars = 2 * (S + SR) + 2 * kAccBufs + 1;
    // per-expert prefix of live token slabs (the compact item list), after the
    // barriers, the TMEM address word and the abort flag
    static constexpr int kOffPrefix = kOffBar + 8 * kNumBars + 16;
    // the scaled byte tables of all 256 E8M0 values (16 bytes each), built once per
    // CTA, where shared memory has room: a decoder thread then loads its two blocks'
    // tables instead of building them
    static constexpr int kOffTab = (kOffPrefix + 4 * (kPrefixExperts + 1) + 15) & ~15;
    static constexpr bool kSmemTable = 1024 + kOffTab + 4096 <= 232448;
    static constexpr int kSmemBytes = 1024 + (kSmemTable ? kOffTab + 4096 : kOffTab);
    static_assert(kTok == 64 || kTok == 128 || kTok == 256, "MMA N");
    static_assert(kKS == kK || (kKS == 2 * kK && kExt == 0 && (kIssuers == 4 || kMTw == 2)),
                  "K per slice");
    static_assert(kMTw == 1 || kMTw == 2, "weight tiles per item");
    static_assert(kExt == 0 || (kExt == kXExtBox && kMTw == 1 && kTok == 256), "slab extension");
    static_assert(kDecodeWarps % kWarpsPerSlice == 0, "decoder groups");
    static_assert(kEpiWarps % 4 == 0 && kDecodeWarps % 4 == 0, "warps per TMEM lane quarter");
    // a decoder group's ring positions advance by kGroups per slice and wrap with
    // one subtraction, so neither ring may be shorter than kGroups
    static_assert(kGroups <= S && kGroups <= SR, "ring depth below the decoder group count");
    // one issuer: accumulators and the whole ring fit; several: 16-column partials and
    // the whole ring fit, and 64-column partials leave at least 8 ring stages
    static_assert(kIssuers == 1 ? kAColBase + S * kAStageCols <= (int)kTmemCols
                                : kIssuers * 16 + S * kAStageCols <= (int)kTmemCols &&
                                      kIssuers * 64 + 8 * 32 <= (int)kTmemCols &&
                                      kIssuers * 32 + 4 * kAStageCols <= (int)kTmemCols,
                  "tensor memory columns");
    static_assert(kSmemBytes <= 232448, "shared memory per block");
    // several issuers: four (one per decoder group and epilogue warp), one weight tile,
    // one accumulator buffer, ring stages in whole rounds of the four groups. The last
    // is what keeps the parity waits sound: stage s is then used by one decoder group
    // and one issuer only, so nobody reaches use u of a stage before use u - 1 is under
    // way. With another ring length a stage's uses pass between groups, a fast waiter
    // can be a whole use ahead, and a parity wait cannot tell phase u from u - 2 (a
    // 7-stage ring faulted on GB300 that way).
    static_assert(kIssuers == 1 || (kIssuers == 4 && kGroups == 4 && kEpiWarps == 4 && kMTw == 1 &&
                                    kAccBufs == 1 && kExt == 0 && S % 4 == 0 && kEpiWarp0 % 4 == 0),
                  "issuer layout");
};

// Up to 64 tokens per expert (decode-time batches): one 128-row weight tile per
// item (more items than SMs several times over), the MMA's N cut to the expert's
// tokens rounded up to 16, activation boxes only as tall as the capacity, four MMA
// issuers with partial accumulators of the capacity rounded up to 16 columns each,
// K slices of 128 in a ring of 4 stages (one per decoder group) and a weight ring of
// 12. (With a capacity of 33 to 64 it measured 12-15% faster than the 128-token
// configuration on 32 x 2880 x 2880, 2-3% slower on 32 x 5760 x 2880, and 4% faster
// over a 64-token MoE layer step.)
using CfgTiny = TmemCfg<64, 1, 1, 4, 12, false, 0, 16, 4, true, 4, 2 * kK>;
// Up to 128 tokens per expert: two weight tiles per item (one MMA warp each), one
// accumulator buffer, K slices of 128 in a ring of 2 stages (one per decoder group):
// 0.130 against 0.137 ms with slices of 64 for 32 x 128 tokens x 5760 x 2880.
using CfgSmall = TmemCfg<128, 2, 1, 2, 4, false, 0, 16, 4, true, 1, 2 * kK>;
// More tokens: 256 tokens per item (an expert's last slab up to 320) against one
// weight tile; 12 decoder warps (3 groups) and 8 epilogue warps, so that the
// single accumulator is read out twice as fast at the end of an item.
using CfgLarge = TmemCfg<256, 1, 1, 5, 5, false, 64, 12, 8>;
// Gate/up GEMM of the MoE layer with the activation function in the epilogue.
using CfgGateUp = TmemCfg<128, 2, 1, 2, 4, true, 0, 16, 4, true, 1, 2 * kK>;
// The same for up to 64 tokens per expert: gate and up halves of one weight tile.
using CfgGateUpTiny = TmemCfg<64, 1, 1, 4, 12, true, 0, 16, 4, true, 4, 2 * kK>;
// The same with 256-token slabs (the last up to 320): gate and up halves of one
// weight tile.
using CfgGateUpLarge = TmemCfg<256, 1, 1, 5, 5, true, 64, 12, 8>;

// MXFP4 decode of one word for use as a matrix operand only: every code takes its
// sign, so code 8 comes out as -0.0 instead of +0.0. A product with -0.0 is a zero
// like one with +0.0 and adds nothing to a sum, so a dot product over these values
// equals the one over the exact decode (only an all-zero sum may differ in the sign
// of its zero). Two integer operations fewer per word than mx_decode_word (lookup_word
// keeps only bit 3 of each sign nibble).
__device__ __forceinline__ uint4 mx_decode_word_operand(uint32_t w, const ByteTable &t) {
    return lookup_word(w, t, w);
}

struct Item {
    int64_t row_begin, rows, m0;
    int expert, n0;
    bool live, bad;
};

// Item t of the dense list: weight tile t % n_tiles (fastest), token slab, expert
// (every expert gets the slabs max_rows needs; those past its rows are dead).
__device__ __forceinline__ Item item_at(int64_t t, int n_tiles, int slabs, int tok, int cols,
                                        const int64_t *__restrict__ offsets, int64_t max_rows,
                                        int64_t total_rows) {
    Item it;
    const int64_t rest = t / n_tiles;
    it.n0 = (int)(t - rest * n_tiles) * cols;
    it.expert = (int)(rest / slabs);
    it.m0 = (rest - (int64_t)it.expert * slabs) * tok;
    it.row_begin = __ldg(offsets + it.expert);
    const int64_t end = __ldg(offsets + it.expert + 1);
    it.rows = end - it.row_begin;
    it.bad = it.row_begin < 0 || it.rows < 0 || it.rows > max_rows || end > total_rows;
    it.live = !it.bad && it.m0 < it.rows;
    return it;
}

// Item t of the compact list (live items only): global slab s = t / n_tiles, found
// in the per-expert slab prefix by binary search (an expert with no slab has the
// same prefix as the next one; the last expert with prefix <= s owns slab s).
__device__ __forceinline__ Item item_compact(int64_t t, int n_tiles, int tok, int cols,
                                             const int32_t *prefix, int experts,
                                             const int64_t *__restrict__ offsets) {
    Item it;
    const int64_t s = t / n_tiles;
    it.n0 = (int)(t - s * n_tiles) * cols;
    int lo = 0, hi = experts;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= s) lo = mid; else hi = mid;
    }
    it.expert = lo;
    it.m0 = (s - prefix[lo]) * tok;
    it.row_begin = __ldg(offsets + lo);
    it.rows = __ldg(offsets + lo + 1) - it.row_begin;
    it.live = true;
    it.bad = false;
    return it;
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
mx_moe_gemm_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_x_ext,
                        const __grid_constant__ CUtensorMap map_w,
                        const int64_t *__restrict__ expert_offsets,
                        const uint8_t *__restrict__ w_scales, int32_t experts, int64_t max_rows,
                        int64_t total_rows, int32_t n_rows, int32_t n_out, int32_t k,
                        int32_t x_box_rows, uint16_t *__restrict__ out,
                        int32_t *__restrict__ status) {
    // n_rows: weight rows per expert (2 n_out in gate/up mode); n_out: output columns;
    // x_box_rows: rows of map_x's box (kXBox, or fewer with 64-token items)
    constexpr int kTok = C::kTok, kMTw = C::kMTw, S = C::S, SR = C::SR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_addr(smem);
    const uint32_t x_ring = base + C::kOffX, raw_ring = base + C::kOffRaw;
    const uint32_t bars = base + C::kOffBar;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (S + s); };
    auto full_raw = [&](int s) { return bars + 8u * (2 * S + s); };
    auto empty_raw = [&](int s) { return bars + 8u * (2 * S + SR + s); };
    auto acc_full = [&](int b) { return bars + 8u * (2 * (S + SR) + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (2 * (S + SR) + C::kAccBufs + b); };
    const uint32_t drain_bar = bars + 8u * (2 * (S + SR) + 2 * C::kAccBufs);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + 8 * C::kNumBars);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + C::kOffPrefix);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int n_tiles = (n_out + C::kTileCols - 1) / C::kTileCols;
    const int slabs = (int)((max_rows + kTok - 1) / kTok);
    const int nk = (k + C::kKS - 1) / C::kKS;  // K slices
    const int scale_pitch = k / 32;
    // up to kPrefixExperts experts the CTAs walk live items only; beyond, every
    // expert gets max_rows' slabs and dead items are skipped
    const bool compact = experts <= kPrefixExperts;
    if (compact && warp == 1) {
        // lane l owns experts [l * per, (l + 1) * per): its run of slab counts, then a
        // warp scan of the run totals; an expert with inconsistent offsets gets no slab
        const int per = (experts + 31) / 32;
        const int e0 = lane * per, e1 = e0 + per < experts ? e0 + per : experts;
        int32_t run = 0;
        for (int e = e0; e < e1; ++e) {
            const int64_t rb = __ldg(expert_offsets + e), end = __ldg(expert_offsets + e + 1);
            const int64_t rows = end - rb;
            const bool ok = rb >= 0 && rows >= 0 && rows <= max_rows && end <= total_rows;
            if (!ok && blockIdx.x == 0) atomicExch(status, FP4_ERR_SHAPE);
            prefix[e] = run;
            // slabs of kTok tokens, the last one up to kTok + kExt
            const int64_t n_slabs = rows <= 0 ? 0 : (rows - C::kExt + kTok - 1) / kTok;
            run += ok ? (int32_t)(n_slabs > 1 ? n_slabs : (rows > 0 ? 1 : 0)) : 0;
        }
        int32_t incl = run;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += v;
        }
        for (int e = e0; e < e1; ++e) prefix[e] += incl - run;
        if (lane == 31) prefix[experts] = incl;
    }
    // tokens of an item: kTok, or what is left of the expert's rows; in the compact
    // list an expert's last slab takes up to kTok + kExt
    auto item_tokens = [&](const Item &it) -> int {
        const int64_t left = it.rows - it.m0;  // > 0 for a live item
        if (C::kExt > 0 && compact && left <= kTok + C::kExt) return (int)left;
        return (int)(left < kTok ? left : kTok);
    };
    // MMA N of the first kTok tokens: a slab whose rows fit in 128 takes N = 128 MMAs
    // and one activation box per slice
    auto tok_live = [&](int n_tok) { return (kTok == 256 && n_tok <= 128) ? 128 : kTok; };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            // the activation TMA thread's arrival (with its bytes) and one per decoder warp
            mbar_init(full(s), C::kWarpsPerSlice + 1);
            mbar_init(empty(s), C::kTileIssuers);  // one commit per MMA warp
        }
        for (int s = 0; s < SR; ++s) {
            mbar_init(full_raw(s), 1);
            mbar_init(empty_raw(s), C::kWarpsPerSlice);
        }
        for (int b = 0; b < C::kAccBufs; ++b) {
            mbar_init(acc_full(b), C::kIssuers * C::kTileIssuers);  // one commit per issuer
            mbar_init(acc_empty(b), C::kEpiWarps);
        }
        mbar_init(drain_bar, C::kIssuers * C::kTileIssuers);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
        if (C::kExt > 0)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x_ext)) : "memory");
    }
    if (C::kSmemTable) {
        for (int e = tid; e < 256; e += C::kThreads) {
            const ByteTable t = mx_scaled_table((uint32_t)e);
            st_shared_v4(base + C::kOffTab + 16u * (uint32_t)e, make_uint4(t.lo_a, t.lo_b, t.hi_a, t.hi_b));
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // with several issuers each partial accumulator takes the capacity's columns
    // (x_box_rows) and the ring of decoded slices takes what is left, in whole
    // rounds of the four decoder groups (at most S stages)
    const int acc_stride = C::kIssuers > 1 ? x_box_rows : C::kAccCols;
    const int a_base = C::kIssuers > 1 ? C::kIssuers * acc_stride : C::kAColBase;
    const int s_ring =
        C::kIssuers > 1
            ? ((((int)kTmemCols - a_base) / C::kAStageCols) & ~3) < S
                  ? ((((int)kTmemCols - a_base) / C::kAStageCols) & ~3)
                  : S
            : S;
    const uint32_t tab = base + C::kOffTab;
    const int64_t n_items = compact ? (int64_t)prefix[experts] * n_tiles
                                    : (int64_t)experts * slabs * n_tiles;
    auto item = [&](int64_t t) {
        return compact ? item_compact(t, n_tiles, kTok, C::kTileCols, prefix, experts, expert_offsets)
                       : item_at(t, n_tiles, slabs, kTok, C::kTileCols, expert_offsets, max_rows,
                                 total_rows);
    };

    if (warp < C::kDecodeWarps) {
        // ---- decoders: slice g (counted across this CTA's items) belongs to group g % kGroups ----
        const int quarter = warp & 3;
        const int mt = (warp >> 2) % kMTw;
        const int group = warp / C::kWarpsPerSlice;
        const int r = mt * kWM + quarter * 32 + lane;  // TMEM lane (M row) within the item
        // its row of the packed slice in shared memory: the halves layout takes gate
        // row i from box row i and up row i from box row 64 + i
        const int raw_r = C::kHalves ? (lane >> 4) * (kWM / 2) + quarter * 16 + (lane & 15) : r;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)a_base +
                                   (uint32_t)(mt * (C::kKS / 2));
        bool stop = false;
        uint32_t g0 = 0;  // first slice of the current item
        // ring positions of this group's next slice g (the group's slices are g =
        // group, group + kGroups, ... across items): stage and phase of each ring
        int sr = group % SR, sw = group % s_ring;
        uint32_t pr = (uint32_t)(group / SR) & 1u, pw = (uint32_t)(group / s_ring) & 1u;
        uint32_t g = (uint32_t)group;
        for (int64_t t = blockIdx.x; t < n_items && !stop; t += gridDim.x) {
            const Item it = item(t);
            if (!it.live) continue;
            // the weight row this thread decodes (within the expert) and whether it exists
            const int i_tile = C::kHalves ? quarter * 16 + (lane & 15) : r - mt * kWM;
            const int half = C::kHalves ? lane >> 4 : mt;  // 0 gate, 1 up in gate/up mode
            const int wr = C::kGateUp ? half * n_out + it.n0 + i_tile : it.n0 + r;
            const bool row_ok = C::kGateUp ? it.n0 + i_tile < n_out : wr < n_out;
            const uint8_t *srow = w_scales + ((int64_t)it.expert * n_rows + wr) * scale_pitch;
            // the row's E8M0 bytes of slice kt (kKS / 32 of them); those of the group's
            // next slice are loaded one slice ahead, so their latency hides behind a slice
            auto scale_at = [&](int kt, int h) {
                const int b = (C::kKS / 32) * kt + h;
                return (row_ok && b < scale_pitch) ? ldg_early_u8(srow + b) : 127u;
            };
            const int kt_first = (int)(((uint32_t)group + (uint32_t)C::kGroups -
                                        g0 % (uint32_t)C::kGroups) % (uint32_t)C::kGroups);
            uint32_t next_e[2 * C::kSub];
#pragma unroll
            for (int h = 0; h < 2 * C::kSub; ++h) next_e[h] = scale_at(kt_first, h);
            for (int kt = kt_first; kt < nk; kt += C::kGroups) {
                uint32_t ev[2 * C::kSub];
#pragma unroll
                for (int h = 0; h < 2 * C::kSub; ++h) ev[h] = next_e[h];
                if (kt + C::kGroups < nk) {
#pragma unroll
                    for (int h = 0; h < 2 * C::kSub; ++h) next_e[h] = scale_at(kt + C::kGroups, h);
                }
                const uint32_t e0 = ev[0], e1 = ev[1];
                if (lane == 0 && !mbar_wait_sleep(full_raw(sr), pr)) *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) {  // warp-uniform
                    stop = true;
                    break;
                }
                const uint32_t raw_row = raw_ring + sr * C::kRawBytes + (uint32_t)raw_r * (uint32_t)(C::kKS / 2);
                // 64-byte rows come with the 64-byte swizzle: 16-byte chunk c of row r sits
                // at chunk c ^ (r / 2 % 4), so that 8 consecutive rows' reads of one chunk
                // hit 8 different bank groups
                const uint32_t sw64 = C::kSub == 2 ? (uint32_t)((raw_r >> 1) & 3) : 0u;
                const uint4 w0 = lds_v4(raw_row + 16u * (0u ^ sw64));
                const uint4 w1 = lds_v4(raw_row + 16u * (1u ^ sw64));
                uint4 w2 = w0, w3 = w1;  // the second sub-slice's codes
                if constexpr (C::kSub == 2) {
                    w2 = lds_v4(raw_row + 16u * (2u ^ sw64));
                    w3 = lds_v4(raw_row + 16u * (3u ^ sw64));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_raw(sr));  // the slice's codes are in registers
                ByteTable t0, t1;
                if constexpr (C::kSmemTable) {
                    const uint4 q0 = lds_v4(tab + 16u * e0), q1 = lds_v4(tab + 16u * e1);
                    t0 = ByteTable{q0.x, q0.y, q0.z, q0.w};
                    t1 = ByteTable{q1.x, q1.y, q1.z, q1.w};
                } else {
                    t0 = mx_scaled_table(e0);
                    t1 = mx_scaled_table(e1);
                }
                uint32_t d[32];
                const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = mx_decode_word_operand(words[q], q < 4 ? t0 : t1);
                    d[4 * q + 0] = v.x;
                    d[4 * q + 1] = v.y;
                    d[4 * q + 2] = v.z;
                    d[4 * q + 3] = v.w;
                }
                if (g >= (uint32_t)s_ring && lane == 0 && !mbar_wait_sleep(empty(sw), pw ^ 1u))
                    *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                tmem_st32(lane_addr + (uint32_t)(sw * C::kAStageCols), d);
                tmem_wait_st();
                if constexpr (C::kSub == 2) {
                    // the second 64-wide sub-slice into the next 32 columns
                    ByteTable t2, t3;
                    if constexpr (C::kSmemTable) {
                        const uint4 q2 = lds_v4(tab + 16u * ev[2]), q3 = lds_v4(tab + 16u * ev[3]);
                        t2 = ByteTable{q2.x, q2.y, q2.z, q2.w};
                        t3 = ByteTable{q3.x, q3.y, q3.z, q3.w};
                    } else {
                        t2 = mx_scaled_table(ev[2]);
                        t3 = mx_scaled_table(ev[3]);
                    }
                    const uint32_t words2[8] = {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 v = mx_decode_word_operand(words2[q], q < 4 ? t2 : t3);
                        d[4 * q + 0] = v.x;
                        d[4 * q + 1] = v.y;
                        d[4 * q + 2] = v.z;
                        d[4 * q + 3] = v.w;
                    }
                    tmem_st32(lane_addr + (uint32_t)(sw * C::kAStageCols + kK / 2), d);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full(sw));
                g += C::kGroups;
                if ((sr += C::kGroups) >= SR) { sr -= SR; pr ^= 1u; }
                if ((sw += C::kGroups) >= s_ring) { sw -= s_ring; pw ^= 1u; }
            }
            g0 += (uint32_t)nk;
        }
    } else if (warp < C::kEpiWarp0 + C::kEpiWarps) {
        // ---- epilogue: accumulator (weight rows x tokens) -> bf16 output ----
        // kEpiSubs warps share each TMEM lane quarter and take its chunks in turn; a
        // warp releases the accumulator after its last tcgen05.ld (at once if it has
        // no chunk), so the next item's MMAs wait for the slowest warp's reads only
        constexpr int kEpiSubs = C::kEpiWarps / 4;
        const int quarter = warp & 3;
        const int sub = (warp - C::kEpiWarp0) >> 2;
        // 32 accumulator columns of this thread's lane at `col`: with several issuers
        // the sum of the partials in `pmask`, in issuer order (fp32, round to nearest)
        auto ld32 = [&](uint32_t col, uint32_t(&v)[32], uint32_t pmask) {
            if constexpr (C::kIssuers == 1) {
                tmem_ld32(col, v);
            } else {
                bool first = true;
#pragma unroll 1
                for (int p = 0; p < C::kIssuers; ++p) {
                    if (!((pmask >> p) & 1u)) continue;
                    const uint32_t pc = col + (uint32_t)(p * acc_stride);
                    if (first) {
                        tmem_ld32(pc, v);
                        first = false;
                    } else {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t w[16];
                            tmem_ld16(pc + (uint32_t)(16 * h), w);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[16 * h + i] = __float_as_uint(
                                    __fadd_rn(__uint_as_float(v[16 * h + i]), __uint_as_float(w[i])));
                        }
                    }
                }
            }
        };
        // read-out of one item from accumulator buffer b; `release` is called after
        // this warp's last tcgen05.ld of the item
        auto read_out = [&](const Item &it, int b, uint32_t pmask, auto &&release) {
            const int n_tok = item_tokens(it);  // > 0
            const bool odd = lane & 1;
            const int64_t step2 = 2 * (int64_t)n_out;
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) +
                                   (uint32_t)(b * C::kIssuers * C::kAccCols);
            uint16_t *const obase = out + (it.row_begin + it.m0 + (odd ? 1 : 0)) * n_out;
            if constexpr (C::kHalves) {
                // lanes 0-15 of a warp hold gate rows and lanes 16-31 the up rows of
                // the same 16 output columns. Per 32-token chunk the gate lanes finish
                // tokens 0-15 and the up lanes tokens 16-31: one xor-16 exchange hands
                // each side the other's values for its tokens
                const bool up_lane = lane >= 16;
                const int col = it.n0 + quarter * 16 + (lane & 14);
                const bool col_ok = col < n_out;
                const int t_half = up_lane ? 16 : 0;  // this lane's tokens within a chunk
                const int chunks = (n_tok + 31) / 32;
                if (sub >= chunks) release();
#pragma unroll 1
                for (int q = sub; q < chunks; q += kEpiSubs) {
                    const int c0 = q * 32;
                    uint32_t v[32];
                    ld32(taddr + (uint32_t)c0, v, pmask);
                    if (q + kEpiSubs >= chunks) release();
                    uint16_t *optr = obase + (int64_t)(c0 + t_half) * n_out + col;
                    const int lim = n_tok - c0 - t_half - (odd ? 1 : 0);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        // gate lanes send their gate values of tokens 16-31, up lanes
                        // their up values of tokens 0-15
                        const uint32_t s0 = up_lane ? v[i] : v[16 + i];
                        const uint32_t s1 = up_lane ? v[i + 1] : v[16 + i + 1];
                        const uint32_t r0 = __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
                        const uint32_t r1 = __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
                        const uint32_t g0 = up_lane ? r0 : v[i], u0 = up_lane ? v[16 + i] : r0;
                        const uint32_t g1 = up_lane ? r1 : v[i + 1], u1 = up_lane ? v[16 + i + 1] : r1;
                        const uint32_t mine = pack_bf16x2_rn(silu_mul(g0, u0), silu_mul(g1, u1));
                        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
                        const uint32_t word = odd ? prmt(other, mine, 0x7632u) : prmt(mine, other, 0x5410u);
                        if (col_ok && i < lim) *reinterpret_cast<uint32_t *>(optr) = word;
                        optr += step2;
                    }
                }
            } else if constexpr (C::kGateUp) {
                // column c of the output: gate in accumulator tile 0, up in tile 1
                const int col = it.n0 + quarter * 32 + (lane & ~1);
                const bool col_ok = col < n_out;
                const int chunks = (n_tok + 15) / 16;
                if (sub >= chunks) release();
#pragma unroll 1
                for (int q = sub; q < chunks; q += kEpiSubs) {
                    const int c0 = q * 16;
                    uint32_t gate[16], up[16];
                    tmem_ld16(taddr + (uint32_t)c0, gate);
                    tmem_ld16(taddr + (uint32_t)(kTok + c0), up);
                    if (q + kEpiSubs >= chunks) release();
                    uint16_t *optr = obase + (int64_t)c0 * n_out + col;
                    const int lim = n_tok - c0 - (odd ? 1 : 0);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const uint32_t mine = pack_bf16x2_rn(silu_mul(gate[i], up[i]),
                                                             silu_mul(gate[i + 1], up[i + 1]));
                        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
                        const uint32_t word = odd ? prmt(other, mine, 0x7632u) : prmt(mine, other, 0x5410u);
                        if (col_ok && i < lim) *reinterpret_cast<uint32_t *>(optr) = word;
                        optr += step2;
                    }
                }
            } else {
                // lanes 2i and 2i+1 hold output columns c and c+1 (c even); after an
                // exchange the even lane stores both columns of token t and the odd
                // lane both columns of token t + 1. Chunk q is tile q / per_tile.
                const int per_tile = (n_tok + 31) / 32;
                const int chunks = kMTw * per_tile;
                if (sub >= chunks) release();
#pragma unroll 1
                for (int q = sub; q < chunks; q += kEpiSubs) {
                    const int mt = kMTw == 1 ? 0 : q / per_tile;
                    const int c0 = (q - mt * per_tile) * 32;
                    uint32_t acc[32];
                    ld32(taddr + (uint32_t)(mt * kTok + c0), acc, pmask);
                    if (q + kEpiSubs >= chunks) release();
                    const int col = it.n0 + mt * kWM + quarter * 32 + (lane & ~1);
                    const bool col_ok = col < n_out;
                    uint16_t *optr = obase + (int64_t)c0 * n_out + col;
                    const int lim = n_tok - c0 - (odd ? 1 : 0);  // tokens i (even) with i < lim are stored
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const uint32_t mine =
                            pack_bf16x2_rn(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1]));
                        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
                        const uint32_t word = odd ? prmt(other, mine, 0x7632u) : prmt(mine, other, 0x5410u);
                        if (col_ok && i < lim) *reinterpret_cast<uint32_t *>(optr) = word;
                        optr += step2;
                    }
                }
            }
        };
        if constexpr (C::kIssuers == 1) {
            uint32_t use[2] = {0, 0};
            uint32_t j = 0;  // live items so far
            for (int64_t t = blockIdx.x; t < n_items; t += gridDim.x) {
                const Item it = item(t);
                if (!it.live) continue;
                const int b = C::kAccBufs == 1 ? 0 : (int)(j & 1u);
                const uint32_t u = b ? use[1] : use[0];
                if (lane == 0 && !mbar_wait_sleep(acc_full(b), u & 1u)) *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
                tc_fence_after();
                read_out(it, b, 1u, [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty(b));
                });
                if (b) ++use[1]; else ++use[0];
                ++j;
            }
        } else {
            // ---- issuer i = this warp's lane quarter: the item's K slices of decoder
            // group i (slices g = i mod 4 of this CTA's count) into partial accumulator
            // i, then the read-out of lane quarter i over all partials ----
            const int me = quarter;
            const uint32_t d_col = tmem + (uint32_t)(me * acc_stride);
            const uint32_t a_col0 = tmem + (uint32_t)a_base;
            const uint64_t x_desc0 = kmajor_sw128_desc(x_ring);
            uint32_t g0 = 0;          // this CTA's slices before the current item
            uint32_t items_done = 0;  // live items read out so far
            for (int64_t t = blockIdx.x; t < n_items; t += gridDim.x) {
                const Item it = item(t);
                if (it.bad && me == 0 && lane == 0) atomicExch(status, FP4_ERR_SHAPE);
                if (!it.live) continue;
                const int n_tok = item_tokens(it);
                const uint32_t idesc =
                    instr_desc_bf16<kWM, 16>() + ((uint32_t)(((n_tok + 15) & ~15) - 16) >> 3 << 17);
                const int kt0 = (int)(((uint32_t)me + 4u - (g0 & 3u)) & 3u);  // first slice of mine
                // the previous item's partials must have been read out by all four warps
                if (items_done > 0 && lane == 0 &&
                    !mbar_wait_sleep(acc_empty(0), (items_done - 1u) & 1u))
                    *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
                if (lane == 0) {
                    tc_fence_after();
                    for (int kt = kt0; kt < nk; kt += 4) {
                        const uint32_t gg = g0 + (uint32_t)kt;
                        const int st = (int)(gg % (uint32_t)s_ring);
                        if (!(C::kMmaSleep ? mbar_wait_sleep(full(st), (gg / (uint32_t)s_ring) & 1u)
                                           : mbar_wait_bounded(full(st), (gg / (uint32_t)s_ring) & 1u))) {
                            *abort_flag = 1;
                            break;
                        }
                        tc_fence_after();
                        if constexpr (C::kSub == 2) {
                            const uint64_t xd = x_desc0 + (uint64_t)(st * (C::kXBytes >> 4));
                            mma_slice2_tmem_a_commit(d_col, a_col0 + (uint32_t)(st * C::kAStageCols), xd,
                                                     xd + (uint64_t)(C::kXSubBytes >> 4), idesc,
                                                     kt > kt0 ? 1u : 0u, empty(st));
                        } else {
                            mma_slice_tmem_a_commit(d_col, a_col0 + (uint32_t)(st * C::kAStageCols),
                                                    x_desc0 + (uint64_t)(st * (C::kXBytes >> 4)), idesc,
                                                    kt > kt0 ? 1u : 0u, empty(st));
                        }
                    }
                    mma_commit(acc_full(0));  // arrives once this issuer's MMAs are complete
                }
                __syncwarp();
                if (*abort_flag) break;
                // the partials of the issuers that had a slice of this item
                uint32_t pmask = 0;
                for (int p = 0; p < C::kIssuers; ++p)
                    if ((int)(((uint32_t)p + 4u - (g0 & 3u)) & 3u) < nk) pmask |= 1u << p;
                g0 += (uint32_t)nk;
                if (lane == 0 && !mbar_wait_sleep(acc_full(0), items_done & 1u)) *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
                tc_fence_after();
                read_out(it, 0, pmask, [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty(0));
                });
                ++items_done;
            }
            // every MMA this thread issued completes before tensor memory is released
            if (lane == 0) {
                mma_commit(drain_bar);
                if (!mbar_wait_bounded(drain_bar, 0)) *abort_flag = 1;
            }
        }
    } else if (warp == C::kTmaXWarp && lane == 0) {
        // ---- TMA: activation tiles ----
        // launched behind the kernel that writes the activations (the MoE layer), the
        // kernel may start while that one finishes: the activation loads wait for it
        grid_dependency_wait();
        int s = 0;
        uint32_t ph = 0, g = 0;
        bool stop = false;
        for (int64_t t = blockIdx.x; t < n_items && !stop; t += gridDim.x) {
            const Item it = item(t);
            if (!it.live) continue;
            const int n_tok = item_tokens(it);
            const int row0 = (int)(it.row_begin + it.m0);
            // extended slabs get a loop of their own: this thread is on the critical
            // path, and a branch for the extension box in the plain loop costs ~10%
            if (C::kExt > 0 && n_tok > kTok) {
                for (int kt = 0; kt < nk; ++kt, ++g) {
                    if (g >= (uint32_t)s_ring && !mbar_wait_sleep(empty(s), ph ^ 1u)) *abort_flag = 1;
                    if (*abort_flag) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(full(s), (uint32_t)(kTok / kXBox * kXBoxBytes + kXExtBytes));
                    for (int bx = 0; bx < kTok / kXBox; ++bx)
                        tma_load_2d(x_ring + s * C::kXBytes + bx * kXBoxBytes, &map_x, kt * kK,
                                    row0 + bx * kXBox, full(s));
                    tma_load_2d(x_ring + s * C::kXBytes + kTok / kXBox * kXBoxBytes, &map_x_ext,
                                kt * kK, row0 + kTok, full(s));
                    if (++s == s_ring) { s = 0; ph ^= 1u; }
                }
                continue;
            }
            // 64-token items: one box of x_box_rows rows per 64-wide sub-slice; else
            // tok_live / 128 boxes
            const int boxes = kTok == 64 ? 1 : tok_live(n_tok) / kXBox;
            const uint32_t box_bytes = kTok == 64 ? (uint32_t)x_box_rows * (kK * 2) : (uint32_t)kXBoxBytes;
            for (int kt = 0; kt < nk; ++kt, ++g) {
                if (g >= (uint32_t)s_ring && !mbar_wait_sleep(empty(s), ph ^ 1u)) *abort_flag = 1;
                if (*abort_flag) {
                    stop = true;
                    break;
                }
                mbar_arrive_expect_tx(full(s), (uint32_t)(C::kSub * boxes) * box_bytes);
#pragma unroll
                for (int sub = 0; sub < C::kSub; ++sub)
                    for (int bx = 0; bx < boxes; ++bx)
                        tma_load_2d(x_ring + s * C::kXBytes + sub * C::kXSubBytes + bx * kXBoxBytes, &map_x,
                                    kt * C::kKS + sub * kK, row0 + bx * kXBox, full(s));
                if (++s == s_ring) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp == C::kTmaWWarp && lane == 0) {
        // ---- TMA: packed weight slices ----
        int s = 0;
        uint32_t ph = 0, g = 0;
        bool stop = false;
        for (int64_t t = blockIdx.x; t < n_items && !stop; t += gridDim.x) {
            const Item it = item(t);
            if (!it.live) continue;
            const int w_row = it.expert * n_rows + it.n0;  // gate rows in gate/up mode
            for (int kt = 0; kt < nk; ++kt, ++g) {
                if (g >= (uint32_t)SR && !mbar_wait_sleep(empty_raw(s), ph ^ 1u)) *abort_flag = 1;
                if (*abort_flag) {
                    stop = true;
                    break;
                }
                mbar_arrive_expect_tx(full_raw(s), (uint32_t)C::kRawBytes);
                tma_load_2d(raw_ring + s * C::kRawBytes, &map_w, kt * (C::kKS / 2), w_row, full_raw(s));
                if (C::kGateUp)  // the matching up rows fill the second half of the stage
                    tma_load_2d(raw_ring + s * C::kRawBytes + C::kBoxRows * (C::kKS / 2), &map_w,
                                kt * (C::kKS / 2), w_row + n_out, full_raw(s));
                if (++s == SR) { s = 0; ph ^= 1u; }
            }
        }
    } else if (C::kIssuers == 1 && warp >= C::kMmaWarp && warp < C::kMmaWarp + C::kTileIssuers &&
               lane == 0) {
        // ---- MMA issue: weight tile mt of every item (a thread issues one tcgen05.mma
        // per ~120-200 cycles whatever its N, measured on GB300, so the two 128 x 128
        // tiles of a 128-token item take one issuer each) ----
        const int mt = warp - C::kMmaWarp;
        constexpr uint32_t idesc_full = instr_desc_bf16<kWM, kTok>();
        constexpr uint32_t idesc_half = instr_desc_bf16<kWM, 128>();
        // stage 0 descriptors; stage s and K step kk add s * bytes/16 and kk * 32/16
        const uint64_t x_desc0 = kmajor_sw128_desc(x_ring);
        const uint32_t a_col0 = tmem + (uint32_t)C::kAColBase;
        uint32_t use[2] = {0, 0};
        uint32_t j = 0;
        int st = 0;
        uint32_t ph = 0;
        uint32_t ready = 0;  // the next stage's full barrier was seen complete
        bool stop = false;
        for (int64_t t = blockIdx.x; t < n_items && !stop; t += gridDim.x) {
            const Item it = item(t);
            if (it.bad) atomicExch(status, FP4_ERR_SHAPE);
            if (!it.live) continue;
            const int n_tok = item_tokens(it);
            // 64-token items: N = the item's tokens rounded up to 16
            const uint32_t idesc =
                kTok == 64 ? instr_desc_bf16<kWM, 16>() + ((uint32_t)(((n_tok + 15) & ~15) - 16) >> 3 << 17)
                           : (tok_live(n_tok) == kTok ? idesc_full : idesc_half);
            // an extended slab: tokens kTok.. (N rounded up to 16) into columns kTok..
            const int n_ext = C::kExt > 0 && n_tok > kTok ? (n_tok - kTok + 15) & ~15 : 0;
            const uint32_t idesc_ext = instr_desc_bf16<kWM, 16>() + ((uint32_t)(n_ext - 16) >> 3 << 17);
            const int b = C::kAccBufs == 1 ? 0 : (int)(j & 1u);
            const uint32_t u = b ? use[1] : use[0];
            // the buffer's previous item must have been read out
            if (u > 0 && !(C::kMmaSleep ? mbar_wait_sleep(acc_empty(b), (u - 1u) & 1u)
                                        : mbar_wait_bounded(acc_empty(b), (u - 1u) & 1u)))
                *abort_flag = 1;
            const uint32_t d_col = tmem + (uint32_t)(b * C::kAccCols);
            // separate K loops for extended and plain slabs: every instruction of this
            // thread is tensor-pipe idle time, so the common loop carries no extra branch
            if (C::kExt > 0 && n_ext > 0) {
                for (int kt = 0; kt < nk; ++kt) {
                    if (!ready && !(C::kMmaSleep ? mbar_wait_sleep(full(st), ph)
                                                 : mbar_wait_bounded(full(st), ph))) {
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    const int st_next = st + 1 == S ? 0 : st + 1;
                    const uint32_t ph_next = st + 1 == S ? ph ^ 1u : ph;
                    const uint64_t x_desc = x_desc0 + (uint64_t)(st * (C::kXBytes >> 4));
                    ready = mma_slice_tmem_a_ext(d_col, a_col0 + (uint32_t)(st * C::kAStageCols), x_desc,
                                                 idesc, d_col + (uint32_t)kTok,
                                                 x_desc + (uint64_t)(kTok * kK * 2 >> 4), idesc_ext,
                                                 kt > 0 ? 1u : 0u, empty(st), full(st_next), ph_next);
                    st = st_next;
                    ph = ph_next;
                }
            } else {
                for (int kt = 0; kt < nk; ++kt) {
                    if (!ready && !(C::kMmaSleep ? mbar_wait_sleep(full(st), ph)
                                                 : mbar_wait_bounded(full(st), ph))) {
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    const int st_next = st + 1 == S ? 0 : st + 1;
                    const uint32_t ph_next = st + 1 == S ? ph ^ 1u : ph;
                    if constexpr (C::kSub == 2) {
                        const uint64_t xd = x_desc0 + (uint64_t)(st * (C::kXBytes >> 4));
                        ready = mma_slice2_tmem_a(
                            d_col + (uint32_t)(mt * kTok),
                            a_col0 + (uint32_t)(st * C::kAStageCols + mt * (C::kKS / 2)), xd,
                            xd + (uint64_t)(C::kXSubBytes >> 4), idesc, kt > 0 ? 1u : 0u,
                            empty(st), full(st_next), ph_next);
                    } else {
                        ready = mma_slice_tmem_a(
                            d_col + (uint32_t)(mt * kTok),
                            a_col0 + (uint32_t)(st * C::kAStageCols + mt * (kK / 2)),
                            x_desc0 + (uint64_t)(st * (C::kXBytes >> 4)), idesc, kt > 0 ? 1u : 0u,
                            empty(st), full(st_next), ph_next);
                    }
                    st = st_next;
                    ph = ph_next;
                }
            }
            if (*abort_flag) {
                stop = true;
                break;
            }
            mma_commit(acc_full(b));
            if (b) ++use[1]; else ++use[0];
            ++j;
        }
        // all issued tensor-core work completes before TMEM is released
        mma_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0)) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) atomicExch(status, FP4_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

int sm_count() {
    static thread_local int device = -1, count = 0;
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return 0;
    if (d != device) {
        if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
            return 0;
        device = d;
    }
    return count;
}

// Tensor maps of the activations [total_rows, k] bf16 (64 x 128 boxes and, for
// slab extensions, 64 x 64 boxes; 128-byte swizzle; rows past total_rows and
// columns past k read as zero) and of the packed weights [experts * n_rows, k / 2]
// uint8 (raw_w-byte x box_rows boxes: 32 bytes unswizzled, 64 bytes with the 64-byte
// swizzle; columns past k / 2 read as zero).
cudaError_t tmem_tensor_maps(const uint16_t *a, int64_t total_rows, const uint8_t *w_packed,
                             int64_t experts, int64_t n_rows, int64_t k, int box_rows,
                             int x_box_rows, int raw_w, CUtensorMap *map_x, CUtensorMap *map_x_ext,
                             CUtensorMap *map_w) {
    EncodeTiled encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint32_t elem_strides[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)(total_rows > 0 ? total_rows : 1)};
        const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
        const cuuint32_t box[2] = {kK, (cuuint32_t)x_box_rows};
        if (encode(map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a), dims,
                   strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        const cuuint32_t box_ext[2] = {kK, kXExtBox};
        if (encode(map_x_ext, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a), dims,
                   strides, box_ext, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)(experts * n_rows)};
        const cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
        const cuuint32_t box[2] = {(cuuint32_t)raw_w, (cuuint32_t)box_rows};
        if (encode(map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w_packed), dims,
                   strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   raw_w == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <class C>
cudaError_t launch_tmem(const uint16_t *a, const int64_t *expert_offsets, int64_t experts,
                        int64_t max_rows, int64_t total_rows, const uint8_t *w_packed,
                        const uint8_t *w_scales, int64_t n_rows, int64_t n_out, int64_t k,
                        uint16_t *out, int32_t *status, cudaStream_t stream, bool after_kernel) {
    static thread_local int configured_device = -1;
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (configured_device != device) {
        err = cudaFuncSetAttribute(mx_moe_gemm_kernel<C>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (err != cudaSuccess) return err;
        configured_device = device;
    }
    // 64-token items load activation boxes of the capacity rounded up to 16 rows
    const int x_box_rows =
        C::kTok == 64 ? (int)(((max_rows < 1 ? 1 : max_rows) + 15) & ~(int64_t)15) : kXBox;
    CUtensorMap map_x, map_x_ext, map_w;
    err = tmem_tensor_maps(a, total_rows, w_packed, experts, n_rows, k,
                           C::kBoxRows, x_box_rows, C::kKS / 2, &map_x, &map_x_ext, &map_w);
    if (err != cudaSuccess) return err;
    const int64_t items = experts * ((max_rows + C::kTok - 1) / C::kTok) *
                          ((n_out + C::kTileCols - 1) / C::kTileCols);
    if (items == 0) return cudaSuccess;  // no expert may hold a row (capacity 0): no work
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = (int)(items < sms ? items : sms);
    return launch_kernel(mx_moe_gemm_kernel<C>, dim3(grid), dim3(C::kThreads), C::kSmemBytes,
                         stream, after_kernel, map_x, map_x_ext, map_w, expert_offsets, w_scales,
                         (int32_t)experts, max_rows, total_rows, (int32_t)n_rows, (int32_t)n_out,
                         (int32_t)k, (int32_t)x_box_rows, out, status);
}

}  // namespace

cudaError_t launch_mx_moe_gemm(const uint16_t *a, const int64_t *expert_offsets, int64_t experts,
                               int64_t max_rows, int64_t total_rows, const uint8_t *w_packed,
                               const uint8_t *w_scales, int64_t n, int64_t k, uint16_t *out,
                               int32_t *status, cudaStream_t stream, bool after_kernel) {
    if (max_rows > 128)
        return launch_tmem<CfgLarge>(a, expert_offsets, experts, max_rows, total_rows, w_packed,
                                     w_scales, n, n, k, out, status, stream, after_kernel);
    if (max_rows <= 64)
        return launch_tmem<CfgTiny>(a, expert_offsets, experts, max_rows, total_rows, w_packed,
                                    w_scales, n, n, k, out, status, stream, after_kernel);
    return launch_tmem<CfgSmall>(a, expert_offsets, experts, max_rows, total_rows, w_packed,
                                 w_scales, n, n, k, out, status, stream, after_kernel);
}

cudaError_t launch_mx_moe_gate_up(const uint16_t *x, const int64_t *expert_offsets, int64_t experts,
                                  int64_t max_rows, int64_t total_rows, const uint8_t *w1_packed,
                                  const uint8_t *w1_scales, int64_t n, int64_t k, uint16_t *act,
                                  int32_t *status, cudaStream_t stream, bool after_kernel) {
    if (max_rows > 128)
        return launch_tmem<CfgGateUpLarge>(x, expert_offsets, experts, max_rows, total_rows,
                                           w1_packed, w1_scales, 2 * n, n, k, act, status, stream,
                                           after_kernel);
    if (max_rows <= 64)
        return launch_tmem<CfgGateUpTiny>(x, expert_offsets, experts, max_rows, total_rows,
                                          w1_packed, w1_scales, 2 * n, n, k, act, status, stream,
                                          after_kernel);
    return launch_tmem<CfgGateUp>(x, expert_offsets, experts, max_rows, total_rows, w1_packed,
                                  w1_scales, 2 * n, n, k, act, status, stream, after_kernel);
}

}  // namespace fp4mx
