// decode_attn.cuh -- paged decode attention for sm_103a (kernel templates).
//
// Instantiated by decode_attn.cu (bf16 KV cache) and decode_attn_fp8.cu
// (e4m3 KV cache), one translation unit each so the two compile in parallel.
//
// What it computes: for every sequence b, new query token i and query head h,
//   out = softmax_t(scale * q . K_t) V_t over the logical positions t the
//   causal mask allows (t <= pos = ctx - q_len + i; with a sliding window of
//   W positions also t > pos - W: CS336 lecture-10 notes, Local attention &
//   sparse variants), with K_t, V_t found through
//   the block table (PagedAttention: "Inference Engines", The Breakthrough;
//   CS336 lecture-10 notes, PagedAttention (vLLM)), and query head h reading
//   KV head h / (n_q / n_kv) ("Transformer inference mechanics", MHA versus
//   MQA versus GQA).
//
// How (GB300 design):
//   * A "unit" is one (sequence, KV head).  Its query rows are the G = n_q/n_kv
//     heads of the group times the q_len new tokens (rows = G * q_len <= 128),
//     so every KV tile is fetched from HBM once for all of them.
//   * The whole step is a flat list of (unit, block) work items.  Persistent
//     CTA c (one per SM) takes the contiguous slice [c*W/grid, (c+1)*W/grid)
//     of the W items, so every CTA streams the same number of KV bytes however
//     ragged the context lengths are.  A unit cut by a slice boundary is a
//     split (flash-decoding); its pieces leave (O, m, l) partials that the
//     LSE merge kernel combines.
//   * Warp 8 is the producer: it reads block ids and kIssueLanes (8) of its
//     lanes issue, side by side, 2-D TMA tile loads (128-byte swizzle) of the
//     K and V tiles of each (block, KV head) into a ring of shared-memory
//     stages, each guarded by a full/empty mbarrier pair.  Its walk never stops at unit
//     boundaries, so HBM stays busy while consumers finish a unit.
//   * Warps 0..7 consume, each taking every 8th block (and, for more than 8
//     rows, one 16-row slice of them).  Products run on the tensor cores
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate); the online softmax
//     (running max m and sum l, fp32, base 2) is the FlashAttention recurrence
//     ("Efficient inference", FlashAttention: exact attention without the
//     matrix).  At the end of a unit the warps' partials are combined in
//     shared memory by the same exact rule.
//       - narrow (rows <= 8): tokens on the MMA's M side, S^T = K Q^T and
//         O^T += V^T P^T, rows padded only to 8;
//       - wide (rows > 8): rows on the M side in 16-row slices, S = Q K^T and
//         O += P V.
//   * fp32 output keeps each probability as a bf16 pair (hi + lo) so the PV
//     product keeps ~16 bits of it; bf16 output uses one bf16.
//   * 8-bit (e4m3) caches (KV8): tiles stay as bytes in shared memory and are
//     widened to f16 in registers (every e4m3 value is exact in f16), the
//     products run as f16 mma.sync with Q and P in f16.  K fragments come
//     from plain ldmatrix: lane (g, t) holds bytes 4t..4t+3 of a 16-byte row
//     segment, so in each 16-wide k step logical k (2t, 2t+1) is d (4t, 4t+1)
//     and (2t+8, 2t+9) is d (4t+2, 4t+3); Q is loaded in the same order.  V
//     fragments come from ldmatrix.trans (token pairs of one byte pair) and
//     one byte permute that separates the even and odd d of the pair, so the
//     output columns are d = 32j + 16h + 2c + parity.  The per-head K scale
//     is folded into the score scale and the V scale into the final
//     normalisation.  Rows > 64 use the tensor-memory consumer on f16 copies
//     of the stages (see there).
//
// Bounded waits: every mbarrier wait gives up after a second, records
// kErrTimeout in the workspace and the kernel winds down without hanging.
#pragma once

#include <atomic>
#include <cfloat>
#include <climits>
#include <type_traits>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
// The tensor-memory consumer over an 8-bit cache adds three warps (9, 10, 11)
// that widen stages to f16 beside warps 6 and 7: five converter warps on
// schedulers 2, 3, 1, 2, 3 (two warps on schedulers 2 and 3 alone took
// ~1.2 us per 64-key stage, the pace of the whole pipeline).  ptxas caps a
// thread at 168 registers for 288 and for 384 threads alike.
constexpr int kTmemConverters = 5;
__host__ __device__ constexpr int threads_for(int mode, bool kv8) {
    // tensor-memory consumer: + 3 converter warps over an 8-bit cache; the
    // paired form (mode 3) has eight softmax warps, the producer and two issuers
    return mode == 3 ? kThreads + 2 * 32 : (mode == 2 && kv8 ? kThreads + 3 * 32 : kThreads);
}
constexpr int kMergeSlots = 4;                   // warps that park a partial per merge round
constexpr int kIssueLanes = 8;                   // producer lanes issuing loads side by side
constexpr int kNarrowRows = 8;                   // rows up to which the narrow consumer is used
constexpr int kTmemMinRows = 64;                 // rows above which the TMEM consumer is used

// Per-(block, KV head) scales weigh a block's probabilities by its V scale over
// the largest one seen so far; the weights go to f16 for the MMA, so they carry
// a power-of-two headroom, taken back out of the accumulator at the end, that
// keeps small ratios out of f16's subnormal range: 2^14 where probabilities
// are at most 1 (mma.sync consumers), 2^7 where the lazily rescaled ones reach
// 2^8 (tensor-memory consumer) -- at most 2^15 either way, below f16's 65504.
constexpr float kPShiftSync = 16384.f, kPShiftSyncInv = 1.f / 16384.f;
constexpr float kPShiftTmem = 128.f, kPShiftTmemInv = 1.f / 128.f;

// Consumer modes, chosen by the number of query rows sharing a KV head.
constexpr int kModeWide = 0;    // 8 < rows <= 64: mma.sync, rows on the M side
constexpr int kModeNarrow = 1;  // rows <= 8: mma.sync, tokens on the M side
constexpr int kModeTmem = 2;    // rows > 64: tcgen05, M = 128 row tiles, accumulators in TMEM
constexpr int kModeTmem2 = 3;   // 256-row units: two M = 128 row tiles on every stage (bf16 only)

template <int D, int BS, int MODE, bool KV8 = false, bool BLK = false>
struct AttnCfg {
    static constexpr bool kTmem = MODE == kModeTmem || MODE == kModeTmem2;
    static constexpr int kQRows = MODE == kModeTmem2 ? 256 : 128;  // rows of the query tile
    static_assert(MODE != kModeTmem2 || (!KV8 && !BLK), "the paired form is bf16 only");
    static constexpr int kTileBytes = BS * D * (KV8 ? 1 : 2);  // one K (or V) tile of one (block, head)
    // TMA boxes per tile: bf16 in 64-column (128-byte) boxes; e4m3 rows of D
    // bytes in one box (128-byte swizzle at D = 128, 64-byte at D = 64).
    static constexpr int kBoxes = KV8 ? 1 : D / 64;
    static constexpr int kBoxCols = KV8 ? D : 64;
    static constexpr int kBoxBytes = KV8 ? BS * D : BS * 128;
    // Blocks per ring stage.  TMEM consumer: 64 keys, so one score MMA spans
    // them (N = 64).  mma.sync consumers: enough blocks for 8 KB of K + V --
    // the stream slows down markedly with smaller stages (measured: 4 KB
    // stages ran at ~4.3 TB/s, 8 KB ones at ~6 TB/s, whatever the dtype),
    // since every stage costs a barrier round trip and a producer issue.  A
    // stage is laid out as [K box 0][K box 1 (d 128)][V box 0][V box 1], each
    // region holding the stage's blocks one after another (kRegion bytes), so
    // the rows of all its blocks are contiguous within each 64-column region.
    // (TMEM consumer, bf16 at d 128, through the grouped 4-D views: each half
    // of the stage is [block][8-row group][half][8 rows][128 bytes] instead,
    // one copy per block for K and one for V.)
    static constexpr int kBlocksPerStage =
        kTmem ? 64 / BS : (2 * kTileBytes >= 8192 ? 1 : 8192 / (2 * kTileBytes));
    static constexpr int kRegion = kBlocksPerStage * kBoxBytes;
    static constexpr int kStageBytes = 2 * kBoxes * kRegion;
    // An 8-bit cache keeps a (block, head)'s V rows right after its K rows,
    // so one TMA box of 2 * BS rows fetches both: in its stages block b
    // occupies [K rows][V rows] at b * 2 * kBoxBytes.  (bf16: K region(s),
    // then V region(s), block b at b * kBoxBytes within each.)
    __device__ static uint32_t k_tile(uint32_t stage, int b) {
        return KV8 ? stage + b * 2 * kBoxBytes : stage + b * kBoxBytes;
    }
    __device__ static uint32_t v_tile(uint32_t stage, int b) {
        return KV8 ? stage + b * 2 * kBoxBytes + kBoxBytes
                   : stage + kBoxes * kRegion + b * kBoxBytes;
    }
    // Per-lane floats a warp parks for a merge round: its accumulator, m[2], l[2].
    static constexpr int kLaneFloats = (MODE == kModeNarrow ? D / 4 : D / 2) + 4;
    static constexpr int kMergeBytes = kTmem ? 0 : kMergeSlots * 32 * kLaneFloats * 4;
    // Narrow emit: rows x head_dim fp32 tile (+4 floats of row padding) and (m, l) per row.
    static constexpr int kTileStride = D + 4;
    static constexpr int kEmitBytes =
        MODE == kModeNarrow ? (kNarrowRows * kTileStride + 2 * kNarrowRows) * 4 : 0;
    // TMEM mode over bf16: the unit's 128 (paired: 256) query rows as a
    // swizzled K-major tile, fetched by TMA while the piece before it ends.
    // Over an 8-bit cache the query rows live in tensor memory instead, which
    // leaves the 32 KB to the ring: eight 64-key stages instead of six
    // (measured: MQA verify 51.7 -> 49.7 us, with block scales 62.7 -> 55.8,
    // chunked prefill 125.4 -> 117.3).  Over bf16 the extra stage did not pay
    // for the later query rows (MQA verify 40.2 -> 41.5 us).
    static constexpr int kQTileBytes = (kTmem && !KV8) ? kQRows * D * 2 : 0;
    // TMEM mode over an 8-bit cache: kCvtCopies f16 copies of a 64-key stage
    // (K and V, each 64 rows in D/64 swizzled 64-column regions).  A copy is
    // held from its conversion until its PV product completes; with two, the
    // conversion of stage g + 2 waited for PV(g) and the softmax for that
    // conversion (MQA verify e4m3: one stage per ~1.5 us against ~0.8 over bf16).
    static constexpr int kCvtCopies = 3;
    static constexpr int kCvtRegion = 64 * 128;
    static constexpr int kCvtBytes =
        (kTmem && KV8) ? kCvtCopies * 2 * (D / 64) * kCvtRegion : 0;
    // Per-(block, KV head) scales (BLK): each block of a stage brings 16 bytes
    // {K scale, V scale, 0, 0} with its tiles, into a slot beside the ring;
    // the tensor-memory consumer's converter warps copy a super-block's scales
    // next to its f16 copy (kCvtCopies copies x blocks x {K, V}).
    static constexpr int kSlotBytes = BLK ? kBlocksPerStage * 16 : 0;
    static constexpr int kCvtSlotBytes =
        (BLK && kTmem) ? kCvtCopies * kBlocksPerStage * 8 : 0;
    static constexpr int kScratchBytes =
        kMergeBytes + kEmitBytes + kQTileBytes + kCvtBytes + kCvtSlotBytes;
    static constexpr int kMaxStages = kTmem ? (KV8 ? 24 : 16) : (KV8 ? 48 : 32);
    static constexpr int kBarrierBytes = 2 * kMaxStages * 8;
    static constexpr int kBudget = 227 * 1024 - 1024 - kScratchBytes - kBarrierBytes - 1024;
    // In the mma.sync modes the ring depth is a multiple of the consumer-warp
    // count: block g and block g - kStages then belong to the same warp, so
    // when a warp waits for round r of a stage it has itself already seen
    // round r - 1 complete.  (mbarrier parity waits cannot tell round r from
    // round r - 2; with another warp owning round r - 1 a still-in-flight load
    // would read as complete.)  The TMEM mode has a single consumer thread.
    static constexpr int kStagesRaw = kBudget / (kStageBytes + kSlotBytes);
    static constexpr int kStages =
        kStagesRaw >= kMaxStages ? kMaxStages
                                 : (kTmem ? kStagesRaw : (kStagesRaw / 8) * 8);
    static constexpr int kSmemBytes =
        1024 + kStages * kStageBytes + kScratchBytes + 2 * kStages * 8 + kStages * kSlotBytes;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(kTmem ? kStages >= 2
                                    : (kStages % kConsumerWarps == 0 && kStages >= kConsumerWarps),
                  "ring depth");
    static_assert(kTmem || kStages >= kIssueLanes, "one stage per issue lane");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    // The mma.sync consumers address a block's boxes BS * 128 bytes apart.
    static_assert(kTmem || kBlocksPerStage == 1 || kBoxes == 1, "stage layout");
};

// Byte offset of the 16-byte chunk holding (row, col..col+7) inside a tile
// stored as D/64 boxes of [BS rows][128 bytes] with the TMA 128-byte swizzle
// (16-byte chunk index XOR row % 8 within each 1024-byte atom).
template <int BS>
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return static_cast<uint32_t>((col >> 6) * (BS * 128) + row * 128 +
                                 ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

// Byte offset of (row, byte cb..cb+15) in an e4m3 tile of D-byte rows as the
// TMA unit writes it: 128-byte swizzle at D = 128 (16-byte chunk ^ row % 8),
// 64-byte swizzle at D = 64 (chunk ^ (row / 2) % 4).  cb is a multiple of 16.
template <int D>
__device__ __forceinline__ uint32_t swz8(int row, int cb) {
    if constexpr (D == 128)
        return static_cast<uint32_t>(row * 128 + (((cb >> 4) ^ (row & 7)) << 4));
    else
        return static_cast<uint32_t>(row * 64 + (((cb >> 4) ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ int unit_ctx(const AttnArgs& a, int s, int bs) {
    int ctx = __ldg(a.context_lens + s);
    const int cap = a.max_blocks_per_seq * bs;
    return ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
}

__device__ __forceinline__ int unit_blocks(const AttnArgs& a, int s, int bs) {
    return (unit_ctx(a, s, bs) + bs - 1) / bs;
}

// Query rows come in tiles of a.rows: row R = t * a.rows + r of a unit's
// G * q_len rows belongs to query token R / G and query head h * G + R % G.
// A decode step has one tile; a prefill chunk (many new tokens) has several,
// each its own unit.  Tokens of tile t: first and last.
__device__ __forceinline__ int tile_first_token(const AttnArgs& a, int t) {
    return (t * a.rows) / a.group;
}
__device__ __forceinline__ int tile_last_token(const AttnArgs& a, int t) {
    const int last_row = min(a.rows_total, (t + 1) * a.rows) - 1;
    return last_row / a.group;
}

// Row r of tile t: its query token i and query head hq; false for padding
// rows past the last real row.
__device__ __forceinline__ bool unit_row(const AttnArgs& a, int t, int h, int r, int& i,
                                         int& hq) {
    const int R = t * a.rows + r;
    const bool valid = r < a.rows && R < a.rows_total;
    i = valid ? R / a.group : 0;
    hq = h * a.group + (valid ? R % a.group : 0);
    return valid;
}

// One past the last block a tile whose last query token is last_tok can see:
// that row sits at position ctx - q_len + last_tok and sees nothing later
// (causal).  At least one block when ctx > 0, so a tile whose rows all
// precede the context still writes its zero rows; none when ctx == 0.
// (ctx - q_len + last_tok + 1 <= ctx: no overflow.)
__device__ __forceinline__ int tok_end_block(const AttnArgs& a, int ctx, int last_tok, int bs) {
    const int vis = max(1, min(ctx - a.q_len + last_tok + 1, ctx));
    return static_cast<int>((static_cast<unsigned>(vis) + bs - 1) / static_cast<unsigned>(bs));
}

// First block a tile whose first query token is first_tok can see: with a
// sliding window, its earliest row (position ctx - q_len + first_tok) sees
// nothing before that position minus W - 1, so earlier blocks are never
// read.  Always < tok_end_block of the same tile.
__device__ __forceinline__ int tok_first_block(const AttnArgs& a, int ctx, int first_tok, int bs) {
    if (a.window <= 0) return 0;
    const long long lo = (long long)ctx - a.q_len + first_tok - a.window + 1;
    return lo > 0 ? static_cast<int>(static_cast<unsigned>(lo) / static_cast<unsigned>(bs)) : 0;
}

__device__ __forceinline__ int unit_end_block(const AttnArgs& a, int ctx, int t, int bs) {
    return tok_end_block(a, ctx, tile_last_token(a, t), bs);
}
__device__ __forceinline__ int unit_first_block(const AttnArgs& a, int ctx, int t, int bs) {
    return tok_first_block(a, ctx, tile_first_token(a, t), bs);
}

// The first and last query tokens of tiles 0, 1, 2, ... in turn, without a
// division per tile: the first row t * rows of the tile is carried as a
// token and a row within the token's group.
struct TileSteps {
    int fq, fr, dq, dr, g, qmax;
    __device__ __forceinline__ explicit TileSteps(const AttnArgs& a)
        : fq(0), fr(0), dq(a.rows / a.group), dr(a.rows % a.group), g(a.group), qmax(a.q_len - 1) {}
    __device__ __forceinline__ int first() const { return fq; }
    __device__ __forceinline__ int last() const {  // the row before the next tile's first
        int nq = fq + dq, nr = fr + dr;
        if (nr >= g) {
            nr -= g;
            ++nq;
        }
        return min(nr > 0 ? nq : nq - 1, qmax);
    }
    __device__ __forceinline__ void next() {
        fq += dq;
        fr += dr;
        if (fr >= g) {
            fr -= g;
            ++fq;
        }
    }
};

// Work items (blocks to read) of one KV head of sequence s, over all its tiles.
__device__ __forceinline__ long long head_items(const AttnArgs& a, int ctx, int bs) {
    if (ctx == 0) return 0;
    // One row tile and no window (every decode step): the unit reads every block.
    if (a.q_tiles == 1 && a.window <= 0)
        return static_cast<long long>((static_cast<unsigned>(ctx) + bs - 1) / static_cast<unsigned>(bs));
    TileSteps ts(a);
    long long n = 0;
#pragma unroll 1
    for (int t = 0; t < a.q_tiles; ++t) {
        n += tok_end_block(a, ctx, ts.last(), bs) - tok_first_block(a, ctx, ts.first(), bs);
        ts.next();
    }
    return n;
}

// Position in the flat work list: sequence s, KV head h, row tile t, block j
// of that unit (the unit reads blocks jlo .. nb-1), `left` items still to
// process in this CTA's slice.  Units run tile-fastest, so the tiles of one
// KV head (which read overlapping blocks) follow each other.
struct Walk {
    int s, h, t, j, jlo, nb, ctx;
    long long left;
};

template <int BS>
__device__ __forceinline__ void walk_set_unit(const AttnArgs& a, Walk& w) {
    w.nb = unit_end_block(a, w.ctx, w.t, BS);
    w.jlo = unit_first_block(a, w.ctx, w.t, BS);
    w.j = w.jlo;
}

template <int BS>
__device__ __forceinline__ void walk_next_unit(const AttnArgs& a, Walk& w) {
    if (++w.t == a.q_tiles) {
        w.t = 0;
        if (++w.h == a.n_kv) {
            w.h = 0;
            do {
                ++w.s;
            } while (w.s < a.num_seqs && unit_ctx(a, w.s, BS) == 0);
            w.ctx = w.s < a.num_seqs ? unit_ctx(a, w.s, BS) : 0;
        }
    }
    walk_set_unit<BS>(a, w);
    // The slices cover exactly the items of the units; a walk that ran past
    // the last sequence stops instead of spinning on empty pieces.
    if (w.s >= a.num_seqs) w.left = 0;
}

__device__ __forceinline__ int piece_end(const Walk& w) {
    return (long long)w.nb < (long long)w.j + w.left ? w.nb : static_cast<int>(w.j + w.left);
}

// Block-wide inclusive scan of two 64-bit values per thread (all NT threads);
// s_red holds 2 * NT / 32 values.
template <int NT>
__device__ __forceinline__ void block_inclusive_scan2(long long& c, long long& r, long long* s_red,
                                                      long long& total_c, long long& total_r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long nc = __shfl_up_sync(0xffffffffu, c, off);
        const long long nr = __shfl_up_sync(0xffffffffu, r, off);
        if (lane >= off) {
            c += nc;
            r += nr;
        }
    }
    if (lane == 31) {
        s_red[2 * warp] = c;
        s_red[2 * warp + 1] = r;
    }
    __syncthreads();
    long long bc = 0, br = 0;
    total_c = total_r = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const long long tc = s_red[2 * w], tr = s_red[2 * w + 1];
        if (w < warp) {
            bc += tc;
            br += tr;
        }
        total_c += tc;
        total_r += tr;
    }
    __syncthreads();
    c += bc;
    r += br;
}

// a / b for a >= 0, b > 0: one 32-bit division when both fit, as they do but
// for batches of billions of blocks.
__device__ __forceinline__ long long div_nn(long long a, long long b) {
    if ((((unsigned long long)a | (unsigned long long)b) >> 32) == 0)
        return static_cast<long long>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
    return a / b;
}

// Block item (within the sequence) at cost offset o of a sequence: a position
// inside a unit's fixed-cost prefix maps to the unit's first block.  The map
// is non-decreasing, so consecutive CTAs' slices meet exactly.  Also the
// item's unit (KV head h, row tile t) and block j.
struct ItemPos {
    long long item;
    int h, t, j;
};

template <int BS>
__device__ __forceinline__ ItemPos cost_to_item(const AttnArgs& a, int ctx, long long o) {
    const long long hi = head_items(a, ctx, BS);
    const long long hc = hi + (long long)a.q_tiles * a.unit_cost;
    const long long h = div_nn(o, hc);
    long long o2 = o - h * hc, before = 0;  // o2 < hc: some tile holds it
    ItemPos p;
    p.h = static_cast<int>(h);
    TileSteps ts(a);
#pragma unroll 1
    for (int t = 0;; ++t) {
        const int jlo = tok_first_block(a, ctx, ts.first(), BS);
        const long long n = tok_end_block(a, ctx, ts.last(), BS) - jlo;
        if (o2 < n + a.unit_cost || t + 1 >= a.q_tiles) {
            const long long k = o2 > a.unit_cost ? o2 - a.unit_cost : 0;
            p.item = h * hi + before + k;
            p.t = t;
            p.j = jlo + static_cast<int>(k);
            return p;
        }
        o2 -= n + a.unit_cost;
        before += n;
        ts.next();
    }
}

// The partition weighs a unit as its blocks plus a.unit_cost: the fixed work
// of a unit (query load, cross-warp combine, output) in block equivalents.
// Without it a CTA whose slice covers many short sequences does many units'
// fixed work for the same bytes and finishes last.  A sequence with context
// ctx costs (head_items + q_tiles * unit_cost) * n_kv, nothing when empty.
//
// All threads: this CTA's slice of the flat (unit, block) list -- cost range
// [c*C/grid, (c+1)*C/grid) mapped to block items -- as the walk position of
// its first item.  Each thread takes kSliceSeqs consecutive sequences per
// round, so one round (one load of the context lengths, one scan) covers
// batches of up to kThreads * kSliceSeqs sequences; the thread whose
// sequences hold the slice's first (last) cost position computes its walk
// and publishes it.  s_pos: {start found, item0, end found, item1}.
// This code runs once per launch, so its cost is mostly instruction fetch
// of cold code: it is kept small (no unrolling; one sequence per thread per
// round), which measured several times faster than unrolled variants.
constexpr int kSliceSeqs = 1;

template <int BS, int NT>
__device__ __forceinline__ Walk find_slice(const AttnArgs& a, long long* s_red,
                                           long long* s_pos, Walk* s_walk) {
    const int tid = threadIdx.x, cta = blockIdx.x, grid = gridDim.x;
    constexpr int kRound = NT * kSliceSeqs;
    long long total_c = 0, total_r = 0;
    if (a.num_seqs > kRound) {  // several rounds: totals first
        long long mc = 0, mr = 0;
        for (int s = tid; s < a.num_seqs; s += NT) {
            const int ctx = unit_ctx(a, s, BS);
            const long long hi = head_items(a, ctx, BS);
            mc += ctx > 0 ? (hi + (long long)a.q_tiles * a.unit_cost) * a.n_kv : 0;
            mr += hi * a.n_kv;
        }
        block_inclusive_scan2<NT>(mc, mr, s_red, total_c, total_r);
    }
    long long start = 0, end = 0, base_c = 0, base_r = 0;
    for (int s0 = 0; s0 < a.num_seqs; s0 += kRound) {
        const int sb = s0 + tid * kSliceSeqs;
        int ctx[kSliceSeqs];
        long long vc[kSliceSeqs], vr[kSliceSeqs], ic = 0, ir = 0;
#pragma unroll
        for (int k = 0; k < kSliceSeqs; ++k) ctx[k] = sb + k < a.num_seqs ? unit_ctx(a, sb + k, BS) : 0;
#pragma unroll
        for (int k = 0; k < kSliceSeqs; ++k) {
            const long long hi = head_items(a, ctx[k], BS);
            vc[k] = ctx[k] > 0 ? (hi + (long long)a.q_tiles * a.unit_cost) * a.n_kv : 0;
            vr[k] = hi * a.n_kv;
            ic += vc[k];
            ir += vr[k];
        }
        const long long lc = ic, lr = ir;
        long long rc, rr;
        block_inclusive_scan2<NT>(ic, ir, s_red, rc, rr);
        if (a.num_seqs <= kRound) {
            total_c = rc;
            total_r = rr;
        }
        start = div_nn(total_c * cta, grid);
        end = div_nn(total_c * (cta + 1), grid);
        if (start >= end) break;  // (uniform) an empty slice
        long long ec = base_c + ic - lc, er = base_r + ir - lr;
#pragma unroll
        for (int k = 0; k < kSliceSeqs; ++k) {
            if (vc[k] > 0 && ec <= start && start < ec + vc[k]) {
                const ItemPos p = cost_to_item<BS>(a, ctx[k], start - ec);
                Walk w;
                w.s = sb + k;
                w.ctx = ctx[k];
                w.h = p.h;
                w.t = p.t;
                walk_set_unit<BS>(a, w);
                w.j = p.j;
                w.left = 0;
                *s_walk = w;
                s_pos[1] = er + p.item;
                s_pos[0] = 1;
            }
            if (end < total_c && vc[k] > 0 && ec <= end && end < ec + vc[k]) {
                s_pos[3] = er + cost_to_item<BS>(a, ctx[k], end - ec).item;
                s_pos[2] = 1;
            }
            ec += vc[k];
            er += vr[k];
        }
        base_c += rc;
        base_r += rr;
        __syncthreads();
        if (s_pos[0] >= 0 && (end >= total_c || s_pos[2] >= 0)) break;
    }
    __syncthreads();  // (also publishes the barrier init when no round ran)
    Walk w;
    w.left = 0;
    if (start < end && s_pos[0] >= 0 && (end >= total_c || s_pos[2] >= 0)) {
        w = *s_walk;
        w.left = (end < total_c ? s_pos[3] : total_r) - s_pos[1];
    }
    if (w.left <= 0) {
        w.left = 0;
        w.s = w.h = w.t = w.j = w.jlo = w.nb = w.ctx = 0;
    }
    return w;
}

// ===================== producer warp =====================
// Fills ring stages of SBS blocks each: a piece of n blocks takes ceil(n / SBS)
// stages (the last may be partial), counted from the piece's first block.
// Lanes 0..kIssueLanes-1 fill consecutive stages side by side: one serial
// wait/issue chain per stage would cap the stream (measured with 2, 4 and 8
// lanes: the GQA step took 221.6, 172.2 and 161.3 us).
// ORDERED (the tensor-memory consumer, which frees stages strictly in order):
// stages are refilled one at a time in order, each stage's TMA boxes spread
// over the lanes, so a freed stage is refilled at once instead of waiting for
// the stages issued beside it, and the first stages of a launch land first
// instead of together.
// BLK: each block's 16-byte scale entry comes with its tiles into the stage's
// slot, by an LSU asynchronous copy tracked by the stage's full barrier (as
// 16-byte TMA bulk copies they cost 8-bit GQA 14 us of 115: twice the TMA
// operations per stage); an out-of-range block id (whose tiles read zeros)
// gets a zero slot written by the issuing lane before the stage's arrival.
template <int D, int BS, int kStages, int kStageBytes, int kTileBytes, int kBoxBytes, int kBoxes,
          int kBoxCols, int kRegion, int SBS, bool KV8, bool ORDERED, bool BLK>
__device__ __forceinline__ void produce(const AttnArgs& a, const CUtensorMap* tmap_k,
                                        const CUtensorMap* tmap_v, Walk w, uint8_t* stages,
                                        uint8_t* slots, uint64_t* full_bar, uint64_t* empty_bar,
                                        volatile int* s_abort) {
    // a block's scale entry: (block, head) row of [num_blocks][n_kv][4] fp32
    auto scale_src = [&](int blk) { return a.kv_scales + ((size_t)blk * a.n_kv + w.h) * 4; };
    static_assert(32 % SBS == 0, "stages must not straddle a batch of 32 block ids");
    const int lane = threadIdx.x & 31;
    if (a.test_stall) return;  // failure-path tests: nothing is loaded, every wait expires
    const uint64_t policy = l2_policy_evict_first();
    uint32_t gidx = 0, issued = 0;  // stages; issued: fills actually started (a prefix of gidx)
    bool ok = true;
    while (w.left > 0 && ok) {
        const int j1 = piece_end(w);
        // The consumers load this unit's query rows when they reach it, about a
        // ring later: fetch them into the L2 now (one bulk prefetch per query
        // token of the row tile), so that load does not wait on HBM.
        {
            const int R0 = w.t * a.rows, R1 = min(a.rows_total, R0 + a.rows);
            const int i0 = R0 / a.group, i1 = (R1 - 1) / a.group;
            for (int i = i0 + lane; i <= i1; i += 32) {
                const int lo = max(R0, i * a.group) - i * a.group;
                const int hi = min(R1, (i + 1) * a.group) - i * a.group;
                prefetch_l2_bulk(a.q + (((size_t)w.s * a.q_len + i) * a.n_q + w.h * a.group + lo) * D,
                                 static_cast<uint32_t>((hi - lo) * D * 2));
            }
        }
        const int32_t* bt = a.block_tables + (size_t)w.s * a.max_blocks_per_seq;
        int my = w.j + lane < j1 ? __ldg(bt + w.j + lane) : 0;
        for (int jb = w.j; jb < j1 && ok; jb += 32) {
            const int n = min(32, j1 - jb);
            const int ns = (n + SBS - 1) / SBS;  // stages of this batch
            // The next 32 block ids load while this batch is issued.
            const int nxt = jb + 32 + lane < j1 ? __ldg(bt + jb + 32 + lane) : 0;
            if (lane < n && (my < 0 || my >= a.num_blocks)) {
                if (a.checked) atomicOr(a.err, kErrBadBlock);
                my = -1;  // read as an out-of-bounds (zero-filled) tile
            }
            if (*s_abort) ok = false;  // a consumer gave up
            if constexpr (ORDERED) {
                // boxes per block: K and V halves (bf16), one K and one V box
                // through the grouped 4-D views (bf16, d 128), or one K+V box
                // (8-bit)
                static_assert(SBS * (KV8 ? 1 : 2 * kBoxes) <= 32, "one box per lane");
                const bool g4 = !KV8 && kBoxes == 2 && a.tile_4d;
                const int bpb = KV8 ? 1 : (g4 ? 2 : 2 * kBoxes);
                for (int k = 0; k < ns && ok; ++k) {
                    const int nb = min(SBS, n - k * SBS);
                    const int blk = __shfl_sync(0xffffffffu, my, (k * SBS + lane / bpb) & 31);
                    const uint32_t stage = gidx % kStages;
                    bool good = true;
                    if (lane == 0)
                        good = mbar_wait_bounded(&empty_bar[stage], ((gidx / kStages) & 1u) ^ 1u);
                    good = __shfl_sync(0xffffffffu, good, 0);
                    __syncwarp();
                    if (!good) {
                        ok = false;
                        if (lane == 0) {
                            atomicOr(a.err, kErrTimeout);
                            *s_abort = 1;
                        }
                        break;
                    }
                    // BLK: lane b < nb owns block b's scale slot (one box per block)
                    if constexpr (BLK) {
                        static_assert(KV8, "scale slots assume one box per block");
                        if (lane < nb) {
                            uint8_t* slot = slots + (stage * SBS + lane) * 16;
                            if (blk >= 0) {
                                cp_async_16(slot, scale_src(blk));
                                cp_async_mbar_arrive(&full_bar[stage]);
                            } else {
                                *reinterpret_cast<uint4*>(slot) = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                        __syncwarp();  // the slots' arrivals and zeros before the stage's arrival
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&full_bar[stage], nb * 2 * kTileBytes);
                    if (lane < nb * bpb) {
                        const int b = lane / bpb, box = lane % bpb;
                        const long long y64 = ((long long)blk * a.n_kv + w.h) * a.kv_mul * BS;
                        const bool oob = blk < 0 || y64 >= a.tile_rows_total;
                        const int yk = oob ? a.tile_rows_total : static_cast<int>(y64);
                        if constexpr (KV8) {
                            tma_load_2d(stages + stage * kStageBytes + b * 2 * kBoxBytes, tmap_k,
                                        0, yk, &full_bar[stage], policy);
                        } else if (g4) {
                            // block b's K (box 0) or V (box 1) tile in one copy, as
                            // [8-row group][half][8 rows][128 bytes] at b * 2 * kBoxBytes
                            // of the stage's K or V region
                            const bool isv = box == 1;
                            const int y = isv && !oob ? yk + a.v_row_off : yk;
                            tma_load_4d_hint(stages + stage * kStageBytes +
                                                 (isv ? kBoxes * kRegion : 0) + b * 2 * kBoxBytes,
                                             isv ? tmap_v : tmap_k, 0, 0, 0, y >> 3,
                                             &full_bar[stage], policy);
                        } else {
                            // box: K half (box < kBoxes), then V half
                            const int half = box % kBoxes;
                            const bool isv = box >= kBoxes;
                            const int yv = oob ? a.tile_rows_total : yk + a.v_row_off;
                            tma_load_2d(stages + stage * kStageBytes + b * kBoxBytes +
                                            (isv ? kBoxes + half : half) * kRegion,
                                        isv ? tmap_v : tmap_k, half * kBoxCols, isv ? yv : yk,
                                        &full_bar[stage], policy);
                        }
                    }
                    ++gidx;
                    issued = gidx;
                }
            }
            for (int k0 = 0; !ORDERED && k0 < ns && ok; k0 += kIssueLanes) {
                const int sk = k0 + lane;  // this lane's stage within the batch
                const bool act = lane < kIssueLanes && sk < ns;
                const int nb = SBS == 1 ? 1 : (act ? min(SBS, n - sk * SBS) : 0);
                // Block ids of this lane's stage, fetched before the wait.
                int blks[SBS];
#pragma unroll
                for (int b = 0; b < SBS; ++b)
                    blks[b] = __shfl_sync(0xffffffffu, my, (sk * SBS + b) & 31);
                const uint32_t gl = gidx + lane;
                const uint32_t stage = gl % kStages;
                bool good = true;
                if (act) good = mbar_wait_bounded(&empty_bar[stage], ((gl / kStages) & 1u) ^ 1u);
                const unsigned act_mask = __ballot_sync(0xffffffffu, act);
                const unsigned good_mask = __ballot_sync(0xffffffffu, act && good);
                const unsigned fail = act_mask & ~good_mask;
                // Only the lanes below the first failed wait issue, so the
                // issued fills stay a prefix of the stage sequence.
                const unsigned issue_mask =
                    fail ? (good_mask & ((1u << (__ffs(fail) - 1)) - 1u)) : good_mask;
                const bool do_issue = (issue_mask >> lane) & 1u;
                if constexpr (BLK) {
                    // this lane's stage: a copy for each in-range block, zeros for the rest
                    if (do_issue) {
                        bool copied = false;
#pragma unroll
                        for (int b = 0; b < SBS; ++b) {
                            if (b >= nb) continue;
                            uint8_t* slot = slots + (stage * SBS + b) * 16;
                            if (blks[b] >= 0) {
                                cp_async_16(slot, scale_src(blks[b]));
                                copied = true;
                            } else {
                                *reinterpret_cast<uint4*>(slot) = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                        if (copied) cp_async_mbar_arrive(&full_bar[stage]);
                    }
                }
                if (do_issue) mbar_arrive_expect_tx(&full_bar[stage], nb * 2 * kTileBytes);
#pragma unroll
                for (int b = 0; b < SBS; ++b) {
                    const int blk = blks[b];
                    if (do_issue && b < nb) {
                        // K rows of (block, head) in the 2-D cache view; the V rows
                        // follow them in an 8-bit cache, else they sit at the same
                        // rows of the V cache.  Bad ids read past the end (zeros).
                        const long long y64 = ((long long)blk * a.n_kv + w.h) * a.kv_mul * BS;
                        const bool oob = blk < 0 || y64 >= a.tile_rows_total;
                        const int yk = oob ? a.tile_rows_total : static_cast<int>(y64);
                        const int yv = oob ? a.tile_rows_total : yk + a.v_row_off;
                        if constexpr (KV8) {
                            // one box of 2 * BS rows: the K rows, then the V rows
                            tma_load_2d(stages + stage * kStageBytes + b * 2 * kBoxBytes, tmap_k,
                                        0, yk, &full_bar[stage], policy);
                        } else {
                            uint8_t* kdst = stages + stage * kStageBytes + b * kBoxBytes;
#pragma unroll
                            for (int half = 0; half < kBoxes; ++half) {
                                tma_load_2d(kdst + half * kRegion, tmap_k, half * kBoxCols, yk,
                                            &full_bar[stage], policy);
                                tma_load_2d(kdst + (kBoxes + half) * kRegion, tmap_v,
                                            half * kBoxCols, yv, &full_bar[stage], policy);
                            }
                        }
                    }
                }
                issued = gidx + __popc(issue_mask);
                if (fail) {
                    ok = false;
                    if (lane == 0) {
                        atomicOr(a.err, kErrTimeout);
                        *s_abort = 1;
                    }
                }
                gidx += min(kIssueLanes, ns - k0);
            }
            my = nxt;
        }
        w.left -= j1 - w.j;
        if (w.left > 0) walk_next_unit<BS>(a, w);
    }
    // Do not leave the CTA while copies into its shared memory are in flight.
    if (lane == 0) {
        const uint32_t first = issued > (uint32_t)kStages ? issued - kStages : 0u;
        for (uint32_t qi = first; qi < issued; ++qi)
            if (!mbar_wait_bounded(&full_bar[qi % kStages], (qi / kStages) & 1u)) break;
    }
}

// Wait for a stage as a consumer (all 32 lanes).  The verdict is a warp vote,
// so the warp-collective work that follows runs on all lanes or on none; once
// anything failed the warp stops waiting and the CTA is told.
__device__ __forceinline__ bool consumer_wait(const AttnArgs& a, uint64_t* bar, uint32_t parity,
                                              bool ok, volatile int* s_abort) {
    bool good = ok && !*s_abort;
    if (good && !mbar_wait_bounded(bar, parity)) {
        good = false;
        atomicOr(a.err, kErrTimeout);
        *s_abort = 1;
    }
    return __all_sync(0xffffffffu, good);
}

// Combine two online-softmax states of one row: weights a1, a2 for the two
// accumulators, and the combined (m, l).
__device__ __forceinline__ void merge_weights(float& m, float& l, float m2, float l2, float& a1,
                                              float& a2) {
    const float mn = fmaxf(m, m2);
    const float mb = mn == -INFINITY ? 0.f : mn;
    a1 = fast_exp2(m - mb);
    a2 = fast_exp2(m2 - mb);
    l = a1 * l + a2 * l2;
    m = mn;
}

// ===================== narrow consumer (rows <= 8) =====================
// Warp w takes blocks g == w (mod 8).  Per 16-token tile of a block:
//   S^T[tok][row] = K[tok][:] . Q^T[:][row]       (A = K tile via ldmatrix, B = Q^T)
//   P^T B-fragment = movmatrix.trans of bf16(S^T) (rows move from the column
//                    index of the accumulator to the lane index of the operand)
//   O^T[d][row]  += V^T[d][tok] . P^T[tok][row]    (A = V tile via ldmatrix.trans)
// Lane (g, t) holds rows 2t, 2t+1 of the softmax state; a row's max and sum
// reduce over the 8 lanes sharing t.
//
// Per-(block, KV head) scales (BLK): the K scale of a tile's block joins that
// tile's score scale; the V scale multiplies the tile's probabilities
// relative to vrun, the largest V scale the warp has met in this unit (the
// accumulator is rescaled when vrun grows, the running sum l is not), and the
// accumulator is multiplied by vrun at the unit's end.
template <int D, int BS, bool OUT_F32, bool KV8, bool BLK>
__device__ __forceinline__ void consume_narrow(const AttnArgs& a, Walk w, uint8_t* stages,
                                               const uint8_t* slots, float* scratch,
                                               uint64_t* full_bar, uint64_t* empty_bar,
                                               volatile int* s_abort, int4& info0, int4& info1) {
    using C = AttnCfg<D, BS, kModeNarrow, KV8, BLK>;
    constexpr int kStages = C::kStages;
    constexpr int MT = D / 16;   // 16-wide head_dim tiles (M of the PV product)
    constexpr int KT = D / 16;   // 16-deep k steps of the score product
    constexpr int PT = BS / 16;  // 16-token tiles per block
    constexpr int WN = kConsumerWarps;
    constexpr int SBS = C::kBlocksPerStage;
    constexpr int UT = SBS * PT;  // 16-token tiles per stage
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3, mi = lane >> 3, rr = lane & 7;
    const int R = a.rows, cta = blockIdx.x;
    float* emit_tile = scratch + C::kMergeBytes / 4;
    float* emit_ml = emit_tile + kNarrowRows * C::kTileStride;

    uint32_t gbase = 0;  // sequence number (in this CTA) of the piece's first stage
    bool ok = true;
    int piece = 0;
    while (w.left > 0) {
        const int j0 = w.j, j1 = piece_end(w);
        const int ctx = w.ctx, s = w.s, h = w.h;

        // Q^T as B fragments: (k = head_dim 2t.., n = row g); rows >= R are zero.
        // 8-bit caches: f16, in the permuted k order of the K fragments.
        uint32_t qb[KT][2];
        {
            int i, hq;
            const bool valid = unit_row(a, w.t, h, g, i, hq);
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)s * a.q_len + i) * a.n_q + hq) * D);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                if constexpr (KV8) {
                    const uint2 w2 = valid ? __ldg(reinterpret_cast<const uint2*>(qrow) + kk * 4 + t)
                                           : make_uint2(0u, 0u);
                    qb[kk][0] = bf16x2_to_f16x2(w2.x);
                    qb[kk][1] = bf16x2_to_f16x2(w2.y);
                } else {
                    qb[kk][0] = valid ? __ldg(qrow + kk * 8 + t) : 0u;
                    qb[kk][1] = valid ? __ldg(qrow + kk * 8 + 4 + t) : 0u;
                }
            }
        }
        // Per-unit scales: the K dequantisation scale joins the score scale,
        // the V one the final normalisation (per-block scales come per stage).
        const float sl2 = (KV8 && !BLK) ? a.scale_log2 * __ldg(a.k_scale + h) : a.scale_log2;
        const float vsc = (KV8 && !BLK) ? __ldg(a.v_scale + h) : 1.f;
        float vrun = 0.f;  // BLK: largest V scale of this unit so far
        // Row r sees tokens lo..lim: lim = its position, lo = lim - W + 1
        // with a window (INT_MIN without); padding rows see nothing.
        int lim[2], lo[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            int ie, he;
            lim[e] = unit_row(a, w.t, h, 2 * t + e, ie, he) ? ctx - a.q_len + ie : -1;
            lo[e] = a.window > 0 ? lim[e] - a.window + 1 : INT_MIN;
        }
        // smallest causal limit and largest window start of the tile's real rows
        const int lim_min = ctx - a.q_len + tile_first_token(a, w.t);
        const int lo_max =
            a.window > 0 ? ctx - a.q_len + tile_last_token(a, w.t) - a.window + 1 : INT_MIN;

        float o[MT][4];
#pragma unroll
        for (int n = 0; n < MT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

        // Warp w takes stages q == w (mod WN); stage q holds blocks
        // q*SBS .. q*SBS + nb - 1 of the piece.  Tile u of its SBS * PT
        // 16-token tiles belongs to block u / PT.
        const int ns = (j1 - j0 + SBS - 1) / SBS;
        const int first = static_cast<int>((uint32_t)(warp + WN - (int)(gbase % WN)) % WN);
        for (int q = first; q < ns; q += WN) {
            const uint32_t gidx = gbase + q;
            const uint32_t stage = gidx % kStages;
            ok = consumer_wait(a, &full_bar[stage], (gidx / kStages) & 1u, ok, s_abort);
            const int nb = min(SBS, j1 - j0 - q * SBS);  // blocks in this stage
            if (ok) {
                const uint32_t sb = smem_addr(stages + stage * C::kStageBytes);
                // BLK: this stage's block scales; kf = score scale x K scale,
                // rat = V scale / vrun, vfac rescales the accumulator when vrun grows.
                float kf[SBS], rat[SBS], vfac = 1.f;
#pragma unroll
                for (int b = 0; b < SBS; ++b) kf[b] = sl2;
                if constexpr (BLK) {
                    float vs[SBS], smax = 0.f;
#pragma unroll
                    for (int b = 0; b < SBS; ++b) {
                        const float2 sc = b < nb ? *reinterpret_cast<const float2*>(
                                                       slots + (stage * SBS + b) * 16)
                                                 : make_float2(0.f, 0.f);
                        kf[b] = sl2 * sc.x;
                        vs[b] = sc.y;
                        smax = fmaxf(smax, sc.y);
                    }
                    if (smax > vrun) {
                        vfac = vrun / smax;
                        vrun = smax;
                    }
                    const float rinv = vrun > 0.f ? kPShiftSync / vrun : 0.f;
#pragma unroll
                    for (int b = 0; b < SBS; ++b) rat[b] = vs[b] * rinv;
                }
                // ---- S^T = K Q^T, two interleaved accumulators per 16-token tile
                float st[UT][4], st2[UT][4];
#pragma unroll
                for (int u = 0; u < UT; ++u)
#pragma unroll
                    for (int e = 0; e < 4; ++e) st[u][e] = st2[u][e] = 0.f;
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    const int bi = u / PT, tp = u % PT;
                    if (bi >= nb) continue;
                    const uint32_t kb = C::k_tile(sb, bi);
                    if constexpr (KV8) {
                        // One x4 load: tokens (0-7, 8-15) x bytes (32j.., 32j+16..) = two k steps.
#pragma unroll
                        for (int j = 0; j < D / 32; ++j) {
                            uint32_t r[4];
                            ldmatrix_x4(r, kb + swz8<D>(tp * 16 + (mi & 1) * 8 + rr,
                                                        32 * j + (mi >> 1) * 16));
                            uint32_t k0[4], k1[4];  // A fragments of k steps 2j, 2j + 1
                            e4m3x4_to_f16x2x2(r[0], k0[0], k0[2]);
                            e4m3x4_to_f16x2x2(r[1], k0[1], k0[3]);
                            e4m3x4_to_f16x2x2(r[2], k1[0], k1[2]);
                            e4m3x4_to_f16x2x2(r[3], k1[1], k1[3]);
                            mma_f16_16816(st[u], k0, qb[2 * j][0], qb[2 * j][1]);
                            mma_f16_16816(st2[u], k1, qb[2 * j + 1][0], qb[2 * j + 1][1]);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk) {
                            uint32_t ka[4];
                            ldmatrix_x4(ka, kb + swz<BS>(tp * 16 + (mi & 1) * 8 + rr,
                                                          kk * 16 + (mi >> 1) * 8));
                            if (kk & 1)
                                mma_bf16_16816(st2[u], ka, qb[kk][0], qb[kk][1]);
                            else
                                mma_bf16_16816(st[u], ka, qb[kk][0], qb[kk][1]);
                        }
                    }
                }

                // ---- scale, causal / window / tail mask, online softmax (base 2)
                float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    const int bi = u / PT, tp = u % PT;
                    const int tok0 = (j0 + q * SBS + bi) * BS;
                    const bool need_mask = tok0 + BS - 1 > lim_min || tok0 < lo_max;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float x = (st[u][e] + st2[u][e]) * kf[bi];
                        const int tk = tok0 + tp * 16 + g + (e >> 1) * 8;
                        if (bi >= nb || (need_mask && (tk > lim[e & 1] || tk < lo[e & 1])))
                            x = -INFINITY;
                        st[u][e] = x;
                        mloc[e & 1] = fmaxf(mloc[e & 1], x);
                    }
                }
                float alpha[2], mbase[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mloc[e] = fmaxf(mloc[e], __shfl_xor_sync(0xffffffffu, mloc[e], 4));
                    mloc[e] = fmaxf(mloc[e], __shfl_xor_sync(0xffffffffu, mloc[e], 8));
                    mloc[e] = fmaxf(mloc[e], __shfl_xor_sync(0xffffffffu, mloc[e], 16));
                    const float mnew = fmaxf(m[e], mloc[e]);
                    mbase[e] = mnew == -INFINITY ? 0.f : mnew;
                    alpha[e] = fast_exp2(m[e] - mbase[e]);
                    m[e] = mnew;
                }
                float rsum[2] = {0.f, 0.f};
#pragma unroll
                for (int u = 0; u < UT; ++u) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p = fast_exp2(st[u][e] - mbase[e & 1]);
                        st[u][e] = p;
                        rsum[e & 1] += p;
                    }
                }
                l[0] = l[0] * alpha[0] + rsum[0];
                l[1] = l[1] * alpha[1] + rsum[1];
                if constexpr (BLK) {
                    // the accumulator also follows vrun; the probabilities of each
                    // block are weighed by its V scale relative to vrun
                    alpha[0] *= vfac;
                    alpha[1] *= vfac;
#pragma unroll
                    for (int u = 0; u < UT; ++u)
#pragma unroll
                        for (int e = 0; e < 4; ++e) st[u][e] *= rat[u / PT];
                }
                if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
                    for (int n = 0; n < MT; ++n) {
                        o[n][0] *= alpha[0];
                        o[n][1] *= alpha[1];
                        o[n][2] *= alpha[0];
                        o[n][3] *= alpha[1];
                    }
                }

                // ---- P^T as B fragments: pack (tok g, rows 2t..) then transpose
                // (bf16 against a bf16 cache, f16 against an 8-bit one)
                uint32_t pb[UT][2], pl[UT][2];
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    if constexpr (KV8) {
                        const uint32_t h0 = pack_f16x2(st[u][0], st[u][1]);
                        const uint32_t h1 = pack_f16x2(st[u][2], st[u][3]);
                        pb[u][0] = movmatrix_trans(h0);
                        pb[u][1] = movmatrix_trans(h1);
                        if (OUT_F32) {
                            pl[u][0] = movmatrix_trans(pack_f16x2(st[u][0] - f16_lo_to_f32(h0),
                                                                  st[u][1] - f16_hi_to_f32(h0)));
                            pl[u][1] = movmatrix_trans(pack_f16x2(st[u][2] - f16_lo_to_f32(h1),
                                                                  st[u][3] - f16_hi_to_f32(h1)));
                        }
                    } else {
                        const uint32_t h0 = pack_bf16x2(st[u][0], st[u][1]);
                        const uint32_t h1 = pack_bf16x2(st[u][2], st[u][3]);
                        pb[u][0] = movmatrix_trans(h0);
                        pb[u][1] = movmatrix_trans(h1);
                        if (OUT_F32) {
                            pl[u][0] = movmatrix_trans(pack_bf16x2(st[u][0] - bf16_lo_to_f32(h0),
                                                                   st[u][1] - bf16_hi_to_f32(h0)));
                            pl[u][1] = movmatrix_trans(pack_bf16x2(st[u][2] - bf16_lo_to_f32(h1),
                                                                   st[u][3] - bf16_hi_to_f32(h1)));
                        }
                    }
                }

                // ---- O^T += V^T P^T (V rows past the context are zeroed: they may hold NaN)
#pragma unroll
                for (int u = 0; u < UT; ++u) {
                    const int bi = u / PT, tp = u % PT;
                    if (bi >= nb) continue;
                    const uint32_t vb = C::v_tile(sb, bi);
                    const int tok0 = (j0 + q * SBS + bi) * BS;
                    // Only a unit's last block reaches past the context: the
                    // masked form runs there alone (the warp-uniform branch
                    // spares every other tile the mask instructions).
                    auto pv_tile = [&](auto masked) {
                        constexpr bool kMasked = decltype(masked)::value;
                        uint32_t vm0 = 0xFFFFFFFFu, vm8 = 0xFFFFFFFFu;
                        if (kMasked) {
                            const int ta = tok0 + tp * 16 + 2 * t;
                            vm0 = (ta < ctx ? 0x0000FFFFu : 0u) |
                                  (ta + 1 < ctx ? 0xFFFF0000u : 0u);
                            vm8 = (ta + 8 < ctx ? 0x0000FFFFu : 0u) |
                                  (ta + 9 < ctx ? 0xFFFF0000u : 0u);
                        }
                        if constexpr (KV8) {
                            // x4.trans over tokens (0-7, 8-15) x bytes (32j.., 32j+16..): lane
                            // (g, t) gets d (2g, 2g+1) of tokens (2t, 2t+1); the permute splits
                            // them into the even-d and odd-d A fragments (M rows g, g+8 are
                            // d 32j + 2g (+1) and 32j + 16 + 2g (+1)).
#pragma unroll
                            for (int j = 0; j < D / 32; ++j) {
                                uint32_t r[4];
                                ldmatrix_x4_trans(r, vb + swz8<D>(tp * 16 + (mi & 1) * 8 + rr,
                                                                  32 * j + (mi >> 1) * 16));
                                uint32_t ev[4], od[4];
#pragma unroll
                                for (int mm = 0; mm < 4; ++mm)
                                    e4m3x4_to_f16x2x2(prmt(r[mm], 0u, 0x3120u), ev[mm], od[mm]);
                                uint32_t ae[4] = {ev[0], ev[2], ev[1], ev[3]};
                                uint32_t ao[4] = {od[0], od[2], od[1], od[3]};
                                if constexpr (kMasked) {
                                    ae[0] &= vm0; ae[1] &= vm0; ae[2] &= vm8; ae[3] &= vm8;
                                    ao[0] &= vm0; ao[1] &= vm0; ao[2] &= vm8; ao[3] &= vm8;
                                }
                                mma_f16_16816(o[2 * j], ae, pb[u][0], pb[u][1]);
                                mma_f16_16816(o[2 * j + 1], ao, pb[u][0], pb[u][1]);
                                if (OUT_F32) {
                                    mma_f16_16816(o[2 * j], ae, pl[u][0], pl[u][1]);
                                    mma_f16_16816(o[2 * j + 1], ao, pl[u][0], pl[u][1]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int dm = 0; dm < MT; ++dm) {
                                uint32_t va[4];
                                ldmatrix_x4_trans(va, vb + swz<BS>(tp * 16 + (mi >> 1) * 8 + rr,
                                                                    dm * 16 + (mi & 1) * 8));
                                if constexpr (kMasked) {
                                    va[0] &= vm0;
                                    va[1] &= vm0;
                                    va[2] &= vm8;
                                    va[3] &= vm8;
                                }
                                mma_bf16_16816(o[dm], va, pb[u][0], pb[u][1]);
                                if (OUT_F32) mma_bf16_16816(o[dm], va, pl[u][0], pl[u][1]);
                            }
                        }
                    };
                    if (tok0 + BS > ctx)
                        pv_tile(std::true_type{});
                    else
                        pv_tile(std::false_type{});
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
        }
        gbase += ns;

        // ---- row sums across the 8 lanes of a row, then combine the warps' partials
        if constexpr (BLK) {  // the accumulator in value units (vrun is warp-uniform)
            const float back = vrun * kPShiftSyncInv;
#pragma unroll
            for (int n = 0; n < MT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] *= back;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
        }
        for (int step = WN >> 1; step >= 1; step >>= 1) {
            if (warp >= step && warp < 2 * step) {
                float* sl = scratch + (size_t)(warp - step) * 32 * C::kLaneFloats;
#pragma unroll
                for (int n = 0; n < MT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sl[(n * 4 + e) * 32 + lane] = o[n][e];
                sl[(MT * 4 + 0) * 32 + lane] = m[0];
                sl[(MT * 4 + 1) * 32 + lane] = m[1];
                sl[(MT * 4 + 2) * 32 + lane] = l[0];
                sl[(MT * 4 + 3) * 32 + lane] = l[1];
            }
            named_barrier_sync(1, kConsumerThreads);
            if (warp < step) {
                const float* sl = scratch + (size_t)warp * 32 * C::kLaneFloats;
                float a1[2], a2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    merge_weights(m[e], l[e], sl[(MT * 4 + e) * 32 + lane],
                                  sl[(MT * 4 + 2 + e) * 32 + lane], a1[e], a2[e]);
#pragma unroll
                for (int n = 0; n < MT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[n][e] = a1[e & 1] * o[n][e] + a2[e & 1] * sl[(n * 4 + e) * 32 + lane];
            }
            named_barrier_sync(1, kConsumerThreads);
        }

        // ---- emit (warp 0): through a row-major tile, then 16-byte stores
        const bool first_piece = j0 == w.jlo, last_piece = j1 == w.nb;
        const bool whole = first_piece && last_piece;
        if (warp == 0) {
            float scl[2];
#pragma unroll
            for (int e = 0; e < 2; ++e)
                scl[e] = (whole ? (l[e] > 0.f ? 1.f / l[e] : 0.f) : 1.f) * vsc;
#pragma unroll
            for (int n = 0; n < MT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // d of accumulator element (n, e): see the PV product above
                    const int dcol = KV8 ? (n >> 1) * 32 + (e >> 1) * 16 + 2 * g + (n & 1)
                                         : n * 16 + g + (e >> 1) * 8;
                    emit_tile[(2 * t + (e & 1)) * C::kTileStride + dcol] = o[n][e] * scl[e & 1];
                }
            if (g == 0) {
                emit_ml[(2 * t) * 2 + 0] = m[0];
                emit_ml[(2 * t) * 2 + 1] = l[0];
                emit_ml[(2 * t + 1) * 2 + 0] = m[1];
                emit_ml[(2 * t + 1) * 2 + 1] = l[1];
            }
            __syncwarp();
            if (whole) {
                constexpr int V = OUT_F32 ? 4 : 8;  // elements per 16-byte store
                for (int idx = lane; idx < R * (D / V); idx += 32) {
                    const int r = idx / (D / V), c = (idx % (D / V)) * V;
                    int i, hq;
                    if (!unit_row(a, w.t, h, r, i, hq)) continue;
                    const size_t ob = (((size_t)s * a.q_len + i) * a.n_q + hq) * D + c;
                    const float* src = emit_tile + r * C::kTileStride + c;
                    if (OUT_F32) {
                        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + ob) =
                            make_float4(src[0], src[1], src[2], src[3]);
                    } else {
                        uint4 v;
                        v.x = pack_bf16x2(src[0], src[1]);
                        v.y = pack_bf16x2(src[2], src[3]);
                        v.z = pack_bf16x2(src[4], src[5]);
                        v.w = pack_bf16x2(src[6], src[7]);
                        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ob) = v;
                    }
                }
            } else {
                const int slot = piece == 0 ? 0 : 1;
                const size_t rec = (size_t)cta * 2 + slot;
                for (int idx = lane; idx < R * (D / 4); idx += 32) {
                    const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
                    const float* src = emit_tile + r * C::kTileStride + c;
                    *reinterpret_cast<float4*>(a.rec_o + (rec * R + r) * D + c) =
                        make_float4(src[0], src[1], src[2], src[3]);
                }
                if (lane < R)
                    *reinterpret_cast<float2*>(a.rec_ml + (rec * R + lane) * 2) =
                        make_float2(emit_ml[lane * 2], emit_ml[lane * 2 + 1]);
                const int4 rinfo = make_int4(
                    s, h, kRecValid | (first_piece ? kRecFirst : 0) | (last_piece ? kRecLast : 0),
                    w.t);
                if (slot == 0)
                    info0 = rinfo;
                else
                    info1 = rinfo;
            }
            __syncwarp();
        }
        ++piece;
        w.left -= j1 - w.j;
        if (w.left > 0) walk_next_unit<BS>(a, w);
    }
}

// ===================== wide consumer (rows > 8) =====================
// Warp w owns 16-row slice (w % WM) of the unit's rows and blocks g == w / WM
// (mod WN), WM * WN = 8.  S = Q K^T (A = Q rows, B = K via ldmatrix), P stays
// in registers as the A operand of O += P V (B = V via ldmatrix.trans).
// Per-(block, KV head) scales (BLK): as in the narrow consumer -- the K scale
// of a chunk's block joins its score scale, its V scale weighs the chunk's
// probabilities relative to vrun, and the accumulator follows vrun.
template <int D, int BS, bool OUT_F32, bool KV8, bool BLK>
__device__ __forceinline__ void consume_wide(const AttnArgs& a, Walk w, uint8_t* stages,
                                             const uint8_t* slots, float* scratch,
                                             uint64_t* full_bar, uint64_t* empty_bar,
                                             volatile int* s_abort, int4& info0, int4& info1) {
    using C = AttnCfg<D, BS, kModeWide, KV8, BLK>;
    constexpr int kStages = C::kStages;
    constexpr int SBS = C::kBlocksPerStage;
    constexpr int NT = D / 8;    // 8-wide output column tiles
    constexpr int KT = D / 16;   // 16-deep k steps over head_dim
    constexpr int PT = BS / 16;  // 16-token chunks per block
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int WM = a.warp_rows;
    const int WN = kConsumerWarps / WM;
    const int mt = warp % WM;   // which 16-row slice of the unit's rows
    const int col = warp / WM;  // which residue class of blocks
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const int cta = blockIdx.x;

    uint32_t gbase = 0;
    bool ok = true;
    int piece = 0;
    while (w.left > 0) {
        const int j0 = w.j, j1 = piece_end(w);
        const int ctx = w.ctx, s = w.s, h = w.h;

        // Query fragments of this unit's two rows per thread (rows >= a.rows are zero).
        uint32_t qf[KT][4];
        int lim[2], lo[2];  // row sees tokens lo..lim (lo = INT_MIN without a window)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = mt * 16 + g + hh * 8;
            int i, hq;
            const bool valid = unit_row(a, w.t, h, r, i, hq);
            lim[hh] = valid ? ctx - a.q_len + i : -1;
            lo[hh] = a.window > 0 ? lim[hh] - a.window + 1 : INT_MIN;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)s * a.q_len + i) * a.n_q + hq) * D);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                if constexpr (KV8) {
                    // f16, in the permuted k order of the 8-bit K fragments
                    const uint2 w2 = valid ? __ldg(reinterpret_cast<const uint2*>(qrow) + kk * 4 + t)
                                           : make_uint2(0u, 0u);
                    qf[kk][hh] = bf16x2_to_f16x2(w2.x);
                    qf[kk][2 + hh] = bf16x2_to_f16x2(w2.y);
                } else {
                    qf[kk][hh] = valid ? __ldg(qrow + kk * 8 + t) : 0u;
                    qf[kk][2 + hh] = valid ? __ldg(qrow + kk * 8 + 4 + t) : 0u;
                }
            }
        }
        const float sl2 = (KV8 && !BLK) ? a.scale_log2 * __ldg(a.k_scale + h) : a.scale_log2;
        const float vsc = (KV8 && !BLK) ? __ldg(a.v_scale + h) : 1.f;
        float vrun = 0.f, vinv = 0.f;  // BLK: largest V scale of this unit so far; headroom / it
        // smallest causal limit and largest window start of the tile's real rows
        const int lim_min = ctx - a.q_len + tile_first_token(a, w.t);
        const int lo_max =
            a.window > 0 ? ctx - a.q_len + tile_last_token(a, w.t) - a.window + 1 : INT_MIN;

        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

        // Column col takes stages q == col (mod WN); stage q holds blocks
        // q*SBS .. q*SBS + nb - 1 of the piece.
        const int ns = (j1 - j0 + SBS - 1) / SBS;
        const int first = static_cast<int>((uint32_t)(col + WN - (int)(gbase % WN)) % WN);
        for (int q = first; q < ns; q += WN) {
            const uint32_t gidx = gbase + q;
            const uint32_t stage = gidx % kStages;
            ok = consumer_wait(a, &full_bar[stage], (gidx / kStages) & 1u, ok, s_abort);
            const int nb = min(SBS, j1 - j0 - q * SBS);  // blocks in this stage
            if (ok) {
                const uint32_t sb = smem_addr(stages + stage * C::kStageBytes);
                const uint8_t* sslot = slots + stage * SBS * 16;  // BLK: the blocks' scales
                if constexpr (BLK) {
                    float smax = 0.f;
                    for (int b = 0; b < nb; ++b)
                        smax = fmaxf(smax, reinterpret_cast<const float*>(sslot + b * 16)[1]);
                    if (smax > vrun) {
                        const float vfac = vrun / smax;
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) o[n][e] *= vfac;
                        vrun = smax;
                        vinv = kPShiftSync / smax;
                    }
                }

                // The stage's blocks are taken 16 tokens at a time (one
                // online-softmax update per chunk): chunk u is token tile
                // u % PT of block u / PT.  This keeps the live registers low.
#pragma unroll 1
                for (int u = 0; u < nb * PT; ++u) {
                    const int bi = u / PT, tp = u % PT;
                    const int j = j0 + q * SBS + bi;
                    const uint32_t kbase = C::k_tile(sb, bi);
                    const uint32_t vbase = C::v_tile(sb, bi);
                    // ---- S = Q K^T over 16 tokens
                    float sc[2][4];
#pragma unroll
                    for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                    if constexpr (KV8) {
                        // x4: tokens (0-7, 8-15) x bytes (32j.., 32j+16..); lane (g, t)
                        // holds d 4t..4t+3 of token g: (lo pair, hi pair) = (b0, b1).
#pragma unroll
                        for (int j = 0; j < D / 32; ++j) {
                            uint32_t r[4];
                            ldmatrix_x4(r, kbase + swz8<D>(tp * 16 + (mi & 1) * 8 + rr,
                                                           32 * j + (mi >> 1) * 16));
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                uint32_t b0, b1;
                                e4m3x4_to_f16x2x2(r[m], b0, b1);
                                mma_f16_16816(sc[m & 1], qf[2 * j + (m >> 1)], b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk) {
                            uint32_t b[4];
                            ldmatrix_x4(b, kbase + swz<BS>(tp * 16 + (mi >> 1) * 8 + rr,
                                                            kk * 16 + (mi & 1) * 8));
                            mma_bf16_16816(sc[0], qf[kk], b[0], b[1]);
                            mma_bf16_16816(sc[1], qf[kk], b[2], b[3]);
                        }
                    }

                    // ---- scale, causal / window / tail mask, online softmax (base 2)
                    const int tok0 = j * BS + tp * 16;
                    const bool need_mask = tok0 + 15 > lim_min || tok0 < lo_max;
                    float kfb = sl2, ratb = 1.f;  // BLK: this block's score factor, V weight
                    if constexpr (BLK) {
                        const float2 bsc = *reinterpret_cast<const float2*>(sslot + bi * 16);
                        kfb = sl2 * bsc.x;
                        ratb = bsc.y * vinv;
                    }
                    float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float x = sc[n][e] * kfb;
                            const int tk = tok0 + n * 8 + 2 * t + (e & 1);
                            if (need_mask && (tk > lim[e >> 1] || tk < lo[e >> 1])) x = -INFINITY;
                            sc[n][e] = x;
                            mloc[e >> 1] = fmaxf(mloc[e >> 1], x);
                        }
                    }
                    float alpha[2], mbase[2];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        mloc[hh] = fmaxf(mloc[hh], __shfl_xor_sync(0xffffffffu, mloc[hh], 1));
                        mloc[hh] = fmaxf(mloc[hh], __shfl_xor_sync(0xffffffffu, mloc[hh], 2));
                        const float mnew = fmaxf(m[hh], mloc[hh]);
                        mbase[hh] = mnew == -INFINITY ? 0.f : mnew;
                        alpha[hh] = fast_exp2(m[hh] - mbase[hh]);
                        m[hh] = mnew;
                    }
                    float rsum[2] = {0.f, 0.f};
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p = fast_exp2(sc[n][e] - mbase[e >> 1]);
                            sc[n][e] = p;
                            rsum[e >> 1] += p;
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) l[hh] = l[hh] * alpha[hh] + rsum[hh];
                    if constexpr (BLK) {
#pragma unroll
                        for (int n = 0; n < 2; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) sc[n][e] *= ratb;
                    }
                    if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            o[n][0] *= alpha[0];
                            o[n][1] *= alpha[0];
                            o[n][2] *= alpha[1];
                            o[n][3] *= alpha[1];
                        }
                    }

                    // ---- P as bf16 (f16 for an 8-bit cache) A fragments (fp32
                    //      output: hi + lo pair)
                    uint32_t pa[4], pl[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int n = q2 >> 1;
                        const int e = (q2 & 1) * 2;
                        const float p0 = sc[n][e], p1 = sc[n][e + 1];
                        if constexpr (KV8) {
                            pa[q2] = pack_f16x2(p0, p1);
                            if (OUT_F32)
                                pl[q2] = pack_f16x2(p0 - f16_lo_to_f32(pa[q2]),
                                                    p1 - f16_hi_to_f32(pa[q2]));
                        } else {
                            pa[q2] = pack_bf16x2(p0, p1);
                            if (OUT_F32)
                                pl[q2] = pack_bf16x2(p0 - bf16_lo_to_f32(pa[q2]),
                                                     p1 - bf16_hi_to_f32(pa[q2]));
                        }
                    }

                    // ---- O += P V (V rows past the context are zeroed: they may hold NaN)
                    uint32_t vm0 = 0xFFFFFFFFu, vm8 = 0xFFFFFFFFu;
                    if (tok0 + 16 > ctx) {
                        const int ta = tok0 + 2 * t;
                        vm0 = (ta < ctx ? 0x0000FFFFu : 0u) | (ta + 1 < ctx ? 0xFFFF0000u : 0u);
                        vm8 = (ta + 8 < ctx ? 0x0000FFFFu : 0u) | (ta + 9 < ctx ? 0xFFFF0000u : 0u);
                    }
                    if constexpr (KV8) {
                        // x4.trans over tokens (0-7, 8-15) x bytes (32j.., 32j+16..) and a
                        // byte permute: B fragments of the output columns
                        // d = 32j + 16h + 2c + parity, tile index 4j + 2h + parity.
#pragma unroll
                        for (int j = 0; j < D / 32; ++j) {
                            uint32_t r[4];
                            ldmatrix_x4_trans(r, vbase + swz8<D>(tp * 16 + (mi & 1) * 8 + rr,
                                                                 32 * j + (mi >> 1) * 16));
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {  // d 32j + 16 hh ..
                                uint32_t e0, o0, e1, o1;    // tokens 0-7 / 8-15, even / odd d
                                e4m3x4_to_f16x2x2(prmt(r[2 * hh], 0u, 0x3120u), e0, o0);
                                e4m3x4_to_f16x2x2(prmt(r[2 * hh + 1], 0u, 0x3120u), e1, o1);
                                e0 &= vm0;
                                o0 &= vm0;
                                e1 &= vm8;
                                o1 &= vm8;
                                mma_f16_16816(o[4 * j + 2 * hh], pa, e0, e1);
                                mma_f16_16816(o[4 * j + 2 * hh + 1], pa, o0, o1);
                                if (OUT_F32) {
                                    mma_f16_16816(o[4 * j + 2 * hh], pl, e0, e1);
                                    mma_f16_16816(o[4 * j + 2 * hh + 1], pl, o0, o1);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int dp = 0; dp < D / 16; ++dp) {
                            uint32_t b[4];
                            ldmatrix_x4_trans(b, vbase + swz<BS>(tp * 16 + (mi & 1) * 8 + rr,
                                                                  dp * 16 + (mi >> 1) * 8));
                            b[0] &= vm0;
                            b[1] &= vm8;
                            b[2] &= vm0;
                            b[3] &= vm8;
                            mma_bf16_16816(o[2 * dp], pa, b[0], b[1]);
                            mma_bf16_16816(o[2 * dp + 1], pa, b[2], b[3]);
                            if (OUT_F32) {
                                mma_bf16_16816(o[2 * dp], pl, b[0], b[1]);
                                mma_bf16_16816(o[2 * dp + 1], pl, b[2], b[3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
        }
        gbase += ns;

        // ---- row sums across the quad, then combine the WN column partials
        if constexpr (BLK) {  // the accumulator in value units (vrun is warp-uniform)
            const float back = vrun * kPShiftSyncInv;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] *= back;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
            l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
        }
        for (int step = WN >> 1; step >= 1; step >>= 1) {
            if (col >= step && col < 2 * step) {
                float* sl = scratch + (size_t)((col - step) * WM + mt) * 32 * C::kLaneFloats;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sl[(n * 4 + e) * 32 + lane] = o[n][e];
                sl[(NT * 4 + 0) * 32 + lane] = m[0];
                sl[(NT * 4 + 1) * 32 + lane] = m[1];
                sl[(NT * 4 + 2) * 32 + lane] = l[0];
                sl[(NT * 4 + 3) * 32 + lane] = l[1];
            }
            named_barrier_sync(1, kConsumerThreads);
            if (col < step) {
                const float* sl = scratch + (size_t)(col * WM + mt) * 32 * C::kLaneFloats;
                float a1[2], a2[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    merge_weights(m[hh], l[hh], sl[(NT * 4 + hh) * 32 + lane],
                                  sl[(NT * 4 + 2 + hh) * 32 + lane], a1[hh], a2[hh]);
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[n][e] = a1[e >> 1] * o[n][e] + a2[e >> 1] * sl[(n * 4 + e) * 32 + lane];
            }
            named_barrier_sync(1, kConsumerThreads);
        }

        // ---- emit: a whole unit goes straight to `out`; a piece becomes a record
        const bool first_piece = j0 == w.jlo, last_piece = j1 == w.nb;
        if (col == 0) {
            if (first_piece && last_piece) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g + hh * 8;
                    int i, hq;
                    if (!unit_row(a, w.t, h, r, i, hq)) continue;
                    const float inv = (l[hh] > 0.f ? 1.f / l[hh] : 0.f) * vsc;
                    const size_t ob = (((size_t)s * a.q_len + i) * a.n_q + hq) * D;
                    if constexpr (KV8) {
                        // tiles 4j + 2h + {0, 1} hold d = 32j + 16h + 4t + {0, 2} / {1, 3}
#pragma unroll
                        for (int n = 0; n < NT; n += 2) {
                            const size_t d0 = ob + (n >> 2) * 32 + ((n >> 1) & 1) * 16 + 4 * t;
                            const float v0 = o[n][2 * hh] * inv, v1 = o[n + 1][2 * hh] * inv;
                            const float v2 = o[n][2 * hh + 1] * inv, v3 = o[n + 1][2 * hh + 1] * inv;
                            if (OUT_F32)
                                *reinterpret_cast<float4*>(static_cast<float*>(a.out) + d0) =
                                    make_float4(v0, v1, v2, v3);
                            else
                                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + d0) =
                                    make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
                        }
                    } else {
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            const float v0 = o[n][2 * hh] * inv, v1 = o[n][2 * hh + 1] * inv;
                            if (OUT_F32)
                                *reinterpret_cast<float2*>(static_cast<float*>(a.out) + ob +
                                                           n * 8 + 2 * t) = make_float2(v0, v1);
                            else
                                *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + ob +
                                                             n * 8 + 2 * t) = pack_bf16x2(v0, v1);
                        }
                    }
                }
            } else {
                const int slot = piece == 0 ? 0 : 1;
                const size_t rec = (size_t)cta * 2 + slot;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g + hh * 8;
                    if (r >= a.rows) continue;
                    float* ro = a.rec_o + (rec * a.rows + r) * D;
                    if constexpr (KV8) {
#pragma unroll
                        for (int n = 0; n < NT; n += 2)
                            *reinterpret_cast<float4*>(ro + (n >> 2) * 32 + ((n >> 1) & 1) * 16 +
                                                       4 * t) =
                                make_float4(o[n][2 * hh] * vsc, o[n + 1][2 * hh] * vsc,
                                            o[n][2 * hh + 1] * vsc, o[n + 1][2 * hh + 1] * vsc);
                    } else {
#pragma unroll
                        for (int n = 0; n < NT; ++n)
                            *reinterpret_cast<float2*>(ro + n * 8 + 2 * t) =
                                make_float2(o[n][2 * hh], o[n][2 * hh + 1]);
                    }
                    if (t == 0)
                        *reinterpret_cast<float2*>(a.rec_ml + (rec * a.rows + r) * 2) =
                            make_float2(m[hh], l[hh]);
                }
                const int4 rinfo = make_int4(
                    s, h, kRecValid | (first_piece ? kRecFirst : 0) | (last_piece ? kRecLast : 0),
                    w.t);
                if (slot == 0)
                    info0 = rinfo;
                else
                    info1 = rinfo;
            }
        }
        ++piece;
        w.left -= j1 - w.j;
        if (w.left > 0) walk_next_unit<BS>(a, w);
    }
}

// ===================== TMEM consumer (rows > 64) =====================
// One row tile (R <= 128 rows, on the MMA's M = 128; rows >= R are padding
// whose scores are all masked) per unit, accumulators in TMEM.
// Keys are taken kKeys = 64 at a time: one ring stage holds a super-block
// of 64 / BS blocks with their K rows (and V rows) contiguous, so the three
// roles synchronise once per 64 keys and one score MMA spans them all:
//   warp 4, lane 0 -- QK issuer: S[g&1] = Q K^T for the super-block
//                     (tcgen05.mma, M = 128, N = 64; A = Q tile, B = K
//                     stage, both K-major) once its stage has landed and the
//                     softmax has loaded S[g&1] of super-block g-2;
//   warps 0..3     -- softmax, one thread per row (TMEM lane = row, so a row's
//                     max and sum never leave the thread): P[q&1] = bf16 of
//                     2^(S*scale - m) into TMEM, running sum l; O is rescaled
//                     in TMEM only when a row's max grew by more than 2^8 (the
//                     stale max is used consistently in P and l: exact);
//   warp 5, lane 0 -- PV issuer: O += P[g&1] V over the super-block's keys
//                     (A from TMEM, B = V stage, MN-major), then releases
//                     the stage.
// Scores therefore run up to two super-blocks ahead of the softmax, and the
// PV update of one overlaps the softmax of the next.  TMEM columns: O
// [0, 128), S 2 x 64 from 128, P 2 x 32 from 256, the low halves of P for
// fp32 output 2 x 32 from 320.
// Over an 8-bit cache (KV8) five converter warps (6, 7, 9, 10, 11) widen each
// landed stage into one of three f16 copies (K and V in the layout the bf16
// stages have, V rows past the context zeroed) and free the stage; the MMAs read the copies as kind::f16
// with Q and P in f16 (every e4m3 value is exact in f16), and the PV product
// frees the copy.  The per-head K scale joins the score scale, the V scale
// the normalisation.
// The query tile of unit (sequence s, KV head h, row tile t) by TMA (query
// map present): D/64 boxes of 64 columns x a.rows rows, landing as the
// swizzled K-major tile the score MMA reads (64-column region r at
// r * QROWS * 128 bytes); completes on `bar`.  Rows of a
// partial tile past a.rows keep stale bits; their scores are all masked.
template <int D, int QROWS>
__device__ __forceinline__ void issue_q_tile(const AttnArgs& a, const CUtensorMap* tmap_q,
                                             uint8_t* qtile, uint64_t* bar, int s, int h, int t) {
    const int r0 = t * a.rows;
    const int y = h * a.group + r0 % a.group, z = s * a.q_len + r0 / a.group;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(D / 64) * 128u * static_cast<uint32_t>(a.rows));
#pragma unroll
    for (int half = 0; half < D / 64; ++half)
        tma_load_3d(qtile + half * QROWS * 128, tmap_q, half * 64, y, z, bar);
}

// Per-(block, KV head) scales (BLK, 8-bit cache only): the converter warps
// copy each super-block's K and V scales beside its f16 copy; the softmax
// multiplies each key's raw score by the score scale times its block's K
// scale before taking the row maximum, and weighs each block's probabilities
// by its V scale relative to vrun, the largest V scale of the unit so far (O
// is rescaled in TMEM when vrun grows, together with a grown maximum).
//
// T2 = 2 (the paired form, 256-row units over a bf16 cache, bf16 output):
// the unit's rows are two 128-row sub-tiles that share every stage.  Softmax
// warps 0-3 take sub-tile 0 and warps 4-7 sub-tile 1 (TMEM lanes again 0..127,
// in their own columns: O of sub-tile u at u * 128, its score slot at 256 +
// u * 64, its two P buffers at 384 + u * 64); warp 9 issues both score
// products of a stage, warp 10 both PV products, and a stage is freed when
// both are done.  Each sub-tile has one score slot: the softmax reads S at
// the start of its round, so the next stage's product can refill the slot
// while the exponentials run.  Half the stages per score FLOP (the producer
// spends ~60 ns of TMA issue per box, which bounded the one-tile form on
// chunked prefill) at the price of a 64 KB query tile (a five-stage ring).
template <int D, int BS, bool OUT_F32, bool KV8, bool BLK, int T2 = 1>
__device__ __forceinline__ void consume_tmem(const AttnArgs& a, Walk w, uint8_t* stages,
                                             const uint8_t* slots, uint8_t* qtile,
                                             const CUtensorMap* tmap_q, uint64_t* full_bar,
                                             uint64_t* empty_bar, uint64_t* tcb, uint32_t* s_tmem,
                                             volatile int* s_abort, int4& info0, int4& info1) {
    static_assert(!BLK || KV8, "block scales come with the 8-bit cache");
    static_assert(T2 == 1 || (!KV8 && !OUT_F32), "the paired form: bf16 cache, bf16 output");
    using C = AttnCfg<D, BS, T2 == 2 ? kModeTmem2 : kModeTmem, KV8, BLK>;
    constexpr int kStages = C::kStages;
    constexpr int kKeys = 64;                  // keys per softmax round
    constexpr int SB = C::kBlocksPerStage;     // blocks per super-block (= per stage)
    static_assert(SB * BS == kKeys, "a stage holds one super-block");
    constexpr uint32_t kTmemCols = 512;
    // O of sub-tile u at kColO + 128 u; score slots of 64 columns from kColS;
    // P buffers of 32 columns from kColP (two per sub-tile); fp32 output's low
    // halves of P from kColPL (one-tile form only)
    constexpr uint32_t kColO = 0, kColS = T2 == 2 ? 256 : 128, kColP = T2 == 2 ? 384 : 256,
                       kColPL = 320;
    // Over an 8-bit cache the query rows are the score product's A operand in
    // tensor memory, columns kColQ .. kColQ + D/2 (two f16 per column, the
    // lower index in the low half), each softmax thread storing its own row;
    // over bf16 the products read a query tile in shared memory.
    constexpr bool kQT = KV8;
    constexpr uint32_t kColQ = 384;
    constexpr int KT = D / 16;   // k steps of S = Q K^T
    constexpr int kQHalf = C::kQRows * 128;  // bytes of one 64-column half of the Q tile
    // warps 0..5 take part (paired: 0..7, 9, 10), and the converter warps 6, 7,
    // 9, 10, 11 over an 8-bit cache
    constexpr int kParty = KV8 ? threads_for(kModeTmem, true) - 32 : (T2 == 2 ? 320 : 192);
    constexpr int kQKWarp = T2 == 2 ? 9 : 4, kPVWarp = T2 == 2 ? 10 : 5;
    constexpr int kHalves = D / 64;          // 64-column regions of an f16 K or V copy
    // tcb: [0..1] S ready, [2..3] S read (per score slot), [4..7] P ready, [8..11] PV done
    //      (per sub-tile u and P buffer b: 2u + b), [12] QK teardown, [13] PV teardown,
    //      [14..16] f16 copy ready, [17..19] f16 copy read, [20] Q landed (TMA) or
    //      stored (tensor memory), [21] Q read
    uint64_t* s_full = tcb;
    uint64_t* s_free = tcb + 2;
    uint64_t* p_full = tcb + 4;
    uint64_t* pv_done = tcb + 8;
    constexpr uint32_t kCopies = C::kCvtCopies;
    uint64_t* cvt_full = tcb + 14;  // 8-bit cache: f16 copy [g % kCopies] ready
    uint64_t* cvt_free = tcb + 17;  // 8-bit cache: f16 copy [g % kCopies] read by its PV product
    uint64_t* q_full = tcb + 20;    // query tile landed (TMA), or stored into tensor memory
    uint64_t* q_empty = tcb + 21;   // the piece's score products have read the query tile
    // Score slot of stage g for sub-tile u, and the parity of its g-th use.
    auto sslot = [](uint32_t g, int u) -> uint32_t { return T2 == 2 ? (uint32_t)u : (g & 1u); };
    auto spar = [](uint32_t g) -> uint32_t { return T2 == 2 ? (g & 1u) : ((g >> 1) & 1u); };
    // f16 copies (8-bit cache): copy c at cvt + c * kCopy, K regions then V regions
    uint8_t* cvt = qtile + C::kQTileBytes;
    constexpr int kCopy = 2 * kHalves * C::kCvtRegion;
    // BLK: scales of the super-block in f16 copy c: [c][block][K, V]
    float* cvt_sc = reinterpret_cast<float*>(cvt + C::kCvtBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!KV8 && T2 == 1 && warp > 5) return;  // warps 6, 7 have no part in this mode over bf16
    const bool softmax = warp < 4 * T2;
    const int sub = T2 == 2 ? ((warp >> 2) & 1) : 0;  // softmax threads: their sub-tile
    const int row = threadIdx.x & 127;                // softmax threads: row = TMEM lane
    const int trow = sub * 128 + row;                 // ... and their row of the unit's tile
    const int R = a.rows, cta = blockIdx.x;

    if (warp == 0) tmem_alloc(s_tmem, kTmemCols);
    tc_fence_before();
    named_barrier_sync(2, kParty);
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const uint32_t tlane = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t idesc_qk = KV8 ? umma_idesc_f16(128, kKeys, false) : umma_idesc_bf16(128, kKeys, false);
    const uint32_t idesc_pv = KV8 ? umma_idesc_f16(128, D, true) : umma_idesc_bf16(128, D, true);
    const uint32_t q_saddr = smem_addr(qtile);
    // bf16 tiles at d 128 by one 4-D copy each: a stage's K and V regions are
    // [block][8-row group][half][8 rows][128 bytes] (uniform 2048-byte stride
    // between 8-row groups, halves 1024 bytes apart)
    const bool g4 = !KV8 && C::kBoxes == 2 && a.tile_4d;

    auto issuer_fail = [&](bool& ok) {
        ok = false;
        atomicOr(a.err, kErrTimeout);
        *s_abort = 1;
    };
    // 8-bit cache: this thread's query row of the unit at walk position wq,
    // or null for a row outside the unit.
    auto q_row_src = [&](const Walk& wq) -> const uint4* {
        int iq = 0, hq = 0;
        if (!unit_row(a, wq.t, wq.h, trow, iq, hq)) return nullptr;
        return reinterpret_cast<const uint4*>(a.q + (((size_t)wq.s * a.q_len + iq) * a.n_q + hq) * D);
    };
    // ... as raw bf16 pairs (zeros outside the unit): tensor-memory columns
    // 0..31 of the row in q0, 32..63 (head_dim 128) in q1.
    auto q_rows_load = [&](const Walk& wq, uint32_t (&q0)[32], uint32_t (&q1)[32]) {
        const uint4* src = q_row_src(wq);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = src ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            if (c < 8) {
                q0[4 * c] = v.x, q0[4 * c + 1] = v.y, q0[4 * c + 2] = v.z, q0[4 * c + 3] = v.w;
            } else {
                q1[4 * c - 32] = v.x, q1[4 * c - 31] = v.y, q1[4 * c - 30] = v.z,
                q1[4 * c - 29] = v.w;
            }
        }
    };
    // ... widened to f16 (the f16 products take f16 on both sides), stored
    // as the thread's lane of the A operand, and announced to the score issuer.
    auto q_rows_store = [&](uint32_t (&q0)[32], uint32_t (&q1)[32]) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            q0[j] = bf16x2_to_f16x2(q0[j]);
            if (D == 128) q1[j] = bf16x2_to_f16x2(q1[j]);
        }
        tmem_st32(tlane + kColQ, q0);
        if constexpr (D == 128) tmem_st32(tlane + kColQ + 32, q1);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(q_full);
    };

    uint32_t gbase = 0;  // sequence number (in this CTA) of the piece's first stage
    bool ok = true;
    int piece = 0;
    // QK issuer: a query-tile TMA not yet seen to land (the first was issued
    // before the consumers started).
    bool q_pending = a.q_tma && w.left > 0;
    uint32_t q_pending_par = 0;
    while (w.left > 0) {
        const int j0 = w.j, j1 = piece_end(w), n = j1 - j0;
        const int nsb = (n + SB - 1) / SB;
        const int ctx = w.ctx, s = w.s, h = w.h;
        int lim = -1, lo = INT_MIN, i_row = 0, hq_row = 0;
        bool row_ok = false;
        if (softmax) {
            row_ok = unit_row(a, w.t, h, trow, i_row, hq_row);
            lim = row_ok ? ctx - a.q_len + i_row : -1;
            if (a.window > 0) lo = lim - a.window + 1;
        }
        if constexpr (kQT) {
            // The first piece's query rows; each later piece's are stored by
            // the piece before it, ahead of its output, from the L2, where
            // they are fetched now.
            if (softmax) {
                if (piece == 0) {
                    uint32_t q0[32], q1[32];
                    q_rows_load(w, q0, q1);
                    q_rows_store(q0, q1);
                }
                Walk wn = w;
                wn.left -= j1 - w.j;
                if (wn.left > 0) {
                    walk_next_unit<BS>(a, wn);
                    if (const uint4* src = q_row_src(wn)) prefetch_l2_bulk(src, D * 2);
                }
            }
        } else if (softmax && !a.q_tma) {
            // This unit's query rows into the swizzled Q tile (the previous
            // unit's score products finished: each of them was waited for).
            const bool valid = row_ok;
            const uint4* qrow = reinterpret_cast<const uint4*>(
                a.q + (((size_t)s * a.q_len + i_row) * a.n_q + hq_row) * D);
            uint4 qv[D / 8];
#pragma unroll
            for (int c = 0; c < D / 8; ++c) qv[c] = valid ? __ldg(qrow + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
                *reinterpret_cast<uint4*>(qtile + (c >> 3) * kQHalf + trow * 128 +
                                          (((c & 7) ^ (trow & 7)) << 4)) = qv[c];
            fence_proxy_async_smem();
        }
        if (!kQT && !a.q_tma) {
            tc_fence_before();
            named_barrier_sync(2, kParty);  // Q tile ready; the previous unit's O has been read
            tc_fence_after();
        }
        // (With TMA query tiles, or query rows in tensor memory, the roles need
        // no barrier per piece: the issuer waits for the rows, and the first PV
        // product of a piece, which overwrites O, waits for P of its first
        // super-block, which the softmax threads write only after reading the
        // previous O.)

        if (warp == kQKWarp) {
            // ===================== QK issuer =====================
            if (lane == 0 && ok && (kQT || a.q_tma)) {
                // This piece's query rows: stored into tensor memory by the
                // softmax threads, or the tile landed in shared memory.
                if (*s_abort || !mbar_wait_bounded(q_full, piece & 1))
                    issuer_fail(ok);
                else
                    q_pending = false;
                tc_fence_after();
            }
            if (lane == 0 && ok) {
                // A score slot is reused by the stage T2 later (paired: the same
                // sub-tile's next stage; else the stage after next).
                constexpr uint32_t kReuse = T2 == 2 ? 1u : 2u;
                for (int q = 0; q < nsb && ok; ++q) {
                    const uint32_t g = gbase + q, st = g % kStages;
                    if (*s_abort ||
                        !(KV8 ? mbar_wait_bounded(&cvt_full[g % kCopies], (g / kCopies) & 1u)
                              : mbar_wait_bounded(&full_bar[st], (g / kStages) & 1u))) {
                        issuer_fail(ok);
                        break;
                    }
                    // Rows past the stage's blocks (a partial last super-block)
                    // hold stale keys; the softmax masks their columns.
                    const uint32_t kb = KV8 ? smem_addr(cvt + (g % kCopies) * kCopy)
                                            : smem_addr(stages + st * C::kStageBytes);
                    constexpr uint32_t kKRegion = KV8 ? C::kCvtRegion : C::kRegion;
#pragma unroll
                    for (int u = 0; u < T2; ++u) {
                        const uint32_t slot = sslot(g, u);
                        if (g >= kReuse && (*s_abort || !mbar_wait_bounded(&s_free[slot],
                                                                          spar(g - kReuse)))) {
                            issuer_fail(ok);
                            break;
                        }
                        tc_fence_after();
                        const uint32_t scol = tbase + kColS + slot * kKeys;
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk) {
                            const uint64_t bd =
                                g4 ? umma_smem_desc(kb + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048)
                                   : umma_smem_desc(kb + (kk >> 2) * kKRegion + (kk & 3) * 32, 16,
                                                    1024);
                            if constexpr (kQT) {
                                // 16 query columns = 8 tensor-memory columns per k step
                                umma_ts(scol, tbase + kColQ + kk * 8, bd, idesc_qk, kk > 0 ? 1u : 0u);
                            } else {
                                const uint64_t ad = umma_smem_desc(
                                    q_saddr + (kk >> 2) * kQHalf + u * 128 * 128 + (kk & 3) * 32, 16,
                                    1024);
                                umma_ss(scol, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                            }
                        }
                        umma_commit(&s_full[slot]);
                    }
                }
            }
            if (lane == 0 && ok && !kQT && a.q_tma) {
                // The next piece's query tile, once this piece's score
                // products have read this one.
                Walk wn = w;
                wn.left -= j1 - w.j;
                if (wn.left > 0) walk_next_unit<BS>(a, wn);
                if (wn.left > 0) {
                    umma_commit(q_empty);
                    if (!mbar_wait_bounded(q_empty, piece & 1)) {
                        issuer_fail(ok);
                    } else {
                        issue_q_tile<D, C::kQRows>(a, tmap_q, qtile, q_full, wn.s, wn.h, wn.t);
                        q_pending = true;
                        q_pending_par = (piece + 1) & 1;
                    }
                }
            }
            __syncwarp();
        } else if (warp == kPVWarp) {
            // ===================== PV issuer =====================
            if (lane == 0 && ok) {
                for (int q = 0; q < nsb && ok; ++q) {
                    const uint32_t g = gbase + q, st = g % kStages;
                    // Only the keys of the stage's blocks enter the product.
                    const int nk16 = min(SB, n - q * SB) * (BS / 16);
                    const uint32_t vb =
                        KV8 ? smem_addr(cvt + (g % kCopies) * kCopy) + kHalves * C::kCvtRegion
                            : smem_addr(stages + st * C::kStageBytes) + C::kBoxes * C::kRegion;
                    // The V rows of 16 keys, the distance to their second
                    // 64-column half and between their 8-row groups: halves of
                    // all the stage's blocks apart (2-D copies), or the grouped
                    // 4-D layout's 1024 and 2048 bytes.
                    const uint32_t vlbo = KV8 ? C::kCvtRegion : (g4 ? 1024u : C::kRegion);
                    const uint32_t vsbo = g4 ? 2048u : 1024u;
                    const uint32_t pcol = (g & 1u) * (kKeys / 2);
#pragma unroll
                    for (int u = 0; u < T2; ++u) {
                        const uint32_t pb = 2u * u + (g & 1u);  // P buffer of sub-tile u
                        if (*s_abort || !mbar_wait_bounded(&p_full[pb], (g >> 1) & 1u)) {
                            issuer_fail(ok);
                            break;
                        }
                        tc_fence_after();
                        // The softmax saw S of this stage, so its score product
                        // (with the other sub-tile's, the only readers of the
                        // stage's K) has completed.
                        const uint32_t ocol = tbase + kColO + u * 128;
                        const uint32_t pc = tbase + kColP + u * kKeys + pcol;
                        for (int kk = 0; kk < nk16; ++kk) {
                            const uint32_t vrow = g4 ? kk * 4096 : kk * 16 * 128;
                            const uint64_t bd = umma_smem_desc(vb + vrow, vlbo, vsbo);
                            umma_ts(ocol, pc + kk * 8, bd, idesc_pv, (q > 0 || kk > 0) ? 1u : 0u);
                            if (OUT_F32)
                                umma_ts(ocol, tbase + kColPL + pcol + kk * 8, bd, idesc_pv, 1u);
                        }
                        umma_commit(&pv_done[pb]);  // its P buffer is free; O is current
                    }
                    if (!ok) break;
                    if (KV8)
                        umma_commit(&cvt_free[g % kCopies]);  // the f16 copy is consumed
                    else
                        umma_commit(&empty_bar[st]);  // K and V of this stage are consumed
                }
            }
            __syncwarp();
        } else if (!softmax) {
            // ===================== f16 copies (8-bit cache; five warps) ============
            if constexpr (KV8) {
                // A stage's 2 x 64 rows (K rows, then V rows) are 2 * kRounds rounds
                // of 32 (row, 16-byte chunk) items; round k goes to converter k % 5
                // (warps 6, 7, 9, 10, 11).  Each converter arrives on its own when its
                // rounds are done (the copy-ready and stage-free barriers count 5).
                const int ci = warp < kConsumerWarps ? warp - 6 : warp - 7;
                constexpr int kChunks = D / 16;             // 16-byte e4m3 chunks per row
                constexpr int kRounds = 64 * kChunks / 32;  // rounds of K (or of V)
                constexpr int kAll = 2 * kRounds;
                constexpr int kMine = (kAll + kTmemConverters - 1) / kTmemConverters;
                constexpr int kBatch = 4;  // rounds whose loads are issued together
                for (int q = 0; q < nsb; ++q) {
                    const uint32_t g = gbase + q, st = g % kStages;
                    bool good = !*s_abort && mbar_wait_bounded(&full_bar[st], (g / kStages) & 1u);
                    if (good && g >= kCopies)
                        good = mbar_wait_bounded(&cvt_free[g % kCopies],
                                                 ((g - kCopies) / kCopies) & 1u);
                    if (!__all_sync(0xffffffffu, good)) {
                        if (lane == 0) {
                            atomicOr(a.err, kErrTimeout);
                            *s_abort = 1;
                        }
                        break;
                    }
                    tc_fence_after();
                    const int nb = min(SB, n - q * SB);
                    const int tok0 = (j0 + q * SB) * BS;
                    if constexpr (BLK) {
                        // the blocks' scales (K: converter 0, V: converter 1), before the
                        // stage is given back
                        if (ci < 2 && lane < nb)
                            cvt_sc[((g % kCopies) * SB + lane) * 2 + ci] =
                                reinterpret_cast<const float*>(slots + (st * SB + lane) * 16)[ci];
                    }
                    const uint8_t* stage_src = stages + st * C::kStageBytes;
                    uint8_t* copy = cvt + (g % kCopies) * kCopy;
                    // Rows of blocks past the stage's last are read (they lie inside the
                    // stage) and replaced by zeros, as are keys past the context.
#pragma unroll
                    for (int j0r = 0; j0r < kMine; j0r += kBatch) {
                        uint4 v[kBatch];
                        bool res[kBatch];
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int k = ci + kTmemConverters * (j0r + u);
                            res[u] = false;
                            if (j0r + u < kMine && k < kAll) {
                                const int isv = k / kRounds, it = lane + 32 * (k % kRounds);
                                const int nrow = it / kChunks, cb = it % kChunks;
                                const int b = nrow / BS, r = nrow % BS;
                                res[u] = b < nb && tok0 + nrow < ctx;  // a resident key
                                v[u] = *reinterpret_cast<const uint4*>(
                                    stage_src + isv * C::kBoxBytes + b * 2 * C::kBoxBytes +
                                    swz8<D>(r, cb * 16));
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int k = ci + kTmemConverters * (j0r + u);
                            if (!(j0r + u < kMine && k < kAll)) continue;
                            const int isv = k / kRounds, it = lane + 32 * (k % kRounds);
                            const int nrow = it / kChunks, cb = it % kChunks;
                            uint4 o0, o1;
                            e4m3x4_to_f16x2x2(v[u].x, o0.x, o0.y);
                            e4m3x4_to_f16x2x2(v[u].y, o0.z, o0.w);
                            e4m3x4_to_f16x2x2(v[u].z, o1.x, o1.y);
                            e4m3x4_to_f16x2x2(v[u].w, o1.z, o1.w);
                            if (!res[u]) o0 = o1 = make_uint4(0u, 0u, 0u, 0u);
                            // f16 chunks 2cb, 2cb + 1 (d 16cb ..): region (2cb) / 8, chunk (2cb) % 8
                            uint8_t* row = copy + isv * kHalves * C::kCvtRegion +
                                           ((2 * cb) / 8) * C::kCvtRegion + nrow * 128;
                            const int c0 = (2 * cb) % 8;
                            *reinterpret_cast<uint4*>(row + ((c0 ^ (nrow & 7)) << 4)) = o0;
                            *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (nrow & 7)) << 4)) = o1;
                        }
                    }
                    fence_proxy_async_smem();  // the copy, for the tensor cores
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&cvt_full[g % kCopies]);
                        mbar_arrive(&empty_bar[st]);  // (every converter: the e4m3 stage is free)
                    }
                }
            }
        } else {
            // ===================== softmax (thread = row) =====================
            // Scores stay raw: the row's extreme is taken over raw scores and
            // the exponent of a key is S * sl2 - S_ext * sl2, so the extreme
            // key itself weighs 1 (to the rounding of S_ext * sl2, ~1e-7
            // relative, which cancels against the same weight in l).  Over a negative scale the largest
            // scaled score is the smallest raw one; a zero scale makes every
            // visible score 0 (S is replaced by 0 and scaled by 1).  m_used is
            // the scaled running max, mr_used the raw score it came from.
            float m_used = -INFINITY, mr_used = 0.f, l = 0.f;
            // BLK: scores arrive already multiplied by their block's factor (score
            // scale x K scale), so the row extreme is a plain maximum.
            const float sl2_in = BLK ? 1.f
                                 : KV8 ? a.scale_log2 * __ldg(a.k_scale + h) : a.scale_log2;
            const bool zero_scale = sl2_in == 0.f;
            const float sl2 = zero_scale ? 1.f : sl2_in;
            const bool neg = sl2 < 0.f;
            float vrun = 0.f, vinv = 0.f;  // BLK: largest V scale of the unit so far; headroom / it
            const float hidden = neg ? INFINITY : -INFINITY;  // a masked raw score
            const int lim_min = ctx - a.q_len + tile_first_token(a, w.t);
            const int lo_max =
                a.window > 0 ? ctx - a.q_len + tile_last_token(a, w.t) - a.window + 1 : INT_MIN;
            for (int q = 0; q < nsb; ++q) {
                const uint32_t sq = gbase + q;  // this super-block's stage
                const int nb = min(SB, n - q * SB);
                ok = consumer_wait(a, &s_full[sslot(sq, sub)], spar(sq), ok, s_abort);
                if (!ok) continue;
                tc_fence_after();
                float x[kKeys];
                {
                    uint32_t s0[32], s1[32];
                    tmem_ld32(tlane + kColS + sslot(sq, sub) * kKeys, s0);
                    tmem_ld32(tlane + kColS + sslot(sq, sub) * kKeys + 32, s1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        x[c] = __uint_as_float(s0[c]);
                        x[32 + c] = __uint_as_float(s1[c]);
                    }
                    tc_fence_before();
                    mbar_arrive(&s_free[sslot(sq, sub)]);  // the score slot may be refilled
                }
                // BLK: the blocks' scales (written by the converter warps, acquired through
                // their copy-ready barrier, whose phase for this super-block has completed)
                float rat[SB], vfac = 1.f;
                bool vgrow = false;
                if constexpr (BLK) {
                    ok = consumer_wait(a, &cvt_full[sq % kCopies], (sq / kCopies) & 1u, ok,
                                       s_abort);
                    if (!ok) continue;
                    float kf[SB], vs[SB], smax = 0.f;
#pragma unroll
                    for (int b = 0; b < SB; ++b) {
                        const float2 sc = b < nb ? *reinterpret_cast<const float2*>(
                                                       cvt_sc + ((sq % kCopies) * SB + b) * 2)
                                                 : make_float2(0.f, 0.f);
                        kf[b] = a.scale_log2 * sc.x;
                        vs[b] = sc.y;
                        smax = fmaxf(smax, sc.y);
                    }
#pragma unroll
                    for (int c = 0; c < kKeys; ++c) x[c] *= kf[c / BS];
                    if (smax > vrun) {
                        vgrow = true;
                        vfac = vrun / smax;
                        vrun = smax;
                        vinv = kPShiftTmem / smax;
                    }
#pragma unroll
                    for (int b = 0; b < SB; ++b) rat[b] = vs[b] * vinv;
                }
                if (zero_scale) {
#pragma unroll
                    for (int c = 0; c < kKeys; ++c) x[c] = 0.f;
                }
                const int tok0 = (j0 + q * SB) * BS;  // first key of the super-block
                const int nkeys = nb * BS;            // columns past it hold stale scores
                if (nkeys < kKeys || tok0 + kKeys - 1 > lim_min || tok0 < lo_max) {
#pragma unroll
                    for (int c = 0; c < kKeys; ++c)
                        if (c >= nkeys || tok0 + c > lim || tok0 + c < lo) x[c] = hidden;
                }
                // The row's extreme raw score: a tree of three-input max (min).
                float t[22];
                if (!neg) {
#pragma unroll
                    for (int i = 0; i < 21; ++i) t[i] = max3f(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
                    t[21] = x[63];
#pragma unroll
                    for (int i = 0; i < 7; ++i) t[i] = max3f(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
                    t[0] = max3f(max3f(t[0], t[1], t[2]), max3f(t[3], t[4], t[5]),
                                 max3f(t[6], t[21], t[21]));
                } else {
#pragma unroll
                    for (int i = 0; i < 21; ++i) t[i] = min3f(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
                    t[21] = x[63];
#pragma unroll
                    for (int i = 0; i < 7; ++i) t[i] = min3f(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
                    t[0] = min3f(min3f(t[0], t[1], t[2]), min3f(t[3], t[4], t[5]),
                                 min3f(t[6], t[21], t[21]));
                }
                const float mloc = t[0] == hidden ? -INFINITY : t[0] * sl2;
                // This P buffer was last read by the PV of super-block q - 2.
                if (q > 1) {
                    ok = consumer_wait(a, &pv_done[2 * sub + (sq & 1u)], ((sq - 2) >> 1) & 1u, ok,
                                       s_abort);
                    if (!ok) continue;
                    tc_fence_after();
                }
                const bool grow = mloc > m_used + 8.f;
                if (__any_sync(0xffffffffu, grow) || vgrow) {  // (vgrow is CTA-uniform)
                    // O may only be rescaled once the previous super-block's PV is done.
                    if (q > 0) {
                        ok = consumer_wait(a, &pv_done[2 * sub + ((sq - 1) & 1u)],
                                           ((sq - 1) >> 1) & 1u, ok, s_abort);
                        if (!ok) continue;
                        tc_fence_after();
                    }
                    // alpha rescales weights taken against the old raw extreme
                    // to the new one, in the same arithmetic as the weights.
                    const float alpha = m_used == -INFINITY ? 0.f
                                        : grow             ? fast_exp2((mr_used - t[0]) * sl2)
                                                           : 1.f;
                    if (grow) {
                        m_used = mloc;
                        mr_used = t[0];
                    }
                    l *= alpha;
                    if (q > 0) {
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t ov[32];
                            tmem_ld32(tlane + kColO + sub * 128 + c0, ov);
                            tmem_wait_ld();
                            const float oscale = alpha * vfac;
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                ov[c] = __float_as_uint(__uint_as_float(ov[c]) * oscale);
                            tmem_st32(tlane + kColO + sub * 128 + c0, ov);
                        }
                        tmem_wait_st();
                    }
                }
                // With m_used = -inf every score of the row is masked (hidden
                // scales to -inf): the offset mr_used = 0 gives p = 0 for all.
                // The exponent S * sl2 - mr_used * sl2 is one FMA per key (the
                // extreme key's weight is 1 within a few ulp of its exponent).
                const float msl = mr_used * sl2;
                uint32_t ph[kKeys / 2], pl[kKeys / 2];
                float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
                for (int c = 0; c < kKeys; c += 4) {
                    float p0 = fast_exp2(fmaf(x[c], sl2, -msl));
                    float p1 = fast_exp2(fmaf(x[c + 1], sl2, -msl));
                    float p2 = fast_exp2(fmaf(x[c + 2], sl2, -msl));
                    float p3 = fast_exp2(fmaf(x[c + 3], sl2, -msl));
                    rs0 += p0;
                    rs1 += p1;
                    rs2 += p2;
                    rs3 += p3;
                    if constexpr (BLK) {  // four keys of one block (BS is a multiple of 4)
                        const float r = rat[c / BS];
                        p0 *= r;
                        p1 *= r;
                        p2 *= r;
                        p3 *= r;
                    }
                    if constexpr (KV8) {
                        ph[c / 2] = pack_f16x2(p0, p1);
                        ph[c / 2 + 1] = pack_f16x2(p2, p3);
                        if (OUT_F32) {
                            pl[c / 2] = pack_f16x2(p0 - f16_lo_to_f32(ph[c / 2]),
                                                   p1 - f16_hi_to_f32(ph[c / 2]));
                            pl[c / 2 + 1] = pack_f16x2(p2 - f16_lo_to_f32(ph[c / 2 + 1]),
                                                       p3 - f16_hi_to_f32(ph[c / 2 + 1]));
                        }
                    } else {
                        ph[c / 2] = pack_bf16x2(p0, p1);
                        ph[c / 2 + 1] = pack_bf16x2(p2, p3);
                        if (OUT_F32) {
                            pl[c / 2] = pack_bf16x2(p0 - bf16_lo_to_f32(ph[c / 2]),
                                                    p1 - bf16_hi_to_f32(ph[c / 2]));
                            pl[c / 2 + 1] = pack_bf16x2(p2 - bf16_lo_to_f32(ph[c / 2 + 1]),
                                                        p3 - bf16_hi_to_f32(ph[c / 2 + 1]));
                        }
                    }
                }
                const float rs = (rs0 + rs1) + (rs2 + rs3);
                l += rs;
                tmem_st32(tlane + kColP + sub * kKeys + (sq & 1u) * (kKeys / 2), ph);
                if (OUT_F32) tmem_st32(tlane + kColPL + (sq & 1u) * (kKeys / 2), pl);
                tmem_wait_st();
                // V rows past the context may hold NaN; 0 * NaN would poison O.
                // Only a unit's last block reaches past the context, and it is
                // the last block of its super-block.
                const int tokl = tok0 + (nb - 1) * BS;
                // (Paired: sub-tile 0 alone; the PV issuer takes sub-tile 1
                // after sub-tile 0's P, so after these zeros.)
                if (!KV8 && sub == 0 && tokl + BS > ctx) {  // (the f16 copies come zeroed there)
                    uint8_t* vt = stages + (sq % kStages) * C::kStageBytes +
                                  C::kBoxes * C::kRegion +
                                  (nb - 1) * (g4 ? 2 * C::kBoxBytes : C::kBoxBytes);
                    const int valid = ctx - tokl;  // >= 1: the block holds a resident token
                    const int chunks = (BS - valid) * 8;  // 16-byte chunks per 64-column half
                    for (int qq = row; qq < chunks * (D / 64); qq += 128) {
                        const int half = qq / chunks, rq = qq % chunks;
                        const int r = valid + (rq >> 3);  // the row, and its chunk rq & 7
                        const int off = g4 ? (r >> 3) * 2048 + half * 1024 + (r & 7) * 128
                                           : half * C::kRegion + r * 128;
                        *reinterpret_cast<uint4*>(vt + off + (rq & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(&p_full[2 * sub + (sq & 1u)]);
            }

            if constexpr (kQT) {
                // The next piece's query rows, before this piece's output, so
                // that its score products overlap the output's stores.  They
                // may be overwritten now: this piece's last S was read above,
                // so every score product that read them has completed.
                Walk wn = w;
                wn.left -= j1 - w.j;
                if (wn.left > 0) {
                    walk_next_unit<BS>(a, wn);
                    uint32_t q0[32], q1[32];
                    q_rows_load(wn, q0, q1);
                    q_rows_store(q0, q1);
                }
            }

            // ---- epilogue: the last PV, then O out of TMEM row by row
            if (nsb > 0) {
                const uint32_t sl = gbase + nsb - 1;
                ok = consumer_wait(a, &pv_done[2 * sub + (sl & 1u)], (sl >> 1) & 1u, ok, s_abort);
            }
            tc_fence_after();
            const bool first_piece = j0 == w.jlo, last_piece = j1 == w.nb;
            const bool whole = first_piece && last_piece;
            if (ok) {
                const float vsc = BLK ? vrun * kPShiftTmemInv : KV8 ? __ldg(a.v_scale + h) : 1.f;
                const float scl = (whole ? (l > 0.f ? 1.f / l : 0.f) : 1.f) * vsc;
                const size_t rec = (size_t)cta * 2 + (piece == 0 ? 0 : 1);
                if (whole && !OUT_F32) {
                    // bf16 rows: each thread its own row, 16 bytes per store
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32(tlane + kColO + sub * 128 + c0, ov);
                        tmem_wait_ld();
                        if (row_ok) {
                            const size_t ob =
                                (((size_t)s * a.q_len + i_row) * a.n_q + hq_row) * D + c0;
                            uint4* op = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ob);
#pragma unroll
                            for (int c = 0; c < 32; c += 8)
                                op[c / 8] = make_uint4(
                                    pack_bf16x2(__uint_as_float(ov[c]) * scl, __uint_as_float(ov[c + 1]) * scl),
                                    pack_bf16x2(__uint_as_float(ov[c + 2]) * scl, __uint_as_float(ov[c + 3]) * scl),
                                    pack_bf16x2(__uint_as_float(ov[c + 4]) * scl, __uint_as_float(ov[c + 5]) * scl),
                                    pack_bf16x2(__uint_as_float(ov[c + 6]) * scl, __uint_as_float(ov[c + 7]) * scl));
                        }
                    }
                } else if constexpr (BLK) {
                    // Per-block scales: fp32 rows one per thread.  (This
                    // instantiation runs 384 threads at the 168-register cap;
                    // the 16x256b form below measured 1.6 us slower here.)
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32(tlane + kColO + sub * 128 + c0, ov);
                        tmem_wait_ld();
                        if (whole ? row_ok : trow < R) {
                            float* op =
                                whole ? static_cast<float*>(a.out) +
                                            (((size_t)s * a.q_len + i_row) * a.n_q + hq_row) * D + c0
                                      : a.rec_o + (rec * R + trow) * D + c0;
#pragma unroll
                            for (int c = 0; c < 32; c += 4)
                                *reinterpret_cast<float4*>(op + c) = make_float4(
                                    __uint_as_float(ov[c]) * scl, __uint_as_float(ov[c + 1]) * scl,
                                    __uint_as_float(ov[c + 2]) * scl, __uint_as_float(ov[c + 3]) * scl);
                        }
                    }
                } else {
                    // fp32 rows (a record keeps o unnormalised: scl is then the V
                    // scale, 1 for bf16; or an fp32 output row).  O is read in the
                    // 16x256b shape, so four lanes store 32 contiguous bytes of one
                    // row and a store instruction reaches 8 rows, not 32 (the
                    // per-row form took ~1.5 us per 64 KB record).
                    const int g8 = lane >> 2, q4 = lane & 3;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        const int rq = (warp & 3) * 32 + hh * 16;  // first row of the half
                        float* dst[2];
                        float sc[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            // tile row; lane r % 32 holds its scl
                            const int r = sub * 128 + rq + g8 + 8 * u;
                            sc[u] = __shfl_sync(0xffffffffu, scl, (r & 31));
                            dst[u] = nullptr;
                            if (whole) {
                                int ir = 0, hr = 0;
                                if (unit_row(a, w.t, h, r, ir, hr))
                                    dst[u] = static_cast<float*>(a.out) +
                                             (((size_t)s * a.q_len + ir) * a.n_q + hr) * D;
                            } else if (r < R) {
                                dst[u] = a.rec_o + (rec * R + r) * D;
                            }
                        }
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t ov[16];
                            tmem_ld_16x256b_x4(tbase + ((uint32_t)rq << 16) + kColO + sub * 128 + c0,
                                               ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int c = c0 + 8 * j + 2 * q4;
#pragma unroll
                                for (int u = 0; u < 2; ++u)
                                    if (dst[u])
                                        *reinterpret_cast<float2*>(dst[u] + c) =
                                            make_float2(__uint_as_float(ov[4 * j + 2 * u]) * sc[u],
                                                        __uint_as_float(ov[4 * j + 2 * u + 1]) * sc[u]);
                            }
                        }
                    }
                }
                if (!whole) {
                    if (trow < R)
                        *reinterpret_cast<float2*>(a.rec_ml + (rec * R + trow) * 2) = make_float2(m_used, l);
                    if (trow == 0) {
                        const int4 rinfo = make_int4(
                            s, h, kRecValid | (first_piece ? kRecFirst : 0) | (last_piece ? kRecLast : 0),
                            w.t);
                        if (piece == 0)
                            info0 = rinfo;
                        else
                            info1 = rinfo;
                    }
                }
            }
            tc_fence_before();
        }
        gbase += nsb;
        ++piece;
        w.left -= j1 - w.j;
        if (w.left > 0) walk_next_unit<BS>(a, w);
    }
    // Teardown: no tensor-core operation may still be running when TMEM is
    // freed, and no query-tile copy may still be landing.
    if ((warp == kQKWarp || warp == kPVWarp) && lane == 0) {
        uint64_t* bar = &tcb[warp == kQKWarp ? 12 : 13];
        umma_commit(bar);
        (void)mbar_wait_bounded(bar, 0u);
        if (warp == kQKWarp && q_pending) (void)mbar_wait_bounded(q_full, q_pending_par);
    }
    tc_fence_before();
    named_barrier_sync(2, kParty);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ===================== kernel =====================
template <int D, int BS, bool OUT_F32, int MODE, bool KV8, bool BLK>
__global__ void __launch_bounds__(threads_for(MODE, KV8), 1)
    paged_decode_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ CUtensorMap tmap_q, const AttnArgs a) {
    using C = AttnCfg<D, BS, MODE, KV8, BLK>;
    constexpr int kStages = C::kStages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stages = smem;
    float* scratch = reinterpret_cast<float*>(smem + kStages * C::kStageBytes);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStages * C::kStageBytes +
                                                     C::kScratchBytes);
    uint64_t* empty_bar = full_bar + kStages;
    // BLK: the scale slots of the ring, kBlocksPerStage x 16 bytes per stage
    uint8_t* slots = reinterpret_cast<uint8_t*>(empty_bar + kStages);

    constexpr int NT = threads_for(MODE, KV8);
    __shared__ long long s_red[2 * NT / 32];
    __shared__ long long s_pos[4];
    __shared__ Walk s_walk;
    __shared__ int s_abort;
    // TMEM modes: S ready/read (x2 each), P ready, PV done (x4 each), 2
    // teardowns, over an 8-bit cache f16 copy ready / free (x3 each), query
    // rows ready, query tile read
    __shared__ uint64_t s_tcb[22];
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Arrivals that release a stage: one per 16-row slice (wide), one warp
    // (narrow), one tensor-core commit (TMEM mode), the five converter warps
    // (TMEM mode over an 8-bit cache).
    const int releases =
        MODE == kModeWide ? a.warp_rows : (MODE == kModeTmem && KV8 ? kTmemConverters : 1);
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], releases);
        }
        if (C::kTmem) {
            // S ready (a commit), S read (128 rows), P ready (128 rows) and
            // PV done (a commit) per sub-tile and buffer, two issuer
            // teardowns (a commit each), f16
            // copy ready (the converter warps) / free (a commit), query rows
            // stored in tensor memory (128 rows; 8-bit cache) or the query
            // tile landed (the TMA; bf16), query tile read (a commit)
            const uint32_t cvt = KV8 ? (uint32_t)kTmemConverters : 1u;
            const uint32_t qin = KV8 ? 128u : 1u;
            const uint32_t counts[22] = {1,   1,   128, 128, 128, 128, 128, 128, 1,   1, 1,
                                         1,   1,   1,   cvt, cvt, cvt, 1,   1,   1,   qin, 1};
            static_assert(C::kCvtCopies == 3, "barrier counts: three f16 copies");
            for (int i = 0; i < 22; ++i) mbar_init(&s_tcb[i], counts[i]);
        }
        fence_barrier_init();
        s_abort = 0;
        for (int i = 0; i < 4; ++i) s_pos[i] = -1;
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
        // Small tables read piecemeal later, fetched into the L2 now with one
        // sequential prefetch per CTA (each CTA a 1/grid share): the block
        // tables, which the producers read right after the work partition, and
        // (per-block scales) the scale entries, one 16-byte read per block that
        // from HBM cost a random access each (8-bit GQA 116.0 -> 101.3 us without them).
        auto share = [&](const void* base, size_t bytes) {
            const size_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
            const size_t lo = per * blockIdx.x;
            if (lo < bytes) {
                const size_t n = bytes - lo < per ? bytes - lo : per;
                prefetch_l2_bulk(static_cast<const uint8_t*>(base) + lo, static_cast<uint32_t>(n));
            }
        };
        // (the tables are only 4-byte aligned: the prefetch covers the 16-byte-aligned
        // interior of their span and never reaches past it)
        const uintptr_t tb = reinterpret_cast<uintptr_t>(a.block_tables);
        const uintptr_t t0 = (tb + 15) & ~uintptr_t(15);
        const uintptr_t t1 = (tb + (size_t)a.num_seqs * a.max_blocks_per_seq * 4) & ~uintptr_t(15);
        if (t1 > t0) share(reinterpret_cast<const void*>(t0), t1 - t0);
        if (BLK) share(a.kv_scales, (size_t)a.num_blocks * a.n_kv * 16);
    }
    const Walk w0 = find_slice<BS, NT>(a, s_red, s_pos, &s_walk);  // also publishes the barrier init
    // This kernel is launched as a programmatic dependent of the previous
    // kernel on the stream: the work partition above (which reads only the
    // context lengths) may overlap it, e.g. the cache append that precedes
    // every decode step; nothing else is read or written before it completes.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Let the merge kernel (launched as a programmatic dependent) be scheduled
    // early; it waits for this whole grid before reading anything.
    if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Tensor-memory consumer with TMA query tiles (bf16 cache): the first
    // tile is issued before the producer's first stage, so it is not queued
    // behind the ring fill.
    if constexpr (C::kTmem && !KV8) {
        if (a.q_tma) {
            if (warp == (MODE == kModeTmem2 ? 9 : 4)) {  // the QK issuer
                if (lane == 0 && w0.left > 0)
                    issue_q_tile<D, C::kQRows>(a, &tmap_q, reinterpret_cast<uint8_t*>(scratch),
                                               &s_tcb[20], w0.s, w0.h, w0.t);
                __syncwarp();
                named_barrier_arrive(3, 64);
            } else if (warp == kConsumerWarps) {
                named_barrier_sync(3, 64);
            }
        }
    }
    if (warp == kConsumerWarps) {
        produce<D, BS, kStages, C::kStageBytes, C::kTileBytes, C::kBoxBytes, C::kBoxes,
                C::kBoxCols, C::kRegion, C::kBlocksPerStage, KV8, C::kTmem, BLK>(
            a, &tmap_k, &tmap_v, w0, stages, slots, full_bar, empty_bar, &s_abort);
        return;
    }

    // Sequences with nothing resident produce zero rows (and are checked).
    for (int s = blockIdx.x; s < a.num_seqs; s += gridDim.x) {
        const int raw = __ldg(a.context_lens + s);
        if (a.checked && tid == 0 &&
            (raw < 0 || raw > a.max_blocks_per_seq * BS || (raw > 0 && raw < a.q_len)))
            atomicOr(a.err, kErrBadContext);
        if (unit_blocks(a, s, BS) == 0) {
            const size_t n = (size_t)a.q_len * a.n_q * D;
            const size_t o0 = (size_t)s * n;
            for (size_t e = tid; e < n; e += kConsumerThreads) {
                if (OUT_F32)
                    static_cast<float*>(a.out)[o0 + e] = 0.f;
                else
                    static_cast<uint16_t*>(a.out)[o0 + e] = 0;
            }
        }
    }

    int4 info0 = make_int4(0, 0, 0, 0), info1 = make_int4(0, 0, 0, 0);
    if (w0.left <= 0) info0.z = info1.z = kRecEmpty;
    if constexpr (MODE == kModeNarrow)
        consume_narrow<D, BS, OUT_F32, KV8, BLK>(a, w0, stages, slots, scratch, full_bar,
                                                 empty_bar, &s_abort, info0, info1);
    else if constexpr (MODE == kModeWide)
        consume_wide<D, BS, OUT_F32, KV8, BLK>(a, w0, stages, slots, scratch, full_bar, empty_bar,
                                               &s_abort, info0, info1);
    else
        consume_tmem<D, BS, OUT_F32, KV8, BLK, MODE == kModeTmem2 ? 2 : 1>(
            a, w0, stages, slots, reinterpret_cast<uint8_t*>(scratch), &tmap_q, full_bar,
            empty_bar, s_tcb, &s_tmem, &s_abort, info0, info1);
    if (tid == 0) {
        a.rec_info[(size_t)blockIdx.x * 2 + 0] = info0;
        a.rec_info[(size_t)blockIdx.x * 2 + 1] = info1;
    }
}

// ---------------------------------------------------------------------------
template <int D, int BS, bool F32, int MODE, bool KV8, bool BLK>
static cudaError_t launch_one(const AttnArgs& a, const AttnMaps& m, int grid,
                              cudaStream_t stream) {
    auto kern = paged_decode_attn_kernel<D, BS, F32, MODE, KV8, BLK>;
    const int smem = AttnCfg<D, BS, MODE, KV8, BLK>::kSmemBytes;
    // The shared-memory opt-in is set once per device for each instantiation.
    static std::atomic<unsigned long long> opted_in{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(opted_in.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        opted_in.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads_for(MODE, KV8), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.early_start ? 1 : 0;  // without it, griddepcontrol.wait returns at once
    e = cudaLaunchKernelEx(&cfg, kern, m.k, m.v, m.q, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Consumer by rows per KV head: narrow (<= 8), wide, TMEM (> 64).
template <int D, int BS, bool KV8, bool BLK>
static cudaError_t launch_shape(const AttnArgs& a, const AttnMaps& m, bool out_f32, int grid,
                                cudaStream_t stream) {
    if (a.rows <= kNarrowRows)
        return out_f32 ? launch_one<D, BS, true, kModeNarrow, KV8, BLK>(a, m, grid, stream)
                       : launch_one<D, BS, false, kModeNarrow, KV8, BLK>(a, m, grid, stream);
    if (a.rows > 128) {  // the paired form: bf16 cache and output only (chosen by the host)
        if constexpr (!KV8 && !BLK) {
            if (!out_f32) return launch_one<D, BS, false, kModeTmem2, false, false>(a, m, grid, stream);
        }
        return cudaErrorInvalidValue;
    }
    if (a.rows > kTmemMinRows)
        return out_f32 ? launch_one<D, BS, true, kModeTmem, KV8, BLK>(a, m, grid, stream)
                       : launch_one<D, BS, false, kModeTmem, KV8, BLK>(a, m, grid, stream);
    return out_f32 ? launch_one<D, BS, true, kModeWide, KV8, BLK>(a, m, grid, stream)
                   : launch_one<D, BS, false, kModeWide, KV8, BLK>(a, m, grid, stream);
}

template <bool KV8, bool BLK>
static cudaError_t launch_decode_attn_kv(const AttnArgs& a, const AttnMaps& m, int head_dim,
                                         int block_size, bool out_f32, int grid,
                                         cudaStream_t stream) {
    if (head_dim == 128 && block_size == 16)
        return launch_shape<128, 16, KV8, BLK>(a, m, out_f32, grid, stream);
    if (head_dim == 128 && block_size == 32)
        return launch_shape<128, 32, KV8, BLK>(a, m, out_f32, grid, stream);
    if (head_dim == 64 && block_size == 16)
        return launch_shape<64, 16, KV8, BLK>(a, m, out_f32, grid, stream);
    if (head_dim == 64 && block_size == 32)
        return launch_shape<64, 32, KV8, BLK>(a, m, out_f32, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
