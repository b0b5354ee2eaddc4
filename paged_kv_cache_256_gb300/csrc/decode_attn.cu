// decode_attn.cu -- paged decode attention for sm_103a.
//
// What it computes: for every sequence b, new query token i and query head h,
//   out = softmax_t(scale * q . K_t) V_t over the logical positions t the
//   causal mask allows (t <= ctx - q_len + i), with K_t, V_t found through
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
//   * Warp 8 is the producer: it reads block ids, and one lane issues 2-D TMA
//     tile loads (128-byte swizzle) of the K and V tiles of each
//     (block, KV head) into a ring of shared-memory stages, each guarded by a
//     full/empty mbarrier pair.  Its walk never stops at unit boundaries, so
//     HBM stays busy while consumers finish a unit.
//   * Warps 0..7 consume.  Warp w owns 16-row tile (w % WM) of the unit and
//     every WN-th block (WN = 8 / WM).  Scores S = Q K^T and the update
//     O += P V run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//     accumulate); the online softmax (running max m and sum l, fp32, base 2)
//     is the FlashAttention recurrence ("Efficient inference", FlashAttention:
//     exact attention without the matrix).  At the end of a unit the WN
//     column partials are combined in shared memory by the same exact rule.
//   * fp32 output keeps each probability as a bf16 pair (hi + lo) so the PV
//     product keeps ~16 bits of it; bf16 output uses one bf16.
//
// Bounded waits: every mbarrier wait gives up after a second, records
// kErrTimeout in the workspace and the kernel winds down without hanging.
#include <cfloat>
#include <climits>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kMergeSlots = 4;                   // (WN / 2) * WM is at most 4
constexpr int kIssueLanes = 4;                   // producer lanes issuing loads side by side

template <int D, int BS>
struct AttnCfg {
    static constexpr int kTileBytes = BS * D * 2;  // one K (or V) tile of one (block, head)
    static constexpr int kStageBytes = 2 * kTileBytes;
    // The ring depth is a multiple of the consumer-warp count: block g and
    // block g - kStages then belong to the same warp, so when a warp waits for
    // round r of a stage it has itself already seen round r - 1 complete.
    // (mbarrier parity waits cannot tell round r from round r - 2; with
    // another warp owning round r - 1 a still-in-flight load would read as
    // complete.)
    static constexpr int kStagesRaw = (160 * 1024) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 32 ? 32 : (kStagesRaw / 8) * 8;
    static constexpr int kBoxBytes = BS * 128;  // one 64-column swizzled box
    static constexpr int kLaneFloats = D / 2 + 4;  // o (D/8 n-tiles x 4) + m[2] + l[2]
    static constexpr int kScratchBytes = kMergeSlots * 32 * kLaneFloats * 4;
    static constexpr int kBarrierBytes = 2 * kStages * 8;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kScratchBytes + kBarrierBytes;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kStages % 8 == 0 && kStages >= 8, "ring depth must be a multiple of 8 warps");
};

// Byte offset of the 16-byte chunk holding (row, col..col+7) inside a tile
// stored as D/64 boxes of [BS rows][128 bytes] with the TMA 128-byte swizzle
// (16-byte chunk index XOR row % 8 within each 1024-byte atom).
template <int BS>
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return static_cast<uint32_t>((col >> 6) * (BS * 128) + row * 128 +
                                 ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

__device__ __forceinline__ int unit_blocks(const AttnArgs& a, int s, int bs) {
    int ctx = __ldg(a.context_lens + s);
    const int cap = a.max_blocks_per_seq * bs;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    return (ctx + bs - 1) / bs;
}

__device__ __forceinline__ int unit_ctx(const AttnArgs& a, int s, int bs) {
    int ctx = __ldg(a.context_lens + s);
    const int cap = a.max_blocks_per_seq * bs;
    return ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
}

// Position in the flat work list: sequence s, KV head h, block j of that unit,
// `left` items still to process in this CTA's slice.
struct Walk {
    int s, h, j, nb, ctx;
    long long left;
};

template <int BS>
__device__ __forceinline__ void walk_next_unit(const AttnArgs& a, Walk& w) {
    w.j = 0;
    if (++w.h == a.n_kv) {
        w.h = 0;
        do {
            ++w.s;
            w.nb = w.s < a.num_seqs ? unit_blocks(a, w.s, BS) : 1;
        } while (w.nb == 0);
        w.ctx = unit_ctx(a, w.s, BS);
    }
}

// Block-wide inclusive scan of one 64-bit value per thread (all kThreads).
__device__ __forceinline__ long long block_inclusive_scan(long long v, long long* s_red,
                                                          long long& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        long long n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) s_red[warp] = v;
    __syncthreads();
    long long before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const long long t = s_red[w];
        if (w < warp) before += t;
        total += t;
    }
    __syncthreads();
    return v + before;
}

template <int D, int BS, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const AttnArgs a) {
    using C = AttnCfg<D, BS>;
    constexpr int kStages = C::kStages;
    constexpr int NT = D / 8;    // 8-wide output column tiles
    constexpr int KT = D / 16;   // 16-deep k steps over head_dim
    constexpr int ST = BS / 8;   // 8-token score tiles per block
    constexpr int PT = BS / 16;  // 16-token k steps of the PV product

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stages = smem;
    float* scratch = reinterpret_cast<float*>(smem + kStages * C::kStageBytes);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStages * C::kStageBytes +
                                                     C::kScratchBytes);
    uint64_t* empty_bar = full_bar + kStages;

    __shared__ long long s_red[kThreads / 32];
    __shared__ long long s_start[2];
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int WM = a.warp_rows;
    const int WN = kConsumerWarps / WM;
    const int cta = blockIdx.x, grid = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], WM);
        }
        fence_barrier_init();
        s_abort = 0;
        s_start[0] = -1;
        s_start[1] = 0;
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }

    // ---- this CTA's slice of the flat (unit, block) work list --------------
    long long mine = 0;
    for (int s = tid; s < a.num_seqs; s += kThreads) mine += unit_blocks(a, s, BS);
    long long total_blocks;
    (void)block_inclusive_scan(mine, s_red, total_blocks);  // also publishes barrier init
    const long long W = total_blocks * a.n_kv;
    const long long start = (W * cta) / grid;
    const long long end = (W * (cta + 1)) / grid;

    if (start < end) {
        long long base = 0;
        for (int s0 = 0; s0 < a.num_seqs; s0 += kThreads) {
            const int s = s0 + tid;
            const long long v = s < a.num_seqs ? (long long)unit_blocks(a, s, BS) * a.n_kv : 0;
            long long chunk;
            const long long incl = block_inclusive_scan(v, s_red, chunk);
            const long long excl = incl - v;
            if (v > 0 && base + excl <= start && start < base + incl) {
                s_start[0] = s;
                s_start[1] = start - (base + excl);
            }
            base += chunk;
            __syncthreads();
            if (s_start[0] >= 0) break;
        }
    }
    __syncthreads();

    Walk w0;
    w0.left = end - start;
    if (w0.left > 0) {
        w0.s = static_cast<int>(s_start[0]);
        w0.nb = unit_blocks(a, w0.s, BS);
        w0.ctx = unit_ctx(a, w0.s, BS);
        w0.h = static_cast<int>(s_start[1] / w0.nb);
        w0.j = static_cast<int>(s_start[1] % w0.nb);
    } else {
        w0.s = w0.h = w0.j = w0.nb = w0.ctx = 0;
    }

    if (warp == kConsumerWarps) {
        // ===================== producer warp =====================
        const uint64_t policy = l2_policy_evict_first();
        uint32_t gidx = 0, issued = 0;  // issued: fills actually started (a prefix of gidx)
        bool ok = true;
        Walk w = w0;
        while (w.left > 0 && ok) {
            const int j1 = (long long)w.nb < (long long)w.j + w.left ? w.nb
                                                                     : static_cast<int>(w.j + w.left);
            const int32_t* bt = a.block_tables + (size_t)w.s * a.max_blocks_per_seq;
            int my = w.j + lane < j1 ? __ldg(bt + w.j + lane) : 0;
            for (int jb = w.j; jb < j1 && ok; jb += 32) {
                const int n = min(32, j1 - jb);
                // The next 32 block ids load while this batch is issued.
                const int nxt = jb + 32 + lane < j1 ? __ldg(bt + jb + 32 + lane) : 0;
                if (lane < n && (my < 0 || my >= a.num_blocks)) {
                    if (a.checked) atomicOr(a.err, kErrBadBlock);
                    my = -1;  // read as an out-of-bounds (zero-filled) tile
                }
                if (*((volatile int*)&s_abort)) ok = false;  // a consumer gave up
                // Lanes 0..kIssueLanes-1 issue the next blocks side by side:
                // one serial wait/issue chain per block would cap the stream.
                for (int k0 = 0; k0 < n && ok; k0 += kIssueLanes) {
                    const int kk = k0 + lane;
                    const int blk = __shfl_sync(0xffffffffu, my, kk & 31);
                    const bool act = lane < kIssueLanes && kk < n;
                    const uint32_t gl = gidx + lane;
                    const uint32_t stage = gl % kStages;
                    bool good = true;
                    if (act) good = mbar_wait_bounded(&empty_bar[stage], ((gl / kStages) & 1u) ^ 1u);
                    const unsigned act_mask = __ballot_sync(0xffffffffu, act);
                    const unsigned good_mask = __ballot_sync(0xffffffffu, act && good);
                    const unsigned fail = act_mask & ~good_mask;
                    // Only the lanes below the first failed wait issue, so the
                    // issued fills stay a prefix of the block sequence.
                    const unsigned issue_mask =
                        fail ? (good_mask & ((1u << (__ffs(fail) - 1)) - 1u)) : good_mask;
                    if ((issue_mask >> lane) & 1u) {
                        mbar_arrive_expect_tx(&full_bar[stage], 2 * C::kTileBytes);
                        const long long y64 = ((long long)blk * a.n_kv + w.h) * BS;
                        const int y = (blk < 0 || y64 >= a.tile_rows_total)
                                          ? a.tile_rows_total
                                          : static_cast<int>(y64);
                        uint8_t* kdst = stages + stage * C::kStageBytes;
                        uint8_t* vdst = kdst + C::kTileBytes;
#pragma unroll
                        for (int half = 0; half < D / 64; ++half) {
                            tma_load_2d(kdst + half * C::kBoxBytes, &tmap_k, half * 64, y,
                                        &full_bar[stage], policy);
                            tma_load_2d(vdst + half * C::kBoxBytes, &tmap_v, half * 64, y,
                                        &full_bar[stage], policy);
                        }
                    }
                    issued = gidx + __popc(issue_mask);
                    if (fail) {
                        ok = false;
                        if (lane == 0) {
                            atomicOr(a.err, kErrTimeout);
                            *((volatile int*)&s_abort) = 1;
                        }
                    }
                    gidx += min(kIssueLanes, n - k0);
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
        return;
    }

    // ===================== consumer warps =====================
    // Sequences with nothing resident produce zero rows (and are checked).
    for (int s = cta; s < a.num_seqs; s += grid) {
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

    const int mt = warp % WM;  // which 16-row tile of the unit's rows
    const int col = warp / WM; // which residue class of blocks
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix index, row within matrix
    const int G = a.group;

    int4 info0 = make_int4(0, 0, 0, 0), info1 = make_int4(0, 0, 0, 0);
    if (w0.left <= 0) info0.z = info1.z = kRecEmpty;

    uint32_t gidx = 0;
    bool ok = true;
    int piece = 0;
    Walk w = w0;
    while (w.left > 0) {
        const int j0 = w.j;
        const int j1 = (long long)w.nb < (long long)w.j + w.left ? w.nb
                                                                 : static_cast<int>(w.j + w.left);
        const int ctx = w.ctx;
        const int s = w.s, h = w.h;

        // Query fragments of this unit's two rows per thread (rows >= a.rows are zero).
        uint32_t qf[KT][4];
        int lim[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = mt * 16 + g + hh * 8;
            const bool valid = r < a.rows;
            const int i = valid ? r / G : 0;
            const int hq = h * G + (valid ? r % G : 0);
            lim[hh] = valid ? ctx - a.q_len + i : -1;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                a.q + (((size_t)s * a.q_len + i) * a.n_q + hq) * D);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                qf[kk][hh] = valid ? __ldg(qrow + kk * 8 + t) : 0u;
                qf[kk][2 + hh] = valid ? __ldg(qrow + kk * 8 + 4 + t) : 0u;
            }
        }
        const int lim_min = ctx - a.q_len;  // smallest causal limit of a real row

        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

        for (int j = j0; j < j1; ++j, ++gidx) {
            if ((int)(gidx % (uint32_t)WN) != col) continue;
            const uint32_t stage = gidx % kStages;
            if (ok && *((volatile int*)&s_abort)) ok = false;  // another warp gave up
            if (ok && !mbar_wait_bounded(&full_bar[stage], (gidx / kStages) & 1u)) {
                ok = false;
                atomicOr(a.err, kErrTimeout);
                *((volatile int*)&s_abort) = 1;
            }
            if (ok) {
                const uint32_t kbase = smem_addr(stages + stage * C::kStageBytes);
                const uint32_t vbase = kbase + C::kTileBytes;

                // ---- S = Q K^T over this block's BS tokens
                float sc[ST][4];
#pragma unroll
                for (int n = 0; n < ST; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
#pragma unroll
                    for (int tp = 0; tp < PT; ++tp) {
                        uint32_t b[4];
                        const int tok = tp * 16 + (mi >> 1) * 8 + rr;
                        const int dc = kk * 16 + (mi & 1) * 8;
                        ldmatrix_x4(b, kbase + swz<BS>(tok, dc));
                        mma_bf16_16816(sc[2 * tp], qf[kk], b[0], b[1]);
                        mma_bf16_16816(sc[2 * tp + 1], qf[kk], b[2], b[3]);
                    }
                }

                // ---- scale, causal / tail mask, online softmax (base 2)
                const int tok0 = j * BS;
                const bool need_mask = tok0 + BS - 1 > lim_min;
                float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int n = 0; n < ST; ++n) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float x = sc[n][e] * a.scale_log2;
                        if (need_mask) {
                            const int tk = tok0 + n * 8 + 2 * t + (e & 1);
                            if (tk > lim[e >> 1]) x = -INFINITY;
                        }
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
                for (int n = 0; n < ST; ++n) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p = fast_exp2(sc[n][e] - mbase[e >> 1]);
                        sc[n][e] = p;
                        rsum[e >> 1] += p;
                    }
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) l[hh] = l[hh] * alpha[hh] + rsum[hh];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    o[n][0] *= alpha[0];
                    o[n][1] *= alpha[0];
                    o[n][2] *= alpha[1];
                    o[n][3] *= alpha[1];
                }

                // ---- P as bf16 A fragments (fp32 output: hi + lo pair)
                uint32_t pa[PT][4];
                uint32_t pl[PT][4];
#pragma unroll
                for (int tp = 0; tp < PT; ++tp) {
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int n = 2 * tp + (q2 >> 1);
                        const int e = (q2 & 1) * 2;
                        const float p0 = sc[n][e], p1 = sc[n][e + 1];
                        pa[tp][q2] = pack_bf16x2(p0, p1);
                        if (OUT_F32)
                            pl[tp][q2] = pack_bf16x2(p0 - bf16_lo_to_f32(pa[tp][q2]),
                                                     p1 - bf16_hi_to_f32(pa[tp][q2]));
                    }
                }

                // ---- O += P V (V rows past the context are zeroed: they may hold NaN)
                const bool need_vmask = tok0 + BS > ctx;
#pragma unroll
                for (int tp = 0; tp < PT; ++tp) {
                    uint32_t vm0 = 0xFFFFFFFFu, vm8 = 0xFFFFFFFFu;
                    if (need_vmask) {
                        const int ta = tok0 + tp * 16 + 2 * t;
                        vm0 = (ta < ctx ? 0x0000FFFFu : 0u) | (ta + 1 < ctx ? 0xFFFF0000u : 0u);
                        vm8 = (ta + 8 < ctx ? 0x0000FFFFu : 0u) | (ta + 9 < ctx ? 0xFFFF0000u : 0u);
                    }
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        uint32_t b[4];
                        const int tok = tp * 16 + (mi & 1) * 8 + rr;
                        const int dc = dp * 16 + (mi >> 1) * 8;
                        ldmatrix_x4_trans(b, vbase + swz<BS>(tok, dc));
                        b[0] &= vm0;
                        b[1] &= vm8;
                        b[2] &= vm0;
                        b[3] &= vm8;
                        mma_bf16_16816(o[2 * dp], pa[tp], b[0], b[1]);
                        mma_bf16_16816(o[2 * dp + 1], pa[tp], b[2], b[3]);
                        if (OUT_F32) {
                            mma_bf16_16816(o[2 * dp], pl[tp], b[0], b[1]);
                            mma_bf16_16816(o[2 * dp + 1], pl[tp], b[2], b[3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
        }

        // ---- row sums across the quad, then combine the WN column partials
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
                for (int hh = 0; hh < 2; ++hh) {
                    const float m2 = sl[(NT * 4 + hh) * 32 + lane];
                    const float l2 = sl[(NT * 4 + 2 + hh) * 32 + lane];
                    const float mn = fmaxf(m[hh], m2);
                    const float mb = mn == -INFINITY ? 0.f : mn;
                    a1[hh] = fast_exp2(m[hh] - mb);
                    a2[hh] = fast_exp2(m2 - mb);
                    l[hh] = a1[hh] * l[hh] + a2[hh] * l2;
                    m[hh] = mn;
                }
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[n][e] = a1[e >> 1] * o[n][e] + a2[e >> 1] * sl[(n * 4 + e) * 32 + lane];
            }
            named_barrier_sync(1, kConsumerThreads);
        }

        // ---- emit: a whole unit goes straight to `out`; a piece becomes a record
        const bool first = j0 == 0, last = j1 == w.nb;
        if (col == 0) {
            if (first && last) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = mt * 16 + g + hh * 8;
                    if (r >= a.rows) continue;
                    const int i = r / G, hq = h * G + r % G;
                    const float inv = l[hh] > 0.f ? 1.f / l[hh] : 0.f;
                    const size_t ob = (((size_t)s * a.q_len + i) * a.n_q + hq) * D;
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const float v0 = o[n][2 * hh] * inv, v1 = o[n][2 * hh + 1] * inv;
                        if (OUT_F32)
                            *reinterpret_cast<float2*>(static_cast<float*>(a.out) + ob + n * 8 +
                                                       2 * t) = make_float2(v0, v1);
                        else
                            *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + ob +
                                                         n * 8 + 2 * t) = pack_bf16x2(v0, v1);
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
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        *reinterpret_cast<float2*>(ro + n * 8 + 2 * t) =
                            make_float2(o[n][2 * hh], o[n][2 * hh + 1]);
                    if (t == 0)
                        *reinterpret_cast<float2*>(a.rec_ml + (rec * a.rows + r) * 2) =
                            make_float2(m[hh], l[hh]);
                }
                const int4 rinfo = make_int4(s, h, kRecValid | (first ? kRecFirst : 0) |
                                                       (last ? kRecLast : 0), 0);
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
    if (tid == 0) {
        a.rec_info[(size_t)cta * 2 + 0] = info0;
        a.rec_info[(size_t)cta * 2 + 1] = info1;
    }
}

// ---------------------------------------------------------------------------
int decode_attn_smem_bytes(int head_dim, int block_size) {
    if (head_dim == 128 && block_size == 16) return AttnCfg<128, 16>::kSmemBytes;
    if (head_dim == 128 && block_size == 32) return AttnCfg<128, 32>::kSmemBytes;
    if (head_dim == 64 && block_size == 16) return AttnCfg<64, 16>::kSmemBytes;
    if (head_dim == 64 && block_size == 32) return AttnCfg<64, 32>::kSmemBytes;
    return -1;
}

template <int D, int BS, bool F32>
static cudaError_t launch_one(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t stream) {
    auto kern = paged_decode_attn_kernel<D, BS, F32>;
    const int smem = AttnCfg<D, BS>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

cudaError_t launch_decode_attn(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                               int head_dim, int block_size, bool out_f32, int grid,
                               cudaStream_t stream) {
#define PKV_DISPATCH(D_, BS_)                                                         \
    if (head_dim == D_ && block_size == BS_)                                          \
        return out_f32 ? launch_one<D_, BS_, true>(a, tk, tv, grid, stream)           \
                       : launch_one<D_, BS_, false>(a, tk, tv, grid, stream);
    PKV_DISPATCH(128, 16)
    PKV_DISPATCH(128, 32)
    PKV_DISPATCH(64, 16)
    PKV_DISPATCH(64, 32)
#undef PKV_DISPATCH
    return cudaErrorInvalidValue;
}

}  // namespace pkv
