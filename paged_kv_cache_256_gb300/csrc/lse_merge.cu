// lse_merge.cu -- combine the split pieces of a (sequence, KV head) unit.
//
// Each piece of a unit -- a (sequence, KV head, row tile) -- that the
// attention kernel split across CTAs left, per query row, its running max m (base-2 domain), running sum l and
// unnormalised output o.  The exact combination is
//     M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p,
// the rescale-and-combine rule of the online softmax ("Efficient inference",
// FlashAttention: exact attention without the matrix; FlashDecoding is named
// in CS336 lecture-10 notes, PagedAttention (vLLM)).  Pieces with l == 0 (no
// visible key) weigh nothing, and a row whose pieces are all empty is zero.
//
// Grid (attention CTAs) x (row groups); each warp merges kMergeRowsPerWarp
// output rows.  (The paired form's 256-row units take the second kernel
// below, lse_merge_units_kernel.)  Block (c, y) looks at the records of attention CTA c: if one
// of them starts a split unit (the unit's first block, not its last), its
// warps find the CTAs c+1, c+2, ... holding the unit's other pieces with a
// lane-parallel ballot over their records and combine their rows.  Every
// split unit has exactly one starting piece, so each unit is merged exactly
// once.  The loads are arranged in as few dependent rounds as possible: the
// records of CTA c and of the next 32 CTAs together; then every piece's
// (m, l) (lane k <-> piece k) together with the outputs of the first
// kMergeChunk pieces; M, the weights and the denominator follow from
// registers.  Pieces come in groups of 32 and the running combination is
// rescaled when a later group raises M (the same exact rule).
//
// The kernel is launched as a programmatic dependent of the attention kernel:
// it may start while the attention grid drains and waits (griddepcontrol)
// for the attention grid to finish before reading any record.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

// Warps per block: 8 for units of up to 64 rows; 4 for 128-row units (MQA
// verify, prefill tiles), whose eight times as many blocks then start two to
// an SM beside the attention CTAs (measured: MQA verify 40.1 -> 39.4 us,
// prefill 97.0 -> 96.4 us; GQA slower with 4).
constexpr int kMergeRowsPerWarp = 2;
constexpr int kMergeChunk = 4;  // pieces whose outputs are loaded together

template <int V>
struct VecF;
template <>
struct VecF<4> {
    __device__ static void load(const float* p, float (&x)[4]) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    }
};
template <>
struct VecF<2> {
    __device__ static void load(const float* p, float (&x)[2]) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x;
        x[1] = v.y;
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <int D, bool OUT_F32, int kMergeWarps>
__global__ void __launch_bounds__(kMergeWarps * 32, 32 / kMergeWarps)
    lse_merge_kernel(const AttnArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int V = D / 32;  // consecutive columns per lane
    constexpr int RW = kMergeRowsPerWarp;
    const int c = blockIdx.x, grid = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (blockIdx.y * kMergeWarps + warp) * RW;  // this warp's first row
    if (r0 >= a.rows) return;

    // First load round: CTA c's records and the first records of CTAs c+1 .. c+32.
    const int4 i1 = a.rec_info[(size_t)c * 2 + 1];
    const int4 i0 = a.rec_info[(size_t)c * 2 + 0];
    const int cn = c + 1 + lane;
    const int4 nx = cn < grid ? a.rec_info[(size_t)cn * 2] : make_int4(0, 0, 0, 0);
    int first_rec;
    int4 head;
    if (i1.z & kRecValid) {
        first_rec = c * 2 + 1;
        head = i1;
    } else if ((i0.z & kRecValid) && (i0.z & kRecFirst) && !(i0.z & kRecLast)) {
        first_rec = c * 2;
        head = i0;
    } else {
        return;
    }
    const int s = head.x, h = head.y, tile = head.w;

    // The unit's last piece: the first CTA after c whose first record closes
    // the unit, with only this unit's pieces or empty CTAs between.
    int npc = -1;  // the pieces are c (first_rec) and the CTAs c+1 .. c+npc
    for (int base = c + 1; base < grid && npc < 0; base += 32) {
        const int c2 = base + lane;
        const int4 in = base == c + 1 ? nx : (c2 < grid ? a.rec_info[(size_t)c2 * 2] : make_int4(0, 0, 0, 0));
        const bool same =
            c2 < grid && (in.z & kRecValid) && in.x == s && in.y == h && in.w == tile;
        const bool cont = same || (c2 < grid && (in.z & kRecEmpty));
        const unsigned ends = __ballot_sync(0xffffffffu, (same && (in.z & kRecLast)) || !cont);
        if (ends) {
            const int k = __ffs(ends) - 1;
            const bool closed = __shfl_sync(0xffffffffu, same && (in.z & kRecLast), k);
            if (!closed) {
                if (lane == 0) atomicOr(a.err, kErrInternal);
                return;
            }
            npc = base + k - c;
        }
    }
    if (npc < 0) {
        if (lane == 0) atomicOr(a.err, kErrInternal);
        return;
    }

    float M[RW], den[RW], acc[RW][V];
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
        M[rr] = -INFINITY;
        den[rr] = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[rr][v] = 0.f;
    }
    // Flags of CTA c + lane (lanes >= 1), from the first load round.
    const int z_near = __shfl_sync(0xffffffffu, nx.z, (lane + 31) & 31);
    for (int kg = 0; kg <= npc; kg += 32) {
        // Lane k <-> piece kg + k: its record, or -1 (past the unit, or an
        // empty CTA whose slots hold nothing of it).
        const int k = kg + lane;
        int rec = -1;
        if (k == 0) {
            rec = first_rec;
        } else if (k <= npc) {
            const int z = kg == 0 ? z_near : a.rec_info[(size_t)(c + k) * 2].z;
            if (!(z & kRecEmpty)) rec = (c + k) * 2;
        }
        const int cnt = min(32, npc + 1 - kg);  // pieces of this group
        float2 ml[RW];
#pragma unroll
        for (int rr = 0; rr < RW; ++rr)
            ml[rr] = (rec >= 0 && r0 + rr < a.rows)
                         ? *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec * a.rows + r0 + rr) * 2)
                         : make_float2(-INFINITY, 0.f);
        for (int q0 = 0; q0 < cnt; q0 += kMergeChunk) {
            float x[kMergeChunk][RW][V];
            int live = 0;
#pragma unroll
            for (int u = 0; u < kMergeChunk; ++u) {
                const int q = q0 + u;
                const int rq = __shfl_sync(0xffffffffu, rec, q & 31);
                const bool ok = q < cnt && rq >= 0;
                live |= ok ? 1 << u : 0;
#pragma unroll
                for (int rr = 0; rr < RW; ++rr) {
                    if (ok && r0 + rr < a.rows)
                        VecF<V>::load(a.rec_o + ((size_t)rq * a.rows + r0 + rr) * D + lane * V, x[u][rr]);
                    else
#pragma unroll
                        for (int v = 0; v < V; ++v) x[u][rr][v] = 0.f;
                }
            }
            float wk[RW];
#pragma unroll
            for (int rr = 0; rr < RW; ++rr) {
                if (q0 == 0) {
                    // The group's largest running max; pieces with l == 0 weigh nothing.
                    const float mg = warp_max(ml[rr].y > 0.f ? ml[rr].x : -INFINITY);
                    if (mg > M[rr]) {
                        const float f = M[rr] == -INFINITY ? 0.f : fast_exp2(M[rr] - mg);
                        den[rr] *= f;
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[rr][v] *= f;
                        M[rr] = mg;
                    }
                }
                wk[rr] = ml[rr].y > 0.f ? fast_exp2(ml[rr].x - M[rr]) : 0.f;
                if (q0 == 0) den[rr] += warp_sum(wk[rr] * ml[rr].y);
            }
#pragma unroll
            for (int u = 0; u < kMergeChunk; ++u) {
#pragma unroll
                for (int rr = 0; rr < RW; ++rr) {
                    const float w = __shfl_sync(0xffffffffu, wk[rr], (q0 + u) & 31);
                    if ((live >> u & 1) && w != 0.f) {
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[rr][v] += w * x[u][rr][v];
                    }
                }
            }
        }
    }

    const int G = a.group;
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
        const int r = r0 + rr;
        // Row r of the unit's row tile: query token i, query head hq (padding
        // rows of a partial last tile have no output).
        const int R = tile * a.rows + r;
        if (r >= a.rows || R >= a.rows_total) continue;
        const float inv = den[rr] > 0.f ? 1.f / den[rr] : 0.f;
        const int i = R / G, hq = h * G + R % G;
        const size_t ob = (((size_t)s * a.q_len + i) * a.n_q + hq) * D + lane * V;
        if (OUT_F32) {
            float* op = static_cast<float*>(a.out) + ob;
#pragma unroll
            for (int v = 0; v < V; ++v) op[v] = acc[rr][v] * inv;
        } else {
            uint32_t* op = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + ob);
#pragma unroll
            for (int v = 0; v < V; v += 2)
                op[v / 2] = pack_bf16x2(acc[rr][v] * inv, acc[rr][v + 1] * inv);
        }
    }
}

// The paired tensor-memory form's 256-row units, over at most kUnitMaxGrid
// attention CTAs.  One block per (attention CTA, row group) left most of the
// blocks waiting for a later launch wave (chunked prefill: block starts
// spread over 8 us after the attention grid ended).  Here a grid of
// kUnitBlocksPerSm blocks per attention CTA lists the split units once per
// block -- every CTA's records into shared memory, one thread per CTA finds
// the unit its records start and counts its pieces -- and the blocks take
// (unit, 16-row group) items in turn.  An item's rows of up to kUnitPieces
// pieces arrive by one bulk copy each (a piece's record rows are contiguous:
// 8 KB at head_dim 128) into shared memory, beside plain loads of their
// (m, l); 16 threads share a row, each combining head_dim / 16 columns by the
// same exact rule.  Measured (attention call, trimmed means of the same
// buffers): chunked prefill 78.5 -> 76.6 us; for 128-row units it was no
// faster (MQA verify e4m3 48.3 -> 49.9 us), so those keep the kernel above.
constexpr int kUnitRows = 16;        // rows of a work item
constexpr int kUnitPieces = 4;       // pieces staged per round
constexpr int kUnitThreads = 256;    // 16 threads per row
constexpr int kUnitMaxGrid = 256;    // attention CTAs whose records a block lists
constexpr int kUnitBlocksPerSm = 4;  // merge blocks per attention CTA

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kUnitThreads, kUnitBlocksPerSm)
    lse_merge_units_kernel(const AttnArgs a, int attn_grid) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int CW = D / 16;  // columns per thread: CW / 4 groups of 4, 64 columns apart
    extern __shared__ __align__(128) float s_buf[];  // [kUnitPieces][kUnitRows][D]
    __shared__ int4 s_info[kUnitMaxGrid][2];
    __shared__ int s_cta[kUnitMaxGrid], s_first[kUnitMaxGrid], s_npc[kUnitMaxGrid];
    __shared__ int s_wn[kUnitThreads / 32];
    __shared__ int s_n;
    __shared__ __align__(8) uint64_t s_bar;
    const int tid = threadIdx.x;
    static_assert(kUnitMaxGrid <= kUnitThreads, "one thread per attention CTA");
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_barrier_init();
    }
    for (int c = tid; c < attn_grid; c += kUnitThreads) {
        s_info[c][0] = a.rec_info[(size_t)c * 2];
        s_info[c][1] = a.rec_info[(size_t)c * 2 + 1];
    }
    __syncthreads();
    // The split units: the one each CTA's records start (its last piece, or a
    // first piece that does not close its unit), with the CTAs c+1 .. c+npc
    // that hold its other pieces (only its pieces or empty CTAs between).
    // Thread c takes CTA c (attn_grid <= kUnitThreads); the list is in CTA
    // order, the same in every block, which take its items in turn.
    const int c = tid;
    int first = -1, npc = -1;
    if (c < attn_grid) {
        const int4 i0 = s_info[c][0], i1 = s_info[c][1];
        int4 head = make_int4(0, 0, 0, 0);
        if (i1.z & kRecValid) {
            first = c * 2 + 1;
            head = i1;
        } else if ((i0.z & kRecValid) && (i0.z & kRecFirst) && !(i0.z & kRecLast)) {
            first = c * 2;
            head = i0;
        }
        if (first >= 0) {
            for (int c2 = c + 1; c2 < attn_grid; ++c2) {
                const int4 in = s_info[c2][0];
                const bool same =
                    (in.z & kRecValid) && in.x == head.x && in.y == head.y && in.w == head.w;
                if (same && (in.z & kRecLast)) {
                    npc = c2 - c;
                    break;
                }
                if (!same && !(in.z & kRecEmpty)) break;
            }
            if (npc < 0) {
                if (blockIdx.x == 0) atomicOr(a.err, kErrInternal);
                first = -1;
            }
        }
    }
    const unsigned listed = __ballot_sync(0xffffffffu, first >= 0);
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 0) s_wn[warp] = __popc(listed);
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kUnitThreads / 32; ++w) {
        base += w < warp ? s_wn[w] : 0;
        total += s_wn[w];
    }
    if (first >= 0) {
        const int k = base + __popc(listed & ((1u << lane) - 1u));
        s_cta[k] = c;
        s_first[k] = first;
        s_npc[k] = npc;
    }
    if (tid == 0) s_n = total;
    __syncthreads();

    const int groups = (a.rows + kUnitRows - 1) / kUnitRows;
    const int n_items = s_n * groups;
    // 16 threads per row; a group of 4 columns per thread and 64-column chunk,
    // so each chunk's loads and stores are contiguous across the 16 threads
    const int row = tid >> 4, col = (tid & 15) * 4;
    const uint64_t pol = l2_policy_evict_first();
    uint32_t phase = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int u = it / groups, r0 = (it - u * groups) * kUnitRows;
        const int cu = s_cta[u], np = s_npc[u], fr = s_first[u];
        const int4 head = s_info[cu][fr & 1];
        const int nrows = min(kUnitRows, a.rows - r0);
        const int r = r0 + row;
        float M = -INFINITY, den = 0.f, acc[CW];
#pragma unroll
        for (int v = 0; v < CW; ++v) acc[v] = 0.f;
        for (int k0 = 0; k0 <= np; k0 += kUnitPieces) {
            // piece k0 + j's record, or -1 (past the unit, or an empty CTA)
            int rec[kUnitPieces];
#pragma unroll
            for (int j = 0; j < kUnitPieces; ++j) {
                const int k = k0 + j;
                rec[j] = k > np ? -1
                         : k == 0 ? fr
                                  : ((s_info[cu + k][0].z & kRecEmpty) ? -1 : (cu + k) * 2);
            }
            if (tid == 0) {
                const uint32_t bytes = static_cast<uint32_t>(nrows) * D * 4u;
                uint32_t total = 0;
#pragma unroll
                for (int j = 0; j < kUnitPieces; ++j) total += rec[j] >= 0 ? bytes : 0u;
                mbar_arrive_expect_tx(&s_bar, total);
#pragma unroll
                for (int j = 0; j < kUnitPieces; ++j)
                    if (rec[j] >= 0)
                        bulk_load(s_buf + j * kUnitRows * D, a.rec_o + ((size_t)rec[j] * a.rows + r0) * D,
                                  bytes, &s_bar, pol);
            }
            float2 ml[kUnitPieces];
#pragma unroll
            for (int j = 0; j < kUnitPieces; ++j)
                ml[j] = (rec[j] >= 0 && row < nrows)
                            ? *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec[j] * a.rows + r) * 2)
                            : make_float2(-INFINITY, 0.f);
            const bool good = mbar_wait_bounded(&s_bar, phase);
            phase ^= 1u;
            if (__syncthreads_or(!good)) {  // (copies that never land: the context is failing)
                if (tid == 0) atomicOr(a.err, kErrTimeout);
                return;
            }
            // The round's largest running max (pieces with l == 0 weigh nothing),
            // then each piece's weight against the unit's running max.
            float mg = -INFINITY;
#pragma unroll
            for (int j = 0; j < kUnitPieces; ++j)
                if (ml[j].y > 0.f) mg = fmaxf(mg, ml[j].x);
            if (mg > M) {
                const float f = M == -INFINITY ? 0.f : fast_exp2(M - mg);
                den *= f;
#pragma unroll
                for (int v = 0; v < CW; ++v) acc[v] *= f;
                M = mg;
            }
#pragma unroll
            for (int j = 0; j < kUnitPieces; ++j) {
                if (!(ml[j].y > 0.f)) continue;
                const float w = fast_exp2(ml[j].x - M);
                den += w * ml[j].y;
                const float* x = s_buf + (j * kUnitRows + row) * D + col;
#pragma unroll
                for (int v = 0; v < CW / 4; ++v) {
                    const float4 q = *reinterpret_cast<const float4*>(x + 64 * v);
                    acc[4 * v] += w * q.x;
                    acc[4 * v + 1] += w * q.y;
                    acc[4 * v + 2] += w * q.z;
                    acc[4 * v + 3] += w * q.w;
                }
            }
            __syncthreads();  // every thread has read the staged rows
        }
        // Row r of the unit's row tile: query token i, query head hq (padding
        // rows of a partial last tile have no output).
        const int R = head.w * a.rows + r;
        if (row >= nrows || R >= a.rows_total) continue;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int G = a.group, i = R / G, hq = head.y * G + R % G;
        const size_t ob = (((size_t)head.x * a.q_len + i) * a.n_q + hq) * D + col;
#pragma unroll
        for (int v = 0; v < CW / 4; ++v) {
            if (OUT_F32)
                *reinterpret_cast<float4*>(static_cast<float*>(a.out) + ob + 64 * v) =
                    make_float4(acc[4 * v] * inv, acc[4 * v + 1] * inv, acc[4 * v + 2] * inv,
                                acc[4 * v + 3] * inv);
            else
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + ob + 64 * v) =
                    make_uint2(pack_bf16x2(acc[4 * v] * inv, acc[4 * v + 1] * inv),
                               pack_bf16x2(acc[4 * v + 2] * inv, acc[4 * v + 3] * inv));
        }
    }
}

template <int D, bool F32, int kMergeWarps>
static cudaError_t launch_merge_one(const AttnArgs& a, int grid, cudaStream_t stream) {
    constexpr int kRowsPerBlock = kMergeWarps * kMergeRowsPerWarp;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, (a.rows + kRowsPerBlock - 1) / kRowsPerBlock, 1);
    cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, F32, kMergeWarps>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool F32>
static cudaError_t launch_merge_units(const AttnArgs& a, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid * kUnitBlocksPerSm, 1, 1);
    cfg.blockDim = dim3(kUnitThreads, 1, 1);
    cfg.dynamicSmemBytes = kUnitPieces * kUnitRows * D * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_units_kernel<D, F32>, a, grid);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool F32>
static cudaError_t launch_merge_rows(const AttnArgs& a, int grid, cudaStream_t stream) {
    if (a.rows > 128 && grid <= kUnitMaxGrid) return launch_merge_units<D, F32>(a, grid, stream);
    return a.rows > 64 ? launch_merge_one<D, F32, 4>(a, grid, stream)
                       : launch_merge_one<D, F32, 8>(a, grid, stream);
}

cudaError_t launch_lse_merge(const AttnArgs& a, int head_dim, bool out_f32, int grid,
                             cudaStream_t stream) {
    if (head_dim == 128)
        return out_f32 ? launch_merge_rows<128, true>(a, grid, stream)
                       : launch_merge_rows<128, false>(a, grid, stream);
    if (head_dim == 64)
        return out_f32 ? launch_merge_rows<64, true>(a, grid, stream)
                       : launch_merge_rows<64, false>(a, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
