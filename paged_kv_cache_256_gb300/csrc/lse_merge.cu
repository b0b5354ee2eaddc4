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
// Grid (attention CTAs) x (row groups of 8); one warp per output row.  Block
// (c, y) looks at the records of attention CTA c: if one of them starts a
// split unit (the unit's first block, not its last), its warps find the
// CTAs c+1, c+2, ... holding the unit's other pieces with a lane-parallel
// ballot over their records and combine rows 8y..8y+7.  Every split unit has
// exactly one starting piece, so each unit is merged exactly once.  All loads
// of one row are independent of each other, so a row costs a few memory
// latencies whatever the number of pieces.
//
// The kernel is launched as a programmatic dependent of the attention kernel:
// it may start while the attention grid drains and waits (griddepcontrol)
// for the attention grid to finish before reading any record.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kMergeRowsPerBlock = 8;
constexpr int kMergeThreads = kMergeRowsPerBlock * 32;

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const AttnArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int V = D / 32;  // consecutive columns per lane
    const int c = blockIdx.x, grid = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y * kMergeRowsPerBlock + warp;
    if (r >= a.rows) return;

    const int4 i1 = a.rec_info[(size_t)c * 2 + 1];
    const int4 i0 = a.rec_info[(size_t)c * 2 + 0];
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
    // Row r of the unit's row tile: query token i, query head hq (padding rows of
    // a partial last tile have no output).
    const int R = tile * a.rows + r;
    if (R >= a.rows_total) return;

    // Pieces: first_rec, then the first record of every non-empty CTA in
    // (c, c_end].  Find c_end 32 CTAs at a time.
    int c_end = -1;
    for (int base = c + 1; base < grid && c_end < 0; base += 32) {
        const int c2 = base + lane;
        int4 in = make_int4(0, 0, 0, 0);
        if (c2 < grid) in = a.rec_info[(size_t)c2 * 2];
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
            c_end = base + k;
        }
    }
    if (c_end < 0) {
        if (lane == 0) atomicOr(a.err, kErrInternal);
        return;
    }

    // Pass 1 (lane k <-> piece k of each group of 32): largest running max and
    // the weighted denominator.
    const int npieces = c_end - c + 1;  // candidate slots; empty CTAs weigh 0
    float M = -INFINITY;
    for (int k0 = 0; k0 < npieces; k0 += 32) {
        const int k = k0 + lane;
        if (k < npieces) {
            const int rec = k == 0 ? first_rec : (c + k) * 2;
            const bool live = k == 0 || !(a.rec_info[(size_t)(c + k) * 2].z & kRecEmpty);
            if (live) {
                const float2 ml = *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec * a.rows + r) * 2);
                if (ml.y > 0.f) M = fmaxf(M, ml.x);
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float mb = M == -INFINITY ? 0.f : M;

    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    float den = 0.f;
    for (int k0 = 0; k0 < npieces; k0 += 32) {
        const int k = k0 + lane;
        float wk = 0.f, lk = 0.f;
        if (k < npieces) {
            const int rec = k == 0 ? first_rec : (c + k) * 2;
            const bool live = k == 0 || !(a.rec_info[(size_t)(c + k) * 2].z & kRecEmpty);
            if (live) {
                const float2 ml = *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec * a.rows + r) * 2);
                if (ml.y > 0.f) {
                    wk = fast_exp2(ml.x - mb);
                    lk = ml.y;
                }
            }
        }
        float dpart = wk * lk;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, off);
        den += dpart;
        // Pass 2: every lane accumulates its V columns over the group's pieces.
        const int cnt = min(32, npieces - k0);
        for (int q = 0; q < cnt; ++q) {
            const float wq = __shfl_sync(0xffffffffu, wk, q);
            if (wq == 0.f) continue;  // uniform across the warp
            const int kq = k0 + q;
            const int rec = kq == 0 ? first_rec : (c + kq) * 2;
            const float* ro = a.rec_o + ((size_t)rec * a.rows + r) * D + lane * V;
            if (V == 4) {
                const float4 x = *reinterpret_cast<const float4*>(ro);
                acc[0] += wq * x.x;
                acc[1] += wq * x.y;
                acc[2] += wq * x.z;
                acc[3] += wq * x.w;
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) acc[v] += wq * ro[v];
            }
        }
    }

    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int G = a.group;
    const int i = R / G, hq = h * G + R % G;
    const size_t ob = (((size_t)s * a.q_len + i) * a.n_q + hq) * D + lane * V;
    if (OUT_F32) {
        float* op = static_cast<float*>(a.out) + ob;
#pragma unroll
        for (int v = 0; v < V; ++v) op[v] = acc[v] * inv;
    } else {
        uint32_t* op = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + ob);
#pragma unroll
        for (int v = 0; v < V; v += 2) op[v / 2] = pack_bf16x2(acc[v] * inv, acc[v + 1] * inv);
    }
}

template <int D, bool F32>
static cudaError_t launch_merge_one(const AttnArgs& a, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, (a.rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, F32>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const AttnArgs& a, int head_dim, bool out_f32, int grid,
                             cudaStream_t stream) {
    if (head_dim == 128)
        return out_f32 ? launch_merge_one<128, true>(a, grid, stream)
                       : launch_merge_one<128, false>(a, grid, stream);
    if (head_dim == 64)
        return out_f32 ? launch_merge_one<64, true>(a, grid, stream)
                       : launch_merge_one<64, false>(a, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
