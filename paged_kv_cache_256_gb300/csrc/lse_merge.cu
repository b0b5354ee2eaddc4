// lse_merge.cu -- combine the split pieces of a (sequence, KV head) unit.
//
// Each piece of a unit that the attention kernel split across CTAs left, per
// query row, its running max m (base-2 domain), running sum l and
// unnormalised output o.  The exact combination is
//     M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p,
// the rescale-and-combine rule of the online softmax ("Efficient inference",
// FlashAttention: exact attention without the matrix; FlashDecoding is named
// in CS336 lecture-10 notes, PagedAttention (vLLM)).  Pieces with l == 0 (no
// visible key) weigh nothing, and a row whose pieces are all empty is zero.
//
// Merge CTA c looks at the records of attention CTA c: if one of them starts
// a split unit (the unit's first block, not its last), it walks forward over
// CTAs c+1, c+2, ... whose first record continues that unit until the piece
// holding the unit's last block, and writes the merged rows.  Every split
// unit has exactly one starting piece, so each unit is merged exactly once.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kMergeThreads = 128;

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const AttnArgs a) {
    constexpr int V = D / 32;  // consecutive columns per lane
    const int c = blockIdx.x, grid = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
    const int s = head.x, h = head.y;

    // Find the CTA holding the unit's last piece.
    int c_end = c;
    bool closed = false;
    for (int c2 = c + 1; c2 < grid; ++c2) {
        const int4 in = a.rec_info[(size_t)c2 * 2];
        if (in.z & kRecEmpty) continue;
        if (!(in.z & kRecValid) || in.x != s || in.y != h) break;
        c_end = c2;
        if (in.z & kRecLast) {
            closed = true;
            break;
        }
    }
    if (!closed) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrInternal);
        return;
    }

    const int G = a.group;
    for (int r = warp; r < a.rows; r += kMergeThreads / 32) {
        // pass 1: the largest running max among non-empty pieces
        float M = -INFINITY;
        for (int c2 = c; c2 <= c_end; ++c2) {
            const int rec = c2 == c ? first_rec : c2 * 2;
            if (c2 != c && (a.rec_info[(size_t)c2 * 2].z & kRecEmpty)) continue;
            const float2 ml = *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec * a.rows + r) * 2);
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        const float mb = M == -INFINITY ? 0.f : M;
        // pass 2: weighted sums
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        float den = 0.f;
        for (int c2 = c; c2 <= c_end; ++c2) {
            const int rec = c2 == c ? first_rec : c2 * 2;
            if (c2 != c && (a.rec_info[(size_t)c2 * 2].z & kRecEmpty)) continue;
            const float2 ml = *reinterpret_cast<const float2*>(a.rec_ml + ((size_t)rec * a.rows + r) * 2);
            if (!(ml.y > 0.f)) continue;
            const float wgt = fast_exp2(ml.x - mb);
            den += wgt * ml.y;
            const float* ro = a.rec_o + ((size_t)rec * a.rows + r) * D + lane * V;
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] += wgt * ro[v];
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int i = r / G, hq = h * G + r % G;
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
}

cudaError_t launch_lse_merge(const AttnArgs& a, int head_dim, bool out_f32, int grid,
                             cudaStream_t stream) {
    if (head_dim == 128) {
        if (out_f32)
            lse_merge_kernel<128, true><<<grid, kMergeThreads, 0, stream>>>(a);
        else
            lse_merge_kernel<128, false><<<grid, kMergeThreads, 0, stream>>>(a);
    } else if (head_dim == 64) {
        if (out_f32)
            lse_merge_kernel<64, true><<<grid, kMergeThreads, 0, stream>>>(a);
        else
            lse_merge_kernel<64, false><<<grid, kMergeThreads, 0, stream>>>(a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pkv
