// kv_append.cu -- writes into the paged cache: each step's new K/V rows, and
// whole-block copies for copy-on-write.
//
// For token i with slot s = slot_mapping[i] in [0, num_blocks * block_size):
//   cache[s / block_size][g][s % block_size][:] = new[i][g][:]  for every KV head g,
// a bit copy for K and V ("Transformer inference mechanics", What the KV cache
// stores per layer: the cache gains the new token's K/V each step).  Other
// slots are skipped, so a padding token (slot -1) writes nothing.
//
// One thread moves one 16-byte chunk; consecutive threads cover consecutive
// chunks of the same row, then the K row and the V row of the same
// (token, head), so both the reads of k_new/v_new and the writes into the
// cache are full 16-byte vector accesses.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     const int32_t* __restrict__ slot_mapping, long long num_tokens, int n_kv,
                     int chunks, int block_size, long long num_slots, uint4* __restrict__ k_cache,
                     uint4* __restrict__ v_cache) {
    // The attention call that follows may start its work partition now (it
    // reads no cache before this grid completes).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long total = num_tokens * n_kv * 2 * chunks;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int chunk = static_cast<int>(idx % chunks);
        long long rest = idx / chunks;
        const int which = static_cast<int>(rest & 1);  // 0: K, 1: V
        rest >>= 1;
        const int g = static_cast<int>(rest % n_kv);
        const long long tok = rest / n_kv;
        const long long slot = __ldg(slot_mapping + tok);
        if (slot < 0 || slot >= num_slots) continue;
        const long long blk = slot / block_size, off = slot % block_size;
        const size_t dst = (((size_t)blk * n_kv + g) * block_size + off) * chunks + chunk;
        const size_t src = ((size_t)tok * n_kv + g) * chunks + chunk;
        if (which == 0)
            k_cache[dst] = __ldg(k_new + src);
        else
            v_cache[dst] = __ldg(v_new + src);
    }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             int num_tokens, int n_kv, int head_dim, int block_size,
                             int num_blocks, void* k_cache, void* v_cache, int num_sms,
                             cudaStream_t stream) {
    const int chunks = head_dim / 8;
    const long long total = (long long)num_tokens * n_kv * 2 * chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    kv_append_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        num_tokens, n_kv, chunks, block_size, (long long)num_blocks * block_size,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache));
    return cudaGetLastError();
}

// The quantising append into an 8-bit (e4m3) cache, laid out as
// [num_blocks][n_kv][2][block_size][head_dim] (each (block, head)'s K rows,
// then its V rows): the code stored for value x of KV head g is the e4m3
// nearest to x / scale[g] -- the quotient rounded
// to fp32 (IEEE division), then to e4m3 with ties to even, saturating at
// +-448 -- so a cached value decodes to code * scale[g] ("Efficient
// inference", Quantization: quantise and dequantise through a scale).  One
// thread turns 8 bf16 (16 bytes) into 8 codes (8 bytes).
__device__ __forceinline__ uint32_t quantise4(uint32_t lo2, uint32_t hi2, float sc) {
    const float x0 = __fdiv_rn(bf16_lo_to_f32(lo2), sc), x1 = __fdiv_rn(bf16_hi_to_f32(lo2), sc);
    const float x2 = __fdiv_rn(bf16_lo_to_f32(hi2), sc), x3 = __fdiv_rn(bf16_hi_to_f32(hi2), sc);
    return f32x2_to_e4m3x2(x0, x1) | (f32x2_to_e4m3x2(x2, x3) << 16);
}

__global__ void __launch_bounds__(256)
    kv_append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                         const int32_t* __restrict__ slot_mapping, long long num_tokens, int n_kv,
                         int chunks, int block_size, long long num_slots,
                         const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                         uint2* __restrict__ kv_cache) {
    // The attention call that follows may start its work partition now (it
    // reads no cache before this grid completes).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long total = num_tokens * n_kv * 2 * chunks;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int chunk = static_cast<int>(idx % chunks);
        long long rest = idx / chunks;
        const int which = static_cast<int>(rest & 1);  // 0: K, 1: V
        rest >>= 1;
        const int g = static_cast<int>(rest % n_kv);
        const long long tok = rest / n_kv;
        const long long slot = __ldg(slot_mapping + tok);
        if (slot < 0 || slot >= num_slots) continue;
        const long long blk = slot / block_size, off = slot % block_size;
        const size_t dst =
            ((((size_t)blk * n_kv + g) * 2 + which) * block_size + off) * chunks + chunk;
        const size_t src = ((size_t)tok * n_kv + g) * chunks + chunk;
        const uint4 x = __ldg((which == 0 ? k_new : v_new) + src);
        const float sc = __ldg((which == 0 ? k_scale : v_scale) + g);
        kv_cache[dst] = make_uint2(quantise4(x.x, x.y, sc), quantise4(x.z, x.w, sc));
    }
}

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new,
                                 const int32_t* slot_mapping, int num_tokens, int n_kv,
                                 int head_dim, int block_size, int num_blocks,
                                 const float* k_scale, const float* v_scale, void* kv_cache,
                                 int num_sms, cudaStream_t stream) {
    const int chunks = head_dim / 8;
    const long long total = (long long)num_tokens * n_kv * 2 * chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    kv_append_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        num_tokens, n_kv, chunks, block_size, (long long)num_blocks * block_size, k_scale,
        v_scale, static_cast<uint2*>(kv_cache));
    return cudaGetLastError();
}

// The quantising append into an 8-bit cache with one scale per (block, KV
// head) (layout as above, scales [num_blocks][n_kv][4] fp32 = K scale, V
// scale, reserved, reserved).  A scale follows the values of its block: it is
// the smallest power of two 2^e (e >= -126) that keeps the block's largest
// finite value within 448, it only grows while the block fills, and when it
// grows the block's resident rows (those below the call's first offset in
// the block) are re-quantised by the power-of-two ratio -- exact except for
// values that fall below the normal e4m3 range.  A block written from offset
// 0 starts over (its stored scale is ignored); scale 0 stands for "nothing
// but zeros so far".  ("Efficient inference", Quantization: quantise and
// dequantise through a scale.)
//
// One warp per (token, KV head).  The warp of the first token of a run --
// consecutive tokens (skipped slots aside) landing in one block -- handles
// the whole run for its head, K then V: the largest |x| over the run's rows,
// the new scale, the re-quantised resident rows, the run's codes, the scale
// entry.  Every other warp returns.  Lanes take 4 consecutive elements of a
// row at a time.
constexpr int kAppendWarps = 4;  // small CTAs: a decode step's few runs spread over more SMs

// The smallest power of two s = 2^e, e >= -126, with a <= 448 * s (a > 0,
// finite).  r = fp32(a / 448) rounds across no power of two that matters:
// a has 8 significant bits, so when a / 448 exceeds 2^e it does so by at
// least 1/224 of it, far more than fp32 rounding; hence ceil(log2(r)) is
// exactly the wanted e.
__device__ __forceinline__ float pow2_scale_for(float a) {
    const float r = __fdiv_rn(a, 448.f);
    const uint32_t u = __float_as_uint(r);
    int e = static_cast<int>((u >> 23) & 0xFF) - 127;  // floor(log2 r) for normal r
    if ((u & 0x7FFFFFu) != 0) ++e;                      // not a power of two: round up
    if (((u >> 23) & 0xFF) == 0) e = -126;              // r subnormal or 0: below 2^-126
    if (e < -126) e = -126;
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Division by a block scale s.  The scales this append sets are powers of two
// 2^e (-126 <= e <= 127), and for those x / s and x * 2^-e are the same real
// number rounded once, so multiplying by the exact reciprocal gives the IEEE
// quotient bit for bit (subnormal and overflowing results included); any
// other stored scale is divided by.
struct DivBy {
    float s, inv;
    bool pow2;
    __device__ __forceinline__ explicit DivBy(float sc) : s(sc) {
        const uint32_t u = __float_as_uint(sc), ex = (u >> 23) & 0xFFu;
        pow2 = (u & 0x807FFFFFu) == 0u && ex >= 1u && ex <= 253u;
        inv = pow2 ? __uint_as_float((254u - ex) << 23) : 0.f;
    }
    __device__ __forceinline__ float operator()(float x) const {
        return pow2 ? x * inv : __fdiv_rn(x, s);
    }
};

// Four bf16 (two 32-bit words) -> four e4m3 codes of x / s (x itself for s == 0).
__device__ __forceinline__ uint32_t quantise4_by(uint32_t lo2, uint32_t hi2, const DivBy& d) {
    float x0 = bf16_lo_to_f32(lo2), x1 = bf16_hi_to_f32(lo2);
    float x2 = bf16_lo_to_f32(hi2), x3 = bf16_hi_to_f32(hi2);
    if (d.s > 0.f) {
        x0 = d(x0);
        x1 = d(x1);
        x2 = d(x2);
        x3 = d(x3);
    }
    return f32x2_to_e4m3x2(x0, x1) | (f32x2_to_e4m3x2(x2, x3) << 16);
}

// Four codes re-quantised from scale s_old to s_new: e4m3 of fp32(fp32(v * s_old) / s_new).
__device__ __forceinline__ uint32_t requantise4(uint32_t codes, float s_old, const DivBy& d) {
    uint32_t lo, hi;  // f16 pairs of bytes (0, 1) and (2, 3); every e4m3 value is exact in f16
    e4m3x4_to_f16x2x2(codes, lo, hi);
    const float v0 = d(f16_lo_to_f32(lo) * s_old);
    const float v1 = d(f16_hi_to_f32(lo) * s_old);
    const float v2 = d(f16_lo_to_f32(hi) * s_old);
    const float v3 = d(f16_hi_to_f32(hi) * s_old);
    return f32x2_to_e4m3x2(v0, v1) | (f32x2_to_e4m3x2(v2, v3) << 16);
}

__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_fp8_block_kernel(const uint16_t* __restrict__ k_new,
                               const uint16_t* __restrict__ v_new,
                               const int32_t* __restrict__ slot_mapping, int num_tokens, int n_kv,
                               int head_dim, int block_size, long long num_slots,
                               uint8_t* __restrict__ kv_cache, float* __restrict__ kv_scales) {
    // The attention call that follows may start its work partition now (it
    // reads no cache before this grid completes).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    // (the host limits num_tokens * n_kv to fewer than 2^31)
    const unsigned item = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (item >= static_cast<unsigned>(num_tokens * n_kv)) return;
    const int t = static_cast<int>(item / static_cast<unsigned>(n_kv));
    const int g = static_cast<int>(item % static_cast<unsigned>(n_kv));
    // (the host limits the slots to fewer than 2^31: 32-bit arithmetic throughout)
    const int nslots = static_cast<int>(num_slots);
    const unsigned ubs = static_cast<unsigned>(block_size);
    auto valid = [&](int s) { return s >= 0 && s < nslots; };
    auto block_of = [&](int s) { return static_cast<int>(static_cast<unsigned>(s) / ubs); };
    auto offset_of = [&](int s) { return static_cast<int>(static_cast<unsigned>(s) % ubs); };
    // First round of loads, all independent: this token's slot and the 32
    // slots on either side of it (the usual run fits in them).
    const int slot = __ldg(slot_mapping + t);
    const int pb0 = t - 1 - lane, pf0 = t + 1 + lane;
    const int sb0 = pb0 >= 0 ? __ldg(slot_mapping + pb0) : -1;
    const int sf0 = pf0 < num_tokens ? __ldg(slot_mapping + pf0) : -1;
    if (!valid(slot)) return;
    const int blk = block_of(slot);

    // Does the nearest earlier valid token land in the same block?  (Lanes look
    // 32 tokens back at a time; the answer is warp-uniform.)
    for (int base = t - 1; base >= 0; base -= 32) {
        const int p = base - lane;
        const int sp = base == t - 1 ? sb0 : (p >= 0 ? __ldg(slot_mapping + p) : -1);
        const unsigned vm = __ballot_sync(0xffffffffu, p >= 0 && valid(sp));
        if (vm) {
            const int sprev = __shfl_sync(0xffffffffu, sp, __ffs(vm) - 1);
            if (block_of(sprev) == blk) return;  // not the run's first token
            break;
        }
    }
    // The run: tokens t .. end-1 (skipped slots included), and its lowest offset.
    int end = t + 1;
    int o_min = offset_of(slot);
    for (int base = t + 1; base < num_tokens; base += 32) {
        const int p = base + lane;
        const int sp = base == t + 1 ? sf0 : (p < num_tokens ? __ldg(slot_mapping + p) : -1);
        const bool other = p < num_tokens && valid(sp) && block_of(sp) != blk;
        const unsigned stop = __ballot_sync(0xffffffffu, other || p >= num_tokens);
        const int lim = stop ? __ffs(stop) - 1 : 32;  // lanes below lim are in the run
        int off = (lane < lim && valid(sp)) ? offset_of(sp) : block_size;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) off = min(off, __shfl_xor_sync(0xffffffffu, off, o));
        o_min = min(o_min, off);
        end = base + lim;
        if (stop) break;
    }

    // Second round, all independent: the block's scale entry and the run's K
    // and V rows (largest finite |x| of each).
    float* entry = kv_scales + ((size_t)blk * n_kv + g) * 4;
    const float2 s_old2 = o_min > 0 ? *reinterpret_cast<const float2*>(entry) : make_float2(0.f, 0.f);
    float amax[2] = {0.f, 0.f};
#pragma unroll 4
    for (int j = t; j < end; ++j) {
        const int sj = __ldg(slot_mapping + j);
        if (!valid(sj)) continue;
        const size_t rowo = ((size_t)j * n_kv + g) * head_dim;
        for (int e = lane * 4; e < head_dim; e += 128) {
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>((which == 0 ? k_new : v_new) + rowo + e));
                const float x[4] = {bf16_lo_to_f32(v.x), bf16_hi_to_f32(v.x), bf16_lo_to_f32(v.y),
                                    bf16_hi_to_f32(v.y)};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (isfinite(x[k])) amax[which] = fmaxf(amax[which], fabsf(x[k]));
            }
        }
    }
    float s_new2[2];
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        float m = amax[which];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s_old = which == 0 ? s_old2.x : s_old2.y;
        float s_new = s_old;
        if (m > 0.f) s_new = fmaxf(s_old, pow2_scale_for(m));
        s_new2[which] = s_new;
        uint8_t* rows = kv_cache + (((size_t)blk * n_kv + g) * 2 + which) * (size_t)block_size * head_dim;
        if (s_new > s_old && s_old > 0.f) {  // re-quantise the resident rows
            const DivBy d(s_new);
            for (int r = 0; r < o_min; ++r)
                for (int e = lane * 4; e < head_dim; e += 128) {
                    uint32_t* cp = reinterpret_cast<uint32_t*>(rows + (size_t)r * head_dim + e);
                    *cp = requantise4(*cp, s_old, d);
                }
        }
    }
    // The run's codes, in call order (a later token on the same offset writes
    // after an earlier one), then the scale entry.
    const DivBy dk(s_new2[0]), dv(s_new2[1]);
    for (int j = t; j < end; ++j) {
        const int sj = __ldg(slot_mapping + j);
        if (!valid(sj)) continue;
        const size_t rowo = ((size_t)j * n_kv + g) * head_dim;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            uint8_t* dst = kv_cache + (((size_t)blk * n_kv + g) * 2 + which) * (size_t)block_size * head_dim +
                           (size_t)offset_of(sj) * head_dim;
            for (int e = lane * 4; e < head_dim; e += 128) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>((which == 0 ? k_new : v_new) + rowo + e));
                *reinterpret_cast<uint32_t*>(dst + e) = quantise4_by(v.x, v.y, which == 0 ? dk : dv);
            }
        }
        __syncwarp();
    }
    if (lane == 0) *reinterpret_cast<float4*>(entry) = make_float4(s_new2[0], s_new2[1], 0.f, 0.f);
}

cudaError_t launch_kv_append_fp8_block(const void* k_new, const void* v_new,
                                       const int32_t* slot_mapping, int num_tokens, int n_kv,
                                       int head_dim, int block_size, int num_blocks,
                                       void* kv_cache, float* kv_scales, cudaStream_t stream) {
    const long long items = (long long)num_tokens * n_kv;
    const long long blocks = (items + kAppendWarps - 1) / kAppendWarps;
    kv_append_fp8_block_kernel<<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, stream>>>(
        static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), slot_mapping,
        num_tokens, n_kv, head_dim, block_size, (long long)num_blocks * block_size,
        static_cast<uint8_t*>(kv_cache), kv_scales);
    return cudaGetLastError();
}

// One thread moves one 16-byte chunk of a (K or V) block; consecutive threads
// cover consecutive chunks of the same block, so reads and writes are full
// 16-byte vector accesses over whole contiguous blocks.
// scales (8-bit cache with per-block scales): the [num_blocks][n_kv][4] fp32
// scale tensor, n_kv 16-byte chunks per block, copied by the threads that
// would copy V (an interleaved cache has no separate V).
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ pairs, int num_pairs, int num_blocks,
                       long long chunks_per_block, uint4* __restrict__ scales, int n_kv) {
    const long long total = (long long)num_pairs * 2 * chunks_per_block;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long chunk = idx % chunks_per_block;
        const long long rest = idx / chunks_per_block;
        const int which = static_cast<int>(rest & 1);  // 0: K, 1: V
        const int p = static_cast<int>(rest >> 1);
        const int src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst) continue;
        if (which == 1 && scales != nullptr) {
            if (chunk < n_kv)
                scales[(size_t)dst * n_kv + chunk] = scales[(size_t)src * n_kv + chunk];
            continue;
        }
        uint4* cache = which == 0 ? k_cache : v_cache;
        if (cache == nullptr) continue;  // one interleaved cache: its blocks hold K and V
        cache[(size_t)dst * chunks_per_block + chunk] = cache[(size_t)src * chunks_per_block + chunk];
    }
}

// elem_bytes * n_kv * block_size * head_dim bytes per block of each cache; a
// null v_cache (an interleaved 8-bit cache) copies k_cache only.
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int n_kv, int head_dim, int block_size,
                               int elem_bytes, void* scales, int num_sms, cudaStream_t stream) {
    const long long chunks = (long long)n_kv * block_size * head_dim * elem_bytes / 16;
    const long long total = (long long)num_pairs * 2 * chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    copy_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, num_pairs, num_blocks,
        chunks, static_cast<uint4*>(scales), n_kv);
    return cudaGetLastError();
}

}  // namespace pkv
