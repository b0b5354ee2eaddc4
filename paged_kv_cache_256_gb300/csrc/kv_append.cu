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

// One thread moves one 16-byte chunk of a (K or V) block; consecutive threads
// cover consecutive chunks of the same block, so reads and writes are full
// 16-byte vector accesses over whole contiguous blocks.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ pairs, int num_pairs, int num_blocks,
                       long long chunks_per_block) {
    const long long total = (long long)num_pairs * 2 * chunks_per_block;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long chunk = idx % chunks_per_block;
        const long long rest = idx / chunks_per_block;
        const int which = static_cast<int>(rest & 1);  // 0: K, 1: V
        const int p = static_cast<int>(rest >> 1);
        const int src = __ldg(pairs + 2 * p), dst = __ldg(pairs + 2 * p + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst) continue;
        uint4* cache = which == 0 ? k_cache : v_cache;
        if (cache == nullptr) continue;  // one interleaved cache: its blocks hold K and V
        cache[(size_t)dst * chunks_per_block + chunk] = cache[(size_t)src * chunks_per_block + chunk];
    }
}

// elem_bytes * n_kv * block_size * head_dim bytes per block of each cache; a
// null v_cache (an interleaved 8-bit cache) copies k_cache only.
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int n_kv, int head_dim, int block_size,
                               int elem_bytes, int num_sms, cudaStream_t stream) {
    const long long chunks = (long long)n_kv * block_size * head_dim * elem_bytes / 16;
    const long long total = (long long)num_pairs * 2 * chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    copy_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, num_pairs, num_blocks,
        chunks);
    return cudaGetLastError();
}

}  // namespace pkv
