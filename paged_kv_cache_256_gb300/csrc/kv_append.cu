// kv_append.cu -- write each step's new K/V rows into their paged-cache slots.
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

namespace pkv {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     const int32_t* __restrict__ slot_mapping, long long num_tokens, int n_kv,
                     int chunks, int block_size, long long num_slots, uint4* __restrict__ k_cache,
                     uint4* __restrict__ v_cache) {
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

}  // namespace pkv
