// decode_attn.cu -- the paged decode-attention kernels for bf16 KV caches
// (templates in decode_attn.cuh).
#include "decode_attn.cuh"

namespace pkv {

cudaError_t launch_decode_attn(const AttnArgs& a, const AttnMaps& maps, int head_dim,
                               int block_size, bool out_f32, int grid, cudaStream_t stream) {
    return launch_decode_attn_kv<false, false>(a, maps, head_dim, block_size, out_f32, grid,
                                               stream);
}

}  // namespace pkv
