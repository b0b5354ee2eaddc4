// decode_attn_fp8.cu -- the paged decode-attention kernels for 8-bit (e4m3)
// KV caches with per-KV-head scales (templates in decode_attn.cuh).
#include "decode_attn.cuh"

namespace pkv {

cudaError_t launch_decode_attn_fp8(const AttnArgs& a, const AttnMaps& maps, int head_dim,
                                   int block_size, bool out_f32, int grid, cudaStream_t stream) {
    return launch_decode_attn_kv<true, false>(a, maps, head_dim, block_size, out_f32, grid,
                                              stream);
}

}  // namespace pkv
