// pkv_internal.h -- declarations shared by the C-ABI front end and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

// Record flags of a split piece (see decode_attn.cu).
constexpr int kRecValid = 1;  // the slot holds a piece of a split unit
constexpr int kRecFirst = 2;  // the piece starts at the unit's first block
// (record info = {sequence, KV head, flags, row tile})
constexpr int kRecLast = 4;   // the piece ends at the unit's last block
constexpr int kRecEmpty = 8;  // the CTA owned no blocks at all

constexpr unsigned kErrInternal = 8u;  // inconsistent split records (after a timeout)

struct AttnArgs {
    const uint16_t* q;            // [num_seqs][q_len][n_q][head_dim] bf16
    const int32_t* block_tables;  // [num_seqs][max_blocks_per_seq]
    const int32_t* context_lens;  // [num_seqs]
    void* out;                    // [num_seqs][q_len][n_q][head_dim] bf16 or f32
    unsigned* err;                // workspace error word
    int4* rec_info;               // [grid][2] {seq, kv head, flags, row tile}
    float* rec_ml;                // [grid][2][rows][2] {m (log2 domain), l}
    float* rec_o;                 // [grid][2][rows][head_dim] unnormalised output
    int num_seqs;
    int q_len;
    int n_q;
    int n_kv;
    int group;       // n_q / n_kv
    int rows;        // query rows per row tile: rows_total if <= 128, else <= 128 (whole tokens when they fit)
    int rows_total;  // group * q_len: query rows sharing one KV head
    int q_tiles;     // ceil(rows_total / rows): row tiles per (sequence, KV head)
    int max_blocks_per_seq;
    int num_blocks;
    int tile_rows_total;  // rows of the 2-D cache view: num_blocks * n_kv * kv_mul * block_size
    int kv_mul;           // 1: separate K and V caches; 2: one cache, K rows then V rows
    int v_row_off;        // rows from a tile's K rows to its V rows (0 or block_size)
    int warp_rows;        // 16-row tiles per KV unit (1, 2, 4 or 8)
    const float* k_scale;  // 8-bit caches: [n_kv] dequantisation scales (else unused)
    const float* v_scale;
    int window;        // 0: full causal attention; W > 0: a row sees its last W positions
    int unit_cost;     // a unit's fixed work in block equivalents (work partition weight)
    int checked;
    int test_stall;    // failure-path tests: the producer issues nothing
    float scale_log2;  // scale * log2(e): scores are kept in the base-2 domain
    int q_tma;         // tensor-memory consumer, bf16 cache: query tiles arrive by TMA (the q map is valid)
    int early_start;   // launched as a programmatic dependent of the previous kernel
    const float* kv_scales;  // per-(block, KV head) scales [num_blocks][n_kv][4], or null
    int tile_4d;  // the K and V maps are grouped 4-D views: a whole tile in one copy
};

// The tensor maps of one attention launch: the K and V cache views and the
// query tiles (tensor-memory consumer).  With AttnArgs::tile_4d the K and V
// views are four-dimensional: {64 columns, 8 rows, 2 column halves, row groups}.
// Workspace bytes of an attention call in its one-tile form (the least any
// call of these sizes needs; pkv_paged_decode_attn_workspace_size reports
// the paired form's, which some calls use).  0 for invalid shapes.
size_t attn_workspace_min_bytes(int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                                int block_size, unsigned flags);

struct AttnMaps {
    CUtensorMap k, v, q;
};

struct WorkspaceLayout {
    size_t err_off, info_off, ml_off, o_off, total;
};

WorkspaceLayout workspace_layout(int grid, int rows, int head_dim);


cudaError_t launch_decode_attn(const AttnArgs& a, const AttnMaps& maps, int head_dim,
                               int block_size, bool out_f32, int grid, cudaStream_t stream);

cudaError_t launch_decode_attn_fp8(const AttnArgs& a, const AttnMaps& maps, int head_dim,
                                   int block_size, bool out_f32, int grid, cudaStream_t stream);

cudaError_t launch_decode_attn_fp8_block(const AttnArgs& a, const AttnMaps& maps, int head_dim,
                                         int block_size, bool out_f32, int grid,
                                         cudaStream_t stream);

cudaError_t launch_lse_merge(const AttnArgs& a, int head_dim, bool out_f32, int grid,
                             cudaStream_t stream);

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             int num_tokens, int n_kv, int head_dim, int block_size,
                             int num_blocks, void* k_cache, void* v_cache, int num_sms,
                             cudaStream_t stream);

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new,
                                 const int32_t* slot_mapping, int num_tokens, int n_kv,
                                 int head_dim, int block_size, int num_blocks,
                                 const float* k_scale, const float* v_scale, void* kv_cache,
                                 int num_sms, cudaStream_t stream);

cudaError_t launch_kv_append_fp8_block(const void* k_new, const void* v_new,
                                       const int32_t* slot_mapping, int num_tokens, int n_kv,
                                       int head_dim, int block_size, int num_blocks,
                                       void* kv_cache, float* kv_scales, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int n_kv, int head_dim, int block_size,
                               int elem_bytes, void* scales, int num_sms, cudaStream_t stream);

}  // namespace pkv
