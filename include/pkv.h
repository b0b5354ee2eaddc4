/*
 * pkv.h -- C ABI of the paged decode-attention library (libpkv.so, GB300 / sm_103a).
 *
 * The library computes one decode step of attention over a KV cache that is
 * stored in fixed-size blocks and reached through per-sequence block tables
 * (PagedAttention: "Inference Engines", The Breakthrough, PagedAttention
 * paragraph; CS336 lecture-10 notes, PagedAttention (vLLM)), and writes each
 * step's new keys and values into that cache.
 *
 * Conventions shared by every entry point
 *   - Pointers named *_cache, q, out, k_new, v_new, block_tables,
 *     context_lens, slot_mapping and workspace are DEVICE pointers owned by
 *     the caller.  The library allocates no device memory and keeps no
 *     per-call state; it only caches per-device attributes and driver entry
 *     points.
 *   - bf16 tensors are passed as raw 16-bit patterns (`const void *`).
 *   - `stream` is a cudaStream_t passed as `void *` (NULL = legacy default
 *     stream) and must belong to the current CUDA device.  Calls are
 *     asynchronous on that stream: a PKV_OK return means "validated and
 *     launched"; faults inside a kernel surface at the next synchronisation.
 *   - Programmatic overlap: the attention kernel is launched as a
 *     programmatic dependent of the kernel before it on the stream, and the
 *     append kernels let their dependents start at once.  So an attention
 *     call right after an append begins its work partition (it reads
 *     context_lens, and nothing else) while the append runs, and reads the
 *     caches, q and block_tables, and writes anything, only after it has
 *     completed.  A preceding kernel that does not signal early completion
 *     (any kernel outside this library) is waited for as usual; one that
 *     does must not write context_lens, unless the call passes
 *     PKV_FLAG_NO_EARLY_START.
 *   - Argument checks run on the host before anything is launched; a failed
 *     check returns a status and launches nothing.
 *   - Device pointers to bf16 / fp32 tensors must be 16-byte aligned, int32
 *     arrays 4-byte aligned.
 *   - Every index is int32; products that address memory are computed in 64 bits.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,     /* null pointer, negative size, n_q % n_kv != 0, misalignment */
    PKV_ERR_UNSUPPORTED = 2,     /* valid but outside the built kernels (head_dim, block_size, rows) */
    PKV_ERR_WORKSPACE = 3,       /* workspace missing or smaller than the size query asked for */
    PKV_ERR_CUDA = 4,            /* a CUDA runtime / driver call or a launch failed */
    PKV_ERR_BAD_BLOCK_TABLE = 5, /* CHECKED mode found a block index or context length out of range */
    PKV_ERR_TIMEOUT = 6,         /* a bounded in-kernel wait gave up (the kernel returned early) */
    PKV_ERR_OUT_OF_BLOCKS = 7    /* the block pool has too few free blocks (nothing was changed) */
} pkv_status;

/* kv_dtype values (pkv_attn_params). */
#define PKV_KV_BF16 0     /* caches hold bf16 */
#define PKV_KV_FP8_E4M3 1 /* caches hold e4m3 codes with per-KV-head scales */
#define PKV_KV_FP8_E4M3_BLOCK 2 /* e4m3 codes with one scale per (block, KV head) */

/* out_dtype values. */
#define PKV_OUT_BF16 0 /* round-to-nearest-even bf16 */
#define PKV_OUT_F32 1  /* fp32 (debug / tight-parity path; probabilities kept to ~16 bits) */

/* flags bits. */
#define PKV_FLAG_CHECKED 0x1u /* bounds-check block indices and context lengths on the device */
/* For tests of the failure path only: the attention kernel issues no loads,
 * so every bounded in-kernel wait expires (after about a second), the kernel
 * winds down and pkv_check_error reports PKV_ERR_TIMEOUT.  The output of
 * such a call is not valid; the context stays usable. */
#define PKV_FLAG_TEST_STALL 0x2u
/* pkv_copy_blocks: the cache is the interleaved 8-bit (e4m3) cache. */
#define PKV_FLAG_KV_FP8 0x4u
/* Attention calls: launch the attention kernel as an ordinary (not a
 * programmatic) dependent of the kernel before it, so it reads nothing,
 * context_lens included, before that kernel has completed.  For callers whose
 * preceding kernel signals early completion and writes context_lens. */
#define PKV_FLAG_NO_EARLY_START 0x8u
/* pkv_copy_blocks: the 8-bit cache has per-(block, KV head) scales; v_cache
 * is then its scale tensor, copied with the blocks (needs PKV_FLAG_KV_FP8). */
#define PKV_FLAG_KV_BLOCK_SCALES 0x10u
/* Attention calls on a bf16 cache with head_dim 128 and more than 64 query
 * rows per KV head: fetch each K and V tile as two 64-column copies, the
 * form used when the CUDA driver declines the one-copy (four-dimensional) views
 * of the caches.  Results are bit-identical either way; tests use it to run
 * both. */
#define PKV_FLAG_TILE_2D 0x20u
/* Attention calls: keep one tile of at most 128 query rows per unit even
 * where two would be taken together (the paired form: bf16 cache, bf16
 * output, more than 128 query rows per KV head; it also falls back to one
 * tile when the workspace is smaller than the size query reports).  Results
 * agree within the stated tolerance; tests use it to run both forms. */
#define PKV_FLAG_ONE_TILE 0x40u
/* Bits 16..31 force the number of attention CTAs (0 = one per SM).  Tests
 * use it to move where long contexts are split; results stay within the
 * stated tolerance for every value. */
#define PKV_FLAG_GRID_SHIFT 16
#define PKV_FLAG_GRID(n) (((unsigned)(n) & 0xFFFFu) << PKV_FLAG_GRID_SHIFT)

/*
 * pkv_paged_decode_attn -- one decode step of paged attention.
 *
 * Computes, for every sequence b, new query token i < q_len and query head h,
 *     out[b][i][h] = softmax_t( scale * q[b][i][h] . K_b[t] ) . V_b[t],
 *     over logical positions t <= context_lens[b] - q_len + i,
 * the causal decoder attention of "Transformer inference mechanics", What Q,
 * K, and V do in causal attention, with K_b, V_b read through the block
 * table.  Query head h reads KV head h / (n_q / n_kv): MHA when n_kv == n_q,
 * GQA for groups, MQA when n_kv == 1 ("Transformer inference mechanics", MHA
 * versus MQA versus GQA).  Each KV block is read once for all query heads of
 * its group and all q_len tokens.  Long contexts are split across CTAs and
 * combined with a log-sum-exp merge (FlashDecoding, named in CS336 lecture-10
 * notes, PagedAttention (vLLM); exact combination of partial softmax
 * results, "Efficient inference", FlashAttention section).
 *
 * Layouts (all row-major, contiguous):
 *   q            [num_seqs][q_len][n_q][head_dim]           bf16
 *   k_cache      [num_blocks][n_kv][block_size][head_dim]    bf16 (v_cache alike)
 *   block_tables [num_seqs][max_blocks_per_seq]              int32 physical block ids
 *   context_lens [num_seqs]                                  int32 resident tokens,
 *                including the q_len new ones (their K/V must already be appended)
 *   out          [num_seqs][q_len][n_q][head_dim]            bf16 or fp32 (out_dtype)
 *   Token t of sequence b lives in block block_tables[b][t / block_size] at
 *   offset t % block_size.  Only entries t / block_size < ceil(ctx/block_size)
 *   are read; slots past the context in the last block are never used, and
 *   may hold any bits (NaN included).
 *
 * q_len new tokens per sequence: 1 for plain decoding, a few for a
 *   speculative-verify step, or a whole prompt chunk (paged / chunked
 *   prefill: the prompt pass before decoding, "Efficient inference", Two
 *   phases, two bottlenecks; chunked prefill is named among the scheduling
 *   techniques in "Transformer inference mechanics", A better connection
 *   map).  The rows = (n_q / n_kv) * q_len query rows that share a KV head
 *   are processed in tiles of at most 128 (whole query tokens when one
 *   token's heads fit); each tile reads only the blocks its rows can see.
 * Supported: head_dim in {64, 128}; block_size in {16, 32}; q_len <= 65536;
 *   rows <= 2^24; num_blocks * n_kv * block_size < 2^31.
 * Rows that see no key (context_lens[b] == 0, or < q_len) are written as zeros.
 *
 * workspace: device memory of at least pkv_paged_decode_attn_workspace_size(...)
 *   bytes, zero-filled once before its first use; the library leaves it
 *   reusable (its error word is cleared by pkv_check_error).  One workspace
 *   must not be shared by calls that may run concurrently.
 * flags: PKV_FLAG_CHECKED makes the kernel validate every block index it
 *   reads (0 <= id < num_blocks) and every context length
 *   (0 <= ctx <= max_blocks_per_seq * block_size, ctx == 0 or ctx >= q_len);
 *   violations are clamped, recorded in the workspace and reported by
 *   pkv_check_error as PKV_ERR_BAD_BLOCK_TABLE.  Without it, context lengths
 *   are still clamped to the table width and an out-of-range block id reads
 *   zeros (the tensor-memory-access unit fills out-of-bounds tiles), so no
 *   call reads outside the caches.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE
 *   or PKV_ERR_CUDA.  num_seqs == 0 returns PKV_OK and launches nothing.
 */
int pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                          int block_size, int max_blocks_per_seq, int num_blocks,
                          float scale, void *out, int out_dtype,
                          void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream);

/*
 * pkv_paged_decode_attn_ex -- pkv_paged_decode_attn with every argument in
 * one struct, plus the options the positional form does not have.
 *
 * window: 0 = full causal attention (exactly pkv_paged_decode_attn).  W > 0
 *   is sliding-window (local) attention: query token i, at position
 *   pos = context_lens[b] - q_len + i, sees only positions pos - W + 1 .. pos,
 *   its own and the W - 1 before it (CS336 lecture-10 notes, Local attention &
 *   sparse variants).  KV blocks that no row of a sequence can see are not
 *   read, so a step costs about min(ctx, W + q_len) tokens per sequence.  The
 *   cache itself is unchanged: the caller may keep or release blocks that
 *   have left every window.  W >= max_blocks_per_seq * block_size is the same
 *   as 0.  W < 0 returns PKV_ERR_INVALID_ARG.
 * kv_dtype: PKV_KV_BF16, or PKV_KV_FP8_E4M3 for an 8-bit cache -- fewer
 *   bytes per cached element, dequantised through a scale ("Efficient
 *   inference", Quantization: fewer bytes per weight; CS336 lecture-10 notes,
 *   Quantization & pruning).  The cache is then ONE tensor of e4m3 codes
 *   (OCP FP8 E4M3: bias 7, largest finite 448, no infinity) passed as
 *   k_cache, with v_cache NULL:
 *       kv_cache [num_blocks][n_kv][2][block_size][head_dim]   (1 byte each)
 *   -- for every (block, KV head) its K rows, then its V rows, so the two
 *   tiles a KV head reads from a block are one contiguous 2 * block_size *
 *   head_dim run (random 4 KB runs stream much faster than 2 KB ones).
 *   k_scale / v_scale are DEVICE fp32 arrays [n_kv]: the value of code c in
 *   KV head g is c * k_scale[g] for K and c * v_scale[g] for V.
 *   The result is the attention over those values.  Inside the kernel Q and
 *   the probabilities are rounded to f16 (|q| must stay below 65504), the
 *   products accumulate in fp32.  pkv_kv_append_fp8 writes such a cache.
 *   The cache pointer must be 16-byte aligned.  k_scale / v_scale are
 *   ignored for PKV_KV_BF16.  Any other kv_dtype, a non-NULL v_cache with an
 *   8-bit cache or a NULL one with bf16, returns PKV_ERR_INVALID_ARG.
 *   PKV_KV_FP8_E4M3_BLOCK: the same 8-bit cache, but each (block, KV head)
 *   has its own scales, so a scale follows the values of its block
 *   (pkv_kv_append_fp8_block sets them):
 *       kv_scales [num_blocks][n_kv][4]   fp32, 16-byte aligned
 *   holding the K scale, the V scale and two reserved words per (block,
 *   head).  Token t of sequence b decodes as code * the scale of block
 *   block_tables[b][t / block_size].  k_scale / v_scale are ignored; a NULL
 *   or misaligned kv_scales returns PKV_ERR_INVALID_ARG.  A block id outside
 *   [0, num_blocks) reads zero codes and zero scales (as for bf16).
 * Every other field, the layouts and the return codes are those of
 * pkv_paged_decode_attn.  `p` is read during the call only.
 */
typedef struct pkv_attn_params {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int num_seqs;
    int q_len;
    int n_q;
    int n_kv;
    int head_dim;
    int block_size;
    int max_blocks_per_seq;
    int num_blocks;
    float scale;
    void *out;
    int out_dtype;
    void *workspace;
    size_t workspace_bytes;
    unsigned flags;
    int window;
    int kv_dtype;
    const float *k_scale;
    const float *v_scale;
    const float *kv_scales; /* PKV_KV_FP8_E4M3_BLOCK only */
} pkv_attn_params;

int pkv_paged_decode_attn_ex(const pkv_attn_params *p, void *stream);

/*
 * Bytes of workspace pkv_paged_decode_attn needs for these sizes on the
 * current device (the split-K partials of at most two pieces per CTA plus
 * an error word).  max_context_len is accepted for interface stability and
 * does not change the result.  Returns 0 for arguments the call would reject.
 */
size_t pkv_paged_decode_attn_workspace_size(int num_seqs, int q_len, int n_q, int n_kv,
                                            int head_dim, int block_size,
                                            int max_context_len, unsigned flags);

/*
 * pkv_paged_decode_attn_noalloc -- pkv_paged_decode_attn without a caller workspace.
 *
 * The pages have no counterpart to this entry point.  It is for callers that
 * cannot allocate device memory at all: a plugin inside another inference
 * engine whose per-step hook must not allocate, a process whose device memory
 * is reserved up front by some other pool, or a latency-critical loop that
 * must never reach cudaMalloc / cudaFree (which can synchronise the device).
 *
 * Arguments and results are those of pkv_paged_decode_attn minus the
 * workspace: the split-K records live in a scratch array of 24 MiB that the
 * library holds in the device memory of every GPU that loads it, until the
 * process exits.  The call allocates nothing.
 *   - Sizes whose workspace would exceed 24 MiB return PKV_ERR_WORKSPACE
 *     (every supported shape fits at up to 180 SMs; a forced CTA count in
 *     `flags` can exceed it).
 *   - PKV_FLAG_CHECKED and PKV_FLAG_TEST_STALL return PKV_ERR_UNSUPPORTED:
 *     device-side reports would land in the scratch array, which the caller
 *     cannot read.  For the same reason an expired in-kernel wait is not
 *     reported by this call.
 *   - The first call on a device looks up the scratch array's device address
 *     (with that device current); make that first call before any stream
 *     capture on the device.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that may overlap
 *     on the GPU -- different streams, or different host threads -- race on
 *     it: issue them on one stream.
 */
int pkv_paged_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                                  int block_size, int max_blocks_per_seq, int num_blocks,
                                  float scale, void *out, int out_dtype, unsigned flags,
                                  void *stream);

/*
 * pkv_kv_append -- write this step's new keys and values into the paged cache.
 *
 * For every token i < num_tokens with 0 <= slot_mapping[i] < num_blocks * block_size:
 *   k_cache[slot / block_size][g][slot % block_size][:] = k_new[i][g][:]   for all g < n_kv
 *   (v_cache likewise).  The copy is bit-exact; every other cache byte is unchanged.
 * Slots outside that range (e.g. -1 for padding tokens) are skipped.
 * ("Transformer inference mechanics", What the KV cache stores per layer:
 * the cache gains the new token's K/V each step.)
 * Layouts: k_new, v_new [num_tokens][n_kv][head_dim] bf16; slot_mapping
 *   [num_tokens] int32; caches as for pkv_paged_decode_attn.  head_dim must be
 *   a multiple of 8.  Two tokens naming the same slot leave either one's row.
 * flags: reserved, pass 0.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_CUDA; num_tokens == 0 launches nothing.
 */
int pkv_kv_append(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                  int num_tokens, int n_kv, int head_dim, int block_size, int num_blocks,
                  void *k_cache, void *v_cache, unsigned flags, void *stream);

/*
 * pkv_kv_append_fp8 -- pkv_kv_append into an 8-bit (e4m3) cache.
 *
 * For every valid slot (as in pkv_kv_append) and KV head g, element e of the
 * new key row is stored as the e4m3 code nearest to k_new[i][g][e] /
 * k_scale[g]: the quotient is rounded to fp32 (IEEE division), then to e4m3
 * with ties to the even code; quotients beyond +-448 (and infinities) store
 * +-448, NaN stores 0x7F.  V likewise with v_scale.  Quantise through a
 * scale: "Efficient inference", Quantization: fewer bytes per weight.
 * k_scale, v_scale: DEVICE fp32 [n_kv]; kv_cache: the interleaved 8-bit cache
 *   [num_blocks][n_kv][2][block_size][head_dim] bytes (K rows at [..][0], V
 *   rows at [..][1]), 16-byte aligned; k_new, v_new as for pkv_kv_append.
 * flags: reserved, pass 0.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_CUDA; num_tokens == 0 launches nothing.
 */
int pkv_kv_append_fp8(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                      int num_tokens, int n_kv, int head_dim, int block_size, int num_blocks,
                      const float *k_scale, const float *v_scale, void *kv_cache,
                      unsigned flags, void *stream);

/*
 * pkv_kv_append_fp8_block -- quantising append into an 8-bit (e4m3) cache
 * whose scales are per (block, KV head) (PKV_KV_FP8_E4M3_BLOCK).
 *
 * Quantise through a scale ("Efficient inference", Quantization: fewer bytes
 * per weight; CS336 lecture-10 notes, Quantization & pruning: bf16 -> fp8),
 * with the scale kept per block so that it follows the data.  For every
 * block B that receives tokens in this call and every KV head, for K and V
 * separately:
 *   - the run = the call's tokens whose slots fall in B, o_min their lowest
 *     offset; rows below o_min are the block's resident rows;
 *   - s_old = the stored scale if o_min > 0, else 0 (a block written from
 *     offset 0 starts over); scale 0 means "nothing but zeros so far";
 *   - a = the largest finite |x| of the run's new rows;
 *   - s_new = s_old if a == 0, else the larger of s_old and 2^e, the smallest
 *     power of two (e >= -126) with a <= 448 * 2^e, so no new value saturates;
 *   - if s_new > s_old > 0 the resident rows are re-quantised: code c becomes
 *     the e4m3 nearest to fp32(fp32(value(c) * s_old) / s_new) -- exact, the
 *     ratio being a power of two, except where a value falls below the
 *     normal e4m3 range (2^-6 * s_new);
 *   - each new row stores the e4m3 nearest to fp32(x / s_new) (ties to even;
 *     NaN stores 0x7F, infinities +-448; with s_new == 0 every value is 0 or
 *     non-finite and stores its own code); the scale entry becomes s_new and
 *     its two reserved words 0.
 * Precondition: the tokens that land in one block are consecutive entries of
 *   slot_mapping, ignoring skipped slots (as they are when each sequence's
 *   new tokens are listed together, in order).  Otherwise two parts of the
 *   call update the same block at once and its codes and scale are
 *   unspecified; nothing outside that block changes.  Two tokens naming the
 *   same slot leave the later one's row.
 * k_new, v_new [num_tokens][n_kv][head_dim] bf16 (head_dim a multiple of 8,
 *   at most 1024); slot_mapping [num_tokens] int32; kv_cache the interleaved
 *   cache [num_blocks][n_kv][2][block_size][head_dim] (16-byte aligned);
 *   kv_scales [num_blocks][n_kv][4] fp32 (16-byte aligned), read and written.
 * A freshly allocated block needs no initialisation (its first token lands at
 *   offset 0).  flags: reserved, pass 0.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED (more than 2^31
 * rows or slots) or PKV_ERR_CUDA; num_tokens == 0 launches nothing.
 */
int pkv_kv_append_fp8_block(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                            int num_tokens, int n_kv, int head_dim, int block_size,
                            int num_blocks, void *kv_cache, float *kv_scales, unsigned flags,
                            void *stream);

/*
 * pkv_copy_blocks -- copy whole physical blocks (every KV head, K and V).
 *
 * For each pair p < num_pairs: block pairs[2p+1] of k_cache and of v_cache
 * becomes a bit copy of block pairs[2p].  This is the copy half of
 * copy-on-write: a block shared by several sequences (a common prefix) is
 * duplicated before one of them writes into it ("Inference Engines", The
 * Breakthrough, PagedAttention paragraph; CS336 lecture-10 notes,
 * PagedAttention (vLLM): copy-on-write at the block level).
 * pairs: device int32 [num_pairs][2]; pairs with an id outside
 *   [0, num_blocks) or with src == dst are skipped.  A destination must not
 *   also be a source in the same call.
 * Caches as for pkv_paged_decode_attn (head_dim a multiple of 8); with
 * PKV_FLAG_KV_FP8 in flags, k_cache is the interleaved 8-bit cache (each
 * block holds K and V) and v_cache must be NULL -- or, with
 * PKV_FLAG_KV_BLOCK_SCALES as well, the cache's [num_blocks][n_kv][4] fp32
 * scale tensor (16-byte aligned), whose entries are copied with the blocks.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_CUDA; num_pairs == 0 launches nothing.
 */
int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int num_pairs,
                    int num_blocks, int n_kv, int head_dim, int block_size, unsigned flags,
                    void *stream);

/*
 * Block pool -- host-side allocator of physical blocks with reference counts
 * (on-demand allocation, prefix sharing, copy-on-write: "Transformer inference
 * mechanics", FlashAttention versus PagedAttention; "Inference Engines", The
 * Breakthrough).  Pure host bookkeeping: it never touches device memory.
 * Every call either succeeds completely or changes nothing.  A pool is not
 * thread-safe: callers serialise access.
 */
typedef struct pkv_block_pool pkv_block_pool;

/* All num_blocks blocks free (reference count 0).  NULL on bad sizes or no memory. */
pkv_block_pool *pkv_pool_create(int num_blocks, int block_size);
void pkv_pool_destroy(pkv_block_pool *pool);
/* Free blocks, or -1 for a NULL pool. */
int pkv_pool_num_free(const pkv_block_pool *pool);
/* Reference count of a block (0 = free), or -1 for a bad pool or id. */
int pkv_pool_refcount(const pkv_block_pool *pool, int block);
/* Take n free blocks (reference count 1 each) into out_blocks[0..n).
 * PKV_ERR_OUT_OF_BLOCKS if fewer than n are free. */
int pkv_pool_alloc(pkv_block_pool *pool, int n, int32_t *out_blocks);
/* One more owner for each listed block (a forked sequence or a shared prefix);
 * every block must be in use. */
int pkv_pool_share(pkv_block_pool *pool, const int32_t *blocks, int n);
/* One owner fewer for each listed block; a block whose count reaches 0 is free
 * again.  Fails (changing nothing) if a count would go below 0. */
int pkv_pool_release(pkv_block_pool *pool, const int32_t *blocks, int n);
/*
 * Make room for n_new tokens at the end of one sequence.
 * table[0..*nblocks) is the sequence's block-table row (host memory, room for
 * max_blocks entries) and ctx its resident token count.  Every block that
 * will receive a new token is made exclusively owned: if it is shared, a
 * fresh block takes its place in the table, the pair (old, new) is appended
 * to copy_pairs (room for 2 * ceil(n_new / block_size + 1) ints) and the old
 * block loses this owner; blocks are appended to the table as needed and
 * *nblocks is updated.  slot_out[i] is the cache slot of new token i
 * (block * block_size + offset), ready for pkv_kv_append; *num_pairs is the
 * number of copies to make with pkv_copy_blocks before appending.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_OUT_OF_BLOCKS.
 */
int pkv_pool_append_slots(pkv_block_pool *pool, int32_t *table, int *nblocks, int max_blocks,
                          int ctx, int n_new, int32_t *slot_out, int32_t *copy_pairs,
                          int *num_pairs);

/*
 * Synchronise `stream`, read and clear the error word of `workspace`.
 * Returns PKV_OK, PKV_ERR_BAD_BLOCK_TABLE (CHECKED mode saw a bad block id or
 * context length), PKV_ERR_TIMEOUT (a bounded wait inside the kernel expired;
 * that call's output is not valid), PKV_ERR_INVALID_ARG (null workspace) or
 * PKV_ERR_CUDA.  Not usable inside CUDA-graph capture (it synchronises).
 */
int pkv_check_error(const void *workspace, void *stream);

/*
 * KV-cache bytes M_kv = 2 * layers * n_kv * head_dim * tokens * elem_bytes
 * ("Inference Engines", The Mathematics; "Efficient inference", Key ideas),
 * where tokens = sequence length x batch.  Returns -1 for a negative argument.
 */
int64_t pkv_kv_bytes(int layers, int n_kv, int head_dim, int elem_bytes, int64_t tokens);

/* Static, human-readable name of a pkv_status value. */
const char *pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/*
 * Diagnostics (not part of the attention path).
 *
 * pkv_read_stream -- read `bytes` of device memory at `buf` once, with 16-byte
 * vector loads from ctas_per_sm (1..4) CTAs of 512 threads per SM, and XOR
 * the data into the device word *sink.  Its rate is a practical read peak of
 * the device (a copy's rate counts reads and writes together), and reading
 * more than the L2 holds evicts everything the L2 held before.
 * buf 16-byte aligned, bytes a multiple of 16, sink 4-byte aligned.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_CUDA; bytes == 0 launches nothing.
 */
int pkv_read_stream(const void *buf, size_t bytes, unsigned *sink, int ctas_per_sm,
                    void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
