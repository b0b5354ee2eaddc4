// pkv_noalloc.cu -- paged decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attn needs a caller-provided workspace for the split-K
// records of long contexts.  Some callers have no way to provide one: an
// inference-engine plugin whose per-step hook is forbidden to allocate, a
// process whose device memory is handed out up front by another component's
// pool, or a latency-critical loop that must never hit cudaMalloc/cudaFree
// (both can synchronise the device).  For them this file owns a fixed scratch
// array in the library's own device memory and passes it as the workspace.
//
// The array lives in every GPU that loads the library until the process
// exits.  Its device address is looked up once per device (with that device
// current) by the first call made on that device; nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(24) << 20;  // 24 MiB
constexpr int kMaxDevices = 64;

// Device memory shared by every call on a device.  In host code this name is
// only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_scratch on the current device, looked up on first use.
int scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return PKV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode_attn_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
    int block_size, int max_blocks_per_seq, int num_blocks, float scale, void* out,
    int out_dtype, unsigned flags, void* stream) {
    // Device-side reports (CHECKED mode, an expired wait) land in the scratch
    // array, which this caller cannot read back.  Refuse CHECKED rather than
    // drop its reports, and refuse the test-only stall flag, whose only effect
    // here would be an invalid output with PKV_OK.
    if (flags & (PKV_FLAG_CHECKED | PKV_FLAG_TEST_STALL)) return PKV_ERR_UNSUPPORTED;
    // The one-tile form's need: a call whose paired form does not fit the
    // scratch runs in the one-tile form.
    const size_t need = pkv::attn_workspace_min_bytes(num_seqs, q_len, n_q, n_kv, head_dim,
                                                      block_size, flags);
    if (need == 0 || num_seqs == 0) {
        // Invalid shapes (or an empty batch): the regular entry point gives the
        // precise status and launches nothing.
        return pkv_paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                     q_len, n_q, n_kv, head_dim, block_size,
                                     max_blocks_per_seq, num_blocks, scale, out, out_dtype,
                                     nullptr, 0, flags, stream);
    }
    if (need > kScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the fixed 24 MiB
    void* scratch = nullptr;
    const int st = scratch_on_current_device(&scratch);
    if (st != PKV_OK) return st;
    // Nothing in the scratch has to start at zero: each call rewrites every
    // split record it later reads, and the error word is never read here.
    return pkv_paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                 q_len, n_q, n_kv, head_dim, block_size, max_blocks_per_seq,
                                 num_blocks, scale, out, out_dtype, scratch, kScratchBytes, flags,
                                 stream);
}
