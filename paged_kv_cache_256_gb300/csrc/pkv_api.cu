// pkv_api.cu -- the C ABI declared in include/pkv.h.
//
// Host side only: argument checks (no launch on failure), the tensor maps
// that let the TMA unit fetch (block, KV head) tiles of the caches, the
// workspace layout, and the launches.  The kernels live in decode_attn.cu,
// lse_merge.cu and kv_append.cu.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/pkv.h"
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kMaxDevices = 64;

int sm_count(int dev) {
    static int cache[kMaxDevices] = {0};
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a cache: rows = num_blocks * n_kv * block_size, columns =
// head_dim elements.  bf16: one box = 64 columns x block_size rows with the
// 128-byte swizzle.  e4m3 (kv8; one cache whose (block, head) tiles hold the
// K rows, then the V rows): one box = a whole row of head_dim bytes x
// block_size rows, 128-byte swizzle at head_dim 128, 64-byte at 64.
bool make_cache_map(CUtensorMap* map, const void* base, int head_dim, long long rows,
                    int block_size, bool kv8) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * (kv8 ? 1 : 2)};
    // e4m3: one box covers a (block, head)'s K rows and the V rows after them
    cuuint32_t box[2] = {kv8 ? (cuuint32_t)head_dim : 64u,
                         (cuuint32_t)(kv8 ? 2 * block_size : block_size)};
    cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapSwizzle swz = (!kv8 || head_dim == 128) ? CU_TENSOR_MAP_SWIZZLE_128B
                                                             : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = fn(map, kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Grouped 4-D view of a bf16 cache with head_dim 128 for the tensor-memory
// consumer: {64 columns, 8 rows, 2 column halves, row groups of 8}, strides
// 256 (row), 128 (half) and 2048 (group) bytes.  One box of 64 x 8 x 2 x
// block_size/8 brings a whole (block, KV head) tile and lands it as
// [8-row group][half][8 rows][128 bytes], 128-byte swizzled: the 8-row groups
// of consecutive blocks then lie at one stride (2048 bytes) and the halves
// 1024 bytes apart, the K-major layout the N = 64 score product and the
// MN-major layout the PV product read -- one copy per tile where the 2-D view
// needs two.  The strides are not in increasing order (the half stride lies
// inside a row); a driver that declines such a view returns an error and the
// caller keeps the 2-D view.  rows is a multiple of 8 (block_size is).
bool make_cache_map_4d(CUtensorMap* map, const void* base, long long rows, int block_size) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64u, 8u, 2u, (cuuint64_t)(rows / 8)};
    cuuint64_t strides[3] = {256u, 128u, 2048u};
    cuuint32_t box[4] = {64u, 8u, 2u, (cuuint32_t)(block_size / 8)};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Encoding a tensor map is a driver call; decode loops pass the same caches
// every step, so the last few encodings are kept (keyed by everything that
// goes into them).
struct MapKey {
    const void* base;
    long long rows;
    int head_dim, block_size;
    bool kv8, grouped;
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kMapCache = 8;
std::mutex g_map_mutex;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool cached_cache_map(CUtensorMap* map, const void* base, int head_dim, long long rows,
                      int block_size, bool kv8, bool grouped = false) {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (const MapEntry& e : g_maps)
        if (e.used && e.key.base == base && e.key.rows == rows && e.key.head_dim == head_dim &&
            e.key.block_size == block_size && e.key.kv8 == kv8 && e.key.grouped == grouped) {
            *map = e.map;
            return true;
        }
    if (grouped ? !make_cache_map_4d(map, base, rows, block_size)
                : !make_cache_map(map, base, head_dim, rows, block_size, kv8))
        return false;
    MapEntry& e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.key = MapKey{base, rows, head_dim, block_size, kv8, grouped};
    e.map = *map;
    e.used = true;
    return true;
}

// 3-D view of the queries for the tensor-memory consumer: [tokens =
// num_seqs * q_len][n_q heads][head_dim] bf16, one box = 64 columns x by
// heads x bz tokens with the 128-byte swizzle, so a row tile lands as the
// K-major operand the score MMA reads (row r = token-major, head-minor).
bool make_q_map(CUtensorMap* map, const void* q, int head_dim, int n_q, long long tokens, int by,
                int bz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_q, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_q * head_dim * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)by, (cuuint32_t)bz};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct QMapKey {
    const void* q;
    long long tokens;
    int head_dim, n_q, by, bz;
};
struct QMapEntry {
    QMapKey key;
    CUtensorMap map;
    bool used;
};
QMapEntry g_qmaps[kMapCache];
int g_qmap_next = 0;

bool cached_q_map(CUtensorMap* map, const void* q, int head_dim, int n_q, long long tokens, int by,
                  int bz) {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (const QMapEntry& e : g_qmaps)
        if (e.used && e.key.q == q && e.key.tokens == tokens && e.key.head_dim == head_dim &&
            e.key.n_q == n_q && e.key.by == by && e.key.bz == bz) {
            *map = e.map;
            return true;
        }
    if (!make_q_map(map, q, head_dim, n_q, tokens, by, bz)) return false;
    QMapEntry& e = g_qmaps[g_qmap_next];
    g_qmap_next = (g_qmap_next + 1) % kMapCache;
    e.key = QMapKey{q, tokens, head_dim, n_q, by, bz};
    e.map = *map;
    e.used = true;
    return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kTileRows = 128;
constexpr int kMaxQLen = 1 << 16;
constexpr long long kMaxRowsTotal = 1LL << 24;

int warp_rows_for(int rows) {
    const int tiles = (rows + 15) / 16;
    return tiles <= 1 ? 1 : tiles <= 2 ? 2 : tiles <= 4 ? 4 : 8;
}

// Number of attention CTAs: forced by the flags, else one per SM.
int attn_grid(unsigned flags, int dev) {
    const int forced = (int)((flags >> PKV_FLAG_GRID_SHIFT) & 0xFFFFu);
    if (forced > 0) return forced;
    return sm_count(dev);
}

int check_shape(int num_seqs, int q_len, int n_q, int n_kv, int head_dim, int block_size) {
    if (num_seqs < 0 || q_len < 1 || n_q < 1 || n_kv < 1 || head_dim < 1 || block_size < 1)
        return PKV_ERR_INVALID_ARG;
    if (n_q % n_kv != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (q_len > kMaxQLen || (long long)(n_q / n_kv) * q_len > kMaxRowsTotal)
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// A unit's fixed work (query load, cross-warp combine, output) in blocks of
// streaming time: the weight the work partition gives each unit on top of
// its blocks.  Measured per consumer on GB300 with the L2 evicted before each
// call (ragged GQA, MQA verify and chunked-prefill batches; uniform contexts
// do not care): rows <= 8 -- 10 for bf16 (GQA 168.4 / 166.4 / 163.9 / 164.4 /
// 166.3 us at 6 / 8 / 10 / 12 / 16), 32 for 8-bit blocks, which stream in
// half the time while the unit's fixed work grows (Q widened to f16);
// 8 < rows <= 64 with an 8-bit cache -- 4 (every row-slice warp widens each
// tile, so blocks cost more); tensor-memory consumer -- 12 (the O read-out
// per unit and the pipeline fill; MQA verify 41.5 / 41.5 / 41.9 us at 10 /
// 12 / 16), 14 over an 8-bit cache, whose eight-stage ring streams blocks
// faster than its units' fixed work (MQA verify 49.7 / 47.6 / 49.7 / 51.7 us
// at 10 / 14 / 18 / 22, with block scales 55.8 / 53.8 / 55.8 / 57.8, chunked
// prefill 117.2 / 113.3 / 109.0 / 111.1).
// Per-block scales (fetched with the tiles by LSU copies) leave these weights
// as they are (8-bit GQA with block scales 100.4 us at 32, 104.3 at 24).
int unit_cost_for(int rows, bool kv8) {
    if (rows > 128) return 16;  // the paired tensor-memory form (bf16 only)
    if (rows <= 8) return kv8 ? 32 : 10;
    if (rows > 64) return kv8 ? 14 : 12;
    return kv8 ? 4 : 6;
}

// Query rows sharing one KV head are processed in tiles of at most 128,
// holding whole query tokens when a token's group of heads fits in a tile.
int tile_rows(int n_q, int n_kv, int q_len) {
    const int group = n_q / n_kv;
    const int rows_total = group * q_len;
    if (rows_total <= kTileRows) return rows_total;
    return group <= kTileRows ? (kTileRows / group) * group : kTileRows;
}

// Rows of the paired tensor-memory form: two tiles per unit when a KV head
// has more than one tile of more than 64 rows; else the one-tile rows.
int paired_rows(int n_q, int n_kv, int q_len) {
    const int rows = tile_rows(n_q, n_kv, q_len);
    return (rows > 64 && (n_q / n_kv) * q_len > rows) ? 2 * rows : rows;
}

// A tile as one TMA box of the query map (by heads x bz tokens): whole
// tokens of `group` heads, or part of one token's heads when a token's
// group spans several tiles.  0 when a tile cannot be one box.
bool q_box(int group, int rows, int* by, int* bz) {
    if (rows % group == 0) {
        *by = group;
        *bz = rows / group;
    } else if (group % rows == 0) {
        *by = rows;
        *bz = 1;
    } else {
        return false;
    }
    return *by <= 256 && *bz <= 256;
}

}  // namespace

WorkspaceLayout workspace_layout(int grid, int rows, int head_dim) {
    WorkspaceLayout L;
    L.err_off = 0;
    L.info_off = 256;
    L.ml_off = round_up(L.info_off + (size_t)grid * 2 * sizeof(int4), 256);
    L.o_off = round_up(L.ml_off + (size_t)grid * 2 * rows * 2 * sizeof(float), 256);
    L.total = round_up(L.o_off + (size_t)grid * 2 * rows * head_dim * sizeof(float), 256);
    return L;
}

}  // namespace pkv

using namespace pkv;

namespace pkv {
size_t attn_workspace_min_bytes(int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                                int block_size, unsigned flags) {
    if (check_shape(num_seqs, q_len, n_q, n_kv, head_dim, block_size) != PKV_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int grid = attn_grid(flags, dev);
    if (grid <= 0) return 0;
    return workspace_layout(grid, tile_rows(n_q, n_kv, q_len), head_dim).total;
}
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 10200; }

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_BAD_BLOCK_TABLE: return "PKV_ERR_BAD_BLOCK_TABLE";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
        case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
        default: return "PKV_ERR_UNKNOWN";
    }
}

int64_t pkv_kv_bytes(int layers, int n_kv, int head_dim, int elem_bytes, int64_t tokens) {
    if (layers < 0 || n_kv < 0 || head_dim < 0 || elem_bytes < 0 || tokens < 0) return -1;
    return (int64_t)2 * layers * n_kv * head_dim * elem_bytes * tokens;
}

size_t pkv_paged_decode_attn_workspace_size(int num_seqs, int q_len, int n_q, int n_kv,
                                            int head_dim, int block_size, int max_context_len,
                                            unsigned flags) {
    (void)max_context_len;
    if (check_shape(num_seqs, q_len, n_q, n_kv, head_dim, block_size) != PKV_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int grid = attn_grid(flags, dev);
    if (grid <= 0) return 0;
    // sized for the larger tiling the call may choose (the paired form)
    return workspace_layout(grid, paired_rows(n_q, n_kv, q_len), head_dim).total;
}


int pkv_paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          int num_seqs, int q_len, int n_q, int n_kv, int head_dim,
                          int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                          void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                          unsigned flags, void* stream) {
    pkv_attn_params p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.q_len = q_len;
    p.n_q = n_q;
    p.n_kv = n_kv;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.scale = scale;
    p.out = out;
    p.out_dtype = out_dtype;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    p.flags = flags;
    p.window = 0;
    p.kv_dtype = PKV_KV_BF16;
    return pkv_paged_decode_attn_ex(&p, stream);
}

int pkv_paged_decode_attn_ex(const pkv_attn_params* p, void* stream) {
    if (!p) return PKV_ERR_INVALID_ARG;
    const void *q = p->q, *k_cache = p->k_cache, *v_cache = p->v_cache;
    const int32_t *block_tables = p->block_tables, *context_lens = p->context_lens;
    const int num_seqs = p->num_seqs, q_len = p->q_len, n_q = p->n_q, n_kv = p->n_kv;
    const int head_dim = p->head_dim, block_size = p->block_size;
    const int max_blocks_per_seq = p->max_blocks_per_seq, num_blocks = p->num_blocks;
    const float scale = p->scale;
    void* out = p->out;
    const int out_dtype = p->out_dtype;
    void* workspace = p->workspace;
    const size_t workspace_bytes = p->workspace_bytes;
    const unsigned flags = p->flags;
    int st = check_shape(num_seqs, q_len, n_q, n_kv, head_dim, block_size);
    if (st != PKV_OK) return st;
    if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32) return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (p->window < 0) return PKV_ERR_INVALID_ARG;
    if (p->kv_dtype != PKV_KV_BF16 && p->kv_dtype != PKV_KV_FP8_E4M3 &&
        p->kv_dtype != PKV_KV_FP8_E4M3_BLOCK)
        return PKV_ERR_INVALID_ARG;
    const bool blk = p->kv_dtype == PKV_KV_FP8_E4M3_BLOCK;
    const bool kv8 = p->kv_dtype == PKV_KV_FP8_E4M3 || blk;
    if (num_seqs == 0) return PKV_OK;
    if (kv8 && !blk &&
        (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 4) || !aligned(p->v_scale, 4)))
        return PKV_ERR_INVALID_ARG;
    if (blk && (!p->kv_scales || !aligned(p->kv_scales, 16))) return PKV_ERR_INVALID_ARG;
    // An 8-bit cache is one interleaved tensor, passed as k_cache; v_cache is NULL.
    if (kv8 ? v_cache != nullptr : v_cache == nullptr) return PKV_ERR_INVALID_ARG;
    if (!q || !k_cache || !block_tables || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || (!kv8 && !aligned(v_cache, 16)) ||
        !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    const long long rows_total = (long long)num_blocks * n_kv * (kv8 ? 2 : 1) * block_size;
    if (rows_total >= (1LL << 31) - 64) return PKV_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * block_size >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int grid0 = attn_grid(flags, dev);
    if (grid0 <= 0) return PKV_ERR_CUDA;
    // Query rows per unit: one tile of at most 128 rows, or over a bf16 cache
    // with bf16 output two such tiles (the paired tensor-memory form, which
    // reads each stage once for both) when the workspace holds their records.
    const int q_rows_total = (n_q / n_kv) * q_len;
    const int rows1 = tile_rows(n_q, n_kv, q_len);
    const int rows2 = paired_rows(n_q, n_kv, q_len);
    const bool pair_ok = rows2 > rows1 && !kv8 && out_dtype == PKV_OUT_BF16 &&
                         !(flags & PKV_FLAG_ONE_TILE);
    int rows = rows1, q_tiles = 1, grid = grid0;
    WorkspaceLayout L;
    for (int attempt = pair_ok ? 0 : 1; attempt < 2; ++attempt) {
        rows = attempt == 0 ? rows2 : rows1;
        q_tiles = (q_rows_total + rows - 1) / rows;
        grid = grid0;
        // No more CTAs than (unit, block) items the call can have.
        if (((flags >> PKV_FLAG_GRID_SHIFT) & 0xFFFFu) == 0) {
            const long long items = (long long)num_seqs * n_kv * q_tiles * max_blocks_per_seq;
            if (items < grid) grid = (int)items;
        }
        L = workspace_layout(grid, rows, head_dim);
        if (workspace && workspace_bytes >= L.total) break;
    }
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;

    AttnMaps maps;
    std::memset(&maps, 0, sizeof maps);
    // The tensor-memory consumer over a bf16 head_dim-128 cache takes each K
    // and V tile in one copy through the grouped 4-D views where the CUDA driver
    // accepts them; everything else reads through the 2-D views.
    int tile_4d = 0;
    if (!kv8 && head_dim == 128 && rows > 64 && !(flags & PKV_FLAG_TILE_2D) &&
        cached_cache_map(&maps.k, k_cache, head_dim, rows_total, block_size, false, true) &&
        cached_cache_map(&maps.v, v_cache, head_dim, rows_total, block_size, false, true))
        tile_4d = 1;
    if (!tile_4d &&
        (!cached_cache_map(&maps.k, k_cache, head_dim, rows_total, block_size, kv8) ||
         !cached_cache_map(&maps.v, kv8 ? k_cache : v_cache, head_dim, rows_total, block_size,
                           kv8)))
        return PKV_ERR_CUDA;
    // The tensor-memory consumer (more than 64 rows) over a bf16 cache takes
    // its query tiles by TMA when a tile is one box; otherwise its threads
    // load them.  (Over an 8-bit cache its threads store their query rows,
    // widened to f16, into tensor memory.)
    int q_tma = 0, by = 0, bz = 0;
    if (rows > 64 && !kv8 && (long long)num_seqs * q_len < (1LL << 31) &&
        q_box(n_q / n_kv, rows, &by, &bz)) {
        if (!cached_q_map(&maps.q, q, head_dim, n_q, (long long)num_seqs * q_len, by, bz))
            return PKV_ERR_CUDA;
        q_tma = 1;
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    AttnArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.err = reinterpret_cast<unsigned*>(ws + L.err_off);
    a.rec_info = reinterpret_cast<int4*>(ws + L.info_off);
    a.rec_ml = reinterpret_cast<float*>(ws + L.ml_off);
    a.rec_o = reinterpret_cast<float*>(ws + L.o_off);
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.group = n_q / n_kv;
    a.rows = rows;
    a.rows_total = q_rows_total;
    a.q_tiles = q_tiles;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.tile_rows_total = (int)rows_total;
    a.kv_mul = kv8 ? 2 : 1;
    a.v_row_off = kv8 ? block_size : 0;
    a.warp_rows = warp_rows_for(rows);
    a.unit_cost = unit_cost_for(rows, kv8);
    a.k_scale = (kv8 && !blk) ? p->k_scale : nullptr;
    a.v_scale = (kv8 && !blk) ? p->v_scale : nullptr;
    a.kv_scales = blk ? p->kv_scales : nullptr;
    // A window at least as wide as any context is no window.
    a.window = (long long)p->window >= (long long)max_blocks_per_seq * block_size ? 0 : p->window;
    a.checked = (flags & PKV_FLAG_CHECKED) ? 1 : 0;
    a.test_stall = (flags & PKV_FLAG_TEST_STALL) ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.q_tma = q_tma;
    a.early_start = (flags & PKV_FLAG_NO_EARLY_START) ? 0 : 1;
    a.tile_4d = tile_4d;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = out_dtype == PKV_OUT_F32;
    const cudaError_t le =
        blk   ? launch_decode_attn_fp8_block(a, maps, head_dim, block_size, f32, grid, s)
        : kv8 ? launch_decode_attn_fp8(a, maps, head_dim, block_size, f32, grid, s)
              : launch_decode_attn(a, maps, head_dim, block_size, f32, grid, s);
    if (le != cudaSuccess) return PKV_ERR_CUDA;
    if (grid > 1 && launch_lse_merge(a, head_dim, f32, grid, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int pkv_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                  int num_tokens, int n_kv, int head_dim, int block_size, int num_blocks,
                  void* k_cache, void* v_cache, unsigned flags, void* stream) {
    (void)flags;
    if (num_tokens < 0 || n_kv < 1 || head_dim < 8 || head_dim % 8 != 0 || block_size < 1 ||
        num_blocks < 1)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 4))
        return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return PKV_ERR_CUDA;
    if (launch_kv_append(k_new, v_new, slot_mapping, num_tokens, n_kv, head_dim, block_size,
                         num_blocks, k_cache, v_cache, sms,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int pkv_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                      int num_tokens, int n_kv, int head_dim, int block_size, int num_blocks,
                      const float* k_scale, const float* v_scale, void* kv_cache,
                      unsigned flags, void* stream) {
    (void)flags;
    if (num_tokens < 0 || n_kv < 1 || head_dim < 8 || head_dim % 8 != 0 || block_size < 1 ||
        num_blocks < 1)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_cache || !k_scale || !v_scale)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return PKV_ERR_CUDA;
    if (launch_kv_append_fp8(k_new, v_new, slot_mapping, num_tokens, n_kv, head_dim, block_size,
                             num_blocks, k_scale, v_scale, kv_cache, sms,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int pkv_kv_append_fp8_block(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                            int num_tokens, int n_kv, int head_dim, int block_size,
                            int num_blocks, void* kv_cache, float* kv_scales, unsigned flags,
                            void* stream) {
    (void)flags;
    if (num_tokens < 0 || n_kv < 1 || head_dim < 8 || head_dim % 8 != 0 || head_dim > 1024 ||
        block_size < 1 || num_blocks < 1)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_cache || !kv_scales) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 4) || !aligned(kv_scales, 16))
        return PKV_ERR_INVALID_ARG;
    if ((long long)num_tokens * n_kv >= (1LL << 31) ||
        (long long)num_blocks * block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;
    if (launch_kv_append_fp8_block(k_new, v_new, slot_mapping, num_tokens, n_kv, head_dim,
                                   block_size, num_blocks, kv_cache, kv_scales,
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                    int num_blocks, int n_kv, int head_dim, int block_size, unsigned flags,
                    void* stream) {
    // An 8-bit cache is one tensor whose blocks hold K and V (1 byte each): a
    // block is as many bytes as a bf16 K block, and there is no V pointer;
    // with per-block scales, v_cache is the scale tensor, copied with the blocks.
    const bool kv8 = (flags & PKV_FLAG_KV_FP8) != 0;
    const bool blk = (flags & PKV_FLAG_KV_BLOCK_SCALES) != 0;
    if (blk && !kv8) return PKV_ERR_INVALID_ARG;
    if (num_pairs < 0 || num_blocks < 1 || n_kv < 1 || head_dim < 8 || head_dim % 8 != 0 ||
        block_size < 1 || ((long long)n_kv * block_size * head_dim * 2) % 16 != 0)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !pairs || ((kv8 && !blk) ? v_cache != nullptr : v_cache == nullptr))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || (v_cache && !aligned(v_cache, 16)) || !aligned(pairs, 4))
        return PKV_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return PKV_ERR_CUDA;
    if (launch_copy_blocks(k_cache, kv8 ? nullptr : v_cache, pairs, num_pairs, num_blocks, n_kv,
                           head_dim, block_size, 2, blk ? v_cache : nullptr, sms,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int pkv_check_error(const void* workspace, void* stream) {
    if (!workspace) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (word == 0) return PKV_OK;
    if (cudaMemset(const_cast<void*>(workspace), 0, sizeof word) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (word & kErrTimeout) return PKV_ERR_TIMEOUT;
    if (word & (kErrBadBlock | kErrBadContext)) return PKV_ERR_BAD_BLOCK_TABLE;
    return PKV_ERR_CUDA;
}

}  // extern "C"
