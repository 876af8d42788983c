// api.cu -- the extern "C" entry points declared in include/pagedkv.h.
//
// Responsibilities: argument validation (before anything is enqueued), the
// split-KV partition plan, workspace carving, TMA tensor-map encoding and the
// kernel launches on the caller's stream.  No allocation, no synchronisation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/pagedkv.h"
#include "launch.h"

namespace {

using pkv::kBlockSize;
using pkv::kHeadDim;

constexpr int kMaxDevices = 64;
constexpr int kMinPartBlocks = 16;      // automatic plans never go below 256 tokens per partition
constexpr int kDefaultPartBlocks = 64;  // 1024 tokens
constexpr int kMaxAutoParts = 32;       // automatic bf16 decode plans: at most 32 partitions per sequence
constexpr int kDecodeCtasPerSm = 3;     // resident decode CTAs per SM (64 KB of shared memory each)
constexpr int kDecodeFp8CtasPerSm = 4;  // resident FP8 decode CTAs per SM (52 KB each, 128 registers)
constexpr size_t kStatusBytes = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- per-device caches -----------------------------------------------------------
std::atomic<int> g_sm_count[kMaxDevices];
std::once_flag g_decode_prepared[kMaxDevices];
std::once_flag g_prefill_prepared[kMaxDevices];
std::once_flag g_decode_fp8_prepared[kMaxDevices];
cudaError_t g_decode_prep_err[kMaxDevices];
cudaError_t g_decode_fp8_prep_err[kMaxDevices];
cudaError_t g_prefill_prep_err[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int sm_count(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ---- tensor maps -------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Pool tensor [num_blocks][n_kv][16][128] bf16 viewed as 4-D (dims inner->outer:
// head_dim, slot, head, block); box = 64 dims x 16 slots, 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const void *base, int32_t num_blocks, int32_t n_kv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kBlockSize),
                                static_cast<cuuint64_t>(n_kv), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                   static_cast<cuuint64_t>(kHeadDim) * 2 * kBlockSize,
                                   static_cast<cuuint64_t>(kHeadDim) * 2 * kBlockSize * n_kv};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kBlockSize), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An FP8 pool [num_blocks][n_kv][16][128] of one-byte codes viewed as 4-D; one box
// = a whole 2 KB (block, head) tile (128 codes = 128 bytes x 16 slots), 128-byte swizzle.
bool encode_pool_map_fp8(CUtensorMap *map, const void *base, int32_t num_blocks, int32_t n_kv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kBlockSize),
                                static_cast<cuuint64_t>(n_kv), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kHeadDim) * kBlockSize,
                                   static_cast<cuuint64_t>(kHeadDim) * kBlockSize * n_kv};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kBlockSize), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same pool viewed as 5-D so that ONE box is a whole 4 KB (block, head) tile
// in the order the tensor core wants it: dims inner->outer are 64 dims (128 B),
// 8 slots (stride 256 B), the two 64-dim halves (stride 128 B), the two 8-slot
// groups (stride 2 KB) and the (block, head) tile index block * n_kv + head
// (stride 4 KB).  The box (64, 8, 2, 2, 1) lands in shared memory as
// [slot group][dim half][8 slots][128 B], i.e. four 1 KB swizzle atoms.
bool encode_pool_tile_map(CUtensorMap *map, const void *base, int32_t num_blocks, int32_t n_kv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t tiles = static_cast<uint64_t>(num_blocks) * static_cast<uint64_t>(n_kv);
    if (tiles > static_cast<uint64_t>(INT32_MAX)) return false;  // tile index is a 32-bit coordinate
    const cuuint64_t dims[5] = {64, 8, 2, 2, static_cast<cuuint64_t>(tiles)};
    const cuuint64_t strides[4] = {256, 128, 2048, 4096};
    const cuuint32_t box[5] = {64, 8, 2, 2, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row tensor [rows][n_q][128] (the chunk's q, bf16, or its output, bf16 or fp32)
// viewed as 3-D (head_dim, head, row); box = 128 bytes of dims (bf16: 64, fp32:
// 32) x G heads x (128 / G) rows, 128-byte swizzle: one box is 128 tile rows of
// 128 bytes ordered (row, head), the layout of the Q tile and of a staged
// output tile.
bool encode_rows_map(CUtensorMap *map, const void *base, int32_t rows, int32_t n_q, int32_t group, bool fp32) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = fp32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(n_q),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * es, static_cast<cuuint64_t>(kHeadDim) * es * n_q};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(group),
                               static_cast<cuuint32_t>(128 / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- validation helpers -------------------------------------------------------------
int check_cache(const pkv_cache_desc *c) {
    if (!c) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks < 1 || c->num_kv_heads < 1) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize || c->head_dim != kHeadDim || c->dtype != PKV_DTYPE_BF16)
        return PKV_ERR_UNSUPPORTED;
    // The pool's byte size must stay addressable by the kernels' 64-bit index math
    // and by the 32-bit block coordinate of the tensor map.
    return PKV_OK;
}

// A pool of FP8 (E4M3) codes, for the *_fp8 entry points.
int check_cache_fp8(const pkv_cache_desc *c) {
    if (!c) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks < 1 || c->num_kv_heads < 1) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlockSize || c->head_dim != kHeadDim || c->dtype != PKV_DTYPE_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int check_group(int32_t n_q, int32_t n_kv) {
    if (n_q < 1 || n_q % n_kv != 0) return PKV_ERR_INVALID_ARG;
    const int32_t G = n_q / n_kv;
    if (G > 8 && G % 8 != 0) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// ---- decode plan -----------------------------------------------------------------------
// Workspace layout: [status word | part_m | part_l | part_o], each region
// 256-byte aligned; only the status word when nothing is split.
struct DecodePlan {
    int32_t part_blocks;
    int32_t max_parts;
    size_t off_m, off_l, off_o, total;
};

// rows_per_seq: query rows per sequence (1 for decode, q_per_seq for verify).
DecodePlan plan_decode(int32_t num_seqs, int32_t n_q, int32_t max_blocks, int32_t part_blocks,
                       int32_t rows_per_seq = 1) {
    DecodePlan pl{};
    pl.part_blocks = part_blocks >= max_blocks ? max_blocks : part_blocks;
    pl.max_parts = (max_blocks + pl.part_blocks - 1) / pl.part_blocks;
    if (pl.max_parts <= 1) {
        pl.off_m = pl.off_l = pl.off_o = pl.total = kStatusBytes;
        return pl;
    }
    const size_t rows = static_cast<size_t>(num_seqs) * rows_per_seq * n_q * pl.max_parts;
    pl.off_m = kStatusBytes;
    pl.off_l = pl.off_m + align_up(rows * 4, 256);
    pl.off_o = pl.off_l + align_up(rows * 4, 256);
    pl.total = pl.off_o + align_up(rows * kHeadDim * 4, 256);
    return pl;
}

int32_t auto_part_blocks(int32_t num_seqs, int32_t n_kv, int32_t head_splits, int32_t max_blocks, int sms,
                         bool cap_parts, bool fp8 = false, bool window_span = false) {
    // Partitions of 1024 tokens (measured best on ragged 8B-shaped batches and
    // 70B-shaped B=8 long contexts) keep CTAs uniform and the merge small; a
    // context that fits one partition is not split.  Three refinements, each
    // measured on a GB300 (decode call, L2 flushed):
    //  (a) contexts of at most two default partitions whose unsplit grid already
    //      covers every SM within one wave of resident CTAs are not split at all:
    //      a second, ragged wave and the merge cost more than the split gains
    //      (B=32 x 2048 tokens, 8 KV heads: 47.8 us unsplit vs 58.0 us);
    //  (b) for the bf16 decode (cap_parts), at most 32 partitions per sequence,
    //      since the merge folds a row's partitions in sequence (B=1 x 128K
    //      tokens: 90.8 us with 4096-token partitions vs 103.1 us with 1024);
    //      the FP8 decode and verify, bound by instruction issue, keep the finer
    //      split (B=1 x 128K: 69.8 vs 73.3 us and 176 vs 184 us);
    //  (c) when few (sequence, head) units exist the partitions shrink (not below
    //      256 tokens, nor below (b)'s floor) until the grid covers every SM twice.
    const int64_t units = static_cast<int64_t>(num_seqs) * n_kv * head_splits;
    const int64_t nsm = sms > 0 ? sms : 148;
    // (e) a sliding window that bounds every long sequence's span (window_span: the
    //     span, W / 16 + 1 blocks, is shorter than the table) gives CTAs of about
    //     equal length, so splitting buys no balance, and the default partition
    //     leaves a one-block tail partition (W = 1024: 64 + 1 blocks): spans up to 4
    //     default partitions are not split when the units cover every SM (8B-shaped
    //     B=64, back to back: W = 1024, 47.1 vs 52.1 us; W = 1536, 60.2 vs 62.1;
    //     W = 2048, 69.6 vs 72.0; W = 3000, 84.3 vs 85.9; MHA B=32 x 2048: W = 1024,
    //     79.1 vs 81.8; W = 1536, 115.5 vs 118.5).
    if (window_span && units >= nsm && max_blocks <= 4 * kDefaultPartBlocks) return max_blocks;
    if (fp8) {
        // The FP8 decode moves half the bytes per CTA, so it prefers fewer, longer
        // CTAs (back-to-back decode calls, GB300): contexts of at most 2048 tokens
        // whose units fill every SM are not split (MHA B=32 x 2048: 94.8 us vs
        // 101.3 us with 1024-token partitions), and contexts of 16K tokens and more
        // double the partition while at least 3 CTAs per SM remain (B=8 x 32K:
        // 4096-token partitions, 108.4 vs 113.3 us; B=1 x 128K: 2048-token, 62.7 vs
        // 72.3 us).  Ragged batches of shorter contexts keep 1024-token partitions
        // (8B-shaped B=64: 68.5 us; 2048-token partitions: 80.5 us).
        if (max_blocks <= 2 * kDefaultPartBlocks && units >= nsm) return std::max(max_blocks, kMinPartBlocks);
        if (max_blocks >= 16 * kDefaultPartBlocks) {
            int32_t pb = kDefaultPartBlocks;
            while (units * ((max_blocks + 2 * pb - 1) / (2 * pb)) >= kDecodeCtasPerSm * nsm) pb *= 2;
            return pb;
        }
    }
    if (max_blocks <= 2 * kDefaultPartBlocks && units >= nsm && units <= nsm * kDecodeCtasPerSm)
        return std::max(max_blocks, kMinPartBlocks);  // (a)
    int32_t floor_pb = kMinPartBlocks;  // (b)
    while (cap_parts && floor_pb < max_blocks && (max_blocks + floor_pb - 1) / floor_pb > kMaxAutoParts)
        floor_pb *= 2;
    int32_t pb = std::max(kDefaultPartBlocks, floor_pb);
    const int64_t want = nsm * 2;  // (c)
    while (pb > floor_pb && units * ((max_blocks + pb - 1) / pb) < want) pb /= 2;
    pb = std::max(pb, floor_pb);
    // (d) a grid a little over one wave of resident CTAs (its second wave a few
    //     CTAs) takes instead the most partitions that fit in one wave, when those
    //     still give every SM a CTA (MQA-shaped B=32 x 2048, 32 query heads over one
    //     KV head, L2 flushed: 3 partitions of 688 tokens, 23.2 us, against 4 of 512,
    //     29.3 us, and 4 of 768 or 1024, 25.2 us).
    const int64_t slots = nsm * (fp8 ? kDecodeFp8CtasPerSm : kDecodeCtasPerSm);
    const int64_t parts = (max_blocks + pb - 1) / pb;
    if (units * parts > slots && units * parts < 2 * slots) {
        const int64_t fit = slots / units;
        if (fit >= 1 && units * fit >= nsm) {
            const int32_t pb1 = static_cast<int32_t>((max_blocks + fit - 1) / fit);
            if (pb1 >= floor_pb) pb = pb1;
        }
    }
    return pb;
}

}  // namespace

extern "C" {

int pagedkv_version(void) { return 100; }

const char *pagedkv_status_string(int status) {
    switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: invalid argument";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: unsupported shape or type";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: CUDA runtime error";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS: not enough free blocks";
    default: return "unknown pagedkv status";
    }
}

int kv_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens, const pkv_cache_desc *cache,
                         void *stream) {
    if (int rc = check_cache(cache)) return rc;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 4))
        return PKV_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return PKV_ERR_CUDA;
    const cudaError_t e =
        pkv::launch_kv_cache_write(key, value, k_cache, v_cache, slot_mapping, num_tokens, cache->num_kv_heads,
                                   cache->num_blocks, sm_count(dev), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int kv_reshape_and_cache_fp8(const void *key, const void *value, void *k_cache, void *v_cache, float *k_scale,
                             float *v_scale, const int32_t *slot_mapping, int32_t num_tokens, const pkv_cache_desc *cache,
                             void *stream) {
    if (int rc = check_cache_fp8(cache)) return rc;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_scale, 16) || !aligned(v_scale, 16) || !aligned(slot_mapping, 4))
        return PKV_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return PKV_ERR_CUDA;
    const cudaError_t e = pkv::launch_kv_cache_write_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                                                         num_tokens, cache->num_kv_heads, cache->num_blocks,
                                                         sm_count(dev), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale, const int32_t *block_pairs,
                   int32_t num_pairs, const pkv_cache_desc *cache, void *stream) {
    if (!cache || cache->num_blocks < 1 || cache->num_kv_heads < 1) return PKV_ERR_INVALID_ARG;
    if (cache->block_size != kBlockSize || cache->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
    const bool fp8 = cache->dtype == PKV_DTYPE_FP8_E4M3;
    if (!fp8 && cache->dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (num_pairs < 0 || num_pairs > 65535) return PKV_ERR_INVALID_ARG;  // one CTA column per pair
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !block_pairs || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_pairs, 4))
        return PKV_ERR_INVALID_ARG;
    if (fp8 ? (!k_scale || !v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16)) : (k_scale || v_scale))
        return PKV_ERR_INVALID_ARG;
    const cudaError_t e = pkv::launch_kv_copy_blocks(k_cache, v_cache, k_scale, v_scale, block_pairs, num_pairs,
                                                     cache->num_kv_heads, fp8 ? 1 : 2, cache->num_blocks,
                                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                      int32_t partition_size, const pkv_cache_desc *cache) {
    // The workspace does not depend on the cache's element type.
    if ((check_cache(cache) != PKV_OK && check_cache_fp8(cache) != PKV_OK) || num_seqs < 1 || max_blocks_per_seq < 1)
        return 0;
    if (check_group(num_q_heads, cache->num_kv_heads) != PKV_OK) return 0;
    if (partition_size < 0 || partition_size % kBlockSize != 0) return 0;
    const int32_t pb = partition_size > 0 ? partition_size / kBlockSize : kMinPartBlocks;
    return plan_decode(num_seqs, num_q_heads, max_blocks_per_seq, pb).total;
}

int32_t paged_attention_decode_partitions(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                          int32_t partition_size, int32_t window, const pkv_cache_desc *cache) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    if (int rc = cache->dtype == PKV_DTYPE_FP8_E4M3 ? check_cache_fp8(cache) : check_cache(cache)) return rc;
    if (int rc = check_group(num_q_heads, cache->num_kv_heads)) return rc;
    if (num_seqs < 1 || num_seqs > 65535 || max_blocks_per_seq < 1 || window < 0) return PKV_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % kBlockSize != 0) return PKV_ERR_INVALID_ARG;
    // The same plan as the decode entry points: blocks a row can touch, CTAs per KV head.
    const int32_t span = window > 0 ? static_cast<int32_t>(std::min<int64_t>(
                                          max_blocks_per_seq, (static_cast<int64_t>(window) + 15) / kBlockSize + 1))
                                    : max_blocks_per_seq;
    const int32_t G = num_q_heads / cache->num_kv_heads;
    const int32_t head_splits = G / (G < 8 ? G : 8);
    int32_t pb = partition_size / kBlockSize;
    if (partition_size == 0) {
        const int dev = current_device();
        if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
        const bool fp8 = cache->dtype == PKV_DTYPE_FP8_E4M3;
        pb = auto_part_blocks(num_seqs, cache->num_kv_heads, head_splits, span, sm_count(dev), !fp8, fp8,
                              span < max_blocks_per_seq);
    }
    return plan_decode(num_seqs, num_q_heads, span, pb).max_parts;
}

namespace {

// Shared by the decode entry points; window = 0 means no sliding window; k_scale /
// v_scale non-null select the FP8 cache (cache->dtype PKV_DTYPE_FP8_E4M3); new_key /
// new_value non-null append each sequence's new row at position ctx - 1 in the same launch.
int decode_impl(void *out, int32_t out_dtype, const void *q, const void *k_cache, const void *v_cache,
                const float *k_scale, const float *v_scale, const int32_t *block_tables,
                const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                float scale, int32_t window, int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                size_t workspace_bytes, void *stream, const void *new_key = nullptr,
                const void *new_value = nullptr) {
    const bool fp8 = k_scale != nullptr;
    const bool append = new_key != nullptr;
    if (append && (fp8 || !new_value || !aligned(new_key, 16) || !aligned(new_value, 16))) return PKV_ERR_INVALID_ARG;
    if (int rc = fp8 ? check_cache_fp8(cache) : check_cache(cache)) return rc;
    if (fp8 && (!v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16))) return PKV_ERR_INVALID_ARG;
    if (int rc = check_group(num_q_heads, cache->num_kv_heads)) return rc;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_DTYPE_FLOAT32 && out_dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 1 || num_seqs > 65535 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_blocks_per_seq) * kBlockSize > INT32_MAX) return PKV_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % kBlockSize != 0) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
    if (window < 0) return PKV_ERR_INVALID_ARG;
    // Blocks one row can touch: all of its table, or at most ceil(W / 16) + 1 under a window.
    const int32_t span_blocks =
        window > 0 ? static_cast<int32_t>(std::min<int64_t>(max_blocks_per_seq, (static_cast<int64_t>(window) + 15) /
                                                                                         kBlockSize + 1))
                   : max_blocks_per_seq;
    // The documented contract: at least what paged_attention_workspace_size() answers for
    // the blocks a row can touch (for a window that is no more than for the whole table).
    if (workspace_bytes <
        paged_attention_workspace_size(num_seqs, num_q_heads, span_blocks, partition_size, cache))
        return PKV_ERR_WORKSPACE_TOO_SMALL;

    const int32_t n_kv = cache->num_kv_heads;
    const int32_t G = num_q_heads / n_kv;
    const int32_t hpc = G < 8 ? G : 8;  // query heads per CTA; larger groups are split over CTAs
    const int32_t head_splits = G / hpc;
    if (static_cast<int64_t>(n_kv) * head_splits > 65535) return PKV_ERR_UNSUPPORTED;

    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    const int sms = sm_count(dev);

    const int32_t pb = partition_size > 0 ? partition_size / kBlockSize
                                          : auto_part_blocks(num_seqs, n_kv, head_splits, span_blocks, sms, !fp8, fp8,
                                                             span_blocks < max_blocks_per_seq);
    const DecodePlan pl = plan_decode(num_seqs, num_q_heads, span_blocks, pb);
    if (workspace_bytes < pl.total) return PKV_ERR_WORKSPACE_TOO_SMALL;  // cannot happen for auto plans

    CUtensorMap kmap, vmap;
    if (fp8 ? (!encode_pool_map_fp8(&kmap, k_cache, cache->num_blocks, n_kv) ||
               !encode_pool_map_fp8(&vmap, v_cache, cache->num_blocks, n_kv))
            : (!encode_pool_map(&kmap, k_cache, cache->num_blocks, n_kv) ||
               !encode_pool_map(&vmap, v_cache, cache->num_blocks, n_kv)))
        return PKV_ERR_CUDA;

    if (fp8) {
        std::call_once(g_decode_fp8_prepared[dev], [&] { g_decode_fp8_prep_err[dev] = pkv::decode_fp8_prepare_device(); });
        if (g_decode_fp8_prep_err[dev] != cudaSuccess) return PKV_ERR_CUDA;
    } else {
        std::call_once(g_decode_prepared[dev], [&] { g_decode_prep_err[dev] = pkv::decode_prepare_device(); });
        if (g_decode_prep_err[dev] != cudaSuccess) return PKV_ERR_CUDA;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    pkv::DecodeParams p{};
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.part_m = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_m) : nullptr;
    p.part_l = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_l) : nullptr;
    p.part_o = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_o) : nullptr;
    p.num_seqs = num_seqs;
    p.n_q = num_q_heads;
    p.n_kv = n_kv;
    p.group = G;
    p.heads_per_cta = hpc;
    p.head_splits = head_splits;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.part_blocks = pl.part_blocks;
    p.max_parts = pl.max_parts;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.out_bf16 = out_dtype == PKV_DTYPE_BF16;
    p.window = window;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (append) {
        pkv::DecodeParamsAppend pa{};
        static_cast<pkv::DecodeParams &>(pa) = p;
        pa.new_k = new_key;
        pa.new_v = new_value;
        pa.k_cache = const_cast<void *>(k_cache);
        pa.v_cache = const_cast<void *>(v_cache);
        e = pkv::launch_paged_decode_append(kmap, vmap, pa, s);
    } else if (fp8) {
        pkv::DecodeParamsFp8 p8{};
        static_cast<pkv::DecodeParams &>(p8) = p;
        p8.k_scale = k_scale;
        p8.v_scale = v_scale;
        e = pkv::launch_paged_decode_fp8(kmap, vmap, p8, s);
    } else {
        e = pkv::launch_paged_decode(kmap, vmap, p, s);
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int paged_attention_decode(void *out, int32_t out_dtype, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t partition_size,
                           const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(out, out_dtype, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, 0, partition_size, cache, workspace, workspace_bytes,
                       stream);
}

int paged_attention_decode_append(void *out, int32_t out_dtype, const void *q, const void *key, const void *value,
                                  void *k_cache, void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_blocks_per_seq, float scale, int32_t partition_size,
                                  const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes, void *stream) {
    if (!key || !value) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, 0, partition_size, cache, workspace, workspace_bytes,
                       stream, key, value);
}

int paged_attention_decode_window(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                                  int32_t window, int32_t partition_size, const pkv_cache_desc *cache,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (window < 1) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, window, partition_size, cache, workspace,
                       workspace_bytes, stream);
}

int paged_attention_decode_fp8(void *out, int32_t out_dtype, const void *q, const void *k_cache, const void *v_cache,
                               const float *k_scale, const float *v_scale, const int32_t *block_tables,
                               const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t max_blocks_per_seq, float scale, int32_t window, int32_t partition_size,
                               const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes, void *stream) {
    if (!k_scale || !v_scale || window < 0) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, window, partition_size, cache, workspace,
                       workspace_bytes, stream);
}

size_t paged_attention_prefill_workspace_size(int32_t num_seqs, int32_t num_q_heads, const pkv_cache_desc *cache) {
    if ((check_cache(cache) != PKV_OK && check_cache_fp8(cache) != PKV_OK) || num_seqs < 1) return 0;
    if (check_group(num_q_heads, cache->num_kv_heads) != PKV_OK) return 0;
    return kStatusBytes;
}

namespace {

// Split-KV plan of the prefill kernel.  Its CTAs (one per KV head, sequence and
// pair of 128-row tiles; one CTA per SM) can be too few to fill the GPU -- a
// long chunk of one or two sequences, or a verify of few sequences -- and then
// each pair's key tiles are cut into `splits` ranges whose partials (m, l, O)
// the merge kernel folds ("LLM 推理全过程的维度变化与核心公式", section "工程优化
// 怎么嵌进公式": Flash-Decoding's split of cache_len and log-sum-exp reduction
// apply to the rows of a chunk alike).  The count is chosen from the sizes
// alone (context lengths are device data): at least 8 key tiles of the longest
// possible context per split, and the number of waves of CTAs closest to whole.
// Workspace: [status | part_m | part_l | part_o], each region 256-byte aligned.
struct PrefillPlan {
    int32_t splits;
    size_t off_m, off_l, off_o, total;
};
PrefillPlan plan_prefill(int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t total_rows, int32_t max_q_len,
                         int32_t max_blocks, int64_t sms) {
    PrefillPlan pl{1, kStatusBytes, kStatusBytes, kStatusBytes, kStatusBytes};
    const int32_t G = n_q / n_kv;
    if (G < 1 || 128 % G != 0 || max_q_len < 1 || total_rows < 1) return pl;
    const int64_t tiles = (static_cast<int64_t>(max_q_len) + 128 / G - 1) / (128 / G);
    const int64_t units = static_cast<int64_t>(n_kv) * num_seqs * ((tiles + 1) / 2);
    const int64_t key_tiles = (static_cast<int64_t>(max_blocks) * kBlockSize + 127) / 128;
    const int64_t max_splits = std::min<int64_t>(16, key_tiles / 8);
    if (sms < 1 || units >= sms || max_splits < 2) return pl;
    double best = 0.0;
    for (int64_t sp = 2; sp <= max_splits; ++sp) {
        if (units * sp < sms) continue;
        const double waves = static_cast<double>(units * sp) / static_cast<double>(sms);
        const double eff = waves / std::ceil(waves);
        if (eff > best + 1e-9) {
            best = eff;
            pl.splits = static_cast<int32_t>(sp);
        }
        if (eff >= 0.9) break;  // the fewest splits that fill the waves well
    }
    if (pl.splits <= 1) pl.splits = static_cast<int32_t>(max_splits);  // under one wave even so: take them all
    if ((tiles + 1) / 2 * pl.splits > 65535) {  // grid z: pairs x splits
        pl.splits = 1;
        return pl;
    }
    const size_t rows = static_cast<size_t>(total_rows) * n_q * pl.splits;
    pl.off_m = kStatusBytes;
    pl.off_l = pl.off_m + align_up(rows * 4, 256);
    pl.off_o = pl.off_l + align_up(rows * 4, 256);
    pl.total = pl.off_o + align_up(rows * kHeadDim * 4, 256);
    return pl;
}

int64_t device_sms_or_default() {
    const int dev = current_device();
    return dev >= 0 && dev < kMaxDevices ? sm_count(dev) : 152;
}

}  // namespace

size_t paged_attention_prefill_chunk_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t total_q_rows,
                                                    int32_t max_q_len, int32_t max_blocks_per_seq,
                                                    const pkv_cache_desc *cache) {
    if ((check_cache(cache) != PKV_OK && check_cache_fp8(cache) != PKV_OK) || num_seqs < 1 || max_blocks_per_seq < 1)
        return 0;
    if (check_group(num_q_heads, cache->num_kv_heads) != PKV_OK || total_q_rows < 0 || max_q_len < 0) return 0;
    return plan_prefill(num_seqs, num_q_heads, cache->num_kv_heads, total_q_rows, max_q_len, max_blocks_per_seq,
                        device_sms_or_default())
        .total;
}

namespace {

// Shared by the prefill-chunk and verify entry points.  cu_q_lens null: every sequence
// has uniform_q_len rows (sequence b owns rows b * uniform_q_len ..).
int prefill_impl(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens, int32_t uniform_q_len,
                 int32_t max_q_len, int32_t total_q_rows, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                 int32_t max_blocks_per_seq, float scale, const pkv_cache_desc *cache, void *workspace,
                 size_t workspace_bytes, void *stream, int32_t window = 0, const float *k_scale = nullptr,
                 const float *v_scale = nullptr) {
    // FP8 cache: E4M3 codes with per-slot scales, expanded to bf16 in shared memory.
    const bool fp8 = k_scale != nullptr;
    if (int rc = fp8 ? check_cache_fp8(cache) : check_cache(cache)) return rc;
    if (fp8 && (!v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16))) return PKV_ERR_INVALID_ARG;
    if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (window < 0) return PKV_ERR_INVALID_ARG;
    const int32_t G = num_q_heads / cache->num_kv_heads;
    // A 128-row MMA tile packs 128 / G query positions x the G heads of one KV group.
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PKV_ERR_UNSUPPORTED;
    if (!out || !q || (!cu_q_lens && uniform_q_len < 1) || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_DTYPE_FLOAT32 && out_dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 1 || num_seqs > 65535 || max_blocks_per_seq < 1 || max_q_len < 0 || total_q_rows < 0)
        return PKV_ERR_INVALID_ARG;
    if ((static_cast<int64_t>(max_q_len) + 127) / 128 * G > 65535) return PKV_ERR_UNSUPPORTED;  // grid z
    if (static_cast<int64_t>(max_blocks_per_seq) * kBlockSize > INT32_MAX) return PKV_ERR_INVALID_ARG;
    // K/V tiles are addressed by the 32-bit index block * n_kv + head.
    if (static_cast<int64_t>(cache->num_blocks) * cache->num_kv_heads > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(cu_q_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < kStatusBytes) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (max_q_len == 0 || total_q_rows == 0) return PKV_OK;

    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    // Split-KV when the CTAs cannot fill the GPU and the workspace holds the partials
    // (a workspace of the status word alone keeps one CTA per pair of row tiles).
    PrefillPlan pl = plan_prefill(num_seqs, num_q_heads, cache->num_kv_heads, total_q_rows, max_q_len,
                                  max_blocks_per_seq, sm_count(dev));
    if (pl.splits > 1 && workspace_bytes < pl.total) pl.splits = 1;

    CUtensorMap qmap, kmap, vmap, omap;
    if (!encode_rows_map(&qmap, q, total_q_rows, num_q_heads, G, false) ||
        !encode_rows_map(&omap, out, total_q_rows, num_q_heads, G, out_dtype == PKV_DTYPE_FLOAT32) ||
        !(fp8 ? encode_pool_map_fp8(&kmap, k_cache, cache->num_blocks, cache->num_kv_heads)
              : encode_pool_tile_map(&kmap, k_cache, cache->num_blocks, cache->num_kv_heads)) ||
        !(fp8 ? encode_pool_map_fp8(&vmap, v_cache, cache->num_blocks, cache->num_kv_heads)
              : encode_pool_tile_map(&vmap, v_cache, cache->num_blocks, cache->num_kv_heads)))
        return PKV_ERR_CUDA;
    std::call_once(g_prefill_prepared[dev], [&] { g_prefill_prep_err[dev] = pkv::prefill_prepare_device(); });
    if (g_prefill_prep_err[dev] != cudaSuccess) return PKV_ERR_CUDA;

    pkv::PrefillParams p{};
    p.out = out;
    p.cu_q_lens = cu_q_lens;
    p.uniform_q_len = cu_q_lens ? 0 : uniform_q_len;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = static_cast<uint32_t *>(workspace);
    p.num_seqs = num_seqs;
    p.n_q = num_q_heads;
    p.n_kv = cache->num_kv_heads;
    p.group = G;
    p.rows_per_tile = 128 / G;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.total_rows = total_q_rows;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.out_bf16 = out_dtype == PKV_DTYPE_BF16;
    p.window = window;
    p.k_scale = k_scale;
    p.v_scale = fp8 ? v_scale : nullptr;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.kv_splits = pl.splits;
    p.part_m = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.off_m) : nullptr;
    p.part_l = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.off_l) : nullptr;
    p.part_o = pl.splits > 1 ? reinterpret_cast<float *>(ws + pl.off_o) : nullptr;
    if (pkv::launch_prefill_chunk(qmap, kmap, vmap, omap, p, max_q_len, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace

int paged_attention_prefill_chunk(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens,
                                  int32_t max_q_len, int32_t total_q_rows, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                                  const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (!cu_q_lens) return PKV_ERR_INVALID_ARG;
    return prefill_impl(out, out_dtype, q, cu_q_lens, 0, max_q_len, total_q_rows, k_cache, v_cache, block_tables,
                        context_lens, num_seqs, num_q_heads, max_blocks_per_seq, scale, cache, workspace,
                        workspace_bytes, stream);
}

int paged_attention_prefill_chunk_window(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens,
                                         int32_t max_q_len, int32_t total_q_rows, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_blocks_per_seq, float scale, int32_t window,
                                         const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                                         void *stream) {
    if (!cu_q_lens || window < 1) return PKV_ERR_INVALID_ARG;
    return prefill_impl(out, out_dtype, q, cu_q_lens, 0, max_q_len, total_q_rows, k_cache, v_cache, block_tables,
                        context_lens, num_seqs, num_q_heads, max_blocks_per_seq, scale, cache, workspace,
                        workspace_bytes, stream, window);
}

int paged_attention_prefill_chunk_fp8(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens,
                                      int32_t max_q_len, int32_t total_q_rows, const void *k_cache,
                                      const void *v_cache, const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t window,
                                      const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                                      void *stream) {
    if (!cu_q_lens || !k_scale || !v_scale || window < 0) return PKV_ERR_INVALID_ARG;
    return prefill_impl(out, out_dtype, q, cu_q_lens, 0, max_q_len, total_q_rows, k_cache, v_cache, block_tables,
                        context_lens, num_seqs, num_q_heads, max_blocks_per_seq, scale, cache, workspace,
                        workspace_bytes, stream, window, k_scale, v_scale);
}

namespace {
constexpr int32_t kMaxVerifyRows = 16;  // draft positions per sequence
// SMs the verify routing below counts with: the current device's, else 152 (GB300).
int64_t route_sms() {
    const int dev = current_device();
    return dev >= 0 && dev < kMaxDevices ? sm_count(dev) : 152;
}

// Verify runs on the decode kernel (the G x k (position, head) columns of a KV head
// shared out over ceil(G * k / 16) CTAs of up to 16 MMA columns, 8 over an FP8
// cache, each reading the K/V) or on the prefill kernel (uniform q_len, K/V read
// once per row tile, split-KV when its CTAs cannot fill the GPU).  The decode
// route's time grows with the columns; the prefill route's is flat in k.
// Measured on a GB300 (us, decode route / prefill route):
//   8B-shaped B=64, G=4, k = 2 4 6 8 12 16:  104/207 128/207 191/207 206/207 296/207 388/207
//     FP8:                                   78/243 134/244 189/244 244/244 357/244 471/244
//   70B-shaped B=8 x 32K, G=8, k = 1 2 4 8 16: 171/283 200/286 295/290 570/295 1122/310
//     FP8:                                   116/338 195/340 373/343 730/350 1445/364
// so the prefill kernel is taken from G * k >= 32 columns on, where it can pack
// the group (G in {1, 2, 4, 8, 16}); below, the decode kernel.
bool verify_on_prefill(bool /*fp8*/, int32_t /*num_seqs*/, int32_t q_per_seq, int32_t G, int32_t /*n_kv*/) {
    if (G > 16 || 128 % G != 0) return false;
    return static_cast<int64_t>(G) * q_per_seq >= 32;
}
// CTAs per KV head and the columns each takes (the last one may take fewer): up to
// 16 columns (two 8-column MMA tiles) per CTA, 8 over an FP8 cache (one tile).
int32_t verify_splits(int32_t cols, bool fp8 = false) { return fp8 ? (cols + 7) / 8 : (cols + 15) / 16; }
int32_t verify_cols_per_cta(int32_t cols, bool fp8 = false) {
    return (cols + verify_splits(cols, fp8) - 1) / verify_splits(cols, fp8);
}

}  // namespace

size_t paged_attention_verify_workspace_size_on(int32_t kernel, int32_t num_seqs, int32_t q_per_seq,
                                                int32_t num_q_heads, int32_t max_blocks_per_seq,
                                                int32_t partition_size, const pkv_cache_desc *cache) {
    if (!cache) return 0;
    const bool fp8 = cache->dtype == PKV_DTYPE_FP8_E4M3;
    if ((fp8 ? check_cache_fp8(cache) : check_cache(cache)) != PKV_OK || num_seqs < 1 || max_blocks_per_seq < 1)
        return 0;
    if (q_per_seq < 1 || q_per_seq > kMaxVerifyRows) return 0;
    if (check_group(num_q_heads, cache->num_kv_heads) != PKV_OK) return 0;
    if (partition_size < 0 || partition_size % kBlockSize != 0) return 0;
    if (kernel < PKV_VERIFY_AUTO || kernel > PKV_VERIFY_PREFILL_KERNEL) return 0;
    const int32_t G = num_q_heads / cache->num_kv_heads;
    if (kernel == PKV_VERIFY_PREFILL_KERNEL && (G > 16 || 128 % G != 0)) return 0;
    if (kernel == PKV_VERIFY_PREFILL_KERNEL ||
        (kernel == PKV_VERIFY_AUTO && verify_on_prefill(fp8, num_seqs, q_per_seq, G, cache->num_kv_heads))) {
        if (static_cast<int64_t>(num_seqs) * q_per_seq > INT32_MAX) return 0;
        return plan_prefill(num_seqs, num_q_heads, cache->num_kv_heads, num_seqs * q_per_seq, q_per_seq,
                            max_blocks_per_seq, route_sms())
            .total;
    }
    const int32_t pb = partition_size > 0 ? partition_size / kBlockSize : kMinPartBlocks;
    return plan_decode(num_seqs, num_q_heads, max_blocks_per_seq, pb, q_per_seq).total;
}

size_t paged_attention_verify_workspace_size(int32_t num_seqs, int32_t q_per_seq, int32_t num_q_heads,
                                             int32_t max_blocks_per_seq, int32_t partition_size,
                                             const pkv_cache_desc *cache) {
    return paged_attention_verify_workspace_size_on(PKV_VERIFY_AUTO, num_seqs, q_per_seq, num_q_heads,
                                                    max_blocks_per_seq, partition_size, cache);
}

int paged_attention_verify_on_prefill(int32_t num_seqs, int32_t q_per_seq, int32_t num_q_heads,
                                      const pkv_cache_desc *cache) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    const bool fp8 = cache->dtype == PKV_DTYPE_FP8_E4M3;
    if (int rc = fp8 ? check_cache_fp8(cache) : check_cache(cache)) return rc;
    if (int rc = check_group(num_q_heads, cache->num_kv_heads)) return rc;
    if (num_seqs < 1 || q_per_seq < 1 || q_per_seq > kMaxVerifyRows) return PKV_ERR_INVALID_ARG;
    return verify_on_prefill(fp8, num_seqs, q_per_seq, num_q_heads / cache->num_kv_heads, cache->num_kv_heads) ? 1
                                                                                                                : 0;
}

namespace {

// Shared by paged_attention_verify and paged_attention_verify_window (window 0: none).
// k_scale / v_scale non-null: an FP8 cache (cache->dtype PKV_DTYPE_FP8_E4M3).  The
// kernel is chosen by verify_on_prefill.
int verify_impl(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq, const void *k_cache,
                const void *v_cache, const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t partition_size, int32_t window,
                const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes, void *stream,
                const float *k_scale = nullptr, const float *v_scale = nullptr, int32_t kernel = PKV_VERIFY_AUTO) {
    if (window < 0) return PKV_ERR_INVALID_ARG;
    const bool fp8 = k_scale != nullptr;
    if (int rc = fp8 ? check_cache_fp8(cache) : check_cache(cache)) return rc;
    if (fp8 && (!v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16))) return PKV_ERR_INVALID_ARG;
    if (int rc = check_group(num_q_heads, cache->num_kv_heads)) return rc;
    if (q_per_seq < 1 || q_per_seq > kMaxVerifyRows) return PKV_ERR_INVALID_ARG;
    if (kernel < PKV_VERIFY_AUTO || kernel > PKV_VERIFY_PREFILL_KERNEL) return PKV_ERR_INVALID_ARG;
    const int32_t G = num_q_heads / cache->num_kv_heads;
    if (kernel == PKV_VERIFY_PREFILL_KERNEL && (G > 16 || 128 % G != 0)) return PKV_ERR_UNSUPPORTED;
    if (kernel == PKV_VERIFY_PREFILL_KERNEL ||
        (kernel == PKV_VERIFY_AUTO && verify_on_prefill(fp8, num_seqs, q_per_seq, G, cache->num_kv_heads))) {
        // Prefill kernel, uniform rows: sequence b owns q rows b * q_per_seq .. + q_per_seq - 1.
        if (static_cast<int64_t>(num_seqs) * q_per_seq > INT32_MAX) return PKV_ERR_INVALID_ARG;
        return prefill_impl(out, out_dtype, q, nullptr, q_per_seq, q_per_seq, num_seqs * q_per_seq, k_cache, v_cache,
                            block_tables, context_lens, num_seqs, num_q_heads, max_blocks_per_seq, scale, cache,
                            workspace, workspace_bytes, stream, window, k_scale, v_scale);
    }
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_DTYPE_FLOAT32 && out_dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 1 || num_seqs > 65535 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_blocks_per_seq) * kBlockSize > INT32_MAX) return PKV_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % kBlockSize != 0) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < paged_attention_verify_workspace_size_on(PKV_VERIFY_DECODE_KERNEL, num_seqs, q_per_seq,
                                                                   num_q_heads, max_blocks_per_seq, partition_size,
                                                                   cache))
        return PKV_ERR_WORKSPACE_TOO_SMALL;

    const int32_t n_kv = cache->num_kv_heads;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    const int sms = sm_count(dev);
    const int32_t cols = G * q_per_seq;
    const int32_t splits = verify_splits(cols, fp8);
    // grid y of the decode kernel (KV heads x splits) and of the merge kernel (rows)
    if (static_cast<int64_t>(n_kv) * splits > 65535 || static_cast<int64_t>(num_seqs) * q_per_seq > 65535)
        return PKV_ERR_UNSUPPORTED;
    // Blocks a sequence's rows can touch: all of its table, or under a window the
    // keys from the first row's window start (ctx - k + 1 - W) to ctx - 1.
    const int32_t span =
        window > 0 ? static_cast<int32_t>(std::min<int64_t>(
                         max_blocks_per_seq, (static_cast<int64_t>(window) + q_per_seq - 1 + 15) / kBlockSize + 1))
                   : max_blocks_per_seq;
    const int32_t pb = partition_size > 0 ? partition_size / kBlockSize
                                          : auto_part_blocks(num_seqs, n_kv, splits, span, sms, false, false,
                                                             span < max_blocks_per_seq);
    const DecodePlan pl = plan_decode(num_seqs, num_q_heads, span, pb, q_per_seq);
    if (workspace_bytes < pl.total) return PKV_ERR_WORKSPACE_TOO_SMALL;

    CUtensorMap kmap, vmap;
    if (fp8 ? (!encode_pool_map_fp8(&kmap, k_cache, cache->num_blocks, n_kv) ||
               !encode_pool_map_fp8(&vmap, v_cache, cache->num_blocks, n_kv))
            : (!encode_pool_map(&kmap, k_cache, cache->num_blocks, n_kv) ||
               !encode_pool_map(&vmap, v_cache, cache->num_blocks, n_kv)))
        return PKV_ERR_CUDA;
    if (fp8) {
        std::call_once(g_decode_fp8_prepared[dev], [&] { g_decode_fp8_prep_err[dev] = pkv::decode_fp8_prepare_device(); });
        if (g_decode_fp8_prep_err[dev] != cudaSuccess) return PKV_ERR_CUDA;
    } else {
        std::call_once(g_decode_prepared[dev], [&] { g_decode_prep_err[dev] = pkv::decode_prepare_device(); });
        if (g_decode_prep_err[dev] != cudaSuccess) return PKV_ERR_CUDA;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    pkv::DecodeParamsFp8Verify p{};
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.part_m = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_m) : nullptr;
    p.part_l = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_l) : nullptr;
    p.part_o = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.off_o) : nullptr;
    p.num_seqs = num_seqs;
    p.n_q = num_q_heads;
    p.n_kv = n_kv;
    p.group = G;
    p.heads_per_cta = verify_cols_per_cta(cols, fp8);  // the CTA's share of the q_per_seq x G columns
    p.head_splits = splits;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.part_blocks = pl.part_blocks;
    p.max_parts = pl.max_parts;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.out_bf16 = out_dtype == PKV_DTYPE_BF16;
    p.window = window;
    p.q_per_seq = q_per_seq;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    cudaError_t e;
    if (fp8) {
        e = pkv::launch_paged_verify_fp8(kmap, vmap, p, static_cast<cudaStream_t>(stream));
    } else {
        pkv::DecodeParamsVerify pv{};
        static_cast<pkv::DecodeParams &>(pv) = static_cast<const pkv::DecodeParams &>(p);
        pv.q_per_seq = q_per_seq;
        e = pkv::launch_paged_verify(kmap, vmap, pv, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int paged_attention_verify(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                           int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                           int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return verify_impl(out, out_dtype, q, q_per_seq, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, partition_size, 0, cache, workspace, workspace_bytes,
                       stream);
}

int paged_attention_verify_window(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq,
                                  const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_blocks_per_seq, float scale, int32_t partition_size, int32_t window,
                                  const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (window < 1) return PKV_ERR_INVALID_ARG;
    return verify_impl(out, out_dtype, q, q_per_seq, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, partition_size, window, cache, workspace,
                       workspace_bytes, stream);
}

int paged_attention_verify_on(int32_t kernel, void *out, int32_t out_dtype, const void *q, int32_t q_per_seq,
                              const void *k_cache, const void *v_cache, const float *k_scale, const float *v_scale,
                              const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                              int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t window,
                              int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                              size_t workspace_bytes, void *stream) {
    if ((k_scale == nullptr) != (v_scale == nullptr)) return PKV_ERR_INVALID_ARG;
    return verify_impl(out, out_dtype, q, q_per_seq, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, partition_size, window, cache, workspace,
                       workspace_bytes, stream, k_scale, v_scale, kernel);
}

int paged_attention_verify_fp8(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq, const void *k_cache,
                               const void *v_cache, const float *k_scale, const float *v_scale,
                               const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                               int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t window,
                               int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                               size_t workspace_bytes, void *stream) {
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return verify_impl(out, out_dtype, q, q_per_seq, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, max_blocks_per_seq, scale, partition_size, window, cache, workspace,
                       workspace_bytes, stream, k_scale, v_scale);
}


// ---- decode without a caller workspace ------------------------------------------
// The scratch that paged_attention_decode would take as its workspace, as one
// file-scope device array.  Host code must not use the symbol itself as a
// pointer (it names a host-side shadow); it uses the device address obtained
// once per device with cudaGetSymbolAddress.
static_assert(PKV_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");
static __device__ __align__(256) uint8_t g_decode_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on `dev` (which must be current); nullptr on
// failure.  Only a successful lookup is kept, so a failed first call (for example
// one made during stream capture) is retried by the next one.
void *decode_scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) == cudaSuccess) g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}
}  // namespace

int paged_attention_decode_static_scratch(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, float scale, int32_t partition_size,
                                          const pkv_cache_desc *cache, uint32_t *status, void *stream) {
    if (int rc = check_cache(cache)) return rc;
    if (int rc = check_group(num_q_heads, cache->num_kv_heads)) return rc;
    if (status && !aligned(status, 4)) return PKV_ERR_INVALID_ARG;
    const size_t need =
        paged_attention_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq, partition_size, cache);
    if (need == 0) return PKV_ERR_INVALID_ARG;
    if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    uint8_t *scratch = static_cast<uint8_t *>(decode_scratch_address(dev));
    if (!scratch) return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // What must start at zero: the status word alone (the split-KV partials are
    // always written before they are read).
    static_assert(kStatusBytes <= PKV_STATIC_SCRATCH_BYTES, "the status word lies inside the scratch array");
    if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess) return PKV_ERR_CUDA;
    const int rc = paged_attention_decode(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                          num_q_heads, max_blocks_per_seq, scale, partition_size, cache, scratch,
                                          PKV_STATIC_SCRATCH_BYTES, stream);
    if (rc != PKV_OK) return rc;
    if (status && cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // extern "C"
