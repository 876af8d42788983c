// cache_write.cu -- K1: append new tokens' K/V to the paged pool through slot_mapping.
//
// For token t, KV head h: the 256-byte row key[t][h][:] goes to slot
// s = slot_mapping[t], i.e. block s / 16, offset s % 16 of the pool laid out
// [num_blocks][n_kv][16][128] ("LLM 推理全过程的维度变化与核心公式", section
// "Decode 阶段维度流转": KV_Cache[:, :, cache_len, :] = K_new, V_new; vLLM
// concepts deep dive, section 1: kernels write new K/V through the slot mapping).
//
// One thread moves one 16-byte vector of K and the matching vector of V, so
// reads are fully coalesced and each (token, head) row is written as one
// contiguous 256-byte run.  HBM bound: 2 x 2 x T x n_kv x 256 bytes.
//
// FP8 caches (E4M3 codes plus one fp32 scale per token and KV head: the INT8 /
// FP8 KV Cache item of "LLM 推理全过程的维度变化与核心公式", section "KV Cache 的
// 形状与增长", per-token quantisation): one warp per (token, head) row, four
// values per lane.  With a = max(max_k |x_k|, 2^-100): inv = 448 / a, code_k =
// E4M3(x_k * inv) (nearest even, saturating), scale = a / 448 -- each a single
// correctly rounded fp32 operation, so codes and scales are reproducible.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

__global__ void __launch_bounds__(256)
kv_cache_write_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ k_cache,
                      uint4 *__restrict__ v_cache, const int32_t *__restrict__ slot_mapping, int64_t total_vec,
                      int32_t n_kv, int64_t num_slots) {
    griddep_launch_dependents();
    griddep_wait();  // the previous kernel on the stream may still read the pool
    constexpr int kVecPerRow = kHeadDim * 2 / 16;  // 16 vectors of 8 bf16 per (token, head) row
    const int64_t vec_per_tok = static_cast<int64_t>(n_kv) * kVecPerRow;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vec; i += stride) {
        const int64_t t = i / vec_per_tok;
        const int64_t r = i - t * vec_per_tok;  // h * 16 + c
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0 || slot >= num_slots) continue;  // padding token or out-of-range slot: no write
        const int64_t blk = slot / kBlockSize;
        const int64_t off = slot - blk * kBlockSize;
        const int64_t h = r / kVecPerRow;
        const int64_t c = r - h * kVecPerRow;
        const int64_t dst = ((blk * n_kv + h) * kBlockSize + off) * kVecPerRow + c;
        const uint4 kv = __ldg(key + i);
        const uint4 vv = __ldg(value + i);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

// Block copy at a branch point: CTA (i, c) copies block pairs[2i] onto block
// pairs[2i+1] of cache c (0: K, 1: V), the block's codes then (FP8) its scales,
// in coalesced 16-byte vectors.  Ids outside [0, num_blocks) skip the pair.
__global__ void __launch_bounds__(256)
kv_copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, uint4 *__restrict__ k_scale,
                      uint4 *__restrict__ v_scale, const int32_t *__restrict__ pairs, int64_t block_vec,
                      int64_t scale_vec, int32_t num_blocks) {
    griddep_launch_dependents();
    griddep_wait();  // kernels before us may still read or write the pool
    const int64_t src = __ldg(pairs + 2 * blockIdx.x), dst = __ldg(pairs + 2 * blockIdx.x + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return;
    uint4 *data = blockIdx.y == 0 ? k_cache : v_cache;
    for (int64_t i = threadIdx.x; i < block_vec; i += blockDim.x) data[dst * block_vec + i] = data[src * block_vec + i];
    uint4 *sc = blockIdx.y == 0 ? k_scale : v_scale;
    if (sc)
        for (int64_t i = threadIdx.x; i < scale_vec; i += blockDim.x) sc[dst * scale_vec + i] = sc[src * scale_vec + i];
}

__global__ void __launch_bounds__(256)
kv_cache_write_fp8_kernel(const uint2 *__restrict__ key, const uint2 *__restrict__ value, uint32_t *__restrict__ k_cache,
                          uint32_t *__restrict__ v_cache, float *__restrict__ k_scale, float *__restrict__ v_scale,
                          const int32_t *__restrict__ slot_mapping, int64_t rows, int32_t n_kv, int64_t num_slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // Rows 0 .. rows-1 are K rows (token t, head h as t * n_kv + h), then the V rows.
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < 2 * rows; r += stride) {
        const bool is_v = r >= rows;
        const int64_t rr = is_v ? r - rows : r;
        const int64_t t = rr / n_kv, h = rr - t * n_kv;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0 || slot >= num_slots) continue;  // padding token or out-of-range slot: no write
        const uint2 x = __ldg((is_v ? value : key) + rr * 32 + lane);  // values 4 lane .. 4 lane + 3
        const float v0 = __uint_as_float(x.x << 16), v1 = __uint_as_float(x.x & 0xffff0000u);
        const float v2 = __uint_as_float(x.y << 16), v3 = __uint_as_float(x.y & 0xffff0000u);
        float a = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        a = fmaxf(a, 0x1p-100f);
        const float inv = __fdiv_rn(448.f, a);
        const uint32_t codes = f32x2_to_e4m3x2(__fmul_rn(v0, inv), __fmul_rn(v1, inv)) |
                               (f32x2_to_e4m3x2(__fmul_rn(v2, inv), __fmul_rn(v3, inv)) << 16);
        const int64_t blk = slot / kBlockSize;
        const int64_t row = (blk * n_kv + h) * kBlockSize + (slot - blk * kBlockSize);
        (is_v ? v_cache : k_cache)[row * 32 + lane] = codes;
        if (lane == 0) (is_v ? v_scale : k_scale)[row] = __fdiv_rn(a, 448.f);
    }
}

}  // namespace

cudaError_t launch_kv_cache_write_fp8(const void *key, const void *value, void *k_cache, void *v_cache, float *k_scale,
                                      float *v_scale, const int32_t *slot_mapping, int32_t num_tokens, int32_t n_kv,
                                      int32_t num_blocks, int sm_count, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(num_tokens) * n_kv;
    if (rows == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (2 * rows * 32 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(kv_cache_write_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                      static_cast<const uint2 *>(key), static_cast<const uint2 *>(value),
                      static_cast<uint32_t *>(k_cache), static_cast<uint32_t *>(v_cache), k_scale, v_scale,
                      slot_mapping, rows, n_kv, static_cast<int64_t>(num_blocks) * kBlockSize);
}

cudaError_t launch_kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale, const int32_t *pairs,
                                  int32_t num_pairs, int32_t n_kv, int32_t elem_bytes, int32_t num_blocks,
                                  cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t block_vec = static_cast<int64_t>(n_kv) * kBlockSize * kHeadDim * elem_bytes / 16;
    const int64_t scale_vec = static_cast<int64_t>(n_kv) * kBlockSize * 4 / 16;  // fp32 per (slot, head)
    return launch_pdl(kv_copy_blocks_kernel, dim3(static_cast<unsigned>(num_pairs), 2), dim3(256), 0, stream,
                      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), reinterpret_cast<uint4 *>(k_scale),
                      reinterpret_cast<uint4 *>(v_scale), pairs, block_vec, scale_vec, num_blocks);
}

cudaError_t launch_kv_cache_write(const void *key, const void *value, void *k_cache, void *v_cache,
                                  const int32_t *slot_mapping, int32_t num_tokens, int32_t n_kv,
                                  int32_t num_blocks, int sm_count, cudaStream_t stream) {
    const int64_t total_vec = static_cast<int64_t>(num_tokens) * n_kv * (kHeadDim * 2 / 16);
    if (total_vec == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total_vec + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(kv_cache_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, total_vec, n_kv,
                      static_cast<int64_t>(num_blocks) * kBlockSize);
}

}  // namespace pkv
