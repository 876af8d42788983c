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

}  // namespace

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
