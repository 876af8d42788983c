// launch.h -- internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel on the stream drains; every kernel here executes
// griddepcontrol.wait before touching global memory, so stream order holds.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;

// Device status bits (mirror the PKV_STATUS_* values of the public header).
constexpr uint32_t kStatusBadContextLen = 0x1u;
constexpr uint32_t kStatusBadBlockId = 0x2u;
constexpr uint32_t kStatusBadQLen = 0x4u;
constexpr uint32_t kStatusTimeout = 0x8u;

// ---- K1: cache write ----------------------------------------------------------
cudaError_t launch_kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale, const int32_t *pairs,
                                  int32_t num_pairs, int32_t n_kv, int32_t elem_bytes, int32_t num_blocks,
                                  cudaStream_t stream);
cudaError_t launch_kv_cache_write_fp8(const void *key, const void *value, void *k_cache, void *v_cache, float *k_scale,
                                      float *v_scale, const int32_t *slot_mapping, int32_t num_tokens, int32_t n_kv,
                                      int32_t num_blocks, int sm_count, cudaStream_t stream);
cudaError_t launch_kv_cache_write(const void *key, const void *value, void *k_cache, void *v_cache,
                                  const int32_t *slot_mapping, int32_t num_tokens, int32_t n_kv,
                                  int32_t num_blocks, int sm_count, cudaStream_t stream);

// ---- K2: decode with optional split-KV, K3: its log-sum-exp merge -----------------
struct DecodeParams {
    const void *q;               // bf16 [num_seqs][n_q][128]
    void *out;                   // [num_seqs][n_q][128], f32 or bf16
    const int32_t *block_tables; // [num_seqs][max_blocks]
    const int32_t *context_lens; // [num_seqs]
    float *part_m;               // [num_seqs][n_q][max_parts]   (log2 domain, scale folded in)
    float *part_l;               // [num_seqs][n_q][max_parts]
    float *part_o;               // [num_seqs][n_q][max_parts][128] (unnormalised)
    uint32_t *status;            // device status word
    int32_t num_seqs, n_q, n_kv;
    int32_t group;               // G = n_q / n_kv
    int32_t heads_per_cta;       // min(G, 8)
    int32_t head_splits;         // G / heads_per_cta
    int32_t max_blocks;          // block-table row length
    int32_t num_blocks;          // pool size
    int32_t part_blocks;         // blocks per partition
    int32_t max_parts;           // partitions of the longest possible context
    float scale_log2;            // scale * log2(e)
    int32_t out_bf16;            // 1: bf16 output, 0: f32
    int32_t window;              // sliding window W (keys j >= ctx - W visible); 0: none
};

// The FP8 decode's parameters: the same plus the per-token scales (a separate
// type, so the bf16 kernels' parameter block stays as it is).
struct DecodeParamsFp8 : DecodeParams {
    const float *k_scale;  // [num_blocks][n_kv][16]
    const float *v_scale;
};

// Multi-token verify on the decode kernel: each sequence has q_per_seq query rows
// (positions ctx - q_per_seq .. ctx - 1, causal among themselves); a CTA's MMA
// columns are the group's (position, head) pairs, heads_per_cta = G * q_per_seq <= 8.
struct DecodeParamsVerify : DecodeParams {
    int32_t q_per_seq;
};

// Multi-token verify over an FP8 cache (one 8-column MMA tile per CTA).
struct DecodeParamsFp8Verify : DecodeParamsFp8 {
    int32_t q_per_seq;
};

// Decode with the step's token appended in the same launch: new_k / new_v (bf16
// [num_seqs][n_kv][128]) hold each sequence's new K/V row, which belongs at
// position ctx - 1.  The CTAs that read the sequence's last block put the row
// into their shared-memory copy of that block, and the first CTA of each KV
// head's last partition writes it to the pool (k_cache / v_cache), so no CTA of
// the launch reads the slot from memory.
struct DecodeParamsAppend : DecodeParams {
    const void *new_k;
    const void *new_v;
    void *k_cache;
    void *v_cache;
};

// The log-sum-exp merge of split partials (m, l, O) into out, one CTA per (row,
// query head): rows_per_seq maps a row to its sequence's context length when the
// partition count follows from it (fixed_parts = 0); fixed_parts > 0 merges that
// many partials per row (the prefill's key splits).
cudaError_t launch_merge(const DecodeParams &p, int rows, int rows_per_seq, int fixed_parts, cudaStream_t stream);

// Shared-memory bytes of the decode kernel; sets its dynamic shared memory limit.
size_t decode_smem_bytes();
cudaError_t decode_prepare_device();
// Enqueues the decode kernel and, when a context is split into partitions, the
// merge kernel, both with programmatic dependent launch.
cudaError_t launch_paged_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                                cudaStream_t stream);
// The FP8 (E4M3 codes + per-token scales) decode: its own stage layout, same merge.
size_t decode_fp8_smem_bytes();
cudaError_t decode_fp8_prepare_device();
cudaError_t launch_paged_decode_fp8(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsFp8 &p,
                                    cudaStream_t stream);
cudaError_t launch_paged_verify(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsVerify &p,
                                cudaStream_t stream);
cudaError_t launch_paged_verify_fp8(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsFp8Verify &p,
                                    cudaStream_t stream);
cudaError_t launch_paged_decode_append(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsAppend &p,
                                       cudaStream_t stream);

// ---- K4: causal chunked prefill on tcgen05 ---------------------------------------
struct PrefillParams {
    void *out;                   // [total_rows][n_q][128]
    const int32_t *cu_q_lens;    // [num_seqs + 1]; null: every sequence has uniform_q_len rows
    const int32_t *block_tables; // [num_seqs][max_blocks]
    const int32_t *context_lens; // [num_seqs]
    uint32_t *status;
    int32_t num_seqs, n_q, n_kv, group;
    int32_t rows_per_tile;       // query positions per 128-row tile (128 / G)
    int32_t max_blocks, num_blocks;
    int32_t total_rows;
    float scale_log2;
    int32_t out_bf16;
    int32_t uniform_q_len;       // rows per sequence when cu_q_lens is null
    int32_t window;              // sliding window W (> 0): a row at pos sees pos - W < j <= pos; 0: none
    const float *k_scale;        // FP8 cache: per-slot scales [num_blocks][n_kv][16]; null for bf16
    const float *v_scale;
    // Split-KV (kv_splits > 1): CTA split s of a pair of row tiles takes key tiles
    // [s * per, (s + 1) * per) of the pair's n key tiles (per = ceil(n / kv_splits)) and
    // writes the unnormalised partial (m, l, O) of every row it owns to part_* (indexed
    // [(row * n_q + head) * kv_splits + s]); the merge kernel folds the splits.
    int32_t kv_splits;
    float *part_m, *part_l, *part_o;
};

size_t prefill_smem_bytes();
cudaError_t prefill_prepare_device();
cudaError_t launch_prefill_chunk(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const CUtensorMap &omap, const PrefillParams &p, int max_q_len, cudaStream_t stream);

}  // namespace pkv
