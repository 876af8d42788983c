// decode.cu -- paged decode attention: one CTA per sequence x KV head x
// partition serves the whole GQA group; the partitions of a split context are
// combined by a separate log-sum-exp merge kernel (Flash-Decoding) launched
// right behind the decode grid with programmatic dependent launch.
//
// What is computed ("LLM 推理全过程的维度变化与核心公式", section "Decode 阶段
// 维度流转"; "注意力演进与推理流程", section 3.1):
//   s_j = scale * <q[b][h], K_b[j][g]>,   g = floor(h / G),  j < ctx_b
//   out[b][h] = sum_j softmax(s)_j V_b[j][g]
// with K_b[j] at row j % 16 of physical block block_tables[b][j / 16].
//
// Design (GB300, HBM bound: every K/V byte is read once per KV head):
//  * One CTA serves all G query heads of a KV head (up to 8; larger groups are
//    split over CTAs), so each 4 KB (block, head) tile of K and of V is fetched
//    from HBM once.  A context is cut into partitions of `part_blocks` blocks
//    that run as independent CTAs (grid = partitions x heads x sequences).
//  * Inside a CTA each warp owns every NW-th block of the partition and runs
//    its own pipeline: lane 0 issues TMA tensor copies (128-byte swizzle) of the
//    block's K and V tiles into a ring of ST stages, completing on one mbarrier
//    per stage; the warp consumes stage after stage with no CTA-wide barrier.
//  * The group's dot products run on the tensor cores with warp-level MMA
//    (m16n8k16, bf16 in, fp32 accumulate), in the transposed form
//    S^T[16 keys x 8 heads] = K[16 x 128] Q^T[128 x 8] so that up to 8 heads fill
//    the n = 8 side, and O^T[128 x 8] += V^T[128 x 16] P^T[16 x 8].  The softmax
//    is the fp32 online softmax (running max m, running sum l, rescale of O when
//    m rises) with max reductions by warp shuffles across the 8 lanes that share
//    a head column; probabilities go from the S^T accumulator layout to the
//    B-operand layout of the second MMA with movmatrix transposes, as a bf16
//    head plus a bf16 remainder so that rounding P to bf16 costs no accuracy.
//  * Keys at or past ctx (the tail of the last block) are masked by index, never
//    by value, and their V rows are zeroed in registers, so stale or NaN bytes in
//    unused slots cannot leak into the result.
//  * FP8 (E4M3) caches (FP8 = true): a stage holds the block's 2 KB K and V code
//    tiles (one TMA box each) and their 64 B scale rows (bulk copies); the MMAs
//    run in fp16 as laid out in decode_core.cuh, the K scale multiplies the
//    scores and the V scale is folded into P.  Bytes per token and head halve.
//  * Sliding window W ("LLM 推理全过程的维度变化与核心公式", section "KV Cache 的
//    形状与增长": only the most recent W tokens' K and V are kept): the row sees
//    keys j >= j0 = max(0, ctx - W); partitions cover only the blocks from
//    j0 / 16 on, so whole blocks before the window are never fetched, and the
//    keys of the first block that precede j0 are masked like the tail.
//  * At the end the warps' (m, l, O) are combined through shared memory; with a
//    single partition the CTA writes out = O / l directly, otherwise it writes
//    the unnormalised partial (m, l, O) to the workspace, and lse_merge_kernel
//    folds the partitions of each (sequence, query head) row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "decode_core.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

template <bool FP8, bool VERIFY, bool APPEND = false>
using DecodeParamsT = std::conditional_t<
    FP8, std::conditional_t<VERIFY, DecodeParamsFp8Verify, DecodeParamsFp8>,
    std::conditional_t<VERIFY, DecodeParamsVerify, std::conditional_t<APPEND, DecodeParamsAppend, DecodeParams>>>;

// NCT: 8-column MMA tiles per CTA (2 only for multi-token verify with 9..16 columns).
// APPEND: the step's new K/V row of each sequence is appended in this launch.
template <int NW, int ST, bool FP8, bool VERIFY = false, int NCT = 1, bool APPEND = false>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeParamsT<FP8, VERIFY, APPEND> p) {
    constexpr uint32_t kStage = FP8 ? kStageBytes8 : kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem =
        reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Verify with several CTAs per KV head: the split is the fastest grid index, so
    // the CTAs that read the same K/V tiles run side by side and share them in L2.
    const int part = VERIFY ? static_cast<int>(blockIdx.x) / p.head_splits : static_cast<int>(blockIdx.x);
    const int hs = VERIFY ? static_cast<int>(blockIdx.y) * p.head_splits + static_cast<int>(blockIdx.x) % p.head_splits
                          : static_cast<int>(blockIdx.y);
    const int b = blockIdx.z;
    const int g = hs / p.head_splits;
    static_assert(NCT == 1 || (NCT == 2 && VERIFY && !FP8), "two column tiles: verify only");
    static_assert(!APPEND || (!FP8 && !VERIFY && NCT == 1), "append: bf16 decode only");
    const int hpc = p.heads_per_cta;
    const int hsl = hs - g * p.head_splits;  // this CTA's share of the group's columns
    const int h0 = g * p.group + hsl * hpc;
    // Columns of this CTA: decode, heads h0 .. h0 + hpc - 1; verify, the group's
    // (position, head) pairs hsl * hpc .. (the last share may be shorter).
    int ncols = hpc;
    if constexpr (VERIFY) ncols = min(hpc, p.group * p.q_per_seq - hsl * hpc);
    // q / out row (in units of 128-element head rows) of CTA column c: decode, head h0 + c of
    // sequence b; verify, column cg = hsl * hpc + c is position cg / G of sequence b's
    // q_per_seq rows and head g * G + cg % G.
    auto col_row = [&](int c) -> size_t {
        if constexpr (VERIFY) {
            const int cg = hsl * hpc + c;
            return (static_cast<size_t>(b) * p.q_per_seq + cg / p.group) * p.n_q + static_cast<size_t>(g) * p.group +
                   cg % p.group;
        } else {
            return static_cast<size_t>(b) * p.n_q + h0 + c;
        }
    };

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    griddep_launch_dependents();
    griddep_wait();  // inputs written by the previous kernel on the stream (e.g. the KV append)

    // ---- sequence extent (device data: checked, never trusted) ----
    int ctx = __ldg(p.context_lens + b);
    const int max_ctx = p.max_blocks * kBlockSize;
    const bool ctx_ok = ctx >= 1 && ctx <= max_ctx;
    if (!ctx_ok) {
        if (part == 0 && threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusBadContextLen);
        ctx = ctx < 1 ? 0 : max_ctx;
    }
    if constexpr (VERIFY) {
        if (ctx > 0 && ctx < p.q_per_seq) {  // the rows being verified must already be in the cache
            if (part == 0 && threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusBadQLen);
            ctx = 0;
        }
    }
    if (ctx == 0) {
        if (part == 0)
            for (int i = threadIdx.x; i < ncols * kHeadDim; i += NW * 32)
                store_out(p.out, p.out_bf16, col_row(i >> 7) * kHeadDim + (i & 127), 0.f);
        return;
    }
    const int nblocks = (ctx + kBlockSize - 1) / kBlockSize;
    int j0 = (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;  // first visible key
    if constexpr (VERIFY) {  // the earliest verified row (position ctx - q_per_seq) bounds the window
        if (p.window > 0) j0 = max(0, ctx - p.q_per_seq + 1 - p.window);
    }
    const int first_blk = j0 / kBlockSize;
    const int nparts = (nblocks - first_blk + p.part_blocks - 1) / p.part_blocks;
    if (part >= nparts) return;
    const int blk_begin = first_blk + part * p.part_blocks;
    const int nblk = min(p.part_blocks, nblocks - blk_begin);
    const int nmine = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;
    const int32_t *table = p.block_tables + static_cast<size_t>(b) * p.max_blocks;

    // Append: lane l holds 16 bytes of the new row (K for lanes 0-15, V for 16-31;
    // dims 64 * ((l >> 3) & 1) + 8 * (l & 7) ..), loaded early by the last partition's CTAs.
    uint4 app = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (APPEND) {
        if (ctx_ok && part == nparts - 1) {
            const size_t e = (static_cast<size_t>(b) * p.n_kv + g) * kHeadDim + 64 * ((lane >> 3) & 1) + 8 * (lane & 7);
            const void *src = lane < 16 ? p.new_k : p.new_v;
            app = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(src) + e));
        }
    }

    const uint32_t stage_base = smem_u32(smem) + warp * (ST * kStage);
    // FP8: the scale rows of each stage sit after all warps' code rings.
    const uint32_t scale_base = smem_u32(smem) + NW * ST * kStage + warp * (FP8 ? ST * kStageScaleBytes : 0);
    const uint32_t bar_base = smem_u32(smem) + NW * ST * kStage + (FP8 ? NW * ST * kStageScaleBytes : 0) + warp * ST * 8;

    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(bar_base + 8 * s, FP8 ? kFp8StageArrivals : 1);
        fence_mbar_init();
    }
    __syncwarp();
    constexpr int kIssueLanes = FP8 ? 8 : 1;  // lanes that take part in a stage's copies

    // Lanes < kIssueLanes: start the copies of this warp's i-th block into stage i % ST.
    auto issue = [&](int i) {
        const int s = i % ST;
        const int j = blk_begin + warp + NW * i;
        int phys = __ldg(table + j);
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) phys = 0;  // masked below
        if constexpr (FP8)
            issue_block_copy_fp8(&kmap, &vmap, p.k_scale, p.v_scale, stage_base + s * kStage,
                                 scale_base + s * kStageScaleBytes, bar_base + 8 * s, g, p.n_kv, phys, lane);
        else
            issue_block_copy(&kmap, &vmap, stage_base + s * kStage, bar_base + 8 * s, g, phys);
    };
    if (lane < kIssueLanes)
        for (int i = 0; i < ST && i < nmine; ++i) issue(i);

    // ---- Q^T as the B operand (16 dims x 8 heads per k-step), kept in registers ----
    const int n = lane >> 2;  // head column of B / row group of C
    const int q4 = lane & 3;
    uint32_t bqt[NCT][8][2];
    auto &bq = bqt[0];
    float sl2 = p.scale_log2;
    if constexpr (FP8 && VERIFY) {
        const int qexp = load_q_frag_fp8_row(bq, p.q, col_row(n), n < ncols, lane);
        sl2 *= ldexpf(1.f, -qexp);
    } else if constexpr (FP8) {
        const int qexp = load_q_frag_fp8(bq, p.q, static_cast<size_t>(b) * p.n_q + h0, hpc, lane);
        sl2 *= ldexpf(1.f, -qexp);
    } else if constexpr (VERIFY) {
#pragma unroll
        for (int t = 0; t < NCT; ++t) load_q_frag_row(bqt[t], p.q, col_row(8 * t + n), 8 * t + n < ncols, lane);
    } else {
        load_q_frag(bq, p.q, static_cast<size_t>(b) * p.n_q + h0, hpc, lane);
    }
    // Verify: the absolute causal bound (exclusive) of this lane's columns 8t + 2*q4 and 8t + 2*q4 + 1.
    int pos_end[NCT][2] = {};
    if constexpr (VERIFY) {
#pragma unroll
        for (int t = 0; t < NCT; ++t)
#pragma unroll
            for (int u = 0; u < 2; ++u)
                pos_end[t][u] = ctx - p.q_per_seq + (hsl * hpc + 8 * t + 2 * q4 + u) / p.group + 1;
    }

    DecodeAcc acct[NCT];
    auto &acc = acct[0];
#pragma unroll
    for (int t = 0; t < NCT; ++t) acct[t].reset();

    int consumed = 0;
    bool timed_out = false;
    for (int i = 0; i < nmine; ++i) {
        const int s = i % ST;
        const uint32_t bar = bar_base + 8 * s;
        bool ok = mbar_wait(bar, (i / ST) & 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            timed_out = true;
            break;
        }
        const int j = blk_begin + warp + NW * i;
        const int phys = __ldg(table + j);
        int valid = min(kBlockSize, ctx - j * kBlockSize);
        const int lo = j == first_blk ? j0 - j * kBlockSize : 0;
        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
            valid = 0;
            if (lane == 0 && p.status) atomicOr(p.status, kStatusBadBlockId);
        }
        const uint32_t kb = stage_base + s * kStage;
        if constexpr (APPEND) {
            if (ctx_ok && j == nblocks - 1 && valid > 0) {
                // The new row r of the last block: into this warp's copy of the block (K and V,
                // 16 bytes per lane at the swizzled position) and, from one CTA per KV head, to the pool.
                const int r = (ctx - 1) & (kBlockSize - 1);
                const int box = (lane >> 3) & 1, ch = lane & 7;
                sts128(kb + (lane >> 4) * kTileBytes + box * kBoxBytes + r * 128 + ((ch ^ (r & 7)) << 4), app);
                if (hsl == 0) {
                    void *pool = lane < 16 ? p.k_cache : p.v_cache;
                    const size_t e = ((static_cast<size_t>(phys) * p.n_kv + g) * kBlockSize + r) * kHeadDim +
                                     64 * box + 8 * ch;
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pool) + e) = app;
                }
                __syncwarp();
            }
        }
        if constexpr (FP8 && VERIFY) {
            const int w = p.window > 0 ? p.window : (1 << 30);
            const int lim0 = pos_end[0][0] - j * kBlockSize, lim1 = pos_end[0][1] - j * kBlockSize;
            decode_block_fp8<true>(acc, bq, kb, kb + kTileBytes8, scale_base + s * kStageScaleBytes, lo, valid, sl2,
                                   lane, lim0, lim1, lim0 - w, lim1 - w);
        } else if constexpr (FP8) {
            decode_block_fp8(acc, bq, kb, kb + kTileBytes8, scale_base + s * kStageScaleBytes, lo, valid, sl2, lane);
        } else if constexpr (VERIFY && NCT == 2) {
            // column window starts (pos_end - W; far below any key without a window)
            const int w = p.window > 0 ? p.window : (1 << 30);
            const int lim[2][2] = {{pos_end[0][0] - j * kBlockSize, pos_end[0][1] - j * kBlockSize},
                                   {pos_end[1][0] - j * kBlockSize, pos_end[1][1] - j * kBlockSize}};
            const int low[2][2] = {{lim[0][0] - w, lim[0][1] - w}, {lim[1][0] - w, lim[1][1] - w}};
            decode_block_x2(acct, bqt, kb, kb + kTileBytes, lo, valid, sl2, lane, lim, low);
        } else if constexpr (VERIFY) {
            const int w = p.window > 0 ? p.window : (1 << 30);
            const int lim0 = pos_end[0][0] - j * kBlockSize, lim1 = pos_end[0][1] - j * kBlockSize;
            decode_block<true>(acc, bq, kb, kb + kTileBytes, lo, valid, sl2, lane, lim0, lim1, lim0 - w, lim1 - w);
        } else
            decode_block(acc, bq, kb, kb + kTileBytes, lo, valid, sl2, lane);
        consumed = i + 1;

        __syncwarp();
        if (lane < kIssueLanes && i + ST < nmine) {
            fence_proxy_async_smem();
            issue(i + ST);
        }
    }

    if (timed_out) {
        if (lane == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        // Let this warp's copies still in flight land before the CTA exits.
        const int issued = min(nmine, consumed + ST);
        for (int i = consumed; i < issued; ++i) mbar_wait(bar_base + 8 * (i % ST), (i / ST) & 1);
    }

    if constexpr (FP8) fp8_finish(acc);
    // Full row sums of this warp: add the shares of the 8 lanes of a head column.
#pragma unroll
    for (int t = 0; t < NCT; ++t) acct[t].reduce_sums();

    // ---- combine the warps of the CTA (shared memory reused after the pipeline) ----
    constexpr int kCols = 8 * NCT;  // MMA columns per warp
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(smem);  // [NW][kCols][128]
    float *red_m = red_o + NW * kCols * kHeadDim;    // [NW][kCols]
    float *red_l = red_m + NW * kCols;               // [NW][kCols]
#pragma unroll
    for (int t = 0; t < NCT; ++t) {
        const int c0 = warp * kCols + 8 * t + 2 * q4;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            // O^T fragment rows n and n + 8 of MMA mt are dims d0 and d1 (bf16: 16mt + n, +8;
            // FP8: the permuted order 16n + 2mt, +1)
            const int d0 = FP8 ? 16 * n + 2 * mt : 16 * mt + n;
            const int d1 = FP8 ? d0 + 1 : d0 + 8;
            red_o[c0 * kHeadDim + d0] = acct[t].o[mt][0];
            red_o[(c0 + 1) * kHeadDim + d0] = acct[t].o[mt][1];
            red_o[c0 * kHeadDim + d1] = acct[t].o[mt][2];
            red_o[(c0 + 1) * kHeadDim + d1] = acct[t].o[mt][3];
        }
        if (lane < 4) {
            red_m[c0] = acct[t].m0;
            red_m[c0 + 1] = acct[t].m1;
            red_l[c0] = acct[t].l0;
            red_l[c0 + 1] = acct[t].l1;
        }
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < ncols * kHeadDim; idx += NW * 32) {
        const int hh = idx >> 7, d = idx & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * kCols + hh]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = fast_exp2(red_m[w * kCols + hh] - Mu);
            L += f * red_l[w * kCols + hh];
            O += f * red_o[(w * kCols + hh) * kHeadDim + d];
        }
        const size_t row = col_row(hh);
        if (nparts == 1) {
            store_out(p.out, p.out_bf16, row * kHeadDim + d, L > 0.f ? O / L : 0.f);
        } else {
            const size_t pi = row * p.max_parts + part;
            p.part_o[pi * kHeadDim + d] = O;
            if (d == 0) {
                p.part_m[pi] = M;
                p.part_l[pi] = L;
            }
        }
    }
}

}  // namespace

namespace {

// Log-sum-exp merge of the partitions (one CTA per query row and query head):
//   out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p
// ("LLM 推理全过程的维度变化与核心公式", section "工程优化怎么嵌进公式", Flash
// Decoding; scores in the log2 domain).  8 warps fold the partitions
// p = w, w + 8, ...; lane owns dims 4*lane .. 4*lane + 3.
constexpr int kMergeWarps = 8;
// Calls whose rows have at most this many partitions fold them with one warp per
// (row, query head); more go to one CTA per (row, query head), whose warps fold the
// partitions in parallel (measured, decode call back to back: 8B-shaped batch, 4
// partitions, 91.7 -> 90.9 us with the warp fold; MQA sweep, 3, 23.6 -> 23.3; 70B
// verify k = 16 on the split prefill, 7, 291.2 -> 284.1; mixed batch, 8, 159.3 ->
// 159.9; 70B-shaped B=8 and B=1, 32, 165.0 -> 174.2 and 84.6 -> 91.9).
constexpr int kMergeWarpMaxParts = 7;

// Rows r = blockIdx.y, + gridDim.y, ... < rows.  fixed_parts > 0: every row has that
// many partials (the prefill's key splits); 0: a row's partition count follows
// from its sequence's context length as the decode kernel derived it.
__global__ void __launch_bounds__(kMergeWarps * 32)
    lse_merge_kernel(const DecodeParams p, int rows, int rows_per_seq, int fixed_parts) {
    __shared__ float red_o[kMergeWarps][kHeadDim];
    __shared__ float red_x[kMergeWarps];
    __shared__ float red_l[kMergeWarps];
    const int h = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();  // the producing grid's partials
    for (int r = blockIdx.y; r < rows; r += gridDim.y) {  // q row r of the call (decode: r = b)
        int nparts = fixed_parts;
        if (nparts == 0) {
            const int b = r / rows_per_seq;  // its sequence
            int ctx = __ldg(p.context_lens + b);
            const int max_ctx = p.max_blocks * kBlockSize;
            ctx = ctx < 1 ? 0 : (ctx > max_ctx ? max_ctx : ctx);
            // first visible key of the call's earliest row of this sequence, as the decode kernel has it
            // (decode: rows_per_seq = 1, key ctx - W; verify: the first of the q_per_seq rows)
            const int first_blk = (p.window > 0 ? max(0, ctx - rows_per_seq + 1 - p.window) : 0) / kBlockSize;
            nparts = ((ctx + kBlockSize - 1) / kBlockSize - first_blk + p.part_blocks - 1) / p.part_blocks;
        }
        if (nparts <= 1) continue;  // written directly by the decode kernel (CTA-uniform)
        const size_t base = (static_cast<size_t>(r) * p.n_q + h) * p.max_parts;
        float M = -INFINITY;
        for (int i = threadIdx.x; i < nparts; i += kMergeWarps * 32) M = fmaxf(M, __ldcg(p.part_m + base + i));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (lane == 0) red_x[warp] = M;
        __syncthreads();
        M = red_x[0];
#pragma unroll
        for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, red_x[w]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int i = warp; i < nparts; i += kMergeWarps) {
            const float f = fast_exp2(__ldcg(p.part_m + base + i) - Mu);
            L += f * __ldcg(p.part_l + base + i);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (base + i) * kHeadDim) + lane);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
        }
        reinterpret_cast<float4 *>(red_o[warp])[lane] = acc;
        if (lane == 0) red_l[warp] = L;
        __syncthreads();
        if (threadIdx.x < kHeadDim) {
            float Ls = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) {
                Ls += red_l[w];
                O += red_o[w][threadIdx.x];
            }
            store_out(p.out, p.out_bf16, (static_cast<size_t>(r) * p.n_q + h) * kHeadDim + threadIdx.x,
                      Ls > 0.f ? O / Ls : 0.f);
        }
        __syncthreads();  // red_* are reused by the next row
    }
    // The next kernel on the stream (often the next step's decode) launches only as
    // the merge ends: launched earlier, its CTAs would take whatever SM slots were
    // free while this step's grids still ran, and a grid of few CTAs (one long
    // sequence: 256 CTAs) would start unevenly spread over the SMs (B=1 x 128K,
    // back-to-back steps: 85.0 us per step against 109.6 with the trigger at the
    // merge's start; the 8B-shaped batch of 2048 CTAs is unchanged).
    griddep_launch_dependents();
}

// The same fold with one warp per (row, query head) and eight per CTA, for calls
// with few partitions per row: lane i holds partition i's weight (32 at a time),
// each partition's O row arrives as one float4 per lane, and no shared memory or
// CTA barrier is involved (the one-CTA-per-row kernel spends most of a short fold
// on its barriers and on CTA scheduling: 2048 CTAs for the 8B-shaped batch).
constexpr int kMergeRowsPerCta = 8;
__global__ void __launch_bounds__(kMergeRowsPerCta * 32)
    lse_merge_warp_kernel(const DecodeParams p, int rows, int rows_per_seq, int fixed_parts) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_wait();  // the producing grid's partials
    const int64_t total = static_cast<int64_t>(rows) * p.n_q;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * kMergeRowsPerCta + warp; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * kMergeRowsPerCta) {
        const int r = static_cast<int>(idx / p.n_q), h = static_cast<int>(idx % p.n_q);
        int nparts = fixed_parts;
        if (nparts == 0) {  // as in lse_merge_kernel: the partitions of row r's sequence
            const int b = r / rows_per_seq;
            int ctx = __ldg(p.context_lens + b);
            const int max_ctx = p.max_blocks * kBlockSize;
            ctx = ctx < 1 ? 0 : (ctx > max_ctx ? max_ctx : ctx);
            const int first_blk = (p.window > 0 ? max(0, ctx - rows_per_seq + 1 - p.window) : 0) / kBlockSize;
            nparts = ((ctx + kBlockSize - 1) / kBlockSize - first_blk + p.part_blocks - 1) / p.part_blocks;
        }
        if (nparts <= 1) continue;  // written directly by the producing kernel (warp-uniform)
        const size_t base = (static_cast<size_t>(r) * p.n_q + h) * p.max_parts;
        float M = -INFINITY;
        for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(p.part_m + base + i));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = 0; i0 < nparts; i0 += 32) {
            float f = 0.f;
            if (i0 + lane < nparts) {
                f = fast_exp2(__ldcg(p.part_m + base + i0 + lane) - Mu);
                L += f * __ldcg(p.part_l + base + i0 + lane);
            }
            const int n = min(32, nparts - i0);
            const float4 *po = reinterpret_cast<const float4 *>(p.part_o + (base + i0) * kHeadDim) + lane;
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const float fj = __shfl_sync(0xffffffffu, f, j);
                const float4 v = __ldcg(po + static_cast<size_t>(j) * (kHeadDim / 4));
                acc.x += fj * v.x;
                acc.y += fj * v.y;
                acc.z += fj * v.z;
                acc.w += fj * v.w;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (L > 0.f) {
            acc.x /= L;
            acc.y /= L;
            acc.z /= L;
            acc.w /= L;
        } else {
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // (4-byte stores: the output is only required to be 4-byte aligned)
        const size_t o = (static_cast<size_t>(r) * p.n_q + h) * kHeadDim + 4 * lane;
        if (p.out_bf16) {
            __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) + o);
            ob[0] = __floats2bfloat162_rn(acc.x, acc.y);
            ob[1] = __floats2bfloat162_rn(acc.z, acc.w);
        } else {
            float *of = static_cast<float *>(p.out) + o;
            of[0] = acc.x;
            of[1] = acc.y;
            of[2] = acc.z;
            of[3] = acc.w;
        }
    }
    griddep_launch_dependents();  // (as lse_merge_kernel: the next grid launches as the merge ends)
}

}  // namespace

cudaError_t launch_merge(const DecodeParams &p, int rows, int rows_per_seq, int fixed_parts, cudaStream_t stream) {
    const int64_t pairs = static_cast<int64_t>(rows) * p.n_q;
    if (p.max_parts <= kMergeWarpMaxParts) {
        const int64_t ctas = (pairs + kMergeRowsPerCta - 1) / kMergeRowsPerCta;
        return launch_pdl(lse_merge_warp_kernel, dim3(static_cast<unsigned>(ctas < 65535 * 16 ? ctas : 65535 * 16)),
                          dim3(kMergeRowsPerCta * 32), 0, stream, p, rows, rows_per_seq, fixed_parts);
    }
    return launch_pdl(lse_merge_kernel, dim3(p.n_q, rows < 65535 ? rows : 65535), dim3(kMergeWarps * 32), 0, stream, p,
                      rows, rows_per_seq, fixed_parts);
}

namespace {

template <int NW, int ST, bool FP8 = false, bool VERIFY = false, int NCT = 1, bool APPEND = false>
cudaError_t launch_variant(const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const DecodeParamsT<FP8, VERIFY, APPEND> &p, cudaStream_t stream) {
    const dim3 grid = VERIFY ? dim3(p.max_parts * p.head_splits, p.n_kv, p.num_seqs)
                             : dim3(p.max_parts, p.n_kv * p.head_splits, p.num_seqs);
    cudaError_t e = launch_pdl(paged_decode_kernel<NW, ST, FP8, VERIFY, NCT, APPEND>, grid, dim3(NW * 32),
                               FP8 ? decode_fp8_smem_bytes() : decode_smem_bytes(), stream, kmap, vmap, p);
    if (e != cudaSuccess) return e;
    int rows_per_seq = 1;
    if constexpr (VERIFY) rows_per_seq = p.q_per_seq;
    if (p.max_parts > 1) e = launch_merge(p, p.num_seqs * rows_per_seq, rows_per_seq, 0, stream);
    return e;
}

// The bf16 decode: 4 warps, 2 stages of one K and one V tile per warp; 64 KB of
// shared memory let 3 CTAs share an SM (measured best of 4 x 2, 4 x 3, 4 x 4
// and 8 x 2 warps x stages).
constexpr int kWarps = 4, kStages = 2;

// The FP8 decode: 4 warps, 3 stages of 4 KB codes (+ 128 B of scales) per warp;
// 128 registers and 52 KB of shared memory let 4 CTAs share an SM.
constexpr int kFp8Warps = 4, kFp8Stages = 3;

}  // namespace

size_t decode_smem_bytes() {
    // stage ring + mbarriers + 1 KB for aligning the base to the 1 KB swizzle period
    return static_cast<size_t>(kWarps) * kStages * kStageBytes + static_cast<size_t>(kWarps) * kStages * 8 + 1024;
}

cudaError_t decode_prepare_device() {
    const int smem = static_cast<int>(decode_smem_bytes());
    cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<kWarps, kStages, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(paged_decode_kernel<kWarps, kStages, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(paged_decode_kernel<kWarps, kStages, false, true, 2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(paged_decode_kernel<kWarps, kStages, false, false, 1, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

size_t decode_fp8_smem_bytes() {
    return static_cast<size_t>(kFp8Warps) * kFp8Stages * (kStageBytes8 + kStageScaleBytes + 8) + 1024;
}

cudaError_t decode_fp8_prepare_device() {
    const cudaError_t e =
        cudaFuncSetAttribute(paged_decode_kernel<kFp8Warps, kFp8Stages, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(decode_fp8_smem_bytes()));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(paged_decode_kernel<kFp8Warps, kFp8Stages, true, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(decode_fp8_smem_bytes()));
}

cudaError_t launch_paged_verify_fp8(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsFp8Verify &p,
                                    cudaStream_t stream) {
    if (p.heads_per_cta > 8) return cudaErrorInvalidValue;  // one 8-column MMA tile per CTA
    return launch_variant<kFp8Warps, kFp8Stages, true, true>(kmap, vmap, p, stream);
}

cudaError_t launch_paged_decode_fp8(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsFp8 &p,
                                    cudaStream_t stream) {
    return launch_variant<kFp8Warps, kFp8Stages, true>(kmap, vmap, p, stream);
}

cudaError_t launch_paged_verify(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsVerify &p,
                                cudaStream_t stream) {
    if (p.heads_per_cta > 16) return cudaErrorInvalidValue;
    // 9..16 columns: two 8-column MMA tiles per warp
    return p.heads_per_cta > 8 ? launch_variant<kWarps, kStages, false, true, 2>(kmap, vmap, p, stream)
                               : launch_variant<kWarps, kStages, false, true>(kmap, vmap, p, stream);
}

cudaError_t launch_paged_decode_append(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParamsAppend &p,
                                       cudaStream_t stream) {
    return launch_variant<kWarps, kStages, false, false, 1, true>(kmap, vmap, p, stream);
}

cudaError_t launch_paged_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                                cudaStream_t stream) {
    return launch_variant<kWarps, kStages>(kmap, vmap, p, stream);
}

}  // namespace pkv
