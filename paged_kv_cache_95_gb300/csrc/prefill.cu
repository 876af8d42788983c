// prefill.cu -- K4: causal chunked-prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// What is computed ("注意力演进与推理流程", section 1.1 and 变革 3; "LLM 推理全过程的
// 维度变化与核心公式", Chunked Prefill paragraph): sequence b has q_len new query
// rows at absolute positions c + i (c = ctx - q_len); row i of head h sees keys
// j <= c + i of KV head g = floor(h / G):
//     out[i][h] = sum_{j <= c+i} softmax_j(scale <q_i,h, K_j,g>) V_j,g
//
// Tiling (one CTA = one 128-row tile of one sequence and one KV group):
//  * The 128 rows of the MMA tile pack 128/G query positions x the G heads of
//    the group (row r = position (r / G), head (r % G)), so every K/V tile is
//    shared by the whole group.  Q is loaded once by TMA (128-byte swizzle).
//  * Keys are walked in tiles of 128 (= 8 paged blocks of 16).  Each paged
//    block's K and V tile (2 x 4 KB) is gathered with TMA from the block table
//    into a 2-stage ring; the blocks' halves are placed so that every operand
//    is one canonical 128-byte-swizzled UMMA layout: K as a K-major B operand,
//    V as an MN-major B operand.
//  * S = Q K^T (M=128, N=128, K=128) goes to tensor memory columns [0, 128).
//    The 128 threads each own one tensor-memory lane (= one row): they load the
//    row, apply the causal/length mask by index, update the running max and sum
//    (fp32, log2 domain) and write P = 2^(s - m) into shared memory in the
//    K-major layout of the A operand, as a bf16 head plus a bf16 remainder (the
//    remainder goes into the K tile, which S = Q K^T no longer needs), so that
//    P V = P_hi V + P_lo V keeps the weights to ~2^-17 relative.
//  * O += P_hi V + P_lo V (M=128, N=128 dims, K=128 keys) accumulates in tensor memory
//    columns [128, 256).  The running max used as the exponent reference is only
//    raised when a row's max grows by more than 2^8, in which case the row's O
//    is rescaled in tensor memory; P stays <= 256, safe in bf16/fp32.
//  * Epilogue: O / l from tensor memory to global memory.
//  * Keys at or past the context length and keys of blocks with an invalid id
//    are masked by index and their V rows are zeroed in shared memory, so stale
//    or NaN bytes cannot reach the result.
//
// Every mbarrier wait is bounded; on a timeout the CTA records
// PKV_STATUS_TIMEOUT, drains its outstanding copies and MMAs (bounded) and
// frees its tensor memory before returning.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kHalfTile = 128 * 128;        // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kOpBytes = 2 * kHalfTile;     // 32 KB: a 128 x 128 bf16 operand (lo | hi halves)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK0 = kOffQ + kOpBytes;    // stage s: K at kOffK0 + s * 2 * kOpBytes, V right after
constexpr uint32_t kOffP = kOffK0 + 4 * kOpBytes;
constexpr uint32_t kOffBar = kOffP + kOpBytes;   // mbarriers: q_full, kv_full[2], s_done, o_done
constexpr uint32_t kOffTmem = kOffBar + 64;
constexpr uint32_t kSmemBytes = kOffTmem + 16 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;              // S: [0,128), O: [128,256)

// Instruction descriptor, kind::f16: D f32, A/B bf16, M = 128, N = 128.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBase;               // A K-major, B K-major
constexpr uint32_t kIdescPV = kIdescBase | (1u << 16);  // B MN-major

// Shared-memory matrix descriptor for a 128-byte-swizzled canonical layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void store_row(void *out, int32_t bf16, size_t base, const float *v, int n, float inv) {
    if (bf16) {
        uint32_t *o = reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(out) + base);
        for (int i = 0; i < n; i += 2) o[i / 2] = pack_bf16x2(v[i] * inv, v[i + 1] * inv);
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
        for (int i = 0; i < n; i += 4) o[i / 4] = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem =
        reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int tile = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int G = p.group;
    const int rpt = p.rows_per_tile;

    if (tid == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    griddep_launch_dependents();
    griddep_wait();  // the KV append (or any producer of q) before us on the stream

    // ---- sequence extent (device data: checked) ----
    const int row0 = __ldg(p.cu_q_lens + b);
    const int q_len = __ldg(p.cu_q_lens + b + 1) - row0;
    const int ctx = __ldg(p.context_lens + b);
    if (q_len < 0 || q_len > ctx || ctx > p.max_blocks * kBlockSize || row0 < 0 || row0 + q_len > p.total_rows) {
        if (tile == 0 && g == 0 && tid == 0 && p.status) atomicOr(p.status, kStatusBadQLen);
        return;
    }
    const int i0 = tile * rpt;
    if (i0 >= q_len) return;
    const int rows_here = min(rpt, q_len - i0);
    const int c = ctx - q_len;
    const int last_pos = c + i0 + rows_here - 1;
    const int n_keys = last_pos + 1;  // keys 0 .. last_pos
    const int n_ktiles = (n_keys + 127) / 128;
    const int nblocks = (ctx + kBlockSize - 1) / kBlockSize;
    const int32_t *table = p.block_tables + static_cast<size_t>(b) * p.max_blocks;

    const uint32_t bar_q = sbase + kOffBar;
    const uint32_t bar_kv0 = bar_q + 8;  // kv_full[0], kv_full[1]
    const uint32_t bar_s = bar_q + 24;
    const uint32_t bar_o = bar_q + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(bar_kv0, 1);
        mbar_init(bar_kv0 + 8, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off;        // this warp's S lanes
    const uint32_t t_o = tmem + lane_off + 128;  // this warp's O lanes

    // Thread 0 gathers key tile kt (8 paged blocks) into stage kt & 1.
    auto issue_kv = [&](int kt) {
        const int s = kt & 1;
        const uint32_t kbase = sbase + kOffK0 + s * 2 * kOpBytes;
        const uint32_t vbase = kbase + kOpBytes;
        const uint32_t bar = bar_kv0 + 8 * s;
        int nload = 0;
        for (int t = 0; t < 8; ++t) nload += (kt * 8 + t < nblocks) ? 1 : 0;
        mbar_arrive_expect_tx(bar, nload * 4 * 2048);
        for (int t = 0; t < 8; ++t) {
            const int jb = kt * 8 + t;
            if (jb >= nblocks) break;
            int phys = __ldg(table + jb);
            if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) phys = 0;  // masked below
            tma_load_4d(kbase + t * 2048, &kmap, bar, 0, 0, g, phys);
            tma_load_4d(kbase + kHalfTile + t * 2048, &kmap, bar, 64, 0, g, phys);
            tma_load_4d(vbase + t * 2048, &vmap, bar, 0, 0, g, phys);
            tma_load_4d(vbase + kHalfTile + t * 2048, &vmap, bar, 64, 0, g, phys);
        }
    };

    if (tid == 0) {
        mbar_arrive_expect_tx(bar_q, kOpBytes);
        tma_load_3d(sbase + kOffQ, &qmap, bar_q, 0, g * G, row0 + i0);
        tma_load_3d(sbase + kOffQ + kHalfTile, &qmap, bar_q, 64, g * G, row0 + i0);
        issue_kv(0);
        if (n_ktiles > 1) issue_kv(1);
    }

    // This thread's row of the tile.
    const int r = tid;
    const int ii = r / G;
    const bool row_valid = ii < rows_here;
    const int pos = c + i0 + (row_valid ? ii : 0);
    const int limit = min(pos, ctx - 1);  // visible keys: j <= limit
    const float sl2 = p.scale_log2;

    float m_ref = -INFINITY;  // exponent reference (raised lazily)
    float l = 0.f;
    bool fail = !mbar_wait(bar_q, 0);
    int kt = 0;
    for (; kt < n_ktiles && !fail; ++kt) {
        const int s = kt & 1;
        const uint32_t kbase = sbase + kOffK0 + s * 2 * kOpBytes;
        const uint32_t vbase = kbase + kOpBytes;
        fail |= !mbar_wait(bar_kv0 + 8 * s, (kt >> 1) & 1);
        if (__syncthreads_or(fail)) {
            fail = true;
            break;
        }

        // Which of this tile's blocks have an invalid id (their keys are masked).
        uint32_t bad = 0;
        for (int t = 0; t < 8; ++t) {
            const int jb = kt * 8 + t;
            if (jb < nblocks && static_cast<unsigned>(__ldg(table + jb)) >= static_cast<unsigned>(p.num_blocks))
                bad |= 1u << t;
        }
        if (bad && tid == 0 && p.status) atomicOr(p.status, kStatusBadBlockId);

        // ---- S = Q K^T ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = (kk >> 2) * kHalfTile, koff = (kk & 3) * 32;
                const uint64_t ad = sw128_desc(sbase + kOffQ + half + koff, 16, 1024);
                const uint64_t bd = sw128_desc(kbase + half + koff, 16, 1024);
                umma_bf16(tmem, ad, bd, kIdescQK, kk > 0);
            }
            umma_commit(bar_s);
        }
        fail |= !mbar_wait(bar_s, kt & 1);
        tc_fence_after();

        // ---- softmax on this thread's row ----
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x32(t_s + 32 * q, sr[q]);
        tmem_wait_ld();
        const int key0 = kt * 128;
        float mt = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int j = key0 + 32 * q + k;
                const bool ok = j <= limit && !((bad >> ((32 * q + k) >> 4)) & 1u);
                const float v = ok ? __uint_as_float(sr[q][k]) * sl2 : -INFINITY;
                sr[q][k] = __float_as_uint(v);
                mt = fmaxf(mt, v);
            }
        float alpha = 1.f;
        if (mt > m_ref + 8.f || (m_ref == -INFINITY && mt != -INFINITY)) {
            alpha = fast_exp2(m_ref - mt);  // 0 when m_ref = -inf
            m_ref = mt;
        }
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;

        // The previous P V must be done before P is overwritten and O is rescaled.
        if (kt > 0) fail |= !mbar_wait(bar_o, (kt - 1) & 1);
        tc_fence_after();
        if (tid == 0 && kt >= 1 && kt + 1 < n_ktiles) issue_kv(kt + 1);  // stage (kt+1)&1 is free now

        // P as bf16, K-major 128-byte-swizzled rows: chunk c of row r at c ^ (r & 7).
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t prow = sbase + kOffP + (q >> 1) * kHalfTile + r * 128;
            const uint32_t plow = kbase + (q >> 1) * kHalfTile + r * 128;  // remainder: into the spent K tile
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                uint32_t w[4], x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pa = fast_exp2(__uint_as_float(sr[q][8 * c8 + 2 * e]) - mu);
                    const float pb = fast_exp2(__uint_as_float(sr[q][8 * c8 + 2 * e + 1]) - mu);
                    rs += pa + pb;
                    w[e] = pack_bf16x2(pa, pb);
                    x[e] = pack_bf16x2(pa - __uint_as_float(w[e] << 16), pb - __uint_as_float(w[e] & 0xffff0000u));
                }
                const int chunk = (q & 1) * 4 + c8;
                const uint32_t sw = ((chunk ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + sw), "r"(w[0]), "r"(w[1]),
                             "r"(w[2]), "r"(w[3])
                             : "memory");
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(plow + sw), "r"(x[0]), "r"(x[1]),
                             "r"(x[2]), "r"(x[3])
                             : "memory");
            }
        }
        l = l * alpha + rs;

        // Rescale O rows whose reference max moved (warp-uniform tensor-memory access).
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t orow[32];
                tmem_ld_32x32b_x32(t_o + 32 * q, orow);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) orow[k] = __float_as_uint(__uint_as_float(orow[k]) * alpha);
                tmem_st_32x32b_x32(t_o + 32 * q, orow);
            }
            tmem_wait_st();
        }

        // Zero V rows of keys no row may see (past the context, or of a bad block).
        {
            const int rv = ctx - key0;  // keys [rv, 128) are past the context
            if (rv < 128 || bad) {
                for (int idx = tid; idx < 128 * 16; idx += kThreads) {
                    const int key = idx >> 4, ch = idx & 15;
                    if (key >= rv || ((bad >> (key >> 4)) & 1u)) {
                        const uint32_t addr = vbase + (ch >> 3) * kHalfTile + key * 128 + (ch & 7) * 16;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                    }
                }
            }
        }

        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            fail = true;
            break;
        }

        // ---- O += P_hi V + P_lo V ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t aoff = (t >> 2) * kHalfTile + (t & 3) * 32;
                const uint64_t bd = sw128_desc(vbase + t * 2048, kHalfTile, 1024);
                umma_bf16(tmem + 128, sw128_desc(sbase + kOffP + aoff, 16, 1024), bd, kIdescPV,
                          (kt > 0 || t > 0) ? 1u : 0u);
                umma_bf16(tmem + 128, sw128_desc(kbase + aoff, 16, 1024), bd, kIdescPV, 1u);
            }
            umma_commit(bar_o);
        }
    }

    if (!fail) {
        fail |= !mbar_wait(bar_o, (n_ktiles - 1) & 1);
        tc_fence_after();
    }
    if (__syncthreads_or(fail)) {
        if (tid == 0) {
            if (p.status) atomicOr(p.status, kStatusTimeout);
            // Best effort: let outstanding copies and MMAs finish before freeing.
            mbar_wait(bar_o, (max(kt, 1) - 1) & 1);
        }
    } else {
        // ---- epilogue: out = O / l ----
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow_base =
            (static_cast<size_t>(row0 + i0 + ii) * p.n_q + static_cast<size_t>(g) * G + (r % G)) * kHeadDim;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t orow[32];
            tmem_ld_32x32b_x32(t_o + 32 * q, orow);
            tmem_wait_ld();
            if (row_valid) store_row(p.out, p.out_bf16, orow_base + 32 * q, reinterpret_cast<float *>(orow), 32, inv);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes; }

cudaError_t prefill_prepare_device() {
    return cudaFuncSetAttribute(prefill_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
}

cudaError_t launch_prefill_chunk(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const PrefillParams &p, int max_q_len, cudaStream_t stream) {
    const dim3 grid((max_q_len + p.rows_per_tile - 1) / p.rows_per_tile, p.n_kv, p.num_seqs);
    return launch_pdl(prefill_chunk_kernel, grid, dim3(kThreads), kSmemBytes, stream, qmap, kmap, vmap, p);
}

}  // namespace pkv
