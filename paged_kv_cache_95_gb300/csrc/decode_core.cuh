// decode_core.cuh -- the per-block math of paged decode attention (one warp,
// one 16-token block), used by the decode kernel in decode.cu.
//
// One warp processes one 16-token paged block of one KV head for up to 8 query
// heads of its GQA group ("注意力演进与推理流程", section 3.1: head h reads KV
// group floor(h / G)):
//   S^T[16 keys x 8 heads] = K[16 x 128] Q^T[128 x 8]      (mma.sync m16n8k16)
//   online softmax in the log2 domain (running max m, sum l, rescale of O)
//   O^T[128 x 8] += V^T[128 x 16] P^T[16 x 8]
// K and V tiles sit in shared memory as two 2 KB boxes each (64 dims x 16 rows,
// 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)), so the
// ldmatrix reads are bank-conflict free.
#pragma once

#include <cuda_bf16.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

constexpr uint32_t kTileBytes = kBlockSize * kHeadDim * 2;  // 4096 B: one (block, head) tile
constexpr uint32_t kBoxBytes = kTileBytes / 2;              // 2048 B: 16 rows x 64 dims (128-B rows)
constexpr uint32_t kStageBytes = 2 * kTileBytes;            // K tile + V tile

__device__ __forceinline__ void store_out(void *out, int32_t bf16, size_t idx, float v) {
    if (bf16)
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(out)[idx] = v;
}

// Online-softmax state of one warp for the 8 head columns of its MMA tile.  Lane
// (n = lane / 4, q4 = lane % 4) holds columns 2*q4 and 2*q4 + 1: the running max
// (identical across the 8 lanes of a column), its share of the running sum, and
// O^T rows 16*mt + n and 16*mt + n + 8 of those columns.
struct DecodeAcc {
    float m0, m1, l0, l1;
    float o[8][4];
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
    // Add up the 8 lanes' shares of the running sums (result in every lane).
    __device__ __forceinline__ void reduce_sums() {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }
};

// Q^T as the B operand of S^T = K Q^T: for k-step kk, lane (n, q4) holds head n,
// dims 16*kk + 2*q4 (+1) and 16*kk + 8 + 2*q4 (+1).  Heads n >= hpc are zero.
__device__ __forceinline__ void load_q_frag(uint32_t (&bq)[8][2], const void *q, size_t head0_row, int hpc,
                                            int lane) {
    const int n = lane >> 2, q4 = lane & 3;
    const bool hv = n < hpc;
    const uint32_t *qrow =
        reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(q) + (head0_row + n) * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        bq[kk][0] = hv ? __ldg(qrow + (16 * kk + 2 * q4) / 2) : 0u;
        bq[kk][1] = hv ? __ldg(qrow + (16 * kk + 8 + 2 * q4) / 2) : 0u;
    }
}

// One block: kb / vb are the shared addresses of the stage's K and V tiles;
// keys >= valid are masked by index (their V rows are zeroed in registers, so
// stale or NaN bytes in unused slots never reach the result).
__device__ __forceinline__ void decode_block(DecodeAcc &acc, const uint32_t (&bq)[8][2], uint32_t kb, uint32_t vb,
                                             int valid, float sl2, int lane) {
    const int n = lane >> 2, q4 = lane & 3;
    const int kkey = (lane & 7) | (((lane >> 3) & 1) << 3);  // K: matrices (keys 0-7 | 8-15) x (dims lo | hi)
    const int khi = lane >> 4;
    const int vkey = (lane & 7) | ((lane >> 4) << 3);        // V: matrices (dims lo | hi) x (keys 0-7 | 8-15)
    const int vhi = (lane >> 3) & 1;

    // S^T = K Q^T  (rows: keys, columns: heads)
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int chunk = 2 * kk + khi;
        const uint32_t addr = kb + (chunk >> 3) * kBoxBytes + kkey * 128 + (((chunk & 7) ^ (lane & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4(a, addr);
        mma_bf16_16816(c, a, bq[kk][0], bq[kk][1]);
    }

    // Online softmax in the log2 domain (scale * log2(e) folded into the scores).
    const int key_a = n, key_b = n + 8;
    const float s00 = key_a < valid ? c[0] * sl2 : -INFINITY;
    const float s01 = key_a < valid ? c[1] * sl2 : -INFINITY;
    const float s10 = key_b < valid ? c[2] * sl2 : -INFINITY;
    const float s11 = key_b < valid ? c[3] * sl2 : -INFINITY;
    float bm0 = fmaxf(s00, s10), bm1 = fmaxf(s01, s11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    const float mn0 = fmaxf(acc.m0, bm0), mn1 = fmaxf(acc.m1, bm1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(acc.m0 - mu0), al1 = fast_exp2(acc.m1 - mu1);
    const float p00 = fast_exp2(s00 - mu0), p01 = fast_exp2(s01 - mu1);
    const float p10 = fast_exp2(s10 - mu0), p11 = fast_exp2(s11 - mu1);
    acc.l0 = acc.l0 * al0 + p00 + p10;
    acc.l1 = acc.l1 * al1 + p01 + p11;
    acc.m0 = mn0;
    acc.m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        acc.o[mt][0] *= al0;
        acc.o[mt][1] *= al1;
        acc.o[mt][2] *= al0;
        acc.o[mt][3] *= al1;
    }

    // P (C layout: row key, col head) -> P^T in the B-operand layout.  P is
    // split into a bf16 head and a bf16 remainder (P = hi + lo to ~2^-17), so
    // the weights keep fp32-like precision through the bf16 MMA.
    const uint32_t ph0 = pack_bf16x2(p00, p01), ph1 = pack_bf16x2(p10, p11);
    const uint32_t pl0 = pack_bf16x2(p00 - __uint_as_float(ph0 << 16), p01 - __uint_as_float(ph0 & 0xffff0000u));
    const uint32_t pl1 = pack_bf16x2(p10 - __uint_as_float(ph1 << 16), p11 - __uint_as_float(ph1 & 0xffff0000u));
    const uint32_t pb0 = movmatrix_trans(ph0);  // keys 0-7
    const uint32_t pb1 = movmatrix_trans(ph1);  // keys 8-15
    const uint32_t pr0 = movmatrix_trans(pl0);
    const uint32_t pr1 = movmatrix_trans(pl1);

    // Zero V rows of keys >= valid (their P is 0, but 0 * NaN would not be).
    uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
    if (valid < kBlockSize) {
        const int ka = 2 * q4, kb2 = 2 * q4 + 8;
        vm_lo = (ka < valid ? 0x0000ffffu : 0u) | (ka + 1 < valid ? 0xffff0000u : 0u);
        vm_hi = (kb2 < valid ? 0x0000ffffu : 0u) | (kb2 + 1 < valid ? 0xffff0000u : 0u);
    }

    // O^T += V^T P^T  (rows: head dims, columns: heads)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int chunk = 2 * mt + vhi;
        const uint32_t addr = vb + (chunk >> 3) * kBoxBytes + vkey * 128 + (((chunk & 7) ^ (lane & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4_trans(a, addr);
        a[0] &= vm_lo;
        a[1] &= vm_lo;
        a[2] &= vm_hi;
        a[3] &= vm_hi;
        mma_bf16_16816(acc.o[mt], a, pb0, pb1);
        mma_bf16_16816(acc.o[mt], a, pr0, pr1);
    }
}

// Copies of one (block, head) K and V tile into a stage: four TMA boxes of 64
// dims x 16 slots, completing on `bar` with 8 KB of transactions.
__device__ __forceinline__ void issue_block_copy(const CUtensorMap *kmap, const CUtensorMap *vmap, uint32_t dst,
                                                 uint32_t bar, int kv_head, int phys_block) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_4d(dst, kmap, bar, 0, 0, kv_head, phys_block);
    tma_load_4d(dst + kBoxBytes, kmap, bar, 64, 0, kv_head, phys_block);
    tma_load_4d(dst + kTileBytes, vmap, bar, 0, 0, kv_head, phys_block);
    tma_load_4d(dst + kTileBytes + kBoxBytes, vmap, bar, 64, 0, kv_head, phys_block);
}

}  // namespace pkv
