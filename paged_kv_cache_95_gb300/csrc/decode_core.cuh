// decode_core.cuh -- the per-block math of paged decode attention (one warp,
// one 16-token block), used by the decode kernel in decode.cu.
//
// One warp processes one 16-token paged block of one KV head for up to 8 query
// heads of its GQA group ("注意力演进与推理流程", section 3.1: head h reads KV
// group floor(h / G)):
//   S^T[16 keys x 8 heads] = K[16 x 128] Q^T[128 x 8]      (mma.sync m16n8k16)
//   online softmax in the log2 domain (lazy exponent reference m, sum l,
//   rescale of O when m is raised)
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
constexpr int kNoVexp = 1 << 20;                            // "no V scale seen yet"
constexpr uint32_t kBoxBytes = kTileBytes / 2;              // 2048 B: 16 rows x 64 dims (128-B rows)
constexpr uint32_t kStageBytes = 2 * kTileBytes;            // K tile + V tile

__device__ __forceinline__ void store_out(void *out, int32_t bf16, size_t idx, float v) {
    if (bf16)
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(out)[idx] = v;
}

// Online-softmax state of one warp for the 8 head columns of its MMA tile.  Lane
// (n = lane / 4, q4 = lane % 4) holds columns 2*q4 and 2*q4 + 1: the exponent
// reference m (identical across the 8 lanes of a column), its share of the
// running sum l = sum 2^(s - m), and O^T rows 16*mt + n and 16*mt + n + 8 of
// those columns (O = sum 2^(s - m) v).  The reference is lazy: it is raised (and
// l and O rescaled) only when a score exceeds it by more than kLazyExp, so every
// weight stays <= 2^kLazyExp and most blocks skip the block maximum and the
// rescale; the result is the same softmax, since out = O / l for any reference.
constexpr float kLazyExp = 8.f;
struct DecodeAcc {
    float m0, m1, l0, l1;
    float o[8][4];
    // FP8 only: O is held times 2^vexp (vexp set by the largest V scale seen so
    // far, which it puts in [2, 4)); vthr = 2^(2 - vexp): a V scale at or above it
    // lowers vexp.
    int vexp;
    float vthr, vup;  // vup = 2^vexp (0 before the first V scale)
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        vexp = kNoVexp;
        vthr = vup = 0.f;
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

// Q^T as the B operand of S^T = K Q^T: for k-step kk, lane (n, q4) holds column n
// (q row `row`, i.e. q + row * 128), dims 16*kk + 2*q4 (+1) and 16*kk + 8 + 2*q4 (+1).
// Columns with hv false are zero.
__device__ __forceinline__ void load_q_frag_row(uint32_t (&bq)[8][2], const void *q, size_t row, bool hv, int lane) {
    const int q4 = lane & 3;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(q) + row * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        bq[kk][0] = hv ? __ldg(qrow + (16 * kk + 2 * q4) / 2) : 0u;
        bq[kk][1] = hv ? __ldg(qrow + (16 * kk + 8 + 2 * q4) / 2) : 0u;
    }
}

// Decode: column n is head head0_row + n (heads n >= hpc are zero).
__device__ __forceinline__ void load_q_frag(uint32_t (&bq)[8][2], const void *q, size_t head0_row, int hpc,
                                            int lane) {
    const int n = lane >> 2;
    load_q_frag_row(bq, q, head0_row + n, n < hpc, lane);
}

// O columns 2*q4 and 2*q4 + 1 of this lane times a0 and a1.
__device__ __forceinline__ void rescale_o(DecodeAcc &acc, float a0, float a1) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        acc.o[mt][0] *= a0;
        acc.o[mt][1] *= a1;
        acc.o[mt][2] *= a0;
        acc.o[mt][3] *= a1;
    }
}
// Raises the exponent references of this lane's two columns when a score of the
// block exceeds them by more than kLazyExp (a warp vote; most blocks skip it):
// the column's block maximum becomes its reference and l and O are rescaled.
__device__ __forceinline__ void raise_reference(DecodeAcc &acc, float s00, float s01, float s10, float s11) {
    const bool up = s00 > acc.m0 + kLazyExp || s10 > acc.m0 + kLazyExp || s01 > acc.m1 + kLazyExp ||
                    s11 > acc.m1 + kLazyExp;
    if (!__any_sync(0xffffffffu, up)) return;
    float bm0 = fmaxf(s00, s10), bm1 = fmaxf(s01, s11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    float al0 = 1.f, al1 = 1.f;
    if (bm0 > acc.m0 + kLazyExp) {  // also the first visible key (m = -inf: alpha = 0, l and O are 0)
        al0 = fast_exp2(acc.m0 - bm0);
        acc.m0 = bm0;
    }
    if (bm1 > acc.m1 + kLazyExp) {
        al1 = fast_exp2(acc.m1 - bm1);
        acc.m1 = bm1;
    }
    acc.l0 *= al0;
    acc.l1 *= al1;
    rescale_o(acc, al0, al1);
}

// One block: kb / vb are the shared addresses of the stage's K and V tiles;
// only keys lo <= k < valid take part (lo > 0 only in the block where a sliding
// window starts); the others are masked by index and their V rows are zeroed in
// registers, so stale or NaN bytes in those slots never reach the result.
// Multi-token verify: column 2*q4 (2*q4 + 1) of this lane also only sees keys
// k < lim0 (lim1) -- its causal bound -- and, with a sliding window (LOW), keys
// k >= low0 (low1); keys between a column's bounds and [lo, valid) hold valid
// data, so only their weight is zeroed.
template <bool LOW = false>
__device__ __forceinline__ void decode_block(DecodeAcc &acc, const uint32_t (&bq)[8][2], uint32_t kb, uint32_t vb,
                                             int lo, int valid, float sl2, int lane, int lim0 = kBlockSize,
                                             int lim1 = kBlockSize, int low0 = 0, int low1 = 0) {
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
    const bool in_a = key_a >= lo && key_a < valid, in_b = key_b >= lo && key_b < valid;
    bool v00 = in_a && key_a < lim0, v01 = in_a && key_a < lim1;
    bool v10 = in_b && key_b < lim0, v11 = in_b && key_b < lim1;
    if constexpr (LOW) {
        v00 = v00 && key_a >= low0;
        v01 = v01 && key_a >= low1;
        v10 = v10 && key_b >= low0;
        v11 = v11 && key_b >= low1;
    }
    const float s00 = v00 ? c[0] * sl2 : -INFINITY;
    const float s01 = v01 ? c[1] * sl2 : -INFINITY;
    const float s10 = v10 ? c[2] * sl2 : -INFINITY;
    const float s11 = v11 ? c[3] * sl2 : -INFINITY;
    raise_reference(acc, s00, s01, s10, s11);
    const float mu0 = acc.m0 == -INFINITY ? 0.f : acc.m0;
    const float mu1 = acc.m1 == -INFINITY ? 0.f : acc.m1;
    const float p00 = fast_exp2(s00 - mu0), p01 = fast_exp2(s01 - mu1);
    const float p10 = fast_exp2(s10 - mu0), p11 = fast_exp2(s11 - mu1);
    acc.l0 += p00 + p10;
    acc.l1 += p01 + p11;

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

    // Zero V rows of keys outside [lo, valid) (their P is 0, but 0 * NaN would not be).
    uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
    if (lo > 0 || valid < kBlockSize) {
        auto keep = [&](int k) { return k >= lo && k < valid; };
        const int ka = 2 * q4, kb2 = 2 * q4 + 8;
        vm_lo = (keep(ka) ? 0x0000ffffu : 0u) | (keep(ka + 1) ? 0xffff0000u : 0u);
        vm_hi = (keep(kb2) ? 0x0000ffffu : 0u) | (keep(kb2 + 1) ? 0xffff0000u : 0u);
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

// One block for two 8-column tiles of the same KV head (16 MMA columns, e.g.
// multi-token verify with G x q_per_seq in 9..16): each K and V fragment is read
// from shared memory once and feeds both tiles' MMAs; each tile keeps its own
// online-softmax state.  lim[t][0..1] are the causal bounds (exclusive, relative
// to the block) of this lane's columns 2*q4 and 2*q4 + 1 of tile t; low[t][0..1]
// their sliding-window starts (inclusive; 0 or below without a window).
__device__ __forceinline__ void decode_block_x2(DecodeAcc (&acc)[2], const uint32_t (&bq)[2][8][2], uint32_t kb,
                                                uint32_t vb, int lo, int valid, float sl2, int lane,
                                                const int (&lim)[2][2], const int (&low)[2][2]) {
    const int n = lane >> 2, q4 = lane & 3;
    const int kkey = (lane & 7) | (((lane >> 3) & 1) << 3);
    const int khi = lane >> 4;
    const int vkey = (lane & 7) | ((lane >> 4) << 3);
    const int vhi = (lane >> 3) & 1;

    // S^T = K Q^T for both column tiles
    float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int chunk = 2 * kk + khi;
        const uint32_t addr = kb + (chunk >> 3) * kBoxBytes + kkey * 128 + (((chunk & 7) ^ (lane & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4(a, addr);
        mma_bf16_16816(c[0], a, bq[0][kk][0], bq[0][kk][1]);
        mma_bf16_16816(c[1], a, bq[1][kk][0], bq[1][kk][1]);
    }

    // Online softmax per tile; P^T fragments (bf16 head + remainder) per tile.
    const int key_a = n, key_b = n + 8;
    const bool in_a = key_a >= lo && key_a < valid, in_b = key_b >= lo && key_b < valid;
    uint32_t pb[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const float s00 = in_a && key_a < lim[t][0] && key_a >= low[t][0] ? c[t][0] * sl2 : -INFINITY;
        const float s01 = in_a && key_a < lim[t][1] && key_a >= low[t][1] ? c[t][1] * sl2 : -INFINITY;
        const float s10 = in_b && key_b < lim[t][0] && key_b >= low[t][0] ? c[t][2] * sl2 : -INFINITY;
        const float s11 = in_b && key_b < lim[t][1] && key_b >= low[t][1] ? c[t][3] * sl2 : -INFINITY;
        raise_reference(acc[t], s00, s01, s10, s11);
        const float mu0 = acc[t].m0 == -INFINITY ? 0.f : acc[t].m0;
        const float mu1 = acc[t].m1 == -INFINITY ? 0.f : acc[t].m1;
        const float p00 = fast_exp2(s00 - mu0), p01 = fast_exp2(s01 - mu1);
        const float p10 = fast_exp2(s10 - mu0), p11 = fast_exp2(s11 - mu1);
        acc[t].l0 += p00 + p10;
        acc[t].l1 += p01 + p11;
        const uint32_t ph0 = pack_bf16x2(p00, p01), ph1 = pack_bf16x2(p10, p11);
        const uint32_t pl0 = pack_bf16x2(p00 - __uint_as_float(ph0 << 16), p01 - __uint_as_float(ph0 & 0xffff0000u));
        const uint32_t pl1 = pack_bf16x2(p10 - __uint_as_float(ph1 << 16), p11 - __uint_as_float(ph1 & 0xffff0000u));
        pb[t][0] = movmatrix_trans(ph0);
        pb[t][1] = movmatrix_trans(ph1);
        pb[t][2] = movmatrix_trans(pl0);
        pb[t][3] = movmatrix_trans(pl1);
    }

    uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
    if (lo > 0 || valid < kBlockSize) {
        auto keep = [&](int k) { return k >= lo && k < valid; };
        const int ka = 2 * q4, kb2 = 2 * q4 + 8;
        vm_lo = (keep(ka) ? 0x0000ffffu : 0u) | (keep(ka + 1) ? 0xffff0000u : 0u);
        vm_hi = (keep(kb2) ? 0x0000ffffu : 0u) | (keep(kb2 + 1) ? 0xffff0000u : 0u);
    }

    // O^T += V^T P^T for both tiles (one V fragment per 16 dims)
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
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            mma_bf16_16816(acc[t].o[mt], a, pb[t][0], pb[t][1]);
            mma_bf16_16816(acc[t].o[mt], a, pb[t][2], pb[t][3]);
        }
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

// ---- FP8 (E4M3) cache: one code per element, one fp32 scale per (slot, head) ----
//
// The MMAs run in fp16, which holds every E4M3 value exactly.  S^T = K Q^T
// contracts over the head dims in a permuted order -- k-step kk, lane column
// t = lane % 4 covers dims 32t + 4kk + {0,1} and 32t + 4kk + {2,3} -- so each lane
// reads 32 contiguous code bytes of a key row; Q follows the same order (the dot
// product does not depend on it).  O^T += V^T P^T assigns fragment row g of MMA
// mt to output dim 16g + 2mt and row g + 8 to 16g + 2mt + 1, so each lane reads
// 16 contiguous code bytes of four key rows and builds key pairs with byte
// permutes; the combine step undoes the order.
constexpr uint32_t kTileBytes8 = kBlockSize * kHeadDim;   // 2 KB: 16 slots x 128 codes
constexpr uint32_t kStageBytes8 = 2 * kTileBytes8;        // K tile + V tile
constexpr uint32_t kScaleBytes = kBlockSize * 4;          // 64 B: one (block, head)'s scales
constexpr uint32_t kStageScaleBytes = 2 * kScaleBytes;    // K scales + V scales

// Q (bf16) as fp16 B fragments in the permuted dim order, times 2^qexp.  qexp is
// chosen so that the largest |q| of the CTA's heads lands in [2^13, 2^14): the
// power-of-two scaling is exact and keeps every value inside the fp16 range.
// Returns qexp (the caller multiplies the scores by 2^-qexp).
// Column n reads q row `row` (multiples of 128 elements); columns with hv false are zero.
__device__ __forceinline__ int load_q_frag_fp8_row(uint32_t (&bq)[8][2], const void *q, size_t row, bool hv,
                                                   int lane) {
    const int q4 = lane & 3;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(q) + row * kHeadDim);
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        bq[kk][0] = hv ? __ldg(qrow + (32 * q4 + 4 * kk) / 2) : 0u;
        bq[kk][1] = hv ? __ldg(qrow + (32 * q4 + 4 * kk + 2) / 2) : 0u;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            amax = fmaxf(amax, fabsf(__uint_as_float(bq[kk][j] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(bq[kk][j] & 0xffff0000u)));
        }
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int qexp = 0;
    if (amax > 0.f) {
        const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127;  // floor(log2) for normals
        qexp = min(100, max(-100, 13 - e));
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float lo = ldexpf(__uint_as_float(bq[kk][j] << 16), qexp);
            const float hi = ldexpf(__uint_as_float(bq[kk][j] & 0xffff0000u), qexp);
            bq[kk][j] = pack_f16x2(lo, hi);
        }
    return qexp;
}

// Decode: column n is head head0_row + n (heads n >= hpc are zero).
__device__ __forceinline__ int load_q_frag_fp8(uint32_t (&bq)[8][2], const void *q, size_t head0_row, int hpc,
                                               int lane) {
    const int n = lane >> 2;
    return load_q_frag_fp8_row(bq, q, head0_row + n, n < hpc, lane);
}

// One FP8 block.  kb / vb: the stage's K and V code tiles (16 rows x 128 B,
// 128-byte swizzled); sc: its scales (16 K scales, then 16 V scales).  Keys
// outside [lo, valid) are masked by index; their V codes and scales are never
// used, so stale or NaN bytes in those slots do not reach the result.
// fsl2 = scale * log2(e) * 2^-qexp.
//
// V scales are folded into the weights: P'' = p * sv * 2^vexp, with vexp the
// running exponent that puts the largest V scale seen so far in [2, 4); with the
// lazy reference p <= 2^8, so P'' <= 2^10 and every weight that matters is a
// normal fp16 number; O is held times 2^vexp (rescaled with the softmax
// correction when vexp drops) and brought back by fp8_finish().  P'' goes in as
// an fp16 head + remainder.
// Multi-token verify (BOUNDS): column 2*q4 (2*q4 + 1) of this lane only sees keys
// low0 <= k < lim0 (low1 <= k < lim1) of the block; those keys hold valid data,
// so only their weight is zeroed.
template <bool BOUNDS = false>
__device__ __forceinline__ void decode_block_fp8(DecodeAcc &acc, const uint32_t (&bq)[8][2], uint32_t kb,
                                                 uint32_t vb, uint32_t sc, int lo, int valid, float fsl2, int lane,
                                                 int lim0 = kBlockSize, int lim1 = kBlockSize, int low0 = 0,
                                                 int low1 = 0) {
    const int n = lane >> 2, q4 = lane & 3;
    const int key_a = n, key_b = n + 8;
    const bool in_a = key_a >= lo && key_a < valid, in_b = key_b >= lo && key_b < valid;

    // S^T = K Q^T: key rows n and n + 8, code bytes 32*q4 .. +31 (chunks 2*q4, 2*q4+1, swizzled);
    // two accumulators halve the dependent MMA chain.
    const uint32_t sw = static_cast<uint32_t>(n & 7);
    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 ka = lds128(kb + key_a * 128 + (((2 * q4 + h) ^ sw) << 4));
        const uint4 kb4 = lds128(kb + key_b * 128 + (((2 * q4 + h) ^ sw) << 4));
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb4.x, kb4.y, kb4.z, kb4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kk = 4 * h + i;
            uint32_t a[4];
            e4m3x4_to_f16x2x2(wa[i], a[0], a[2]);
            e4m3x4_to_f16x2x2(wb[i], a[1], a[3]);
            if (i & 1)
                mma_f16_16816(c2, a, bq[kk][0], bq[kk][1]);
            else
                mma_f16_16816(c, a, bq[kk][0], bq[kk][1]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] += c2[j];

    // Scores with each key's K scale; online softmax in the log2 domain.
    const float fa = lds_f32(sc + 4 * key_a) * fsl2, fb = lds_f32(sc + 4 * key_b) * fsl2;
    bool v00 = in_a, v01 = in_a, v10 = in_b, v11 = in_b;
    if constexpr (BOUNDS) {
        v00 = v00 && key_a < lim0 && key_a >= low0;
        v01 = v01 && key_a < lim1 && key_a >= low1;
        v10 = v10 && key_b < lim0 && key_b >= low0;
        v11 = v11 && key_b < lim1 && key_b >= low1;
    }
    const float s00 = v00 ? c[0] * fa : -INFINITY;
    const float s01 = v01 ? c[1] * fa : -INFINITY;
    const float s10 = v10 ? c[2] * fb : -INFINITY;
    const float s11 = v11 ? c[3] * fb : -INFINITY;
    const float sva = in_a ? lds_f32(sc + kScaleBytes + 4 * key_a) : 0.f;
    const float svb = in_b ? lds_f32(sc + kScaleBytes + 4 * key_b) : 0.f;
    // Lazy exponent reference (as for bf16) and lazy V exponent: both are revisited only
    // when a score exceeds its column's reference by more than kLazyExp or a V scale
    // reaches vthr (one warp vote; most blocks skip the reductions and the rescale).
    const bool raise = s00 > acc.m0 + kLazyExp || s10 > acc.m0 + kLazyExp || s01 > acc.m1 + kLazyExp ||
                       s11 > acc.m1 + kLazyExp || sva >= acc.vthr || svb >= acc.vthr;
    if (__any_sync(0xffffffffu, raise)) {
        float bm0 = fmaxf(s00, s10), bm1 = fmaxf(s01, s11), svmax = fmaxf(sva, svb);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            svmax = fmaxf(svmax, __shfl_xor_sync(0xffffffffu, svmax, off));
        }
        float as0 = 1.f, as1 = 1.f;  // softmax corrections (l and O)
        if (bm0 > acc.m0 + kLazyExp) {
            as0 = fast_exp2(acc.m0 - bm0);
            acc.m0 = bm0;
        }
        if (bm1 > acc.m1 + kLazyExp) {
            as1 = fast_exp2(acc.m1 - bm1);
            acc.m1 = bm1;
        }
        acc.l0 *= as0;
        acc.l1 *= as1;
        // A larger V scale lowers vexp (svmax * 2^vexp in [2, 4)): O, held times 2^vexp,
        // shrinks by the same power of two.
        float f = 1.f;
        if (svmax > 0.f && svmax >= acc.vthr) {
            const int ve = 1 - (static_cast<int>((__float_as_uint(svmax) >> 23) & 0xff) - 127);
            f = acc.vexp == kNoVexp ? 1.f : ldexpf(1.f, ve - acc.vexp);
            acc.vexp = ve;
            acc.vthr = ldexpf(1.f, 2 - ve);
            acc.vup = ldexpf(1.f, ve);
        }
        rescale_o(acc, as0 * f, as1 * f);
    }
    const float mu0 = acc.m0 == -INFINITY ? 0.f : acc.m0;
    const float mu1 = acc.m1 == -INFINITY ? 0.f : acc.m1;
    const float p00 = fast_exp2(s00 - mu0), p01 = fast_exp2(s01 - mu1);
    const float p10 = fast_exp2(s10 - mu0), p11 = fast_exp2(s11 - mu1);
    acc.l0 += p00 + p10;
    acc.l1 += p01 + p11;

    const float wa2 = sva * acc.vup, wb2 = svb * acc.vup;
    const float q00 = p00 * wa2, q01 = p01 * wa2, q10 = p10 * wb2, q11 = p11 * wb2;
    const uint32_t ph0 = pack_f16x2(q00, q01), ph1 = pack_f16x2(q10, q11);
    const float2 h0 = unpack_f16x2(ph0), h1 = unpack_f16x2(ph1);
    const uint32_t pl0 = pack_f16x2(q00 - h0.x, q01 - h0.y), pl1 = pack_f16x2(q10 - h1.x, q11 - h1.y);
    const uint32_t pb0 = movmatrix_trans(ph0), pb1 = movmatrix_trans(ph1);
    const uint32_t pr0 = movmatrix_trans(pl0), pr1 = movmatrix_trans(pl1);

    // V^T: key rows 2*q4, 2*q4+1, 2*q4+8, 2*q4+9, code bytes 16n .. 16n+15 (chunk n, swizzled);
    // masked keys contribute zero codes.
    auto keep = [&](int k) { return k >= lo && k < valid; };
    const int k0 = 2 * q4;
    uint4 v0 = lds128(vb + k0 * 128 + ((n ^ (k0 & 7)) << 4));
    uint4 v1 = lds128(vb + (k0 + 1) * 128 + ((n ^ ((k0 + 1) & 7)) << 4));
    uint4 v2 = lds128(vb + (k0 + 8) * 128 + ((n ^ ((k0 + 8) & 7)) << 4));
    uint4 v3 = lds128(vb + (k0 + 9) * 128 + ((n ^ ((k0 + 9) & 7)) << 4));
    if (lo > 0 || valid < kBlockSize) {  // (warp-uniform: only the window's first block and the last one)
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        if (!keep(k0)) v0 = zero;
        if (!keep(k0 + 1)) v1 = zero;
        if (!keep(k0 + 8)) v2 = zero;
        if (!keep(k0 + 9)) v3 = zero;
    }
    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
    const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        // bytes 2mt, 2mt+1 of each row: [row k.b, row k+1.b, row k.b+1, row k+1.b+1]
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t pa = __byte_perm(w0[mt >> 1], w1[mt >> 1], sel);
        const uint32_t pb = __byte_perm(w2[mt >> 1], w3[mt >> 1], sel);
        uint32_t a[4];
        e4m3x4_to_f16x2x2(pa, a[0], a[1]);
        e4m3x4_to_f16x2x2(pb, a[2], a[3]);
        mma_f16_16816(acc.o[mt], a, pb0, pb1);
        mma_f16_16816(acc.o[mt], a, pr0, pr1);
    }
}

// After the last FP8 block: O back to its true scale (it is held times 2^vexp).
__device__ __forceinline__ void fp8_finish(DecodeAcc &acc) {
    if (acc.vexp == kNoVexp) return;  // no key seen: O is zero
    const float down = ldexpf(1.f, -acc.vexp);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc.o[mt][j] *= down;
}

// Copies of one (block, head) FP8 tile pair and its scales into a stage, run by
// lanes 0-7 of the warp: lane 0 sends the two 2 KB code tiles through the TMA unit
// (4 KB of transactions on `bar`); lanes 0-3 / 4-7 each copy 16 B of the K / V scale
// row with cp.async and arrive on `bar` when it lands (so `bar` counts 1 + 8
// arrivals per phase).  Keeping the 64 B rows off the TMA unit halves the TMA
// operations per block.
constexpr uint32_t kFp8StageArrivals = 1 + 8;
__device__ __forceinline__ void issue_block_copy_fp8(const CUtensorMap *kmap, const CUtensorMap *vmap,
                                                     const float *k_scale, const float *v_scale, uint32_t dst,
                                                     uint32_t dst_scale, uint32_t bar, int kv_head, int n_kv,
                                                     int phys_block, int lane) {
    if (lane == 0) {
        mbar_arrive_expect_tx(bar, kStageBytes8);
        tma_load_4d(dst, kmap, bar, 0, 0, kv_head, phys_block);
        tma_load_4d(dst + kTileBytes8, vmap, bar, 0, 0, kv_head, phys_block);
    }
    const size_t row = (static_cast<size_t>(phys_block) * n_kv + kv_head) * kBlockSize;
    const int part = lane & 3;
    cp_async_16(dst_scale + (lane < 4 ? 0u : kScaleBytes) + 16u * part, (lane < 4 ? k_scale : v_scale) + row + 4 * part);
    cp_async_mbar_arrive_noinc(bar);
}

}  // namespace pkv
