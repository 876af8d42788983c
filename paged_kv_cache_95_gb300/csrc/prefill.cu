// prefill.cu -- K4: causal chunked-prefill attention over the paged cache on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// What is computed ("注意力演进与推理流程", section 1.1 and 变革 3; "LLM 推理全过程的
// 维度变化与核心公式", Chunked Prefill paragraph): sequence b has q_len new query
// rows at absolute positions c + i (c = ctx - q_len); row i of head h sees keys
// j <= c + i of KV head g = floor(h / G):
//     out[i][h] = sum_{j <= c+i} softmax_j(scale <q_i,h, K_j,g>) V_j,g
//
// Tiling (one CTA = two 128-row tiles of one sequence and one KV group):
//  * The 128 rows of an MMA tile pack 128/G query positions x the G heads of
//    the group (row r = position (r / G), head (r % G)), so every K/V tile is
//    shared by the whole group.  A CTA holds two adjacent row tiles (Q0 and
//    Q1, loaded once by TMA, 128-byte swizzle) and walks the key tiles once for
//    both: each K and V tile copied into shared memory feeds two tiles' MMAs,
//    which halves the copy bytes per flop (the copies landing in shared memory
//    are what limits a one-tile CTA).  Tile 0 stops at its own last key tile.
//  * Keys are walked in tiles of 128 (= 8 paged blocks of 16).  Each paged
//    block's K and V tiles (4 KB each) are gathered from the block table with
//    ONE TMA copy apiece into separate 2-deep K and V rings.  The copy's 5-D
//    view of the pool lands a tile as [slot group (keys 0-7 | 8-15)][dim half]
//    [8 slots][128 B], four 1 KB 128-byte-swizzle atoms, so that eight tiles
//    side by side form one canonical UMMA operand: K as a K-major B operand
//    (8-key groups 2 KB apart, the upper dim half 1 KB in), V per 16-key step
//    as an MN-major B operand (dim halves 1 KB apart, key groups 2 KB apart).
//
// Warp roles (warp specialisation, all hand-offs through mbarriers):
//  * warps 16 and 18: TMA producers for K and V.  Lane t < 8 reads block t of
//    a key tile from the block table (one tile ahead) and issues that block's
//    copy: the eight copies go out as one warp instruction.  A K slot is
//    refilled once both tiles' S MMAs that read it complete, a V slot once
//    both tiles' P V MMAs complete.
//  * warp 17 (one lane): MMA issuer; also owns the tensor-memory allocation
//    (all 512 columns: S/P of tile t in [128t, 128t+128), O of tile t in
//    [256 + 128t, +128)).  Per key tile k it issues, in this order,
//        S0(k) = Q0 K(k)^T,  P1(k-1) V(k-1),  S1(k) = Q1 K(k)^T,  P0(k) V(k)
//    (M=128, N=128), so the tensor core computes one tile's MMAs while the
//    other tile's softmax runs (ping-pong).  An S MMA overwrites the columns
//    of the P that the P V MMA issued just before it reads; MMAs of one thread
//    execute in order, and the commit after S_t(k) completes only when every
//    earlier MMA has, so when the softmax sees S_t(k) the previous P_t V is
//    already in O_t.  The thread waits only for the P barriers (and K(0)):
//    softmax warp 0 checks that V(k) and K(k+1) have landed before its pass
//    over key tile k, so every P barrier also covers the copies the MMAs after
//    it read (a wait on the issuing thread lets the tensor pipe run dry).
//  * warps 0-15 (512 threads) work on tile 0's scores, then on tile 1's, for
//    each key tile (the MMAs of one tile run while the other tile's softmax
//    does): warps w, w+4, w+8, w+12 own tensor-memory lanes 32*(w%4) .. +31
//    (= tile rows) and split the 128 columns in quarters, so each thread holds
//    32 scores of one row in registers, applies the causal/length mask by
//    index (skipped for fully visible chunks), and the four quarters exchange
//    their row maxima through shared memory (a 128-thread named barrier per row
//    quarter) -- in the plain chunk only when a vote over those 128 threads
//    says a weight against the current reference may pass 2^8.  Each updates
//    its quarter of the running sum (fp32, log2 domain, pairs of keys in packed
//    f32x2 arithmetic) and writes P = 2^(s - m) back over its 32 columns, in one
//    store, as [16 columns bf16 head | 16 columns bf16 remainder] (head = P
//    truncated to bf16, remainder = the rest, by mixed-precision FMAs, rounded to
//    bf16; P V = P_hi V + P_lo V keeps the weights to ~2^-16 relative).  The
//    exponent reference is only raised when a row's max grows by more than 2^8,
//    in which case the row's O is rescaled in tensor memory; P stays <= 256.
//  * Epilogue per tile after its last P V: O / l from tensor memory; a full
//    tile is staged in a free ring in the output tensor map's 128-byte-swizzled
//    layout and leaves by TMA store; a ragged last tile by 16-byte stores of its
//    valid rows only (a whole-box store would overwrite the next sequence).
//    When both tiles end at the same key tile, tile 0's epilogue (staged in the
//    K ring) runs while tile 1's last P V is still in the pipe; otherwise both
//    tiles' last P V first (tile 0: the V ring, tile 1: the K ring).
//  * Keys at or past the context length and keys of blocks with an invalid id
//    are masked by index and their V rows are zeroed in shared memory (once,
//    before the first P V that reads them), so stale or NaN bytes cannot reach
//    the result.
//
// Every mbarrier wait is bounded; a role whose wait runs out raises a
// CTA-wide abort flag, the others stop at their next wait, the CTA records
// PKV_STATUS_TIMEOUT and frees its tensor memory before returning.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kRowTiles = 2;      // 128-row Q tiles per CTA
constexpr int kSoftmaxWarps = 16;  // warps w, w+4, w+8, w+12 share lanes 32*(w%4).. and split the columns
constexpr int kProducerK = kSoftmaxWarps;              // warp 16
constexpr int kMmaWarp = kProducerK + 1;               // warp 17
constexpr int kProducerV = kProducerK + 2;             // warp 18
constexpr int kThreads = (kProducerV + 1) * 32;        // 608

constexpr uint32_t kHalfTile = 128 * 128;     // 16 KB: 128 rows x 128 bytes (Q dim half; staged output box)
constexpr uint32_t kOpBytes = 2 * kHalfTile;  // 32 KB: a 128 x 128 bf16 operand
constexpr uint32_t kBlkBytes = 4096;          // one paged (block, head) tile inside a K/V operand
constexpr int kStagesK = 2;                                // K ring depth
constexpr int kStagesV = 2;                                // V ring depth
constexpr uint32_t kOffQ = 0;                              // Q tiles: [tile][dim half][128 rows][128 B]
constexpr uint32_t kOffK = kOffQ + kRowTiles * kOpBytes;   // K ring: kStagesK x 32 KB
constexpr uint32_t kOffV = kOffK + kStagesK * kOpBytes;    // V ring: kStagesV x 32 KB
constexpr uint32_t kOffBar = kOffV + kStagesV * kOpBytes;
// q_full, k_full/k_empty[kStagesK], v_full/v_empty[kStagesV], then per tile s_full, p_full, o_done,
// then (FP8 cache) k_conv[kStagesK] (a V stage's expansion is covered by the P barriers)
constexpr int kBarTile = 1 + 2 * kStagesK + 2 * kStagesV;
constexpr int kBarConv = kBarTile + 3 * kRowTiles;
constexpr uint32_t kNumBars = kBarConv + kStagesK;
constexpr uint32_t kOffTmem = kOffBar + 8 * 24;
constexpr uint32_t kOffAbort = kOffTmem + 8;
constexpr uint32_t kXchBytes = 2 * 4 * 128 * 4;  // per tile: row maxima [key tile & 1][column quarter][128]
constexpr uint32_t kOffXch = kOffAbort + 8;
// The dynamic shared memory is declared 1024-byte aligned (the swizzle period of
// the TMA/UMMA operands); the kernel checks it and refuses to run otherwise.
// FP8 cache: the key tiles' per-slot scales, [K slot | V slot][8 blocks][16 slots] fp32.
// K scales are read by tile 1's softmax after the K stage is released (its S is
// done), so they live in a ring twice as deep as the K ring: key tile kt's K
// scales in slot kt % kScaleSlotsK stay until key tile kt + 2 kStagesK loads,
// which waits for S of key tile kt + kStagesK, i.e. for both tiles' softmax of
// key tile kt.  V scales share the V stage's life (released after both P V).
constexpr uint32_t kScaleStage = 8 * kBlockSize * 4;  // 512 B
constexpr int kScaleSlotsK = 2 * kStagesK;
constexpr uint32_t kOffScale = kOffXch + kRowTiles * kXchBytes;
constexpr uint32_t kSmemBytes = kOffScale + (kScaleSlotsK + kStagesV) * kScaleStage;
constexpr uint32_t kCodeOff = kOpBytes / 2;  // FP8 codes land in the upper half of a stage, then expand to bf16
constexpr uint32_t kCodeTile = kBlockSize * kHeadDim;  // 2 KB: one (block, head) tile of E4M3 codes
constexpr uint32_t kTmemCols = 512;  // S/P of tile t: [128t, 128t + 128); O of tile t: [256 + 128t, +128)
constexpr uint32_t kTmemO = 256;
static_assert(kSmemBytes <= 232448, "prefill shared memory exceeds the per-CTA limit");
static_assert(kNumBars <= 24, "barrier area");
static_assert(kOffScale % 16 == 0, "bulk copies land on 16-byte boundaries");

// Instruction descriptor, kind::f16: D f32, A/B bf16, M = 128, N = 128.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBase;               // A K-major, B K-major
constexpr uint32_t kIdescPV = kIdescBase | (1u << 16);  // B MN-major

// Two fp32 values from shared memory.
__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
    float2 r;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(r.x), "=f"(r.y) : "r"(addr));
    return r;
}

// Sixteen E4M3 codes (dims d .. d + 15) to bf16 (exact: E4M3 values are bf16
// values): w0 holds dims d .. d + 7, w1 dims d + 8 .. d + 15.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 &c, uint4 &w0, uint4 &w1) {
    auto two = [](uint32_t f16x2) {
        const float2 f = unpack_f16x2(f16x2);
        return pack_bf16x2(f.x, f.y);
    };
    uint32_t a, b;
    e4m3x4_to_f16x2x2(c.x, a, b);
    w0.x = two(a);
    w0.y = two(b);
    e4m3x4_to_f16x2x2(c.y, a, b);
    w0.z = two(a);
    w0.w = two(b);
    e4m3x4_to_f16x2x2(c.z, a, b);
    w1.x = two(a);
    w1.y = two(b);
    e4m3x4_to_f16x2x2(c.w, a, b);
    w1.z = two(a);
    w1.w = two(b);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled canonical layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// 32 consecutive output values of one row (v scaled by inv) straight to global
// memory in 16-byte stores; base is a multiple of 32 elements.
__device__ __forceinline__ void store_row(void *out, int32_t bf16, size_t base, const uint32_t (&v)[32], float inv) {
    auto f = [&](int i) { return __uint_as_float(v[i]) * inv; };
    if (bf16) {
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + base);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            o[c] = make_uint4(pack_bf16x2(f(8 * c), f(8 * c + 1)), pack_bf16x2(f(8 * c + 2), f(8 * c + 3)),
                              pack_bf16x2(f(8 * c + 4), f(8 * c + 5)), pack_bf16x2(f(8 * c + 6), f(8 * c + 7)));
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
#pragma unroll
        for (int c = 0; c < 8; ++c) o[c] = make_float4(f(4 * c), f(4 * c + 1), f(4 * c + 2), f(4 * c + 3));
    }
}

// The same 32 values (dims 64 * hc + 32 * q ..) into the staged output tile: boxes
// of 128 rows x 128 bytes (bf16: 64 dims, fp32: 32 dims), 16-byte chunk c of row
// r at chunk c ^ (r & 7) -- the layout the output tensor map's TMA store reads.
__device__ __forceinline__ void stage_row(uint32_t stage, int32_t bf16, int r, int hc, int q, const uint32_t (&v)[32],
                                          float inv) {
    auto f = [&](int i) { return __uint_as_float(v[i]) * inv; };
    if (bf16) {
        const uint32_t row = stage + hc * (128 * 128) + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((4 * q + c) ^ (r & 7)) << 4)),
                         "r"(pack_bf16x2(f(8 * c), f(8 * c + 1))), "r"(pack_bf16x2(f(8 * c + 2), f(8 * c + 3))),
                         "r"(pack_bf16x2(f(8 * c + 4), f(8 * c + 5))), "r"(pack_bf16x2(f(8 * c + 6), f(8 * c + 7)))
                         : "memory");
    } else {
        const uint32_t row = stage + (2 * hc + q) * (128 * 128) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ (r & 7)) << 4)), "f"(f(4 * c)),
                         "f"(f(4 * c + 1)), "f"(f(4 * c + 2)), "f"(f(4 * c + 3))
                         : "memory");
    }
}

// 608 threads, one CTA per SM (200 KB of shared memory); 19 warps put five on
// some SM sub-partition, whose 16K registers then allow 96 a thread.
// WINDOW: sliding-window instantiation (p.window > 0); the plain one compiles
// without any of the window's bookkeeping.  SPLIT: split-KV instantiation
// (p.kv_splits > 1: partials to the workspace for the merge kernel); the
// unsplit one compiles with one split as a constant.  (With the split count a
// runtime value in the unsplit kernel, ragged row tiles of multi-sequence
// batches came out wrong on the GPU -- rows written with other rows' values or
// not at all -- while the same source with the count constant, and the split
// path itself, matched the oracle; the cause was not found, so the unsplit
// kernel keeps the count constant.)  FP8: the cache holds E4M3 codes with
// per-slot scales (p.k_scale / p.v_scale): each block's 2 KB code tile lands in
// the upper half of a ring stage and the softmax warps expand it in place to the
// bf16 operand layout (E4M3 values are exact in bf16) between two key tiles'
// softmax passes; the K scale multiplies the scores and the V scale the weights
// that enter P V (the row sums keep the unscaled weights).
// P - head for a pair, head = the packed bf16 pair `h` (the low half goes with p.x):
// mixed-precision FMAs (bf16 operands, fp32 addend), exact since head is P truncated.
__device__ __forceinline__ float2 minus_bf16x2(float2 p, uint32_t h) {
    float2 d;
    asm("{\n\t.reg .b16 lo, hi, m;\n\tmov.b32 {lo, hi}, %2;\n\tmov.b16 m, 0xBF80;\n\t"
        "fma.rn.f32.bf16 %0, lo, m, %3;\n\tfma.rn.f32.bf16 %1, hi, m, %4;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(h), "f"(p.x), "f"(p.y));
    return d;
}

// OR of `pred` over the `nthreads` threads of named barrier `id` (a barrier as well).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %2, 0;\n\t"
        "barrier.cta.red.or.pred q, %1, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(static_cast<uint32_t>(pred)), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <bool WINDOW, bool FP8, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                         const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Grid (KV group, sequence, pair of row tiles x key split), pairs in reverse:
    // later rows see more keys, so the longest CTAs start first and the last wave
    // is short; the splits of a pair are adjacent.
    const int g = blockIdx.x;
    const int b = blockIdx.y;
    const int S = SPLIT ? p.kv_splits : 1;
    const int pair = static_cast<int>(gridDim.z) / S - 1 - static_cast<int>(blockIdx.z) / S;
    const int split = static_cast<int>(blockIdx.z) % S;
    const int G = p.group;
    const int rpt = p.rows_per_tile;

    if (tid == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        prefetch_tensormap(&omap);
    }
    griddep_launch_dependents();
    griddep_wait();  // the KV append (or any producer of q) before us on the stream
    if (sbase & 1023u) {  // operands need the 1 KB swizzle alignment
        if (tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        return;
    }

    // ---- sequence extent (device data: checked) ----
    const int row0 = p.cu_q_lens ? __ldg(p.cu_q_lens + b) : b * p.uniform_q_len;
    const int q_len = p.cu_q_lens ? __ldg(p.cu_q_lens + b + 1) - row0 : p.uniform_q_len;
    const int ctx = __ldg(p.context_lens + b);
    // Split-KV: this split's partial for rows [r_lo, r_hi) of the pair is empty
    // (m = -inf, l = 0, O = 0): the merge then gives those rows nothing from it.
    auto empty_partials = [&](int r_lo, int r_hi) {
        for (int idx = tid; idx < max(0, r_hi - r_lo) * G * 32; idx += kThreads) {
            const int i = r_lo + idx / (G * 32), h = (idx / 32) % G, c4 = idx % 32;
            const size_t pi = (static_cast<size_t>(row0 + i) * p.n_q + static_cast<size_t>(g) * G + h) * S + split;
            reinterpret_cast<float4 *>(p.part_o + pi * kHeadDim)[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 == 0) {
                p.part_m[pi] = -INFINITY;
                p.part_l[pi] = 0.f;
            }
        }
    };
    if (q_len < 0 || q_len > ctx || ctx > p.max_blocks * kBlockSize || row0 < 0 || row0 + q_len > p.total_rows) {
        if (pair == 0 && split == 0 && g == 0 && tid == 0 && p.status) atomicOr(p.status, kStatusBadQLen);
        // The sequence's rows read as zeros when they can be addressed (this CTA's
        // two row tiles of its KV group; 16-byte stores, out is 16-byte aligned).
        if (S > 1 && q_len > 0 && row0 >= 0 && row0 + q_len <= p.total_rows) {
            empty_partials(2 * pair * rpt, min(q_len, (2 * pair + 2) * rpt));
        } else if (q_len > 0 && row0 >= 0 && row0 + q_len <= p.total_rows) {
            const int r_lo = 2 * pair * rpt, r_hi = min(q_len, r_lo + 2 * rpt);
            const int chunks = p.out_bf16 ? 16 : 32;  // 16-byte chunks per (row, head)
            const int per_row = G * chunks;
            for (int idx = tid; idx < max(0, r_hi - r_lo) * per_row; idx += kThreads) {
                const int i = r_lo + idx / per_row, h = (idx % per_row) / chunks, c = idx % chunks;
                const size_t elem =
                    (static_cast<size_t>(row0 + i) * p.n_q + static_cast<size_t>(g) * G + h) * kHeadDim;
                reinterpret_cast<uint4 *>(static_cast<char *>(p.out) + elem * (p.out_bf16 ? 2 : 4))[c] =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }
    const int c = ctx - q_len;
    // Row tile t of the pair: rows i0(t) .. i0(t) + rows(t) - 1 (0 rows: past the
    // chunk), keys 0 .. c + i0(t) + rows(t) - 1, key tiles nt(t); nt(1) >= nt(0)
    // whenever tile 1 has rows.
    auto tile_i0 = [&](int t) { return (2 * pair + t) * rpt; };
    auto tile_rows = [&](int t) { return max(0, min(rpt, q_len - tile_i0(t))); };
    // Sliding window W: a row at position pos sees keys pos - W < j <= pos.  The
    // CTA's earliest row sees nothing before kfirst, so key tiles before kt0 are
    // never visited and blocks before fb are never read (their table entries may
    // be stale).  Key tiles are counted from kt0 below: loop index kt is key tile
    // kt0 + kt (keys 128 (kt0 + kt) ..).
    const int W = WINDOW ? p.window : 0;
    const int kfirst = W > 0 ? max(0, c + tile_i0(0) + 1 - W) : 0;
    int kt0 = kfirst / 128;
    const int fb = kfirst / kBlockSize;
    auto tile_nt = [&](int t) {
        return tile_rows(t) > 0 ? (c + tile_i0(t) + tile_rows(t) + 127) / 128 - kt0 : 0;
    };
    int nt0 = tile_nt(0), nt1 = tile_nt(1);
    int n_tiles = max(nt0, nt1);
    if (S > 1) {
        // This split's key tiles [ks, ke) of the pair's n_tiles; counted from kt0 + ks below.
        const int per = (n_tiles + S - 1) / S;
        const int ks = min(n_tiles, split * per), ke = min(n_tiles, ks + per);
        nt0 = max(0, min(nt0, ke) - ks);
        nt1 = max(0, min(nt1, ke) - ks);
        kt0 += ks;
        n_tiles = max(nt0, nt1);
        if (n_tiles == 0) {
            empty_partials(tile_i0(0), tile_i0(0) + tile_rows(0) + tile_rows(1));
            return;
        }
    }
    if (n_tiles == 0) return;
    const int nblocks = (ctx + kBlockSize - 1) / kBlockSize;
    const int32_t *table = p.block_tables + static_cast<size_t>(b) * p.max_blocks;

    const uint32_t bar_q = sbase + kOffBar;
    // K slot kt % kStagesK (use kt / kStagesK), V slot kt % kStagesV; per tile t: S, P and O barriers.
    auto k_full = [&](int st) { return sbase + kOffBar + 8 * (1 + st); };
    auto k_empty = [&](int st) { return sbase + kOffBar + 8 * (1 + kStagesK + st); };
    auto v_full = [&](int st) { return sbase + kOffBar + 8 * (1 + 2 * kStagesK + st); };
    auto v_empty = [&](int st) { return sbase + kOffBar + 8 * (1 + 2 * kStagesK + kStagesV + st); };
    auto s_full = [&](int t) { return sbase + kOffBar + 8 * (kBarTile + t); };
    auto p_full = [&](int t) { return sbase + kOffBar + 8 * (kBarTile + kRowTiles + t); };
    auto o_done = [&](int t) { return sbase + kOffBar + 8 * (kBarTile + 2 * kRowTiles + t); };
    auto k_conv = [&](int st) { return sbase + kOffBar + 8 * (kBarConv + st); };  // FP8: K stage in bf16
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + kOffAbort);

    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int st = 0; st < kStagesK; ++st) {
            mbar_init(k_full(st), 1);
            mbar_init(k_empty(st), 1);
        }
        for (int st = 0; st < kStagesV; ++st) {
            mbar_init(v_full(st), 1);
            mbar_init(v_empty(st), 1);
        }
        for (int t = 0; t < kRowTiles; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), kSoftmaxWarps);
            mbar_init(o_done(t), 1);
        }
        for (int st = 0; st < kStagesK; ++st) mbar_init(k_conv(st), kSoftmaxWarps);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // A bounded wait that gives up at once after another role gave up.
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity)) return true;
        *abort_flag = 1u;
        return false;
    };
    // The same for a whole warp: lane 0 polls (one poller per warp keeps the
    // barrier words free for the copies' transaction updates), the warp barrier
    // hands its view of memory to the other lanes.
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
        bool ok = false;
        if (lane == 0) ok = wait(bar, parity);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        return ok;
    };

    if (warp == kProducerK || warp == kProducerV) {
        // ---------------- TMA producers: warp 16 fills the K ring, warp 18 the V ring ----------------
        const bool is_k = warp == kProducerK;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t ring = sbase + (is_k ? kOffK : kOffV);
        const int stages = is_k ? kStagesK : kStagesV;
        if (is_k && lane == 0) {  // both Q tiles (rows past the chunk read as zeros or are never stored)
            mbar_arrive_expect_tx(bar_q, kRowTiles * kOpBytes);
            for (int t = 0; t < kRowTiles; ++t) {
                tma_load_3d(sbase + kOffQ + t * kOpBytes, &qmap, bar_q, 0, g * G, row0 + tile_i0(t));
                tma_load_3d(sbase + kOffQ + t * kOpBytes + kHalfTile, &qmap, bar_q, 64, g * G, row0 + tile_i0(t));
            }
        }
        // (block, head) tile index of key tile kt's t-th paged block, read by lane t
        // (one parallel load per tile); invalid ids and blocks before the window
        // fetch tile 0 and are masked.
        auto tile_index = [&](int kt) -> int {
            const int jb = (kt0 + kt) * 8 + lane;
            int mine = 0;
            if (lane < 8 && (!WINDOW || jb >= fb) && jb < nblocks) {
                mine = __ldg(table + jb);
                if (static_cast<unsigned>(mine) >= static_cast<unsigned>(p.num_blocks)) mine = 0;
            }
            return mine * p.n_kv + g;
        };
        // All lanes walk the schedule (lane 0 waits for the warp); lane t
        // issues block t.  The next tile's table entries are read before this tile's wait.
        int next = tile_index(0);
        for (int kt = 0; kt < n_tiles; ++kt) {
            const int mine = next;
            if (kt + 1 < n_tiles) next = tile_index(kt + 1);
            const int st = kt % stages;
            if (kt >= stages &&
                !warp_wait(is_k ? k_empty(st) : v_empty(st), ((kt / stages) - 1) & 1))
                break;
            const uint32_t bar = is_k ? k_full(st) : v_full(st);
            const uint32_t dst = ring + st * kOpBytes;
            const int nload = min(8, nblocks - (kt0 + kt) * 8);
            if constexpr (FP8) {
                // Block t's 2 KB code tile (one box: 128 codes x 16 slots, 128-byte swizzle) into the
                // stage's upper half, and its 64 B of scales into the key tile's scale slot (K: slot
                // kt % kScaleSlotsK of the deeper K-scale ring; V: the V stage's slot).
                if (lane == 0) mbar_arrive_expect_tx(bar, nload * (kCodeTile + kBlockSize * 4));
                __syncwarp();
                if (lane < nload) {
                    const int phys = mine / p.n_kv;
                    tma_load_4d(dst + kCodeOff + lane * kCodeTile, map, bar, 0, 0, g, phys);
                    const float *sc = is_k ? p.k_scale : p.v_scale;
                    const int slot = is_k ? kt % kScaleSlotsK : kScaleSlotsK + st;
                    bulk_copy_g2s(sbase + kOffScale + slot * kScaleStage + lane * 64,
                                  sc + (static_cast<size_t>(phys) * p.n_kv + g) * kBlockSize, 64, bar);
                }
            } else {
                if (lane == 0) mbar_arrive_expect_tx(bar, nload * kBlkBytes);
                __syncwarp();
                if (lane < nload) tma_load_5d(dst + lane * kBlkBytes, map, bar, 0, 0, 0, 0, mine);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer: S0(k), P1(k-1) V(k-1), S1(k), P0(k) V(k) ----------------
        if (lane == 0) {
            auto mma_s = [&](int t, int kt) {
                const uint32_t kb = sbase + kOffK + (kt % kStagesK) * kOpBytes;
                const uint32_t qb = sbase + kOffQ + t * kOpBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // 16 dims per step: dim half kk / 4, 32 B into the row
                    const uint32_t qoff = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
                    umma_bf16(tmem + 128 * t, sw128_desc(qb + qoff, 16, 1024), sw128_desc(kb + koff, 16, 2048),
                              kIdescQK, kk > 0);
                }
                umma_commit(s_full(t));
            };
            auto mma_pv = [&](int t, int kt) {
                const uint32_t vb = sbase + kOffV + (kt % kStagesV) * kOpBytes;
#pragma unroll
                for (int s8 = 0; s8 < 8; ++s8) {
                    // keys 16 s8 .. +15: half s8 / 4, 32-key chunk (s8 / 2) % 2, [16 head | 16 remainder] columns
                    const uint32_t a_hi = tmem + 128 * t + (s8 >> 2) * 64 + ((s8 >> 1) & 1) * 32 + (s8 & 1) * 8;
                    const uint64_t bd = sw128_desc(vb + s8 * kBlkBytes, 1024, 2048);
                    umma_bf16_tmem_a(tmem + kTmemO + 128 * t, a_hi, bd, kIdescPV, (kt > 0 || s8 > 0) ? 1u : 0u);
                    umma_bf16_tmem_a(tmem + kTmemO + 128 * t, a_hi + 16, bd, kIdescPV, 1u);
                }
                umma_commit(o_done(t));
            };
            bool ok = wait(bar_q, 0);
            for (int kt = 0; ok && kt <= n_tiles; ++kt) {
                const int st_k = kt % kStagesK, st_v = kt % kStagesV;
                // K(kt) waited for (just before the first S that reads it).  bf16: only K(0)
                // here; for kt > 0 the P barrier of key tile kt - 1 that this thread waited
                // for already covers K(kt), since softmax warp 0 checks it before its pass
                // (every wait here drains the tensor pipe for about 115 cycles).  A P
                // barrier also covers its key tile's V: bf16, by the same check; FP8,
                // because every softmax warp expands its share of V(kt) (and fences it for
                // the tensor core) before its pass over key tile kt.
                bool k_ready = false;
                auto need_k = [&]() -> bool {
                    if (!k_ready) {
                        if ((FP8 || kt == 0) && !wait(FP8 ? k_conv(st_k) : k_full(st_k), (kt / kStagesK) & 1))
                            return false;
                        tc_fence_after();
                        k_ready = true;
                    }
                    return true;
                };
                if (kt < nt0) {
                    if (!(ok = need_k())) break;
                    mma_s(0, kt);
                }
                if (kt >= 1 && kt - 1 < nt1) {  // tile 1's P V of the previous key tile
                    const int pk = kt - 1;
                    if (!(ok = wait(p_full(1), pk & 1))) break;
                    tc_fence_after();
                    mma_pv(1, pk);
                    umma_commit(v_empty(pk % kStagesV));  // both tiles' P V of key tile pk are issued
                }
                if (kt < nt1) {
                    if (!(ok = need_k())) break;
                    mma_s(1, kt);
                }
                if (kt < n_tiles) umma_commit(k_empty(st_k));  // both tiles' S of key tile kt are issued
                if (kt < nt0) {
                    if (!(ok = wait(p_full(0), kt & 1))) break;
                    tc_fence_after();
                    mma_pv(0, kt);
                    if (kt >= nt1) umma_commit(v_empty(st_v));  // tile 1 does not read this key tile
                }
            }
        }
    } else {
        // ---------------- softmax warps: both tiles in turn; one row and one column quarter per thread ----------------
        // (every wait decision is made warp-uniform, so the .sync.aligned tensor-memory
        // loads and stores below always see the full warp)
        const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31 (warp % 4 == quarter)
        const int cq = warp >> 2;      // column quarter: keys / O dims [32*cq, 32*cq + 32)
        const int r = quarter * 32 + lane;
        const int ii = r / G;
        const float sl2 = p.scale_log2;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float *xch = reinterpret_cast<float *>(smem + kOffXch);  // [tile][key tile & 1][quarter][row]; then row sums
        const uint32_t row_bar = 1 + quarter;  // named barriers 1..4: the four warps of a row quarter
        auto row_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(row_bar) : "memory"); };

        // Per tile: the row's last visible key, running exponent reference and row-sum share.
        int limit[kRowTiles], first[kRowTiles];
        float m_ref[kRowTiles], l[kRowTiles];
        // The vote (plain chunk and window, bf16, unsplit): up to key tile exact_until[t]
        // some row of tile t has no reference yet, so those passes take the row maximum
        // directly (CTA-uniform): the first key tile, or under a window the key tile
        // where the tile's last row's window starts.
        constexpr bool kVote = !FP8 && !SPLIT;
        int exact_until[kRowTiles];
#pragma unroll
        for (int t = 0; t < kRowTiles; ++t) {
            const int pos = c + tile_i0(t) + (ii < tile_rows(t) ? ii : 0);
            limit[t] = min(pos, ctx - 1);                  // visible keys: first <= j <= limit
            first[t] = WINDOW ? max(0, pos + 1 - W) : 0;
            m_ref[t] = -INFINITY;
            l[t] = 0.f;
            exact_until[t] = WINDOW ? max(0, c + tile_i0(t) + tile_rows(t) - W) / 128 - kt0 : 0;
        }

        // The four warps of a row quarter pass exactly one row barrier per (key tile,
        // tile) and two per tile in the epilogue on every path: after a wait gives up
        // (`alive` false) the loops keep turning without work, so the named barriers
        // always match and never hang.
        bool alive = true;
        // FP8: key tile kx's K (is_v false) or V codes, once landed, expanded in place to
        // the bf16 operand layout by all 512 softmax threads (a CTA-uniform call): each
        // thread takes two 16-code chunks of a slot row (chunk c: block c / 128, slot
        // (c / 8) % 16, dims 16 (c % 8) ..), reads them, and after a barrier over all
        // softmax warps (so every code is read before any bf16 overwrites it) writes
        // them as two swizzled 16-byte bf16 chunks.  V rows no row may see (past the
        // context, of an invalid block or of a block before the window) become zeros,
        // and so do their V scales (before the barrier, so every later reader sees
        // it): a masked key then enters P V with weight p * 0 = 0 whatever stale or
        // uninitialised scale its slot held.
        auto expand = [&](bool is_v, int kx) {
            const int stages = is_v ? kStagesV : kStagesK;
            const int st = kx % stages;
            const uint32_t stage = sbase + (is_v ? kOffV : kOffK) + st * kOpBytes;
            const bool ok = alive && warp_wait(is_v ? v_full(st) : k_full(st), (kx / stages) & 1);
            uint32_t zmask = 0;
            int rvx = 128;
            if (is_v) {
                const int jb = (kt0 + kx) * 8 + lane;
                const bool bad_lane = lane < 8 && (!WINDOW || jb >= fb) && jb < nblocks &&
                                      static_cast<unsigned>(__ldg(table + jb)) >= static_cast<unsigned>(p.num_blocks);
                zmask = __ballot_sync(0xffffffffu, bad_lane);
                if constexpr (WINDOW) zmask |= (1u << min(8, max(0, fb - (kt0 + kx) * 8))) - 1u;
                rvx = ctx - (kt0 + kx) * 128;
            }
            uint4 cd[2];
            bool zero[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int cc = tid + i * kSoftmaxWarps * 32;
                const int blk = cc >> 7, sl = (cc >> 3) & 15, ch = cc & 7;
                zero[i] = is_v && (blk * 16 + sl >= rvx || ((zmask >> blk) & 1u));
                cd[i] = make_uint4(0u, 0u, 0u, 0u);
                if (ok && !zero[i]) cd[i] = lds128(stage + kCodeOff + blk * kCodeTile + sl * 128 + ((ch ^ (sl & 7)) << 4));
                if (ok && zero[i] && ch == 0)
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kOffScale + (kScaleSlotsK + st) * kScaleStage +
                                                                  (blk * kBlockSize + sl) * 4),
                                 "f"(0.f)
                                 : "memory");
            }
            asm volatile("bar.sync 10, %0;" ::"r"(kSoftmaxWarps * 32) : "memory");
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int cc = tid + i * kSoftmaxWarps * 32;
                const int blk = cc >> 7, sl = (cc >> 3) & 15, ch = cc & 7;
                uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
                if (!zero[i]) e4m3x16_to_bf16(cd[i], w0, w1);
                const int s8 = sl & 7, j0 = 2 * (ch & 3);
                const uint32_t row = stage + blk * kBlkBytes + (sl >> 3) * 2048 + (ch >> 2) * 1024 + s8 * 128;
                if (ok) {
                    sts128(row + ((j0 ^ s8) << 4), w0);
                    sts128(row + (((j0 + 1) ^ s8) << 4), w1);
                }
            }
            fence_proxy_async_smem();  // generic stores -> the tensor core (async proxy)
            __syncwarp();
            if (ok && lane == 0 && !is_v) mbar_arrive(k_conv(st));
            alive = ok;
        };
        if constexpr (FP8) {
            expand(false, 0);
            expand(true, 0);
        }
        for (int kt = 0; kt < n_tiles; ++kt) {
            // Which of this key tile's blocks have an invalid id (flagged) or lie wholly
            // before the window (never read): their keys are masked.  Lane j < 8
            // checks block j, a ballot shares the answer.
            const int jb = (kt0 + kt) * 8 + lane;
            const bool bad_lane = lane < 8 && (!WINDOW || jb >= fb) && jb < nblocks &&
                                  static_cast<unsigned>(__ldg(table + jb)) >= static_cast<unsigned>(p.num_blocks);
            const uint32_t invalid = __ballot_sync(0xffffffffu, bad_lane);
            if (invalid && tid == 0 && p.status) atomicOr(p.status, kStatusBadBlockId);
            uint32_t bad = invalid;
            if constexpr (WINDOW) bad |= (1u << min(8, max(0, fb - (kt0 + kt) * 8))) - 1u;
            const int kc = (kt0 + kt) * 128 + 32 * cq;  // first key of this thread's chunk
            const int rv = ctx - (kt0 + kt) * 128;      // keys [rv, 128) of the key tile are past the context

#pragma unroll
            for (int t = 0; t < kRowTiles; ++t) {
                // FP8: the next key tile's K right after tile 0's pass (S0(kt+1) waits for it).
                if constexpr (FP8) {
                    if (t == 1 && kt + 1 < n_tiles) expand(false, kt + 1);
                }
                if (kt >= (t == 0 ? nt0 : nt1)) continue;  // (CTA-uniform)
                // bf16: before its pass over S_t(kt) (while the MMAs still run), warp 0 checks that
                // V(kt) and K(kt + 1) have landed, so that the P barrier it arrives on covers
                // them and the MMA thread does not wait for copies itself.
                if (!FP8 && warp == 0)
                    alive = alive && warp_wait(v_full(kt % kStagesV), (kt / kStagesV) & 1) &&
                            (kt + 1 >= n_tiles ||
                             warp_wait(k_full((kt + 1) % kStagesK), ((kt + 1) / kStagesK) & 1));
                const bool exact = !kVote || kt <= exact_until[t];  // (CTA-uniform)
                alive = alive && warp_wait(s_full(t), kt & 1);
                if (!alive) {  // (the exchange -- and the vote before it -- of the other warps)
                    if (!exact) bar_red_or(row_bar, 128, true);
                    row_sync();
                    continue;
                }
                tc_fence_after();
                const uint32_t t_s = lane_base + 128 * t + 32 * cq;
                const uint32_t t_o = lane_base + kTmemO + 128 * t + 32 * cq;
                float *xm = xch + ((t * 2 + (kt & 1)) * 4) * 128;

                // This thread's 32 scores, masked by index (keys past the row's position or in a bad block).
                auto load_scores = [&](uint32_t(&vv)[32]) {
                    tmem_ld_32x32b_x32(t_s, vv);
                    if constexpr (FP8) {  // scores times each key's K scale
                        const uint32_t ks = sbase + kOffScale + (kt % kScaleSlotsK) * kScaleStage + 128 * cq;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint4 w = lds128(ks + 16 * i);
                            const float2 a = fmul2(make_float2(__uint_as_float(vv[4 * i]), __uint_as_float(vv[4 * i + 1])),
                                                   make_float2(__uint_as_float(w.x), __uint_as_float(w.y)));
                            const float2 c = fmul2(make_float2(__uint_as_float(vv[4 * i + 2]), __uint_as_float(vv[4 * i + 3])),
                                                   make_float2(__uint_as_float(w.z), __uint_as_float(w.w)));
                            vv[4 * i] = __float_as_uint(a.x);
                            vv[4 * i + 1] = __float_as_uint(a.y);
                            vv[4 * i + 2] = __float_as_uint(c.x);
                            vv[4 * i + 3] = __float_as_uint(c.y);
                        }
                    }
                    if (!(kc + 31 <= limit[t] && (!WINDOW || kc >= first[t]) && !((bad >> (2 * cq)) & 3u))) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const bool ok = kc + k <= limit[t] && (!WINDOW || kc + k >= first[t]) &&
                                            !((bad >> ((32 * cq + k) >> 4)) & 1u);
                            if (!ok) vv[k] = __float_as_uint(-INFINITY);
                        }
                    }
                };
                uint32_t v[32];
                load_scores(v);
                // The exponent reference m: raised to the exact row maximum (exchanged between
                // the four warps of the row quarter; O and l rescaled) when that maximum passes
                // it by more than 2^8 -- also at the first visible key (m_ref = -inf).
                float alpha = 1.f;
                auto raise_reference = [&](const uint32_t(&vv)[32]) {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int k = 0; k < 32; k += 2)
                        mx[(k >> 1) & 3] = fmax3(mx[(k >> 1) & 3], __uint_as_float(vv[k]), __uint_as_float(vv[k + 1]));
                    xm[cq * 128 + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                    row_sync();
                    const float mraw = fmaxf(fmaxf(xm[r], xm[128 + r]), fmaxf(xm[256 + r], xm[384 + r]));
                    const float mt = mraw == -INFINITY ? -INFINITY : mraw * sl2;  // scale > 0 keeps the order
                    if (mt > m_ref[t] + 8.f) {
                        alpha = fast_exp2(m_ref[t] - mt);  // 0 when m_ref = -inf
                        m_ref[t] = mt;
                    }
                    // Rescale O: every earlier P V of this tile completed before S(kt) did.
                    if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        uint32_t orow[32];
                        tmem_ld_32x32b_x32(t_o, orow);
#pragma unroll
                        for (int k = 0; k < 32; ++k) orow[k] = __float_as_uint(__uint_as_float(orow[k]) * alpha);
                        tmem_st_32x32b_x32(t_o, orow);
                    }
                };
                // P = 2^(s * scale * log2(e) - m) and this thread's share of the row sum.
                const float2 sl2v = make_float2(sl2, sl2);
                float2 pr2[16];
                auto weights = [&](const uint32_t(&vv)[32]) -> float {
                    const float mu = m_ref[t] == -INFINITY ? 0.f : m_ref[t];
                    const float2 nmu = make_float2(-mu, -mu);
                    float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 x =
                            ffma2(make_float2(__uint_as_float(vv[2 * e]), __uint_as_float(vv[2 * e + 1])), sl2v, nmu);
                        pr2[e] = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        if (e & 1)
                            rs1 = fadd2(rs1, pr2[e]);
                        else
                            rs0 = fadd2(rs0, pr2[e]);
                    }
                    const float2 rs = fadd2(rs0, rs1);
                    return rs.x + rs.y;
                };
                float rsum;
                // The FP8 and split instantiations take the exact maximum every pass (the split
                // kernel spills with the vote's live weights, 294 -> 322 us on the 70B verify;
                // FP8 measured slower with the vote, 95.7 -> 97.8 us).
                if (exact) {
                    raise_reference(v);
                    rsum = weights(v);
                } else {
                    // The weights against the current reference first; the maximum is
                    // taken and exchanged only when a thread's 32 weights sum past 2^8 (then
                    // some weight may exceed 2^8) or the row has no reference yet -- one vote
                    // per pass instead of a maximum over every key and an exchange, which
                    // leaves the integer pipe to the MMA thread (mixed chunk 68.8 -> 66.4 us).
                    bool need = m_ref[t] == -INFINITY;
                    rsum = 0.f;
                    if (!need) {
                        rsum = weights(v);
                        need = !(rsum <= 256.f);
                    }
                    if (bar_red_or(row_bar, 128, need)) {
                        uint32_t v2[32];  // S is still in tensor memory: reloaded, so v dies above
                        load_scores(v2);
                        raise_reference(v2);
                        rsum = weights(v2);
                    }
                }

                // P written back over the chunk's 32 columns as [16 columns bf16 head | 16
                // columns bf16 remainder] (two keys per column, the lower key in the low
                // half); pairs of keys go through packed f32x2 arithmetic.
                uint32_t pk[32];  // [16 columns of heads | 16 columns of remainders], one store
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 pr = pr2[e];
                    // FP8: the weights entering P V carry each key's V scale (a masked key's
                    // scale was zeroed by the expansion); the row sums keep the plain weights.
                    float2 pw = pr;
                    if constexpr (FP8) {
                        const float2 sv =
                            lds_f32x2(sbase + kOffScale + (kScaleSlotsK + kt % kStagesV) * kScaleStage + 128 * cq + 8 * e);
                        pw = fmul2(pr, sv);
                    }
                    // head: the upper 16 bits of each (bf16 truncation, exact in fp32);
                    // remainder: P - head >= 0 (exact in fp32), rounded to nearest bf16.
                    // (remainder by mixed-precision FMAs instead of masks and a subtraction:
                    // no integer work, 65.2 -> 64.1 us on the mixed chunk)
                    pk[e] = __byte_perm(__float_as_uint(pw.x), __float_as_uint(pw.y), 0x7632);
                    const float2 rr = minus_bf16x2(pw, pk[e]);
                    pk[16 + e] = pack_bf16x2(rr.x, rr.y);
                }
                tmem_st_32x32b_x32(t_s, pk);  // (one store instead of two: 69.9 -> 69.0 us on the mixed chunk)
                tmem_wait_st();
                l[t] = l[t] * alpha + rsum;

                // Zero V rows of keys no row may see (past the context, of a bad block or
                // of a block before the window), once per key tile, by the first tile that
                // reads it, before its P V.
                if (!FP8 && (rv < 128 || bad) && t == (kt < nt0 ? 0 : 1)) {  // (FP8: done by expand)
                    alive = warp_wait(v_full(kt % kStagesV), (kt / kStagesV) & 1);
                    if (!alive) continue;
                    const uint32_t vb = sbase + kOffV + (kt % kStagesV) * kOpBytes;
                    for (int idx = tid; idx < 128 * 16; idx += kSoftmaxWarps * 32) {
                        const int key = idx >> 4, ch = idx & 15;  // (all 16 chunks of a row: swizzle is moot)
                        if (key >= rv || ((bad >> (key >> 4)) & 1u)) {
                            const uint32_t addr = vb + (key >> 4) * kBlkBytes + ((key >> 3) & 1) * 2048 +
                                                  (ch >> 3) * 1024 + (key & 7) * 128 + (ch & 7) * 16;
                            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                        }
                    }
                    fence_proxy_async_smem();  // zeroed V rows -> the tensor core (async proxy)
                }
                // (P itself goes through tensor memory: the tcgen05 fence below orders it; the
                // proxy fence costs 150-350 cycles per pass, so only passes that zeroed V rows
                // pay it; FP8 fences its expansions where it writes them.)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            // FP8: the next key tile's V (every warp's share is written before its P arrivals
            // for key tile kt + 1, which the P V MMAs of that key tile wait for).
            if constexpr (FP8) {
                if (kt + 1 < n_tiles) expand(true, kt + 1);
            }
        }

        // ---- epilogue per tile: out = O / l (the four column quarters add their row sums) ----
        // A full tile is staged in a free ring for a TMA store.  When both tiles end at the
        // same key tile, tile 0's epilogue runs while tile 1's last P V is still in the
        // pipe: tile 0 is staged in the K ring (free once tile 0's last P V completed,
        // since every S was issued before it), tile 1 in the V ring after its own last P V.
        // Otherwise both tiles' last P V first (tile 0: the V ring, tile 1: the K ring).
        const bool early = nt0 == nt1;  // CTA-uniform
        bool done = alive;
        // both tiles' row sums, added over the four column quarters through shared memory
        row_sync();  // the last maxima have been read: the exchange area is free
        xch[cq * 128 + r] = l[0];
        xch[512 + cq * 128 + r] = l[1];
        row_sync();
        if (!early) {
            if (nt0 > 0) done = done && warp_wait(o_done(0), (nt0 - 1) & 1);
            if (nt1 > 0) done = done && warp_wait(o_done(1), (nt1 - 1) & 1);
        }
#pragma unroll 1
        for (int t = 0; t < kRowTiles; ++t) {
            const int my_nt = t == 0 ? nt0 : nt1;
            if (early && my_nt > 0) done = done && warp_wait(o_done(t), (my_nt - 1) & 1);
            const int i0 = tile_i0(t);
            const int rows_here = tile_rows(t);
            const bool row_valid = ii < rows_here;
            const bool staged = S == 1 && rows_here == rpt;  // CTA-uniform
            const uint32_t stage = sbase + ((t == 0) != early ? kOffV : kOffK);
            // Split-KV: row (row0 + i0 + ii, head g G + r % G)'s partial of this split.
            auto part_index = [&]() {
                return (static_cast<size_t>(row0 + i0 + ii) * p.n_q + static_cast<size_t>(g) * G + (r % G)) * S + split;
            };
            if (S > 1 && my_nt == 0 && row_valid) {  // no key tile of this split reaches the tile
                const size_t pi = part_index();
                float4 *po = reinterpret_cast<float4 *>(p.part_o + pi * kHeadDim + 32 * cq);
#pragma unroll
                for (int k = 0; k < 8; ++k) po[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cq == 0) {
                    p.part_m[pi] = -INFINITY;
                    p.part_l[pi] = 0.f;
                }
            }
            if (my_nt > 0 && done) {
                tc_fence_after();
                const float *xl = xch + 512 * t;
                const float lt = (xl[r] + xl[128 + r]) + (xl[256 + r] + xl[384 + r]);
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                uint32_t orow[32];
                tmem_ld_32x32b_x32(lane_base + kTmemO + 128 * t + 32 * cq, orow);
                if (S > 1) {
                    // the unnormalised partial: O and l relative to the row's exponent reference m
                    if (row_valid) {
                        const size_t pi = part_index();
                        float4 *po = reinterpret_cast<float4 *>(p.part_o + pi * kHeadDim + 32 * cq);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            po[k] = make_float4(__uint_as_float(orow[4 * k]), __uint_as_float(orow[4 * k + 1]),
                                                __uint_as_float(orow[4 * k + 2]), __uint_as_float(orow[4 * k + 3]));
                        if (cq == 0) {
                            p.part_m[pi] = m_ref[t];
                            p.part_l[pi] = lt;
                        }
                    }
                } else if (staged) {
                    stage_row(stage, p.out_bf16, r, cq >> 1, cq & 1, orow, inv);
                } else if (row_valid) {
                    const size_t base =
                        (static_cast<size_t>(row0 + i0 + ii) * p.n_q + static_cast<size_t>(g) * G + (r % G)) *
                            kHeadDim +
                        32 * cq;
                    store_row(p.out, p.out_bf16, base, orow, inv);
                }
            }
            if (staged) {
                // Every softmax warp reaches this barrier on every path (staged is CTA-uniform).
                fence_proxy_async_smem();
                asm volatile("bar.sync 9, %0;" ::"r"(kSoftmaxWarps * 32) : "memory");
                if (tid == 0 && !*abort_flag) {
                    const int nbox = p.out_bf16 ? 2 : 4;
#pragma unroll 1
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_store_3d(&omap, stage + bx * kHalfTile, bx * (p.out_bf16 ? 64 : 32), g * G, row0 + i0);
                    bulk_commit_group();
                    bulk_wait_group_read_all();  // shared memory must outlive the reads
                }
            }
        }
    }

    // ---- teardown: every role is done (or gave up); free tensor memory ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag) {
        if (tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
        // Best effort: let MMAs still in flight finish before the columns are freed.
        if (warp == kMmaWarp && lane == 0) {
            if (nt0 > 0) mbar_wait(o_done(0), (nt0 - 1) & 1);
            if (nt1 > 0) mbar_wait(o_done(1), (nt1 - 1) & 1);
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes; }

template <bool WINDOW, bool FP8>
cudaError_t prepare_pair(int smem) {
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_kernel<WINDOW, FP8, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(prefill_chunk_kernel<WINDOW, FP8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
}

cudaError_t prefill_prepare_device() {
    const int smem = static_cast<int>(kSmemBytes);
    cudaError_t e = prepare_pair<false, false>(smem);
    if (e == cudaSuccess) e = prepare_pair<true, false>(smem);
    if (e == cudaSuccess) e = prepare_pair<false, true>(smem);
    if (e == cudaSuccess) e = prepare_pair<true, true>(smem);
    return e;
}

cudaError_t launch_prefill_chunk(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const CUtensorMap &omap, const PrefillParams &p, int max_q_len, cudaStream_t stream) {
    // One CTA per pair of row tiles and key split.
    const int tiles = (max_q_len + p.rows_per_tile - 1) / p.rows_per_tile;
    const dim3 grid(p.n_kv, p.num_seqs, (tiles + 1) / 2 * p.kv_splits);
    const bool fp8 = p.k_scale != nullptr;
    const bool split = p.kv_splits > 1;
    auto kernel = split ? (p.window > 0 ? (fp8 ? prefill_chunk_kernel<true, true, true>
                                               : prefill_chunk_kernel<true, false, true>)
                                        : (fp8 ? prefill_chunk_kernel<false, true, true>
                                               : prefill_chunk_kernel<false, false, true>))
                        : (p.window > 0 ? (fp8 ? prefill_chunk_kernel<true, true, false>
                                               : prefill_chunk_kernel<true, false, false>)
                                        : (fp8 ? prefill_chunk_kernel<false, true, false>
                                               : prefill_chunk_kernel<false, false, false>));
    cudaError_t e = launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, stream, qmap, kmap, vmap, omap, p);
    if (e != cudaSuccess || p.kv_splits <= 1) return e;
    // The splits' partials, folded per (row, query head) by the decode path's merge kernel.
    DecodeParams m{};
    m.out = p.out;
    m.context_lens = p.context_lens;
    m.part_m = p.part_m;
    m.part_l = p.part_l;
    m.part_o = p.part_o;
    m.n_q = p.n_q;
    m.max_parts = p.kv_splits;
    m.out_bf16 = p.out_bf16;
    return launch_merge(m, p.total_rows, 1, p.kv_splits, stream);
}

}  // namespace pkv
