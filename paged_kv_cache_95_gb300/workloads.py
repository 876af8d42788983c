"""Seeded synthetic workloads for paged KV-cache attention.

This module only *constructs inputs*: random bf16 values, context lengths,
the placement of logical KV blocks in a physical block pool, the block tables
and the slot numbers at which the new tokens' K/V are to be appended.  It holds
none of the attention arithmetic and is shared by the CUDA path, the oracle and
the benchmark, so that both sides consume identical bit patterns.

Shapes and structure follow the five workloads used for parity and
measurement (head_dim 128, 16-token blocks, bf16 K/V/q ~ N(0,1)):

* ``tiny``            B=2, 32/8 heads, contexts {10, 17}, 16-block pool whose
                      physical blocks are randomly permuted; 2 appended tokens.
* ``llama3_8b_b64``   B=64, 32/8 heads, contexts ~ U[512, 4096], pool sized
                      1.2x the blocks needed, tables randomly scattered.
* ``sweep_mha`` / ``sweep_gqa`` / ``sweep_mqa``
                      B=32, context 2048, 32 query heads over 32 / 8 / 1 KV
                      heads, identical seeded q for the three variants.
* ``llama3_70b_b8_32k`` / ``llama3_70b_b1_128k``
                      64/8 heads; B=8 at 32768 and B=1 at 131072.
* ``mixed``           32/8 heads; 4 sequences with a 512-token causal chunk
                      over 1024 cached tokens, 60 decodes with contexts
                      ~ U[256, 8192] of which 16 share one 1024-token prefix
                      (64 identical physical blocks).

Layouts (the pages fix none; PagedAttention only changes the layout, see
"LLM 推理全过程的维度变化与核心公式", section "KV Cache 的形状与增长"):

* k_cache, v_cache : uint16 (bf16 bits) [num_blocks, n_kv, block_size, head_dim]
* block_tables     : int32 [B, max_blocks]; entries past ceil(ctx/16) hold the
                     id of a NaN-filled block that must never be read
* context_lens     : int32 [B]; includes the tokens appended in this step
* q                : uint16 [rows, n_q, head_dim]; cu_q_lens int32 [B+1]
* new_key/new_value: uint16 [T_new, n_kv, head_dim]; slot_mapping int32 [T_new]

Before the append, every pool slot that no sequence owns, and every slot that
the append is about to fill, holds bf16 NaN, so a kernel that reads a slot it
should not (or reads a slot before the append wrote it) produces NaN.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

HEAD_DIM = 128
BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)

WORKLOAD_NAMES = (
    "tiny",
    "llama3_8b_b64",
    "sweep_mha",
    "sweep_gqa",
    "sweep_mqa",
    "llama3_70b_b8_32k",
    "llama3_70b_b1_128k",
    "mixed",
)

# Seed = 1000 + index of the workload family (tiny=0 ... mixed=4).
_FAMILY_SEED = {
    "tiny": 1000,
    "llama3_8b_b64": 1001,
    "sweep_mha": 1002,
    "sweep_gqa": 1002,
    "sweep_mqa": 1002,
    "llama3_70b_b8_32k": 1003,
    "llama3_70b_b1_128k": 1003,
    "mixed": 1004,
}


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    big = u > np.uint32(0xFFFF7FFF)  # (negative NaNs) the 32-bit sum would wrap: redo those in 64 bits
    if big.any():
        w = u[big].astype(np.uint64)
        r[big] = ((w + 0x7FFF + ((w >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class Batch:
    """The sequences of one attention call (decode or chunked prefill)."""

    q: np.ndarray  # uint16 [rows, n_q, d]
    cu_q_lens: np.ndarray  # int32 [B+1]
    block_tables: np.ndarray  # int32 [B, max_blocks]
    context_lens: np.ndarray  # int32 [B]
    # Logical (unpaged) K/V per sequence, including the appended tokens; only
    # materialised on request (small cases), for the contiguous brute force.
    logical_k: Optional[List[np.ndarray]] = None
    logical_v: Optional[List[np.ndarray]] = None

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_q_lens).astype(np.int32)


@dataclass
class Workload:
    name: str
    n_q: int
    n_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    poison_block: int
    k_cache: np.ndarray  # uint16 [num_blocks, n_kv, bs, d], state before the append
    v_cache: np.ndarray
    new_key: np.ndarray  # uint16 [T_new, n_kv, d]
    new_value: np.ndarray
    slot_mapping: np.ndarray  # int32 [T_new]
    scale: float
    decode: Optional[Batch] = None
    chunk: Optional[Batch] = None
    shared_prefix_seqs: List[int] = field(default_factory=list)  # decode-batch indices

    @property
    def group_size(self) -> int:
        return self.n_q // self.n_kv

    def kv_read_bytes(self, batch: Batch) -> int:
        """Logical K+V bytes that attention over ``batch`` reads (bf16)."""
        return int(np.sum(batch.context_lens.astype(np.int64))) * self.n_kv * self.head_dim * 2 * 2


@dataclass
class _SeqSpec:
    ctx: int
    q_len: int
    prefix_group: Optional[int] = None  # sequences in one group share their first blocks


def _build(name, rng, n_q, n_kv, specs, q_override=None, pool_blocks=None,
           shared_prefix_blocks=0, materialize_logical=False, table_width=None, values=True):
    d, bs = HEAD_DIM, BLOCK_SIZE
    nseq = len(specs)
    nblk = [math.ceil(s.ctx / bs) for s in specs]
    groups = sorted({s.prefix_group for s in specs if s.prefix_group is not None})
    unique_needed = sum(nblk) - sum(shared_prefix_blocks for s in specs if s.prefix_group is not None) \
        + shared_prefix_blocks * len(groups)
    if pool_blocks is None:
        pool_blocks = math.ceil(1.2 * unique_needed)
    assert pool_blocks > unique_needed, "pool needs at least one spare (poison) block"

    # Physical placement: a random permutation of the pool, handed out in order.
    perm = rng.permutation(pool_blocks).astype(np.int32)
    cursor = 0
    group_blocks = {}
    for gi in groups:
        group_blocks[gi] = perm[cursor:cursor + shared_prefix_blocks]
        cursor += shared_prefix_blocks
    tables = []
    for s, nb in zip(specs, nblk):
        if s.prefix_group is not None:
            own = perm[cursor:cursor + nb - shared_prefix_blocks]
            cursor += nb - shared_prefix_blocks
            tables.append(np.concatenate([group_blocks[s.prefix_group], own]))
        else:
            tables.append(perm[cursor:cursor + nb])
            cursor += nb
    poison_block = int(perm[cursor])  # never owned by any sequence
    width = table_width if table_width is not None else max(nblk)
    block_tables = np.full((nseq, width), poison_block, dtype=np.int32)
    for i, t in enumerate(tables):
        block_tables[i, :len(t)] = t

    if not values:
        # Structure only (the physical placement above was drawn first, so tables,
        # lengths and slots equal those of the full build); no K/V/q values.
        slots = []
        for i, s in enumerate(specs):
            npos = np.arange(s.ctx - s.q_len, s.ctx)
            slots.append((block_tables[i, npos // bs].astype(np.int64) * bs + npos % bs).astype(np.int32))
        cu = np.zeros(nseq + 1, dtype=np.int32)
        cu[1:] = np.cumsum([s.q_len for s in specs])
        batch = Batch(q=None, cu_q_lens=cu, block_tables=block_tables,
                      context_lens=np.array([s.ctx for s in specs], dtype=np.int32))
        wl = Workload(name=name, n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs, num_blocks=pool_blocks,
                      poison_block=poison_block, k_cache=None, v_cache=None, new_key=None, new_value=None,
                      slot_mapping=np.concatenate(slots).astype(np.int32),
                      scale=float(np.float32(1.0 / math.sqrt(d))))
        return wl, batch

    k_cache = np.full((pool_blocks, n_kv, bs, d), BF16_NAN, dtype=np.uint16)
    v_cache = np.full((pool_blocks, n_kv, bs, d), BF16_NAN, dtype=np.uint16)

    # Shared prefixes: one draw per group.
    group_kv = {}
    for gi in groups:
        npos = shared_prefix_blocks * bs
        group_kv[gi] = (_normal_bf16(rng, (npos, n_kv, d)), _normal_bf16(rng, (npos, n_kv, d)))

    new_k, new_v, slots = [], [], []
    logical_k = [] if materialize_logical else None
    logical_v = [] if materialize_logical else None
    for i, s in enumerate(specs):
        ctx, q_len = s.ctx, s.q_len
        if s.prefix_group is not None:
            pk, pv = group_kv[s.prefix_group]
            rest = ctx - pk.shape[0]
            lk = np.concatenate([pk, _normal_bf16(rng, (rest, n_kv, d))])
            lv = np.concatenate([pv, _normal_bf16(rng, (rest, n_kv, d))])
        else:
            lk = _normal_bf16(rng, (ctx, n_kv, d))
            lv = _normal_bf16(rng, (ctx, n_kv, d))
        cached = ctx - q_len
        # Place the already-cached tokens; the q_len new tokens are appended later.
        pos = np.arange(cached)
        phys = block_tables[i, pos // bs]
        k_cache[phys, :, pos % bs, :] = lk[:cached]
        v_cache[phys, :, pos % bs, :] = lv[:cached]
        npos = np.arange(cached, ctx)
        slots.append((block_tables[i, npos // bs].astype(np.int64) * bs + npos % bs).astype(np.int32))
        new_k.append(lk[cached:])
        new_v.append(lv[cached:])
        if materialize_logical:
            logical_k.append(lk)
            logical_v.append(lv)

    q_rows = sum(s.q_len for s in specs)
    q = q_override if q_override is not None else _normal_bf16(rng, (q_rows, n_q, d))
    assert q.shape == (q_rows, n_q, d)
    cu = np.zeros(nseq + 1, dtype=np.int32)
    cu[1:] = np.cumsum([s.q_len for s in specs])
    batch = Batch(q=q, cu_q_lens=cu, block_tables=block_tables,
                  context_lens=np.array([s.ctx for s in specs], dtype=np.int32),
                  logical_k=logical_k, logical_v=logical_v)
    wl = Workload(name=name, n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs,
                  num_blocks=pool_blocks, poison_block=poison_block,
                  k_cache=k_cache, v_cache=v_cache,
                  new_key=np.concatenate(new_k), new_value=np.concatenate(new_v),
                  slot_mapping=np.concatenate(slots).astype(np.int32),
                  scale=float(np.float32(1.0 / math.sqrt(d))))
    return wl, batch


def _split_batch(batch: Batch, idx: np.ndarray) -> Batch:
    """Sub-batch of the sequences ``idx`` (their q rows, tables, lengths)."""
    q_lens = batch.q_lens
    rows = np.concatenate([np.arange(batch.cu_q_lens[i], batch.cu_q_lens[i + 1]) for i in idx])
    cu = np.zeros(len(idx) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens[idx])
    used = int(max(math.ceil(int(batch.context_lens[i]) / BLOCK_SIZE) for i in idx))
    return Batch(q=None if batch.q is None else np.ascontiguousarray(batch.q[rows]), cu_q_lens=cu,
                 block_tables=np.ascontiguousarray(batch.block_tables[idx, :used]),
                 context_lens=np.ascontiguousarray(batch.context_lens[idx]),
                 logical_k=None if batch.logical_k is None else [batch.logical_k[i] for i in idx],
                 logical_v=None if batch.logical_v is None else [batch.logical_v[i] for i in idx])


def make_workload(name: str, seed: Optional[int] = None, materialize_logical: bool = False,
                  batch_scale: float = 1.0, values: bool = True) -> Workload:
    """Build one named workload.  ``seed`` defaults to 1000 + family index.

    ``batch_scale`` < 1 keeps the same per-sequence structure but fewer
    sequences (used for bounded CPU samples); 1.0 is the full workload.
    ``values=False`` builds the structure alone (contexts, block tables, slot
    mapping, identical to the full build's) and leaves K/V/q to the caller.
    """
    if name not in _FAMILY_SEED:
        raise ValueError(f"unknown workload {name!r}; expected one of {WORKLOAD_NAMES}")
    seed = _FAMILY_SEED[name] if seed is None else seed
    rng = np.random.default_rng(seed)

    def nb(b):
        return max(1, int(round(b * batch_scale)))

    if name == "tiny":
        specs = [_SeqSpec(10, 1), _SeqSpec(17, 1)]
        wl, b = _build(name, rng, 32, 8, specs, pool_blocks=16,
                       materialize_logical=materialize_logical, values=values)
        wl.decode = b
        return wl

    if name == "llama3_8b_b64":
        ctx = rng.integers(512, 4096, size=nb(64), endpoint=True)
        specs = [_SeqSpec(int(c), 1) for c in ctx]
        wl, b = _build(name, rng, 32, 8, specs, materialize_logical=materialize_logical, values=values)
        wl.decode = b
        return wl

    if name.startswith("sweep_"):
        n_kv = {"sweep_mha": 32, "sweep_gqa": 8, "sweep_mqa": 1}[name]
        B = nb(32)
        q = _normal_bf16(rng, (B, 32, HEAD_DIM)) if values else None  # identical across the three variants
        sub = np.random.default_rng([seed, n_kv])
        specs = [_SeqSpec(2048, 1) for _ in range(B)]
        wl, b = _build(name, sub, 32, n_kv, specs, q_override=q,
                       materialize_logical=materialize_logical, values=values)
        wl.decode = b
        return wl

    if name in ("llama3_70b_b8_32k", "llama3_70b_b1_128k"):
        B, ctx = (8, 32768) if name.endswith("32k") else (1, 131072)
        sub = np.random.default_rng([seed, B])
        specs = [_SeqSpec(ctx, 1) for _ in range(nb(B))]
        wl, b = _build(name, sub, 64, 8, specs, materialize_logical=materialize_logical, values=values)
        wl.decode = b
        return wl

    if name == "mixed":
        n_chunk, n_dec = nb(4), nb(60)
        dec_ctx = rng.integers(256, 8192, size=n_dec, endpoint=True)
        eligible = np.flatnonzero(dec_ctx > 1024)
        n_share = min(max(1, int(round(16 * batch_scale))), len(eligible))
        shared = np.sort(rng.choice(eligible, size=n_share, replace=False))
        specs = [_SeqSpec(1536, 512) for _ in range(n_chunk)]
        for i, c in enumerate(dec_ctx):
            specs.append(_SeqSpec(int(c), 1, prefix_group=0 if i in set(shared.tolist()) else None))
        wl, full = _build(name, rng, 32, 8, specs, shared_prefix_blocks=1024 // BLOCK_SIZE,
                          materialize_logical=materialize_logical, values=values)
        wl.chunk = _split_batch(full, np.arange(n_chunk))
        wl.decode = _split_batch(full, np.arange(n_chunk, n_chunk + n_dec))
        wl.shared_prefix_seqs = [int(i) for i in shared]
        return wl

    raise AssertionError(name)


def make_custom(n_q: int, n_kv: int, contexts, q_lens=None, seed: int = 0,
                shared_prefix: Optional[List[int]] = None, shared_prefix_blocks: int = 0,
                pool_blocks: Optional[int] = None, materialize_logical: bool = True,
                table_width: Optional[int] = None, name: str = "custom"):
    """A small ad-hoc workload: one batch with the given contexts and query lengths.

    Sequences listed in ``shared_prefix`` share their first
    ``shared_prefix_blocks`` physical blocks.  Returns (workload, batch).
    """
    rng = np.random.default_rng(seed)
    q_lens = [1] * len(contexts) if q_lens is None else list(q_lens)
    shared = set(shared_prefix or [])
    specs = [_SeqSpec(int(c), int(ql), 0 if i in shared else None)
             for i, (c, ql) in enumerate(zip(contexts, q_lens))]
    wl, batch = _build(name, rng, n_q, n_kv, specs, pool_blocks=pool_blocks,
                       shared_prefix_blocks=shared_prefix_blocks,
                       materialize_logical=materialize_logical, table_width=table_width)
    return wl, batch


def shard_for_rank(name: str, rank: int, world_size: int, **kw) -> Workload:
    """Weak scaling: every rank builds its own full-size batch from its own seed."""
    base = _FAMILY_SEED[name]
    return make_workload(name, seed=base + 7919 * rank if world_size > 1 else base, **kw)
