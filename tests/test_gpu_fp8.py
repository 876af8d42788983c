"""FP8 (E4M3) KV cache on the GPU against the fp64 oracle.

The cache write must be bit-exact (codes and fp32 scales: the quantisation is
taken in fp32, one correctly rounded operation per step, on both sides).  The
decode over the FP8 pool is compared with the oracle's attention over the same
dequantised values (code * scale) within the decode tolerances (max abs 4e-3,
max rel 1e-2); the quantisation error itself is the cache's, not the kernel's.
Source: "LLM 推理全过程的维度变化与核心公式", section "KV Cache 的形状与增长",
INT8 / FP8 KV Cache item (per-token quantisation).

Initial pools are the bf16 workloads' pools quantised row by row by the
oracle, so unowned slots and the slots about to be appended hold the NaN code
(their rows are bf16 NaN): reading any of them shows up as non-finite output.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, bf16_to_dev, i32_to_dev, status_word, torch
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


def fp8_pool(wl):
    """Quantise every slot of the workload's bf16 pool (slot order) with the oracle."""
    nb, n_kv, bs, d = wl.k_cache.shape
    rows_k = wl.k_cache.transpose(0, 2, 1, 3).reshape(nb * bs, n_kv, d)  # [slot][head][d]
    rows_v = wl.v_cache.transpose(0, 2, 1, 3).reshape(nb * bs, n_kv, d)
    kc = np.zeros((nb, n_kv, bs, d), dtype=np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, n_kv, bs), dtype=np.float32)
    vs = np.zeros_like(ks)
    return oracle.kv_reshape_and_cache_fp8(rows_k, rows_v, kc, vc, ks, vs, np.arange(nb * bs, dtype=np.int32))


class Fp8Dev:
    def __init__(self, wl):
        t = torch()
        self.wl = wl
        self.host = fp8_pool(wl)
        self.k_cache, self.v_cache, self.k_scale, self.v_scale = (t.from_numpy(a.copy()).cuda() for a in self.host)
        self.after = oracle.kv_reshape_and_cache_fp8(wl.new_key, wl.new_value, *self.host, wl.slot_mapping)

    def append(self):
        P.kv_reshape_and_cache_fp8(bf16_to_dev(self.wl.new_key), bf16_to_dev(self.wl.new_value), self.k_cache,
                                   self.v_cache, self.k_scale, self.v_scale, i32_to_dev(self.wl.slot_mapping))

    def decode(self, batch, window=0, partition_size=0, out_dtype=None):
        t = torch()
        q = bf16_to_dev(batch.q)
        out = t.empty(q.shape, dtype=out_dtype or t.float32, device="cuda")
        ws = P.paged_attention_decode(out, q, self.k_cache, self.v_cache, i32_to_dev(batch.block_tables),
                                      i32_to_dev(batch.context_lens), self.wl.scale, window=window,
                                      partition_size=partition_size, k_scale=self.k_scale, v_scale=self.v_scale)
        return out, ws

    def prefill(self, batch, window=0, out_dtype=None, tables=None):
        t = torch()
        q = bf16_to_dev(batch.q)
        out = t.full(q.shape, float("nan"), dtype=out_dtype or t.float32, device="cuda")  # every row is written
        ws = P.paged_attention_prefill_chunk(out, q, i32_to_dev(batch.cu_q_lens), int(batch.q_lens.max()),
                                             self.k_cache, self.v_cache,
                                             i32_to_dev(batch.block_tables if tables is None else tables),
                                             i32_to_dev(batch.context_lens), self.wl.scale, window=window,
                                             k_scale=self.k_scale, v_scale=self.v_scale)
        return out, ws

    def oracle(self, batch, window=0):
        kc, vc, ks, vs = self.after
        return oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                      self.wl.scale, n_q=self.wl.n_q, window=window, k_scale=ks, v_scale=vs)


_pools = {}


def pool(name):
    """The named workload on an FP8 pool, appended on the GPU (built once per module)."""
    if name not in _pools:
        d = Fp8Dev(W.make_workload(name, materialize_logical=False))
        d.append()
        _pools[name] = d
    return _pools[name]


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64"])
def test_fp8_cache_write_bit_exact(name):
    d = pool(name)
    torch().cuda.synchronize()
    for dev, ref in zip((d.k_cache, d.v_cache, d.k_scale, d.v_scale), d.after):
        got = dev.cpu().numpy()
        assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), "FP8 cache write differs from the oracle"


def test_fp8_cache_write_extreme_rows():
    """Rows of zeros, tiny values, huge values and mixed signs quantise exactly as the oracle."""
    t = torch()
    rng = np.random.default_rng(50)
    n_kv, T = 2, 12
    x = rng.standard_normal((T, n_kv, 128)).astype(np.float32)
    x[0] = 0.0
    x[1] *= 1e-30
    x[2] *= 1e30
    x[3, 0] = 448.0
    x[4, :, ::2] = -x[4, :, ::2] * 1000
    x[5] = 1e-38
    key, value = W.bf16_bits_from_f32(x), W.bf16_bits_from_f32(x[::-1].copy())
    nb = 4
    host = (np.zeros((nb, n_kv, 16, 128), np.uint8), np.zeros((nb, n_kv, 16, 128), np.uint8),
            np.zeros((nb, n_kv, 16), np.float32), np.zeros((nb, n_kv, 16), np.float32))
    slots = np.array([3, 17, 40, 63, 0, 5, 33, 34, 35, 50, -1, 62], dtype=np.int32)
    ref = oracle.kv_reshape_and_cache_fp8(key, value, *host, slots)
    dev = [t.from_numpy(a.copy()).cuda() for a in host]
    P.kv_reshape_and_cache_fp8(bf16_to_dev(key), bf16_to_dev(value), *dev, i32_to_dev(slots))
    t.cuda.synchronize()
    for g, r in zip(dev, ref):
        assert np.array_equal(g.cpu().numpy().view(np.uint8), r.view(np.uint8))


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64", "sweep_mqa", "sweep_mha"])
def test_fp8_decode_parity(name):
    d = pool(name)
    wl = d.wl
    out, ws = d.decode(wl.decode)
    assert_close(out.cpu().numpy(), d.oracle(wl.decode), what=f"fp8 decode {name}")
    assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 8), (64, 8), (32, 1), (128, 8)])
def test_fp8_decode_edge_lengths_all_groups(n_q, n_kv):
    ctx = [1, 2, 15, 16, 17, 31, 33, 255, 256, 257, 1000]
    wl, batch = W.make_custom(n_q, n_kv, ctx, seed=400 + n_q + n_kv, materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    ref = d.oracle(batch)
    for part in (0, 16, 256):
        out, ws = d.decode(batch, partition_size=part)
        assert_close(out.cpu().numpy(), ref, what=f"fp8 G={n_q // n_kv} part={part}")
        assert status_word(ws) == 0


def test_fp8_decode_window_and_bf16_out():
    t = torch()
    wl, batch = W.make_custom(32, 8, [40, 300, 1024, 17], seed=410, materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    for win in (16, 100):
        out, ws = d.decode(batch, window=win)
        assert_close(out.cpu().numpy(), d.oracle(batch, window=win), what=f"fp8 W={win}")
    o16, _ = d.decode(batch, out_dtype=t.bfloat16)
    o32, _ = d.decode(batch)
    want = o32.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(o16.view(t.int16).cpu().numpy().astype(np.int32) - want)) <= 1


@pytest.mark.parametrize("n_q,n_kv,k", [(32, 8, 1), (32, 8, 2), (64, 8, 4), (32, 32, 16), (32, 1, 3)])
def test_fp8_verify_parity(n_q, n_kv, k):
    """Verify over the FP8 cache: row i at pos = ctx - k + i sees keys j <= pos (and
    pos - W < j under a window).  On the decode kernel (forced), one 8-column MMA tile
    per CTA, so G * k = 8, 32, 96 columns take 1, 4, 12 CTAs per KV head, with split
    partitions; on the library's own route (paged_attention_verify_fp8) too."""
    t = torch()
    ctx = [max(c, k) for c in (16, 17, 33, 100, 256, 257, 700, 1000)] + [k, k + 1]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * len(ctx), seed=560 + 3 * k + n_q // n_kv,
                              materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    q = bf16_to_dev(batch.q)
    for win in (0, 17, 300):
        ref = d.oracle(batch, window=win)
        for kernel, part in ((P.PKV_VERIFY_DECODE_KERNEL, 0), (P.PKV_VERIFY_DECODE_KERNEL, 16),
                             (P.PKV_VERIFY_AUTO, 0)):
            out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
            ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                          i32_to_dev(batch.context_lens), wl.scale, partition_size=part,
                                          window=win, k_scale=d.k_scale, v_scale=d.v_scale, kernel=kernel)
            assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} k={k} W={win} kernel={kernel} part={part}")
            assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv,k,nseq", [(32, 8, 16, 16), (32, 2, 8, 24)])
def test_fp8_verify_prefill_route(n_q, n_kv, k, nseq):
    """FP8 verify with many columns (G * k = 64 over 128 KV-head units, 128 over 48)
    runs on the FP8 prefill kernel: parity with the oracle, and the result is
    bit-identical to paged_attention_prefill_chunk_fp8 with k rows per sequence (the
    route's own kernel, with the same split plan)."""
    t = torch()
    base = (16, 17, 33, 100, 256, 257, 700, 1000, 5, 129, 128, 300, 64, 999, 2000, 31)
    ctx = [max(base[i % len(base)] + 7 * (i // len(base)), k) for i in range(nseq)]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * nseq, seed=580 + k + n_q // n_kv,
                              materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    q = bf16_to_dev(batch.q)
    for win in (0, 17, 300):
        ref = d.oracle(batch, window=win)
        out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
        ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                      i32_to_dev(batch.context_lens), wl.scale, window=win,
                                      k_scale=d.k_scale, v_scale=d.v_scale)
        assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} k={k} W={win}")
        assert status_word(ws) == 0
        pf, _ = d.prefill(batch, window=win)
        assert t.equal(out, pf), "FP8 verify did not take the prefill route"


def test_fp8_verify_last_row_is_fp8_decode():
    t = torch()
    k = 4
    wl, batch = W.make_custom(32, 8, [40, 300, 1024], q_lens=[k] * 3, seed=570, materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    q = bf16_to_dev(batch.q)
    out = t.empty(q.shape, dtype=t.float32, device="cuda")
    P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                             i32_to_dev(batch.context_lens), wl.scale, k_scale=d.k_scale, v_scale=d.v_scale)
    last = np.arange(1, 4) * k - 1
    dec_batch = W.Batch(q=batch.q[last], cu_q_lens=np.arange(4, dtype=np.int32), block_tables=batch.block_tables,
                        context_lens=batch.context_lens)
    dec, _ = d.decode(dec_batch)
    assert np.max(np.abs(out.cpu().numpy()[last] - dec.cpu().numpy())) <= 2e-5


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 8), (64, 8), (32, 2), (32, 16)])
def test_fp8_prefill_parity(n_q, n_kv):
    """Causal chunks over an FP8 cache on the tensor-core prefill: chunk lengths from
    one row to several row tiles, contexts spanning several key tiles with ragged
    tails, with and without a sliding window."""
    ctx = [1, 7, 40, 33, 300, 128, 600, 1100]
    q_lens = [1, 7, 32, 33, 100, 128, 129, 300]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=420 + n_q + n_kv, materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    for win in (0, 17, 300):
        ref = d.oracle(batch, window=win)
        out, ws = d.prefill(batch, window=win)
        assert_close(out.cpu().numpy(), ref, what=f"fp8 prefill G={n_q // n_kv} W={win}")
        assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv", [(32, 8), (32, 32)])
def test_fp8_prefill_and_decode_large_score_range(n_q, n_kv):
    """q scaled by 12 over an FP8 cache: the exponent reference (and, in the decode,
    the V exponent) is raised in the middle of sequences, O rescaled."""
    ctx = [1500, 900, 2000, 300]
    q_lens = [300, 129, 64, 200]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=430 + n_q + n_kv, materialize_logical=False)
    q = W.bf16_bits_from_f32(W.f32_from_bf16_bits(batch.q) * np.float32(12.0))
    batch = W.Batch(q=q, cu_q_lens=batch.cu_q_lens, block_tables=batch.block_tables, context_lens=batch.context_lens)
    d = Fp8Dev(wl)
    d.append()
    for win in (0, 700):
        out, ws = d.prefill(batch, window=win)
        assert_close(out.cpu().numpy(), d.oracle(batch, window=win), what=f"fp8 prefill q x12 W={win}")
        assert status_word(ws) == 0
    last = batch.cu_q_lens[1:] - 1
    dec_batch = W.Batch(q=batch.q[last], cu_q_lens=np.arange(len(ctx) + 1, dtype=np.int32),
                        block_tables=batch.block_tables, context_lens=batch.context_lens)
    out, ws = d.decode(dec_batch)
    assert_close(out.cpu().numpy(), d.oracle(dec_batch), what="fp8 decode q x12")
    assert status_word(ws) == 0


def test_fp8_prefill_mixed_chunks_stale_entries_and_bf16_out():
    """The mixed workload's 512-row chunks over 1024 cached tokens on an FP8 pool:
    plain, and under a 300-token window with invalid ids in the table entries wholly
    before every row's window (never read, no flag); bf16 output too."""
    t = torch()
    wl = W.make_workload("mixed", materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    ch = wl.chunk
    ref = d.oracle(ch)
    out, ws = d.prefill(ch)
    assert_close(out.cpu().numpy(), ref, what="fp8 mixed chunks")
    assert status_word(ws) == 0
    # bf16 output: the fp32 result rounded to nearest-even within one bf16 ulp, and
    # within the relative bound against the oracle (a bf16 half-ulp alone exceeds the
    # absolute bound once |out| >= 2)
    out16, _ = d.prefill(ch, out_dtype=t.bfloat16)
    want = out.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    got = out16.view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(got - want)) <= 1
    rel = np.abs(out16.float().cpu().numpy() - ref) / np.maximum(np.abs(ref), 1.0)
    assert rel.max() <= 1e-2, rel.max()
    win = 300
    tables = ch.block_tables.copy()
    for b in range(ch.num_seqs):
        c = int(ch.context_lens[b]) - int(ch.q_lens[b])
        tables[b, :max(0, c + 1 - win) // 16] = wl.k_cache.shape[0] + 11
    out, ws = d.prefill(ch, window=win, tables=tables)
    assert_close(out.cpu().numpy(), d.oracle(ch, window=win), what="fp8 mixed chunks, W=300")
    assert status_word(ws) == 0


def test_fp8_prefill_invalid_block_is_masked_and_flagged():
    """An out-of-range block id inside the context: its keys are left out (the oracle
    given the same table skips them too) and the bad-block status bit is set."""
    wl, batch = W.make_custom(32, 8, [300, 600], q_lens=[100, 200], seed=431, materialize_logical=False)
    d = Fp8Dev(wl)
    d.append()
    tables = batch.block_tables.copy()
    tables[1, 3] = wl.k_cache.shape[0] + 5
    out, ws = d.prefill(batch, tables=tables)
    assert status_word(ws) & P.PKV_STATUS_BAD_BLOCK_ID
    ok = out[:100].cpu().numpy()  # sequence 0 does not touch the bad entry
    assert_close(ok, d.oracle(batch)[:100], what="fp8 prefill, sequence beside a bad block")
    assert np.all(np.isfinite(out.cpu().numpy()))
