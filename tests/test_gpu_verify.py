"""Multi-token verify (paged_attention_verify) against the fp64 oracle (GPU).

Row i of sequence b sits at position ctx_b - k + i and sees keys j <= ctx_b - k + i
("LLM 推理全过程的维度变化与核心公式", section "工程优化怎么嵌进公式", Speculative
Decoding: the target model checks the k draft positions in one pass) -- the
oracle's causal-chunk rule with q_len = k.  The decode kernel (one 8-column MMA
tile per CTA up to 8 columns, two tiles up to 16, more CTAs per KV head above
that, ragged shares included) and the tcgen05 prefill kernel (taken when G * k
columns over enough sequences x KV heads make it faster, and G packs its tiles)
are both covered, and a test pins which one a batch takes.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_helpers import DevWorkload, assert_close, bf16_to_dev, i32_to_dev, oracle_after_append, status_word, torch
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CTX = [16, 17, 33, 100, 256, 257, 700, 1000]


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


def _on_decode(G, k, nseq, n_kv):
    """The library's route: the prefill kernel when it can pack the group and G k >= 32."""
    if G > 16 or 128 % G:
        return True
    return G * k < 32


def _verify(d, batch, k, partition_size=0, out_dtype=None, context_lens=None, window=0, tables=None):
    t = torch()
    q = bf16_to_dev(batch.q)
    out = t.full(q.shape, float("nan"), dtype=out_dtype or t.float32, device="cuda")  # every row is written
    lens = batch.context_lens if context_lens is None else context_lens
    ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache,
                                  i32_to_dev(batch.block_tables if tables is None else tables), i32_to_dev(lens),
                                  d.wl.scale, partition_size=partition_size, window=window)
    return out, ws


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 16), (48, 16), (32, 8), (64, 8), (32, 2), (32, 1)])
@pytest.mark.parametrize("k", [1, 2, 3, 4, 7, 8, 16])
def test_verify_parity(n_q, n_kv, k):
    ctx = [max(c, k) for c in CTX] + [k, k + 1]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * len(ctx), seed=500 + 7 * k + n_q // n_kv,
                              materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens, wl.scale,
                                 n_q=wl.n_q)
    G = n_q // n_kv
    on_decode = _on_decode(G, k, len(ctx), n_kv)
    for part in ((0, 16, 256) if on_decode else (0,)):
        out, ws = _verify(d, batch, k, partition_size=part)
        assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} k={k} part={part}")
        assert status_word(ws) == 0


def test_verify_last_row_is_decode_and_bf16_out():
    """Row k-1 of each sequence equals the decode of that token."""
    t = torch()
    k = 4
    wl, batch = W.make_custom(32, 8, [40, 300, 1024], q_lens=[k] * 3, seed=520, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    out, _ = _verify(d, batch, k)
    last = np.arange(1, 4) * k - 1
    dq = bf16_to_dev(batch.q[last])
    dout = t.empty(dq.shape, dtype=t.float32, device="cuda")
    P.paged_attention_decode(dout, dq, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                             i32_to_dev(batch.context_lens), wl.scale)
    assert np.max(np.abs(out.cpu().numpy()[last] - dout.cpu().numpy())) <= 2e-5
    o16, _ = _verify(d, batch, k, out_dtype=t.bfloat16)
    want = out.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(o16.view(t.int16).cpu().numpy().astype(np.int32) - want)) <= 1


@pytest.mark.parametrize("n_q,n_kv,k", [(32, 8, 2), (64, 8, 4), (64, 8, 8)])  # decode: 1 and 2 CTAs; prefill
def test_verify_short_context_flags(n_q, n_kv, k):
    wl, batch = W.make_custom(n_q, n_kv, [50, 60], q_lens=[k, k], seed=530 + k, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    lens = batch.context_lens.copy()
    lens[1] = k - 1
    t = torch()
    q = bf16_to_dev(batch.q)
    out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")  # every row must be written
    ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables), i32_to_dev(lens),
                                  d.wl.scale)
    assert status_word(ws) & P.PKV_STATUS_BAD_Q_LEN
    o = out.cpu().numpy()
    assert np.all(o[k:] == 0.0)          # the flagged sequence gets zero rows
    assert np.all(np.isfinite(o[:k]))    # the valid one is computed


@pytest.mark.parametrize("n_q,n_kv,k", [(32, 8, 2), (32, 8, 4), (64, 8, 4), (64, 8, 8), (32, 1, 3), (32, 32, 16)])
def test_verify_window_parity(n_q, n_kv, k):
    """Verify under a sliding window: row i at pos = ctx - k + i sees pos - W < j <= pos
    (decode kernel with one or two column tiles and several CTAs per KV head; the
    tcgen05 prefill kernel for G * k > 32), with split partitions, and table entries
    wholly before the first row's window set to invalid ids (never read, no flag)."""
    ctx = [max(c, k) for c in CTX] + [k, k + 1]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * len(ctx), seed=540 + 7 * k + n_q // n_kv,
                              materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    G = n_q // n_kv
    on_decode = _on_decode(G, k, len(ctx), n_kv)
    for win in (1, 5, 16, 17, 100, 300):
        ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                     wl.scale, n_q=wl.n_q, window=win)
        tables = batch.block_tables.copy()
        for b, c in enumerate(batch.context_lens):
            first = max(0, int(c) - k + 1 - win) // 16
            tables[b, :first] = wl.k_cache.shape[0] + 5
        for part in ((0, 16) if on_decode else (0,)):
            out, ws = _verify(d, batch, k, partition_size=part, window=win, tables=tables)
            assert_close(out.cpu().numpy(), ref, what=f"G={G} k={k} W={win} part={part}")
            assert status_word(ws) == 0


def test_verify_window_errors():
    wl, batch = W.make_custom(32, 8, [50], q_lens=[4], seed=545, materialize_logical=False)
    d = DevWorkload(wl)
    with pytest.raises(P.PagedKVError):
        _verify(d, batch, 4, window=-1)


@pytest.mark.parametrize("n_q,n_kv,k,nseq", [(32, 8, 16, 16), (64, 8, 16, 12), (64, 8, 8, 4), (32, 8, 16, 3)])
def test_verify_route_by_units(n_q, n_kv, k, nseq):
    """G * k = 64 or 128 columns over 24-128 sequence x KV-head units: the prefill
    kernel (splitting the keys where its CTAs cannot fill the GPU); the result is
    bit-identical to paged_attention_prefill_chunk with k rows per sequence (same
    split plan), and both kernels forced match the oracle."""
    t = torch()
    base = (16, 17, 33, 100, 256, 257, 700, 1000, 5, 129, 128, 300, 64, 999, 2000, 31)
    ctx = [max(base[i], k) for i in range(nseq)]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * nseq, seed=590 + k + nseq, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens, wl.scale,
                                 n_q=wl.n_q)
    G = n_q // n_kv
    on_decode = _on_decode(G, k, nseq, n_kv)
    for part in ((0, 16) if on_decode else (0,)):
        out, ws = _verify(d, batch, k, partition_size=part)
        assert_close(out.cpu().numpy(), ref, what=f"G={G} k={k} B={nseq} part={part}")
        assert status_word(ws) == 0
    c = P.CacheDesc(wl.num_blocks, 16, n_kv, 128, P.PKV_DTYPE_BF16)
    assert P.load_library().paged_attention_verify_on_prefill(nseq, k, n_q, ctypes.byref(c)) == (0 if on_decode else 1)
    if not on_decode:
        pf, _ = d.prefill(batch)
        assert t.equal(out, pf), "verify did not take the prefill route"
    q = bf16_to_dev(batch.q)
    for kernel in (P.PKV_VERIFY_DECODE_KERNEL, P.PKV_VERIFY_PREFILL_KERNEL):
        o = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
        P.paged_attention_verify(o, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                 i32_to_dev(batch.context_lens), wl.scale, kernel=kernel)
        assert_close(o.cpu().numpy(), ref, what=f"G={G} k={k} B={nseq} kernel={kernel}")


@pytest.mark.parametrize("n_q,n_kv,k", [(32, 8, 1), (32, 8, 4), (32, 8, 16), (64, 8, 2), (64, 8, 16), (32, 32, 3),
                                        (32, 2, 7), (32, 16, 5)])
def test_verify_on_each_kernel(n_q, n_kv, k):
    """paged_attention_verify_on with each kernel forced: both match the oracle."""
    ctx = [max(c, k) for c in CTX]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=[k] * len(ctx), seed=540 + 3 * k + n_q // n_kv,
                              materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens, wl.scale,
                                 n_q=wl.n_q)
    t = torch()
    q = bf16_to_dev(batch.q)
    for kernel in (P.PKV_VERIFY_DECODE_KERNEL, P.PKV_VERIFY_PREFILL_KERNEL):
        out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
        ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                      i32_to_dev(batch.context_lens), wl.scale, kernel=kernel)
        assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} k={k} kernel={kernel}")
        assert status_word(ws) == 0


def test_verify_long_contexts_few_sequences_on_each_kernel():
    """Two sequences over long contexts: the prefill kernel splits the keys (its
    workspace holds the partials), the decode kernel splits them into partitions;
    both match the oracle, plain and under a window."""
    k = 8
    wl, batch = W.make_custom(64, 8, [20000, 7001], q_lens=[k, k], seed=550, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    t = torch()
    q = bf16_to_dev(batch.q)
    for win in (0, 5000):
        ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                     wl.scale, n_q=wl.n_q, window=win)
        for kernel in (P.PKV_VERIFY_DECODE_KERNEL, P.PKV_VERIFY_PREFILL_KERNEL):
            out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
            ws = P.paged_attention_verify(out, q, k, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                          i32_to_dev(batch.context_lens), wl.scale, kernel=kernel, window=win)
            if kernel == P.PKV_VERIFY_PREFILL_KERNEL:
                assert ws.numel() > 256  # the split plan's partials
            assert_close(out.cpu().numpy(), ref, what=f"k={k} W={win} kernel={kernel}")
            assert status_word(ws) == 0


def test_verify_prefill_kernel_refuses_unpackable_groups():
    t = torch()
    wl, batch = W.make_custom(24, 1, [100, 50], q_lens=[2, 2], seed=560, materialize_logical=False)
    d = DevWorkload(wl)
    q = bf16_to_dev(batch.q)
    out = t.empty(q.shape, dtype=t.float32, device="cuda")
    with pytest.raises(Exception):
        P.paged_attention_verify(out, q, 2, d.k_cache, d.v_cache, i32_to_dev(batch.block_tables),
                                 i32_to_dev(batch.context_lens), wl.scale, kernel=P.PKV_VERIFY_PREFILL_KERNEL,
                                 workspace=t.zeros(1 << 20, dtype=t.uint8, device="cuda"))
