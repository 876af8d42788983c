"""Sliding-window decode (paged_attention_decode_window) and causal prefill chunk
(paged_attention_prefill_chunk_window) against the fp64 oracle (GPU).

A row at position p sees keys p - W < j <= p ("LLM 推理全过程的维度变化与核心公式",
section "KV Cache 的形状与增长", Sliding Window Attention: only the most recent W
tokens' K and V are kept).  Tolerances as for decode: max abs 4e-3, max rel 1e-2.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import DevWorkload, assert_close, oracle_after_append, status_word
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


def _oracle(wl, batch, kc, vc, window):
    return oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                  wl.scale, n_q=wl.n_q, window=window)


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 8), (64, 8), (32, 1), (128, 8)])
def test_window_parity_all_groups(n_q, n_kv):
    ctx = [1, 2, 15, 16, 17, 33, 100, 256, 257, 700, 1500]
    wl, batch = W.make_custom(n_q, n_kv, ctx, seed=300 + n_q + n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    for win in (1, 15, 16, 17, 100, 512, 2000):
        ref = _oracle(wl, batch, kc, vc, win)
        for part in (0, 16):
            out, ws = d.decode(batch, partition_size=part, window=win)
            assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} W={win} part={part}")
            assert status_word(ws) == 0


def test_window_never_reads_blocks_before_it():
    """Table entries wholly before the window may be stale or freed: give them
    invalid ids; the result is unchanged and no bad-block flag is raised."""
    wl, batch = W.make_custom(32, 8, [40, 300, 1024, 17, 999], seed=310, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    for win in (16, 33, 200):
        tables = batch.block_tables.copy()
        for b, ctx in enumerate(batch.context_lens):
            first = max(0, int(ctx) - win) // 16
            tables[b, :first] = wl.k_cache.shape[0] + 7
        ref = _oracle(wl, batch, kc, vc, win)
        out, ws = d.decode(batch, window=win, tables=tables)
        assert_close(out.cpu().numpy(), ref, what=f"W={win}")
        assert status_word(ws) == 0


def test_window_covering_context_matches_plain_decode():
    wl, batch = W.make_custom(32, 8, [5, 64, 333, 1024], seed=311, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                 wl.scale, n_q=wl.n_q)
    out, ws = d.decode(batch, window=1024)
    assert_close(out.cpu().numpy(), ref, what="W >= ctx")


def test_window_long_context():
    """One 128K-token sequence (70B-shaped heads) under a 4096-token window."""
    wl = W.make_workload("llama3_70b_b1_128k", materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ref = _oracle(wl, wl.decode, kc, vc, 4096)
    out, ws = d.decode(wl.decode, window=4096)
    assert_close(out.cpu().numpy(), ref, what="128K, W=4096")
    assert status_word(ws) == 0


def test_window_argument_errors():
    wl, batch = W.make_custom(8, 2, [20], seed=312, materialize_logical=False)
    d = DevWorkload(wl)
    with pytest.raises(P.PagedKVError):
        d.decode(batch, window=-3)


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 8), (64, 8), (32, 2), (32, 16)])
def test_prefill_window_parity(n_q, n_kv):
    """Causal chunks under a window: every row at pos sees pos - W < j <= pos; the
    windows span one key, a partial block, a block, a key tile and beyond."""
    ctx = [1, 7, 40, 33, 300, 128, 600, 1100]
    q_lens = [1, 7, 32, 33, 100, 128, 129, 300]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=320 + n_q + n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    for win in (1, 15, 16, 100, 128, 129, 700, 5000):
        ref = _oracle(wl, batch, kc, vc, win)
        out, ws = d.prefill(batch, window=win)
        assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} W={win}")
        assert status_word(ws) == 0


def test_prefill_window_mixed_chunks_and_stale_entries():
    """The mixed workload's 512-row chunks over 1024 cached tokens under a 300-token
    window; table entries wholly before every row's window get invalid ids: the result
    is unchanged and no bad-block flag is raised."""
    wl = W.make_workload("mixed", materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    kc, vc = oracle_after_append(wl)
    ch = wl.chunk
    win = 300
    ref = _oracle(wl, ch, kc, vc, win)
    tables = ch.block_tables.copy()
    for b in range(ch.num_seqs):
        c = int(ch.context_lens[b]) - int(ch.q_lens[b])
        first = max(0, c + 1 - win) // 16  # the chunk's first row sees nothing before this block
        tables[b, :first] = wl.k_cache.shape[0] + 11
    out, ws = d.prefill(ch, window=win, tables=tables)
    assert_close(out.cpu().numpy(), ref, what="mixed chunks, W=300")
    assert status_word(ws) == 0


def test_prefill_window_covering_context_is_exact():
    """A window at least as long as the context gives the unwindowed result bit for bit."""
    wl, batch = W.make_custom(32, 8, [700, 250, 1536], q_lens=[200, 250, 512], seed=330, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    plain, _ = d.prefill(batch)
    wide, _ = d.prefill(batch, window=1536)
    assert np.array_equal(plain.cpu().numpy(), wide.cpu().numpy())


def test_prefill_window_argument_errors():
    wl, batch = W.make_custom(8, 2, [20], q_lens=[4], seed=331, materialize_logical=False)
    d = DevWorkload(wl)
    with pytest.raises(P.PagedKVError):
        d.prefill(batch, window=-3)
