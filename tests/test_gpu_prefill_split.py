"""Split-KV on the tcgen05 prefill kernel against the fp64 oracle (GPU).

When the prefill kernel's CTAs (one per KV head, sequence and pair of 128-row
tiles) cannot fill the GPU -- a long chunk of one or two sequences, a verify of
few sequences over long contexts -- each pair's key tiles are cut into ranges
whose partials (m, l, O) a log-sum-exp merge folds ("LLM 推理全过程的维度变化与
核心公式", section "工程优化怎么嵌进公式": Flash-Decoding's split of cache_len and
its log-sum-exp reduction, which leave the formula unchanged).  The split is
taken only with a workspace of paged_attention_prefill_chunk_workspace_size()
bytes; a workspace of the status word alone keeps one CTA per pair, and both
must match the oracle.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_helpers import DevWorkload, assert_close, bf16_to_dev, i32_to_dev, oracle_after_append, status_word, torch
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


def _prefill(d, batch, workspace_bytes=None, window=0, tables=None):
    t = torch()
    q = bf16_to_dev(batch.q)
    out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")  # every row is written
    ws = None
    if workspace_bytes is not None:
        ws = t.zeros(workspace_bytes, dtype=t.uint8, device="cuda")
    ws = P.paged_attention_prefill_chunk(out, q, i32_to_dev(batch.cu_q_lens), int(batch.q_lens.max()), d.k_cache,
                                         d.v_cache, i32_to_dev(batch.block_tables if tables is None else tables),
                                         i32_to_dev(batch.context_lens), d.wl.scale, workspace=ws, window=window)
    return out, ws


def _desc(wl):
    return P.CacheDesc(wl.num_blocks, 16, wl.n_kv, 128, P.PKV_DTYPE_BF16)


def _split_bytes(wl, batch):
    return P.paged_attention_prefill_chunk_workspace_size(batch.num_seqs, wl.n_q, int(batch.cu_q_lens[-1]),
                                                          int(batch.q_lens.max()), batch.max_blocks_per_seq,
                                                          _desc(wl))


@pytest.mark.parametrize("n_q,n_kv", [(32, 8), (64, 8), (32, 32), (32, 2)])
def test_prefill_split_long_contexts(n_q, n_kv):
    """Two sequences with short chunks over long contexts (ragged tails, a chunk
    shorter than a row tile): the split plan and the unsplit kernel both match the
    oracle."""
    ctx = [16000, 9001]
    q_lens = [64, 33]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=600 + n_q + n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, *oracle_after_append(wl), batch.block_tables,
                                 batch.context_lens, wl.scale, n_q=wl.n_q)
    nbytes = _split_bytes(wl, batch)
    if n_kv * 2 < 152:
        assert nbytes > 256, "few CTAs over long contexts: the plan splits the keys"
    out, ws = _prefill(d, batch, nbytes)
    assert_close(out.cpu().numpy(), ref, what=f"split G={n_q // n_kv}")
    assert status_word(ws) == 0
    out1, ws1 = _prefill(d, batch, 256)  # the status word alone: no split
    assert_close(out1.cpu().numpy(), ref, what=f"unsplit G={n_q // n_kv}")
    assert status_word(ws1) == 0


def test_prefill_split_large_score_range():
    """q scaled by 12 on the split plan: each key range raises its own exponent
    reference in the middle of the range, and the merge folds partials whose
    references differ by many powers of two."""
    wl, batch = W.make_custom(32, 8, [16000, 9001], q_lens=[64, 33], seed=620, materialize_logical=False)
    q = W.bf16_bits_from_f32(W.f32_from_bf16_bits(batch.q) * np.float32(12.0))
    batch = W.Batch(q=q, cu_q_lens=batch.cu_q_lens, block_tables=batch.block_tables, context_lens=batch.context_lens)
    d = DevWorkload(wl)
    d.append()
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, *oracle_after_append(wl), batch.block_tables,
                                 batch.context_lens, wl.scale, n_q=wl.n_q)
    nbytes = _split_bytes(wl, batch)
    assert nbytes > 256
    out, ws = _prefill(d, batch, nbytes)
    assert_close(out.cpu().numpy(), ref, what="split, q x12")
    assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv", [(32, 8), (64, 8), (32, 16)])
def test_prefill_split_ragged_tiles_many_sequences(n_q, n_kv):
    """Several sequences whose chunks end inside a row tile (and one that is a
    single row), over contexts that end inside a key tile, on the split plan."""
    ctx = [12000, 6001, 9000, 4100, 7777]
    q_lens = [5, 40, 17, 1, 64]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=605 + n_q + n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, *oracle_after_append(wl), batch.block_tables,
                                 batch.context_lens, wl.scale, n_q=wl.n_q)
    nbytes = _split_bytes(wl, batch)
    out, ws = _prefill(d, batch, nbytes)
    assert_close(out.cpu().numpy(), ref, what=f"split, ragged tiles, G={n_q // n_kv}")
    assert status_word(ws) == 0
    out1, ws1 = _prefill(d, batch, 256)
    assert_close(out1.cpu().numpy(), ref, what=f"unsplit, ragged tiles, G={n_q // n_kv}")


def test_prefill_split_window_and_stale_entries():
    """A split chunk under a sliding window, with invalid ids in the table entries
    wholly before every row's window (never read, no flag)."""
    wl, batch = W.make_custom(32, 8, [12000, 7000], q_lens=[100, 17], seed=610, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    win = 3000
    tables = batch.block_tables.copy()
    for b in range(batch.num_seqs):
        c = int(batch.context_lens[b]) - int(batch.q_lens[b])
        tables[b, :max(0, c + 1 - win) // 16] = wl.k_cache.shape[0] + 9
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens, wl.scale,
                                 n_q=wl.n_q, window=win)
    out, ws = _prefill(d, batch, _split_bytes(wl, batch), window=win, tables=tables)
    assert_close(out.cpu().numpy(), ref, what="split, window 3000")
    assert status_word(ws) == 0


def test_prefill_split_bad_block_and_bad_length():
    """Device-side checks under a split: an invalid block id inside one range is
    masked and flagged; a sequence whose q_len exceeds its context gets zero rows."""
    t = torch()
    wl, batch = W.make_custom(32, 8, [9000, 8000], q_lens=[40, 30], seed=611, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    tables = batch.block_tables.copy()
    tables[0, 100] = wl.k_cache.shape[0] + 3
    out, ws = _prefill(d, batch, _split_bytes(wl, batch), tables=tables)
    assert status_word(ws) & P.PKV_STATUS_BAD_BLOCK_ID
    assert np.all(np.isfinite(out.cpu().numpy()))
    # sequence 1 does not touch the bad entry
    sub = W.Batch(q=batch.q[40:], cu_q_lens=np.array([0, 30], np.int32), block_tables=batch.block_tables[1:],
                  context_lens=batch.context_lens[1:])
    kc, vc = oracle_after_append(wl)
    ref1 = oracle.paged_attention(sub.q, sub.cu_q_lens, kc, vc, sub.block_tables, sub.context_lens, wl.scale,
                                  n_q=wl.n_q)
    assert_close(out[40:].cpu().numpy(), ref1, what="split, sequence beside a bad block")
    lens = batch.context_lens.copy()
    lens[1] = 20  # fewer keys than query rows
    q = bf16_to_dev(batch.q)
    out2 = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
    ws2 = t.zeros(_split_bytes(wl, batch), dtype=t.uint8, device="cuda")
    P.paged_attention_prefill_chunk(out2, q, i32_to_dev(batch.cu_q_lens), 40, d.k_cache, d.v_cache,
                                    i32_to_dev(batch.block_tables), i32_to_dev(lens), wl.scale, workspace=ws2)
    t.cuda.synchronize()
    assert status_word(ws2) & P.PKV_STATUS_BAD_Q_LEN
    assert np.all(out2[40:].cpu().numpy() == 0.0)
    ref0 = oracle.paged_attention(batch.q[:40], np.array([0, 40], np.int32), kc, vc, batch.block_tables[:1],
                                  batch.context_lens[:1], wl.scale, n_q=wl.n_q)
    assert_close(out2[:40].cpu().numpy(), ref0, what="split, valid sequence beside a bad length")


def test_verify_70b_shape_on_the_split_prefill_route():
    """The 70B-shaped B=8 x 32K batch verifying k = 16 draft positions runs on the
    prefill kernel (G k = 128 columns over 64 KV-head units), split over the keys;
    two of its sequences are checked against the oracle row by row."""
    t = torch()
    k = 16
    wl = W.make_workload("llama3_70b_b8_32k", values=False)
    b = wl.decode
    assert P.load_library().paged_attention_verify_on_prefill(b.num_seqs, k, wl.n_q, ctypes.byref(_desc(wl))) == 1
    # Values: N(0,1) draws rounded to bf16.  The blocks of the two checked sequences
    # (and q) come from the host generator and are what the oracle reads; the other
    # sequences' blocks are filled on the device.
    checked = (0, 5)
    rng = np.random.default_rng(612)
    nb = wl.num_blocks
    g = t.Generator(device="cuda")
    g.manual_seed(612)
    kc = t.randn((nb, wl.n_kv, 16, 128), generator=g, device="cuda").to(t.bfloat16)
    vc = t.randn((nb, wl.n_kv, 16, 128), generator=g, device="cuda").to(t.bfloat16)
    kh = np.zeros((nb, wl.n_kv, 16, 128), np.uint16)
    vh = np.zeros_like(kh)
    for s in checked:
        blocks = b.block_tables[s, :(int(b.context_lens[s]) + 15) // 16]
        for host, dev in ((kh, kc), (vh, vc)):
            host[blocks] = W.bf16_bits_from_f32(rng.standard_normal((len(blocks), wl.n_kv, 16, 128), dtype=np.float32))
            dev[t.from_numpy(blocks.astype(np.int64)).cuda()] = bf16_to_dev(host[blocks])
    q_bits = W.bf16_bits_from_f32(rng.standard_normal((b.num_seqs * k, wl.n_q, 128), dtype=np.float32))
    q = bf16_to_dev(q_bits)
    out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
    ws = P.paged_attention_verify(out, q, k, kc, vc, i32_to_dev(b.block_tables), i32_to_dev(b.context_lens), wl.scale)
    assert ws.numel() > 256, "the prefill route splits the keys for 64 units"
    assert status_word(ws) == 0
    for s in checked:
        rows = slice(s * k, (s + 1) * k)
        ref = oracle.paged_attention(q_bits[rows], np.array([0, k], np.int32), kh, vh, b.block_tables[s:s + 1],
                                     b.context_lens[s:s + 1], wl.scale, n_q=wl.n_q)
        assert_close(out[rows].cpu().numpy(), ref, what=f"70B verify k=16, sequence {s}")
