"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Cache writes must be bit-exact; attention outputs must satisfy
max |out - ref| <= 4e-3 and max |out - ref| / max(|ref|, 1) <= 1e-2 on the
seeded bf16 workloads, whose unused pool slots hold bf16 NaN so that any read
past a context or of an unowned block shows up as a non-finite output.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import (DevWorkload, assert_close, bf16_to_dev, dev_to_bf16_bits, i32_to_dev, oracle_after_append,
                         oracle_attention, status_word, torch)
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DECODE_WORKLOADS = ["tiny", "llama3_8b_b64", "sweep_mha", "sweep_gqa", "sweep_mqa", "llama3_70b_b8_32k",
                    "llama3_70b_b1_128k", "mixed"]

_cache = {}


def workload(name):
    if name not in _cache:
        wl = W.make_workload(name)
        kc, vc = oracle_after_append(wl)
        _cache[name] = (wl, kc, vc, {})
    return _cache[name]


def oracle_out(name, which):
    wl, kc, vc, memo = workload(name)
    if which not in memo:
        batch = getattr(wl, which)
        memo[which] = oracle_attention(wl, batch, kc, vc)
    return memo[which]


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


# ---- K1: cache write ---------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64", "mixed"])
def test_cache_write_bit_exact(name):
    wl, kc, vc, _ = workload(name)
    d = DevWorkload(wl)
    d.append()
    assert np.array_equal(dev_to_bf16_bits(d.k_cache), kc)
    assert np.array_equal(dev_to_bf16_bits(d.v_cache), vc)


def test_cache_write_skips_padding_and_out_of_range_slots():
    wl, batch = W.make_custom(32, 8, [20, 40, 7], seed=21)
    slots = wl.slot_mapping.copy()
    slots[0] = -1
    slots[2] = wl.num_blocks * 16 + 3  # past the pool: must not be written
    kc, vc = oracle.kv_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, slots)
    d = DevWorkload(wl)
    d.slot_mapping = i32_to_dev(slots)
    d.append()
    torch().cuda.synchronize()
    assert np.array_equal(dev_to_bf16_bits(d.k_cache), kc)
    assert np.array_equal(dev_to_bf16_bits(d.v_cache), vc)


# ---- K2 + K3: decode ---------------------------------------------------------------

@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_decode_parity(name):
    wl, _, _, _ = workload(name)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.decode(wl.decode)
    assert_close(out.cpu().numpy(), oracle_out(name, "decode"), what=name)
    assert status_word(ws) == 0


@pytest.mark.parametrize("part", [16, 48, 256, 512, 688, 1024, 4096])
def test_decode_partition_invariance(part):
    wl, _, _, _ = workload("llama3_8b_b64")
    d = DevWorkload(wl)
    d.append()
    out, _ = d.decode(wl.decode, partition_size=part)
    assert_close(out.cpu().numpy(), oracle_out("llama3_8b_b64", "decode"), what=f"partition {part}")


def test_decode_repeated_calls_share_a_workspace():
    """Reusing one workspace for many calls (with different partition sizes)
    gives bitwise-identical results: no state carries over between calls."""
    t = torch()
    wl, _, _, _ = workload("llama3_8b_b64")
    d = DevWorkload(wl)
    d.append()
    first, ws = d.decode(wl.decode, partition_size=256)
    for part in (256, 512, 256, 0, 256):
        again, _ = d.decode(wl.decode, partition_size=part, workspace=ws)
        if part == 256:
            assert t.equal(first, again)
    assert status_word(ws) == 0
    assert_close(first.cpu().numpy(), oracle_out("llama3_8b_b64", "decode"))


def test_decode_bf16_output_is_rounded_f32():
    t = torch()
    wl, _, _, _ = workload("llama3_8b_b64")
    d = DevWorkload(wl)
    d.append()
    o32, _ = d.decode(wl.decode)
    o16, _ = d.decode(wl.decode, out_dtype=t.bfloat16)
    want = o32.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    got = o16.view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(got - want)) <= 1  # within one bf16 ulp of the rounded fp32 result
    ref = oracle_out("llama3_8b_b64", "decode")
    rel = np.abs(o16.float().cpu().numpy() - ref) / np.maximum(np.abs(ref), 1.0)
    assert rel.max() <= 1e-2


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 16), (32, 8), (64, 8), (32, 4), (32, 2), (32, 1), (64, 4)])
def test_decode_edge_lengths_all_groups(n_q, n_kv):
    ctx = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000]
    wl, batch = W.make_custom(n_q, n_kv, ctx, seed=n_q + 7 * n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    ref = oracle_attention(wl, batch)
    for part in (0, 16, 256):
        out, ws = d.decode(batch, partition_size=part)
        assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} part={part}")
        assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv,B,lo,hi", [(64, 8, 1000, 1, 300), (32, 32, 300, 1, 40), (32, 1, 700, 1, 2000),
                                             (32, 8, 1025, 1, 600)])
def test_decode_many_short_sequences(n_q, n_kv, B, lo, hi):
    """Many short (and some long) sequences in one call, against the oracle."""
    ctx = np.random.default_rng(B).integers(lo, hi, size=B, endpoint=True)
    wl, batch = W.make_custom(n_q, n_kv, ctx.tolist(), seed=B, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.decode(batch)
    assert_close(out.cpu().numpy(), oracle_attention(wl, batch), what=f"B={B} G={n_q // n_kv}")
    assert status_word(ws) == 0


def test_decode_block_permutation_is_bitwise_invariant():
    t = torch()
    wl, batch = W.make_custom(32, 8, [700, 33, 1500, 16], seed=31, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    a, _ = d.decode(batch, partition_size=256)
    perm = np.random.default_rng(5).permutation(wl.num_blocks)
    inv = t.from_numpy(np.argsort(perm)).cuda()
    d.k_cache = d.k_cache[inv].contiguous()  # block i moves to position perm[i]
    d.v_cache = d.v_cache[inv].contiguous()
    batch.block_tables = perm[batch.block_tables].astype(np.int32)
    b, _ = d.decode(batch, partition_size=256)
    assert t.equal(a, b)


def test_decode_shared_prefix_matches_private_copies_bitwise():
    t = torch()
    wl, batch = W.make_custom(32, 8, [1200, 900, 1500], seed=32, shared_prefix=[0, 1, 2], shared_prefix_blocks=40,
                              materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    shared, _ = d.decode(batch)
    tables = batch.block_tables.copy()
    src = []
    nb = wl.num_blocks
    for b in (1, 2):
        for j in range(40):
            src.append(tables[b, j])
            tables[b, j] = nb
            nb += 1
    idx = t.from_numpy(np.array(src, dtype=np.int64)).cuda()
    d.k_cache = t.cat([d.k_cache, d.k_cache[idx]]).contiguous()
    d.v_cache = t.cat([d.v_cache, d.v_cache[idx]]).contiguous()
    batch.block_tables = tables
    private, _ = d.decode(batch)
    assert t.equal(shared, private)
    assert_close(shared.cpu().numpy(), oracle_attention(wl, batch, dev_to_bf16_bits(d.k_cache),
                                                        dev_to_bf16_bits(d.v_cache)))


def test_decode_device_side_checks_flag_and_never_fault():
    t = torch()
    wl, batch = W.make_custom(32, 8, [100, 40, 60, 30], seed=33, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    tables = batch.block_tables.copy()
    tables[0, 2] = wl.num_blocks + 5   # out of range
    tables[1, 0] = -3                  # negative
    lens = batch.context_lens.copy()
    lens[2] = 0                        # empty sequence
    lens[3] = tables.shape[1] * 16 + 1000  # longer than its table row
    q = bf16_to_dev(batch.q)
    out = t.full(q.shape, 7.0, dtype=t.float32, device="cuda")
    ws = t.zeros(P.paged_attention_workspace_size(4, 32, tables.shape[1], 0, P.cache_desc(d.k_cache)),
                 dtype=t.uint8, device="cuda")
    P.paged_attention_decode(out, q, d.k_cache, d.v_cache, i32_to_dev(tables), i32_to_dev(lens), wl.scale,
                             workspace=ws)
    t.cuda.synchronize()
    st = status_word(ws)
    assert st & P.PKV_STATUS_BAD_BLOCK_ID
    assert st & P.PKV_STATUS_BAD_CONTEXT_LEN
    assert not st & P.PKV_STATUS_TIMEOUT
    o = out.cpu().numpy()
    assert np.all(o[2] == 0.0)         # empty sequence -> zero rows
    assert np.all(np.isfinite(o[:2]))  # bad blocks contribute nothing, no NaN


# ---- K4: causal chunked prefill (tcgen05) ---------------------------------------------

def test_prefill_parity_mixed():
    wl, _, _, _ = workload("mixed")
    d = DevWorkload(wl)
    d.append()
    out, ws = d.prefill(wl.chunk)
    assert_close(out.cpu().numpy(), oracle_out("mixed", "chunk"), what="mixed chunk")
    assert status_word(ws) == 0


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 16), (32, 8), (64, 8), (32, 2)])
def test_prefill_ragged_chunks(n_q, n_kv):
    ctx = [1, 7, 40, 33, 300, 128, 600, 1100]
    q_lens = [1, 7, 32, 33, 100, 128, 129, 300]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=n_q * 3 + n_kv, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.prefill(batch)
    assert_close(out.cpu().numpy(), oracle_attention(wl, batch), what=f"G={n_q // n_kv}")
    assert status_word(ws) == 0


def _scaled_q(batch, factor):
    """The batch with q scaled by `factor` (rounded to bf16 again)."""
    q = W.bf16_bits_from_f32(W.f32_from_bf16_bits(batch.q) * np.float32(factor))
    return W.Batch(q=q, cu_q_lens=batch.cu_q_lens, block_tables=batch.block_tables, context_lens=batch.context_lens)


@pytest.mark.parametrize("n_q,n_kv,window", [(32, 8, 0), (32, 32, 0), (64, 8, 0), (32, 8, 700)])
def test_prefill_large_score_range(n_q, n_kv, window):
    """Scores with a wide range (q scaled by 12: score / ln 2 of spread ~17): a row's
    running maximum passes the exponent reference by more than 2^8 again and again
    along the keys, so the reference is raised -- and O and l rescaled in tensor
    memory -- in the middle of a sequence, both on the first key tile's exact path and
    after a vote; the weights of most keys underflow to zero."""
    ctx = [1500, 900, 2000, 300]
    q_lens = [300, 129, 64, 200]
    wl, batch = W.make_custom(n_q, n_kv, ctx, q_lens=q_lens, seed=70 + n_q + n_kv + window,
                              materialize_logical=False)
    batch = _scaled_q(batch, 12.0)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.prefill(batch, window=window)
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                 wl.scale, n_q=wl.n_q, window=window)
    assert_close(out.cpu().numpy(), ref, what=f"G={n_q // n_kv} W={window}, q x12")
    assert status_word(ws) == 0


@pytest.mark.parametrize("part", [0, 256])
def test_decode_large_score_range(part):
    """The decode kernel's lazy reference under the same wide score range."""
    wl, batch = W.make_custom(32, 8, [3000, 1700, 517, 4096], seed=77, materialize_logical=False)
    batch = _scaled_q(batch, 12.0)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.decode(batch, partition_size=part)
    assert_close(out.cpu().numpy(), oracle_attention(wl, batch), what=f"decode, q x12, partition {part}")
    assert status_word(ws) == 0


def test_prefill_bf16_output():
    t = torch()
    wl, batch = W.make_custom(32, 8, [700, 250], q_lens=[200, 250], seed=41, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    o32, _ = d.prefill(batch)
    o16, _ = d.prefill(batch, out_dtype=t.bfloat16)
    want = o32.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    got = o16.view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(got - want)) <= 1


def test_prefill_last_row_matches_decode():
    wl, batch = W.make_custom(32, 8, [900], q_lens=[300], seed=42, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    chunk, _ = d.prefill(batch)
    last = W.Batch(q=batch.q[-1:], cu_q_lens=np.array([0, 1], np.int32), block_tables=batch.block_tables,
                   context_lens=batch.context_lens)
    dec, _ = d.decode(last)
    assert_close(chunk[-1:].cpu().numpy(), dec.cpu().numpy().astype(np.float64), abs_tol=2e-3, what="last row")


def test_prefill_one_chunk_equals_two_chunks():
    wl, batch = W.make_custom(32, 8, [1536], q_lens=[512], seed=43, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    one, _ = d.prefill(batch)
    first = W.Batch(q=batch.q[:256], cu_q_lens=np.array([0, 256], np.int32), block_tables=batch.block_tables,
                    context_lens=np.array([1280], np.int32))
    second = W.Batch(q=batch.q[256:], cu_q_lens=np.array([0, 256], np.int32), block_tables=batch.block_tables,
                     context_lens=np.array([1536], np.int32))
    a, _ = d.prefill(first)
    b, _ = d.prefill(second)
    two = np.concatenate([a.cpu().numpy(), b.cpu().numpy()])
    assert_close(one.cpu().numpy(), two.astype(np.float64), abs_tol=2e-3, what="chunk split")


def test_prefill_bad_block_is_masked_and_flagged():
    """An invalid block id in the first and in a later key tile of one sequence's
    table (unsplit chunk): its keys are masked, the status word flags it, the
    outputs stay finite, and the other sequence matches the oracle."""
    wl, batch = W.make_custom(32, 8, [1400, 1000], q_lens=[300, 200], seed=45, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    tables = batch.block_tables.copy()
    tables[0, 2] = wl.k_cache.shape[0] + 5
    tables[0, 40] = -3
    t = torch()
    ws0 = t.zeros(256, dtype=t.uint8, device="cuda")  # the status word alone: the unsplit kernel
    out, ws = d.prefill(batch, tables=tables, workspace=ws0)
    assert status_word(ws) & P.PKV_STATUS_BAD_BLOCK_ID
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    sub = W.Batch(q=batch.q[300:], cu_q_lens=np.array([0, 200], np.int32), block_tables=batch.block_tables[1:],
                  context_lens=batch.context_lens[1:])
    assert_close(o[300:], oracle_attention(wl, sub), what="sequence beside the bad blocks")


def test_prefill_flags_inconsistent_lengths():
    t = torch()
    wl, batch = W.make_custom(32, 8, [64, 64], q_lens=[16, 16], seed=44, materialize_logical=False)
    d = DevWorkload(wl)
    d.append()
    lens = batch.context_lens.copy()
    lens[1] = 8  # fewer keys than query rows
    q = bf16_to_dev(batch.q)
    out = t.full(q.shape, float("nan"), dtype=t.float32, device="cuda")
    ws = t.zeros(256, dtype=t.uint8, device="cuda")
    P.paged_attention_prefill_chunk(out, q, i32_to_dev(batch.cu_q_lens), 16, d.k_cache, d.v_cache,
                                    i32_to_dev(batch.block_tables), i32_to_dev(lens), wl.scale, workspace=ws)
    t.cuda.synchronize()
    assert status_word(ws) & P.PKV_STATUS_BAD_Q_LEN
    assert np.all(out[16:].cpu().numpy() == 0.0)  # the flagged sequence gets zero rows
    ref = oracle_attention(wl, W.Batch(q=batch.q[:16], cu_q_lens=np.array([0, 16], np.int32),
                                       block_tables=batch.block_tables[:1], context_lens=batch.context_lens[:1]))
    assert_close(out[:16].cpu().numpy(), ref, what="valid sequence still computed")


def test_auto_partitions_follow_the_measured_rules(built_library):
    """The automatic split-KV plan: 1024-token partitions, no split for short
    contexts whose unsplit grid fills one wave, at most 32 partitions per sequence."""
    t = torch()
    P.load_library()
    sms = t.cuda.get_device_properties(0).multi_processor_count
    c = P.CacheDesc(1000, 16, 8, 128, 0)
    n = lambda B, nq, mb: P.paged_attention_decode_partitions(B, nq, mb, 0, c)  # noqa: E731
    assert n(64, 32, 256) == 4          # ragged 8B-shaped batch, contexts up to 4096
    assert n(8, 64, 2048) == 32         # 70B-shaped B=8 x 32K
    assert n(1, 64, 8192) == 32         # B=1 x 128K: capped at 32 (4096-token partitions)
    if sms <= 32 * 8 <= 3 * sms:
        assert n(32, 32, 128) == 1      # B=32 x 2048, 8 KV heads: one wave unsplit
    assert n(2, 32, 2) == 1             # a context inside one partition is never split
    # a sliding window bounding every long sequence's span (W / 16 + 1 blocks): not split
    assert P.paged_attention_decode_partitions(64, 32, 256, 0, c, window=1024) == 1
    assert P.paged_attention_decode_partitions(64, 32, 256, 0, c, window=3000) == 1
    assert P.paged_attention_decode_partitions(64, 32, 4096, 0, c, window=8192) > 1  # 513 blocks: split
    if sms == 152:
        # MQA-shaped B=32 x 2048 (one KV head, 4 CTAs of 8 heads each): 4 partitions
        # of 512 tokens would be 1.12 waves of 3 CTAs per SM; 3 partitions fit one
        c1 = P.CacheDesc(1000, 16, 1, 128, 0)
        assert P.paged_attention_decode_partitions(32, 32, 128, 0, c1) == 3
    # FP8 cache: fewer, longer CTAs (half the bytes per CTA)
    c8 = P.CacheDesc(1000, 16, 8, 128, P.PKV_DTYPE_FP8_E4M3)
    n8 = lambda B, nq, mb: P.paged_attention_decode_partitions(B, nq, mb, 0, c8)  # noqa: E731
    assert n8(64, 32, 256) == 4         # ragged 8B-shaped batch: 1024-token partitions
    if sms == 152:
        assert n8(8, 64, 2048) == 8     # B=8 x 32K: 4096-token partitions
        assert n8(1, 64, 8192) == 64    # B=1 x 128K: 2048-token partitions
    assert n8(32, 256, 128) == 1        # MHA-shaped 2048-token contexts filling the GPU: unsplit


def test_decode_maximum_batch():
    """The largest batch the boundary accepts: 65535 sequences (grid z at its limit),
    contexts 1..39 tokens, one head; the decode and the one-launch decode with the
    append both match the oracle, and the pool holds exactly the oracle's appends."""
    t = torch()
    rng = np.random.default_rng(3)
    ctx = rng.integers(1, 40, size=65535).tolist()
    wl, batch = W.make_custom(1, 1, ctx, seed=5, materialize_logical=False)
    kc, vc = oracle_after_append(wl)
    ref = oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                 wl.scale, n_q=wl.n_q)
    d = DevWorkload(wl)
    d.append()
    out, ws = d.decode(batch)
    assert_close(out.cpu().numpy(), ref, what="B=65535 decode")
    assert status_word(ws) == 0
    # the same step in one launch, on a fresh pool
    d2 = DevWorkload(wl)
    q = bf16_to_dev(batch.q)
    out2 = t.empty(q.shape, dtype=t.float32, device="cuda")
    ws2 = P.paged_attention_decode_append(out2, q, bf16_to_dev(wl.new_key), bf16_to_dev(wl.new_value), d2.k_cache,
                                          d2.v_cache, i32_to_dev(batch.block_tables),
                                          i32_to_dev(batch.context_lens), wl.scale)
    assert_close(out2.cpu().numpy(), ref, what="B=65535 decode with the append")
    assert status_word(ws2) == 0
    assert np.array_equal(dev_to_bf16_bits(d2.k_cache), kc) and np.array_equal(dev_to_bf16_bits(d2.v_cache), vc)
