"""One decode step in one launch (paged_attention_decode_append) against the
fp64 oracle and against the two-call path (GPU).

The call must leave the pool exactly as kv_reshape_and_cache with each
sequence's slot of position ctx - 1 would, and return the attention over the
cache including that row ("LLM 推理全过程的维度变化与核心公式", section "Decode
阶段维度流转": the step's K/V is appended, then the single query row attends over
all of it).  Since the kernel feeds the same bits to the same arithmetic, its
output must also equal the two-call result bit for bit.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import (DevWorkload, assert_close, bf16_to_dev, dev_to_bf16_bits, i32_to_dev, oracle_after_append,
                         oracle_attention, status_word, torch)
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    P.load_library()


def fused(d, batch, partition_size=0, out_dtype=None, tables=None):
    t = torch()
    q = bf16_to_dev(batch.q)
    out = t.empty(q.shape, dtype=out_dtype or t.float32, device="cuda")
    tb = i32_to_dev(batch.block_tables if tables is None else tables)
    ws = P.paged_attention_decode_append(out, q, d.new_key, d.new_value, d.k_cache, d.v_cache, tb,
                                         i32_to_dev(batch.context_lens), d.wl.scale, partition_size=partition_size)
    t.cuda.synchronize()
    return out, ws


def check(wl, batch, parts=(0,)):
    kc, vc = oracle_after_append(wl)
    ref = oracle_attention(wl, batch, kc, vc)
    for part in parts:
        d = DevWorkload(wl)  # fresh pool: the call itself must write the new rows
        out, ws = fused(d, batch, partition_size=part)
        assert status_word(ws) == 0
        assert np.array_equal(dev_to_bf16_bits(d.k_cache), kc), f"K pool differs (part={part})"
        assert np.array_equal(dev_to_bf16_bits(d.v_cache), vc), f"V pool differs (part={part})"
        assert_close(out.cpu().numpy(), ref, what=f"{wl.name} part={part}")
        # the two-call path on the same inputs: identical bits
        d2 = DevWorkload(wl)
        d2.append()
        out2, _ = d2.decode(batch, partition_size=part)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), out2.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64", "sweep_mqa", "sweep_mha"])
def test_decode_append_workloads(name):
    wl = W.make_workload(name, materialize_logical=False)
    check(wl, wl.decode, parts=(0, 256))


@pytest.mark.parametrize("n_q,n_kv", [(32, 32), (32, 8), (64, 8), (32, 2), (32, 1)])
def test_decode_append_edge_lengths(n_q, n_kv):
    ctx = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 1000]
    wl, batch = W.make_custom(n_q, n_kv, ctx, seed=600 + n_q + n_kv, materialize_logical=False)
    check(wl, batch, parts=(0, 16, 256))


def test_decode_append_invalid_last_block_and_bf16_out():
    """A sequence whose last block id is invalid: flagged, nothing written for it, the others exact."""
    t = torch()
    wl, batch = W.make_custom(32, 8, [40, 300, 17, 1024], seed=620, materialize_logical=False)
    tables = batch.block_tables.copy()
    bad = 1
    last = (int(batch.context_lens[bad]) - 1) // 16
    tables[bad, last] = wl.k_cache.shape[0] + 5  # out of range
    d = DevWorkload(wl)
    before_k = dev_to_bf16_bits(d.k_cache)
    out, ws = fused(d, batch, tables=tables)
    assert status_word(ws) & P.PKV_STATUS_BAD_BLOCK_ID
    kc, vc = oracle_after_append(wl)
    got_k = dev_to_bf16_bits(d.k_cache)
    keep = np.ones(len(batch.context_lens), bool)
    keep[bad] = False
    # the bad sequence's slot keeps its old contents; every other new row is written
    slots = wl.slot_mapping
    for b in range(len(keep)):
        blk, row = divmod(int(slots[b]), 16)
        want = kc if keep[b] else before_k
        assert np.array_equal(got_k[blk, :, row], want[blk, :, row])
    ref = oracle_attention(wl, batch, kc, vc)
    assert_close(out.cpu().numpy()[keep], ref[keep], what="valid sequences next to an invalid one")
    # bf16 output: the fp32 result rounded, within one unit
    d2 = DevWorkload(wl)
    o16, _ = fused(d2, batch, out_dtype=t.bfloat16)
    o32, _ = fused(DevWorkload(wl), batch)
    want16 = o32.to(t.bfloat16).view(t.int16).cpu().numpy().astype(np.int32)
    assert np.max(np.abs(o16.view(t.int16).cpu().numpy().astype(np.int32) - want16)) <= 1
