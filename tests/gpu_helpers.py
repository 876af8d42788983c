"""Helpers for the GPU parity tests: upload seeded workloads, run the CUDA path
through the C ABI (ctypes binding), and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np

import oracle
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

ABS_TOL = 4e-3   # max |out - ref| against the fp64 oracle
REL_TOL = 1e-2   # max |out - ref| / max(|ref|, 1)


def torch():
    import torch as t
    return t


def bf16_to_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(t.bfloat16)


def i32_to_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_to_bf16_bits(x) -> np.ndarray:
    t = torch()
    return x.view(t.int16).cpu().numpy().view(np.uint16)


def assert_close(got: np.ndarray, ref: np.ndarray, abs_tol=ABS_TOL, rel_tol=REL_TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), 1.0)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= abs_tol and rel.max() <= rel_tol, \
        f"{what}: max abs err {err.max():.3e} at {i} (got {got[i]:.6f}, ref {ref[i]:.6f}), max rel {rel.max():.3e}"
    return float(err.max())


class DevWorkload:
    """A workload's pool, append inputs and batches on the GPU."""

    def __init__(self, wl: W.Workload):
        self.wl = wl
        self.k_cache = bf16_to_dev(wl.k_cache)
        self.v_cache = bf16_to_dev(wl.v_cache)
        self.new_key = bf16_to_dev(wl.new_key)
        self.new_value = bf16_to_dev(wl.new_value)
        self.slot_mapping = i32_to_dev(wl.slot_mapping)

    def append(self):
        P.kv_reshape_and_cache(self.new_key, self.new_value, self.k_cache, self.v_cache, self.slot_mapping)

    def decode(self, batch: W.Batch, out_dtype=None, partition_size=0, workspace=None, window=0, tables=None):
        t = torch()
        q = bf16_to_dev(batch.q)
        out = t.empty(q.shape, dtype=out_dtype or t.float32, device="cuda")
        tab = batch.block_tables if tables is None else tables
        ws = P.paged_attention_decode(out, q, self.k_cache, self.v_cache, i32_to_dev(tab),
                                      i32_to_dev(batch.context_lens), self.wl.scale, workspace=workspace,
                                      partition_size=partition_size, window=window)
        return out, ws

    def prefill(self, batch: W.Batch, out_dtype=None, workspace=None, window=0, tables=None):
        t = torch()
        q = bf16_to_dev(batch.q)
        out = t.full(q.shape, float("nan"), dtype=out_dtype or t.float32, device="cuda")  # every row is written
        ws = P.paged_attention_prefill_chunk(out, q, i32_to_dev(batch.cu_q_lens), int(batch.q_lens.max()),
                                             self.k_cache, self.v_cache,
                                             i32_to_dev(batch.block_tables if tables is None else tables),
                                             i32_to_dev(batch.context_lens), self.wl.scale, workspace=workspace,
                                             window=window)
        return out, ws


def oracle_after_append(wl: W.Workload):
    return oracle.kv_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)


def oracle_attention(wl: W.Workload, batch: W.Batch, kc=None, vc=None):
    if kc is None:
        kc, vc = oracle_after_append(wl)
    return oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                  wl.scale, n_q=wl.n_q)


def status_word(ws) -> int:
    t = torch()
    return int(ws[:4].view(t.int32).cpu().item()) & 0xFFFFFFFF
