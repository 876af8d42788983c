"""The allocation-free decode entry point, paged_attention_decode_static_scratch.

Some callers cannot allocate device memory where they call attention: code
inside a framework whose allocator owns all device memory, latency-critical
loops where cudaMalloc/cudaFree would synchronise the device, or plugins that
are handed only their inputs and outputs.  For them the library keeps the
split-KV scratch in one fixed device array instead of a workspace argument.

This file is collected last so that, should it fail, a run that stops at the
first failure has already run every other test.  It must pass alone in a
fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

ABS_TOL = 4e-3
REL_TOL = 1e-2


@pytest.fixture(scope="module")
def lib(built_library):
    return P.load_library()


def test_oversized_request_is_rejected_before_any_gpu_work(lib):
    # 4096 sequences x 64 heads x 128 partitions of 256 tokens need far more
    # than the fixed array; the call must refuse on the host.
    c = P.CacheDesc(100000, 16, 8, 128, P.PKV_DTYPE_BF16)
    need = lib.paged_attention_workspace_size(4096, 64, 2048, 256, ctypes.byref(c))
    assert need > P.STATIC_SCRATCH_BYTES
    fake = 0x100000
    rc = lib.paged_attention_decode_static_scratch(fake, P.PKV_DTYPE_FLOAT32, fake, fake, fake, fake, fake, 4096, 64,
                                                   2048, 0.088, 256, ctypes.byref(c), None, None)
    assert rc == P.PKV_ERR_WORKSPACE_TOO_SMALL


def _upload(wl, batch):
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()

    kc, vc = bf(wl.k_cache), bf(wl.v_cache)
    P.kv_reshape_and_cache(bf(wl.new_key), bf(wl.new_value), kc, vc, i32(wl.slot_mapping))
    return kc, vc, bf(batch.q), i32(batch.block_tables), i32(batch.context_lens)


def _close(got, ref):
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), 1.0)
    assert np.all(np.isfinite(got))
    assert err.max() <= ABS_TOL and rel.max() <= REL_TOL, (err.max(), rel.max())


def _oracle(wl, batch):
    import oracle  # the fp64 CPU reference (test infrastructure)
    kc, vc = oracle.kv_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
    return oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                  wl.scale, n_q=wl.n_q)


def _call(lib, out, q, kc, vc, tables, lens, scale, part, status):
    import torch
    desc = P.cache_desc(kc)
    return lib.paged_attention_decode_static_scratch(
        out.data_ptr(), P.PKV_DTYPE_FLOAT32, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(),
        lens.data_ptr(), q.shape[0], q.shape[1], tables.shape[1], scale, part, ctypes.byref(desc),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_decode_and_oracle_on_consecutive_calls(lib):
    import torch
    # Different batches in a row (explicit and automatic partition sizes), so
    # each call runs on scratch that still holds the previous call's data; the
    # last one is a large unsplit batch (many sequences and KV heads, short
    # contexts), where only the status word is cleared.
    cases = [
        W.make_custom(32, 8, [3000, 17, 1025, 2048, 700], seed=51, materialize_logical=False),
        W.make_custom(64, 8, [5000, 260, 4097], seed=52, materialize_logical=False),
        W.make_custom(32, 8, [9000, 33, 4000], seed=53, materialize_logical=False),
        W.make_custom(32, 32, list(np.random.default_rng(54).integers(1, 33, size=1500)), seed=54,
                      materialize_logical=False),
    ]
    for (wl, batch), part in zip(cases, (512, 256, 0, 0)):
        kc, vc, q, tables, lens = _upload(wl, batch)
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        P.paged_attention_decode(ref, q, kc, vc, tables, lens, wl.scale, partition_size=part)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = _call(lib, out, q, kc, vc, tables, lens, wl.scale, part, status)
        assert rc == P.PKV_OK, P.status_string(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        _close(got, ref.cpu().numpy().astype(np.float64))   # the workspace entry point's result
        _close(got, _oracle(wl, batch))                      # the fp64 oracle
        assert int(status.item()) == 0


@pytest.mark.gpu
def test_static_scratch_status_does_not_leak_into_the_next_call(lib):
    import torch
    wl, batch = W.make_custom(32, 8, [700, 40, 3000], seed=55, materialize_logical=False)
    kc, vc, q, tables, lens = _upload(wl, batch)
    bad = lens.clone()
    bad[1] = 0  # an invalid context length: zero output rows and a status bit
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert _call(lib, out, q, kc, vc, tables, bad, wl.scale, 256, status) == P.PKV_OK
    torch.cuda.synchronize()
    assert int(status.item()) & P.PKV_STATUS_BAD_CONTEXT_LEN
    assert np.all(out[1].cpu().numpy() == 0.0)
    assert _call(lib, out, q, kc, vc, tables, lens, wl.scale, 256, status) == P.PKV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _close(out.cpu().numpy(), _oracle(wl, batch))
