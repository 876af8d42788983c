"""The C-ABI library: it loads, exports every declared symbol, and validates
its arguments on the host before anything reaches the GPU (CPU only: every
call below returns from argument checking without a CUDA call)."""
import ctypes
import re

import pytest

from paged_kv_cache_95_gb300 import pagedkv as P

FAKE = 0x100000  # never dereferenced: validation fails before any device access


@pytest.fixture(scope="module")
def lib(built_library):
    return P.load_library()


def declared_symbols():
    text = open(P.HEADER_PATH).read()
    return re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"kv_reshape_and_cache", "paged_attention_decode", "paged_attention_prefill_chunk",
            "paged_attention_workspace_size", "paged_attention_prefill_workspace_size",
            "pagedkv_status_string", "pagedkv_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"libpagedkv.so does not export {name}"


def test_status_strings_and_version(lib):
    for code in (0, -1, -2, -3, -4):
        assert lib.pagedkv_status_string(code)
    assert b"unknown" in lib.pagedkv_status_string(12345)
    assert lib.pagedkv_version() >= 100


def desc(num_blocks=100, bs=16, n_kv=8, d=128, dtype=0):
    return P.CacheDesc(num_blocks, bs, n_kv, d, dtype)


def test_workspace_size_math(lib):
    c = desc()
    # 64 seqs, 32 heads, 256 blocks/seq, 512-token partitions -> 8 parts
    rows = 64 * 32 * 8
    want = 256 + 2 * ((rows * 4 + 255) // 256 * 256) + rows * 128 * 4  # status | m | l | O
    assert lib.paged_attention_workspace_size(64, 32, 256, 512, ctypes.byref(c)) == want
    # a partition that covers the whole context needs only the status word
    assert lib.paged_attention_workspace_size(64, 32, 256, 4096, ctypes.byref(c)) == 256
    # automatic plans are covered by the smallest automatic partition (256 tokens)
    assert lib.paged_attention_workspace_size(64, 32, 256, 0, ctypes.byref(c)) == \
        lib.paged_attention_workspace_size(64, 32, 256, 256, ctypes.byref(c))
    assert lib.paged_attention_workspace_size(64, 32, 256, 100, ctypes.byref(c)) == 0  # not a multiple of 16
    assert lib.paged_attention_workspace_size(64, 30, 256, 0, ctypes.byref(c)) == 0    # 30 % 8 != 0
    assert lib.paged_attention_prefill_workspace_size(4, 32, ctypes.byref(c)) == 256


def test_decode_partitions_with_explicit_size(lib):
    """An explicit partition size gives ceil(blocks a row can touch / partition blocks); no GPU needed."""
    c = desc()
    n = lambda *a: lib.paged_attention_decode_partitions(*a, ctypes.byref(c))  # noqa: E731
    assert n(64, 32, 256, 1024, 0) == 4       # 4096 tokens in 1024-token partitions
    assert n(64, 32, 256, 4096, 0) == 1       # one partition: no merge kernel
    assert n(64, 32, 256, 8192, 0) == 1
    assert n(1, 64, 8192, 1024, 0) == 128
    assert n(1, 64, 8192, 1024, 4096) == 5    # a 4096 window touches at most 257 blocks
    assert n(64, 32, 256, 100, 0) == P.PKV_ERR_INVALID_ARG   # not a multiple of 16
    assert n(64, 30, 256, 1024, 0) == P.PKV_ERR_INVALID_ARG  # 30 % 8 != 0
    assert n(0, 32, 256, 1024, 0) == P.PKV_ERR_INVALID_ARG
    assert n(64, 32, 256, 1024, -1) == P.PKV_ERR_INVALID_ARG
    assert lib.paged_attention_decode_partitions(64, 32, 256, 1024, 0, None) == P.PKV_ERR_INVALID_ARG


def _decode(lib, c, **kw):
    a = dict(out=FAKE, out_dtype=1, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=4, nq=32, mb=8, scale=0.088,
             part=0, ws=FAKE, wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.paged_attention_decode(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"],
                                      a["nq"], a["mb"], a["scale"], a["part"], ctypes.byref(c), a["ws"], a["wsb"],
                                      a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(out=None), P.PKV_ERR_INVALID_ARG),
    (dict(q=None), P.PKV_ERR_INVALID_ARG),
    (dict(bt=None), P.PKV_ERR_INVALID_ARG),
    (dict(ws=None), P.PKV_ERR_INVALID_ARG),
    (dict(B=0), P.PKV_ERR_INVALID_ARG),
    (dict(B=70000), P.PKV_ERR_INVALID_ARG),
    (dict(mb=0), P.PKV_ERR_INVALID_ARG),
    (dict(nq=30), P.PKV_ERR_INVALID_ARG),             # 30 % 8
    (dict(nq=96), P.PKV_ERR_UNSUPPORTED),             # G = 12
    (dict(part=100), P.PKV_ERR_INVALID_ARG),          # not a multiple of 16
    (dict(part=-16), P.PKV_ERR_INVALID_ARG),
    (dict(scale=float("nan")), P.PKV_ERR_INVALID_ARG),
    (dict(out_dtype=7), P.PKV_ERR_UNSUPPORTED),
    (dict(k=FAKE + 8), P.PKV_ERR_INVALID_ARG),        # pool not 16-byte aligned
    (dict(ws=FAKE + 64), P.PKV_ERR_INVALID_ARG),      # workspace not 256-byte aligned
    (dict(part=256, mb=64, wsb=1024), P.PKV_ERR_WORKSPACE_TOO_SMALL),
    (dict(wsb=100), P.PKV_ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_argument_errors(lib, kw, want):
    assert _decode(lib, desc(), **kw) == want


def test_decode_append_argument_errors(lib):
    c = desc()

    def call(**kw):
        a = dict(out=FAKE, q=FAKE, key=FAKE, value=FAKE, k=FAKE, B=4, nq=32, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_decode_append(a["out"], 1, a["q"], a["key"], a["value"], a["k"], FAKE, FAKE, FAKE,
                                                 a["B"], a["nq"], 8, 0.088, 0, ctypes.byref(c), FAKE, a["wsb"], None)
    assert call(key=None) == P.PKV_ERR_INVALID_ARG
    assert call(value=None) == P.PKV_ERR_INVALID_ARG
    assert call(key=FAKE + 8) == P.PKV_ERR_INVALID_ARG     # new rows must be 16-byte aligned
    assert call(value=FAKE + 4) == P.PKV_ERR_INVALID_ARG
    assert call(q=None) == P.PKV_ERR_INVALID_ARG
    assert call(nq=96) == P.PKV_ERR_UNSUPPORTED
    assert call(wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    c8 = desc(dtype=P.PKV_DTYPE_FP8_E4M3)                   # bf16 pool only
    assert lib.paged_attention_decode_append(FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 32, 8, 0.088, 0,
                                             ctypes.byref(c8), FAKE, 1 << 20, None) == P.PKV_ERR_UNSUPPORTED


def test_decode_window_argument_errors(lib):
    c = desc()

    def call(window, **kw):
        a = dict(out=FAKE, out_dtype=1, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=4, nq=32, mb=8, scale=0.088,
                 part=0, ws=FAKE, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_decode_window(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["bt"], a["cl"],
                                                 a["B"], a["nq"], a["mb"], a["scale"], window, a["part"],
                                                 ctypes.byref(c), a["ws"], a["wsb"], None)
    assert call(0) == P.PKV_ERR_INVALID_ARG      # a window holds at least one key
    assert call(-5) == P.PKV_ERR_INVALID_ARG
    assert call(64, q=None) == P.PKV_ERR_INVALID_ARG
    assert call(64, nq=96) == P.PKV_ERR_UNSUPPORTED
    assert call(64, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL


def test_verify_argument_errors(lib):
    c = desc()

    def v(k, **kw):
        a = dict(out=FAKE, q=FAKE, B=4, nq=32, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_verify(a["out"], 1, a["q"], k, FAKE, FAKE, FAKE, FAKE, a["B"], a["nq"], 8, 0.088, 0,
                                          ctypes.byref(c), FAKE, a["wsb"], None)
    assert v(0) == P.PKV_ERR_INVALID_ARG
    assert v(17) == P.PKV_ERR_INVALID_ARG
    assert v(2, q=None) == P.PKV_ERR_INVALID_ARG
    assert v(2, nq=96) == P.PKV_ERR_UNSUPPORTED                 # G = 12
    assert v(2, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL       # decode path (G * k = 8)
    assert v(6, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL       # decode path, two CTAs per KV head (G * k = 24)
    assert v(16, out=FAKE + 4, B=64) == P.PKV_ERR_INVALID_ARG   # prefill path (G * k = 64, 512 units): 16-B out
    ws = lambda k: lib.paged_attention_verify_workspace_size(64, k, 32, 256, 0, ctypes.byref(c))
    assert ws(0) == 0 and ws(17) == 0
    assert ws(16) == 256                                        # prefill path: the status word
    # decode path: partials for 64 * k rows of 32 heads
    assert ws(2) > lib.paged_attention_workspace_size(64, 32, 256, 0, ctypes.byref(c))
    assert ws(6) > ws(4) > ws(2)
    # 4 sequences x 8 KV heads = 32 units fill few SMs: the prefill kernel splits the keys
    # (partials of 4 * k rows of 32 heads per split in the workspace)
    ws4 = lambda k: lib.paged_attention_verify_workspace_size(4, k, 32, 256, 0, ctypes.byref(c))  # noqa: E731
    assert ws4(16) > ws4(8) > 256


def test_fp8_argument_errors(lib):
    c8, c16 = desc(dtype=P.PKV_DTYPE_FP8_E4M3), desc()
    # cache write: needs an FP8 descriptor and both scale arrays
    w = lambda c, **kw: lib.kv_reshape_and_cache_fp8(kw.get("k", FAKE), FAKE, FAKE, FAKE, kw.get("ks", FAKE), FAKE,
                                                     FAKE, kw.get("T", 4), ctypes.byref(c), None)
    assert w(c16) == P.PKV_ERR_UNSUPPORTED
    assert w(c8, ks=None) == P.PKV_ERR_INVALID_ARG
    assert w(c8, ks=FAKE + 4) == P.PKV_ERR_INVALID_ARG   # scales 16-byte aligned
    assert w(c8, T=-1) == P.PKV_ERR_INVALID_ARG
    assert w(c8, T=0) == P.PKV_OK

    def d(c, **kw):
        a = dict(ks=FAKE, vs=FAKE, window=0, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_decode_fp8(FAKE, 1, FAKE, FAKE, FAKE, a["ks"], a["vs"], FAKE, FAKE, 4, 32, 8, 0.088,
                                              a["window"], 0, ctypes.byref(c), FAKE, a["wsb"], None)
    assert d(c16) == P.PKV_ERR_UNSUPPORTED
    assert d(c8, ks=None) == P.PKV_ERR_INVALID_ARG
    assert d(c8, vs=None) == P.PKV_ERR_INVALID_ARG
    assert d(c8, window=-1) == P.PKV_ERR_INVALID_ARG
    assert d(c8, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    # the workspace does not depend on the element type
    assert lib.paged_attention_workspace_size(64, 32, 256, 0, ctypes.byref(c8)) == \
        lib.paged_attention_workspace_size(64, 32, 256, 0, ctypes.byref(c16))


@pytest.mark.parametrize("c,want", [
    (desc(bs=32), P.PKV_ERR_UNSUPPORTED),
    (desc(d=64), P.PKV_ERR_UNSUPPORTED),
    (desc(dtype=1), P.PKV_ERR_UNSUPPORTED),
    (desc(num_blocks=0), P.PKV_ERR_INVALID_ARG),
    (desc(n_kv=0), P.PKV_ERR_INVALID_ARG),
])
def test_cache_descriptor_errors(lib, c, want):
    assert _decode(lib, c) == want
    assert lib.kv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(c), None) == want


def test_cache_write_argument_errors(lib):
    c = desc()
    assert lib.kv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, -1, ctypes.byref(c), None) == P.PKV_ERR_INVALID_ARG
    assert lib.kv_reshape_and_cache(None, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(c), None) == P.PKV_ERR_INVALID_ARG
    assert lib.kv_reshape_and_cache(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(c), None) == \
        P.PKV_ERR_INVALID_ARG
    assert lib.kv_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 4, None, None) == P.PKV_ERR_INVALID_ARG
    # zero tokens: nothing to do, nothing enqueued
    assert lib.kv_reshape_and_cache(None, None, None, None, None, 0, ctypes.byref(c), None) == P.PKV_OK


def test_prefill_argument_errors(lib):
    c = desc()

    def call(**kw):
        a = dict(out=FAKE, dt=1, q=FAKE, cu=FAKE, mq=512, rows=2048, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=4, nq=32,
                 mb=96, scale=0.088, ws=FAKE, wsb=256)
        a.update(kw)
        return lib.paged_attention_prefill_chunk(a["out"], a["dt"], a["q"], a["cu"], a["mq"], a["rows"], a["k"],
                                                 a["v"], a["bt"], a["cl"], a["B"], a["nq"], a["mb"], a["scale"],
                                                 ctypes.byref(c), a["ws"], a["wsb"], None)
    assert call(cu=None) == P.PKV_ERR_INVALID_ARG
    assert call(nq=24) == P.PKV_ERR_UNSUPPORTED         # G = 3 does not tile 128 rows
    assert call(mq=-1) == P.PKV_ERR_INVALID_ARG
    assert call(q=FAKE + 4) == P.PKV_ERR_INVALID_ARG    # TMA needs a 16-byte aligned q
    assert call(out=FAKE + 4) == P.PKV_ERR_INVALID_ARG  # ... and out (full tiles leave by TMA store)
    assert call(wsb=8) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    assert call(ws=None) == P.PKV_ERR_INVALID_ARG
    assert call(mq=0) == P.PKV_OK                        # empty chunk: nothing enqueued


def test_prefill_window_argument_errors(lib):
    c = desc()

    def call(win, **kw):
        a = dict(out=FAKE, dt=1, q=FAKE, cu=FAKE, mq=512, rows=2048, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=4, nq=32,
                 mb=96, scale=0.088, ws=FAKE, wsb=256)
        a.update(kw)
        return lib.paged_attention_prefill_chunk_window(a["out"], a["dt"], a["q"], a["cu"], a["mq"], a["rows"],
                                                        a["k"], a["v"], a["bt"], a["cl"], a["B"], a["nq"], a["mb"],
                                                        a["scale"], win, ctypes.byref(c), a["ws"], a["wsb"], None)
    assert call(0) == P.PKV_ERR_INVALID_ARG              # a window holds at least one token
    assert call(-5) == P.PKV_ERR_INVALID_ARG
    assert call(64, cu=None) == P.PKV_ERR_INVALID_ARG
    assert call(64, nq=24) == P.PKV_ERR_UNSUPPORTED
    assert call(64, wsb=8) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    assert call(64, mq=0) == P.PKV_OK                    # empty chunk: nothing enqueued


def test_verify_window_argument_errors(lib):
    c = desc()

    def v(k, win, **kw):
        a = dict(out=FAKE, q=FAKE, B=4, nq=32, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_verify_window(a["out"], 1, a["q"], k, FAKE, FAKE, FAKE, FAKE, a["B"], a["nq"], 8,
                                                 0.088, 0, win, ctypes.byref(c), FAKE, a["wsb"], None)
    assert v(2, 0) == P.PKV_ERR_INVALID_ARG                     # a window holds at least one token
    assert v(2, -7) == P.PKV_ERR_INVALID_ARG
    assert v(0, 64) == P.PKV_ERR_INVALID_ARG
    assert v(2, 64, nq=96) == P.PKV_ERR_UNSUPPORTED             # G = 12
    assert v(2, 64, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL   # decode path
    assert v(16, 64, out=FAKE + 4, B=64) == P.PKV_ERR_INVALID_ARG  # prefill path (512 units): 16-B out


def test_verify_fp8_argument_errors(lib):
    c8 = desc(dtype=P.PKV_DTYPE_FP8_E4M3)

    def v(k, c=c8, ks=FAKE, vs=FAKE, **kw):
        a = dict(out=FAKE, q=FAKE, B=4, nq=32, wsb=1 << 20)
        a.update(kw)
        return lib.paged_attention_verify_fp8(a["out"], 1, a["q"], k, FAKE, FAKE, ks, vs, FAKE, FAKE, a["B"],
                                              a["nq"], 8, 0.088, 0, 0, ctypes.byref(c), FAKE, a["wsb"], None)
    assert v(2, ks=None) == P.PKV_ERR_INVALID_ARG                # scales are required
    assert v(2, vs=FAKE + 4) == P.PKV_ERR_INVALID_ARG            # ... 16-byte aligned
    assert v(2, c=desc()) == P.PKV_ERR_UNSUPPORTED               # a bf16 cache descriptor
    assert v(0) == P.PKV_ERR_INVALID_ARG
    assert v(2, wsb=100) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    ws = lambda k: lib.paged_attention_verify_workspace_size(64, k, 32, 256, 0, ctypes.byref(c8))  # noqa: E731
    assert ws(6) > ws(4) > 256                                   # decode kernel, one 8-column tile per CTA
    assert ws(16) == 256                                         # G * k = 64 over 512 units: the prefill kernel
    ws4 = lambda k: lib.paged_attention_verify_workspace_size(4, k, 32, 256, 0, ctypes.byref(c8))  # noqa: E731
    assert ws4(16) > ws4(8) > 256                                # 32 units: the prefill kernel splits the keys


def test_prefill_fp8_argument_errors(lib):
    c8 = desc(dtype=P.PKV_DTYPE_FP8_E4M3)

    def f(c=c8, ks=FAKE, vs=FAKE, window=0, cu=FAKE, wsb=1 << 20):
        return lib.paged_attention_prefill_chunk_fp8(FAKE, 1, FAKE, cu, 64, 256, FAKE, FAKE, ks, vs, FAKE, FAKE, 4,
                                                     32, 8, 0.088, window, ctypes.byref(c), FAKE, wsb, None)
    assert f(ks=None) == P.PKV_ERR_INVALID_ARG                   # scales are required
    assert f(vs=None) == P.PKV_ERR_INVALID_ARG
    assert f(ks=FAKE + 4) == P.PKV_ERR_INVALID_ARG               # ... 16-byte aligned
    assert f(cu=None) == P.PKV_ERR_INVALID_ARG
    assert f(window=-1) == P.PKV_ERR_INVALID_ARG
    assert f(c=desc()) == P.PKV_ERR_UNSUPPORTED                  # a bf16 cache descriptor
    assert f(wsb=2) == P.PKV_ERR_WORKSPACE_TOO_SMALL
    assert lib.paged_attention_prefill_workspace_size(4, 32, ctypes.byref(c8)) > 0


# (sequences, q heads, KV heads, k, FP8, the route measured faster on a GB300;
# decode route / prefill route in us, the prefill kernel splitting the keys of the
# 70B-shaped batch): 8B-shaped B=64 (G=4) and 70B-shaped B=8 x 32K (G=8).
MEASURED_VERIFY_ROUTES = [
    *[(64, 32, 8, k, False, "decode") for k in (2, 4, 6)],             # 104-191 vs ~207 us
    *[(64, 32, 8, k, False, "prefill") for k in (12, 16)],             # 296 / 388 vs 207 us
    *[(8, 64, 8, k, False, "decode") for k in (1, 2)],                 # 171 / 200 vs 283 / 286 us
    *[(8, 64, 8, k, False, "prefill") for k in (4, 8, 16)],            # 295 / 570 / 1122 vs 290 / 295 / 310 us
    *[(64, 32, 8, k, True, "decode") for k in (1, 2, 4, 6)],           # 70-189 vs ~244 us
    (64, 32, 8, 16, True, "prefill"),                                  # 471 vs 244 us
    *[(8, 64, 8, k, True, "decode") for k in (1, 2)],                  # 116 / 195 vs 338 / 340 us
    *[(8, 64, 8, k, True, "prefill") for k in (4, 8, 16)],             # 373 / 730 / 1445 vs 343 / 350 / 364 us
]


@pytest.mark.parametrize("nseq,nq,nkv,k,fp8,faster", MEASURED_VERIFY_ROUTES)
def test_verify_route_follows_measurements(lib, nseq, nq, nkv, k, fp8, faster):
    """Without a device the routing counts 152 SMs."""
    c = desc(num_blocks=40000, n_kv=nkv, dtype=P.PKV_DTYPE_FP8_E4M3 if fp8 else 0)
    assert lib.paged_attention_verify_workspace_size(nseq, k, nq, 2048, 0, ctypes.byref(c)) > 0
    route = lib.paged_attention_verify_on_prefill(nseq, k, nq, ctypes.byref(c))
    assert ("prefill" if route == 1 else "decode") == faster


@pytest.mark.parametrize("fp8", [False, True])
def test_verify_route_is_monotone(lib, fp8):
    """More draft positions or more sequences never move a batch from the prefill
    kernel back to the decode kernel (152 SMs without a device), for every group
    size the prefill kernel packs; group sizes it cannot pack never leave the
    decode kernel."""
    def on_prefill(nseq, n_kv, G, k):
        c = desc(num_blocks=40000, n_kv=n_kv, dtype=P.PKV_DTYPE_FP8_E4M3 if fp8 else 0)
        assert lib.paged_attention_verify_workspace_size(nseq, k, G * n_kv, 512, 0, ctypes.byref(c)) > 0
        r = lib.paged_attention_verify_on_prefill(nseq, k, G * n_kv, ctypes.byref(c))
        assert r in (0, 1)
        return r == 1
    for n_kv in (1, 8):
        for G in (1, 2, 4, 8, 16, 24):
            for nseq in (1, 4, 8, 19, 64, 200):
                route = [on_prefill(nseq, n_kv, G, k) for k in range(1, 17)]
                if G == 24:
                    assert not any(route)
                    continue
                assert route == sorted(route), (n_kv, G, nseq)           # once prefill, stays prefill in k
                more = [on_prefill(nseq + 5, n_kv, G, k) for k in range(1, 17)]
                assert all(m or not r for r, m in zip(route, more)), (n_kv, G, nseq)
