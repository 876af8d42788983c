"""fp64 CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline / reference arm may import this package.  The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``pagedkv_oracle.c`` (plain C, fp64, optional OpenMP);
this module compiles it with gcc on first use and wraps it with ctypes.  Every
wrapper takes numpy arrays (bf16 values as uint16 bit patterns) and returns
float64 arrays.

Parity pins: every function here is checked against results fixed by the
pages and by mathematics (tests/test_oracle_pins.py): a contiguous NumPy brute
force, closed forms (one key, constant scores, two keys), the sizes the pages
print (tests/golden/kv_sizes.json), repeat-interleave equivalence of GQA,
block-permutation and shared-prefix invariance, the causal-chunk identities,
the split/merge identity, the sliding-window reductions (a window covering the
context changes nothing, a window of one returns the newest V row), the E4M3
code table fixed by the format definition, and the FP8 path reducing to the
bf16 one on exactly representable values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpagedkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", *extra_flags, src, "-o",
            out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def load_library(path: str = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    if path is None:
        with _lock:
            if _lib is None:
                _lib = _declare(ctypes.CDLL(build()))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
    lib.oracle_kv_bytes_per_token.restype = i64
    lib.oracle_kv_group.argtypes = [i32, i32, i32]
    lib.oracle_kv_group.restype = i32
    lib.oracle_slot_of.argtypes = [P, i32, i32]
    lib.oracle_slot_of.restype = i64
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    lib.oracle_kv_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32]
    lib.oracle_kv_reshape_and_cache.restype = None
    lib.oracle_paged_attention.argtypes = [P, P, P, P, i32, i32, P, P, P, i32, P, i32, i32, i32, i32, f64, i32]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_paged_attention_fp8.argtypes = [P, P, P, P, i32, i32, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                               f64, i32]
    lib.oracle_paged_attention_fp8.restype = ctypes.c_int
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = f64
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_kv_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32]
    lib.oracle_kv_reshape_and_cache_fp8.restype = None
    lib.oracle_copy_blocks.argtypes = [P, P, i32, i64]
    lib.oracle_copy_blocks.restype = None
    lib.oracle_decode_partials.argtypes = [P, P, P, P, i32, i32, P, P, P, i32, P, i32, i32, i32, f64, i32, i32]
    lib.oracle_decode_partials.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [P, P, P, P, i32, i32, i32]
    lib.oracle_lse_merge.restype = None
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def kv_bytes_per_token(layers, n_kv, head_dim, dtype_size, lib=None):
    return int((lib or load_library()).oracle_kv_bytes_per_token(layers, n_kv, head_dim, dtype_size))


def kv_group(h, n_q, n_kv, lib=None):
    return int((lib or load_library()).oracle_kv_group(h, n_q, n_kv))


def slot_of(table_row, pos, block_size, lib=None):
    t, tp = _c(table_row, np.int32)
    return int((lib or load_library()).oracle_slot_of(tp, pos, block_size))


def num_threads(lib=None) -> int:
    return int((lib or load_library()).oracle_num_threads())


def set_num_threads(n: int, lib=None) -> None:
    (lib or load_library()).oracle_set_num_threads(int(n))


def kv_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, lib=None):
    """Return (k_cache', v_cache') with the new tokens written at their slots."""
    lib = lib or load_library()
    num_blocks, n_kv, bs, d = k_cache.shape
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    k, kp = _c(key, np.uint16)
    v, vp = _c(value, np.uint16)
    s, sp = _c(slot_mapping, np.int32)
    lib.oracle_kv_reshape_and_cache(kp, vp, kc.ctypes.data_as(ctypes.c_void_p),
                                    vc.ctypes.data_as(ctypes.c_void_p), sp, int(s.shape[0]),
                                    num_blocks, bs, n_kv, d)
    return kc, vc


def paged_attention(q, cu_q_lens, k_cache, v_cache, block_tables, context_lens, scale,
                    n_q=None, return_lse=False, window=0, k_scale=None, v_scale=None, lib=None):
    """fp64 attention of every query row (decode rows and causal-chunk rows alike).

    window > 0: a row at position p sees keys p - window < j <= p only.
    k_scale / v_scale given: the caches hold E4M3 codes (uint8) with one fp32
    scale per (slot, head), shape [num_blocks][n_kv][block_size]."""
    lib = lib or load_library()
    num_blocks, n_kv, bs, d = k_cache.shape
    fp8 = k_scale is not None
    q_, qp = _c(q, np.uint16)
    rows = q_.shape[0]
    n_q = q_.shape[1] if n_q is None else n_q
    cu, cup = _c(cu_q_lens, np.int32)
    kc, kcp = _c(k_cache, np.uint8 if fp8 else np.uint16)
    vc, vcp = _c(v_cache, np.uint8 if fp8 else np.uint16)
    bt, btp = _c(block_tables, np.int32)
    cl, clp = _c(context_lens, np.int32)
    out = np.zeros((rows, n_q, d), dtype=np.float64)
    lse = np.zeros((rows, n_q), dtype=np.float64) if return_lse else None
    lp = lse.ctypes.data_as(ctypes.c_void_p) if return_lse else None
    if fp8:
        ks, ksp = _c(k_scale, np.float32)
        vs, vsp = _c(v_scale, np.float32)
        rc = lib.oracle_paged_attention_fp8(out.ctypes.data_as(ctypes.c_void_p), lp, qp, cup, int(cl.shape[0]),
                                            n_q, kcp, vcp, ksp, vsp, btp, int(bt.shape[1]), clp, num_blocks,
                                            n_kv, bs, d, float(scale), int(window))
    else:
        rc = lib.oracle_paged_attention(out.ctypes.data_as(ctypes.c_void_p), lp, qp, cup, int(cl.shape[0]),
                                        n_q, kcp, vcp, btp, int(bt.shape[1]), clp, num_blocks, n_kv, bs, d,
                                        float(scale), int(window))
    if rc != 0:
        raise ValueError("oracle_paged_attention rejected its arguments")
    return (out, lse) if return_lse else out


def e4m3_decode(codes, lib=None):
    """Real value of each E4M3 code (uint8 array -> float64 array)."""
    lib = lib or load_library()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e4m3_encode(x, lib=None):
    """Nearest-even E4M3 code of each fp32 value (saturating at 448)."""
    lib = lib or load_library()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def kv_reshape_and_cache_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, lib=None):
    """Return (k_cache', v_cache', k_scale', v_scale') with the new tokens quantised into their slots."""
    lib = lib or load_library()
    num_blocks, n_kv, bs, d = k_cache.shape
    kc = np.array(k_cache, dtype=np.uint8, copy=True)
    vc = np.array(v_cache, dtype=np.uint8, copy=True)
    ks = np.array(k_scale, dtype=np.float32, copy=True)
    vs = np.array(v_scale, dtype=np.float32, copy=True)
    k, kp = _c(key, np.uint16)
    v, vp = _c(value, np.uint16)
    s, sp = _c(slot_mapping, np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    lib.oracle_kv_reshape_and_cache_fp8(kp, vp, ptr(kc), ptr(vc), ptr(ks), ptr(vs), sp, int(s.shape[0]),
                                        num_blocks, bs, n_kv, d)
    return kc, vc, ks, vs


def copy_blocks(cache, pairs, lib=None):
    """Return a copy of `cache` ([num_blocks, ...], any dtype) with block pairs[i][0] copied onto pairs[i][1]."""
    lib = lib or load_library()
    out = np.array(cache, copy=True)
    pr, pp = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), np.int32)
    block_bytes = out.nbytes // out.shape[0]
    lib.oracle_copy_blocks(out.ctypes.data_as(ctypes.c_void_p), pp, int(pr.shape[0]), int(block_bytes))
    return out


def decode_partials(q, k_cache, v_cache, block_tables, context_lens, scale, part_tokens, lib=None):
    """Flash-Decoding partials (m, l, o) of every (sequence, head, part)."""
    lib = lib or load_library()
    num_blocks, n_kv, bs, d = k_cache.shape
    q_, qp = _c(q, np.uint16)
    B, n_q, _ = q_.shape
    cl, clp = _c(context_lens, np.int32)
    max_parts = int(max(1, -(-int(cl.max()) // part_tokens)))
    m = np.zeros((B, n_q, max_parts)); l = np.zeros_like(m)
    o = np.zeros((B, n_q, max_parts, d))
    kc, kcp = _c(k_cache, np.uint16)
    vc, vcp = _c(v_cache, np.uint16)
    bt, btp = _c(block_tables, np.int32)
    rc = lib.oracle_decode_partials(m.ctypes.data_as(ctypes.c_void_p), l.ctypes.data_as(ctypes.c_void_p),
                                    o.ctypes.data_as(ctypes.c_void_p), qp, B, n_q, kcp, vcp, btp,
                                    int(bt.shape[1]), clp, n_kv, bs, d, float(scale), int(part_tokens),
                                    max_parts)
    if rc != 0:
        raise ValueError("oracle_decode_partials rejected its arguments")
    return m, l, o


def lse_merge(m, l, o, lib=None):
    lib = lib or load_library()
    B, n_q, P = m.shape
    d = o.shape[-1]
    out = np.zeros((B, n_q, d))
    m_, mp = _c(m, np.float64)
    l_, lp = _c(l, np.float64)
    o_, op = _c(o, np.float64)
    lib.oracle_lse_merge(out.ctypes.data_as(ctypes.c_void_p), mp, lp, op, B * n_q, P, d)
    return out
