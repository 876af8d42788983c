"""ctypes binding of libpagedkv.so (the C ABI in include/pagedkv.h).

Argument marshalling only: every function checks that the torch tensors it
is given have the dtype, device, shape and contiguity the C ABI documents,
then passes their device pointers, sizes and the current CUDA stream to the
entry point of the same name.  All computation happens in the library's CUDA
kernels; there is no fallback of any kind.  If the library is missing, the
first call raises ``RuntimeError`` (build it with ``__graft_entry__.build()``
or ``python -m paged_kv_cache_95_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

PKV_DTYPE_BF16 = 0
PKV_DTYPE_FLOAT32 = 1
PKV_DTYPE_FP8_E4M3 = 2

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE_TOO_SMALL = -3
PKV_ERR_CUDA = -4
PKV_ERR_OUT_OF_BLOCKS = -5

PKV_STATUS_BAD_CONTEXT_LEN = 0x1
PKV_STATUS_BAD_BLOCK_ID = 0x2
PKV_STATUS_BAD_Q_LEN = 0x4
PKV_STATUS_TIMEOUT = 0x8

PKV_VERIFY_AUTO = -1
PKV_VERIFY_DECODE_KERNEL = 0
PKV_VERIFY_PREFILL_KERNEL = 1

HEAD_DIM = 128
BLOCK_SIZE = 16
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024  # PKV_STATIC_SCRATCH_BYTES

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")
HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedkv.h")

_lock = threading.Lock()
_lib = None


class CacheDesc(ctypes.Structure):
    """Mirror of ``pkv_cache_desc``."""

    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpagedkv.so and declare the C signatures."""
    global _lib
    if path is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                                       "(python -c 'import __graft_entry__ as g; g.build()')")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib):
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(CacheDesc)
    lib.kv_reshape_and_cache.argtypes = [P, P, P, P, P, i32, D, P]
    lib.kv_reshape_and_cache.restype = ctypes.c_int
    lib.paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, D]
    lib.paged_attention_workspace_size.restype = sz
    lib.paged_attention_decode_partitions.argtypes = [i32, i32, i32, i32, i32, D]
    lib.paged_attention_decode_partitions.restype = i32
    lib.paged_attention_decode.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, f32, i32, D, P, sz, P]
    lib.paged_attention_decode.restype = ctypes.c_int
    lib.paged_attention_decode_append.argtypes = [P, i32, P, P, P, P, P, P, P, i32, i32, i32, f32, i32, D, P, sz, P]
    lib.paged_attention_decode_append.restype = ctypes.c_int
    lib.paged_attention_decode_window.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, f32, i32, i32, D, P, sz, P]
    lib.paged_attention_decode_window.restype = ctypes.c_int
    lib.paged_attention_decode_fp8.argtypes = [P, i32, P, P, P, P, P, P, P, i32, i32, i32, f32, i32, i32, D, P, sz, P]
    lib.paged_attention_decode_fp8.restype = ctypes.c_int
    lib.paged_attention_verify_workspace_size.argtypes = [i32, i32, i32, i32, i32, D]
    lib.paged_attention_verify_workspace_size.restype = sz
    lib.paged_attention_verify.argtypes = [P, i32, P, i32, P, P, P, P, i32, i32, i32, f32, i32, D, P, sz, P]
    lib.paged_attention_verify.restype = ctypes.c_int
    lib.paged_attention_verify_window.argtypes = [P, i32, P, i32, P, P, P, P, i32, i32, i32, f32, i32, i32, D, P, sz,
                                                  P]
    lib.paged_attention_verify_window.restype = ctypes.c_int
    lib.paged_attention_verify_fp8.argtypes = [P, i32, P, i32, P, P, P, P, P, P, i32, i32, i32, f32, i32, i32, D, P,
                                               sz, P]
    lib.paged_attention_verify_fp8.restype = ctypes.c_int
    lib.paged_attention_verify_workspace_size_on.argtypes = [i32, i32, i32, i32, i32, i32, D]
    lib.paged_attention_verify_workspace_size_on.restype = sz
    lib.paged_attention_verify_on.argtypes = [i32, P, i32, P, i32, P, P, P, P, P, P, i32, i32, i32, f32, i32, i32, D,
                                              P, sz, P]
    lib.paged_attention_verify_on.restype = ctypes.c_int
    lib.kv_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, P, P, i32, D, P]
    lib.kv_reshape_and_cache_fp8.restype = ctypes.c_int
    lib.paged_attention_prefill_workspace_size.argtypes = [i32, i32, D]
    lib.paged_attention_prefill_workspace_size.restype = sz
    lib.paged_attention_verify_on_prefill.argtypes = [i32, i32, i32, D]
    lib.paged_attention_verify_on_prefill.restype = ctypes.c_int
    lib.paged_attention_prefill_chunk_workspace_size.argtypes = [i32, i32, i32, i32, i32, D]
    lib.paged_attention_prefill_chunk_workspace_size.restype = sz
    lib.paged_attention_prefill_chunk.argtypes = [P, i32, P, P, i32, i32, P, P, P, P, i32, i32, i32, f32, D, P, sz, P]
    lib.paged_attention_prefill_chunk.restype = ctypes.c_int
    lib.paged_attention_prefill_chunk_window.argtypes = [P, i32, P, P, i32, i32, P, P, P, P, i32, i32, i32, f32, i32,
                                                         D, P, sz, P]
    lib.paged_attention_prefill_chunk_window.restype = ctypes.c_int
    lib.paged_attention_prefill_chunk_fp8.argtypes = [P, i32, P, P, i32, i32, P, P, P, P, P, P, i32, i32, i32, f32,
                                                      i32, D, P, sz, P]
    lib.paged_attention_prefill_chunk_fp8.restype = ctypes.c_int
    lib.paged_attention_decode_static_scratch.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, f32, i32, D, P, P]
    lib.paged_attention_decode_static_scratch.restype = ctypes.c_int
    lib.kv_copy_blocks.argtypes = [P, P, P, P, P, i32, D, P]
    lib.kv_copy_blocks.restype = ctypes.c_int
    i64, I = ctypes.c_int64, ctypes.c_int
    lib.pkv_bm_create.argtypes = [i32, ctypes.POINTER(P)]
    lib.pkv_bm_create.restype = I
    lib.pkv_bm_destroy.argtypes = [P]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_num_free.argtypes = [P]
    lib.pkv_bm_num_free.restype = i32
    lib.pkv_bm_ref_count.argtypes = [P, i32, P]
    lib.pkv_bm_ref_count.restype = I
    lib.pkv_bm_add_sequence.argtypes = [P, i64]
    lib.pkv_bm_add_sequence.restype = I
    lib.pkv_bm_fork.argtypes = [P, i64, i64]
    lib.pkv_bm_fork.restype = I
    lib.pkv_bm_append.argtypes = [P, i64, i32, P, P, P]
    lib.pkv_bm_append.restype = I
    lib.pkv_bm_append_batch.argtypes = [P, P, i32, P, P, P, P]
    lib.pkv_bm_append_batch.restype = I
    lib.pkv_bm_free_sequence.argtypes = [P, i64]
    lib.pkv_bm_free_sequence.restype = I
    lib.pkv_bm_sequence_length.argtypes = [P, i64, P]
    lib.pkv_bm_sequence_length.restype = I
    lib.pkv_bm_block_tables.argtypes = [P, P, i32, i32, i32, P, P]
    lib.pkv_bm_block_tables.restype = I
    lib.pkv_bm_publish.argtypes = [P, i64, P, i32]
    lib.pkv_bm_publish.restype = I
    lib.pkv_bm_add_sequence_cached.argtypes = [P, i64, P, i32, P]
    lib.pkv_bm_add_sequence_cached.restype = I
    lib.pagedkv_status_string.argtypes = [ctypes.c_int]
    lib.pagedkv_status_string.restype = ctypes.c_char_p
    lib.pagedkv_version.argtypes = []
    lib.pagedkv_version.restype = ctypes.c_int
    return lib


def status_string(code: int) -> str:
    try:
        return load_library().pagedkv_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def version() -> int:
    return int(load_library().pagedkv_version())


# ---- tensor marshalling ----------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> int:
    return int(t.data_ptr())


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    return int(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check(t, name, dtype, ndim=None, last=None):
    torch = _torch()
    _need(isinstance(t, torch.Tensor), f"{name} must be a torch.Tensor")
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    _need(t.is_contiguous(), f"{name} must be contiguous")
    if ndim is not None:
        _need(t.dim() == ndim, f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if last is not None:
        _need(t.shape[-1] == last, f"{name} last dim must be {last}")


def cache_desc(k_cache) -> CacheDesc:
    """Descriptor of a pool tensor [num_blocks, n_kv, 16, 128]: bf16, or FP8 E4M3 codes
    (torch.float8_e4m3fn or uint8)."""
    torch = _torch()
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    _check(k_cache, "k_cache", k_cache.dtype if fp8 else torch.bfloat16, ndim=4, last=HEAD_DIM)
    nb, n_kv, bs, d = k_cache.shape
    return CacheDesc(int(nb), int(bs), int(n_kv), int(d), PKV_DTYPE_FP8_E4M3 if fp8 else PKV_DTYPE_BF16)


def _out_dtype(out) -> int:
    torch = _torch()
    if out.dtype == torch.float32:
        return PKV_DTYPE_FLOAT32
    if out.dtype == torch.bfloat16:
        return PKV_DTYPE_BF16
    raise ValueError(f"out must be float32 or bfloat16, got {out.dtype}")


def _raise(fn, rc):
    if rc != PKV_OK:
        raise PagedKVError(fn, rc)


# ---- entry points (same names as the C ABI) ----------------------------------------

def kv_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    torch = _torch()
    desc = cache_desc(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(key, "key", torch.bfloat16, ndim=3, last=HEAD_DIM)
    _check(value, "value", torch.bfloat16, ndim=3, last=HEAD_DIM)
    _check(slot_mapping, "slot_mapping", torch.int32, ndim=1)
    T = slot_mapping.shape[0]
    _need(tuple(key.shape) == (T, desc.num_kv_heads, HEAD_DIM), "key must be [num_tokens, n_kv, 128]")
    _need(tuple(value.shape) == tuple(key.shape), "value shape must equal key shape")
    rc = load_library().kv_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                             _ptr(slot_mapping), int(T), ctypes.byref(desc), _stream(stream))
    _raise("kv_reshape_and_cache", rc)


def _check_fp8_pool(k_cache, v_cache, k_scale, v_scale):
    torch = _torch()
    desc = cache_desc(k_cache)
    _need(desc.dtype == PKV_DTYPE_FP8_E4M3, "k_cache must hold E4M3 codes (torch.float8_e4m3fn or uint8)")
    _check(v_cache, "v_cache", k_cache.dtype, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need(t is not None, f"{name} is required for an FP8 cache")
        _check(t, name, torch.float32, ndim=3)
        _need(tuple(t.shape) == tuple(k_cache.shape[:3]), f"{name} must be [num_blocks, n_kv, 16]")
    return desc


def kv_reshape_and_cache_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, stream=None) -> None:
    """Quantise new tokens' K/V to E4M3 (one fp32 scale per token and KV head) into their slots."""
    torch = _torch()
    desc = _check_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    _check(key, "key", torch.bfloat16, ndim=3, last=HEAD_DIM)
    _check(value, "value", torch.bfloat16, ndim=3, last=HEAD_DIM)
    _check(slot_mapping, "slot_mapping", torch.int32, ndim=1)
    T = slot_mapping.shape[0]
    _need(tuple(key.shape) == (T, desc.num_kv_heads, HEAD_DIM), "key must be [num_tokens, n_kv, 128]")
    _need(tuple(value.shape) == tuple(key.shape), "value shape must equal key shape")
    rc = load_library().kv_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                 _ptr(v_scale), _ptr(slot_mapping), int(T), ctypes.byref(desc),
                                                 _stream(stream))
    _raise("kv_reshape_and_cache_fp8", rc)


def kv_copy_blocks(k_cache, v_cache, block_pairs, k_scale=None, v_scale=None, stream=None) -> None:
    """Copy block pairs {source, destination} (int32 CUDA tensor [n, 2]) in both caches
    (and, for an FP8 cache, in both scale arrays)."""
    torch = _torch()
    desc = cache_desc(k_cache)
    _check(v_cache, "v_cache", k_cache.dtype, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(block_pairs, "block_pairs", torch.int32, ndim=2, last=2)
    fp8 = desc.dtype == PKV_DTYPE_FP8_E4M3
    _need(fp8 == (k_scale is not None) and fp8 == (v_scale is not None),
          "k_scale and v_scale are required for an FP8 cache and not allowed otherwise")
    if fp8:
        for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
            _check(t, name, torch.float32, ndim=3)
            _need(tuple(t.shape) == tuple(k_cache.shape[:3]), f"{name} must be [num_blocks, n_kv, 16]")
    rc = load_library().kv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale) if fp8 else None,
                                       _ptr(v_scale) if fp8 else None, _ptr(block_pairs),
                                       int(block_pairs.shape[0]), ctypes.byref(desc), _stream(stream))
    _raise("kv_copy_blocks", rc)


class BlockManager:
    """Host block manager of the paged pool (``pkv_bm_*`` in include/pagedkv.h).

    Sequences are keyed by caller-chosen integers.  ``append`` returns the slot
    mapping of the new tokens and, when the sequence's shared last block had to
    be replaced first, the (source, destination) block pair to copy on the
    device with :func:`kv_copy_blocks` before writing the tokens.
    """

    def __init__(self, num_blocks: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _raise("pkv_bm_create", self._lib.pkv_bm_create(int(num_blocks), ctypes.byref(h)))
        self._h = h
        self.num_blocks = int(num_blocks)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @property
    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        c = ctypes.c_int32()
        _raise("pkv_bm_ref_count", self._lib.pkv_bm_ref_count(self._h, int(block), ctypes.byref(c)))
        return c.value

    def add(self, seq_id: int) -> None:
        _raise("pkv_bm_add_sequence", self._lib.pkv_bm_add_sequence(self._h, int(seq_id)))

    def fork(self, parent_id: int, child_id: int) -> None:
        _raise("pkv_bm_fork", self._lib.pkv_bm_fork(self._h, int(parent_id), int(child_id)))

    def append(self, seq_id: int, num_tokens: int):
        """Returns (slot_mapping int32 numpy [num_tokens], copy pair (src, dst) or None)."""
        import numpy as np
        slots = np.zeros(max(int(num_tokens), 1), dtype=np.int32)
        pair = np.zeros(2, dtype=np.int32)
        n = ctypes.c_int32()
        rc = self._lib.pkv_bm_append(self._h, int(seq_id), int(num_tokens), slots.ctypes.data,
                                     pair.ctypes.data, ctypes.byref(n))
        _raise("pkv_bm_append", rc)
        return slots[:int(num_tokens)], ((int(pair[0]), int(pair[1])) if n.value else None)

    def append_batch(self, seq_ids, num_tokens=None):
        """One call for a batch: returns (slot_mapping int32 [sum of num_tokens],
        copy pairs int32 [n_copies, 2]); num_tokens None means one token each."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = len(ids)
        nt = None if num_tokens is None else np.ascontiguousarray(num_tokens, dtype=np.int32)
        total = n if nt is None else int(nt.sum())
        slots = np.zeros(max(total, 1), dtype=np.int32)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int32)
        c = ctypes.c_int32()
        rc = self._lib.pkv_bm_append_batch(self._h, ids.ctypes.data, n, None if nt is None else nt.ctypes.data,
                                           slots.ctypes.data, pairs.ctypes.data, ctypes.byref(c))
        _raise("pkv_bm_append_batch", rc)
        return slots[:total], pairs[:c.value]

    def free(self, seq_id: int) -> None:
        _raise("pkv_bm_free_sequence", self._lib.pkv_bm_free_sequence(self._h, int(seq_id)))

    def length(self, seq_id: int) -> int:
        n = ctypes.c_int64()
        _raise("pkv_bm_sequence_length", self._lib.pkv_bm_sequence_length(self._h, int(seq_id), ctypes.byref(n)))
        return n.value

    def block_tables(self, seq_ids, max_blocks_per_seq: int, pad_block: int = 0):
        """Returns (block_tables int32 [B, max_blocks], context_lens int32 [B]) as numpy arrays."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.zeros((max(len(ids), 1), int(max_blocks_per_seq)), dtype=np.int32)
        lens = np.zeros(max(len(ids), 1), dtype=np.int32)
        rc = self._lib.pkv_bm_block_tables(self._h, ids.ctypes.data, int(len(ids)), int(max_blocks_per_seq),
                                           int(pad_block), tables.ctypes.data, lens.ctypes.data)
        _raise("pkv_bm_block_tables", rc)
        return tables[:len(ids)], lens[:len(ids)]

    def publish(self, seq_id: int, tokens) -> None:
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _raise("pkv_bm_publish", self._lib.pkv_bm_publish(self._h, int(seq_id), t.ctypes.data, int(t.shape[0])))

    def add_cached(self, seq_id: int, tokens) -> int:
        """New sequence for prompt `tokens`; returns how many leading tokens are already cached."""
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int32()
        rc = self._lib.pkv_bm_add_sequence_cached(self._h, int(seq_id), t.ctypes.data, int(t.shape[0]),
                                                  ctypes.byref(n))
        _raise("pkv_bm_add_sequence_cached", rc)
        return n.value


def paged_attention_workspace_size(num_seqs: int, num_q_heads: int, max_blocks_per_seq: int,
                                   partition_size: int, cache: CacheDesc) -> int:
    return int(load_library().paged_attention_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq,
                                                             partition_size, ctypes.byref(cache)))


def paged_attention_decode_partitions(num_seqs: int, num_q_heads: int, max_blocks_per_seq: int,
                                      partition_size: int, cache: CacheDesc, window: int = 0) -> int:
    """Partitions per sequence the decode entry points use (1: no merge kernel)."""
    n = int(load_library().paged_attention_decode_partitions(num_seqs, num_q_heads, max_blocks_per_seq,
                                                             partition_size, window, ctypes.byref(cache)))
    _raise("paged_attention_decode_partitions", min(n, 0))
    return n


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           workspace=None, partition_size: int = 0, stream=None, window: int = 0,
                           k_scale=None, v_scale=None):
    """Decode attention; ``workspace`` (uint8 CUDA tensor) is allocated if None.
    ``window`` > 0 calls paged_attention_decode_window (each row sees its newest
    ``window`` keys only).  An FP8 pool (E4M3 codes) with ``k_scale`` /
    ``v_scale`` calls paged_attention_decode_fp8."""
    torch = _torch()
    desc = cache_desc(k_cache)
    fp8 = desc.dtype == PKV_DTYPE_FP8_E4M3
    if fp8:
        _check_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    else:
        _need(k_scale is None and v_scale is None, "scales are only for an FP8 cache")
        _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(q, "q", torch.bfloat16, ndim=3, last=HEAD_DIM)
    B, n_q, _ = q.shape
    _check(out, "out", out.dtype, ndim=3)
    _need(tuple(out.shape) == tuple(q.shape), "out must have q's shape")
    _check(block_tables, "block_tables", torch.int32, ndim=2)
    _check(context_lens, "context_lens", torch.int32, ndim=1)
    _need(block_tables.shape[0] == B and context_lens.shape[0] == B, "one table row and length per sequence")
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        nbytes = paged_attention_workspace_size(B, n_q, max_blocks, partition_size, desc)
        _need(nbytes > 0, "invalid sizes for paged_attention_decode")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)  # status word starts clear
    _check(workspace, "workspace", torch.uint8, ndim=1)
    lib = load_library()
    if fp8:
        rc = lib.paged_attention_decode_fp8(
            _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), _ptr(context_lens), int(B), int(n_q), max_blocks, float(scale), int(window),
            int(partition_size), ctypes.byref(desc), _ptr(workspace), int(workspace.numel()), _stream(stream))
        _raise("paged_attention_decode_fp8", rc)
        return workspace
    if window:
        rc = lib.paged_attention_decode_window(
            _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), int(B), int(n_q), max_blocks, float(scale), int(window), int(partition_size),
            ctypes.byref(desc), _ptr(workspace), int(workspace.numel()), _stream(stream))
        _raise("paged_attention_decode_window", rc)
        return workspace
    rc = lib.paged_attention_decode(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        int(B), int(n_q), max_blocks, float(scale), int(partition_size), ctypes.byref(desc), _ptr(workspace),
        int(workspace.numel()), _stream(stream))
    _raise("paged_attention_decode", rc)
    return workspace


def paged_attention_verify(out, q, q_per_seq: int, k_cache, v_cache, block_tables, context_lens, scale: float,
                           workspace=None, partition_size: int = 0, stream=None, window: int = 0,
                           k_scale=None, v_scale=None, kernel: int = -1):
    """Verify k = q_per_seq draft positions per sequence: q / out [num_seqs * k, n_q, 128],
    row i of sequence b at position ctx_b - k + i (causal).  ``window`` > 0: row at pos
    sees pos - window < j <= pos.  An FP8 pool with ``k_scale`` / ``v_scale`` calls
    paged_attention_verify_fp8.  ``kernel`` (PKV_VERIFY_DECODE_KERNEL or
    PKV_VERIFY_PREFILL_KERNEL) forces one kernel through paged_attention_verify_on;
    PKV_VERIFY_AUTO lets the library's measured rule choose.  Returns the workspace."""
    torch = _torch()
    desc = cache_desc(k_cache)
    fp8 = desc.dtype == PKV_DTYPE_FP8_E4M3
    if fp8:
        _check_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    else:
        _need(k_scale is None and v_scale is None, "scales are only for an FP8 cache")
        _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(q, "q", torch.bfloat16, ndim=3, last=HEAD_DIM)
    rows, n_q, _ = q.shape
    _check(out, "out", out.dtype, ndim=3)
    _need(tuple(out.shape) == tuple(q.shape), "out must have q's shape")
    _check(block_tables, "block_tables", torch.int32, ndim=2)
    _check(context_lens, "context_lens", torch.int32, ndim=1)
    B = int(context_lens.shape[0])
    _need(block_tables.shape[0] == B and rows == B * int(q_per_seq), "q must hold q_per_seq rows per sequence")
    max_blocks = int(block_tables.shape[1])
    lib = load_library()
    if workspace is None:
        nbytes = int(lib.paged_attention_verify_workspace_size_on(int(kernel), B, int(q_per_seq), n_q, max_blocks,
                                                                  int(partition_size), ctypes.byref(desc)))
        _need(nbytes > 0, "invalid sizes for paged_attention_verify")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8, ndim=1)
    if kernel != PKV_VERIFY_AUTO:
        rc = lib.paged_attention_verify_on(int(kernel), _ptr(out), _out_dtype(out), _ptr(q), int(q_per_seq),
                                           _ptr(k_cache), _ptr(v_cache), _ptr(k_scale) if fp8 else None,
                                           _ptr(v_scale) if fp8 else None, _ptr(block_tables), _ptr(context_lens), B,
                                           int(n_q), max_blocks, float(scale), int(window), int(partition_size),
                                           ctypes.byref(desc), _ptr(workspace), int(workspace.numel()),
                                           _stream(stream))
        _raise("paged_attention_verify_on", rc)
        return workspace
    if fp8:
        rc = lib.paged_attention_verify_fp8(_ptr(out), _out_dtype(out), _ptr(q), int(q_per_seq), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                            _ptr(context_lens), B, int(n_q), max_blocks, float(scale), int(window),
                                            int(partition_size), ctypes.byref(desc), _ptr(workspace),
                                            int(workspace.numel()), _stream(stream))
        _raise("paged_attention_verify_fp8", rc)
        return workspace
    if window:
        rc = lib.paged_attention_verify_window(_ptr(out), _out_dtype(out), _ptr(q), int(q_per_seq), _ptr(k_cache),
                                               _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, int(n_q),
                                               max_blocks, float(scale), int(partition_size), int(window),
                                               ctypes.byref(desc), _ptr(workspace), int(workspace.numel()),
                                               _stream(stream))
        _raise("paged_attention_verify_window", rc)
        return workspace
    rc = lib.paged_attention_verify(_ptr(out), _out_dtype(out), _ptr(q), int(q_per_seq), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, int(n_q), max_blocks,
                                    float(scale), int(partition_size), ctypes.byref(desc), _ptr(workspace),
                                    int(workspace.numel()), _stream(stream))
    _raise("paged_attention_verify", rc)
    return workspace


def paged_attention_prefill_workspace_size(num_seqs: int, num_q_heads: int, cache: CacheDesc) -> int:
    return int(load_library().paged_attention_prefill_workspace_size(num_seqs, num_q_heads, ctypes.byref(cache)))


def paged_attention_prefill_chunk_workspace_size(num_seqs: int, num_q_heads: int, total_q_rows: int, max_q_len: int,
                                                 max_blocks_per_seq: int, cache: CacheDesc) -> int:
    """Workspace bytes with which the prefill chunk may split its keys (split-KV)."""
    return int(load_library().paged_attention_prefill_chunk_workspace_size(
        num_seqs, num_q_heads, total_q_rows, max_q_len, max_blocks_per_seq, ctypes.byref(cache)))


def paged_attention_prefill_chunk(out, q, cu_q_lens, max_q_len: int, k_cache, v_cache, block_tables, context_lens,
                                  scale: float, workspace=None, stream=None, window: int = 0, k_scale=None,
                                  v_scale=None):
    """Causal chunked-prefill attention; ``workspace`` is allocated if None.
    ``window`` > 0 calls paged_attention_prefill_chunk_window (row at pos sees
    keys pos - window < j <= pos); an FP8 cache with ``k_scale`` / ``v_scale``
    calls paged_attention_prefill_chunk_fp8."""
    torch = _torch()
    fp8 = k_scale is not None or v_scale is not None
    if fp8:
        desc = _check_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    else:
        desc = cache_desc(k_cache)
        _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
        _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(q, "q", torch.bfloat16, ndim=3, last=HEAD_DIM)
    rows, n_q, _ = q.shape
    _check(out, "out", out.dtype, ndim=3)
    _need(tuple(out.shape) == tuple(q.shape), "out must have q's shape")
    _check(cu_q_lens, "cu_q_lens", torch.int32, ndim=1)
    _check(block_tables, "block_tables", torch.int32, ndim=2)
    _check(context_lens, "context_lens", torch.int32, ndim=1)
    B = int(context_lens.shape[0])
    _need(cu_q_lens.shape[0] == B + 1 and block_tables.shape[0] == B, "cu_q_lens is [B+1], block_tables [B, *]")
    if workspace is None:
        nbytes = paged_attention_prefill_chunk_workspace_size(B, n_q, int(rows), int(max_q_len),
                                                              int(block_tables.shape[1]), desc)
        _need(nbytes > 0, "invalid sizes for paged_attention_prefill_chunk")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)  # status word starts clear
    _check(workspace, "workspace", torch.uint8, ndim=1)
    lib = load_library()
    if fp8:
        rc = lib.paged_attention_prefill_chunk_fp8(
            _ptr(out), _out_dtype(out), _ptr(q), _ptr(cu_q_lens), int(max_q_len), int(rows), _ptr(k_cache),
            _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(context_lens), B, int(n_q),
            int(block_tables.shape[1]), float(scale), int(window), ctypes.byref(desc), _ptr(workspace),
            int(workspace.numel()), _stream(stream))
        _raise("paged_attention_prefill_chunk_fp8", rc)
        return workspace
    if window:
        rc = lib.paged_attention_prefill_chunk_window(
            _ptr(out), _out_dtype(out), _ptr(q), _ptr(cu_q_lens), int(max_q_len), int(rows), _ptr(k_cache),
            _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, int(n_q), int(block_tables.shape[1]),
            float(scale), int(window), ctypes.byref(desc), _ptr(workspace), int(workspace.numel()), _stream(stream))
        _raise("paged_attention_prefill_chunk_window", rc)
        return workspace
    rc = lib.paged_attention_prefill_chunk(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(cu_q_lens), int(max_q_len), int(rows), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, int(n_q), int(block_tables.shape[1]),
        float(scale), ctypes.byref(desc), _ptr(workspace), int(workspace.numel()), _stream(stream))
    _raise("paged_attention_prefill_chunk", rc)
    return workspace


def paged_attention_decode_append(out, q, key, value, k_cache, v_cache, block_tables, context_lens, scale: float,
                                  workspace=None, partition_size: int = 0, stream=None):
    """One decode step in one launch: writes ``key`` / ``value`` (bf16
    [B, n_kv, 128], each sequence's row of position ctx - 1) into the pool and
    attends, as kv_reshape_and_cache + paged_attention_decode would."""
    torch = _torch()
    desc = cache_desc(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(q, "q", torch.bfloat16, ndim=3, last=HEAD_DIM)
    B, n_q, _ = q.shape
    n_kv = int(k_cache.shape[1])
    for name, t in (("key", key), ("value", value)):
        _check(t, name, torch.bfloat16, ndim=3, last=HEAD_DIM)
        _need(tuple(t.shape) == (B, n_kv, HEAD_DIM), f"{name} must be [num_seqs, num_kv_heads, 128]")
    _check(out, "out", out.dtype, ndim=3)
    _need(tuple(out.shape) == tuple(q.shape), "out must have q's shape")
    _check(block_tables, "block_tables", torch.int32, ndim=2)
    _check(context_lens, "context_lens", torch.int32, ndim=1)
    _need(block_tables.shape[0] == B and context_lens.shape[0] == B, "one table row and length per sequence")
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        nbytes = paged_attention_workspace_size(B, n_q, max_blocks, partition_size, desc)
        _need(nbytes > 0, "invalid sizes for paged_attention_decode_append")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8, ndim=1)
    rc = load_library().paged_attention_decode_append(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), int(B), int(n_q), max_blocks, float(scale), int(partition_size),
        ctypes.byref(desc), _ptr(workspace), int(workspace.numel()), _stream(stream))
    _raise("paged_attention_decode_append", rc)
    return workspace


def paged_attention_decode_static_scratch(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                          partition_size: int = 0, status=None, stream=None) -> None:
    """Decode attention that allocates nothing: the split-KV scratch is the
    library's fixed device array (STATIC_SCRATCH_BYTES), shared by all calls on
    a device, so calls must not overlap on the GPU.  ``status`` is an optional
    int32 CUDA tensor of one element that receives the call's status bits."""
    torch = _torch()
    desc = cache_desc(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, ndim=4)
    _need(tuple(v_cache.shape) == tuple(k_cache.shape), "v_cache shape must equal k_cache shape")
    _check(q, "q", torch.bfloat16, ndim=3, last=HEAD_DIM)
    B, n_q, _ = q.shape
    _check(out, "out", out.dtype, ndim=3)
    _need(tuple(out.shape) == tuple(q.shape), "out must have q's shape")
    _check(block_tables, "block_tables", torch.int32, ndim=2)
    _check(context_lens, "context_lens", torch.int32, ndim=1)
    if status is not None:
        _check(status, "status", torch.int32, ndim=1)
    rc = load_library().paged_attention_decode_static_scratch(
        _ptr(out), _out_dtype(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        int(B), int(n_q), int(block_tables.shape[1]), float(scale), int(partition_size), ctypes.byref(desc),
        _ptr(status) if status is not None else None, _stream(stream))
    _raise("paged_attention_decode_static_scratch", rc)
