"""Block copy at a branch (kv_copy_blocks) and the host block manager driving the
CUDA path end to end, against the fp64 oracle (GPU).

Sources: xinc.fun archive 233, section 6 (shared prefixes and parallel
candidates reference the same blocks until they branch, where a new block is
allocated); "注意力演进与推理流程", 变革 1 (blocks allocated on demand) and 变革 3
(prefix caching).
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, bf16_to_dev, dev_to_bf16_bits, i32_to_dev, torch
from paged_kv_cache_95_gb300 import pagedkv as P
from paged_kv_cache_95_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BS, D = 16, 128


def test_copy_blocks_bf16_bit_exact(built_library):
    t = torch()
    rng = np.random.default_rng(40)
    nb, n_kv = 64, 8
    k = rng.integers(0, 2 ** 16, size=(nb, n_kv, BS, D), dtype=np.uint16)
    v = rng.integers(0, 2 ** 16, size=(nb, n_kv, BS, D), dtype=np.uint16)
    pairs = np.array([[3, 40], [0, 63], [17, 5], [62, 1], [9, 10], [2, 2 + 30]], dtype=np.int32)
    kd, vd = bf16_to_dev(k), bf16_to_dev(v)
    P.kv_copy_blocks(kd, vd, i32_to_dev(pairs))
    t.cuda.synchronize()
    assert np.array_equal(dev_to_bf16_bits(kd), oracle.copy_blocks(k, pairs))
    assert np.array_equal(dev_to_bf16_bits(vd), oracle.copy_blocks(v, pairs))


def test_copy_blocks_fp8_with_scales(built_library):
    t = torch()
    rng = np.random.default_rng(41)
    nb, n_kv = 32, 2
    k = rng.integers(0, 256, size=(nb, n_kv, BS, D), dtype=np.uint8)
    v = rng.integers(0, 256, size=(nb, n_kv, BS, D), dtype=np.uint8)
    ks = rng.standard_normal((nb, n_kv, BS)).astype(np.float32)
    vs = rng.standard_normal((nb, n_kv, BS)).astype(np.float32)
    pairs = np.array([[1, 30], [31, 0], [7, 8]], dtype=np.int32)
    dev = [t.from_numpy(a.copy()).cuda() for a in (k, v, ks, vs)]
    P.kv_copy_blocks(dev[0], dev[1], i32_to_dev(pairs), k_scale=dev[2], v_scale=dev[3])
    t.cuda.synchronize()
    for d_, a in zip(dev, (k, v, ks, vs)):
        assert np.array_equal(d_.cpu().numpy(), oracle.copy_blocks(a, pairs))


def test_copy_blocks_skips_invalid_ids(built_library):
    t = torch()
    rng = np.random.default_rng(42)
    k = rng.integers(0, 2 ** 16, size=(8, 1, BS, D), dtype=np.uint16)
    kd, vd = bf16_to_dev(k), bf16_to_dev(k)
    P.kv_copy_blocks(kd, vd, i32_to_dev(np.array([[-1, 2], [3, 8], [9, 1], [2, 100]], dtype=np.int32)))
    t.cuda.synchronize()
    assert np.array_equal(dev_to_bf16_bits(kd), k)


class Server:
    """A tiny serving loop on the CUDA path, driven by the block manager.

    The K/V of a token depends on its whole token prefix (as in a real model),
    so sequences with a common prefix hold identical K/V there; the test keeps
    every sequence's logical K/V on the host and checks the kernels' view of
    the pool against the oracle on that contiguous history.
    """

    def __init__(self, num_blocks, n_q, n_kv, seed):
        t = torch()
        self.t = t
        self.n_q, self.n_kv = n_q, n_kv
        self.bm = P.BlockManager(num_blocks)
        nan = np.full((num_blocks, n_kv, BS, D), W.BF16_NAN, dtype=np.uint16)
        self.k_cache, self.v_cache = bf16_to_dev(nan), bf16_to_dev(nan)
        self.tokens, self.logical_k, self.logical_v = {}, {}, {}
        self.rng = np.random.default_rng(seed)
        self.copies = 0

    def _kv(self, toks, p):
        r = np.random.default_rng(abs(hash(tuple(toks[:p + 1]))) % (2 ** 63))
        kv = r.standard_normal((2, self.n_kv, D)).astype(np.float32)
        return W.bf16_bits_from_f32(kv[0]), W.bf16_bits_from_f32(kv[1])

    def write(self, sid, new_tokens):
        slots, pair = self.bm.append(sid, len(new_tokens))
        if pair is not None:  # the branch point: copy the shared block before writing into it
            P.kv_copy_blocks(self.k_cache, self.v_cache, i32_to_dev(np.array([pair], dtype=np.int32)))
            self.copies += 1
        toks = self.tokens[sid]
        ks, vs = [], []
        for tok in new_tokens:
            toks.append(tok)
            k, v = self._kv(toks, len(toks) - 1)
            ks.append(k); vs.append(v)
            self.logical_k[sid].append(k); self.logical_v[sid].append(v)
        P.kv_reshape_and_cache(bf16_to_dev(np.stack(ks)), bf16_to_dev(np.stack(vs)), self.k_cache, self.v_cache,
                               i32_to_dev(slots))

    def new(self, sid, prompt=None, parent=None):
        if parent is not None:
            self.bm.fork(parent, sid)
            self.tokens[sid] = list(self.tokens[parent])
            self.logical_k[sid] = list(self.logical_k[parent]); self.logical_v[sid] = list(self.logical_v[parent])
            return
        n = self.bm.add_cached(sid, prompt)
        self.tokens[sid] = list(prompt[:n])
        self.logical_k[sid] = [self._kv(prompt, p)[0] for p in range(n)]
        self.logical_v[sid] = [self._kv(prompt, p)[1] for p in range(n)]
        self.write(sid, prompt[n:])
        self.bm.publish(sid, self.tokens[sid])
        return n

    def decode_and_check(self, scale):
        t = self.t
        ids = sorted(self.tokens)
        width = max(-(-len(self.tokens[i]) // BS) for i in ids)
        tables, lens = self.bm.block_tables(ids, width, pad_block=0)
        q = W.bf16_bits_from_f32(self.rng.standard_normal((len(ids), self.n_q, D)).astype(np.float32))
        out = t.empty((len(ids), self.n_q, D), dtype=t.float32, device="cuda")
        P.paged_attention_decode(out, bf16_to_dev(q), self.k_cache, self.v_cache, i32_to_dev(tables),
                                 i32_to_dev(lens), scale)
        # oracle on each sequence's own contiguous history (never looks at the pool or the tables)
        lk = [np.stack(self.logical_k[i]) for i in ids]
        lv = [np.stack(self.logical_v[i]) for i in ids]
        nblk = [-(-k.shape[0] // BS) for k in lk]
        kc = np.zeros((sum(nblk), self.n_kv, BS, D), dtype=np.uint16)
        vc = np.zeros_like(kc)
        tab = np.zeros((len(ids), max(nblk)), dtype=np.int32)
        base = 0
        for b, (K, V) in enumerate(zip(lk, lv)):
            for j in range(K.shape[0]):
                kc[base + j // BS, :, j % BS] = K[j]
                vc[base + j // BS, :, j % BS] = V[j]
            tab[b, :nblk[b]] = np.arange(base, base + nblk[b])
            base += nblk[b]
        ref = oracle.paged_attention(q, np.arange(len(ids) + 1, dtype=np.int32), kc, vc, tab, lens, scale,
                                     n_q=self.n_q)
        t.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref, what="served decode")


@pytest.mark.parametrize("seed", [0, 1])
def test_served_sequences_with_forks_and_prefix_reuse(built_library, seed):
    n_q, n_kv = 16, 4
    srv = Server(num_blocks=96, n_q=n_q, n_kv=n_kv, seed=seed)
    rng = np.random.default_rng(100 + seed)
    scale = 1.0 / np.sqrt(D)
    system = [int(x) for x in rng.integers(0, 1000, 37)]  # a shared system prompt
    sid = 0
    for _ in range(3):
        srv.new(sid, system + [int(x) for x in rng.integers(0, 1000, rng.integers(1, 30))])
        sid += 1
    cached = srv.new(sid, system + [5, 6, 7]); sid += 1
    assert cached == 32  # the published system-prompt blocks were taken over
    for step in range(12):
        live = sorted(srv.tokens)
        if step % 4 == 1:  # parallel candidates branch off a live sequence
            srv.new(sid, parent=int(rng.choice(live))); sid += 1
        if step % 5 == 3 and len(live) > 3:
            victim = int(rng.choice(live))
            srv.bm.free(victim)
            for d_ in (srv.tokens, srv.logical_k, srv.logical_v):
                del d_[victim]
        for s_ in sorted(srv.tokens):  # one decode token per live sequence
            srv.write(s_, [int(rng.integers(0, 1000))])
        srv.decode_and_check(scale)
    assert srv.copies > 0
