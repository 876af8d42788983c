"""Host block manager (pkv_bm_* in include/pagedkv.h) against a shadow model (CPU only).

What is checked follows the pages: blocks of 16 tokens handed out on demand
("注意力演进与推理流程", 变革 1), prefixes and parallel candidates sharing physical
blocks until they branch, where a new block is allocated (xinc.fun archive 233,
section 6), and prefix caching that reuses the KV of a repeated prompt prefix
(变革 3).  Block ids themselves are not unique (any free block is a valid
choice), so the tests check what is: every sequence reads back exactly its own
token history from the simulated pool, reference counts equal the number of
tables holding a block, appends never write a shared block, and a failed call
changes nothing.
"""
import numpy as np
import pytest

from paged_kv_cache_95_gb300 import pagedkv as P

BS = 16


def _content(tokens, p):
    """What the pool slot of position p holds: a function of the token prefix (KV depends on it)."""
    return hash(tuple(tokens[:p + 1]))


class Shadow:
    """Plain model: per-sequence token ids, plus the simulated pool (slot -> content)."""

    def __init__(self, bm: P.BlockManager, num_blocks: int):
        self.bm, self.num_blocks = bm, num_blocks
        self.tokens = {}  # seq -> list of token ids
        self.pool = {}    # slot -> content

    def apply_copy(self, pair):
        src, dst = pair
        for o in range(BS):
            if src * BS + o in self.pool:
                self.pool[dst * BS + o] = self.pool[src * BS + o]
            else:
                self.pool.pop(dst * BS + o, None)

    def append(self, sid, new_tokens):
        slots, pair = self.bm.append(sid, len(new_tokens))
        if pair is not None:
            self.apply_copy(pair)
        toks = self.tokens[sid]
        for t, slot in zip(new_tokens, slots):
            toks.append(t)
            self.pool[int(slot)] = _content(toks, len(toks) - 1)
        # the written blocks are private to this sequence
        for slot in slots:
            assert self.bm.ref_count(int(slot) // BS) == 1
        return slots, pair

    def tables(self):
        ids = sorted(self.tokens)
        if not ids:
            return ids, None, None
        width = max(1, max(-(-len(self.tokens[i]) // BS) for i in ids))
        tab, lens = self.bm.block_tables(ids, width, pad_block=-1)
        return ids, tab, lens

    def check(self):
        ids, tab, lens = self.tables()
        refs = np.zeros(self.num_blocks, dtype=np.int64)
        for r, sid in enumerate(ids):
            toks = self.tokens[sid]
            assert lens[r] == len(toks) == self.bm.length(sid)
            nblk = -(-len(toks) // BS)
            assert np.all(tab[r, nblk:] == -1)
            for b in tab[r, :nblk]:
                refs[b] += 1
            for p in range(len(toks)):
                slot = int(tab[r, p // BS]) * BS + p % BS
                assert self.pool.get(slot) == _content(toks, p), (sid, p)
        for b in range(self.num_blocks):
            assert self.bm.ref_count(b) == refs[b], b
        assert self.bm.num_free == self.num_blocks - int(np.count_nonzero(refs))

    def snapshot(self):
        ids, tab, lens = self.tables()
        return (ids, None if tab is None else tab.tolist(), None if lens is None else lens.tolist(),
                self.bm.num_free, [self.bm.ref_count(b) for b in range(self.num_blocks)])


@pytest.fixture
def lib():
    return P.load_library()


def test_cow_at_branch(lib):
    bm = P.BlockManager(8)
    sh = Shadow(bm, 8)
    bm.add(1); sh.tokens[1] = []
    sh.append(1, list(range(20)))               # blocks 0 (full), 1 (4 tokens)
    bm.fork(1, 2); sh.tokens[2] = list(sh.tokens[1])
    assert bm.ref_count(0) == 2 and bm.ref_count(1) == 2
    slots, pair = sh.append(2, [100, 101])     # child writes into the shared partial block
    assert pair is not None and pair[0] == 1 and pair[1] not in (0, 1)
    assert list(slots) == [pair[1] * BS + 4, pair[1] * BS + 5]
    assert bm.ref_count(1) == 1 and bm.ref_count(0) == 2
    slots, pair = sh.append(1, [7])            # parent's block 1 is private again: no copy
    assert pair is None and slots[0] == 1 * BS + 4
    sh.check()


def test_full_shared_block_needs_no_copy(lib):
    bm = P.BlockManager(4)
    sh = Shadow(bm, 4)
    bm.add(1); sh.tokens[1] = []
    sh.append(1, list(range(16)))
    bm.fork(1, 2); sh.tokens[2] = list(sh.tokens[1])
    slots, pair = sh.append(2, [5])            # the next token opens a new block
    assert pair is None and slots[0] // BS not in (0,)
    sh.check()


def test_out_of_blocks_changes_nothing(lib):
    bm = P.BlockManager(3)
    sh = Shadow(bm, 3)
    bm.add(1); sh.tokens[1] = []
    sh.append(1, list(range(40)))              # 3 blocks
    before = sh.snapshot()
    with pytest.raises(P.PagedKVError) as e:
        bm.append(1, 9)
    assert e.value.code == P.PKV_ERR_OUT_OF_BLOCKS
    bm.fork(1, 2); sh.tokens[2] = list(sh.tokens[1])
    with pytest.raises(P.PagedKVError):
        bm.append(2, 1)                         # would need a copy of the shared last block
    assert sh.snapshot()[0] == [1, 2]
    sh.check()
    bm.free(2); del sh.tokens[2]
    assert sh.snapshot()[1:] == before[1:]


def test_argument_errors(lib):
    bm = P.BlockManager(4)
    bm.add(1)
    for call in (lambda: bm.add(1), lambda: bm.fork(9, 10), lambda: bm.fork(1, 1), lambda: bm.free(9),
                 lambda: bm.append(9, 1), lambda: bm.length(9), lambda: bm.ref_count(4),
                 lambda: bm.block_tables([9], 4), lambda: bm.publish(1, [1, 2, 3])):
        with pytest.raises(P.PagedKVError) as e:
            call()
        assert e.value.code == P.PKV_ERR_INVALID_ARG
    bm.append(1, 40)
    with pytest.raises(P.PagedKVError):
        bm.block_tables([1], 2)                 # needs 3 blocks
    with pytest.raises(P.PagedKVError):
        P.BlockManager(0)


def test_prefix_cache_reuse_and_eviction(lib):
    bm = P.BlockManager(10)
    sh = Shadow(bm, 10)
    prompt = list(range(1000, 1040))            # 40 tokens: 2 full blocks + 8
    bm.add(1); sh.tokens[1] = []
    sh.append(1, prompt)
    bm.publish(1, prompt)
    # same prompt: the two full blocks are taken over, the rest is computed
    n = bm.add_cached(2, prompt); sh.tokens[2] = prompt[:n]
    assert n == 32
    sh.append(2, prompt[n:])
    sh.check()
    # a prompt of exactly 32 tokens keeps its last token to compute: one block only
    n = bm.add_cached(3, prompt[:32]); sh.tokens[3] = prompt[:n]
    assert n == 16
    sh.append(3, prompt[n:32])
    # a prompt differing inside block 1 shares only block 0
    other = prompt[:20] + [7] + prompt[21:]
    n = bm.add_cached(4, other); sh.tokens[4] = other[:n]
    assert n == 16
    sh.append(4, other[n:])
    sh.check()
    # freed published blocks stay findable ...
    for sid in (1, 2, 3, 4):
        bm.free(sid); del sh.tokens[sid]
    n = bm.add_cached(5, prompt); sh.tokens[5] = prompt[:n]
    assert n == 32
    sh.append(5, prompt[n:])
    sh.check()
    bm.free(5); del sh.tokens[5]
    # ... until the allocator needs them: filling the pool evicts them
    bm.add(6); sh.tokens[6] = []
    sh.append(6, list(range(10 * BS)))
    assert bm.num_free == 0
    bm.free(6); del sh.tokens[6]
    assert bm.add_cached(7, prompt) == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_every_sequence_intact(lib, seed):
    rng = np.random.default_rng(seed)
    nb = 48
    bm = P.BlockManager(nb)
    sh = Shadow(bm, nb)
    next_id = 0
    prompts = []
    for step in range(400):
        live = sorted(sh.tokens)
        op = rng.choice(["add", "add_cached", "fork", "append", "append", "append", "free", "publish"])
        before = sh.snapshot()
        try:
            if op == "add" or not live and op != "add_cached":
                bm.add(next_id); sh.tokens[next_id] = []; next_id += 1
            elif op == "add_cached":
                base = prompts[rng.integers(len(prompts))] if prompts and rng.random() < 0.8 else []
                cut = int(rng.integers(0, len(base) + 1))
                prompt = list(base[:cut]) + [int(x) for x in rng.integers(0, 50, rng.integers(1, 40))]
                n = bm.add_cached(next_id, prompt)
                assert n % BS == 0 and n < len(prompt)
                sh.tokens[next_id] = prompt[:n]
                sid = next_id; next_id += 1
                sh.append(sid, prompt[n:])
            elif op == "fork":
                parent = int(rng.choice(live))
                bm.fork(parent, next_id); sh.tokens[next_id] = list(sh.tokens[parent]); next_id += 1
            elif op == "append":
                sid = int(rng.choice(live))
                sh.append(sid, [int(x) for x in rng.integers(0, 50, rng.integers(1, 40))])
            elif op == "free":
                sid = int(rng.choice(live))
                prompts.append(list(sh.tokens[sid]))
                bm.free(sid); del sh.tokens[sid]
            elif op == "publish":
                sid = int(rng.choice(live))
                toks = sh.tokens[sid]
                bm.publish(sid, toks[:int(rng.integers(0, len(toks) + 1))])
                prompts.append(list(toks))
        except P.PagedKVError as e:
            assert e.code == P.PKV_ERR_OUT_OF_BLOCKS, e
            if op == "add_cached":  # the sequence was created; its prompt did not fit
                sh.tokens.pop(next_id - 1, None)
                bm.free(next_id - 1)
                continue
            assert sh.snapshot()[1:] == before[1:], f"failed {op} changed the manager"
        sh.check()


def test_append_batch_matches_sequential_appends(lib):
    rng = np.random.default_rng(77)
    a, b = P.BlockManager(200), P.BlockManager(200)
    for m in (a, b):
        for i in range(6):
            m.add(i)
            m.append(i, int(10 + 9 * i))
        m.fork(2, 10)
        m.fork(2, 11)  # three sequences share block(s) of sequence 2
    for _ in range(20):
        ids = rng.permutation([0, 1, 2, 3, 4, 5, 10, 11])[: rng.integers(1, 9)]
        nt = rng.integers(0, 20, len(ids)).astype(np.int32)
        slots, pairs = a.append_batch(ids, nt)
        want_slots, want_pairs = [], []
        for i, n in zip(ids, nt):
            s_, p_ = b.append(int(i), int(n))
            want_slots.extend(s_.tolist())
            if p_ is not None:
                want_pairs.append(list(p_))
        assert slots.tolist() == want_slots
        assert pairs.tolist() == want_pairs
    tabs = lambda m: m.block_tables([0, 1, 2, 3, 4, 5, 10, 11], 64)
    assert all(np.array_equal(x, y) for x, y in zip(tabs(a), tabs(b)))


def test_append_batch_forks_of_one_block(lib):
    """Two forks appending into the same shared partial block in one call: the first
    one copies, the second then owns the block alone and writes in place."""
    bm = P.BlockManager(8)
    bm.add(1)
    bm.append(1, 20)
    bm.fork(1, 2)
    slots, pairs = bm.append_batch([1, 2])
    assert len(pairs) == 1 and pairs[0][0] == 1
    assert slots[0] // BS == pairs[0][1] and slots[1] == 1 * BS + 4
    assert bm.ref_count(1) == 1


def test_append_batch_all_or_nothing(lib):
    bm = P.BlockManager(4)
    for i in range(2):
        bm.add(i)
        bm.append(i, 16)
    before = (bm.num_free, bm.block_tables([0, 1], 4))
    with pytest.raises(P.PagedKVError) as e:
        bm.append_batch([0, 1], [16, 17])   # needs 3 blocks, 2 are free
    assert e.value.code == P.PKV_ERR_OUT_OF_BLOCKS
    for bad in ([0, 0], [0, 9]):
        with pytest.raises(P.PagedKVError) as e:
            bm.append_batch(bad)
        assert e.value.code == P.PKV_ERR_INVALID_ARG
    after = (bm.num_free, bm.block_tables([0, 1], 4))
    assert before[0] == after[0] and all(np.array_equal(x, y) for x, y in zip(before[1], after[1]))
