"""Pins of the oracle block manager against what the pages state.

"Inference optimization" lesson, section "PagedAttention": pages of 16
tokens anywhere in memory, one page table per request, a shared system
prompt stored once and referenced by every request, a private page only when
a request diverges.  "Continuous Batching e PagedAttention no vLLM",
section 3: the last block of a sequence may be partly filled.  Each pin is a
property a wrong manager would break: the logical contents every request
reads back through its table, the reference counts, the page counts of the
shared-prompt example, and the waste bound of partly filled last pages.
"""
import numpy as np
import pytest

from oracle.block_manager import BlockManager, BlockManagerError

B = 16


class Mirror:
    """Token values written through a manager's slots into a simulated pool."""

    def __init__(self, bm: BlockManager):
        self.bm = bm
        self.pool = {}                     # slot -> value
        self.logical = {}                  # seq -> list of values
        self.next = 0

    def _value(self):
        self.next += 1
        return self.next

    def add(self, seq, n):
        vals = [self._value() for _ in range(n)]
        for slot, v in zip(self.bm.add(seq, n), vals):
            self.pool[slot] = v
        self.logical[seq] = vals

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.logical[child] = list(self.logical[parent])

    def append(self, seq):
        slot, copies = self.bm.append(seq)
        for src, dst in copies:                     # copy the whole page first
            for o in range(B):
                if src * B + o in self.pool:
                    self.pool[dst * B + o] = self.pool[src * B + o]
        v = self._value()
        self.pool[slot] = v
        self.logical[seq].append(v)

    def free(self, seq):
        self.bm.free_seq(seq)
        del self.logical[seq]

    def check(self):
        refs = np.zeros(self.bm.num_blocks, dtype=int)
        for seq, vals in self.logical.items():
            table = self.bm.table(seq)
            assert len(table) == -(-len(vals) // B)
            assert len(set(table)) == len(table)
            for b in table:
                refs[b] += 1
            got = [self.pool[table[t // B] * B + t % B] for t in range(len(vals))]
            assert got == vals, f"sequence {seq} reads back other tokens"
        assert list(refs) == self.bm.ref
        assert sorted(self.bm.free) == [b for b in range(self.bm.num_blocks) if refs[b] == 0]


def _random_ops(seed, steps=400, num_blocks=64):
    rng = np.random.default_rng(seed)
    m = Mirror(BlockManager(num_blocks))
    next_id = 0
    for _ in range(steps):
        live = list(m.logical)
        op = rng.integers(0, 10)
        try:
            if op < 2 or not live:
                m.add(next_id, int(rng.integers(0, 40)))
                next_id += 1
            elif op < 4:
                m.fork(int(rng.choice(live)), next_id)
                next_id += 1
            elif op < 9:
                m.append(int(rng.choice(live)))
            else:
                m.free(int(rng.choice(live)))
        except BlockManagerError:
            pass                                   # pool exhausted: state unchanged
        m.check()
    return m


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_every_request_reads_back_its_own_tokens(seed):
    _random_ops(seed)


def test_shared_prompt_is_stored_once():
    # 50 requests share a 512-token system prompt (32 full pages), then each
    # writes 20 tokens of its own: 32 shared pages + 2 private pages each.
    bm = BlockManager(1000)
    bm.add(0, 512)
    for r in range(1, 51):
        bm.fork(0, r)
    bm.free_seq(0)
    for _ in range(20):
        for r in range(1, 51):
            bm.append(r)
    assert bm.num_blocks - bm.num_free() == 32 + 50 * 2
    assert all(bm.ref[b] == 50 for b in bm.table(1)[:32])


def test_divergence_inside_a_page_copies_only_that_page():
    # A 500-token prompt ends in a page holding 4 tokens; each of 3 forks
    # copies that page on its first write, the last one writes in place.
    bm = BlockManager(100)
    bm.add(0, 500)
    shared_last = bm.table(0)[-1]
    for r in (1, 2, 3):
        bm.fork(0, r)
    bm.free_seq(0)
    copies = []
    for r in (1, 2, 3):
        slot, c = bm.append(r)
        copies += c
    assert copies == [(shared_last, 32), (shared_last, 33)]
    assert bm.table(3)[-1] == shared_last and bm.ref[shared_last] == 1
    assert bm.num_blocks - bm.num_free() == 32 + 2


def test_last_page_waste_is_below_one_page_per_sequence():
    bm = BlockManager(500)
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 300, size=30)
    for s, n in enumerate(lens):
        bm.add(s, int(n))
    used = bm.num_blocks - bm.num_free()
    waste = used * B - int(lens.sum())
    assert 0 <= waste <= (B - 1) * len(lens)


def test_freeing_everything_returns_every_page():
    m = _random_ops(9, steps=300)
    for seq in list(m.logical):
        m.free(seq)
    assert m.bm.num_free() == m.bm.num_blocks
    assert all(r == 0 for r in m.bm.ref)


def test_exhaustion_leaves_state_unchanged():
    bm = BlockManager(4)
    bm.add(0, 48)
    before = (bm.table(0), bm.num_free(), list(bm.ref))
    with pytest.raises(BlockManagerError):
        bm.add(1, 40)                               # needs 3 pages, 1 free
    assert (bm.table(0), bm.num_free(), list(bm.ref)) == before
    bm.append(0)                                    # takes the last page
    with pytest.raises(BlockManagerError):
        bm.fork(0, 0)
