"""Host block manager (pa_bm_*), on the CPU, through the C ABI.

Checked against the contract the pages give -- one free list (take from the back, return
to the back), a new block only when a token is the first of a logical block, all of a
sequence's blocks returned when it ends, slot = block_table[pos / 16] * 16 + pos % 16 --
and against a plain Python model of the same list operations, step by step, on random
operation sequences that include forks (shared blocks) and copy on write."""
import numpy as np
import pytest

import paged_decode_attention_reshape_gb300 as pa

B = 16


class Model:
    """The same bookkeeping in plain Python."""

    def __init__(self, nb, ns, mb):
        self.free = list(range(nb - 1, -1, -1))   # back of the list = next block handed out
        self.refs = [0] * nb
        self.seqs = {}
        self.mb = mb

    def take(self):
        b = self.free.pop()
        self.refs[b] = 1
        return b

    def drop(self, b):
        self.refs[b] -= 1
        if self.refs[b] == 0:
            self.free.append(b)

    def append(self, s, n):
        blocks, L = self.seqs.get(s, ([], 0))
        if n == 0:                         # nothing appended: no block taken, no copy
            self.seqs[s] = (blocks, L)
            return "ok", [], None
        end = L + n
        need = -(-end // B)
        if need > self.mb:
            return "invalid", None, None
        cow = L % B != 0 and self.refs[blocks[-1]] > 1
        if need - len(blocks) + cow > len(self.free):
            self.seqs.setdefault(s, (blocks, L))
            return "noblocks", None, None
        blocks = list(blocks)
        pair = None
        if cow:
            old, nb = blocks[-1], self.take()
            self.drop(old)
            blocks[-1] = nb
            pair = (old, nb)
        slots = []
        for pos in range(L, end):
            if pos % B == 0:
                blocks.append(self.take())
            slots.append(blocks[pos // B] * B + pos % B)
        self.seqs[s] = (blocks, end)
        return "ok", slots, pair

    def fork(self, src, dst):
        blocks, L = self.seqs[src]
        self.seqs[dst] = (list(blocks), L)
        for b in blocks:
            self.refs[b] += 1

    def free_seq(self, s):
        blocks, _ = self.seqs.pop(s, ([], 0))
        for b in reversed(blocks):
            self.drop(b)


def check_invariants(m, model, nb, live):
    bt, sl = m.export(sorted(live))
    held = {}
    for i, s in enumerate(sorted(live)):
        L = int(sl[i])
        assert L == m.seq_len(s)
        nblk = -(-L // B)
        assert (bt[i, :nblk] >= 0).all() and (bt[i, nblk:] == -1).all()
        for b in bt[i, :nblk]:
            held[int(b)] = held.get(int(b), 0) + 1
    for b in range(nb):   # a block's count is the number of live sequences holding it
        assert m.refs(b) == held.get(b, 0) == model.refs[b]
    assert m.num_free() == nb - len(held) == len(model.free)


def test_slots_follow_the_block_table_and_blocks_come_off_the_free_list_in_order():
    m = pa.BlockManager(16, 4, 8)
    s0, _ = m.append(0, 37)                 # 3 blocks: 0, 1, 2 (the list hands out ascending ids)
    s1, _ = m.append(1, 5)                  # block 3
    s2, _ = m.append(0, 12)                 # positions 37..48: block 2 fills, block 4 starts at 48
    bt, sl = m.export([0, 1])
    assert list(bt[0, :4]) == [0, 1, 2, 4] and list(bt[1, :1]) == [3] and list(sl) == [49, 5]
    for pos, slot in zip(list(range(37)) + list(range(37, 49)), list(s0) + list(s2)):
        assert slot == bt[0, pos // B] * B + pos % B
    assert s0[20] == 1 * B + 4               # position 20 lies in logical block 1 (physical 1), offset 4
    m.free(0)
    assert m.num_free() == 16 - 1
    s3, _ = m.append(2, 1)                  # freed blocks come back LIFO: the last returned first
    assert s3[0] // B == 0


def test_out_of_blocks_changes_nothing_and_limits():
    m = pa.BlockManager(4, 2, 3)
    m.append(0, 40)                         # 3 blocks
    with pytest.raises(pa.PAError) as e:
        m.append(1, 33)                     # needs 3, 1 free
    assert e.value.status == -9
    assert m.num_free() == 1 and m.seq_len(1) == 0
    with pytest.raises(pa.PAError) as e:
        m.append(0, 9)                      # 49 tokens -> 4 blocks > max_blocks_per_seq
    assert e.value.status == -1
    assert m.seq_len(0) == 40
    with pytest.raises(pa.PAError):
        m.fork(0, 0)
    with pytest.raises(pa.PAError):
        m.append(5, 1)


def test_fork_shares_and_copy_on_write_only_for_a_shared_partial_block():
    m = pa.BlockManager(16, 4, 8)
    m.append(0, 32)                          # two full blocks 0, 1
    m.fork(0, 1)
    assert m.refs(0) == m.refs(1) == 2
    s, cp = m.append(1, 3)                   # starts a new block: no copy needed
    assert cp is None and s[0] // B == 2
    m.fork(1, 2)                             # seq 2 shares 0, 1 and the partial block 2
    s, cp = m.append(2, 1)
    assert cp == (2, 3) and s[0] == 3 * B + 3 and m.refs(2) == 1 and m.refs(3) == 1
    s, cp = m.append(1, 1)                   # block 2 is seq 1's alone again: no copy
    assert cp is None and s[0] == 2 * B + 3
    for q in (0, 1, 2):
        m.free(q)
    assert m.num_free() == 16 and all(m.refs(b) == 0 for b in range(16))


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = np.random.default_rng(seed)
    NB, NS, MB = 40, 6, 10
    m, model = pa.BlockManager(NB, NS, MB), Model(NB, NS, MB)
    live = set()
    for _ in range(300):
        op = rng.choice(["append", "append", "append", "fork", "free"])
        s = int(rng.integers(NS))
        if op == "append":
            n = int(rng.integers(0, 40))
            st, slots, pair = model.append(s, n)
            if st == "ok":
                got, cp = m.append(s, n)
                assert list(got) == slots and cp == pair
                live.add(s)
            else:
                with pytest.raises(pa.PAError) as e:
                    m.append(s, n)
                assert e.value.status == (-9 if st == "noblocks" else -1)
                if st == "noblocks":
                    live.add(s)
        elif op == "fork":
            d = int(rng.integers(NS))
            if s in live and d not in live and d != s:
                m.fork(s, d)
                model.fork(s, d)
                live.add(d)
            else:
                with pytest.raises(pa.PAError):
                    m.fork(s, d)
        else:
            m.free(s)
            model.free_seq(s)
            live.discard(s)
        check_invariants(m, model, NB, live)
