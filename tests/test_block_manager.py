"""Host block manager (pa_bm_*): block tables, shared blocks, prefix cache,
fork, copy-on-write and the CPU swap tier. Host logic only; runs without a
GPU.

The randomized test drives the manager the way a caller does. A simulated
store keeps a token id per (block, slot); the caller applies the manager's
copy-on-write pairs, then writes each sequence's new tokens through its block
table. After every operation these must hold:
  - every live sequence reads back exactly its tokens through its table;
  - no block is written while another sequence also holds it;
  - a prefix-cache hit's blocks already hold the prompt's tokens;
  - reference counts equal the number of tables holding each block;
  - free blocks plus held blocks add up to the pool;
  - a swapped-out sequence reads back its tokens through its host slots,
    each slot held by one sequence, and free plus held slots add up."""
import numpy as np
import pytest

from paged_gqa_decode_02_gb300 import binding as B


def test_tables_and_free_counts():
    bm = B.BlockManager(16, 4)
    assert bm.add_sequence(1, list(range(10))) == 0
    t, n = bm.block_table(1)
    assert n == 10 and list(t) == [0, 1, 2]  # ceil(10 / 4) blocks, handed out in order
    assert bm.num_free_blocks() == 13
    t, n = bm.block_table(1, max_blocks=6)
    assert list(t) == [0, 1, 2, -1, -1, -1]
    with pytest.raises(B.PagedAttnError):
        bm.block_table(1, max_blocks=2)  # does not fit
    bm.free_sequence(1)
    assert bm.num_free_blocks() == 16


def test_prefix_cache_shares_leading_full_blocks_only():
    bs = 4
    bm = B.BlockManager(32, bs)
    a = list(range(100, 114))  # 3 full blocks + 2 tokens
    assert bm.add_sequence(1, a) == 0
    b = a[:8] + [7, 7, 7, 7, 7]  # same first 2 blocks, then different
    assert bm.add_sequence(2, b) == 8
    ta, _ = bm.block_table(1)
    tb, _ = bm.block_table(2)
    assert list(tb[:2]) == list(ta[:2]) and tb[2] != ta[2]
    assert [bm.ref_count(x) for x in ta] == [2, 2, 1, 1]
    # a prompt that is a whole-block prefix but whose tail differs inside a block
    c = a[:6]
    assert bm.add_sequence(3, c) == 4
    # cached blocks outlive their holders and are found again
    bm.free_sequence(1)
    bm.free_sequence(2)
    bm.free_sequence(3)
    assert bm.num_free_blocks() == 32
    assert bm.add_sequence(4, a) == 12
    assert list(bm.block_table(4)[0][:3]) == list(ta[:3])
    # the cache is keyed by the whole chain: same block contents after a
    # different first block do not match
    d = [0, 0, 0, 0] + a[4:12]
    assert bm.add_sequence(5, d) == 0


def test_cache_entries_are_reused_least_recently_released_first():
    bs = 2
    bm = B.BlockManager(6, bs)
    bm.add_sequence(1, [1, 2, 3, 4])  # blocks 0, 1 cached
    bm.add_sequence(2, [5, 6, 7, 8])  # blocks 2, 3 cached
    bm.free_sequence(1)  # released first (tail first)
    bm.free_sequence(2)
    assert bm.num_free_blocks() == 6
    bm.add_sequence(3, [9] * 8)  # 2 free blocks, then the 2 oldest idle cached ones
    assert bm.add_sequence(4, [5, 6, 7, 8]) == 4  # sequence 2's blocks were kept
    bm.free_sequence(4)
    assert bm.add_sequence(5, [1, 2, 3, 4]) == 0  # sequence 1's were reused


def test_blocks_filled_by_appends_join_the_cache():
    bs = 4
    bm = B.BlockManager(16, bs)
    bm.add_sequence(1, [1, 2, 3])
    for t in [4, 5, 6, 7, 8, 9]:
        assert bm.append_tokens(1, [t]) == []
    assert bm.add_sequence(2, [1, 2, 3, 4, 5, 6, 7, 8, 0]) == 8


def test_fork_then_append_copies_the_shared_tail():
    bs = 4
    bm = B.BlockManager(16, bs)
    bm.add_sequence(1, [1, 2, 3, 4, 5, 6])  # blocks 0 (full), 1 (2 of 4)
    bm.fork(1, 2)
    assert [bm.ref_count(x) for x in (0, 1)] == [2, 2]
    copies = bm.append_tokens(2, [7])
    assert copies == [(1, 2)]
    assert list(bm.block_table(2)[0]) == [0, 2] and list(bm.block_table(1)[0]) == [0, 1]
    assert [bm.ref_count(x) for x in (0, 1, 2)] == [2, 1, 1]
    assert bm.append_tokens(1, [8]) == []  # now private: written in place
    # a full shared tail is never copied: the next token opens a new block
    bm.add_sequence(3, [1, 2, 3, 4])
    bm.fork(3, 4)
    assert bm.append_tokens(4, [9]) == []


def test_failed_calls_change_nothing():
    bs = 4
    bm = B.BlockManager(4, bs)
    bm.add_sequence(1, list(range(12)))  # 3 blocks
    free = bm.num_free_blocks()
    with pytest.raises(B.PagedAttnError) as e:
        bm.add_sequence(2, list(range(100, 108)))  # needs 2
    assert e.value.status == 3
    assert bm.num_free_blocks() == free
    with pytest.raises(B.PagedAttnError):
        bm.append_tokens(1, list(range(8)))  # needs 2 more
    assert bm.block_table(1)[1] == 12 and bm.num_free_blocks() == free
    with pytest.raises(B.PagedAttnError):
        bm.add_sequence(1, [1])  # id in use
    with pytest.raises(B.PagedAttnError):
        bm.fork(7, 8)  # no such parent
    with pytest.raises(B.PagedAttnError):
        bm.free_sequence(9)
    assert bm.ref_count(-1) == -1 and bm.ref_count(4) == -1


def test_swap_out_and_in_round_trip():
    bs = 4
    bm = B.BlockManager(8, bs)
    bm.set_cpu_blocks(5)
    bm.add_sequence(1, list(range(10)))  # 3 blocks
    t1, _ = bm.block_table(1)
    copies = bm.swap_out(1)
    assert copies == [(int(t1[0]), 0), (int(t1[1]), 1), (int(t1[2]), 2)]
    assert bm.swapped_slots(1) == [0, 1, 2] and bm.num_free_cpu_blocks() == 2
    assert bm.num_free_blocks() == 8
    for call in (lambda: bm.block_table(1), lambda: bm.append_tokens(1, [5]), lambda: bm.fork(1, 2),
                 lambda: bm.swap_out(1)):
        with pytest.raises(B.PagedAttnError):
            call()
    bm.add_sequence(2, [9] * 30)  # takes all 8 blocks
    with pytest.raises(B.PagedAttnError) as e:
        bm.swap_in(1)  # no GPU blocks: refused, nothing changed
    assert e.value.status == 3 and bm.swapped_slots(1) == [0, 1, 2]
    bm.free_sequence(2)
    back = bm.swap_in(1)
    assert [c for c, _ in back] == [0, 1, 2] and bm.num_free_cpu_blocks() == 5
    t1b, n = bm.block_table(1)
    assert n == 10 and list(t1b) == [g for _, g in back]
    assert bm.append_tokens(1, [10, 11]) == []  # resident again, private tail


def test_swap_out_leaves_shared_blocks_to_their_other_holders():
    bs = 4
    bm = B.BlockManager(8, bs)
    bm.set_cpu_blocks(8)
    bm.add_sequence(1, list(range(6)))  # blocks 0 (full), 1 (half)
    bm.fork(1, 2)
    copies = bm.swap_out(1)
    assert [g for g, _ in copies] == [0, 1]
    assert [bm.ref_count(b) for b in (0, 1)] == [1, 1]  # still held by the child
    assert list(bm.block_table(2)[0]) == [0, 1]
    assert bm.append_tokens(2, [6]) == []  # the child's tail is private now
    bm.free_sequence(1)  # frees the swapped sequence's slots
    assert bm.num_free_cpu_blocks() == 8


def test_swap_refusals_change_nothing():
    bs = 4
    bm = B.BlockManager(8, bs)
    bm.set_cpu_blocks(2)
    bm.add_sequence(1, list(range(12)))  # 3 blocks, 2 slots
    free = bm.num_free_blocks()
    with pytest.raises(B.PagedAttnError) as e:
        bm.swap_out(1)
    assert e.value.status == 3 and bm.num_free_cpu_blocks() == 2 and bm.num_free_blocks() == free
    assert bm.block_table(1)[1] == 12
    with pytest.raises(B.PagedAttnError):
        bm.swap_in(1)  # not swapped out
    bm.add_sequence(2, [1, 2])
    bm.swap_out(2)
    with pytest.raises(B.PagedAttnError):
        bm.set_cpu_blocks(10)  # a slot is in use
    bm.swap_in(2)
    bm.set_cpu_blocks(10)
    assert bm.num_free_cpu_blocks() == 10


def test_prefix_cache_survives_a_swap_out():
    """Swapping a sequence out releases its blocks; full cached blocks stay in
    the prefix cache (their KV is still on the GPU) until reused."""
    bs = 4
    bm = B.BlockManager(16, bs)
    bm.set_cpu_blocks(4)
    prompt = list(range(100, 109))  # 2 full blocks + 1 token
    bm.add_sequence(1, prompt)
    bm.swap_out(1)
    assert bm.add_sequence(2, prompt) == 8


class _Caller:
    """A caller of the manager with a simulated KV store (token ids) and a
    host swap tier."""

    def __init__(self, num_blocks, bs, prefix_cache, rng, cpu_blocks=0):
        self.bm = B.BlockManager(num_blocks, bs, prefix_cache)
        self.bm.set_cpu_blocks(cpu_blocks)
        self.bs, self.nb, self.rng, self.ncpu = bs, num_blocks, rng, cpu_blocks
        self.store = np.full((num_blocks, bs), -1, dtype=np.int64)
        self.cpu_store = np.full((max(cpu_blocks, 1), bs), -1, dtype=np.int64)
        self.seqs = {}  # id -> list of token ids
        self.swapped = set()
        self.next_id = 0

    def _write(self, sid, start, toks):
        table, n = self.bm.block_table(sid)
        for i, t in enumerate(toks):
            pos = start + i
            blk = int(table[pos // self.bs])
            assert self.bm.ref_count(blk) == 1, "write into a shared block"
            self.store[blk, pos % self.bs] = t

    def add(self, prompt):
        sid = self.next_id
        self.next_id += 1
        try:
            cached = self.bm.add_sequence(sid, prompt)
        except B.PagedAttnError as e:
            assert e.status == 3
            return
        assert cached % self.bs == 0 and cached <= len(prompt)
        table, n = self.bm.block_table(sid)
        assert n == len(prompt) and len(table) == -(-len(prompt) // self.bs)
        # cached blocks already hold the prompt's tokens
        for i in range(cached):
            assert self.store[table[i // self.bs], i % self.bs] == prompt[i], "stale prefix-cache hit"
        self._write(sid, cached, prompt[cached:])
        self.seqs[sid] = list(prompt)

    def swap_out(self, sid):
        try:
            copies = self.bm.swap_out(sid)
        except B.PagedAttnError as e:
            assert e.status == 3
            return
        for g, c in copies:
            self.cpu_store[c] = self.store[g]
        self.swapped.add(sid)

    def swap_in(self, sid):
        try:
            copies = self.bm.swap_in(sid)
        except B.PagedAttnError as e:
            assert e.status == 3
            return
        for c, g in copies:
            assert self.bm.ref_count(g) == 1
            self.store[g] = self.cpu_store[c]
        self.swapped.discard(sid)

    def fork(self, parent):
        sid = self.next_id
        self.next_id += 1
        self.bm.fork(parent, sid)
        self.seqs[sid] = list(self.seqs[parent])

    def append(self, sid, toks):
        try:
            copies = self.bm.append_tokens(sid, toks)
        except B.PagedAttnError as e:
            assert e.status == 3
            return
        for src, dst in copies:
            self.store[dst] = self.store[src]
        self._write(sid, len(self.seqs[sid]), toks)
        self.seqs[sid] += list(toks)

    def free(self, sid):
        self.bm.free_sequence(sid)
        del self.seqs[sid]
        self.swapped.discard(sid)

    def check(self):
        held, slots = {}, []
        for sid in self.swapped:
            toks = self.seqs[sid]
            sl = self.bm.swapped_slots(sid)
            assert len(sl) == -(-len(toks) // self.bs)
            got = [int(self.cpu_store[sl[i // self.bs], i % self.bs]) for i in range(len(toks))]
            assert got == toks, f"swapped sequence {sid} reads back wrong tokens"
            slots += sl
        assert len(set(slots)) == len(slots), "a host slot held twice"
        assert self.bm.num_free_cpu_blocks() + len(slots) == self.ncpu
        for sid, toks in self.seqs.items():
            if sid in self.swapped:
                continue
            table, n = self.bm.block_table(sid)
            assert n == len(toks)
            got = [int(self.store[table[i // self.bs], i % self.bs]) for i in range(n)]
            assert got == toks, f"sequence {sid} reads back wrong tokens"
            for b in table:
                held[int(b)] = held.get(int(b), 0) + 1
        for b, c in held.items():
            assert self.bm.ref_count(b) == c
        assert self.bm.num_free_blocks() + len(held) == self.nb


@pytest.mark.parametrize("swap", [False, True])
@pytest.mark.parametrize("prefix_cache", [True, False])
@pytest.mark.parametrize("seed", range(6))
def test_randomized_against_a_simulated_store(seed, prefix_cache, swap):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4, 16]))
    c = _Caller(int(rng.integers(8, 64)), bs, prefix_cache, rng,
                cpu_blocks=int(rng.integers(4, 48)) if swap else 0)
    prompts = [list(rng.integers(0, 3, size=int(rng.integers(1, 5 * bs)))) for _ in range(6)]
    for _ in range(400):
        op = rng.random()
        live = [s for s in c.seqs if s not in c.swapped]
        if swap and c.swapped and op < 0.1:
            c.swap_in(sorted(c.swapped)[int(rng.integers(len(c.swapped)))])
        elif swap and live and op < 0.2:
            c.swap_out(live[int(rng.integers(len(live)))])
        elif op < 0.3 or not live:
            base = prompts[int(rng.integers(len(prompts)))]
            cut = int(rng.integers(1, len(base) + 1))
            tail = list(rng.integers(0, 3, size=int(rng.integers(0, 2 * bs))))
            c.add([int(x) for x in base[:cut] + tail])
        elif op < 0.45:
            c.fork(live[int(rng.integers(len(live)))])
        elif op < 0.85:
            sid = live[int(rng.integers(len(live)))]
            c.append(sid, [int(x) for x in rng.integers(0, 3, size=int(rng.integers(1, bs + 2)))])
        else:
            everyone = list(c.seqs)
            c.free(everyone[int(rng.integers(len(everyone)))])
        c.check()
    for sid in list(c.seqs):
        c.free(sid)
    assert c.bm.num_free_blocks() == c.nb


def test_copy_on_write_without_room_for_the_copy_is_refused():
    """An append that needs a copy-on-write copy but is given no room to
    return it is refused and changes nothing."""
    import ctypes
    bs = 4
    bm = B.BlockManager(8, bs)
    bm.add_sequence(1, [1, 2, 3, 4, 5, 6])
    bm.fork(1, 2)
    before = (list(bm.block_table(2)[0]), bm.num_free_blocks(), bm.ref_count(1))
    tok = (ctypes.c_int32 * 1)(7)
    n = ctypes.c_int32(-1)
    st = B.lib().pa_bm_append_tokens(bm.handle, 2, ctypes.cast(tok, ctypes.c_void_p), 1, None, None, 0,
                                     ctypes.byref(n))
    assert st == 1
    assert (list(bm.block_table(2)[0]), bm.num_free_blocks(), bm.ref_count(1)) == before
    assert bm.block_table(2)[1] == 6
    assert bm.append_tokens(2, [7]) == [(1, 2)]  # with room, the copy is returned
