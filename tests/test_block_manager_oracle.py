"""Pins of the reference block manager: the pages' worked numbers, closed forms and
invariants that a slip in it (a wrong boundary, a lost reference, a key chained on the
wrong parent) would break."""
import collections

import numpy as np
import pytest

from oracle.block_manager import BlockManager, NoBlocks, ROOT_KEY, block_key, key_chain


def check_invariants(bm: BlockManager):
    """Every device block is either in the free queue or read by a resident sequence,
    and its reference count is the number of table entries that name it."""
    refs = collections.Counter()
    host_refs = collections.Counter()
    for s in bm.seqs.values():
        (host_refs if s.swapped else refs).update(s.blocks)
        assert len(s.blocks) == -(-len(s.tokens) // bm.bs)
        assert len(s.keys) == len(s.tokens) // bm.bs
    assert len(set(bm.queue)) == len(bm.queue)
    for b in range(bm.num_blocks):
        assert bm.ref[b] == refs.get(b, 0)
        assert (b in bm.queue) == (bm.ref[b] == 0)
    for h in range(len(bm.host_ref)):
        assert bm.host_ref[h] == host_refs.get(h, 0)
        assert (h in bm.host_free) == (bm.host_ref[h] == 0)
    for k, b in bm.cached.items():
        assert bm.key[b] == k
    assert sum(k is not None for k in bm.key) == len(bm.cached)


def test_prefix_hit_of_the_worked_example():
    """A 2,100-token prompt whose first 2,000 tokens are a shared system prompt holds
    131 full 16-token blocks (2,096 tokens); the first 125 (2,000 tokens) are shared,
    leaving about 100 tokens of prefill on a hit ("PagedAttention and Continuous
    Batching Explained (2026)", section "Prefix caching")."""
    rng = np.random.default_rng(0)
    system = rng.integers(0, 50_000, 2000).tolist()
    a = system + rng.integers(0, 50_000, 100).tolist()
    b = system + rng.integers(0, 50_000, 100).tolist()
    bm = BlockManager(1000, 16, prefix_caching=True)
    assert bm.add_sequence(1, a) == 0
    assert len(bm.seqs[1].keys) == 131 and len(bm.cached) == 131
    assert len(bm.block_table(1)) == 132
    hit = bm.add_sequence(2, b)
    assert hit == 2000 and len(b) - hit == 100
    assert bm.block_table(2)[:125] == bm.block_table(1)[:125]
    assert bm.block_table(2)[125] != bm.block_table(1)[125]
    assert all(bm.refcount(x) == 2 for x in bm.block_table(1)[:125])
    check_invariants(bm)


def test_admission_of_the_measured_capacity():
    """22,048 tokens of cache hold about 34 requests of 512 + 128 = 640 tokens ("KV Cache
    in Serving Engines", section "5. When KV Space Falls Short")."""
    bm = BlockManager(22_048 // 16, 16)
    n = 0
    while bm.can_allocate(640):
        bm.add_sequence(n, list(range(640)))
        n += 1
    assert n == 34
    with pytest.raises(NoBlocks):
        bm.add_sequence(99, list(range(640)))
    check_invariants(bm)


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
def test_waste_is_below_one_block(bs):
    """Blocks are allocated one at a time as the sequence grows, so the only waste is
    the unused tail of the last block ("KV Cache in Serving Engines", "Blocks and Block
    Tables")."""
    rng = np.random.default_rng(bs)
    bm = BlockManager(4000, bs)
    for s in range(20):
        bm.add_sequence(s, [1] * int(rng.integers(1, 300)))
        for _ in range(int(rng.integers(0, 40))):
            bm.append_tokens(s, [2])
        n = bm.num_tokens(s)
        assert 0 <= len(bm.block_table(s)) * bs - n < bs
    check_invariants(bm)


def test_blocks_are_allocated_only_at_block_boundaries():
    bm = BlockManager(10, 4)
    bm.add_sequence(0, [1, 2, 3])
    assert bm.block_table(0) == [0]
    bm.append_tokens(0, [4])  # fills block 0
    assert bm.block_table(0) == [0] and bm.num_free_blocks() == 9
    bm.append_tokens(0, [5])  # position 4 starts block 1
    assert bm.block_table(0) == [0, 1]
    assert bm.slot_mapping([0], [2]).tolist() == [3, 4]


def test_copy_on_write_of_four_samples():
    """Four samples share a prompt whose last block is partly filled; each appends one
    token.  The block is copied only when someone needs to append to it ("KV Cache in
    Serving Engines", section "Sharing Blocks"): three copies, and the fourth sample,
    then its only reader, appends in place."""
    bm = BlockManager(64, 16)
    bm.add_sequence(0, list(range(37)))  # blocks 0, 1, 2 (2 holds 5 tokens)
    for c in (1, 2, 3):
        bm.fork(0, c)
    shared = bm.block_table(0)[-1]
    assert bm.refcount(shared) == 4
    for s in (1, 2, 3, 0):
        bm.append_tokens(s, [100 + s])
    copies = bm.take_copies()
    assert len(copies) == 3 and all(src == shared for src, _ in copies)
    assert bm.block_table(0)[-1] == shared and bm.refcount(shared) == 1
    dsts = [bm.block_table(s)[-1] for s in (1, 2, 3)]
    assert sorted(dsts) == sorted(d for _, d in copies)
    for s in range(4):  # the first two blocks stay shared
        assert bm.block_table(s)[:2] == bm.block_table(0)[:2]
    assert bm.take_copies() == []
    check_invariants(bm)


def test_fork_at_a_block_boundary_copies_nothing():
    bm = BlockManager(16, 16)
    bm.add_sequence(0, list(range(32)))
    bm.fork(0, 1)
    bm.append_tokens(1, [7])
    assert bm.take_copies() == []
    assert bm.block_table(1)[:2] == bm.block_table(0)
    check_invariants(bm)


def test_shared_prefix_of_128_sequences():
    """128 sequences on one 2,048-token prefix: the prefix is stored once and every
    prefix block is read 128 times ("Continuous batching, paged attention, prefix
    caching", section "Prefix caching")."""
    rng = np.random.default_rng(3)
    prefix = rng.integers(0, 1000, 2048).tolist()
    bm = BlockManager(6000, 16, prefix_caching=True)
    for s in range(128):
        suffix = rng.integers(0, 1000, int(rng.integers(1, 513))).tolist()
        hit = bm.add_sequence(s, prefix + suffix)
        assert hit >= (0 if s == 0 else 2048)
    pblocks = bm.block_table(0)[:128]
    for s in range(128):
        assert bm.block_table(s)[:128] == pblocks
    assert all(bm.refcount(b) == 128 for b in pblocks)
    check_invariants(bm)


def test_key_chain_depends_on_every_earlier_block_and_the_extra_keys():
    rng = np.random.default_rng(4)
    t = rng.integers(0, 1000, 64).tolist()
    u = list(t)
    u[3] += 1  # differs in block 0 only
    kt, ku = key_chain(t, 16), key_chain(u, 16)
    assert len(kt) == 4 and all(a != b for a, b in zip(kt, ku))  # every later key changes
    assert key_chain(t, 16, b"tenant-a") != kt
    assert key_chain(t[:63], 16) == kt[:3]  # only full blocks are keyed
    # the same 16 tokens after a different parent give a different key
    assert block_key(ROOT_KEY, t[16:32]) != kt[1]
    assert block_key(kt[0], t[16:32]) == kt[1]


def test_extra_keys_isolate_tenants():
    bm = BlockManager(100, 16, prefix_caching=True)
    toks = list(range(160))
    bm.add_sequence(0, toks, extra=b"salt-a")
    assert bm.add_sequence(1, toks, extra=b"salt-b") == 0
    assert bm.add_sequence(2, toks, extra=b"salt-a") == 160
    check_invariants(bm)


def test_first_miss_ends_the_shared_prefix():
    bm = BlockManager(100, 16, prefix_caching=True)
    a = list(range(96))
    bm.add_sequence(0, a)
    b = list(a)
    b[40] = -5  # block 2 differs; blocks 3, 4, 5 then differ through their parent
    assert bm.add_sequence(1, b) == 32
    check_invariants(bm)


def test_freed_blocks_keep_their_contents_and_tails_are_evicted_first():
    """Blocks of a finished sequence stay reusable until their space is needed; the
    oldest go first, and a sequence's blocks enter the queue tail first ("KV Cache in
    Serving Engines", section "4. Prefix Caching")."""
    bm = BlockManager(8, 4, prefix_caching=True)
    toks = list(range(16))  # 4 full blocks
    bm.add_sequence(0, toks)
    table = bm.block_table(0)
    bm.free_sequence(0)
    assert bm.num_free_blocks() == 8 and len(bm.cached) == 4
    assert bm.queue[-4:] == table[::-1]
    # a new sequence needing 6 blocks takes the 4 never-used ones, then evicts the two
    # tail blocks of the freed sequence
    bm.add_sequence(1, [1000 + i for i in range(24)])
    assert len(bm.cached) == 2 + 6  # head blocks still cached, plus the new full blocks
    assert bm.is_cached(table[0]) and bm.is_cached(table[1])
    assert not bm.is_cached(table[2]) or bm.key[table[2]] != key_chain(toks, 4)[2]
    bm.free_sequence(1)
    assert bm.add_sequence(2, toks) == 8  # the head blocks still hit
    check_invariants(bm)


def test_a_hit_on_an_idle_block_takes_it_out_of_the_queue():
    bm = BlockManager(6, 4, prefix_caching=True)
    bm.add_sequence(0, list(range(8)))
    bm.free_sequence(0)
    assert bm.num_free_blocks() == 6
    assert bm.add_sequence(1, list(range(8)) + [9]) == 8
    assert bm.num_free_blocks() == 3
    check_invariants(bm)


def test_failed_operations_change_nothing():
    bm = BlockManager(4, 4)
    bm.add_sequence(0, list(range(10)))
    before = (list(bm.queue), list(bm.ref), bm.block_table(0))
    with pytest.raises(NoBlocks):
        bm.add_sequence(1, list(range(9)))
    with pytest.raises(NoBlocks):
        bm.append_tokens(0, list(range(7)))
    assert (list(bm.queue), list(bm.ref), bm.block_table(0)) == before
    assert 1 not in bm.seqs
    check_invariants(bm)


def test_swap_round_trip():
    """Pre-emption by swapping to host memory ("Continuous batching and paged
    attention", section "Why they depend on each other"): each distinct block goes out
    once, shared blocks keep their sharing on the host, and coming back restores the
    tables' shape and token counts."""
    bm = BlockManager(32, 4, num_host_blocks=16)
    bm.add_sequence(0, list(range(10)))
    bm.fork(0, 1)
    bm.append_tokens(1, [77])
    bm.take_copies()
    bm.add_sequence(2, list(range(5)))
    shape = {s: (bm.num_tokens(s), len(bm.block_table(s))) for s in (0, 1)}
    shared_before = bm.block_table(0)[:2] == bm.block_table(1)[:2]
    out = bm.swap_out([0, 1])
    assert len(out) == len(set(bm.block_table(0)) | set(bm.block_table(1)))
    assert len({d for d, _ in out}) == len(out) and len({h for _, h in out}) == len(out)
    assert bm.seqs[0].swapped and bm.num_free_host_blocks() == 16 - len(out)
    check_invariants(bm)
    with pytest.raises(RuntimeError):
        bm.append_tokens(0, [1])
    back = bm.swap_in([0, 1])
    assert sorted(h for h, _ in back) == sorted(h for _, h in out)
    assert {s: (bm.num_tokens(s), len(bm.block_table(s))) for s in (0, 1)} == shape
    assert shared_before and bm.block_table(0)[:2] == bm.block_table(1)[:2]
    assert bm.num_free_host_blocks() == 16
    check_invariants(bm)


def test_random_traces_keep_the_invariants():
    rng = np.random.default_rng(11)
    for caching in (False, True):
        bm = BlockManager(200, 8, prefix_caching=caching, num_host_blocks=64)
        live, nxt = [], 0
        for _ in range(600):
            op = rng.integers(0, 6)
            try:
                if op == 0 or not live:
                    n = int(rng.integers(1, 60))
                    bm.add_sequence(nxt, rng.integers(0, 4, n).tolist())
                    live.append(nxt)
                    nxt += 1
                elif op == 1:
                    s = live[rng.integers(len(live))]
                    if not bm.seqs[s].swapped:
                        bm.append_tokens(s, rng.integers(0, 4, int(rng.integers(1, 10))).tolist())
                elif op == 2:
                    s = live[rng.integers(len(live))]
                    if not bm.seqs[s].swapped:
                        bm.fork(s, nxt)
                        live.append(nxt)
                        nxt += 1
                elif op == 3:
                    s = live.pop(rng.integers(len(live)))
                    bm.free_sequence(s)
                elif op == 4:
                    s = live[rng.integers(len(live))]
                    group = [x for x in live if not bm.seqs[x].swapped][:1]
                    if group and not bm.seqs[s].swapped:
                        bm.swap_out([s])
                else:
                    sw = [x for x in live if bm.seqs[x].swapped]
                    if sw:
                        bm.swap_in(sw[:1])
            except NoBlocks:
                pass
            bm.take_copies()
            check_invariants(bm)
