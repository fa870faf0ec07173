"""The C++ block manager against the reference block manager, operation by operation.

Integer work: block ids, reference counts, queue order, cached flags, copy-on-write
pairs, swap pairs, tables and slots must be identical.  Runs on the CPU (the manager
never touches a GPU); the library only has to be built.
"""
import hashlib

import numpy as np
import pytest

from oracle.block_manager import BlockManager as RefManager
from oracle.block_manager import NoBlocks as RefNoBlocks


@pytest.fixture(scope="module")
def bmmod():
    import paged_kv_cache_53_gb300.build as build
    build.build()
    from paged_kv_cache_53_gb300 import block_manager
    return block_manager


@pytest.mark.parametrize("n", [0, 1, 3, 55, 56, 57, 63, 64, 65, 119, 120, 128, 1000, 4133])
def test_sha256_matches_hashlib(bmmod, n):
    data = np.random.default_rng(n).integers(0, 256, n).astype(np.uint8).tobytes()
    assert bmmod.sha256(data) == hashlib.sha256(data).digest()


def test_sha256_of_the_standard_examples(bmmod):
    # the one-block and two-block messages of the Secure Hash Standard's examples
    assert bmmod.sha256(b"abc").hex() == hashlib.sha256(b"abc").hexdigest()
    msg = b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq"
    assert bmmod.sha256(msg) == hashlib.sha256(msg).digest()


def _same_state(bm, ref, live):
    assert bm.num_free_blocks() == ref.num_free_blocks()
    assert bm.num_free_host_blocks() == ref.num_free_host_blocks()
    assert bm.free_queue() == ref.queue
    for b in range(ref.num_blocks):
        assert bm.refcount(b) == ref.refcount(b), b
        assert bm.is_cached(b) == ref.is_cached(b), b
    for s in live:
        assert bm.num_tokens(s) == ref.num_tokens(s)
        if not ref.seqs[s].swapped:
            assert bm.block_table(s) == ref.block_table(s)


def _both(fn_bm, fn_ref, nob):
    """Runs an operation on both managers; both succeed (same result) or both lack
    blocks."""
    try:
        r = fn_ref()
        ok = True
    except RefNoBlocks:
        ok = False
    if ok:
        return r, fn_bm()
    with pytest.raises(nob):
        fn_bm()
    return None, None


@pytest.mark.parametrize("caching", [False, True])
@pytest.mark.parametrize("bs,nb,seed", [(4, 64, 1), (16, 300, 2), (8, 120, 3), (1, 40, 4)])
def test_random_traces_match_the_reference(bmmod, caching, bs, nb, seed):
    rng = np.random.default_rng(seed)
    bm = bmmod.BlockManager(nb, bs, prefix_caching=caching, num_host_blocks=nb // 2)
    ref = RefManager(nb, bs, prefix_caching=caching, num_host_blocks=nb // 2)
    prompts = [rng.integers(0, 3, int(rng.integers(1, 6 * bs))).tolist() for _ in range(6)]
    live, nxt = [], 0
    for step in range(400):
        op = int(rng.integers(0, 8))
        resident = [s for s in live if not ref.seqs[s].swapped]
        swapped = [s for s in live if ref.seqs[s].swapped]
        if op <= 1 or not live:
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(1, len(base) + 1))] + \
                rng.integers(0, 3, int(rng.integers(0, 2 * bs))).tolist()
            extra = [b"", b"", b"salt"][int(rng.integers(3))]
            r, c = _both(lambda: bm.add_sequence(nxt, toks, extra),
                         lambda: ref.add_sequence(nxt, toks, extra), bmmod.NoBlocks)
            assert r == c
            if r is not None:
                live.append(nxt)
            nxt += 1
        elif op == 2 and resident:
            s = resident[int(rng.integers(len(resident)))]
            toks = rng.integers(0, 3, int(rng.integers(1, 2 * bs + 2))).tolist()
            _both(lambda: bm.append_tokens(s, toks), lambda: ref.append_tokens(s, toks),
                  bmmod.NoBlocks)
        elif op == 7 and len(resident) > 1 and rng.random() < 0.5:
            grp = rng.choice(resident, size=min(len(resident), int(rng.integers(2, 6))),
                             replace=False).tolist()
            cnt = rng.integers(0, bs + 2, size=len(grp)).tolist()
            toks = rng.integers(0, 3, int(sum(cnt))).tolist()
            _both(lambda: bm.append_tokens_batch(grp, toks, cnt),
                  lambda: ref.append_tokens_batch(grp, toks, cnt), bmmod.NoBlocks)
        elif op == 3 and resident:
            s = resident[int(rng.integers(len(resident)))]
            bm.fork(s, nxt)
            ref.fork(s, nxt)
            live.append(nxt)
            nxt += 1
        elif op == 4 and live:
            s = live.pop(int(rng.integers(len(live))))
            bm.free_sequence(s)
            ref.free_sequence(s)
        elif op == 5 and resident:
            grp = sorted(set(rng.choice(resident, size=min(2, len(resident)),
                                        replace=False).tolist()))
            r, c = _both(lambda: bm.swap_out(grp), lambda: ref.swap_out(grp), bmmod.NoBlocks)
            if r is not None:
                assert c.tolist() == [list(p) for p in r]
        elif op == 6 and swapped:
            grp = swapped[:1 + int(rng.integers(len(swapped)))]
            r, c = _both(lambda: bm.swap_in(grp), lambda: ref.swap_in(grp), bmmod.NoBlocks)
            if r is not None:
                assert c.tolist() == [list(p) for p in r]
        elif resident:
            q = [int(rng.integers(0, ref.num_tokens(s) + 1)) for s in resident]
            assert np.array_equal(bm.slot_mapping(resident, q), ref.slot_mapping(resident, q))
            w = max(len(ref.block_table(s)) for s in resident) + 1
            t, ctx = bm.block_tables(resident, w)
            assert np.array_equal(t, ref.block_tables(resident, w))
            assert np.array_equal(ctx, ref.context_lens(resident))
        assert bm.take_copies().tolist() == [list(p) for p in ref.take_copies()]
        _same_state(bm, ref, live)


def test_the_worked_prefix_example(bmmod):
    """2,100-token prompts with a common 2,000-token system prompt: 131 full blocks, a
    hit on the first 125 ("PagedAttention and Continuous Batching Explained (2026)",
    section "Prefix caching")."""
    rng = np.random.default_rng(0)
    system = rng.integers(0, 50_000, 2000).tolist()
    bm = bmmod.BlockManager(1000, 16, prefix_caching=True)
    assert bm.add_sequence(1, system + rng.integers(0, 50_000, 100).tolist()) == 0
    assert sum(bm.is_cached(b) for b in bm.block_table(1)) == 131
    assert bm.add_sequence(2, system + rng.integers(0, 50_000, 100).tolist()) == 2000


def test_admission_of_the_measured_capacity(bmmod):
    """22,048 tokens of cache hold 34 requests of 640 tokens ("KV Cache in Serving
    Engines", section "5. When KV Space Falls Short")."""
    bm = bmmod.BlockManager(22_048 // 16, 16)
    n = 0
    while bm.can_allocate(640):
        bm.add_sequence(n, list(range(640)))
        n += 1
    assert n == 34
    with pytest.raises(bmmod.NoBlocks):
        bm.add_sequence(99, list(range(640)))


def test_batch_append_copies_for_all_but_the_last_reader(bmmod):
    """One decode step of four samples on a partly filled shared block, in one call:
    three copies, the last sample appends in place; a shortage changes nothing."""
    bm = bmmod.BlockManager(8, 16)
    ref = RefManager(8, 16)
    for m in (bm, ref):
        m.add_sequence(0, list(range(37)))
        for c in (1, 2, 3):
            m.fork(0, c)
        m.append_tokens_batch([1, 2, 3, 0], [7, 8, 9, 10])
    assert bm.take_copies().tolist() == [list(p) for p in ref.take_copies()]
    assert len(ref.copies) == 0 and bm.num_free_blocks() == ref.num_free_blocks() == 2
    before = [bm.block_table(s) for s in range(4)]
    with pytest.raises(bmmod.NoBlocks):  # 4 x 12 more tokens need 4 blocks, 2 are free
        bm.append_tokens_batch([0, 1, 2, 3], [1] * 48, [12, 12, 12, 12])
    assert [bm.block_table(s) for s in range(4)] == before
    with pytest.raises(bmmod.PaError):
        bm.append_tokens_batch([0, 0], [1, 2])


def test_errors(bmmod):
    from paged_kv_cache_53_gb300 import PaError
    bm = bmmod.BlockManager(8, 4, num_host_blocks=1)
    bm.add_sequence(0, [1, 2, 3, 4, 5])
    with pytest.raises(PaError):
        bm.add_sequence(0, [1])  # exists
    with pytest.raises(PaError):
        bm.append_tokens(7, [1])  # unknown
    with pytest.raises(PaError):
        bm.fork(0, 0)
    with pytest.raises(bmmod.NoBlocks):
        bm.swap_out([0])  # two blocks, one host block
    assert bm.block_table(0) == [0, 1]
    with pytest.raises(PaError):
        bm.swap_in([0])  # resident
    with pytest.raises(PaError):
        bm.slot_mapping([0], [6])  # more query tokens than tokens
    with pytest.raises(PaError):
        bm.block_tables([0], 1)  # too narrow
    with pytest.raises(PaError):
        bmmod.BlockManager(0, 16)
