"""The seeded generators lay out what the pages and the workload recipes describe."""
import numpy as np
import pytest

import oracle
import workloads as W


def _check_tables(step):
    for batch in step.batches():
        for b in range(batch.num_seqs):
            n = oracle.blocks_for_tokens(int(batch.context_lens[b]), step.shape.block_size)
            row = batch.block_tables[b]
            assert (row[:n] >= 0).all() and (row[:n] < step.num_blocks).all()
            assert (row[n:] == W.UNUSED_BLOCK).all()


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_named_workloads_are_well_formed(name):
    step = W.NAMED[name]()
    _check_tables(step)
    sh = step.shape
    assert sh.num_q_heads % sh.num_kv_heads == 0
    # every block id is referenced by at most one table row unless the workload shares
    if step.cow_pairs is None:
        ids = np.concatenate([b.block_tables[b.block_tables >= 0] for b in step.batches()])
        assert len(np.unique(ids)) == len(ids)


def test_tiny_decode():
    s = W.tiny_decode()
    assert s.decode.context_lens.tolist() == [1, 17, 33, 100]
    assert s.num_blocks == 64 and s.shape.dtype == "f32" and s.scale == 1.0 / 8


def test_llama8b_gqa_lengths():
    s = W.llama8b_gqa_decode()
    ctx = s.decode.context_lens
    assert ctx.min() >= 16 and ctx.max() <= 8192 and len(ctx) == 256
    assert s.shape == W.Shape(32, 8, 128, 16, "bf16")


def test_prefix_sharing_cow_layout():
    s = W.prefix_sharing_cow()
    t = s.decode.block_tables
    before = s.decode_tables_before_cow
    # 128 sequences point at one 128-block prefix: refcount 128
    prefix = t[0, :128]
    for b in range(128):
        assert np.array_equal(t[b, :128], prefix)
    assert s.decode.context_lens[:128].min() >= 2049
    assert s.decode.context_lens[:128].max() <= 2048 + 512
    # 8 groups of 4 samples: shared prompt whose last block is partly filled
    pairs = s.cow_pairs
    assert pairs.shape == (24, 2)
    assert len(set(pairs[:, 1].tolist())) == 24
    assert not set(pairs[:, 1].tolist()) & set(pairs[:, 0].tolist())
    for g in range(8):
        rows = range(128 + 4 * g, 128 + 4 * g + 4)
        ctx = int(s.decode.context_lens[rows[0]])
        prompt = ctx - 1
        assert prompt % 16 != 0
        nb = oracle.blocks_for_tokens(prompt, 16)
        assert oracle.blocks_for_tokens(ctx, 16) == nb  # the append lands in the last block
        last = before[rows[0], nb - 1]
        for r in rows:
            assert np.array_equal(before[r, :nb], before[rows[0], :nb])
        # three samples are remapped to copies of the shared last block, one keeps it
        remapped = [r for r in rows if t[r, nb - 1] != last]
        assert len(remapped) == 3
        for r in remapped:
            assert [last, t[r, nb - 1]] in pairs.tolist()


def test_mixed_prefill_decode_layout():
    s = W.mixed_prefill_decode()
    assert s.shape.block_size == 32
    p, d = s.prefill, s.decode
    assert p.query_lens.tolist() == [512] * 8
    ctx0 = p.context_lens - p.query_lens
    assert ctx0[0] == 0 and ctx0[-1] == 16384 and ctx0.min() >= 0 and ctx0.max() <= 16384
    assert d.num_seqs == 248 and (d.context_lens[-8:] == 131072).all()
    assert d.context_lens[:240].min() >= 1024 and d.context_lens[:240].max() <= 32768
    ids = np.concatenate([p.block_tables[p.block_tables >= 0], d.block_tables[d.block_tables >= 0]])
    assert len(np.unique(ids)) == len(ids)


def test_values_are_seeded():
    s = W.decode_step("t", W.Shape(4, 2, 64, 16, "bf16"), [3, 20], seed=9)
    a = W.make_values(s)
    b = W.make_values(s)
    for k in a:
        assert np.array_equal(W.to_numpy(a[k]), W.to_numpy(b[k]))
    assert a["k_cache"].shape == (s.num_blocks, 2, 16, 64)
    assert a["q_decode"].shape == (2, 4, 64)
