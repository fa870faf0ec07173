"""The bench's algorithmic byte and flop counts against plain loops over tiny steps (CPU)."""
import numpy as np

import workloads as W


def _bench():
    import bench
    return bench


def test_decode_algorithmic_bytes_by_hand():
    bench = _bench()
    sh = W.Shape(8, 2, 64, 16, "bf16")
    step = W.decode_step("t", sh, [1, 16, 17, 40], seed=3)
    # K and V rows of every context position per KV head, q and out rows, one table
    # entry per block touched, one length per sequence
    kv = sum(c * 2 * 2 * 64 * 2 for c in [1, 16, 17, 40])
    rows = 4 * 8 * 64
    blocks = 1 + 1 + 2 + 3
    want = kv + rows * 2 + rows * 4 + 4 * blocks + 4 * 4
    assert bench.decode_algorithmic_bytes(step, 4) == want


def test_prefill_flops_and_bytes_by_hand():
    bench = _bench()
    sh = W.Shape(4, 2, 64, 16, "bf16")
    ctx, ql = [5, 40], [3, 17]
    step = W.prefill_step("t", sh, ctx, ql, seed=4)
    pairs = 0
    for c, q in zip(ctx, ql):
        for i in range(q):  # query token i sits at position c - q + i and sees 0 .. itself
            pairs += c - q + i + 1
    assert bench.prefill_useful_flops(step) == 4 * 64 * 4 * pairs
    kv = sum(c * 2 * 2 * 64 * 2 for c in ctx)
    rows = sum(ql) * 4 * 64
    tables = sum(-(-c // 16) for c in ctx) * 4 + 8 * 2
    assert bench.prefill_algorithmic_bytes(step, 2) == kv + rows * 4 + tables


def test_step_roofline_fields_of_the_mixed_workload():
    """The mixed workload's step roofline: decode bytes at HBM speed plus the prefill at
    the slower of its two bounds (the tensor bound here)."""
    bench = _bench()
    step = W.NAMED["mixed_prefill_decode"]()
    dec = bench.decode_algorithmic_bytes(step, 2)
    pf_flops = bench.prefill_useful_flops(step)
    pf_bytes = bench.prefill_algorithmic_bytes(step, 2)
    assert dec > 19e9 and 5e11 < pf_flops < 6e11
    # the prefill batch is compute-bound at any plausible pair of peaks
    assert pf_flops / 1.9e15 > pf_bytes / 7.9e12
    assert np.isclose(pf_flops, 552_859_598_848)
