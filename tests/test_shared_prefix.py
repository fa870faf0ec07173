"""Decode with a shared prefix attended once (pa_decode_shared_prefix) against the float64
oracle, which walks every sequence's full block table on its own.

Bar: the decode bar, max |gpu - oracle| <= 2e-3 on fp32 outputs for fp16/bf16 inputs;
cache writes and copies of the same steps bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun, half_ulp, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _check(pa, step, out_dtype=torch.float32):
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run(out_dtype=out_dtype, share_prefix=True)
    ref = oracle_step(step, kc, vc, vals)
    assert np.array_equal(W.to_numpy(run.vals["k_cache"]), kc)
    assert np.array_equal(W.to_numpy(run.vals["v_cache"]), vc)
    got = to_f64(res["out_decode"])
    err = np.abs(got - ref["out_decode"])
    tol = TOL[step.shape.dtype]
    if out_dtype != torch.float32:
        tol = tol + half_ulp(ref["out_decode"], step.shape.dtype)
    assert np.all(err <= tol), f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}"
    assert pa.get_status() == 0
    return run, res


def test_prefix_sharing_cow_workload(pa):
    """The prefix-sharing workload (128 rows on one 2048-token prefix, 8 groups of 4
    samples with copy-on-write) through the shared-prefix entry point."""
    _check(pa, W.prefix_sharing_cow())


def test_matches_plain_decode(pa):
    """Same inputs through pa_decode and pa_decode_shared_prefix: both within the bar, and
    close to each other (they differ only in summation order)."""
    step = W.prefix_sharing_cow()
    a = StepRun(step).run(kinds=("decode",))["out_decode"]
    b = StepRun(step).run(kinds=("decode",), share_prefix=True)["out_decode"]
    assert torch.max(torch.abs(a - b)).item() <= 2e-3
    assert pa.get_status() == 0


# ------------------------------------------------------------------ shapes and edges
def _suffixes(n, seed, hi=300, with_zero=True):
    rng = np.random.default_rng(seed)
    s = rng.integers(1, hi, size=n, endpoint=True)
    if with_zero and n > 1:
        s[n // 2] = 0  # one row whose context ends at the prefix
    return s


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d,bs", [(128, 16), (128, 32), (64, 16), (64, 32)])
@pytest.mark.parametrize("h_q,h_kv", [(32, 8), (8, 8), (16, 2), (32, 2)])
def test_shapes(pa, dtype, d, bs, h_q, h_kv):
    # 592 = 37 blocks of 16 (not a whole number of 128-token tiles); 576 for block 32
    prefix = 592 if bs == 16 else 576
    step = W.shared_prefix_step("sp", W.Shape(h_q, h_kv, d, bs, dtype), prefix,
                                _suffixes(37, 11), [5, 700, 1], seed=12)
    _check(pa, step)


@pytest.mark.parametrize("n_sharers", [1, 2, 63, 64, 65, 200])
def test_sharer_counts(pa, n_sharers):
    """Ragged query-row tiles: G = 4 rows per sharer, 256 rows per CTA."""
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 1024,
                                _suffixes(n_sharers, n_sharers), [33, 2000], seed=n_sharers)
    _check(pa, step)


@pytest.mark.parametrize("prefix", [16, 128, 144, 4096, 8192])
def test_prefix_lengths(pa, prefix):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), prefix,
                                _suffixes(24, prefix), [prefix + 17], seed=prefix)
    _check(pa, step)


# Bound for large V values: P enters P V as bf16 hi + lo terms, each probability carried to
# a relative error of at most 2^-18, so the output moves by at most 2^-18 * max|v| (fp32
# sums add less); 2^-16 leaves a margin of 4.
def _wide_tol(v_abs_max: float) -> float:
    return TOL["bf16"] + 2.0 ** -16 * v_abs_max


@pytest.mark.parametrize("d", [64, 128])
def test_v_beyond_fp16_range_in_the_prefix(pa, d):
    """bf16 prefix V values far outside fp16's range (and one just inside it, 65280, the
    largest bf16 below 65520): the prefix's P V keeps V in bf16 and carries P as hi + lo
    terms, so outputs must match the oracle, with nothing flagged."""
    step = W.shared_prefix_step("spr", W.Shape(16, 4, d, 16, "bf16"), 512, _suffixes(20, 40),
                                [300], seed=41)
    blocks = step.shared_prefix[0]
    run = StepRun(step)
    v = run.vals["v_cache"]
    v[int(blocks[2]), 1, 3, 5] = -1.0e5   # prefix tile 0 (tokens 32..47), KV head 1
    v[int(blocks[20]), 3, 0, 0] = 3.0e6   # prefix tile 2 (token 320), KV head 3
    v[int(blocks[9]), 0, 7, 2] = 65280.0  # prefix tile 1, KV head 0: fits fp16
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run(share_prefix=True)
    assert pa.get_status() == 0
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(res["out_decode"])
    assert np.isfinite(got).all()
    assert np.abs(got - ref["out_decode"]).max() <= _wide_tol(3.0e6)


@pytest.mark.parametrize("n_sharers,n_others", [(1000, 200), (4300, 200)])
def test_many_sequences_and_sharers(pa, n_sharers, n_others):
    """1,200 sequences (more than the plan kernel has threads), 1,000 of them on one
    prefix: sharer flags and reserved partial slots over many sequences per thread; and
    4,500 sequences, past the 4,096 whose sharer flags the plan keeps in shared memory
    (beyond, it keeps them in the workspace)."""
    rng = np.random.default_rng(38 + n_sharers)
    step = W.shared_prefix_step("spmany", W.Shape(32, 8, 64, 16, "bf16"), 512,
                                rng.integers(1, 40, size=n_sharers),
                                rng.integers(1, 600, size=n_others), seed=38)
    _check(pa, step)


@pytest.mark.parametrize("n_seqs", [1024, 1025])
def test_early_records_boundary(pa, n_seqs):
    """Batches of up to 1,024 sequences let the attention kernel take every sequence's full
    partitions from its own records before the plan is done; one more and it waits for the
    plan's list.  Both sides of the boundary, with many multi-partition sequences."""
    rng = np.random.default_rng(41 + n_seqs)
    n_sharers = 900
    step = W.shared_prefix_step("spedge", W.Shape(32, 8, 64, 16, "bf16"), 256,
                                rng.integers(1, 120, size=n_sharers),
                                rng.integers(1, 300, size=n_seqs - n_sharers), seed=41)
    _check(pa, step)


def _shared_call(pa, run, ws):
    """The shared-prefix decode of `run`'s step (its cache writes already done) into a
    new fp32 output, on the workspace `ws`."""
    st, sh = run.step, run.step.shape
    b, m = st.decode, run.meta["decode"]
    out = torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), dtype=torch.float32,
                      device=run.device)
    blocks, plen, sharers = st.shared_prefix
    pa.decode_shared_prefix(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"],
                            m["bt"], m["ctx"], b.max_ctx, torch.from_numpy(blocks).to(run.device),
                            plen, torch.from_numpy(sharers).to(run.device), st.scale, ws)
    return out


def test_workspace_reused_across_batches(pa):
    """Two batches in turn on one workspace: one whose sequences have many full partitions
    (taken before the plan is done, by a counter the plan resets every call) and one with
    none.  Every call equals, bit for bit, the same call on a fresh workspace."""
    shape = W.Shape(32, 8, 128, 16, "bf16")
    rng = np.random.default_rng(43)
    sa = W.shared_prefix_step("spa", shape, 1024, rng.integers(300, 900, size=96),
                              rng.integers(500, 1500, size=16), seed=43)
    sb = W.shared_prefix_step("spb", shape, 1024, rng.integers(1, 16, size=40), [5, 9],
                              seed=44)
    runs = [StepRun(sa), StepRun(sb)]
    refs = [r.run(kinds=("decode",), share_prefix=True)["out_decode"] for r in runs]
    nbytes = 0
    for r in runs:
        st, sh = r.step, r.step.shape
        nbytes = max(nbytes, pa.decode_shared_prefix_workspace_bytes(
            st.decode.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, st.decode.max_ctx,
            sh.block_size, len(st.shared_prefix[2]), st.shared_prefix[1]))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=runs[0].device)
    for i in (0, 1, 0, 1, 1, 0):
        assert torch.equal(_shared_call(pa, runs[i], ws), refs[i]), i
    assert pa.get_status() == 0


def test_only_sharers_ending_at_the_prefix(pa):
    """A sharer with no context of its own gets the prefix's attention alone (the merge
    normalises its single partial)."""
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 256, [0], [], seed=4)
    _check(pa, step)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_native_output(pa, dtype):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, dtype), 512, _suffixes(50, 3),
                                [100], seed=5)
    _check(pa, step, out_dtype=getattr(torch, {"bf16": "bfloat16", "f16": "float16"}[dtype]))


def test_no_sharers_is_plain_decode_bit_for_bit(pa):
    """num_sharers = 0 runs pa_decode's kernels unchanged."""
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 512, _suffixes(20, 6),
                                [300, 9], seed=6)
    step = W.replace(step, shared_prefix=(step.shared_prefix[0], 512, np.zeros(0, np.int32)))
    a = StepRun(step).run(kinds=("decode",))["out_decode"]
    b = StepRun(step).run(kinds=("decode",), share_prefix=True)["out_decode"]
    assert torch.equal(a, b)
    assert pa.get_status() == 0


def test_is_deterministic(pa):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 2048, _suffixes(96, 8),
                                [512], seed=8)
    a = StepRun(step).run(kinds=("decode",), share_prefix=True)["out_decode"]
    b = StepRun(step).run(kinds=("decode",), share_prefix=True)["out_decode"]
    assert torch.equal(a, b)


def test_bad_prefix_block_is_flagged(pa):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 256, [4, 9], [], seed=9)
    run = StepRun(step)
    blocks, plen, sharers = step.shared_prefix
    bad = blocks.copy()
    bad[3] = step.num_blocks + 5
    run.step = W.replace(step, shared_prefix=(bad, plen, sharers))
    run.run(kinds=("decode",), share_prefix=True)
    assert pa.get_status() & pa.STATUS_BAD_BLOCK


def test_sharer_shorter_than_the_prefix_is_flagged(pa):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 256, [4, 9], [40],
                                seed=10)
    blocks, plen, _ = step.shared_prefix
    run = StepRun(W.replace(step, shared_prefix=(blocks, plen, np.array([0, 2], np.int32))))
    run.run(kinds=("decode",), share_prefix=True)
    assert pa.get_status() & pa.STATUS_BAD_CONTEXT


def test_sharer_index_out_of_range_is_flagged(pa):
    """A sharer index outside the batch (past its end, or negative) sets the bad-context bit
    and is skipped: no read of a query row or write of a partial outside the buffers, and
    the valid sharers' rows come out as without it."""
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 256, [4, 9, 30], [],
                                seed=12)
    blocks, plen, sharers = step.shared_prefix
    good = StepRun(step).run(kinds=("decode",), share_prefix=True)["out_decode"]
    assert pa.get_status() == 0
    for bad in (step.decode.num_seqs + 3, -1):
        with_bad = np.concatenate([sharers, [bad]]).astype(np.int32)
        run = StepRun(W.replace(step, shared_prefix=(blocks, plen, with_bad)))
        out = run.run(kinds=("decode",), share_prefix=True)["out_decode"]
        assert pa.get_status() & pa.STATUS_BAD_CONTEXT
        assert torch.equal(out, good)


def test_rejects_bad_arguments(pa):
    step = W.shared_prefix_step("sp", W.Shape(32, 8, 128, 16, "bf16"), 256, [4, 9], [], seed=1)
    run = StepRun(step)
    blocks, plen, sharers = step.shared_prefix
    for bad in [(blocks, 250, sharers), (blocks, 4096, sharers)]:
        run.step = W.replace(step, shared_prefix=bad)
        with pytest.raises(pa.PaError):
            run.run(kinds=("decode",), share_prefix=True)
    step32 = W.shared_prefix_step("sp", W.Shape(8, 8, 64, 16, "f32"), 64, [4], [], seed=1)
    with pytest.raises(pa.PaError):
        StepRun(step32).run(kinds=("decode",), share_prefix=True)
    pa.get_status()
