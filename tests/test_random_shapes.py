"""Seeded random cases across the supported shapes, against the float64 oracle.

Each case draws, from a fixed seed (every run checks the same cases), a dtype, head dim,
block size, query / KV head counts and a ragged set of lengths that favours the edges (1,
a block, a block +- 1, a 128-token tile +- 1), for decode, chunked prefill and
shared-prefix decode.  The bars are those of the dedicated tests: the step's cache writes
bit for bit, and max |gpu - oracle| <= 2e-3 for fp16/bf16 inputs and 1e-5 for fp32 inputs,
on fp32 outputs.
"""
import numpy as np
import pytest

import workloads as W
from pa_harness import TOL, StepRun, max_abs_err, oracle_step, to_f64

pytestmark = pytest.mark.gpu

# (query heads, KV heads): group sizes 1, 2, 4, 8 and 16
HEADS = [(4, 4), (8, 4), (16, 4), (32, 8), (16, 2), (32, 2), (8, 8)]


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _length(rng, bs, lo, hi):
    edges = [e for e in (1, 2, bs - 1, bs, bs + 1, 127, 128, 129, 255, 256, 257, 513)
             if lo <= e <= hi]
    if edges and rng.random() < 0.5:
        return int(rng.choice(edges))
    return int(rng.integers(lo, hi + 1))


def _shape(rng, dtypes):
    hq, hkv = HEADS[int(rng.integers(len(HEADS)))]
    return W.Shape(hq, hkv, int(rng.choice([64, 128])), int(rng.choice([16, 32])),
                   str(rng.choice(dtypes)))


def _compare(pa, step, kind):
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run(kinds=(kind,), share_prefix=step.shared_prefix is not None)
    ref = oracle_step(step, kc, vc, vals)
    # the step's cache writes, bit for bit (the oracle applied them to its copy of the pool)
    assert np.array_equal(W.to_numpy(run.vals["k_cache"]), kc)
    assert np.array_equal(W.to_numpy(run.vals["v_cache"]), vc)
    got = to_f64(res[f"out_{kind}"])
    assert np.isfinite(got).all()
    err = max_abs_err(got, ref[f"out_{kind}"])
    assert err <= TOL[step.shape.dtype], (step.shape, err)
    assert pa.get_status() == 0


@pytest.mark.parametrize("case", range(32))
def test_random_decode(pa, case):
    rng = np.random.default_rng(53_100 + case)
    shape = _shape(rng, ["bf16", "f16", "f32"])
    n = int(rng.integers(1, 33))
    ctx = [_length(rng, shape.block_size, 1, 3000) for _ in range(n)]
    _compare(pa, W.decode_step("rnd_dec", shape, ctx, seed=53_100 + case), "decode")


@pytest.mark.parametrize("case", range(32))
def test_random_prefill(pa, case):
    rng = np.random.default_rng(53_200 + case)
    shape = _shape(rng, ["bf16", "f16"])
    n = int(rng.integers(1, 9))
    chunks = [_length(rng, shape.block_size, 1, 300) for _ in range(n)]
    ctx = [q + _length(rng, shape.block_size, 1, 1500) - 1 for q in chunks]
    _compare(pa, W.prefill_step("rnd_pre", shape, ctx, chunks, seed=53_200 + case), "prefill")


@pytest.mark.parametrize("case", range(16))
def test_random_shared_prefix(pa, case):
    rng = np.random.default_rng(53_300 + case)
    shape = _shape(rng, ["bf16", "f16"])
    prefix = shape.block_size * int(rng.integers(1, 40))
    sharers = [_length(rng, shape.block_size, 1, 400) for _ in range(int(rng.integers(1, 80)))]
    others = [_length(rng, shape.block_size, 1, 900) for _ in range(int(rng.integers(0, 8)))]
    step = W.shared_prefix_step("rnd_sp", shape, prefix, sharers, others, seed=53_300 + case)
    _compare(pa, step, "decode")
