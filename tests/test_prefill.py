"""Chunked-prefill attention (tcgen05) on the GPU against the float64 oracle.

Bar: max |gpu - oracle| <= 2e-3 on fp32 outputs from fp16/bf16 inputs; native-dtype
outputs may add half an ulp of the output type.  The chunk's slots and cache writes are
compared bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun, blocks_of, half_ulp, max_abs_err, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _check(pa, step, out_dtype=torch.float32, tokens=None):
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run(out_dtype=out_dtype)
    ref = oracle_step(step, kc, vc, vals, prefill_tokens=tokens)
    assert np.array_equal(res["slots_prefill"].cpu().numpy(), ref["slots_prefill"])
    got = to_f64(res["out_prefill"])
    if tokens is not None:
        got = got[tokens]
    err = np.abs(got - ref["out_prefill"])
    tol = TOL[step.shape.dtype]
    if out_dtype != torch.float32:
        tol = tol + half_ulp(ref["out_prefill"], step.shape.dtype)
    assert np.all(err <= tol), f"max err {err.max():.3g}"
    assert pa.get_status() == 0
    return float(err.max())


def test_prefill_small_bf16(pa):
    step = W.prefill_step("p", W.Shape(8, 2, 128, 16, "bf16"), [5, 40], [5, 16], seed=31)
    _check(pa, step)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("h_q,h_kv", [(4, 4), (8, 2), (32, 8), (16, 2), (32, 2)])
def test_prefill_shapes(pa, dtype, d, bs, h_q, h_kv):
    # chunks straddling tile and block edges, contexts starting at 0 and deeper in
    chunks = [1, 5, 31, 33, 64, 129, 200]
    ctx0 = [0, 63, 1, 64, 0, 1000, 77]
    ctx = [c + q for c, q in zip(ctx0, chunks)]
    step = W.prefill_step("pe", W.Shape(h_q, h_kv, d, bs, dtype), ctx, chunks, seed=32)
    _check(pa, step)


def test_prefill_zero_token_chunks(pa):
    """Sequences that append nothing this step sit between ones that do: they get no
    rows and change nothing; the others match the oracle."""
    chunks = [0, 7, 0, 1, 130, 0]
    ctx = [50, 67, 1, 1, 130, 300]
    step = W.prefill_step("pz", W.Shape(32, 8, 128, 16, "bf16"), ctx, chunks, seed=39)
    _check(pa, step)


def test_prefill_many_sequences(pa):
    """More sequences than the plan kernel has threads: 1,500 chunks of 1 to 6 tokens over
    contexts of up to 200 tokens (one work item each per KV head)."""
    rng = np.random.default_rng(37)
    q = rng.integers(1, 6, size=1500, endpoint=True)
    ctx = q + rng.integers(0, 200 - 6, size=1500, endpoint=True)
    step = W.prefill_step("pmany", W.Shape(16, 4, 64, 16, "bf16"), ctx, q, seed=37)
    _check(pa, step)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_native_output(pa, dtype):
    step = W.prefill_step("pn", W.Shape(32, 8, 128, 32, dtype), [512, 700], [512, 100], seed=33)
    _check(pa, step, out_dtype=W._torch_dtype(dtype))


def test_prefill_first_row_of_a_fresh_prompt_is_v0(pa):
    """A chunk that starts at position 0: its first query sees one token, so its output
    is that token's V (bf16 values, exact in fp32)."""
    step = W.prefill_step("p0", W.Shape(8, 8, 128, 16, "bf16"), [20], [20], seed=34)
    run = StepRun(step)
    res = run.run()
    v0 = run.vals["v_new_prefill"][0].float()  # [H_kv, D]
    assert torch.equal(res["out_prefill"][0], v0)


def test_prefill_nan_past_context_is_ignored(pa):
    step = W.prefill_step("pnan", W.Shape(8, 2, 128, 16, "bf16"), [37, 70], [9, 33], seed=35)
    run = StepRun(step)
    b = step.prefill
    for s in range(b.num_seqs):
        ctx = int(b.context_lens[s])
        blk = int(b.block_tables[s, (ctx - 1) // 16])
        run.vals["k_cache"][blk, :, (ctx - 1) % 16 + 1:] = float("nan")
        run.vals["v_cache"][blk, :, (ctx - 1) % 16 + 1:] = float("nan")
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(res["out_prefill"])
    assert np.isfinite(got).all()
    assert max_abs_err(got, ref["out_prefill"]) <= TOL["bf16"]


# Bound for V values outside fp16's range, which the exact pass takes with P as bf16 hi +
# lo terms: each probability is carried to a relative error of at most 2^-18, so the
# output moves by at most 2^-18 * max|v| (fp32 sums add less); 2^-16 leaves a margin of 4.
def _wide_tol(v_abs_max: float) -> float:
    return TOL["bf16"] + 2.0 ** -16 * v_abs_max


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_v_beyond_fp16_range_is_exact(pa, d):
    """P V runs in fp16 with V converted from bf16; a V value of magnitude >= 65520 does not
    fit, and the work items that meet one are computed again with V in bf16 and P as hi +
    lo terms.  Outputs must match the oracle (no status bit: nothing is flagged)."""
    step = W.prefill_step("prange", W.Shape(8, 2, d, 16, "bf16"), [40, 300], [8, 200],
                          seed=36)
    run = StepRun(step)
    b = step.prefill
    # large values in sequence 0's first block (KV head 1) and in sequence 1's context
    blk0 = int(b.block_tables[0, 0])
    run.vals["v_cache"][blk0, 1, 2, 7] = -1.0e5
    run.vals["v_cache"][blk0, 1, 5, 0] = 3.0e6
    blk1 = int(b.block_tables[1, 3])
    run.vals["v_cache"][blk1, 0, 9, 11] = 7.0e4
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()
    assert pa.get_status() == 0
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(res["out_prefill"])
    assert np.isfinite(got).all()
    assert max_abs_err(got, ref["out_prefill"]) <= _wide_tol(3.0e6)


def test_prefill_exact_pass_touches_only_marked_items(pa):
    """Only the work items whose V holds an out-of-range value are computed again: the
    other sequence's outputs equal those of a run without any such value, bit for bit;
    values just inside fp16's range stay on the fast path."""
    shape = W.Shape(32, 8, 128, 32, "bf16")
    step = W.prefill_step("pmark", shape, [600, 700], [300, 200], seed=38)
    clean = StepRun(step)
    blk = int(step.prefill.block_tables[1, 2])
    clean.vals["v_cache"][blk, 3, 1, 2] = 65280.0  # the largest bf16 below 65520
    out_clean = clean.run()["out_prefill"]
    assert pa.get_status() == 0
    run = StepRun(step)
    run.vals["v_cache"][blk, 3, 1, 2] = 65280.0
    blk0 = int(step.prefill.block_tables[0, 1])
    run.vals["v_cache"][blk0, 5, 4, 100] = -2.5e5
    kc, vc = run.host_pool()
    vals = run.host_values()
    out = run.run()["out_prefill"]
    assert pa.get_status() == 0
    n0 = int(step.prefill.query_lens[0])
    assert torch.equal(out[n0:], out_clean[n0:])
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(out)
    assert max_abs_err(got, ref["out_prefill"]) <= _wide_tol(2.5e5)


def test_mixed_prefill_full_size_sampled(pa):
    """The mixed workload's prefill batch at full size (8 chunks of 512 over up to 16,384
    context tokens, block size 32), compared on sampled rows of every sequence that
    include each chunk's first and last token."""
    step = W.mixed_prefill_decode()
    step = W.replace(step, decode=None)
    b = step.prefill
    rng = np.random.default_rng(1)
    tokens = []
    for s in range(b.num_seqs):
        lo, hi = int(b.cu_q_lens[s]), int(b.cu_q_lens[s + 1])
        pick = {lo, lo + 1, hi - 1} | set(rng.integers(lo, hi, size=13).tolist())
        tokens.extend(sorted(pick))
    _check(pa, step, tokens=tokens)


def test_prefill_then_decode_agree_on_the_last_token(pa):
    """The last query of a chunk sees the whole context, like a decode query."""
    shape = W.Shape(32, 8, 128, 16, "bf16")
    ctx = [300, 1000]
    chunks = [50, 128]
    step = W.prefill_step("pd", shape, ctx, chunks, seed=36)
    run = StepRun(step)
    res = run.run()
    last = torch.tensor([49, 50 + 127], device="cuda")
    q_last = run.vals["q_prefill"][last].contiguous()
    m = run.meta["prefill"]
    out = torch.empty(2, 32, 128, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(2, 32, 8, 128, 1000, 16), dtype=torch.uint8,
                     device="cuda")
    pa.decode(out, q_last, run.vals["k_cache"], run.vals["v_cache"], m["bt"], m["ctx"], 1000,
              step.scale, ws)
    torch.cuda.synchronize()
    assert (out - res["out_prefill"][last]).abs().max().item() <= 2e-3
