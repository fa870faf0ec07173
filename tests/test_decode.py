"""Paged decode attention on the GPU against the float64 oracle.

Bar: max |gpu - oracle| <= 2e-3 for fp16/bf16 inputs and <= 1e-5 for fp32 inputs, on fp32
outputs; native-dtype outputs may add half an ulp of the output type.  Slots, cache
writes and block copies of the same steps are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import (TOL, StepRun, blocks_of, half_ulp, max_abs_err, oracle_step, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _full_check(pa, step, out_dtype=torch.float32):
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run(out_dtype=out_dtype)
    ref = oracle_step(step, kc, vc, vals)
    assert np.array_equal(res["slots_decode"].cpu().numpy(), ref["slots_decode"])
    # the cache after the step (copies and writes) is bit-identical
    assert np.array_equal(W.to_numpy(run.vals["k_cache"]), kc)
    assert np.array_equal(W.to_numpy(run.vals["v_cache"]), vc)
    got = to_f64(res["out_decode"])
    err = np.abs(got - ref["out_decode"])
    tol = TOL[step.shape.dtype]
    if out_dtype != torch.float32:
        tol = tol + half_ulp(ref["out_decode"], step.shape.dtype)
    assert np.all(err <= tol), f"max err {err.max():.3g}"
    assert pa.get_status() == 0
    return float(err.max())


# ------------------------------------------------------------------ the named workloads
def test_tiny_decode_fp32(pa):
    step = W.tiny_decode()
    err = _full_check(pa, step)
    assert err <= 1e-5


def test_tiny_decode_single_token_context_returns_v(pa):
    """Context length 1: the output is the freshly written V, exactly."""
    step = W.tiny_decode()
    run = StepRun(step)
    res = run.run()
    out = res["out_decode"].cpu()
    v_new = run.vals["v_new_decode"].cpu()
    assert torch.equal(out[0], v_new[0])  # 4 query heads = 4 KV heads


def test_opt13b_decode_fp16(pa):
    _full_check(pa, W.opt13b_decode())


def test_llama8b_gqa_decode_bf16(pa):
    _full_check(pa, W.llama8b_gqa_decode())


def test_llama8b_gqa_decode_native_bf16_output(pa):
    _full_check(pa, W.llama8b_gqa_decode(), out_dtype=torch.bfloat16)


def test_prefix_sharing_cow(pa):
    step = W.prefix_sharing_cow()
    run = StepRun(step)
    kc, vc = run.host_pool()
    src_before = kc[step.cow_pairs[:, 0]].copy()
    vals = run.host_values()
    res = run.run()
    ref = oracle_step(step, kc, vc, vals)
    k_after = W.to_numpy(run.vals["k_cache"])
    assert np.array_equal(k_after, kc) and np.array_equal(W.to_numpy(run.vals["v_cache"]), vc)
    # the copies left the shared prompt tokens of every source block untouched, and
    # every copy holds those tokens too
    b = step.decode
    for i, (src, dst) in enumerate(step.cow_pairs):
        n = int(b.context_lens[128 + 4 * (i // 3)]) - 1  # prompt length of the group
        assert np.array_equal(k_after[src, :, :n % 16], src_before[i, :, :n % 16])
        assert np.array_equal(k_after[dst, :, :n % 16], src_before[i, :, :n % 16])
    got = to_f64(res["out_decode"])
    assert max_abs_err(got, ref["out_decode"]) <= TOL["bf16"]
    # samples of a group differ only through their appended token
    for g in range(8):
        rows = list(range(128 + 4 * g, 128 + 4 * g + 4))
        n = int(b.context_lens[rows[0]]) - 1
        kk = [W.to_numpy(run.vals["k_cache"])[b.block_tables[r, n // 16], :, : n % 16] for r in rows]
        for x in kk[1:]:
            assert np.array_equal(x, kk[0])
    assert pa.get_status() == 0


def test_mixed_decode_sampled(pa):
    """The long-context decode batch of the mixed workload at full size (split-KV over
    131,072-token contexts), compared on a sample of sequences that includes every
    131,072-token one."""
    step = W.mixed_prefill_decode()
    step = W.replace(step, prefill=None)
    run = StepRun(step)
    b = step.decode
    rng = np.random.default_rng(0)
    seqs = sorted(set(rng.choice(240, size=6, replace=False).tolist()) | set(range(240, 248)))
    block_map = blocks_of(b, seqs, step.shape.block_size)
    kc, vc = run.host_pool(block_map)
    vals = run.host_values()
    res = run.run()
    ref = oracle_step(step, kc, vc, vals, decode_seqs=seqs, block_map=block_map)
    assert np.array_equal(res["slots_decode"].cpu().numpy(), ref["slots_decode"])
    got = to_f64(res["out_decode"])[seqs]
    assert max_abs_err(got, ref["out_decode"]) <= TOL["bf16"]
    assert pa.get_status() == 0


# ------------------------------------------------------------------ edge cases
EDGE_CTX = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257,
            511, 512, 513, 1000, 2047, 2048, 2049, 3001]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("h_q,h_kv", [(4, 4), (8, 4), (16, 4), (16, 2), (32, 2)])
def test_decode_shapes(pa, dtype, d, bs, h_q, h_kv):
    step = W.decode_step("edge", W.Shape(h_q, h_kv, d, bs, dtype), EDGE_CTX, seed=11)
    _full_check(pa, step)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_decode_native_output(pa, dtype):
    step = W.decode_step("edge", W.Shape(32, 8, 128, 16, dtype), EDGE_CTX, seed=12)
    _full_check(pa, step, out_dtype=W._torch_dtype(dtype))


@pytest.mark.parametrize("n,hi,dtype", [(3000, 300, "bf16"), (20000, 9, "f16"), (1500, 40, "f32")])
def test_decode_many_sequences(pa, n, hi, dtype):
    """More sequences than the plan kernel has threads (several per thread), short
    contexts: tens of thousands of single-partition units and their direct outputs."""
    ctx = np.random.default_rng(n).integers(1, hi, size=n, endpoint=True)
    step = W.decode_step("many", W.Shape(16, 4, 64, 16, dtype), ctx, seed=n)
    _full_check(pa, step)


def test_decode_many_partitions_one_sequence(pa):
    """One sequence far longer than the partition size: dozens of partials merged."""
    step = W.decode_step("long1", W.Shape(32, 8, 128, 16, "bf16"), [65536 + 7], seed=13)
    _full_check(pa, step)


def test_decode_empty_context_gives_zeros(pa):
    step = W.decode_step("z", W.Shape(8, 2, 128, 16, "bf16"), [5, 1, 40], seed=14)
    run = StepRun(step)
    run.run()
    b = step.decode
    ctx = torch.tensor([5, 0, 40], dtype=torch.int32, device="cuda")
    out = torch.full((3, 8, 128), 7.0, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(3, 8, 2, 128, 40, 16), dtype=torch.uint8,
                     device="cuda")
    pa.decode(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"],
              run.meta["decode"]["bt"], ctx, 40, step.scale, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]).item() == 0
    assert torch.isfinite(out).all()
    assert pa.get_status() == 0


def test_decode_nan_past_context_is_ignored(pa):
    """Slots past a sequence's context may hold anything, NaN included; they must not
    reach the output."""
    step = W.decode_step("nan", W.Shape(8, 2, 128, 16, "bf16"), [3, 17, 30], seed=15)
    run = StepRun(step)
    b = step.decode
    for s in range(b.num_seqs):
        ctx = int(b.context_lens[s])
        blk = int(b.block_tables[s, (ctx - 1) // 16])
        run.vals["k_cache"][blk, :, (ctx - 1) % 16 + 1:] = float("nan")
        run.vals["v_cache"][blk, :, (ctx - 1) % 16 + 1:] = float("nan")
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(res["out_decode"])
    assert np.isfinite(got).all()
    assert max_abs_err(got, ref["out_decode"]) <= TOL["bf16"]


def test_decode_bad_block_id_is_flagged_and_contained(pa):
    """A corrupt table entry sets the status word; other sequences stay correct."""
    step = W.decode_step("bad", W.Shape(8, 2, 128, 16, "bf16"), [40, 50, 60], seed=16)
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()  # clean run first
    pa.get_status()
    bt = run.meta["decode"]["bt"].clone()
    bt[1, 1] = step.num_blocks + 5
    out = torch.empty_like(res["out_decode"])
    ws = torch.empty(pa.decode_workspace_bytes(3, 8, 2, 128, 60, 16), dtype=torch.uint8,
                     device="cuda")
    pa.decode(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"], bt,
              run.meta["decode"]["ctx"], 60, step.scale, ws)
    assert pa.get_status() & pa.STATUS_BAD_BLOCK
    ref = oracle_step(step, kc, vc, vals)
    got = to_f64(out)
    assert max_abs_err(got[[0, 2]], ref["out_decode"][[0, 2]]) <= TOL["bf16"]


def test_decode_context_past_max_ctx_is_flagged(pa):
    step = W.decode_step("cap", W.Shape(8, 2, 128, 16, "bf16"), [40, 50], seed=17)
    run = StepRun(step)
    run.run()
    pa.get_status()
    out = torch.empty(2, 8, 128, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(2, 8, 2, 128, 45, 16), dtype=torch.uint8,
                     device="cuda")
    pa.decode(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"],
              run.meta["decode"]["bt"], run.meta["decode"]["ctx"], 45, step.scale, ws)
    assert pa.get_status() & pa.STATUS_BAD_CONTEXT
    assert torch.isfinite(out).all()


def test_decode_is_deterministic(pa):
    step = W.llama8b_gqa_decode()
    run = StepRun(step)
    a = run.run()["out_decode"].clone()
    b_ = step.decode
    m = run.meta["decode"]
    out = torch.empty_like(a)
    ws = torch.empty(pa.decode_workspace_bytes(b_.num_seqs, 32, 8, 128, b_.max_ctx, 16),
                     dtype=torch.uint8, device="cuda")
    for _ in range(3):
        pa.decode(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"], m["bt"],
                  m["ctx"], b_.max_ctx, step.scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, a)
