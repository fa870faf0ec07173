"""pa_decode_append (one decode step: cache write of each sequence's new token, then the
decode) against the separate calls and against the float64 oracle.

Bar: cache bytes and slots bit for bit; outputs bit for bit equal to pa_cache_append +
pa_decode on the same inputs (the same kernels over the same bytes) and within the
decode tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _fused(pa, step, out_dtype=torch.float32, with_slots=True):
    """Runs pa_decode_append on a fresh copy of the step's values."""
    run = StepRun(step)
    b, sh, m = step.decode, step.shape, run.meta["decode"]
    kc, vc = run.vals["k_cache"], run.vals["v_cache"]
    out = torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), dtype=out_dtype, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(b.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                               sh.head_dim, b.max_ctx, sh.block_size),
                     dtype=torch.uint8, device="cuda")
    slots = torch.full((b.num_seqs,), -7, dtype=torch.int64, device="cuda") if with_slots else None
    pa.decode_append(out, run.vals["q_decode"], run.vals["k_new_decode"], run.vals["v_new_decode"],
                     kc, vc, m["bt"], m["ctx"], b.max_ctx, step.scale, ws, slots=slots)
    torch.cuda.synchronize()
    return run, out, slots


def _separate(pa, step, out_dtype=torch.float32):
    run = StepRun(step)
    b, sh, m = step.decode, step.shape, run.meta["decode"]
    kc, vc = run.vals["k_cache"], run.vals["v_cache"]
    slots = torch.empty(b.num_seqs, dtype=torch.int64, device="cuda")
    pa.cache_append(run.vals["k_new_decode"], run.vals["v_new_decode"], kc, vc, m["bt"], m["cu"],
                    m["ctx"], 1, slots)
    out = torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), dtype=out_dtype, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(b.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                               sh.head_dim, b.max_ctx, sh.block_size),
                     dtype=torch.uint8, device="cuda")
    pa.decode(out, run.vals["q_decode"], kc, vc, m["bt"], m["ctx"], b.max_ctx, step.scale, ws)
    torch.cuda.synchronize()
    return run, out, slots


@pytest.mark.parametrize("name", ["llama8b_gqa_decode", "opt13b_decode", "tiny_decode"])
def test_workloads_match_separate_calls_and_oracle(pa, name):
    step = W.NAMED[name]()
    ref_run = StepRun(step)
    kc0, vc0 = ref_run.host_pool()
    vals = ref_run.host_values()
    run_f, out_f, slots_f = _fused(pa, step)
    run_s, out_s, slots_s = _separate(pa, step)
    assert pa.get_status() == 0
    assert torch.equal(slots_f, slots_s)
    assert torch.equal(run_f.vals["k_cache"], run_s.vals["k_cache"])
    assert torch.equal(run_f.vals["v_cache"], run_s.vals["v_cache"])
    assert torch.equal(out_f, out_s)
    ref = oracle_step(step, kc0, vc0, vals)
    np.testing.assert_array_equal(slots_f.cpu().numpy(), ref["slots_decode"])
    err = np.abs(to_f64(out_f) - ref["out_decode"])
    assert err.max() <= TOL[step.shape.dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d,bs,hq,hkv", [(128, 16, 32, 8), (64, 32, 16, 16), (128, 32, 16, 1)])
def test_shapes_and_native_output(pa, dtype, d, bs, hq, hkv):
    rng = np.random.default_rng(d + bs + hq)
    ctx = rng.integers(1, 3000, size=37)
    ctx[3] = 1                     # the new token is the whole context
    ctx[5] = bs                    # it ends a block
    ctx[7] = bs + 1                # it opens a block
    step = W.decode_step("da", W.Shape(hq, hkv, d, bs, dtype), ctx, seed=int(ctx.sum()))
    odt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    _, out_f, _ = _fused(pa, step, out_dtype=odt, with_slots=False)
    _, out_s, _ = _separate(pa, step, out_dtype=odt)
    assert torch.equal(out_f, out_s)
    assert pa.get_status() == 0


def test_many_sequences(pa):
    """3,000 sequences (more than the plan kernel's threads) through the fused call."""
    rng = np.random.default_rng(77)
    step = W.decode_step("da_many", W.Shape(32, 8, 64, 16, "bf16"), rng.integers(1, 400, 3000),
                         seed=77)
    run_f, out_f, slots_f = _fused(pa, step)
    run_s, out_s, slots_s = _separate(pa, step)
    assert torch.equal(out_f, out_s) and torch.equal(slots_f, slots_s)
    assert torch.equal(run_f.vals["k_cache"], run_s.vals["k_cache"])
    assert pa.get_status() == 0


def test_back_to_back_steps_reuse_one_workspace(pa):
    """Steps issued back to back on one stream (the plan of step n+1 runs beside step
    n+1's cache write, after step n's merge): every step's output as computed alone."""
    step = W.NAMED["llama8b_gqa_decode"]()
    run = StepRun(step)
    b, sh, m = step.decode, step.shape, run.meta["decode"]
    kc, vc = run.vals["k_cache"], run.vals["v_cache"]
    ws = torch.empty(pa.decode_workspace_bytes(b.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                               sh.head_dim, b.max_ctx, sh.block_size),
                     dtype=torch.uint8, device="cuda")
    outs = [torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), device="cuda")
            for _ in range(6)]
    for o in outs:
        pa.decode_append(o, run.vals["q_decode"], run.vals["k_new_decode"],
                         run.vals["v_new_decode"], kc, vc, m["bt"], m["ctx"], b.max_ctx,
                         step.scale, ws)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert pa.get_status() == 0


def test_empty_context_and_bad_block_are_flagged(pa):
    step = W.decode_step("da_bad", W.Shape(32, 8, 128, 16, "bf16"), [5, 1, 40], seed=5)
    step.decode.context_lens[1] = 0  # no position for the new token
    _fused(pa, step)
    assert pa.get_status() & pa.STATUS_BAD_CONTEXT
    step = W.decode_step("da_bad2", W.Shape(32, 8, 128, 16, "bf16"), [5, 33, 40], seed=6)
    step.decode.block_tables[1, 2] = step.num_blocks + 3  # the new token's block
    _fused(pa, step)
    assert pa.get_status() & pa.STATUS_BAD_BLOCK
