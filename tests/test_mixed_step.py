"""pa_mixed_step (a batch's decodes and prefill chunks side by side on disjoint SMs)
against the same work as separate calls in turn, and against the float64 oracle.

Bar: caches, slots and outputs bit for bit equal to pa_decode_append +
pa_cache_append + pa_prefill_chunk on the same inputs (the same kernels over the same
bytes), and within the tolerances of the oracle on a sample of rows.
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


def _buffers(pa, run, out_dtype):
    st, sh = run.step, run.step.shape
    bufs = {}
    if st.decode is not None:
        b = st.decode
        bufs["decode"] = dict(
            out=torch.empty((b.num_seqs, sh.num_q_heads, sh.head_dim), dtype=out_dtype,
                            device="cuda"),
            slots=torch.full((b.num_seqs,), -9, dtype=torch.int64, device="cuda"),
            workspace=torch.empty(pa.decode_workspace_bytes(b.num_seqs, sh.num_q_heads,
                                                            sh.num_kv_heads, sh.head_dim,
                                                            b.max_ctx, sh.block_size),
                                  dtype=torch.uint8, device="cuda"))
    if st.prefill is not None:
        b = st.prefill
        bufs["prefill"] = dict(
            out=torch.empty((b.num_new_tokens, sh.num_q_heads, sh.head_dim), dtype=out_dtype,
                            device="cuda"),
            slots=torch.full((b.num_new_tokens,), -9, dtype=torch.int64, device="cuda"),
            workspace=torch.empty(max(16, pa.prefill_workspace_bytes(
                b.num_seqs, b.num_new_tokens, b.max_q, sh.num_q_heads, sh.num_kv_heads,
                sh.head_dim, b.max_ctx, sh.block_size)), dtype=torch.uint8, device="cuda"))
    return bufs


def _args(run, bufs):
    st = run.step
    dec = pre = None
    if st.decode is not None:
        m = run.meta["decode"]
        dec = dict(q=run.vals["q_decode"], k_new=run.vals["k_new_decode"],
                   v_new=run.vals["v_new_decode"], block_tables=m["bt"], context_lens=m["ctx"],
                   max_ctx=st.decode.max_ctx, **bufs["decode"])
    if st.prefill is not None:
        m = run.meta["prefill"]
        pre = dict(q=run.vals["q_prefill"], k_new=run.vals["k_new_prefill"],
                   v_new=run.vals["v_new_prefill"], block_tables=m["bt"], cu_q_lens=m["cu"],
                   context_lens=m["ctx"], max_q=st.prefill.max_q, max_ctx=st.prefill.max_ctx,
                   **bufs["prefill"])
    return dec, pre


def _mixed(pa, step, out_dtype=torch.float32):
    run = StepRun(step)
    bufs = _buffers(pa, run, out_dtype)
    dec, pre = _args(run, bufs)
    pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec, prefill=pre)
    torch.cuda.synchronize()
    return run, bufs


def _separate(pa, step, out_dtype=torch.float32):
    run = StepRun(step)
    bufs = _buffers(pa, run, out_dtype)
    dec, pre = _args(run, bufs)
    kc, vc = run.vals["k_cache"], run.vals["v_cache"]
    if dec is not None:
        pa.decode_append(dec["out"], dec["q"], dec["k_new"], dec["v_new"], kc, vc,
                         dec["block_tables"], dec["context_lens"], dec["max_ctx"], step.scale,
                         dec["workspace"], slots=dec["slots"])
    if pre is not None:
        pa.cache_append(pre["k_new"], pre["v_new"], kc, vc, pre["block_tables"], pre["cu_q_lens"],
                        pre["context_lens"], pre["max_q"], pre["slots"])
        pa.prefill_chunk(pre["out"], pre["q"], kc, vc, pre["block_tables"], pre["cu_q_lens"],
                         pre["context_lens"], pre["max_q"], pre["max_ctx"], step.scale,
                         pre["workspace"])
    torch.cuda.synchronize()
    return run, bufs


def _same(run_a, bufs_a, run_b, bufs_b):
    assert torch.equal(run_a.vals["k_cache"], run_b.vals["k_cache"])
    assert torch.equal(run_a.vals["v_cache"], run_b.vals["v_cache"])
    for kind in bufs_a:
        assert torch.equal(bufs_a[kind]["slots"], bufs_b[kind]["slots"]), kind
        assert torch.equal(bufs_a[kind]["out"], bufs_b[kind]["out"]), kind


def test_mixed_workload_matches_separate_calls(pa):
    """The full mixed workload (248 decodes up to 131,072 tokens beside 8 prefill chunks of
    512 tokens over up to 16,384): bit for bit the calls in turn."""
    step = W.mixed_prefill_decode()
    run_m, bufs_m = _mixed(pa, step)
    run_s, bufs_s = _separate(pa, step)
    _same(run_m, bufs_m, run_s, bufs_s)
    assert pa.get_status() == 0


def test_reduced_mixed_step_against_oracle(pa):
    """Decode contexts shrunk to 2% (the prefill batch at full size): every decode row and
    a sample of prefill tokens (first, diagonal-straddling and last of each chunk) against
    the oracle."""
    step = W.mixed_prefill_decode(decode_scale=0.02)
    ref_run = StepRun(step)
    kc, vc = ref_run.host_pool()
    vals = ref_run.host_values()
    run, bufs = _mixed(pa, step)
    cu = step.prefill.cu_q_lens
    toks = sorted({int(t) for b in range(step.prefill.num_seqs)
                   for t in (cu[b], cu[b] + 127, cu[b] + 128, cu[b + 1] - 1)})
    ref = oracle_step(step, kc, vc, vals, prefill_tokens=toks)
    np.testing.assert_array_equal(bufs["decode"]["slots"].cpu().numpy(), ref["slots_decode"])
    np.testing.assert_array_equal(bufs["prefill"]["slots"].cpu().numpy(), ref["slots_prefill"])
    assert np.abs(to_f64(bufs["decode"]["out"]) - ref["out_decode"]).max() <= TOL["bf16"]
    got = to_f64(bufs["prefill"]["out"])[toks]
    assert np.abs(got - ref["out_prefill"]).max() <= TOL["bf16"]
    assert pa.get_status() == 0


@pytest.mark.parametrize("keep", ["decode", "prefill"])
def test_one_batch_alone(pa, keep):
    step = W.mixed_prefill_decode(decode_scale=0.05)
    step = W.replace(step, prefill=None) if keep == "decode" else W.replace(step, decode=None)
    run_m, bufs_m = _mixed(pa, step)
    run_s, bufs_s = _separate(pa, step)
    _same(run_m, bufs_m, run_s, bufs_s)
    assert pa.get_status() == 0


def test_native_output_dtype(pa):
    step = W.mixed_prefill_decode(decode_scale=0.05)
    run_m, bufs_m = _mixed(pa, step, out_dtype=torch.bfloat16)
    run_s, bufs_s = _separate(pa, step, out_dtype=torch.bfloat16)
    _same(run_m, bufs_m, run_s, bufs_s)


def test_captured_in_a_cuda_graph(pa):
    """The side stream forks from and joins the capturing stream: a captured step replays
    to the same bytes as an eager one."""
    step = W.mixed_prefill_decode(decode_scale=0.05)
    run_e, bufs_e = _mixed(pa, step)
    run = StepRun(step)
    kc0, vc0 = run.vals["k_cache"].clone(), run.vals["v_cache"].clone()
    bufs = _buffers(pa, run, torch.float32)
    dec, pre = _args(run, bufs)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec,
                      prefill=pre, stream=s)  # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec,
                          prefill=pre, stream=s)
    for _ in range(2):
        run.vals["k_cache"].copy_(kc0)
        run.vals["v_cache"].copy_(vc0)
        for kind in bufs:
            bufs[kind]["out"].zero_()
        g.replay()
        torch.cuda.synchronize()
        _same(run, bufs, run_e, bufs_e)
    assert pa.get_status() == 0


def test_back_to_back_steps(pa):
    """Steps issued back to back reuse the library's side stream and events."""
    step = W.mixed_prefill_decode(decode_scale=0.05)
    run, bufs = _mixed(pa, step)
    first = {k: v["out"].clone() for k, v in bufs.items()}
    dec, pre = _args(run, bufs)
    for _ in range(4):
        pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec,
                      prefill=pre)
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k]["out"], first[k])
    assert pa.get_status() == 0
