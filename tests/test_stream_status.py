"""Status words of their own for the calls on a stream (pa_set_stream_status).

Two streams, each with a caller-owned word: a data fault in a call on one stream sets a
bit in that stream's word only, the device-wide word stays clear, and removing the entry
sends bits back to the device word.  Calls whose kernels run on the library's side stream
(pa_mixed_step's prefill half) report to the word of the caller's stream.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import StepRun

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _bad_decode(pa, run, stream, bad_block=False, bad_ctx=False):
    step, m = run.step, run.meta["decode"]
    bt = m["bt"].clone()
    if bad_block:
        bt[1, 1] = step.num_blocks + 5
    max_ctx = 45 if bad_ctx else step.decode.max_ctx
    out = torch.empty(step.decode.num_seqs, step.shape.num_q_heads, step.shape.head_dim,
                      device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(step.decode.num_seqs, step.shape.num_q_heads,
                                               step.shape.num_kv_heads, step.shape.head_dim,
                                               max_ctx, step.shape.block_size),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    pa.decode(out, run.vals["q_decode"], run.vals["k_cache"], run.vals["v_cache"], bt,
              m["ctx"], max_ctx, step.scale, ws, stream=stream)
    return out


def test_two_streams_keep_their_bits_apart(pa):
    step = W.decode_step("sw", W.Shape(8, 2, 128, 16, "bf16"), [40, 50, 60], seed=71)
    run = StepRun(step)
    run.run()
    assert pa.get_status() == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    w2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.set_stream_status(s1, w1)
    pa.set_stream_status(s2, w2)
    try:
        _bad_decode(pa, run, s1, bad_block=True)
        _bad_decode(pa, run, s2, bad_ctx=True)
        pa.selftest_wait_timeout(200, s2)
        torch.cuda.synchronize()
        assert int(w1.item()) == pa.STATUS_BAD_BLOCK
        assert int(w2.item()) == pa.STATUS_BAD_CONTEXT | pa.STATUS_TIMEOUT
        assert pa.get_status() == 0  # nothing reached the device-wide word
        # registering a stream again replaces its word
        w3 = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.set_stream_status(s1, w3)
        _bad_decode(pa, run, s1, bad_ctx=True)
        torch.cuda.synchronize()
        assert int(w3.item()) == pa.STATUS_BAD_CONTEXT
        assert int(w1.item()) == pa.STATUS_BAD_BLOCK
    finally:
        pa.set_stream_status(s1, None)
        pa.set_stream_status(s2, None)
    # without an entry the device word gets the bits again
    _bad_decode(pa, run, s1, bad_block=True)
    torch.cuda.synchronize()
    assert pa.get_status() == pa.STATUS_BAD_BLOCK


def test_mixed_step_side_stream_reports_to_the_callers_word(pa):
    """A corrupt block id in the prefill half of pa_mixed_step (run on the library's own
    stream) sets the bit in the word registered for the caller's stream."""
    step = W.replace(W.mixed_prefill_decode(decode_scale=0.02), name="sw_mixed")
    run = StepRun(step)
    sh, d, p = step.shape, step.decode, step.prefill
    md, mp = run.meta["decode"], run.meta["prefill"]
    bt_pre = mp["bt"].clone()
    bt_pre[0, 0] = step.num_blocks + 7
    s = torch.cuda.Stream()
    w = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec = dict(out=torch.empty(d.num_seqs, sh.num_q_heads, sh.head_dim, device="cuda"),
               q=run.vals["q_decode"], k_new=run.vals["k_new_decode"],
               v_new=run.vals["v_new_decode"], block_tables=md["bt"], context_lens=md["ctx"],
               max_ctx=d.max_ctx,
               workspace=torch.empty(pa.decode_workspace_bytes(
                   d.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, d.max_ctx,
                   sh.block_size), dtype=torch.uint8, device="cuda"))
    pre = dict(out=torch.empty(p.num_new_tokens, sh.num_q_heads, sh.head_dim, device="cuda"),
               q=run.vals["q_prefill"], k_new=run.vals["k_new_prefill"],
               v_new=run.vals["v_new_prefill"], block_tables=bt_pre, cu_q_lens=mp["cu"],
               context_lens=mp["ctx"], max_q=p.max_q, max_ctx=p.max_ctx,
               workspace=torch.empty(max(16, pa.prefill_workspace_bytes(
                   p.num_seqs, p.num_new_tokens, p.max_q, sh.num_q_heads, sh.num_kv_heads,
                   sh.head_dim, p.max_ctx, sh.block_size)), dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    pa.set_stream_status(s, w)
    try:
        pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec,
                      prefill=pre, stream=s)
        torch.cuda.synchronize()
        assert int(w.item()) & pa.STATUS_BAD_BLOCK
        assert pa.get_status() == 0
    finally:
        pa.set_stream_status(s, None)
    # the library's side stream and events can be released and are made again on demand
    pa.release_thread_resources()
    pa.release_thread_resources()  # nothing left: a no-op
    pa.mixed_step(run.vals["k_cache"], run.vals["v_cache"], step.scale, decode=dec,
                  prefill=pre, stream=s)
    torch.cuda.synchronize()
    assert pa.get_status() & pa.STATUS_BAD_BLOCK
    pa.release_thread_resources()
