"""pa_decode_static_scratch: paged decode for callers that cannot allocate a workspace.

A caller that has handed all of the GPU's memory to its own pool, or that must not call
cudaMalloc/cudaFree on its path, has no workspace to pass to pa_decode; this entry point
takes its scratch from a fixed array inside the library instead.  It runs the same plan,
attention and merge kernels as pa_decode on the same inputs, and those kernels are
deterministic (the merge reads the partials in a fixed order), so its output must equal
pa_decode's (with a caller-provided workspace) bit for bit, on two calls in a row: the
second call finds the first call's leftovers in the shared array.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun

pytestmark = pytest.mark.gpu

_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


@pytest.fixture(scope="module")
def lib():
    import paged_kv_cache_53_gb300 as pa
    handle = pa.lib()
    fn = handle.pa_decode_static_scratch
    fn.argtypes = [_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]
    fn.restype = _I
    pa.get_status()
    return pa, fn


def _static_decode(pa, fn, out, run):
    st, sh, b, m = run.step, run.step.shape, run.step.decode, run.meta["decode"]
    kc, vc = run.vals["k_cache"], run.vals["v_cache"]
    rc = fn(out.data_ptr(), pa.dtype_code(out.dtype), run.vals["q_decode"].data_ptr(),
            kc.data_ptr(), vc.data_ptr(), m["bt"].data_ptr(), b.block_tables.shape[1],
            m["ctx"].data_ptr(), b.max_ctx, b.num_seqs, sh.num_q_heads, sh.num_kv_heads,
            sh.head_dim, sh.block_size, st.num_blocks, st.scale, pa.dtype_code(kc.dtype),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, pa.lib().pa_last_error_string().decode()


def test_static_scratch_matches_workspace_decode_twice(lib):
    pa, fn = lib
    steps = [W.llama8b_gqa_decode(),
             W.decode_step("second", W.Shape(16, 4, 64, 32, "f16"),
                           [1, 31, 32, 33, 500, 4096, 9000], seed=21)]
    for step in steps:  # two calls in a row, on different shapes
        run = StepRun(step)
        ref = run.run()["out_decode"]  # pa_decode with its own workspace
        out = torch.full_like(ref, float("nan"))
        _static_decode(pa, fn, out, run)
        torch.cuda.synchronize()
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= TOL[step.shape.dtype], err
        assert torch.equal(out, ref), err
    assert pa.get_status() == 0


def test_static_scratch_rejects_sizes_beyond_its_array(lib):
    pa, fn = lib
    need = pa.decode_workspace_bytes(248, 32, 8, 128, 131072, 32)
    assert need > 32 << 20
    rc = fn(None, 2, None, None, None, None, 4096, None, 131072, 248, 32, 8, 128, 32, 200000,
            0.1, 2, None)
    assert rc == 3
    assert "fixed" in pa.lib().pa_last_error_string().decode()
