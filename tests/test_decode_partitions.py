"""Split-KV partitioning does not change the decode result.

pa_decode cuts long contexts into partitions and merges their partial softmax results by
log-sum-exp rescaling; the pages define only the attention itself (the same result as
over a contiguous cache), so every partitioning must give the oracle's output.  The
testing entry point fixes the partition length, from one block per partition (the most
partitions a context can have) to 128 blocks (a single partition for contexts of up to
128 blocks).

Bar: each result within the decode tolerance of the float64 oracle, and every two
partitionings of the same batch within that tolerance of each other; in addition the
pairwise spread must stay below PAIR_TIGHT, far under the tolerance, so that a merge
or partition-boundary mistake that moves only low-order bits is caught too.
"""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun, max_abs_err, oracle_step, to_f64

pytestmark = pytest.mark.gpu

# P carried as a hi + lo pair of 16-bit terms keeps each probability to 2^-17 relative;
# two partitionings round different probabilities, so their outputs (|v| <~ 4) may differ
# by ~6e-5 at the very worst, and fp32 sums add ~1e-6.
PAIR_TIGHT = {"bf16": 2.5e-4, "f16": 2.5e-4, "f32": 5e-6}


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _run_partitions(pa, step, part_blocks_list):
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()  # cache write + pa_decode with the partition size it picks
    ref = oracle_step(step, kc, vc, vals)["out_decode"]
    sh, b, m = step.shape, step.decode, run.meta["decode"]
    outs = {"auto": to_f64(res["out_decode"])}
    for pb in part_blocks_list:
        nbytes = pa.testing_decode_workspace_bytes(b.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                                   sh.head_dim, b.max_ctx, sh.block_size, pb)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = torch.full_like(res["out_decode"], float("nan"))
        pa.testing_decode_partitions(out, run.vals["q_decode"], run.vals["k_cache"],
                                     run.vals["v_cache"], m["bt"], m["ctx"], b.max_ctx,
                                     step.scale, pb, ws)
        torch.cuda.synchronize()
        outs[pb] = to_f64(out)
    assert pa.get_status() == 0
    tol = TOL[sh.dtype]
    for key, got in outs.items():
        assert np.isfinite(got).all(), key
        assert max_abs_err(got, ref) <= tol, (key, max_abs_err(got, ref))
    keys = list(outs)
    for i in range(len(keys)):
        for j in range(i + 1, len(keys)):
            d = max_abs_err(outs[keys[i]], outs[keys[j]])
            assert d <= tol, (keys[i], keys[j], d)
            assert d <= PAIR_TIGHT[sh.dtype], (keys[i], keys[j], d)
    return outs


def test_one_long_sequence_every_partition_count(pa):
    """4,099 tokens = 257 blocks of 16 (the last holding 3 tokens): 257, 129, 37, 5 and 3
    partitions."""
    step = W.decode_step("p_long", W.Shape(32, 8, 128, 16, "bf16"), [4099], seed=31)
    _run_partitions(pa, step, [1, 2, 7, 64, 128])


@pytest.mark.parametrize("dtype,bs,d,h_q,h_kv", [
    ("bf16", 16, 128, 32, 8), ("f16", 32, 128, 32, 8), ("bf16", 16, 64, 16, 2),
    ("f32", 16, 128, 8, 2)])
def test_batch_from_one_partition_to_one_block_each(pa, dtype, bs, d, h_q, h_kv):
    """A GQA batch whose contexts fit one 128-block partition: part_blocks = 128 gives
    every sequence a single partition (its output written directly, no merge), 1 gives
    one partition per block; lengths straddle block and partition edges."""
    ctx = [1, 2, bs - 1, bs, bs + 1, 7 * bs - 1, 7 * bs, 7 * bs + 1, 333, 64 * bs + 5,
           128 * bs - 1, 128 * bs]
    step = W.decode_step("p_batch", W.Shape(h_q, h_kv, d, bs, dtype), ctx, seed=32)
    _run_partitions(pa, step, [1, 2, 7, 64, 128])


def test_partition_sizes_are_validated(pa):
    with pytest.raises(pa.PaError) as e:
        step = W.decode_step("p_bad", W.Shape(8, 2, 128, 16, "bf16"), [40], seed=33)
        run = StepRun(step)
        out = torch.empty(1, 8, 128, device="cuda")
        ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        pa.testing_decode_partitions(out, run.vals["q_decode"], run.vals["k_cache"],
                                     run.vals["v_cache"], run.meta["decode"]["bt"],
                                     run.meta["decode"]["ctx"], 40, step.scale, 129, ws)
    assert e.value.code == 1
