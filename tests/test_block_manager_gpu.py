"""One decode step whose block tables, copy-on-write pairs and slots come from the C++
block manager, run through the device path and compared with the oracle (which runs the
reference block manager, its own copies, cache writes and attention)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle.block_manager import BlockManager as RefManager
from pa_harness import TOL, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def test_decode_step_fed_by_the_block_manager(pa):
    from paged_kv_cache_53_gb300.block_manager import BlockManager
    sh = W.Shape(32, 8, 128, 16, "bf16")
    nb = 256
    bm = BlockManager(nb, 16, prefix_caching=True)
    ref = RefManager(nb, 16, prefix_caching=True)
    rng = np.random.default_rng(21)
    system = rng.integers(0, 30_000, 160).tolist()  # 10 full blocks shared through the cache
    seqs = []
    for s in range(6):
        toks = system + rng.integers(0, 30_000, int(rng.integers(1, 41))).tolist()
        assert bm.add_sequence(s, toks) == ref.add_sequence(s, toks)
        seqs.append(s)
    prompt = rng.integers(0, 30_000, 37).tolist()  # a partly filled last block
    bm.add_sequence(10, prompt)
    ref.add_sequence(10, prompt)
    seqs.append(10)
    for c in (11, 12, 13):  # parallel samples of the prompt
        bm.fork(10, c)
        ref.fork(10, c)
        seqs.append(c)
    new_tok = rng.integers(0, 30_000, len(seqs)).tolist()
    for s, t in zip(seqs, new_tok):
        bm.append_tokens(s, [t])
        ref.append_tokens(s, [t])
    pairs = bm.take_copies()
    ref_pairs = np.asarray(ref.take_copies(), dtype=np.int32).reshape(-1, 2)
    assert pairs.tolist() == ref_pairs.tolist() and len(pairs) == 3
    width = 16
    tables, ctx = bm.block_tables(seqs, width)
    assert np.array_equal(tables, ref.block_tables(seqs, width))
    slots_host = bm.slot_mapping(seqs, [1] * len(seqs))

    # device side: pool, copies, fused slot mapping + cache write, decode
    g = torch.Generator(device="cpu").manual_seed(22)
    kc = W.randn((nb, 8, 16, 128), "bf16", "cpu", g).cuda()
    vc = W.randn((nb, 8, 16, 128), "bf16", "cpu", g).cuda()
    q = W.randn((len(seqs), 32, 128), "bf16", "cpu", g).cuda()
    kn = W.randn((len(seqs), 8, 128), "bf16", "cpu", g).cuda()
    vn = W.randn((len(seqs), 8, 128), "bf16", "cpu", g).cuda()
    kc0, vc0 = W.to_numpy(kc), W.to_numpy(vc)
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    cu = torch.arange(len(seqs) + 1, dtype=torch.int32, device="cuda")
    slots = torch.empty(len(seqs), dtype=torch.int64, device="cuda")
    pa.copy_blocks([kc], [vc], torch.from_numpy(pairs).cuda())
    pa.cache_append(kn, vn, kc, vc, bt, cu, cl, 1, slots)
    out = torch.empty((len(seqs), 32, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(len(seqs), 32, 8, 128, int(ctx.max()), 16),
                     dtype=torch.uint8, device="cuda")
    pa.decode(out, q, kc, vc, bt, cl, int(ctx.max()), 1 / np.sqrt(128), ws)
    torch.cuda.synchronize()
    assert pa.get_status() == 0
    assert np.array_equal(slots.cpu().numpy(), slots_host)

    # oracle side
    ref_slots = ref.slot_mapping(seqs, [1] * len(seqs))
    assert np.array_equal(ref_slots, slots_host)
    oracle.copy_blocks([kc0, vc0], ref_pairs)
    oracle.reshape_and_cache(W.to_numpy(kn), W.to_numpy(vn), kc0, vc0, ref_slots)
    assert np.array_equal(W.to_numpy(kc), kc0) and np.array_equal(W.to_numpy(vc), vc0)
    o = oracle.decode_attention(W.to_numpy(q), kc0, vc0, ref.block_tables(seqs, width),
                                ref.context_lens(seqs), 1 / np.sqrt(128), "bf16")
    assert np.max(np.abs(to_f64(out) - o)) <= TOL["bf16"]
