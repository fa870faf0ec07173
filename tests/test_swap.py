"""pa_swap_blocks (device <-> page-locked host pools) and pre-emption by swap driven by
the C++ block manager, on the GPU, against the oracle.  Copies are bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_harness import TOL, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def _pools(n, shape, dtype, device, seed, pin=False):
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = []
    for _ in range(n):
        t = W.randn(shape, dtype, "cpu", g)
        out.append(t.pin_memory() if pin else t.to(device))
    return out


@pytest.mark.parametrize("dtype,h_kv,d,bs", [("bf16", 8, 128, 16), ("f16", 4, 64, 32),
                                            ("f32", 2, 128, 16)])
@pytest.mark.parametrize("pairs_on", ["cuda", "pinned"])
def test_swap_out_and_in_bit_exact(pa, dtype, h_kv, d, bs, pairs_on):
    layers = 3
    dev = _pools(2 * layers, (40, h_kv, bs, d), dtype, "cuda", 1)
    host = _pools(2 * layers, (24, h_kv, bs, d), dtype, "cpu", 2, pin=True)
    dev0 = [W.to_numpy(t) for t in dev]
    host_np = [W.to_numpy(t) for t in host]
    out_pairs = np.array([[3, 0], [39, 23], [7, 5], [0, 11], [21, 12]], dtype=np.int32)
    pt = torch.from_numpy(out_pairs)
    pt = pt.cuda() if pairs_on == "cuda" else pt.pin_memory()
    pa.swap_blocks(dev[:layers], dev[layers:], host[:layers], host[layers:], pt)
    torch.cuda.synchronize()
    oracle.swap_blocks(dev0, host_np, out_pairs)
    for h, ref in zip(host, host_np):
        assert np.array_equal(W.to_numpy(h), ref)
    # the device blocks are reused, then the host copies come back to other blocks
    for t in dev:
        t[[3, 39, 7, 0, 21]] = 0
    in_pairs = np.array([[0, 30], [23, 3], [5, 8], [11, 9], [12, 39]], dtype=np.int32)
    pt = torch.from_numpy(in_pairs)
    pt = pt.cuda() if pairs_on == "cuda" else pt.pin_memory()
    dev_np = [W.to_numpy(t) for t in dev]
    pa.swap_blocks(host[:layers], host[layers:], dev[:layers], dev[layers:], pt)
    torch.cuda.synchronize()
    oracle.swap_blocks(host_np, dev_np, in_pairs)
    for t, ref in zip(dev, dev_np):
        assert np.array_equal(W.to_numpy(t), ref)
    assert pa.get_status() == 0


def test_device_to_device(pa):
    a = _pools(2, (16, 8, 16, 128), "bf16", "cuda", 3)
    b = _pools(2, (16, 8, 16, 128), "bf16", "cuda", 4)
    a_np, b_np = [W.to_numpy(t) for t in a], [W.to_numpy(t) for t in b]
    pairs = np.array([[1, 2], [15, 0]], dtype=np.int32)
    pa.swap_blocks(a[:1], a[1:], b[:1], b[1:], torch.from_numpy(pairs).cuda())
    oracle.swap_blocks(a_np, b_np, pairs)
    for t, ref in zip(b, b_np):
        assert np.array_equal(W.to_numpy(t), ref)


def test_pageable_host_pool_is_rejected(pa):
    dev = _pools(2, (8, 8, 16, 128), "bf16", "cuda", 5)
    host = [torch.zeros((8, 8, 16, 128), dtype=torch.bfloat16) for _ in range(2)]  # not pinned
    with pytest.raises(pa.PaError, match="page-locked"):
        pa.swap_blocks(dev[:1], dev[1:], host[:1], host[1:],
                       torch.tensor([[0, 0]], dtype=torch.int32, device="cuda"))


def test_pairs_outside_the_pools_are_skipped_and_flagged(pa):
    dev = _pools(2, (8, 8, 16, 128), "bf16", "cuda", 6)
    host = _pools(2, (4, 8, 16, 128), "bf16", "cpu", 7, pin=True)
    host_np = [W.to_numpy(t) for t in host]
    dev_np = [W.to_numpy(t) for t in dev]
    pairs = np.array([[1, 4], [8, 0], [2, 1]], dtype=np.int32)  # host has 4 blocks; dev 8
    pa.swap_blocks(dev[:1], dev[1:], host[:1], host[1:], torch.from_numpy(pairs).cuda())
    assert pa.get_status() & pa.STATUS_BAD_BLOCK
    oracle.swap_blocks(dev_np, host_np, pairs[2:])
    for h, ref in zip(host, host_np):
        assert np.array_equal(W.to_numpy(h), ref)


def test_preemption_by_swap_end_to_end(pa):
    """The block manager admits sequences, pre-empts two of them by swapping their blocks
    to host memory, lets others reuse the freed blocks, and brings them back; the decode
    over the restored tables equals the oracle's decode over the original contents."""
    from paged_kv_cache_53_gb300.block_manager import BlockManager
    sh = W.Shape(32, 8, 128, 16, "bf16")
    nb, nh = 64, 32
    bm = BlockManager(nb, sh.block_size, num_host_blocks=nh)
    rng = np.random.default_rng(9)
    lens = {0: 70, 1: 33, 2: 100, 3: 17}
    for s, n in lens.items():
        bm.add_sequence(s, rng.integers(0, 1000, n).tolist())
    g = torch.Generator(device="cpu").manual_seed(10)
    kc = W.randn((nb, sh.num_kv_heads, sh.block_size, sh.head_dim), "bf16", "cpu", g).cuda()
    vc = W.randn((nb, sh.num_kv_heads, sh.block_size, sh.head_dim), "bf16", "cpu", g).cuda()
    hk = torch.zeros((nh,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    seqs = [0, 1, 2, 3]
    tables0, ctx0 = bm.block_tables(seqs, 8)
    kc0, vc0 = W.to_numpy(kc), W.to_numpy(vc)
    logical = {s: (oracle.gather_context(kc0, tables0[i], ctx0[i]),
                   oracle.gather_context(vc0, tables0[i], ctx0[i])) for i, s in enumerate(seqs)}

    out_pairs = bm.swap_out([1, 2])
    pa.swap_blocks([kc], [vc], [hk], [hv], torch.from_numpy(out_pairs).cuda())
    # another sequence takes the freed blocks and overwrites them
    bm.add_sequence(4, rng.integers(0, 1000, 16 * (nb - 10)).tolist()[:bm.num_free_blocks() * 16])
    for b in bm.block_table(4):
        kc[b] = 7
        vc[b] = -7
    bm.free_sequence(4)
    in_pairs = bm.swap_in([1, 2])
    pa.swap_blocks([hk], [hv], [kc], [vc], torch.from_numpy(in_pairs).cuda())
    torch.cuda.synchronize()
    assert pa.get_status() == 0

    tables, ctx = bm.block_tables(seqs, 8)
    assert np.array_equal(ctx, ctx0)
    kc1, vc1 = W.to_numpy(kc), W.to_numpy(vc)
    for i, s in enumerate(seqs):  # every sequence reads back exactly what it held
        assert np.array_equal(oracle.gather_context(kc1, tables[i], ctx[i]), logical[s][0])
        assert np.array_equal(oracle.gather_context(vc1, tables[i], ctx[i]), logical[s][1])

    q = W.randn((4, sh.num_q_heads, sh.head_dim), "bf16", "cpu", g).cuda()
    out = torch.empty((4, sh.num_q_heads, sh.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(pa.decode_workspace_bytes(4, 32, 8, 128, int(ctx.max()), 16),
                     dtype=torch.uint8, device="cuda")
    pa.decode(out, q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(),
              int(ctx.max()), 1 / np.sqrt(128), ws)
    ref = oracle.decode_attention(W.to_numpy(q), kc0, vc0, tables0, ctx0, 1 / np.sqrt(128),
                                  "bf16")
    assert np.max(np.abs(to_f64(out) - ref)) <= TOL["bf16"]
    assert pa.get_status() == 0
