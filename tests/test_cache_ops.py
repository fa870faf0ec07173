"""Slot mapping, cache write and block copy on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()  # clear
    return pa


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("query_lens,ctx,bs", [
    ([1, 1, 1, 1], [1, 16, 17, 100], 16),
    ([5, 16, 1, 33], [5, 40, 33, 200], 16),
    ([512, 1, 512], [512, 7, 16896], 32),
    ([0, 3, 0], [10, 3, 1], 16),
])
def test_slot_mapping_bit_exact(pa, query_lens, ctx, bs):
    step = W.prefill_step("t", W.Shape(4, 2, 64, bs, "bf16"), ctx, query_lens, seed=1)
    b = step.prefill
    slots = torch.empty(b.num_new_tokens, dtype=torch.int64, device="cuda")
    pa.slot_mapping(slots, _dev(b.block_tables), _dev(b.cu_q_lens), _dev(b.context_lens), bs,
                    step.num_blocks)
    ref = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, bs)
    assert np.array_equal(slots.cpu().numpy(), ref)
    assert pa.get_status() == 0


def test_slot_mapping_flags_positions_outside_the_table(pa):
    tables = np.array([[3, 4], [5, -1]], dtype=np.int32)
    cu = np.array([0, 1, 2], dtype=np.int32)
    ctx = np.array([40, 20], dtype=np.int32)  # sequence 0 past its 2-block table; 1 at block -1
    slots = torch.empty(2, dtype=torch.int64, device="cuda")
    pa.slot_mapping(slots, _dev(tables), _dev(cu), _dev(ctx), 16, 8)
    assert slots.cpu().tolist() == [-1, -1]
    st = pa.get_status()
    assert st & pa.STATUS_BAD_CONTEXT and st & pa.STATUS_BAD_BLOCK


@pytest.mark.parametrize("dtype,h_kv,d,bs", [("bf16", 8, 128, 16), ("f16", 40, 128, 16),
                                            ("f32", 4, 64, 16), ("bf16", 8, 128, 32),
                                            ("f16", 2, 64, 32)])
def test_reshape_and_cache_bit_exact(pa, dtype, h_kv, d, bs):
    step = W.decode_step("t", W.Shape(h_kv, h_kv, d, bs, dtype), [1, bs - 1, bs, bs + 1, 77],
                         seed=3)
    vals = W.make_values(step, "cuda")
    b = step.decode
    kc0, vc0 = W.to_numpy(vals["k_cache"]), W.to_numpy(vals["v_cache"])
    slots_np = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, bs)
    slots_np[2] = -1  # one padding token
    pa.reshape_and_cache(vals["k_new_decode"], vals["v_new_decode"], vals["k_cache"],
                         vals["v_cache"], _dev(slots_np))
    oracle.reshape_and_cache(W.to_numpy(vals["k_new_decode"]), W.to_numpy(vals["v_new_decode"]),
                             kc0, vc0, slots_np)
    assert np.array_equal(W.to_numpy(vals["k_cache"]), kc0)
    assert np.array_equal(W.to_numpy(vals["v_cache"]), vc0)
    assert pa.get_status() == 0


def test_reshape_and_cache_skips_slots_outside_the_pool(pa):
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    pa.reshape_and_cache(kn, kn, kc, vc, _dev(np.array([64, 5], dtype=np.int64)))
    assert pa.get_status() & pa.STATUS_BAD_SLOT
    assert kc.float().sum().item() == 2 * 64 and kc[0, :, 5].float().sum().item() == 128


@pytest.mark.parametrize("dtype,h_kv,d,bs", [("bf16", 8, 128, 16), ("f32", 4, 64, 32)])
def test_copy_blocks_bit_exact(pa, dtype, h_kv, d, bs):
    g = torch.Generator(device="cuda").manual_seed(7)
    layers = 3
    ks = [W.randn((40, h_kv, bs, d), dtype, "cuda", g) for _ in range(layers)]
    vs = [W.randn((40, h_kv, bs, d), dtype, "cuda", g) for _ in range(layers)]
    pairs = np.array([[1, 30], [1, 31], [7, 2], [39, 0]], dtype=np.int32)
    host = [W.to_numpy(t) for t in ks + vs]
    before = [h.copy() for h in host]
    pa.copy_blocks(ks, vs, _dev(pairs))
    oracle.copy_blocks(host, pairs)
    for got, ref, old in zip(ks + vs, host, before):
        got = W.to_numpy(got)
        assert np.array_equal(got, ref)
        for src in pairs[:, 0]:
            assert np.array_equal(got[src], old[src])  # sources untouched
    assert pa.get_status() == 0


def test_copy_blocks_skips_pairs_outside_the_pool(pa):
    kc = torch.arange(4 * 2 * 16 * 64, device="cuda").reshape(4, 2, 16, 64).to(torch.float32)
    ref = kc.clone()
    pa.copy_blocks([kc], [kc.clone()], _dev(np.array([[0, 9], [2, 3]], dtype=np.int32)))
    assert pa.get_status() & pa.STATUS_BAD_BLOCK
    ref[3] = ref[2]
    assert torch.equal(kc, ref)


@pytest.mark.parametrize("query_lens,ctx,bs,dtype", [
    ([1, 1, 1, 1], [1, 16, 17, 100], 16, "bf16"),
    ([5, 16, 1, 33], [5, 40, 33, 200], 16, "f16"),
    ([512, 1, 9], [512, 7, 16896], 32, "bf16"),
    ([0, 3, 0], [10, 3, 1], 16, "f32"),
])
def test_cache_append_bit_exact(pa, query_lens, ctx, bs, dtype):
    """Slot mapping fused with the cache write gives the same slots and pool as the two
    separate operations of the oracle."""
    step = W.prefill_step("a", W.Shape(8, 4, 128, bs, dtype), ctx, query_lens, seed=5)
    b = step.prefill
    vals = W.make_values(step, "cuda")
    kc0, vc0 = W.to_numpy(vals["k_cache"]), W.to_numpy(vals["v_cache"])
    slots = torch.full((b.num_new_tokens,), -7, dtype=torch.int64, device="cuda")
    pa.cache_append(vals["k_new_prefill"], vals["v_new_prefill"], vals["k_cache"],
                    vals["v_cache"], _dev(b.block_tables), _dev(b.cu_q_lens),
                    _dev(b.context_lens), b.max_q, slots)
    ref = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, bs)
    oracle.reshape_and_cache(W.to_numpy(vals["k_new_prefill"]), W.to_numpy(vals["v_new_prefill"]),
                             kc0, vc0, ref)
    assert np.array_equal(slots.cpu().numpy(), ref)
    assert np.array_equal(W.to_numpy(vals["k_cache"]), kc0)
    assert np.array_equal(W.to_numpy(vals["v_cache"]), vc0)
    assert pa.get_status() == 0


def test_cache_append_without_slot_output(pa):
    step = W.decode_step("a2", W.Shape(32, 8, 128, 16, "bf16"), [1, 17, 300], seed=6)
    b = step.decode
    vals = W.make_values(step, "cuda")
    kc0 = W.to_numpy(vals["k_cache"])
    pa.cache_append(vals["k_new_decode"], vals["v_new_decode"], vals["k_cache"], vals["v_cache"],
                    _dev(b.block_tables), _dev(b.cu_q_lens), _dev(b.context_lens), 1)
    ref = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, 16)
    oracle.reshape_and_cache(W.to_numpy(vals["k_new_decode"]), W.to_numpy(vals["v_new_decode"]),
                             kc0, kc0.copy(), ref)
    assert np.array_equal(W.to_numpy(vals["k_cache"]), kc0)
