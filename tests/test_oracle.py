"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks retypes the oracle's own formula: each compares it with a number
the pages print, a closed form, an invariant the pages state, torch's float64 CPU
scaled-dot-product attention on contiguous tensors, or a pure-Python brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")


@pytest.fixture(scope="module")
def pages():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------------------------
# numbers the pages print
# ----------------------------------------------------------------------------------

def test_kv_bytes_per_token_opt13b(pages):
    e = pages["kv_bytes_per_token"][0]
    # the page multiplies layers by the hidden size, i.e. KV heads x head dim as one factor
    assert oracle.kv_bytes_per_token(e["layers"], 1, e["kv_heads_times_head_dim"],
                                     e["bytes_per_value"]) == e["bytes"]
    # and the same with the model's 40 heads of 128
    assert oracle.kv_bytes_per_token(40, 40, 128, 2) == e["bytes"]


def test_kv_bytes_per_token_llama8b(pages):
    e = pages["kv_bytes_per_token"][1]
    assert oracle.kv_bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"],
                                     e["bytes_per_value"]) == e["bytes"]
    s = pages["sequence_cache_bytes"]
    total = s["tokens"] * oracle.kv_bytes_per_token(32, 8, 128, 2)
    assert total == 1_073_741_824
    assert round(total / 1e9, 2) == s["approx_gb"]


def test_paged_tail_waste_example(pages):
    e = pages["paged_tail_waste"]
    blocks = oracle.blocks_for_tokens(e["tokens"], e["block_size"])
    assert blocks * e["block_size"] == e["allocated_slots"]
    assert oracle.tail_waste(e["tokens"], e["block_size"]) == e["wasted_slots"]
    assert e["wasted_slots"] * e["bytes_per_token"] == e["wasted_bytes_approx_mib"] * 2 ** 20


def test_prefix_block_example(pages):
    e = pages["prefix_blocks"]
    assert oracle.full_blocks(e["prompt_tokens"], e["block_size"]) == e["full_blocks"]
    assert e["full_blocks"] * e["block_size"] == e["full_block_tokens"]
    shared = oracle.full_blocks(e["shared_prefix_tokens"], e["block_size"])
    assert shared == e["shared_full_blocks"]
    assert e["prompt_tokens"] - shared * e["block_size"] == e["remaining_prefill_tokens_approx"]


def test_tail_waste_below_one_block(pages):
    bs = pages["tail_waste_bound"]["block_size"]
    for n in range(1, 200):
        w = oracle.tail_waste(n, bs)
        assert 0 <= w < pages["tail_waste_bound"]["max_waste_exclusive"]
        assert oracle.blocks_for_tokens(n, bs) == math.ceil(n / bs)


# ----------------------------------------------------------------------------------
# helpers: contiguous logical caches scattered into a pool by the test itself
# ----------------------------------------------------------------------------------

def _rand(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return W.to_numpy(W.randn(shape, dtype, "cpu", g))


def _scatter(logical_k, logical_v, tables, ctx, num_blocks, block_size, fill_seed, dtype):
    """Places each sequence's contiguous [ctx, H, D] K/V into a noise-filled pool through
    its table (the inverse of a table walk, written independently of the oracle)."""
    h, d = logical_k[0].shape[1], logical_k[0].shape[2]
    kc = _rand((num_blocks, h, block_size, d), dtype, fill_seed)
    vc = _rand((num_blocks, h, block_size, d), dtype, fill_seed + 1)
    for b in range(len(ctx)):
        for t in range(int(ctx[b])):
            blk = tables[b][t // block_size]
            kc[blk, :, t % block_size, :] = logical_k[b][t]
            vc[blk, :, t % block_size, :] = logical_v[b][t]
    return kc, vc


def _problem(ctx, h_q, h_kv, d, bs, dtype, seed, extra_blocks=5):
    rng = np.random.default_rng(seed)
    nblk = [-(-c // bs) for c in ctx]
    nb = sum(nblk) + extra_blocks
    ids = rng.permutation(nb)
    tables = np.full((len(ctx), max(nblk) + 2), -1, dtype=np.int32)
    p = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = ids[p:p + n]
        p += n
    lk = [_rand((c, h_kv, d), dtype, seed * 31 + 2 * b) for b, c in enumerate(ctx)]
    lv = [_rand((c, h_kv, d), dtype, seed * 31 + 2 * b + 1) for b, c in enumerate(ctx)]
    kc, vc = _scatter(lk, lv, tables, ctx, nb, bs, seed + 7, dtype)
    return tables, lk, lv, kc, vc


def _sdpa(q64, k64, v64, scale, mask=None):
    """torch's float64 CPU scaled-dot-product attention; q [R, D], k/v [N, D]."""
    q = torch.from_numpy(q64)[None, None]
    k = torch.from_numpy(k64)[None, None]
    v = torch.from_numpy(v64)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m,
                                                            scale=scale)[0, 0].numpy()


# ----------------------------------------------------------------------------------
# decode attention
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,h_q,h_kv,d,bs", [
    ("f32", 4, 4, 64, 16), ("f16", 8, 2, 64, 16), ("bf16", 8, 2, 128, 32),
    ("bf16", 16, 2, 64, 16), ("f16", 2, 1, 128, 16),
])
def test_decode_matches_torch_sdpa(dtype, h_q, h_kv, d, bs):
    ctx = [1, bs - 1, bs, bs + 1, 3 * bs + 5]
    tables, lk, lv, kc, vc = _problem(ctx, h_q, h_kv, d, bs, dtype, 11)
    q = _rand((len(ctx), h_q, d), dtype, 99)
    scale = 1.0 / math.sqrt(d)
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), scale, dtype)
    g = h_q // h_kv
    for b, c in enumerate(ctx):
        k64, v64, q64 = oracle.widen(lk[b], dtype), oracle.widen(lv[b], dtype), \
            oracle.widen(q[b], dtype)
        for hq in range(h_q):
            ref = _sdpa(q64[hq:hq + 1], k64[:, hq // g], v64[:, hq // g], scale)[0]
            np.testing.assert_allclose(out[b, hq], ref, rtol=0, atol=1e-12)


def test_decode_brute_force_python():
    """A pure-Python loop with math.exp over a tiny GQA problem."""
    ctx = [3, 18]
    h_q, h_kv, d, bs = 4, 2, 8, 16
    tables, lk, lv, kc, vc = _problem(ctx, h_q, h_kv, d, bs, "f32", 5)
    q = _rand((2, h_q, d), "f32", 6)
    scale = 0.3
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), scale, "f32")
    for b, c in enumerate(ctx):
        for hq in range(h_q):
            h = hq // 2
            logits = [scale * sum(float(q[b, hq, i]) * float(lk[b][t, h, i]) for i in range(d))
                      for t in range(c)]
            mx = max(logits)
            w = [math.exp(x - mx) for x in logits]
            z = sum(w)
            for i in range(d):
                ref = sum(w[t] * float(lv[b][t, h, i]) for t in range(c)) / z
                assert abs(out[b, hq, i] - ref) < 1e-12


def test_single_token_context_returns_v_exactly():
    tables, lk, lv, kc, vc = _problem([1, 1, 1], 8, 2, 64, 16, "bf16", 3)
    q = _rand((3, 8, 64), "bf16", 4)
    out = oracle.decode_attention(q, kc, vc, tables, np.array([1, 1, 1]), 0.125, "bf16")
    for b in range(3):
        for hq in range(8):
            assert np.array_equal(out[b, hq], oracle.widen(lv[b][0, hq // 4], "bf16"))


def test_uniform_v_returns_v():
    ctx = [5, 40, 77]
    tables, lk, lv, kc, vc = _problem(ctx, 4, 4, 64, 16, "f32", 8)
    const = _rand((4, 64), "f32", 9)
    for b, c in enumerate(ctx):
        lv[b][:] = const[None]
    kc, vc = _scatter(lk, lv, tables, ctx, kc.shape[0], 16, 21, "f32")
    q = _rand((3, 4, 64), "f32", 10)
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), 0.2, "f32")
    for b in range(3):
        np.testing.assert_allclose(out[b], const.astype(np.float64), rtol=0, atol=1e-12)


def test_permuted_placement_is_invisible():
    """The same logical caches placed at two different sets of physical blocks give the
    same outputs bit for bit (blocks may sit anywhere)."""
    ctx = [20, 33, 64]
    tables, lk, lv, kc, vc = _problem(ctx, 8, 2, 64, 16, "f16", 12)
    q = _rand((3, 8, 64), "f16", 13)
    rng = np.random.default_rng(0)
    perm = rng.permutation(kc.shape[0])
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    kc2, vc2 = _scatter(lk, lv, tables2, ctx, kc.shape[0], 16, 77, "f16")
    a = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), 0.125, "f16")
    b = oracle.decode_attention(q, kc2, vc2, tables2, np.array(ctx), 0.125, "f16")
    assert np.array_equal(a, b)


def test_shared_prefix_equals_unshared_copies():
    """Sequences whose tables point at one physical prefix match sequences holding
    private copies of it."""
    bs, h, d = 16, 2, 64
    prefix = 48
    suffix = [5, 17, 30]
    ctx = [prefix + s for s in suffix]
    pk = _rand((prefix, h, d), "bf16", 40)
    pv = _rand((prefix, h, d), "bf16", 41)
    lk = [np.concatenate([pk, _rand((s, h, d), "bf16", 50 + i)]) for i, s in enumerate(suffix)]
    lv = [np.concatenate([pv, _rand((s, h, d), "bf16", 60 + i)]) for i, s in enumerate(suffix)]
    # private copies
    rng = np.random.default_rng(1)
    nblk = [-(-c // bs) for c in ctx]
    nb = sum(nblk) + 3
    ids = rng.permutation(nb)
    t_priv = np.full((3, max(nblk)), -1, dtype=np.int32)
    p = 0
    for b, n in enumerate(nblk):
        t_priv[b, :n] = ids[p:p + n]
        p += n
    kc1, vc1 = _scatter(lk, lv, t_priv, ctx, nb, bs, 70, "bf16")
    # shared prefix: every row points at the first row's prefix blocks
    t_shared = t_priv.copy()
    t_shared[1:, :prefix // bs] = t_priv[0, :prefix // bs]
    kc2, vc2 = _scatter(lk, lv, t_shared, ctx, nb, bs, 80, "bf16")
    q = _rand((3, 8, d), "bf16", 90)
    a = oracle.decode_attention(q, kc1, vc1, t_priv, np.array(ctx), 0.125, "bf16")
    b = oracle.decode_attention(q, kc2, vc2, t_shared, np.array(ctx), 0.125, "bf16")
    assert np.array_equal(a, b)


def test_zero_scale_gives_mean_of_v():
    ctx = [1, 9, 50]
    tables, lk, lv, kc, vc = _problem(ctx, 4, 2, 64, 16, "f32", 14)
    q = _rand((3, 4, 64), "f32", 15)
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), 0.0, "f32")
    for b in range(3):
        for hq in range(4):
            ref = lv[b][:, hq // 2].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(out[b, hq], ref, rtol=0, atol=1e-12)


def test_dominant_logit_selects_its_value():
    """A query aligned with one key (large positive scale) returns that key's V; a sign
    error would select a different token."""
    ctx = [30]
    tables, lk, lv, kc, vc = _problem(ctx, 2, 1, 64, 16, "f32", 16)
    j = 17
    q = np.zeros((1, 2, 64), dtype=np.float32)
    q[0, 0] = lk[0][j, 0]
    q[0, 1] = -lk[0][j, 0]
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), 100.0, "f32")
    np.testing.assert_allclose(out[0, 0], lv[0][j, 0], rtol=0, atol=1e-9)
    assert not np.allclose(out[0, 1], lv[0][j, 0], atol=1e-3)


def test_gqa_head_mapping():
    """V constant per KV head: query head i must return the constant of KV head
    i // (H_q / H_kv)."""
    h_q, h_kv, d = 8, 2, 64
    ctx = [21]
    tables, lk, lv, kc, vc = _problem(ctx, h_q, h_kv, d, 16, "f32", 17)
    for h in range(h_kv):
        lv[0][:, h, :] = float(h + 1)
    kc, vc = _scatter(lk, lv, tables, ctx, kc.shape[0], 16, 33, "f32")
    q = _rand((1, h_q, d), "f32", 18)
    out = oracle.decode_attention(q, kc, vc, tables, np.array(ctx), 0.125, "f32")
    for hq in range(h_q):
        np.testing.assert_allclose(out[0, hq], float(hq // (h_q // h_kv) + 1), atol=1e-12)


def test_empty_context_gives_zeros():
    tables, lk, lv, kc, vc = _problem([4], 2, 2, 64, 16, "f32", 19)
    q = _rand((1, 2, 64), "f32", 20)
    out = oracle.decode_attention(q, kc, vc, tables, np.array([0]), 0.125, "f32")
    assert not out.any()


# ----------------------------------------------------------------------------------
# chunked prefill
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,h_q,h_kv,d,bs", [("bf16", 8, 2, 64, 16),
                                                 ("f16", 4, 4, 128, 32)])
def test_prefill_matches_torch_sdpa_causal(dtype, h_q, h_kv, d, bs):
    chunks = [5, 16, 1]
    ctx = [5, 40, 33]  # first chunk starts at position 0
    tables, lk, lv, kc, vc = _problem(ctx, h_q, h_kv, d, bs, dtype, 21)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = _rand((int(cu[-1]), h_q, d), dtype, 22)
    scale = 1.0 / math.sqrt(d)
    out = oracle.prefill_chunk_attention(q, kc, vc, tables, cu, np.array(ctx), scale, dtype)
    g = h_q // h_kv
    for b in range(3):
        c0 = ctx[b] - chunks[b]
        mask = np.arange(ctx[b])[None, :] <= (c0 + np.arange(chunks[b]))[:, None]
        k64, v64 = oracle.widen(lk[b], dtype), oracle.widen(lv[b], dtype)
        q64 = oracle.widen(q[cu[b]:cu[b + 1]], dtype)
        for hq in range(h_q):
            ref = _sdpa(q64[:, hq], k64[:, hq // g], v64[:, hq // g], scale, mask)
            np.testing.assert_allclose(out[cu[b]:cu[b + 1], hq], ref, rtol=0, atol=1e-12)


def test_prefill_zero_scale_is_running_mean():
    """With scale 0 query i of a chunk starting at position c0 returns the mean of V over
    positions 0..c0+i; row 0 with c0 = 0 returns V of token 0 exactly."""
    chunk, c0 = 7, 0
    ctx = [c0 + chunk]
    tables, lk, lv, kc, vc = _problem(ctx, 2, 1, 64, 16, "f32", 23)
    q = _rand((chunk, 2, 64), "f32", 24)
    cu = np.array([0, chunk], dtype=np.int32)
    out = oracle.prefill_chunk_attention(q, kc, vc, tables, cu, np.array(ctx), 0.0, "f32")
    v = lv[0][:, 0].astype(np.float64)
    assert np.array_equal(out[0, 0], v[0])
    for i in range(chunk):
        np.testing.assert_allclose(out[i, 1], v[:c0 + i + 1].mean(axis=0), atol=1e-12)
    # a chunk that starts deeper in the context
    chunk, c0 = 5, 21
    ctx = [c0 + chunk]
    tables, lk, lv, kc, vc = _problem(ctx, 2, 1, 64, 16, "f32", 25)
    q = _rand((chunk, 2, 64), "f32", 26)
    cu = np.array([0, chunk], dtype=np.int32)
    out = oracle.prefill_chunk_attention(q, kc, vc, tables, cu, np.array(ctx), 0.0, "f32")
    v = lv[0][:, 0].astype(np.float64)
    for i in range(chunk):
        np.testing.assert_allclose(out[i, 0], v[:c0 + i + 1].mean(axis=0), atol=1e-12)


def test_prefill_last_row_equals_decode():
    """The chunk's last query sees the whole context, exactly like a decode query."""
    ctx = [37, 64]
    chunks = [6, 3]
    tables, lk, lv, kc, vc = _problem(ctx, 8, 2, 64, 16, "bf16", 27)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = _rand((int(cu[-1]), 8, 64), "bf16", 28)
    pre = oracle.prefill_chunk_attention(q, kc, vc, tables, cu, np.array(ctx), 0.125, "bf16")
    last = q[cu[1:] - 1]
    dec = oracle.decode_attention(last, kc, vc, tables, np.array(ctx), 0.125, "bf16")
    np.testing.assert_allclose(pre[cu[1:] - 1], dec, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------------
# slot mapping, cache write, block copy
# ----------------------------------------------------------------------------------

def test_slot_mapping_identity_tables():
    """With table row b = b*W .. b*W+W-1 (a contiguous layout) the slot of position pos is
    (b*W)*bs + pos."""
    bs, width = 16, 8
    ctx = np.array([1, 16, 17, 100], dtype=np.int32)
    ql = np.array([1, 3, 17, 1], dtype=np.int32)
    tables = (np.arange(4)[:, None] * width + np.arange(width)[None, :]).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    slots = oracle.slot_mapping(tables, cu, ctx, bs)
    expect = []
    for b in range(4):
        for pos in range(ctx[b] - ql[b], ctx[b]):
            expect.append(b * width * bs + pos)
    assert slots.tolist() == expect


def test_write_then_walk_round_trip():
    """Writing new tokens through the slot mapping and then walking the table returns them
    as the last positions of each context."""
    step = W.decode_step("t", W.Shape(4, 2, 64, 16, "bf16"), [1, 15, 16, 17, 40], seed=5)
    b = step.decode
    vals = {k: W.to_numpy(v) for k, v in W.make_values(step).items()}
    slots = oracle.slot_mapping(b.block_tables, b.cu_q_lens, b.context_lens, 16)
    kc, vc = vals["k_cache"].copy(), vals["v_cache"].copy()
    oracle.reshape_and_cache(vals["k_new_decode"], vals["v_new_decode"], kc, vc, slots)
    for i in range(b.num_seqs):
        ctx = int(b.context_lens[i])
        k = oracle.gather_context(kc, b.block_tables[i], ctx)
        v = oracle.gather_context(vc, b.block_tables[i], ctx)
        assert np.array_equal(k[-1], vals["k_new_decode"][i])
        assert np.array_equal(v[-1], vals["v_new_decode"][i])
        # earlier positions untouched
        k0 = oracle.gather_context(vals["k_cache"], b.block_tables[i], ctx)
        assert np.array_equal(k[:-1], k0[:-1])
    # exactly B slots changed in the pool
    changed = np.argwhere((kc != vals["k_cache"]).any(axis=(1, 3)))
    assert len({(int(x), int(y)) for x, y in changed}) <= b.num_seqs * 2


def test_negative_slot_is_skipped():
    kc = np.zeros((2, 1, 4, 8), dtype=np.float32)
    vc = np.zeros_like(kc)
    kn = np.ones((2, 1, 8), dtype=np.float32)
    oracle.reshape_and_cache(kn, kn, kc, vc, np.array([-1, 5]))
    assert kc.sum() == 8 and kc[1, 0, 1].sum() == 8


def test_copy_blocks_bits():
    kc = _rand((6, 2, 16, 64), "bf16", 30)
    vc = _rand((6, 2, 16, 64), "bf16", 31)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 4], [1, 5], [2, 0]], dtype=np.int32)
    oracle.copy_blocks([kc, vc], pairs)
    for src, dst in pairs:
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
    for blk in (1, 2, 3):
        assert np.array_equal(kc[blk], k0[blk]) and np.array_equal(vc[blk], v0[blk])


def test_swap_blocks_round_trip_and_fancy_index():
    """Swap-out then swap-in of the same blocks restores the pool; a swap equals numpy's
    fancy-indexed assignment; blocks not named keep their bits."""
    dev = [_rand((8, 2, 16, 64), "bf16", 40 + i) for i in range(4)]  # K, V of two layers
    host = [np.zeros((5, 2, 16, 64), dtype=np.uint16) for _ in range(4)]
    orig = [d.copy() for d in dev]
    out = np.array([[6, 0], [1, 3], [2, 4]], dtype=np.int32)  # (device, host)
    oracle.swap_blocks(dev, host, out)
    for d, h in zip(orig, host):
        ref = np.zeros_like(h)
        ref[out[:, 1]] = d[out[:, 0]]
        assert np.array_equal(h, ref)
    for d in dev:  # the device blocks are reused by someone else meanwhile
        d[[6, 1, 2]] = 0
    back = np.array([[0, 7], [3, 1], [4, 5]], dtype=np.int32)  # (host, device)
    oracle.swap_blocks(host, dev, back)
    for d, o in zip(dev, orig):
        assert np.array_equal(d[7], o[6]) and np.array_equal(d[1], o[1])
        assert np.array_equal(d[5], o[2]) and np.array_equal(d[0], o[0])


def test_widen_bf16_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F], dtype=np.uint16)
    got = oracle.widen(bits, "bf16")
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0 + 2.0 ** -7
    assert got[3] == 0.0 and np.signbit(got[4]) and got[5] == (2 - 2.0 ** -7) * 2.0 ** 127
