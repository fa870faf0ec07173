"""The C-ABI library builds, loads, exports what include/*.h declare, and rejects bad
arguments on the host before anything reaches a GPU.

Every call below fails validation, so no kernel is launched and no device memory is
touched; the pointers passed are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))

FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_53_gb300 import build
    path = build.build()
    import paged_kv_cache_53_gb300 as pa
    return pa.lib(path)


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk", "pa_copy_blocks",
               "pa_slot_mapping"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.pa_version() >= 100


def _err(lib):
    return lib.pa_last_error_string().decode()


def _decode(lib, **kw):
    a = dict(out=FAKE, out_dtype=2, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, maxblk=8, ctx=FAKE,
             max_ctx=128, B=4, Hq=32, Hkv=8, D=128, BS=16, NB=64, scale=0.1, dt=2, ws=FAKE,
             ws_bytes=1 << 30)
    a.update(kw)
    return lib.pa_decode(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["bt"], a["maxblk"],
                         a["ctx"], a["max_ctx"], a["B"], a["Hq"], a["Hkv"], a["D"], a["BS"],
                         a["NB"], a["scale"], a["dt"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code,needle", [
    (dict(D=96), 2, "head_dim"),
    (dict(BS=8), 2, "block_size"),
    (dict(Hq=30), 1, "multiple"),
    (dict(Hq=256, Hkv=8), 2, "group"),
    (dict(dt=7), 1, "dtype"),
    (dict(out_dtype=1), 1, "out_dtype"),
    (dict(q=None), 1, "null"),
    (dict(k=FAKE + 4), 1, "aligned"),
    (dict(ws_bytes=16), 3, "workspace"),
    (dict(maxblk=0), 1, "max_blocks"),
    (dict(NB=0), 1, "positive"),
    (dict(scale=float("nan")), 1, "NaN"),
    (dict(NB=1 << 27, Hkv=8, BS=32), 1, "2^31"),
])
def test_decode_rejects_bad_arguments(lib, kw, code, needle):
    assert _decode(lib, **kw) == code
    assert needle in _err(lib)


def test_zero_sequences_is_a_no_op(lib):
    assert _decode(lib, B=0, out=None, q=None) == 0


def _decode_append(lib, **kw):
    a = dict(out=FAKE, out_dtype=2, q=FAKE, kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, slots=None,
             bt=FAKE, maxblk=8, ctx=FAKE, max_ctx=128, B=4, Hq=32, Hkv=8, D=128, BS=16, NB=64,
             scale=0.1, dt=2, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.pa_decode_append(a["out"], a["out_dtype"], a["q"], a["kn"], a["vn"], a["k"],
                                a["v"], a["slots"], a["bt"], a["maxblk"], a["ctx"], a["max_ctx"],
                                a["B"], a["Hq"], a["Hkv"], a["D"], a["BS"], a["NB"], a["scale"],
                                a["dt"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code,needle", [
    (dict(kn=None), 1, "null"),
    (dict(vn=FAKE + 8), 1, "aligned"),
    (dict(q=None), 1, "null"),
    (dict(D=96), 2, "head_dim"),
    (dict(ws_bytes=16), 3, "workspace"),
    (dict(Hq=30), 1, "multiple"),
])
def test_decode_append_rejects_bad_arguments(lib, kw, code, needle):
    assert _decode_append(lib, **kw) == code
    assert "pa_decode_append" in _err(lib) and needle in _err(lib)


def test_decode_append_zero_sequences_is_a_no_op(lib):
    assert _decode_append(lib, B=0, out=None, q=None, kn=None, vn=None) == 0


def test_workspace_bytes_grow_with_context(lib):
    f = lib.pa_decode_workspace_bytes
    small = f(256, 32, 8, 128, 8192, 16)
    big = f(256, 32, 8, 128, 131072, 16)
    assert 0 < small < big
    assert f(0, 32, 8, 128, 10, 16) == 0


def test_prefill_rejects_bad_arguments(lib):
    args = [FAKE, 2, FAKE, FAKE, FAKE, FAKE, 8, FAKE, FAKE, 2, 16, 8, 128, 32, 8, 128, 16, 64,
            0.1, 0, None, 0, None]  # dtype fp32
    assert lib.pa_prefill_chunk(*args) == 2 and "fp32" in _err(lib)
    args[19] = 2   # bf16
    args[13] = 30  # 30 query heads over 8 KV heads
    assert lib.pa_prefill_chunk(*args) == 1


def test_prefill_with_nothing_to_do_is_a_no_op(lib):
    """No sequences, or no new tokens: nothing is launched (and no device is touched)."""
    base = [None, 2, None, None, None, None, 8, None, None, 0, 16, 8, 128, 32, 8, 128, 16, 64,
            0.1, 2, None, 0, None]
    assert lib.pa_prefill_chunk(*base) == 0          # num_seqs = 0
    no_tokens = list(base)
    no_tokens[9], no_tokens[10] = 4, 0               # 4 sequences, 0 new tokens
    assert lib.pa_prefill_chunk(*no_tokens) == 0


def test_cache_ops_reject_bad_arguments(lib):
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 100, 16, 64, 2, None) == 2
    assert lib.pa_reshape_and_cache(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, 8, 128, 16, 64, 2,
                                    None) == 1
    arr = (ctypes.c_void_p * 1)(FAKE)
    assert lib.pa_copy_blocks(arr, arr, 300, FAKE, 4, 8, 128, 16, 64, 2, None) == 2
    assert lib.pa_slot_mapping(FAKE, None, 8, FAKE, FAKE, 4, 4, 16, 64, None) == 1
    assert lib.pa_slot_mapping(None, None, 8, None, None, 4, 0, 16, 64, None) == 0


def test_get_status_without_output_pointer(lib):
    assert lib.pa_get_status(None) == 1


@pytest.mark.parametrize("us", [0, -5, 2_000_001])
def test_selftest_wait_rejects_timeouts_out_of_range(lib, us):
    # checked before any device is touched
    assert lib.pa_selftest_wait_timeout(us, None) == 1
    assert b"timeout_us" in lib.pa_last_error_string()


def _shared(lib, **kw):
    a = dict(out=FAKE, out_dtype=2, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, maxblk=64, ctx=FAKE,
             max_ctx=1024, B=4, Hq=32, Hkv=8, D=128, BS=16, NB=64, pb=FAKE, plen=512, sh=FAKE,
             nsh=3, scale=0.1, dt=2, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.pa_decode_shared_prefix(
        a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["bt"], a["maxblk"], a["ctx"],
        a["max_ctx"], a["B"], a["Hq"], a["Hkv"], a["D"], a["BS"], a["NB"], a["pb"], a["plen"],
        a["sh"], a["nsh"], a["scale"], a["dt"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code,needle", [
    (dict(plen=500), 1, "multiple of the block size"),
    (dict(plen=2048), 1, "max_ctx"),
    (dict(dt=0, out_dtype=0), 2, "fp16/bf16"),
    (dict(sh=None), 1, "null"),
    (dict(pb=None), 1, "null"),
    (dict(nsh=-1), 1, "negative"),
    (dict(ws_bytes=1 << 20), 3, "workspace"),
    (dict(D=96), 2, "head_dim"),
])
def test_shared_prefix_rejects_bad_arguments(lib, kw, code, needle):
    assert _shared(lib, **kw) == code
    assert needle in _err(lib)


def test_shared_prefix_workspace_bytes(lib):
    f = lib.pa_decode_shared_prefix_workspace_bytes
    plain = lib.pa_decode_workspace_bytes(160, 32, 8, 128, 2560, 16)
    assert f(160, 32, 8, 128, 2560, 16, 0, 2048) == plain  # no sharers: the plain layout
    assert f(160, 32, 8, 128, 2560, 16, 128, 0) == plain
    with_prefix = f(160, 32, 8, 128, 2560, 16, 128, 2048)
    # every sharer keeps one fp32 partial row per query head and prefix split
    assert with_prefix >= plain + 128 * 32 * 128 * 4
    assert f(160, 30, 8, 128, 2560, 16, 128, 2048) == 0


def _mixed_batches():
    import paged_kv_cache_53_gb300 as pa
    dec = pa._DecodeBatch(FAKE, 2, FAKE, FAKE, FAKE, None, FAKE, 8, FAKE, 128, 4, FAKE, 1 << 30)
    pre = pa._PrefillBatch(FAKE, 2, FAKE, FAKE, FAKE, None, FAKE, 8, FAKE, FAKE, 64, 512, 2, 100,
                           FAKE, 1 << 30)
    return dec, pre


def _mixed(lib, dec, pre):
    return lib.pa_mixed_step(ctypes.byref(dec) if dec is not None else None,
                             ctypes.byref(pre) if pre is not None else None, FAKE, FAKE, 32, 8,
                             128, 16, 64, 0.1, 2, None)


def test_mixed_step_with_nothing_to_do(lib):
    dec, pre = _mixed_batches()
    dec.num_seqs = 0
    pre.num_seqs = pre.num_tokens = 0
    assert _mixed(lib, None, None) == 0
    assert _mixed(lib, dec, pre) == 0


@pytest.mark.parametrize("which,field,value,needle", [
    ("dec", "k_new", None, "decode batch: null"),
    ("dec", "v_new", FAKE + 4, "decode batch: K/V pointers"),
    ("pre", "k_new", None, "prefill batch: null"),
    ("pre", "v_new", FAKE + 2, "prefill batch: K/V pointers"),
])
def test_mixed_step_rejects_bad_batches(lib, which, field, value, needle):
    dec, pre = _mixed_batches()
    setattr(dec if which == "dec" else pre, field, value)
    assert _mixed(lib, dec, pre) == 1
    assert "pa_mixed_step" in _err(lib) and needle in _err(lib)


def test_testing_partition_workspace(lib):
    f = lib.pa_testing_decode_workspace_bytes
    assert f(4, 32, 8, 128, 4099, 16, 0) == 0
    assert f(4, 32, 8, 128, 4099, 16, 129) == 0
    sizes = [f(4, 32, 8, 128, 4099, 16, pb) for pb in (1, 2, 7, 64, 128)]
    assert all(a >= b > 0 for a, b in zip(sizes, sizes[1:]))
    # one block per partition: 257 partials per sequence, 32 query heads of 128 fp32 each
    assert sizes[0] >= 4 * 257 * 32 * 128 * 4


@pytest.mark.parametrize("pb", [0, -1, 129])
def test_testing_partitions_rejects_sizes(lib, pb):
    rc = lib.pa_testing_decode_partitions(FAKE, 2, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 128, 4, 32,
                                          8, 128, 16, 64, 0.1, 2, pb, FAKE, 1 << 30, None)
    assert rc == 1 and "part_blocks" in _err(lib)


def test_testing_partitions_checks_workspace(lib):
    rc = lib.pa_testing_decode_partitions(FAKE, 2, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 128, 4, 32,
                                          8, 128, 16, 64, 0.1, 2, 1, FAKE, 1024, None)
    assert rc == 3 and "workspace" in _err(lib)


def test_stream_status_word_must_be_aligned(lib):
    import torch
    rc = lib.pa_set_stream_status(None, FAKE + 2)
    # without a device the call cannot name one (PA_ERR_CUDA); with one, the word is checked
    assert rc == (1 if torch.cuda.is_available() else 4)


def test_release_with_nothing_to_release(lib):
    assert lib.pa_release_thread_resources() == 0
