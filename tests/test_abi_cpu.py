"""Host-side checks of the C ABI: the library builds and loads without a GPU,
exports every function ``include/sa.h`` declares, and rejects bad arguments
with a status and a message before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attention_head_sinks_gb300 import build
    build.build()
    import attention_head_sinks_gb300 as sa
    return sa.lib()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"SA_API\s+[\w\s\*]+?\b(sa_\w+)\s*\(", src))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"sa_varlen_window_fwd", "sa_last_error", "sa_device_error",
            "sa_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    from attention_head_sinks_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_version(lib):
    assert lib.sa_version() == 1


def _window_call(lib, **kw):
    a = dict(q=16, k=16, v=16, cu=16, num_seqs=1, T=128, hq=4, hkv=4, d=80,
             wl=64, wr=64, sinks=16, mode=1, scale=0.1, out=16, lse=16)
    a.update(kw)
    return lib.sa_varlen_window_fwd(
        a["q"], a["k"], a["v"], a["cu"], a["num_seqs"], a["T"], a["hq"], a["hkv"],
        a["d"], a["wl"], a["wr"], a["sinks"], a["mode"], a["scale"], a["out"],
        a["lse"], None)


@pytest.mark.parametrize("kw,needle", [
    (dict(q=None), "NULL"),
    (dict(out=None), "NULL"),
    (dict(mode=7), "sink_mode"),
    (dict(sinks=None, mode=1), "sinks is NULL"),
    (dict(num_seqs=0), "num_seqs"),
    (dict(T=-1), "total_tokens"),
    (dict(hq=6, hkv=4), "multiple"),
    (dict(wl=-1), "window"),
    (dict(scale=0.0), "softmax_scale"),
    (dict(scale=float("inf")), "softmax_scale"),
    (dict(q=18), "misaligned"),
])
def test_window_rejects_bad_arguments(lib, kw, needle):
    st = _window_call(lib, **kw)
    assert st == 1  # SA_ERR_INVALID_ARG
    assert needle in lib.sa_last_error().decode()


def test_window_empty_problem_is_a_no_op(lib):
    assert _window_call(lib, T=0) == 0


def test_python_binding_rejects_cpu_tensors():
    import torch
    import attention_head_sinks_gb300 as sa
    q = torch.zeros(4, 2, 80, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError):
        sa.sa_varlen_window_fwd(q, q, q, cu, 8, 8, None, 0, 0.1)


def _index_call(lib, **kw):
    a = dict(q=16, kv=16, nkv=1000, dqk=576, dv=512, idx=16, topk=2048, nq=64,
             hq=128, sinks=16, mode=2, scale=0.04, out=16, lse=16, ws=16,
             ws_bytes=1 << 40)
    a.update(kw)
    return lib.sa_sparse_index_fwd(
        a["q"], a["kv"], a["nkv"], a["dqk"], a["dv"], a["idx"], a["topk"], a["nq"],
        a["hq"], a["sinks"], a["mode"], a["scale"], a["out"], a["lse"], a["ws"],
        a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(q=None), 1, "NULL"),
    (dict(mode=5), 1, "sink_mode"),
    (dict(sinks=None), 1, "sinks is NULL"),
    (dict(nkv=0), 1, "bad sizes"),
    (dict(dv=600), 1, "bad sizes"),
    (dict(kv=24), 1, "misaligned"),
    (dict(mode=1), 2, "KEY0_BIAS"),
    (dict(nkv=1 << 31), 2, "num_kv"),
    (dict(topk=9000), 2, "topk"),
    (dict(ws=None), 4, "workspace"),
    (dict(ws_bytes=1000), 4, "workspace"),
])
def test_sparse_index_rejects_bad_arguments(lib, kw, status, needle):
    assert _index_call(lib, **kw) == status
    assert needle in lib.sa_last_error().decode()


def _fp8_call(lib, **kw):
    a = dict(q=16, kv=16, ks=16, nkv=1000, dqk=576, dv=512, idx=16, topk=2048, nq=64,
             hq=128, sinks=16, mode=2, scale=0.04, out=16, lse=16, ws=16,
             ws_bytes=1 << 40)
    a.update(kw)
    return lib.sa_sparse_index_fwd_fp8(
        a["q"], a["kv"], a["ks"], a["nkv"], a["dqk"], a["dv"], a["idx"], a["topk"],
        a["nq"], a["hq"], a["sinks"], a["mode"], a["scale"], a["out"], a["lse"], a["ws"],
        a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(ks=None), 1, "NULL"),
    (dict(ks=18), 1, "misaligned"),
    (dict(kv=8), 1, "misaligned"),
    (dict(mode=1), 2, "KEY0_BIAS"),
    (dict(topk=9000), 2, "topk"),
    (dict(ws_bytes=1000), 4, "workspace"),
])
def test_sparse_index_fp8_rejects_bad_arguments(lib, kw, status, needle):
    assert _fp8_call(lib, **kw) == status
    msg = lib.sa_last_error().decode()
    assert needle in msg and msg.startswith("sa_sparse_index_fwd_fp8")


def test_sparse_index_fp8_empty_batch_is_a_no_op(lib):
    assert _fp8_call(lib, nq=0) == 0


def _a256(x):
    return (x + 255) // 256 * 256


def test_sparse_index_workspace_size(lib):
    # compacted index rows (int32 [Nq, topk]), valid count and finished-item
    # counter per query, then, with more than one 256-key item per query, per
    # (query, item, head; head stride rounded to 32): (m, l) fp32, one int8
    # scale exponent per 32 V columns, and the O partial as 512 fp16 values
    head = _a256(64 * 2048 * 4) + 2 * _a256(64 * 4)
    assert lib.sa_sparse_index_workspace_size(64, 128, 512, 2048) == \
        head + _a256(64 * 8 * 2 * 128 * 4) + _a256(64 * 8 * 16 * 128) + \
        64 * 8 * 512 * 128 * 2
    assert lib.sa_sparse_index_workspace_size(3, 40, 512, 300) == \
        _a256(3 * 300 * 4) + 2 * _a256(3 * 4) + _a256(3 * 2 * 2 * 64 * 4) + \
        _a256(3 * 2 * 16 * 64) + 3 * 2 * 512 * 64 * 2
    assert lib.sa_sparse_index_workspace_size(64, 128, 512, 256) == \
        _a256(64 * 256 * 4) + 2 * _a256(64 * 4)
    assert lib.sa_sparse_index_workspace_size(0, 128, 512, 2048) == 0
    assert lib.sa_sparse_index_workspace_size(64, 128, 512, 0) == 0


def test_sparse_index_empty_batch_is_a_no_op(lib):
    assert _index_call(lib, nq=0) == 0


def _noalloc_call(lib, **kw):
    a = dict(q=16, kv=16, nkv=1000, dqk=576, dv=512, idx=16, topk=2048, nq=4,
             hq=128, sinks=16, mode=2, scale=0.04, out=16, lse=16)
    a.update(kw)
    return lib.sa_sparse_index_fwd_noalloc(
        a["q"], a["kv"], a["nkv"], a["dqk"], a["dv"], a["idx"], a["topk"], a["nq"],
        a["hq"], a["sinks"], a["mode"], a["scale"], a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(q=None), 1, "NULL"),
    (dict(mode=5), 1, "sink_mode"),
    (dict(sinks=None), 1, "sinks is NULL"),
    (dict(nkv=0), 1, "bad sizes"),
    (dict(kv=24), 1, "misaligned"),
    (dict(mode=1), 2, "KEY0_BIAS"),
    (dict(nkv=1 << 31), 2, "num_kv"),
    # argument errors come before the scratch-size check, even for sizes
    # whose scratch would exceed the fixed array
    (dict(topk=9000), 2, "topk 9000"),
    (dict(topk=9000, nq=64), 2, "topk 9000"),
    (dict(dv=256), 2, "dqk 576 / dv 256"),
    # 64 queries x 128 heads x 8 items of partials: beyond the fixed 64 MiB
    (dict(nq=64), 2, "64 MiB"),
])
def test_sparse_index_noalloc_rejects_bad_arguments(lib, kw, status, needle):
    assert _noalloc_call(lib, **kw) == status
    msg = lib.sa_last_error().decode()
    assert needle in msg and msg.startswith("sa_sparse_index_fwd_noalloc:"), msg


def test_sparse_index_noalloc_empty_batch_is_a_no_op(lib):
    assert _noalloc_call(lib, nq=0) == 0


def _block_call(lib, **kw):
    a = dict(q=16, k=16, v=16, batch=2, S=8192, hq=32, hkv=4, d=128, tab=16, topk=16,
             bs=64, cu=16, ndocs=6, sinks=16, mode=2, scale=0.08, out=16, lse=16)
    a.update(kw)
    return lib.sa_block_sparse_fwd(
        a["q"], a["k"], a["v"], a["batch"], a["S"], a["hq"], a["hkv"], a["d"], a["tab"],
        a["topk"], a["bs"], a["cu"], a["ndocs"], a["sinks"], a["mode"], a["scale"],
        a["out"], a["lse"], None, 0, None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(q=None), 1, "NULL"),
    (dict(tab=None), 1, "NULL"),
    (dict(mode=3), 1, "sink_mode"),
    (dict(sinks=None), 1, "sinks is NULL"),
    (dict(ndocs=0), 1, "bad sizes"),
    (dict(bs=0), 1, "bad sizes"),
    (dict(hq=30), 1, "multiple"),
    (dict(batch=1 << 20), 1, "2^31"),
    (dict(out=8), 1, "misaligned"),
])
def test_block_sparse_rejects_bad_arguments(lib, kw, status, needle):
    assert _block_call(lib, **kw) == status
    assert needle in lib.sa_last_error().decode()


def test_block_sparse_empty_batch_is_a_no_op(lib):
    assert _block_call(lib, batch=0) == 0


def _merge_call(lib, **kw):
    a = dict(oa=16, la=16, ob=16, lb=16, T=100, H=4, D=80, sinks=16, mode=2, out=16,
             lse=4096)
    a.update(kw)
    return lib.sa_merge_attn_states(a["oa"], a["la"], a["ob"], a["lb"], a["T"], a["H"],
                                    a["D"], a["sinks"], a["mode"], a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(oa=None), 1, "NULL"),
    (dict(mode=7), 1, "sink_mode"),
    (dict(sinks=None), 1, "sinks is NULL"),
    (dict(H=0), 1, "bad sizes"),
    (dict(out=24), 1, "misaligned"),
    (dict(lse=16), 1, "overlaps"),
    (dict(mode=1), 2, "KEY0_BIAS"),
    (dict(D=12), 2, "head_dim"),
])
def test_merge_rejects_bad_arguments(lib, kw, status, needle):
    assert _merge_call(lib, **kw) == status
    assert needle in lib.sa_last_error().decode()


def test_merge_empty_is_a_no_op(lib):
    assert _merge_call(lib, T=0) == 0


def _select_call(lib, **kw):
    a = dict(q=16, k=16, batch=2, S=8192, hi=4, di=128, bs=64, topk=16, tab=16)
    a.update(kw)
    return lib.sa_block_select(a["q"], a["k"], a["batch"], a["S"], a["hi"], a["di"], a["bs"],
                               a["topk"], a["tab"], None)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(q=None), 1, "NULL"),
    (dict(tab=None), 1, "NULL"),
    (dict(hi=0), 1, "bad sizes"),
    (dict(topk=0), 1, "bad sizes"),
    (dict(batch=1 << 20), 1, "2^31"),
    (dict(k=24), 1, "misaligned"),
])
def test_block_select_rejects_bad_arguments(lib, kw, status, needle):
    assert _select_call(lib, **kw) == status
    assert needle in lib.sa_last_error().decode()


def test_block_select_empty_is_a_no_op(lib):
    assert _select_call(lib, batch=0) == 0


def test_block_index_heads_must_divide_kv_heads(lib):
    st = lib.sa_block_sparse_fwd_index_heads(16, 16, 16, 2, 8192, 32, 4, 128, 16, 3, 16, 64,
                                             16, 6, 16, 2, 0.08, 16, 16, None)
    assert st == 1 and "divide" in lib.sa_last_error().decode()
