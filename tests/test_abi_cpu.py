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
