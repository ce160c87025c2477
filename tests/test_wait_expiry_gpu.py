"""The failure path of the bounded waits, on the GPU, without a fault.

Every spin on an mbarrier in the kernels gives up after one second, records a
code in the device error word and lets the kernel return.
``sa_check_wait_expiry`` runs one such wait on a barrier that nothing
arrives on; the host must read the code, and the context must stay usable.
"""
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    import torch
    import attention_head_sinks_gb300 as sa
    from attention_head_sinks_gb300 import workloads as W
    from oracle import sa_oracle as O
    from tests.gpu_util import compare, dev
    assert sa.sa_device_error() == 0
    t0 = time.perf_counter()
    sa.sa_check_wait_expiry()
    code = sa.sa_device_error()        # synchronises, reads, clears
    dt = time.perf_counter() - t0
    assert code == 32, code
    assert 0.9 <= dt < 30.0, dt
    assert sa.sa_device_error() == 0   # cleared
    # a normal call afterwards runs and matches the oracle
    c = W.tiny_window(W.SINK_KEY0_BIAS)
    out, lse = sa.sa_varlen_window_fwd(dev(c.q), dev(c.k), dev(c.v), dev(c.cu_seqlens),
                                       c.window_left, c.window_right, dev(c.sinks), c.mode,
                                       c.scale)
    torch.cuda.synchronize()
    ro, rl, _ = O.window_fwd(c.q, c.k, c.v, c.cu_seqlens, c.window_left, c.window_right,
                             c.sinks, c.mode, c.scale)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= 3e-3 and dl <= 1e-4
    assert sa.sa_device_error() == 0
