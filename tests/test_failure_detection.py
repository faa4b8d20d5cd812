"""Failure detection without a GPU fault.

Every wait in the library's kernels (tensor-core commits, TMA copies) polls an mbarrier a
bounded number of times; when the bound runs out the kernel records a code in the device
error word and returns instead of hanging.  The diagnostic entry point runs that exact
wait on a barrier nothing arrives at, so the timeout path is exercised on demand: the
code must reach the host, the word must clear on read, and the context must stay usable
for ordinary work afterwards.
"""
import ctypes

import numpy as np
import pytest

WAIT_TIMEOUT = 1   # KDA_DEVICE_ERR_WAIT_TIMEOUT in include/kda.h


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    return kda.library()


def test_selftest_rejects_bad_poll_limits_on_the_host(lib):
    assert lib.kda_selftest_bounded_wait(ctypes.c_uint(0), None) == 1
    assert lib.kda_selftest_bounded_wait(ctypes.c_uint((1 << 24) + 1), None) == 1
    assert b"poll_limit" in lib.kda_last_error()


def test_header_documents_the_timeout_code():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")).read()
    m = re.search(r"#define\s+KDA_DEVICE_ERR_WAIT_TIMEOUT\s+(\d+)u", hdr)
    assert m and int(m.group(1)) == WAIT_TIMEOUT


@pytest.mark.gpu
def test_bounded_wait_reports_and_the_context_survives():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    import kda_synth as ks
    from kda_synth.device import to_device, to_host_f64

    assert kda.device_error() == 0
    for limit in (1, 1000):
        kda.selftest_bounded_wait(limit)
        torch.cuda.synchronize()
        assert kda.device_error() == WAIT_TIMEOUT
        assert kda.device_error() == 0           # read clears the word

    # on a side stream as well
    s = torch.cuda.Stream()
    kda.selftest_bounded_wait(64, stream=s)
    s.synchronize()
    assert kda.device_error() == WAIT_TIMEOUT

    # ordinary work afterwards: one decode step of a tiny batch, run twice from the same
    # state, gives identical bits and raises nothing
    w = ks.Workload("after", "decode", 5301, H=2, lengths=[1] * 3, init_state_std=0.02)
    xs = [ks.fill(w.seed, tid, ks.NORMAL, (w.N, w.H * w.d), "bf16") for tid in (1, 2, 3)]
    g = ks.fill(w.seed, ks.TID_G, w.g_kind, (w.N, w.H, w.d), "f32")
    b = ks.fill(w.seed, ks.TID_BETA, ks.SIGMOID, (w.N, w.H), "f32")
    cw, st, cs = w.conv_w(), w.init_state(), w.conv_state()
    outs = []
    for _ in range(2):
        st_d, cs_d = to_device(st), to_device(cs)
        o = kda.kda_recurrent_step(*(to_device(x) for x in xs), to_device(cw), to_device(g), to_device(b),
                                   st_d, cs_d)
        torch.cuda.synchronize()
        outs.append((to_host_f64(o), to_host_f64(st_d)))
    assert np.isfinite(outs[0][0]).all()
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert kda.device_error() == 0
