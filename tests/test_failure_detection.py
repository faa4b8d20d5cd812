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
GATE_RANGE = 2     # KDA_DEVICE_ERR_GATE_RANGE
BETA_RANGE = 4     # KDA_DEVICE_ERR_BETA_RANGE


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


def test_header_documents_the_error_bits():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")).read()
    for name, val in (("WAIT_TIMEOUT", WAIT_TIMEOUT), ("GATE_RANGE", GATE_RANGE), ("BETA_RANGE", BETA_RANGE)):
        m = re.search(r"#define\s+KDA_DEVICE_ERR_%s\s+(\d+)u" % name, hdr)
        assert m and int(m.group(1)) == val, name


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


@pytest.mark.gpu
def test_out_of_range_gates_and_betas_are_reported():
    """The bf16 prefill relies on g in [-5, 0] ("Kimi K3 架构全景", section 02: gate lower bound -5.0)
    and beta in [0, 1]; an input outside them (or not finite) sets its bit of the device error word.
    The values planted here keep every exponent the kernels form finite, so the call completes
    normally; only the report is checked.  In-range inputs, including the bounds themselves,
    raise nothing."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    import kda_synth as ks
    from kda_synth.device import to_device

    w = ks.Workload("range", "prefill", 5302, H=2, lengths=[70, 131])
    q, k, v, g, b = w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta()
    cu = to_device(w.cu_seqlens())
    assert kda.device_error() == 0

    def run(gg, bb):
        kda.kda_chunk_fwd(to_device(q), to_device(k), to_device(v), to_device(gg), to_device(bb), None, cu)
        torch.cuda.synchronize()
        return kda.device_error()

    assert run(g, b) == 0
    edge_g, edge_b = g.copy(), b.copy()
    edge_g[3, 0, :] = -5.0
    edge_g[150, 1, :] = 0.0
    edge_b[5, 0], edge_b[100, 1] = 0.0, 1.0
    assert run(edge_g, edge_b) == 0                       # the bounds themselves are allowed
    for t, h, c, val in ((5, 1, 7, -5.25), (200, 0, 127, 0.5), (69, 1, 0, np.nan), (70, 0, 64, -np.inf)):
        bad = g.copy()
        bad[t, h, c] = val
        assert run(bad, b) == GATE_RANGE, (t, h, c, val)
    for t, h, val in ((0, 0, 1.25), (130, 1, -0.5), (64, 1, np.nan)):
        bad = b.copy()
        bad[t, h] = val
        assert run(g, bad) == BETA_RANGE, (t, h, val)
    bad_g, bad_b = g.copy(), b.copy()
    bad_g[1, 1, 1], bad_b[2, 0] = -6.0, 2.0
    assert run(bad_g, bad_b) == GATE_RANGE | BETA_RANGE   # both bits, one read

    # the bf16 backward checks the same ranges as it reads g and beta
    d_o = to_device(w.qkv("v"))

    def bwd(gg, bb):
        kda.kda_chunk_bwd(to_device(q), to_device(k), to_device(v), to_device(gg), to_device(bb), d_o, cu_seqlens=cu)
        torch.cuda.synchronize()
        return kda.device_error()

    assert bwd(g, b) == 0
    assert bwd(edge_g, edge_b) == 0
    bad = g.copy()
    bad[5, 1, 7] = -5.25
    assert bwd(bad, b) == GATE_RANGE
    bad = g.copy()
    bad[200, 0, 127] = np.nan
    assert bwd(bad, b) == GATE_RANGE
    bad = b.copy()
    bad[130, 1] = -0.5
    assert bwd(g, bad) == BETA_RANGE

    # the decode step checks the same ranges
    wd = ks.Workload("range_dec", "decode", 5303, H=2, lengths=[1] * 3, init_state_std=0.02)
    xs = [to_device(ks.fill(wd.seed, tid, ks.NORMAL, (wd.N, wd.H * wd.d), "bf16")) for tid in (1, 2, 3)]
    gd = ks.fill(wd.seed, ks.TID_G, wd.g_kind, (wd.N, wd.H, wd.d), "f32")
    bd = ks.fill(wd.seed, ks.TID_BETA, ks.SIGMOID, (wd.N, wd.H), "f32")
    cw = to_device(wd.conv_w())

    def step(gg, bb):
        kda.kda_recurrent_step(*xs, cw, to_device(gg), to_device(bb), to_device(wd.init_state()),
                               to_device(wd.conv_state()))
        torch.cuda.synchronize()
        return kda.device_error()

    assert step(gd, bd) == 0
    bad = gd.copy()
    bad[2, 1, 5] = 0.125
    assert step(bad, bd) == GATE_RANGE
    bad = bd.copy()
    bad[1, 0] = -0.01
    assert step(gd, bad) == BETA_RANGE
