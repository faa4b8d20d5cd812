"""kda_chunk_fwd_noalloc: the prefill on the library's static 64 MiB device scratch.

It has no counterpart in the sources; it is the workspace path with the workspace taken from
a scratch array in the library's device image.  CPU tests: the symbol is exported and sizes
whose smallest range does not fit are refused before anything is enqueued.  GPU tests: the
result is bit-identical to kda_chunk_fwd with a caller workspace, also when the static
scratch forces several ranges of chunks (8192 tokens x 96 heads: the workspace path runs the
128 chunk rows as one range, the scratch path in ranges of 6 chunk rows one after the other on
the caller's stream), and on two calls in a row.
"""
import ctypes

import numpy as np
import pytest

import kda_synth as ks

SCRATCH = 64 << 20
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as m
    return m


def _call(lib, **over):
    a = dict(q=P(4096), k=P(4096), v=P(4096), g=P(4096), beta=P(4096), init=None, cu=None, N=1, T=64, H=2,
             dk=128, dv=128, scale=1.0, chunk=64, dtype=1, gate=None, o=P(4096), fs=None, stream=None)
    a.update(over)
    return lib.kda_chunk_fwd_noalloc(a["q"], a["k"], a["v"], a["g"], a["beta"], a["init"], a["cu"], a["N"], a["T"],
                                     a["H"], a["dk"], a["dv"], a["scale"], a["chunk"], a["dtype"], a["gate"], a["o"],
                                     a["fs"], a["stream"])


def test_exported_and_declared(kda):
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")).read()
    assert re.search(r"KDA_API\s+kda_status\s+kda_chunk_fwd_noalloc\s*\(", hdr)
    assert hasattr(kda.library(), "kda_chunk_fwd_noalloc")


def test_oversize_is_refused_on_the_host(kda):
    lib = kda.library()
    UNSUPPORTED, INVALID = 2, 1
    # one chunk row needs 2 x 64 KiB of carried state and 82,432 bytes of operands per head (+ 1 KiB)
    least = kda.kda_chunk_fwd_workspace_size(1, 64, 315, have_cu_seqlens=False)[1]
    assert least > SCRATCH
    assert _call(lib, H=315) == UNSUPPORTED
    assert b"static scratch" in lib.kda_last_error()
    assert kda.kda_chunk_fwd_workspace_size(1, 64, 314, have_cu_seqlens=False)[1] <= SCRATCH
    assert _call(lib, N=0) == INVALID
    assert _call(lib, q=None) == INVALID
    assert _call(lib, dtype=7) == INVALID


@pytest.mark.gpu
@pytest.mark.parametrize("lengths,H", [([130, 1, 0, 257, 5], 3), ([4096], 96), ([8192], 96)])
def test_noalloc_equals_workspace_path(kda, lengths, H):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_synth.device import to_device
    w = ks.Workload("na", "prefill", 108, H=H, lengths=lengths, init_state_std=0.02)
    args = [to_device(x) for x in (w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta(), w.init_state())]
    cu = to_device(w.cu_seqlens()) if w.N > 1 else None
    o1, f1 = kda.kda_chunk_fwd(*args, cu)
    o2, f2 = kda.kda_chunk_fwd_noalloc(*args, cu)
    torch.cuda.synchronize()
    full = kda.kda_chunk_fwd_workspace_size(w.N, w.T, H, have_cu_seqlens=cu is not None)[0]
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    assert np.isfinite(o2.float().cpu().numpy()).all()
    if H == 96:
        assert full > SCRATCH   # 4096 tokens x 96 heads need several ranges in the static scratch
    # the same call twice in a row: the scratch keeps the last call's contents, which must not matter
    o3, f3 = kda.kda_chunk_fwd_noalloc(*args, cu)
    torch.cuda.synchronize()
    assert torch.equal(o3, o1) and torch.equal(f3, f1)
    assert kda.device_error() == 0
