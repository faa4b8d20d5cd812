"""The C ABI without a GPU: the library loads, exports every declared entry point and
rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    return kda.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_header_declares_the_three_operations():
    syms = declared_symbols()
    for name in ("kda_shortconv_l2norm", "kda_chunk_fwd", "kda_recurrent_step"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"


def test_status_strings(lib):
    for code in range(5):
        assert lib.kda_status_string(code).startswith(b"KDA_")
    assert lib.kda_version().decode().count(".") == 2


P = ctypes.c_void_p


def _chunk(lib, **over):
    a = dict(q=P(4096), k=P(4096), v=P(4096), g=P(4096), beta=P(4096), init=None, cu=None, N=1, T=64, H=2,
             dk=128, dv=128, scale=1.0, chunk=64, dtype=1, gate=None, o=P(4096), fs=None, ws=P(4096),
             wsb=1 << 30, stream=None)
    a.update(over)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["init"], a["cu"], a["N"], a["T"], a["H"],
                             a["dk"], a["dv"], a["scale"], a["chunk"], a["dtype"], a["gate"], a["o"], a["fs"],
                             a["ws"], a["wsb"], a["stream"])


def _ws(lib, N, T, H, dtype=1, cu=1):
    full, least = ctypes.c_size_t(0), ctypes.c_size_t(0)
    rc = lib.kda_chunk_fwd_workspace_size(N, T, H, 128, 128, 64, dtype, cu, ctypes.byref(full), ctypes.byref(least))
    return rc, full.value, least.value


def test_workspace_size(lib):
    # carried states 2 x H x 64 KiB, chunk offsets rounded to 1 KiB, 82,432 bytes per chunk and head (the
    # chunk operands, the same layout with and without the fused front end)
    hdr = 2 * 96 * 65536 + 1024
    assert _ws(lib, 1, 8192, 96, cu=0) == (0, hdr + 128 * 96 * 82432, hdr + 96 * 82432)
    assert _ws(lib, 1, 8193, 96, cu=0) == (0, hdr + 129 * 96 * 82432, hdr + 96 * 82432)
    # with cu_seqlens the chunk count is bounded by T / 64 + N
    assert _ws(lib, 32, 520949, 96)[1] == hdr + (520949 // 64 + 32) * 96 * 82432
    assert _ws(lib, 300, 1000, 4)[2] == 2 * 4 * 65536 + 2048 + 4 * 82432
    assert _ws(lib, 1, 0, 96, cu=0)[1] == hdr + 96 * 82432
    assert _ws(lib, 1, 256, 4, dtype=0) == (0, 0, 0)      # the fp32 path needs none
    assert _ws(lib, 2, 256, 4, cu=0)[0] == 1               # several sequences need cu_seqlens
    assert _ws(lib, 1, 256, 4, cu=0)[0] == 0


def test_chunk_fwd_rejects_bad_arguments(lib):
    INVALID, UNSUPPORTED = 1, 2
    assert _chunk(lib, q=None) == INVALID
    assert _chunk(lib, o=P(4100)) == INVALID                 # misaligned
    assert _chunk(lib, dk=64) == UNSUPPORTED
    assert _chunk(lib, chunk=32) == UNSUPPORTED
    assert _chunk(lib, N=2) == INVALID                       # several sequences need cu_seqlens
    assert _chunk(lib, N=0) == INVALID
    assert _chunk(lib, T=-1) == INVALID
    assert _chunk(lib, dtype=7) == INVALID
    assert _chunk(lib, scale=float("nan")) == INVALID
    assert b"must" in lib.kda_last_error()
    least = _ws(lib, 1, 64, 2, cu=0)[2]
    assert _chunk(lib, ws=None) == INVALID                   # the bf16 path needs a workspace
    assert _chunk(lib, wsb=least - 1) == INVALID
    assert _chunk(lib, ws=P(4104), wsb=least) == INVALID     # misaligned workspace
    assert _chunk(lib, T=1 << 31) == INVALID                 # tensor-map coordinates are 32-bit


def test_shortconv_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=P(4096), stride=256, w=P(4096), cu=None, N=1, T=5, H=2, d=128, cs_in=None, cs_out=None, eps=1e-6,
                 dt=1, out=P(4096))
        a.update(over)
        return lib.kda_shortconv_l2norm(a["x"], a["x"], a["x"], a["stride"], a["w"], a["cu"], a["N"], a["T"],
                                        a["H"], a["d"], a["cs_in"], a["cs_out"], a["eps"], a["dt"], a["out"],
                                        a["out"], a["out"], None)
    assert call(x=None) == 1
    assert call(stride=200) == 1          # < H*d
    assert call(stride=260) == 1          # not a multiple of 8
    assert call(d=64) == 2
    assert call(eps=-1.0) == 1
    assert call(cs_in=P(4097)) == 1


def test_recurrent_step_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=P(4096), stride=256, p=P(4096), N=4, H=2, dk=128, dv=128)
        a.update(over)
        return lib.kda_recurrent_step(a["x"], a["x"], a["x"], a["stride"], a["p"], a["p"], a["p"], a["p"], a["p"],
                                      a["N"], a["H"], a["dk"], a["dv"], 1.0, 1e-6, a["p"], None)
    assert call(p=None) == 1
    assert call(N=0) == 1
    assert call(dv=96) == 2
    assert call(stride=8) == 1


def test_chunk_fwd_frontend_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=P(4096), stride=256, w=P(4096), cs_in=None, cs_out=None, eps=1e-6, g=P(4096), b=P(4096),
                 init=None, cu=None, N=1, T=64, H=2, d=128, scale=1.0, chunk=64, gate=None, o=P(1 << 32), fs=None,
                 ws=P(4096), wsb=1 << 30)
        a.update(over)
        return lib.kda_chunk_fwd_frontend(a["x"], a["x"], a["x"], a["stride"], a["w"], a["cs_in"], a["cs_out"],
                                          a["eps"], a["g"], a["b"], a["init"], a["cu"], a["N"], a["T"], a["H"],
                                          a["d"], a["scale"], a["chunk"], a["gate"], a["o"], a["fs"], a["ws"],
                                          a["wsb"], None)
    assert call(x=None) == 1
    assert call(stride=200) == 1          # < H*d
    assert call(stride=260) == 1          # not a multiple of 8
    assert call(d=64) == 2
    assert call(chunk=32) == 2
    assert call(eps=-1.0) == 1
    assert call(ws=None) == 1
    assert call(wsb=1024) == 1 and b"workspace" in lib.kda_last_error()
    assert call(N=2) == 1                 # several sequences need cu_seqlens
    # o holds v during the call: sharing memory with an input is refused before anything is enqueued
    assert call(o=P(4096 + 64 * 256), wsb=1024) == 1                   # inside the raw rows (T x stride x 2 bytes)
    assert b"overlap" in lib.kda_last_error()
    assert call(gate=P(1 << 32), wsb=1024) == 1                        # the output gate in place
    assert b"overlap" in lib.kda_last_error()
    assert call(g=P(1 << 33), o=P((1 << 33) + 4096), wsb=1024) == 1    # inside g (T x H x d x 4 bytes)
    assert b"overlap" in lib.kda_last_error()
    assert call(o=P((1 << 32) + 65536), wsb=1024) == 1                 # clear of every input: the next check
    assert b"workspace" in lib.kda_last_error()


def test_segment_summary_and_combine_reject_bad_arguments(lib):
    def summ(**over):
        a = dict(q=None, k=P(4096), v=P(4096), g=P(4096), b=P(4096), cu=None, N=1, T=64, H=2, dk=128, dv=128,
                 chunk=64, E=P(4096), M=P(4096), ws=P(4096), wsb=1 << 30)
        a.update(over)
        return lib.kda_chunk_segment_summary(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"], a["N"], a["T"],
                                             a["H"], a["dk"], a["dv"], a["chunk"], a["E"], a["M"], a["ws"],
                                             a["wsb"], None)
    assert summ(k=None) == 1
    assert summ(E=None, M=None) == 1       # nothing to compute
    assert summ(v=None) == 1               # the end state needs v
    assert summ(M=P(4100)) == 1            # misaligned
    assert summ(dk=64) == 2
    assert summ(chunk=32) == 2
    assert summ(N=2) == 1                  # several sequences need cu_seqlens
    assert summ(ws=None) == 1
    assert summ(wsb=1024) == 1
    assert summ(T=1 << 31) == 1

    def comb(**over):
        a = dict(S=None, M=P(4096), E=P(4096), out=P(4096), count=1)
        a.update(over)
        return lib.kda_state_combine(a["S"], a["M"], a["E"], a["out"], a["count"], None)
    assert comb(M=None) == 1
    assert comb(E=None) == 1
    assert comb(out=None) == 1
    assert comb(S=P(4100)) == 1            # misaligned
    assert comb(count=-1) == 1
    assert comb(count=1 << 31) == 1


def test_chunk_bwd_rejects_bad_arguments(lib):
    def bwd(**over):
        a = dict(q=P(4096), k=P(4096), v=P(4096), g=P(4096), b=P(4096), init=None, cu=None, N=1, T=64, H=2,
                 dk=128, dv=128, scale=1.0, chunk=64, dtype=1, do=P(4096), dfin=None, dq=P(4096), dk_=P(4096),
                 dv_=P(4096), dg=P(4096), db=P(4096), dinit=None, ws=P(4096), wsb=1 << 40)
        a.update(over)
        return lib.kda_chunk_bwd(a["q"], a["k"], a["v"], a["g"], a["b"], a["init"], a["cu"], a["N"], a["T"], a["H"],
                                 a["dk"], a["dv"], a["scale"], a["chunk"], a["dtype"], a["do"], a["dfin"], a["dq"],
                                 a["dk_"], a["dv_"], a["dg"], a["db"], a["dinit"], a["ws"], a["wsb"], None)
    for name in ("q", "k", "v", "g", "b", "do", "dq", "dk_", "dv_", "dg", "db", "ws"):
        assert bwd(**{name: None}) == 1, name
    assert bwd(dfin=P(4100)) == 1          # misaligned
    assert bwd(dinit=P(4100)) == 1
    assert bwd(dk=64) == 2
    assert bwd(chunk=32) == 2
    assert bwd(dtype=7) == 1
    assert bwd(N=2) == 1                   # several sequences need cu_seqlens
    assert bwd(scale=float("nan")) == 1
    assert bwd(wsb=1024) == 1              # workspace too small
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(1, 8192, 96, 128, 128, 64, ctypes.byref(n)) == 0
    # chunk states and their gradients (2 x 130 slots x 96 heads x 64 KB), six fp32 values per token, head and
    # channel, two per token and head; per slot and head: dgamma and gamma (512 B each), four 64 x 64 matrices,
    # three 64 x 128 tiles; and per slot and head the tensor-core reverse pass's bf16 hi/lo tiles (131,840 B)
    S = 130 * 96
    assert n.value == (2 * S * 65536 + 6 * 8192 * 96 * 512 + 2 * S * 512 + 4 * S * 16384 + 3 * S * 32768 +
                       2 * 8192 * 96 * 4 + S * 131840)
    assert lib.kda_chunk_bwd_workspace_size(1, 64, 2, 64, 128, 64, ctypes.byref(n)) == 2
    assert lib.kda_chunk_bwd_workspace_size(0, 64, 2, 128, 128, 64, ctypes.byref(n)) == 1
