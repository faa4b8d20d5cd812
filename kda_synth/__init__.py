"""Seeded synthetic inputs for the KDA hot path (test and benchmark infrastructure).

This module is the one thing the fp64 oracle (``oracle/``) and the CUDA library
(``gated_delta_rule_53_gb300``) share: it draws numbers, applies a workload's
input distribution and rounds them to the storage type.  It holds none of the
attention arithmetic.  The generator itself lives in ``synth.c`` (its definition
is written out at the top of that file); every element is a pure function of
(seed, tensor id, flat index), so one head of a 40 GB workload can be rebuilt on
its own.

bf16 tensors are returned as ``numpy.uint16`` bit patterns; :func:`bf16_to_f64`
and :func:`bf16_to_f32` widen them exactly.

The five workloads follow the configurations the KDA pages' hot path is
measured on (see :data:`WORKLOADS`): a tiny fp32 prefill, an 8K-token bf16
prefill with 96 heads, a 64-sequence decode step, a 32-sequence packed varlen
prefill and a 262,144-token prefill with the ShortConv front end and output gate.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None

# distribution kinds (must match synth.c)
NORMAL, NEG5_SIGMOID, SIGMOID, NEG_SOFTPLUS5, UNIT_GROUPS = 0, 1, 2, 3, 4
_DT = {"f64": (0, np.float64), "f32": (1, np.float32), "bf16": (2, np.uint16)}

# tensor ids of the generator streams
TID_Q, TID_K, TID_V, TID_G, TID_BETA, TID_STATE, TID_CONV_W, TID_CONV_STATE, TID_GATE, TID_LENGTHS = range(1, 11)
# upstream gradients of a backward: dL/do and dL/dS_final
TID_DO, TID_DSTATE = 11, 12


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_synth.so`` next to it (gcc, portable C99)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_int]
        lib.synth_u64.restype = ctypes.c_int
        lib.synth_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_void_p]
        _lib = lib
    return _lib


def host_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def fill_slice(seed: int, tid: int, kind: int, ld: int, row0: int, nrows: int, col0: int, ncols: int,
               dtype: str = "f32", p0: float = 0.0, p1: float = 1.0, out: np.ndarray | None = None,
               threads: int | None = None) -> np.ndarray:
    """Elements ``(row0 + r) * ld + col0 + c`` of a tensor viewed as rows of length ``ld``."""
    code, npdt = _DT[dtype]
    if out is None:
        out = np.empty((nrows, ncols), dtype=npdt)
    assert out.dtype == npdt and out.flags.c_contiguous and out.size == nrows * ncols
    rc = _load().synth_fill(seed, tid, kind, p0, p1, row0, nrows, ld, col0, ncols,
                            out.ctypes.data, code, threads or host_threads())
    if rc != 0:
        raise ValueError("synth_fill: bad arguments")
    return out


def fill(seed: int, tid: int, kind: int, shape, dtype: str = "f32", p0: float = 0.0, p1: float = 1.0,
         threads: int | None = None) -> np.ndarray:
    """A whole tensor of ``shape`` (flat row-major indices from 0)."""
    shape = tuple(int(s) for s in shape)
    last = shape[-1] if shape else 1
    rows = int(np.prod(shape)) // last if last else 0
    out = fill_slice(seed, tid, kind, last, 0, rows, 0, last, dtype, p0, p1, threads=threads)
    return out.reshape(shape)


def u64(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    if _load().synth_u64(seed, tid, start, count, out.ctypes.data) != 0:
        raise ValueError("synth_u64: bad arguments")
    return out


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(u: np.ndarray) -> np.ndarray:
    return bf16_to_f32(u).astype(np.float64)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def to_f64(a: np.ndarray) -> np.ndarray:
    return bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------------------------

@dataclass
class Workload:
    """One synthetic workload of the hot path.

    ``kind`` is ``"prefill"`` (q, k, v already normalised; kda_chunk_fwd alone),
    ``"frontend"`` (raw inputs through ShortConv+SiLU+L2norm, then kda_chunk_fwd and
    the sigmoid output gate) or ``"decode"`` (one token per sequence through
    kda_recurrent_step).
    """

    name: str
    kind: str
    seed: int
    H: int = 96
    d: int = 128
    lengths: list = field(default_factory=list)   # per-sequence token counts
    dtype: str = "bf16"                            # q, k, v (and o) storage type
    g_kind: int = NEG5_SIGMOID
    init_state_std: float = 0.0                    # 0 => zero initial state
    conv_w_std: float = 0.25
    chunk: int = 64
    scale: float = 1.0
    eps: float = 1e-6

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def varlen(self) -> bool:
        return self.N > 1 and self.kind != "decode"

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    # -- whole tensors ------------------------------------------------------------------------
    def qkv(self, which: str, threads=None) -> np.ndarray:
        """Normalised q / k or raw v, shape [T, H, d] (prefill workloads)."""
        tid = {"q": TID_Q, "k": TID_K, "v": TID_V}[which]
        kind = NORMAL if which == "v" else UNIT_GROUPS
        p1 = 1.0 if which == "v" else float(self.d)
        return fill(self.seed, tid, kind, (self.T, self.H, self.d), self.dtype, 0.0, p1, threads)

    def raw(self, which: str, threads=None) -> np.ndarray:
        """Raw front-end input x_q / x_k / x_v, bf16 [T, H*d] (one row per token)."""
        tid = {"q": TID_Q, "k": TID_K, "v": TID_V}[which]
        return fill(self.seed, tid, NORMAL, (self.T, self.H * self.d), "bf16", 0.0, 1.0, threads)

    def g(self, threads=None) -> np.ndarray:
        return fill(self.seed, TID_G, self.g_kind, (self.T, self.H, self.d), "f32", threads=threads)

    def beta(self, threads=None) -> np.ndarray:
        return fill(self.seed, TID_BETA, SIGMOID, (self.T, self.H), "f32", threads=threads)

    def init_state(self, threads=None):
        if self.init_state_std == 0.0:
            return None
        return fill(self.seed, TID_STATE, NORMAL, (self.N, self.H, self.d, self.d), "f32", 0.0,
                    self.init_state_std, threads)

    def conv_w(self) -> np.ndarray:
        return fill(self.seed, TID_CONV_W, NORMAL, (3 * self.H * self.d, 4), "bf16", 0.0, self.conv_w_std)

    def conv_state(self) -> np.ndarray:
        return fill(self.seed, TID_CONV_STATE, NORMAL, (self.N, 3, 3 * self.H * self.d), "bf16")

    def gate(self, threads=None) -> np.ndarray:
        return fill(self.seed, TID_GATE, NORMAL, (self.T, self.H * self.d), "bf16", 0.0, 1.0, threads)

    # -- one head, for the oracle on workloads too large to hold ------------------------------
    def head_rows(self, tid: int, kind: int, h: int, dtype: str, p1: float = 1.0, width: int | None = None,
                  t0: int = 0, t1: int | None = None):
        """Head ``h``'s ``d`` columns of a [T, H*d]-shaped tensor, tokens [t0, t1)."""
        t1 = self.T if t1 is None else t1
        width = self.H * self.d if width is None else width
        return fill_slice(self.seed, tid, kind, width, t0, t1 - t0, h * self.d, self.d, dtype, 0.0, p1)

    def head_beta(self, h: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        t1 = self.T if t1 is None else t1
        return fill_slice(self.seed, TID_BETA, SIGMOID, self.H, t0, t1 - t0, h, 1, "f32")[:, 0]

    def head_state(self, n: int, h: int):
        if self.init_state_std == 0.0:
            return None
        dd = self.d * self.d
        return fill_slice(self.seed, TID_STATE, NORMAL, self.H * dd, n, 1, h * dd, dd, "f32", 0.0,
                          self.init_state_std).reshape(self.d, self.d)


def varlen_lengths(seed: int, n: int, lo: int = 1024, hi: int = 32768) -> list:
    """Lengths uniform in [lo, hi]: lo + (bits mod (hi - lo + 1)) from the lengths stream."""
    b = u64(seed, TID_LENGTHS, 0, n)
    return [int(lo + int(x) % (hi - lo + 1)) for x in b]


def workload(name: str) -> Workload:
    """The five named workloads (seed = 53000 + their number)."""
    if name == "tiny_fp32":
        return Workload(name, "prefill", 53001, H=4, lengths=[256], dtype="f32")
    if name == "prefill_8k":
        return Workload(name, "prefill", 53002, H=96, lengths=[8192])
    if name == "decode_64":
        return Workload(name, "decode", 53003, H=96, lengths=[1] * 64, init_state_std=0.02)
    if name == "varlen_32":
        return Workload(name, "prefill", 53004, H=96, lengths=varlen_lengths(53004, 32),
                        init_state_std=0.02)
    if name == "long_256k":
        return Workload(name, "frontend", 53005, H=96, lengths=[262144], g_kind=NEG_SOFTPLUS5)
    raise KeyError(name)


WORKLOADS = ("tiny_fp32", "prefill_8k", "decode_64", "varlen_32", "long_256k")
