"""Kimi Delta Attention (KDA) on one GB300: thin Python binding of ``libkda.so``.

Every function here marshals torch tensors into the C ABI declared in
``include/kda.h`` (device pointers, sizes, the current CUDA stream) and calls
it; all arithmetic runs in the library's CUDA kernels.  PyTorch provides device
memory and streams only.  There is no CPU fallback: if ``libkda.so`` has not
been built (``python -m gated_delta_rule_53_gb300.build``), or no CUDA device is
present, the calls raise.

Entry points (same names as the C ABI):

* :func:`kda_shortconv_l2norm` — ShortConv(4) + SiLU on q, k, v; L2 norm of q, k.
* :func:`kda_chunk_fwd` — chunkwise prefill (``chunk_kda``), optional output gate.
* :func:`kda_recurrent_step` — fused single-token decode (``fused_recurrent_kda``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["kda_shortconv_l2norm", "kda_chunk_fwd", "kda_chunk_fwd_frontend", "kda_chunk_fwd_noalloc",
           "kda_chunk_fwd_workspace_size", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size",
           "kda_chunk_segment_summary", "kda_state_combine", "kda_gate_generator",
           "kda_recurrent_step", "library",
           "KDAError", "device_error", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkda.so")
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
_lib = None


class KDAError(RuntimeError):
    pass


def library() -> ctypes.CDLL:
    """The loaded ``libkda.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KDAError(f"{LIB_PATH} is missing: build it with `python -m gated_delta_rule_53_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.kda_shortconv_l2norm.argtypes = [P, P, P, I64, P, P, I32, I64, I32, I32, P, P, F, I32, P, P, P, P]
        SZ = ctypes.c_size_t
        lib.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, F, I32, I32, P, P, P, P, SZ, P]
        lib.kda_chunk_fwd_frontend.argtypes = [P, P, P, I64, P, P, P, F, P, P, P, P, I32, I64, I32, I32, F, I32, P, P,
                                               P, P, SZ, P]
        lib.kda_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, F, I32, I32, P, P, P, P]
        lib.kda_chunk_fwd_workspace_size.argtypes = [I32, I64, I32, I32, I32, I32, I32, I32, ctypes.POINTER(SZ),
                                                     ctypes.POINTER(SZ)]
        lib.kda_recurrent_step.argtypes = [P, P, P, I64, P, P, P, P, P, I32, I32, I32, I32, F, F, P, P]
        lib.kda_chunk_segment_summary.argtypes = [P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, P, P, P, SZ, P]
        lib.kda_state_combine.argtypes = [P, P, P, P, I64, P]
        lib.kda_chunk_bwd.argtypes = [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, F, I32, I32, P, P, P, P, P, P, P,
                                      P, P, SZ, P]
        lib.kda_chunk_bwd_workspace_size.argtypes = [I32, I64, I32, I32, I32, I32, ctypes.POINTER(SZ)]
        lib.kda_gate_generator.argtypes = [P, I64, I32, P, P, P, I32, I32, I32, P, P, P, P]
        for f in (lib.kda_shortconv_l2norm, lib.kda_chunk_fwd, lib.kda_recurrent_step, lib.kda_device_error,
                  lib.kda_chunk_fwd_workspace_size, lib.kda_chunk_fwd_noalloc, lib.kda_chunk_fwd_frontend):
            f.restype = ctypes.c_int
        lib.kda_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.kda_selftest_bounded_wait.argtypes = [ctypes.c_uint, ctypes.c_void_p]
        lib.kda_selftest_bounded_wait.restype = ctypes.c_int
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_version.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        lib = library()
        raise KDAError(f"{what}: {lib.kda_status_string(rc).decode()} — {lib.kda_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise KDAError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise KDAError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise KDAError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise KDAError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def device_error() -> int:
    """Read and clear the library's device error word (synchronises the device)."""
    code = ctypes.c_uint(0)
    _check(library().kda_device_error(ctypes.byref(code)), "kda_device_error")
    return int(code.value)


def selftest_bounded_wait(poll_limit: int = 1000, stream=None) -> None:
    """Launch the diagnostic kernel whose barrier wait always runs out (see include/kda.h)."""
    _check(library().kda_selftest_bounded_wait(int(poll_limit), _stream(stream)), "kda_selftest_bounded_wait")


def kda_shortconv_l2norm(xq, xk, xv, conv_w, H: int, cu_seqlens=None, conv_state_in=None, conv_state_out=None,
                         eps: float = 1e-6, out_dtype=torch.bfloat16, q=None, k=None, v=None, stream=None):
    """ShortConv(4) + SiLU on raw bf16 rows x* [T, >=H*128] (row stride = x.stride(0));
    returns (q, k, v) [T, H, 128] with q, k L2-normalised per head."""
    d = 128
    T = xq.shape[0]
    for name, x in (("xq", xq), ("xk", xk), ("xv", xv)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
            raise KDAError(f"{name} must be a CUDA bf16 [T, width] tensor with unit inner stride")
        if x.shape[0] != T or x.stride(0) != xq.stride(0):
            raise KDAError("xq, xk, xv must share shape and row stride")
    _dev(conv_w, "conv_w", torch.bfloat16, (3 * H * d, 4))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(conv_state_in, "conv_state_in", torch.bfloat16, (N, 3, 3 * H * d))
    _dev(conv_state_out, "conv_state_out", torch.bfloat16, (N, 3, 3 * H * d))
    outs = []
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t is None:
            t = torch.empty((T, H, d), dtype=out_dtype, device=xq.device)
        outs.append(_dev(t, name, out_dtype, (T, H, d)))
    dt = KDA_DTYPE_BF16 if out_dtype == torch.bfloat16 else KDA_DTYPE_F32
    rc = library().kda_shortconv_l2norm(_ptr(xq), _ptr(xk), _ptr(xv), xq.stride(0), _ptr(conv_w), _ptr(cu_seqlens),
                                        N, T, H, d, _ptr(conv_state_in), _ptr(conv_state_out), float(eps), dt,
                                        _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _stream(stream))
    _check(rc, "kda_shortconv_l2norm")
    return tuple(outs)


WORKSPACE_LIMIT = 8 << 30  # default cap of the prefill workspace (bytes); larger problems run in ranges


def kda_chunk_fwd_workspace_size(N: int, T: int, H: int, dtype=torch.bfloat16, have_cu_seqlens: bool = True,
                                 dk: int = 128, dv: int = 128, chunk_size: int = 64):
    """(full_bytes, min_bytes) of the prefill workspace for these sizes (0, 0 for fp32)."""
    full, least = ctypes.c_size_t(0), ctypes.c_size_t(0)
    dt = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_F32
    _check(library().kda_chunk_fwd_workspace_size(N, T, H, dk, dv, chunk_size, dt, 1 if have_cu_seqlens else 0,
                                                  ctypes.byref(full), ctypes.byref(least)),
           "kda_chunk_fwd_workspace_size")
    return int(full.value), int(least.value)


def kda_chunk_fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale: float = 1.0, chunk_size: int = 64,
                  out_gate=None, o=None, final_state=None, output_final_state: bool = True, workspace=None,
                  workspace_limit: int = WORKSPACE_LIMIT, stream=None):
    """Chunkwise KDA prefill.  q, k, v [T, H, 128] (bf16 or fp32, q and k L2-normalised),
    g fp32 [T, H, 128] in [-5, 0], beta fp32 [T, H], init_state fp32 [N, H, 128, 128] or None,
    cu_seqlens int32 [N+1] or None, out_gate bf16 [T, H*128] or None.  workspace: a uint8 CUDA
    tensor, or None to take one of min(full, workspace_limit) bytes (at least the minimum) from
    PyTorch's allocator.  Returns (o [T, H, 128], final_state [N, H, 128, 128] or None)."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise KDAError("q, k, v must be bf16 or fp32")
    _dev(q, "q", dtype); _dev(k, "k", dtype, (T, H, dk)); _dev(v, "v", dtype, (T, H, dv))
    _dev(g, "g", torch.float32, (T, H, dk)); _dev(beta, "beta", torch.float32, (T, H))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(init_state, "init_state", torch.float32, (N, H, dv, dk))
    _dev(out_gate, "out_gate", torch.bfloat16, (T, H * dv))
    if o is None:
        o = torch.empty((T, H, dv), dtype=dtype, device=q.device)
    _dev(o, "o", dtype, (T, H, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    _dev(final_state, "final_state", torch.float32, (N, H, dv, dk))
    dt = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_F32
    if workspace is None and dt == KDA_DTYPE_BF16:
        full, least = kda_chunk_fwd_workspace_size(N, T, H, dtype, cu_seqlens is not None, dk, dv, chunk_size)
        workspace = torch.empty(max(least, min(full, int(workspace_limit))), dtype=torch.uint8, device=q.device)
    if workspace is not None:
        _dev(workspace, "workspace", torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel()
    rc = library().kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                                 N, T, H, dk, dv, float(scale), int(chunk_size), dt, _ptr(out_gate), _ptr(o),
                                 _ptr(final_state), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "kda_chunk_fwd")
    return o, final_state


def kda_chunk_bwd_workspace_size(N: int, T: int, H: int, dk: int = 128, dv: int = 128, chunk_size: int = 64) -> int:
    n = ctypes.c_size_t(0)
    _check(library().kda_chunk_bwd_workspace_size(N, T, H, dk, dv, chunk_size, ctypes.byref(n)),
           "kda_chunk_bwd_workspace_size")
    return int(n.value)


def kda_chunk_bwd(q, k, v, g, beta, d_o, init_state=None, cu_seqlens=None, d_final_state=None, scale: float = 1.0,
                  chunk_size: int = 64, output_d_init_state: bool = True, workspace=None, stream=None):
    """Backward of kda_chunk_fwd.  q, k, v, d_o [T, H, 128] in one dtype (bf16 or fp32); g, beta, init_state,
    cu_seqlens as kda_chunk_fwd; d_final_state fp32 [N, H, 128, 128] or None (= zeros).  workspace: a uint8
    CUDA tensor of at least kda_chunk_bwd_workspace_size bytes, or None to take one from PyTorch's allocator.
    Returns fp32 (dq, dk, dv, dg, dbeta, d_init_state or None)."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise KDAError("q, k, v, d_o must be bf16 or fp32")
    _dev(q, "q", dtype); _dev(k, "k", dtype, (T, H, dk)); _dev(v, "v", dtype, (T, H, dv))
    _dev(d_o, "d_o", dtype, (T, H, dv))
    _dev(g, "g", torch.float32, (T, H, dk)); _dev(beta, "beta", torch.float32, (T, H))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(init_state, "init_state", torch.float32, (N, H, dv, dk))
    _dev(d_final_state, "d_final_state", torch.float32, (N, H, dv, dk))
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dkk, dg = (torch.empty((T, H, dk), **f32) for _ in range(3))
    dvv, db = torch.empty((T, H, dv), **f32), torch.empty((T, H), **f32)
    d_init = torch.empty((N, H, dv, dk), **f32) if output_d_init_state else None
    if workspace is None:
        workspace = torch.empty(kda_chunk_bwd_workspace_size(N, T, H, dk, dv, chunk_size), dtype=torch.uint8,
                                device=q.device)
    _dev(workspace, "workspace", torch.uint8)
    dt = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_F32
    rc = library().kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                                 N, T, H, dk, dv, float(scale), int(chunk_size), dt, _ptr(d_o), _ptr(d_final_state),
                                 _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg), _ptr(db), _ptr(d_init), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(rc, "kda_chunk_bwd")
    return dq, dkk, dvv, dg, db, d_init


def kda_chunk_segment_summary(k, g, beta, v=None, q=None, cu_seqlens=None, end_state=True, transition=True,
                              workspace=None, workspace_limit: int = WORKSPACE_LIMIT, stream=None):
    """Per (sequence, head) segment: E = final state from a zero start and M = its transition operator
    (the segment maps an entering state S to S M + E).  k, v (and optionally q) bf16 [T, H, 128], g fp32
    [T, H, 128], beta fp32 [T, H].  end_state / transition: True (allocate), a fp32 [N, H, 128, 128]
    CUDA tensor, or False/None (skip).  Returns (E or None, M or None)."""
    T, H, dk = k.shape
    _dev(k, "k", torch.bfloat16)
    _dev(q, "q", torch.bfloat16, (T, H, dk)); _dev(v, "v", torch.bfloat16, (T, H, dk))
    _dev(g, "g", torch.float32, (T, H, dk)); _dev(beta, "beta", torch.float32, (T, H))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    outs = []
    for want, name in ((end_state, "end_state"), (transition, "transition")):
        if want is True:
            want = torch.empty((N, H, dk, dk), dtype=torch.float32, device=k.device)
        elif want is False:
            want = None
        _dev(want, name, torch.float32, (N, H, dk, dk))
        outs.append(want)
    E, M = outs
    if workspace is None:
        full, least = kda_chunk_fwd_workspace_size(N, T, H, torch.bfloat16, cu_seqlens is not None, dk, dk, 64)
        workspace = torch.empty(max(least, min(full, int(workspace_limit))), dtype=torch.uint8, device=k.device)
    _dev(workspace, "workspace", torch.uint8)
    rc = library().kda_chunk_segment_summary(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N,
                                             T, H, dk, dk, 64, _ptr(E), _ptr(M), _ptr(workspace), workspace.numel(),
                                             _stream(stream))
    _check(rc, "kda_chunk_segment_summary")
    return E, M


def kda_state_combine(S_in, M, E, out=None, stream=None):
    """S_in M + E over the leading dimensions of fp32 [..., 128, 128] CUDA tensors (S_in None: E)."""
    shape = E.shape
    if len(shape) < 2 or tuple(shape[-2:]) != (128, 128):
        raise KDAError("E must be [..., 128, 128]")
    _dev(E, "E", torch.float32); _dev(M, "M", torch.float32, tuple(shape)); _dev(S_in, "S_in", torch.float32, tuple(shape))
    if out is None:
        out = torch.empty_like(E)
    _dev(out, "out", torch.float32, tuple(shape))
    count = E.numel() // (128 * 128)
    _check(library().kda_state_combine(_ptr(S_in), _ptr(M), _ptr(E), _ptr(out), count, _stream(stream)),
           "kda_state_combine")
    return out


def kda_gate_generator(x, w_gate_a, w_b, a_head, H: int, d: int = 128, gate=None, g=None, z=None, stream=None):
    """Output gate bf16 [T, H*d] and decay gate g fp32 [T, H, d] = max(-5, -softplus(x W_a^T W_b^T + a_h))
    from x bf16 [T, hidden]; w_gate_a bf16 [H*d + rank, hidden] (W_gate rows, then W_a rows), w_b bf16
    [H*d, rank], a_head fp32 [H].  Returns (gate, g)."""
    T, hidden = x.shape
    rank = w_gate_a.shape[0] - H * d
    _dev(x, "x", torch.bfloat16); _dev(w_gate_a, "w_gate_a", torch.bfloat16, (H * d + rank, hidden))
    _dev(w_b, "w_b", torch.bfloat16, (H * d, rank)); _dev(a_head, "a_head", torch.float32, (H,))
    if gate is None:
        gate = torch.empty((T, H * d), dtype=torch.bfloat16, device=x.device)
    if g is None:
        g = torch.empty((T, H, d), dtype=torch.float32, device=x.device)
    if z is None:
        z = torch.empty((max(T, 1), rank), dtype=torch.bfloat16, device=x.device)
    _dev(gate, "gate", torch.bfloat16, (T, H * d)); _dev(g, "g", torch.float32, (T, H, d)); _dev(z, "z", torch.bfloat16)
    _check(library().kda_gate_generator(_ptr(x), T, hidden, _ptr(w_gate_a), _ptr(w_b), _ptr(a_head), H, d, rank,
                                        _ptr(gate), _ptr(g), _ptr(z), _stream(stream)), "kda_gate_generator")
    return gate, g


def kda_chunk_fwd_frontend(xq, xk, xv, conv_w, g, beta, H: int, init_state=None, cu_seqlens=None,
                           conv_state_in=None, conv_state_out=None, eps: float = 1e-6, scale: float = 1.0,
                           chunk_size: int = 64, out_gate=None, o=None, final_state=None,
                           output_final_state: bool = True, workspace=None, workspace_limit: int = WORKSPACE_LIMIT,
                           stream=None):
    """kda_shortconv_l2norm (bf16) + kda_chunk_fwd (bf16) in one pass: raw bf16 xq, xk, xv [T, >=H*128]
    (one row stride), conv_w bf16 [3*H*128, 4], g fp32 [T, H, 128], beta fp32 [T, H].
    Returns (o bf16 [T, H, 128], final_state or None)."""
    d = 128
    T = xq.shape[0]
    for name, x in (("xq", xq), ("xk", xk), ("xv", xv)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1 or x.shape[0] != T:
            raise KDAError(f"{name} must be a CUDA bf16 [T, width] tensor with unit inner stride")
        if x.stride(0) != xq.stride(0):
            raise KDAError("xq, xk, xv must share their row stride")
    _dev(conv_w, "conv_w", torch.bfloat16, (3 * H * d, 4))
    _dev(g, "g", torch.float32, (T, H, d)); _dev(beta, "beta", torch.float32, (T, H))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(init_state, "init_state", torch.float32, (N, H, d, d))
    _dev(conv_state_in, "conv_state_in", torch.bfloat16, (N, 3, 3 * H * d))
    _dev(conv_state_out, "conv_state_out", torch.bfloat16, (N, 3, 3 * H * d))
    _dev(out_gate, "out_gate", torch.bfloat16, (T, H * d))
    if o is None:
        o = torch.empty((T, H, d), dtype=torch.bfloat16, device=xq.device)
    _dev(o, "o", torch.bfloat16, (T, H, d))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32, device=xq.device)
    _dev(final_state, "final_state", torch.float32, (N, H, d, d))
    if workspace is None:
        full, least = kda_chunk_fwd_workspace_size(N, T, H, torch.bfloat16, cu_seqlens is not None, d, d, chunk_size)
        workspace = torch.empty(max(least, min(full, int(workspace_limit))), dtype=torch.uint8, device=xq.device)
    _dev(workspace, "workspace", torch.uint8)
    rc = library().kda_chunk_fwd_frontend(_ptr(xq), _ptr(xk), _ptr(xv), xq.stride(0), _ptr(conv_w),
                                          _ptr(conv_state_in), _ptr(conv_state_out), float(eps), _ptr(g), _ptr(beta),
                                          _ptr(init_state), _ptr(cu_seqlens), N, T, H, d, float(scale),
                                          int(chunk_size), _ptr(out_gate), _ptr(o), _ptr(final_state),
                                          _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "kda_chunk_fwd_frontend")
    return o, final_state


def kda_chunk_fwd_noalloc(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale: float = 1.0,
                          chunk_size: int = 64, out_gate=None, o=None, final_state=None,
                          output_final_state: bool = True, stream=None):
    """kda_chunk_fwd on the library's static 64 MiB scratch instead of a workspace (no allocation
    for it); raises KDAError when the sizes need more than that.  Calls must not overlap."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise KDAError("q, k, v must be bf16 or fp32")
    _dev(q, "q", dtype); _dev(k, "k", dtype, (T, H, dk)); _dev(v, "v", dtype, (T, H, dv))
    _dev(g, "g", torch.float32, (T, H, dk)); _dev(beta, "beta", torch.float32, (T, H))
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(init_state, "init_state", torch.float32, (N, H, dv, dk))
    _dev(out_gate, "out_gate", torch.bfloat16, (T, H * dv))
    if o is None:
        o = torch.empty((T, H, dv), dtype=dtype, device=q.device)
    _dev(o, "o", dtype, (T, H, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    _dev(final_state, "final_state", torch.float32, (N, H, dv, dk))
    dt = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_F32
    rc = library().kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                                         _ptr(cu_seqlens), N, T, H, dk, dv, float(scale), int(chunk_size), dt,
                                         _ptr(out_gate), _ptr(o), _ptr(final_state), _stream(stream))
    _check(rc, "kda_chunk_fwd_noalloc")
    return o, final_state


def kda_recurrent_step(xq, xk, xv, conv_w, g, beta, state, conv_state, scale: float = 1.0, eps: float = 1e-6,
                       o=None, stream=None):
    """One fused decode step, in place on ``state`` (fp32 [N, H, 128, 128]) and
    ``conv_state`` (bf16 [N, 3, 3*H*128]).  x* raw bf16 [N, >=H*128]; g fp32 [N, H, 128];
    beta fp32 [N, H].  Returns o bf16 [N, H, 128]."""
    N, H, dv, dk = state.shape
    for name, x in (("xq", xq), ("xk", xk), ("xv", xv)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1 or x.shape[0] != N:
            raise KDAError(f"{name} must be a CUDA bf16 [N, width] tensor with unit inner stride")
        if x.stride(0) != xq.stride(0):
            raise KDAError("xq, xk, xv must share their row stride")
    _dev(conv_w, "conv_w", torch.bfloat16, (3 * H * dk, 4))
    _dev(g, "g", torch.float32, (N, H, dk)); _dev(beta, "beta", torch.float32, (N, H))
    _dev(state, "state", torch.float32); _dev(conv_state, "conv_state", torch.bfloat16, (N, 3, 3 * H * dk))
    if o is None:
        o = torch.empty((N, H, dv), dtype=torch.bfloat16, device=state.device)
    _dev(o, "o", torch.bfloat16, (N, H, dv))
    rc = library().kda_recurrent_step(_ptr(xq), _ptr(xk), _ptr(xv), xq.stride(0), _ptr(conv_w), _ptr(g), _ptr(beta),
                                      _ptr(state), _ptr(conv_state), N, H, dk, dv, float(scale), float(eps), _ptr(o),
                                      _stream(stream))
    _check(rc, "kda_recurrent_step")
    return o
