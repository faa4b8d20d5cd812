"""fp64 CPU oracle for Kimi Delta Attention (KDA) — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and the two
share no code; the only thing both sides take is the seeded input generator
``kda_synth``.

The arithmetic lives in ``kda_oracle.c`` (plain C99, fp64, one thread per
(sequence, head) chain), compiled with gcc into ``_oracle.so`` next to it:

* :func:`kda_tokenloop` — the recurrence one token at a time, the definition of
  the result ("Kimi-K3 深度解析", section 三, "KDA 的关键改进").
* :func:`kda_chunked` — the same result chunk by chunk (the ``chunk_kda`` form named
  in "Kimi K3 架构全景", section 02), checked against the token loop.
* :func:`shortconv_silu_l2norm` — ShortConv(kernel 4) + SiLU on q, k, v and the L2
  norm of q and k ("深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA).
* :func:`output_gate` — o * sigmoid(gate), the full-rank output gate (same paragraph).
* :func:`recurrent_step` — one decode step: the front end on one token per
  sequence followed by one step of the token loop (``fused_recurrent_kda``).
* :func:`gate_generator` — the decay gate and the full-rank output gate from the layer input,
  as read from "深入 Kimi-K3: Hugging Face 仓库分析" (paragraph on KDA: a low-rank projection plus a
  per-head parameter, floored at -5): gate = x W_gate^T, g = max(-5, -softplus(x W_a^T W_b^T + a_h)).
* :func:`kda_tokenloop_bwd` — the gradients of a loss with respect to q, k, v, g, beta and the
  initial state, by reverse mode through the token loop (the backward of ``chunk_kda``; the
  pages name the operator and its training use, "月之暗面发布Kimi K3开源大模型技术报告", 架构).
* :func:`kda_chunked_bwd` — the same gradients by the chain rule through the chunk form (fp64
  numpy), checked against the token loop's reverse mode: the algebra the GPU backward follows.
* :func:`transition` — a segment's transition operator M = X_1 ... X_L with
  X_t = Diag(alpha_t)(I - beta_t k_t k_t^T), formed as a literal product of dense
  matrices: a segment maps its entering state S to S M + E (E its end state from zero),
  which is how a state is carried across segments of one sequence.

All arrays are fp64 numpy arrays in the layouts of ``kda_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable C99, -O2, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                                   "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
        lib.oracle_kda_tokenloop.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, P, P, ctypes.c_int]
        lib.oracle_kda_chunked.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, I, P, P, ctypes.c_int]
        lib.oracle_kda_transition.argtypes = [P, P, P, P, I, I, I, I, P, ctypes.c_int]
        lib.oracle_kda_tokenloop_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, P, P, P, P, P, P, P, P,
                                                 ctypes.c_int]
        lib.oracle_shortconv_silu_l2norm.argtypes = [P, P, P, I, P, P, I, I, I, I, P, D, P, P, P, P,
                                                     ctypes.c_int]
        for f in (lib.oracle_kda_tokenloop, lib.oracle_kda_chunked, lib.oracle_shortconv_silu_l2norm,
                  lib.oracle_kda_transition, lib.oracle_kda_tokenloop_bwd):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _f64(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return None, 1
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    assert cu[0] == 0 and cu[-1] == T
    return cu, len(cu) - 1


def _kda(fn, q, k, v, g, beta, init_state, cu_seqlens, scale, chunk, nthreads):
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (T, H, dk) and g.shape == (T, H, dk) and v.shape == (T, H, dv)
    assert beta.shape == (T, H)
    cu, N = _cu(cu_seqlens, T)
    s0 = _f64(init_state)
    if s0 is not None:
        assert s0.shape == (N, H, dv, dk)
    o = np.empty((T, H, dv), np.float64)
    fs = np.empty((N, H, dv, dk), np.float64)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), _ptr(cu), N, T, H, dk, dv, float(scale)]
    if chunk is not None:
        args.append(int(chunk))
    args += [_ptr(o), _ptr(fs), nthreads or threads()]
    if fn(*args) != 0:
        raise ValueError("oracle rejected its arguments")
    return o, fs


def kda_tokenloop(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=1.0, nthreads=None):
    """(o [T,H,dv], final_state [N,H,dv,dk]) by the per-token recurrence."""
    return _kda(_load().oracle_kda_tokenloop, q, k, v, g, beta, init_state, cu_seqlens, scale, None, nthreads)


def kda_chunked(q, k, v, g, beta, init_state=None, cu_seqlens=None, scale=1.0, chunk=64, nthreads=None):
    """The same pair computed chunk by chunk (unit-triangular solve per chunk)."""
    return _kda(_load().oracle_kda_chunked, q, k, v, g, beta, init_state, cu_seqlens, scale, chunk, nthreads)


def kda_tokenloop_bwd(q, k, v, g, beta, d_o, init_state=None, cu_seqlens=None, scale=1.0, d_final=None,
                      nthreads=None):
    """Gradients of a loss through the per-token recurrence, by reverse mode: given dL/do [T,H,dv] and
    dL/dS_end [N,H,dv,dk] (None = 0), returns (dq, dk [T,H,dk], dv [T,H,dv], dg [T,H,dk],
    dbeta [T,H], dL/dS0 [N,H,dv,dk])."""
    return _bwd(_load().oracle_kda_tokenloop_bwd, q, k, v, g, beta, d_o, init_state, cu_seqlens, scale, d_final,
                nthreads)


def _bwd(fn, q, k, v, g, beta, d_o, init_state, cu_seqlens, scale, d_final, nthreads):
    q, k, v, g, beta, d_o = (_f64(x) for x in (q, k, v, g, beta, d_o))
    T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (T, H, dk) and g.shape == (T, H, dk) and v.shape == (T, H, dv) and d_o.shape == (T, H, dv)
    assert beta.shape == (T, H)
    cu, N = _cu(cu_seqlens, T)
    s0, dfin = _f64(init_state), _f64(d_final)
    for x in (s0, dfin):
        if x is not None:
            assert x.shape == (N, H, dv, dk)
    dq, dkk, dg = (np.empty((T, H, dk)) for _ in range(3))
    dvv, db, ds0 = np.empty((T, H, dv)), np.empty((T, H)), np.empty((N, H, dv, dk))
    if fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), _ptr(cu), N, T, H, dk, dv, float(scale),
          _ptr(d_o), _ptr(dfin), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg), _ptr(db), _ptr(ds0),
          nthreads or threads()) != 0:
        raise ValueError("oracle rejected its arguments")
    return dq, dkk, dvv, dg, db, ds0


def _chunk_bwd_chain(q, k, v, g, beta, S0, d_o, d_final, scale, C):
    """One (sequence, head) chain: the chain rule through the chunk form, chunk by chunk.

    Per chunk with S0 entering it, G the running sum of g, A the pair products with their decays
    e^{G_ic - G_jc} (A_kk = Diag(beta) B strictly below the diagonal, A_qk on and below it):
      forward  R = V - (K e^G) S0^T,  V' = (I + A_kk)^-1 Diag(beta) R,
               O = scale ((Q e^G) S0^T + A_qk V'),  S_next = S0 Diag(e^{G_last}) + V'^T (K e^{G_last - G})
      reverse  dV' = scale A_qk^T dO + (K e^{G_last - G}) dS_next^T,  dZ = (I + A_kk)^-T dV',
               dS0 = dS_next Diag(e^{G_last}) + scale dO^T (Q e^G) - (Diag(beta) dZ)^T (K e^G)
    and inside the chunk the gradients of every factor above, with G's gradient summed backwards
    into g's.  Every exponent e^{G_ic - G_jc} used has j <= i (never positive)."""
    T, dk = q.shape
    fw, S = [], S0.copy()
    for a in range(0, T, C):
        z = min(a + C, T)
        L = z - a
        qq, kk, vv, gg, bb = q[a:z], k[a:z], v[a:z], g[a:z], beta[a:z]
        G = np.cumsum(gg, 0)
        low, lowd = np.tril(np.ones((L, L)), -1), np.tril(np.ones((L, L)))
        D = G[:, None, :] - G[None, :, :]                         # [i, j, c]
        E = np.exp(np.where(lowd[:, :, None] > 0, D, -np.inf))     # e^{G_ic - G_jc} for j <= i, else 0
        B = np.einsum("ic,jc,ijc->ij", kk, kk, E) * low
        Aqk = np.einsum("ic,jc,ijc->ij", qq, kk, E)
        Akk = bb[:, None] * B
        Kg, Qg, Kr, gam = kk * np.exp(G), qq * np.exp(G), kk * np.exp(G[-1] - G), np.exp(G[-1])
        R = vv - Kg @ S.T
        Vp = np.linalg.solve(np.eye(L) + Akk, bb[:, None] * R)
        fw.append((a, z, S.copy(), G, E, B, Aqk, Akk, Kg, Qg, Kr, gam, R, Vp, low, lowd))
        S = S * gam[None, :] + Vp.T @ Kr
    dq, dkk, dg = np.zeros_like(q), np.zeros_like(k), np.zeros_like(g)
    dvv, db = np.zeros_like(v), np.zeros_like(beta)
    dS = d_final.copy()
    for (a, z, S0c, G, E, B, Aqk, Akk, Kg, Qg, Kr, gam, R, Vp, low, lowd) in reversed(fw):
        L = z - a
        qq, kk, bb, dO = q[a:z], k[a:z], beta[a:z], d_o[a:z]
        dVp = scale * Aqk.T @ dO + Kr @ dS.T
        dZ = np.linalg.solve((np.eye(L) + Akk).T, dVp)
        dQg, dKg, dKr = scale * dO @ S0c, -(bb[:, None] * dZ) @ S0c, Vp @ dS
        dgam = np.sum(dS * S0c, axis=0)
        dAqk = scale * (dO @ Vp.T) * lowd
        dAkk = -(dZ @ Vp.T) * low
        dB = bb[:, None] * dAkk
        dvv[a:z] = bb[:, None] * dZ
        db[a:z] = np.sum(dZ * R, axis=1) + np.sum(dAkk * B, axis=1)
        rowQ = np.einsum("ij,jc,ijc->ic", dAqk, kk, E)
        colQ = np.einsum("ij,ic,ijc->jc", dAqk, qq, E)
        rowK = np.einsum("ij,jc,ijc->ic", dB, kk, E)
        colK = np.einsum("ij,ic,ijc->jc", dB, kk, E)
        dq[a:z] = rowQ + dQg * np.exp(G)
        dkk[a:z] = rowK + colQ + colK + dKg * np.exp(G) + dKr * np.exp(G[-1] - G)
        dG = qq * rowQ + kk * rowK - kk * (colQ + colK) + dQg * Qg + dKg * Kg - dKr * Kr
        dG[-1] += np.sum(dKr * Kr, axis=0) + dgam * gam
        dg[a:z] = np.cumsum(dG[::-1], 0)[::-1]
        dS = dS * gam[None, :] + scale * dO.T @ Qg - (bb[:, None] * dZ).T @ Kg
    return dq, dkk, dvv, dg, db, dS


def kda_chunked_bwd(q, k, v, g, beta, d_o, init_state=None, cu_seqlens=None, scale=1.0, d_final=None, chunk=64):
    """The same gradients as kda_tokenloop_bwd, by the chain rule through the chunk form (fp64 numpy):
    the algebra the GPU backward follows, checked against the token loop's reverse mode."""
    q, k, v, g, beta, d_o = (_f64(x) for x in (q, k, v, g, beta, d_o))
    T, H, dk = q.shape
    dv = v.shape[-1]
    cu, N = _cu(cu_seqlens, T)
    bounds = [0, T] if cu is None else list(cu)
    s0, dfin = _f64(init_state), _f64(d_final)
    dq, dkk, dg = (np.zeros((T, H, dk)) for _ in range(3))
    dvv, db, ds0 = np.zeros((T, H, dv)), np.zeros((T, H)), np.zeros((N, H, dv, dk))
    for n in range(N):
        a, z = bounds[n], bounds[n + 1]
        for h in range(H):
            S0 = s0[n, h] if s0 is not None else np.zeros((dv, dk))
            dF = dfin[n, h] if dfin is not None else np.zeros((dv, dk))
            if z == a:
                ds0[n, h] = dF
                continue
            out = _chunk_bwd_chain(q[a:z, h], k[a:z, h], v[a:z, h], g[a:z, h], beta[a:z, h], S0, d_o[a:z, h], dF,
                                   float(scale), int(chunk))
            dq[a:z, h], dkk[a:z, h], dvv[a:z, h], dg[a:z, h], db[a:z, h], ds0[n, h] = out
    return dq, dkk, dvv, dg, db, ds0


def transition(k, g, beta, cu_seqlens=None, nthreads=None):
    """M [N, H, dk, dk]: each (sequence, head) segment's product X_1 ... X_L of
    X_t = Diag(exp g_t)(I - beta_t k_t k_t^T), so that the segment maps S to S M + E."""
    k, g, beta = (_f64(x) for x in (k, g, beta))
    T, H, dk = k.shape
    assert g.shape == (T, H, dk) and beta.shape == (T, H)
    cu, N = _cu(cu_seqlens, T)
    M = np.empty((N, H, dk, dk), np.float64)
    if _load().oracle_kda_transition(_ptr(k), _ptr(g), _ptr(beta), _ptr(cu), N, T, H, dk, _ptr(M),
                                     nthreads or threads()) != 0:
        raise ValueError("oracle rejected its arguments")
    return M


def gate_generator(x, w_gate_a, w_b, a_head, H, d):
    """(gate [T, H*d], g [T, H, d]) in fp64: gate = x W_gate^T; z = x W_a^T; y = z W_b^T + a_h (a_h the
    head's parameter on each of its d channels); g = max(-5, -softplus(y)), softplus(y) = log(1 + e^y).
    w_gate_a stacks W_gate (H*d rows) over W_a (rank rows)."""
    x, w_gate_a, w_b, a_head = (_f64(t) for t in (x, w_gate_a, w_b, a_head))
    hd = H * d
    gate = x @ w_gate_a[:hd].T
    z = x @ w_gate_a[hd:].T
    y = z @ w_b.T + np.repeat(a_head, d)[None, :]
    g = np.maximum(-5.0, -np.logaddexp(0.0, y))
    return gate, g.reshape(x.shape[0], H, d)


def shortconv_silu_l2norm(xq, xk, xv, conv_w, H, d, cu_seqlens=None, conv_state_in=None, eps=1e-6,
                          want_state=True, nthreads=None):
    """Front end.  x*: [T, >=H*d] raw rows; conv_w: [3*H*d, 4] (q|k|v channel blocks,
    taps oldest..current); conv_state_in: [N, 3, 3*H*d] or None (zeros).
    Returns q, k, v [T, H, d] and the carried state [N, 3, 3*H*d] (or None)."""
    xq, xk, xv, w = (_f64(x) for x in (xq, xk, xv, conv_w))
    T, ld = xq.shape
    assert xk.shape == (T, ld) and xv.shape == (T, ld) and w.shape == (3 * H * d, 4)
    cu, N = _cu(cu_seqlens, T)
    cs = _f64(conv_state_in)
    if cs is not None:
        assert cs.shape == (N, 3, 3 * H * d)
    q = np.empty((T, H, d)); k = np.empty((T, H, d)); v = np.empty((T, H, d))
    cs_out = np.empty((N, 3, 3 * H * d)) if want_state else None
    rc = _load().oracle_shortconv_silu_l2norm(_ptr(xq), _ptr(xk), _ptr(xv), ld, _ptr(w), _ptr(cu), N, T, H, d,
                                              _ptr(cs), float(eps), _ptr(q), _ptr(k), _ptr(v), _ptr(cs_out),
                                              nthreads or threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return q, k, v, cs_out


def output_gate(o, gate):
    """o * sigmoid(gate); o [T, H, dv], gate [T, H*dv]."""
    o = np.asarray(o, np.float64)
    gt = np.asarray(gate, np.float64).reshape(o.shape)
    return o * (1.0 / (1.0 + np.exp(-gt)))


def recurrent_step(xq, xk, xv, conv_w, g, beta, state, conv_state, H, d, scale=1.0, eps=1e-6, nthreads=None):
    """One decode step for N sequences of one token each.

    x*: [N, H*d] raw; g: [N, H, d]; beta: [N, H]; state [N, H, d, d]; conv_state [N, 3, 3*H*d].
    Returns (o [N, H, d], new state, new conv_state)."""
    N = np.asarray(xq).shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    q, k, v, cs = shortconv_silu_l2norm(xq, xk, xv, conv_w, H, d, cu, conv_state, eps, True, nthreads)
    o, s = kda_tokenloop(q, k, v, g, beta, state, cu, scale, nthreads)
    return o, s, cs


def state_numel(layers: int, H: int, dk: int, dv: int) -> int:
    """Values of recurrent state one sequence holds across ``layers`` KDA layers."""
    return int(layers) * int(H) * int(dv) * int(dk)


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, accumulated in fp64."""
    x = np.asarray(x, np.float64).ravel(); ref = np.asarray(ref, np.float64).ravel()
    den = float(np.sqrt(np.dot(ref, ref)))
    num = float(np.sqrt(np.dot(x - ref, x - ref)))
    return num / den if den > 0 else num


def max_abs(x, ref) -> float:
    x = np.asarray(x, np.float64); ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref))) if x.size else 0.0
