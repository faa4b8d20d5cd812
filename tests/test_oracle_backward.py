"""Pins for the oracle's backward (reverse mode through the token loop): checked against
central finite differences of the forward, against the transition operator of a segment, against
closed forms of the no-update case and against linearity in the upstream gradients."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _inputs(rng, lengths, H, dk, dv, decay=0.2):
    T = sum(lengths)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -decay * 5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, dk))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    s0 = 0.5 * rng.standard_normal((len(lengths), H, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, g, b, s0, cu


def _central_differences(orc, bwd):
    """L = sum(o * Wo) + sum(S_end * Ws); every input element perturbed by +-h in fp64 and compared
    with bwd's gradients (AssertionError on the first mismatch)."""
    rng = np.random.default_rng(11)
    lengths, H, dk, dv, scale = [3, 0, 5], 2, 5, 4, 0.7
    q, k, v, g, b, s0, cu = _inputs(rng, lengths, H, dk, dv)
    Wo = rng.standard_normal((sum(lengths), H, dv))
    Ws = rng.standard_normal(s0.shape)

    def loss(q, k, v, g, b, s0):
        o, fs = orc.kda_tokenloop(q, k, v, g, b, s0, cu, scale)
        return float(np.sum(o * Wo) + np.sum(fs * Ws))

    grads = bwd(q, k, v, g, b, Wo, s0, cu, scale, Ws)
    h = 1e-5
    args = [q, k, v, g, b, s0]
    names = ["q", "k", "v", "g", "beta", "S0"]
    for a, (x, gx) in enumerate(zip(args, grads)):
        num = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = list(args), list(args)
            ap[a], am[a] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        assert np.max(np.abs(num)) > 1e-3, names[a]   # the loss depends on every input
        assert np.max(np.abs(gx - num)) <= 1e-7 * (1.0 + np.max(np.abs(num))), names[a]


def test_backward_matches_central_differences(orc):
    _central_differences(orc, lambda *a: orc.kda_tokenloop_bwd(*a[:9], d_final=a[9]))


BWD_MUTANTS = {
    "dq_unscaled": ("dqt[j] += c->scale * s * dot[i];", "dqt[j] += s * dot[i];"),
    "dbeta_drops_prediction": ("db += acc * (vt[i] - p[i]);", "db += acc * vt[i];"),
    "dv_drops_beta": ("dvt[i] = bt * acc;", "dvt[i] = acc;"),
    "dg_reads_wrong_gradient": ("dgt[j] += sb * st[i * dk + j];", "dgt[j] += Sb[i * dk + j] * st[i * dk + j];"),
    "gradient_not_decayed": ("Sb[i * dk + j] = sb * alpha[j];", "Sb[i * dk + j] = sb;"),
    "dk_drops_prediction_path": ("dkt[j] += st[i * dk + j] * pb;", "dkt[j] -= st[i * dk + j] * pb;"),
    "output_gradient_transposed": ("Sb[i * dk + j] += c->scale * dot[i] * qt[j];",
                                   "Sb[i * dk + j] += c->scale * dot[j % dv] * qt[i % dk];"),
}


def test_backward_mutants_are_caught(orc):
    """A plausible slip in the reverse pass (planted in a copy of the oracle's C source) fails the
    central-difference pin."""
    import ctypes
    import os
    import shutil
    import subprocess
    import tempfile
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                            "kda_oracle.c")).read()
    a = src.index("static void tokenloop_bwd_chain(")
    z = src.index("\n}\n", a) + 3
    body = src[a:z]
    tmp = tempfile.mkdtemp(prefix="kda_bwd_mutants_")
    try:
        for name, (old, new) in BWD_MUTANTS.items():
            assert body.count(old) == 1, name
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(src[:a] + body.replace(old, new) + src[z:])
            so = os.path.join(tmp, f"{name}.so")
            subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-pthread", "-o", so, path, "-lm"])
            lib = ctypes.CDLL(so)
            P, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            lib.oracle_kda_tokenloop_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, P, P, P, P, P, P, P, P,
                                                     ctypes.c_int]
            lib.oracle_kda_tokenloop_bwd.restype = ctypes.c_int
            fn = lib.oracle_kda_tokenloop_bwd
            with pytest.raises(AssertionError):
                _central_differences(orc, lambda *x: orc._bwd(fn, *x, 1))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_backward_initial_state_through_the_transition(orc):
    """With do = 0 the gradient reaching S0 is dS_end M^T, M the segment's product of
    Diag(alpha_t)(I - beta_t k_t k_t^T), formed by the oracle's literal operator product."""
    rng = np.random.default_rng(12)
    lengths, H, dk, dv = [7, 2], 2, 6, 5
    q, k, v, g, b, s0, cu = _inputs(rng, lengths, H, dk, dv, decay=0.1)
    dfin = rng.standard_normal(s0.shape)
    *_, ds0 = orc.kda_tokenloop_bwd(q, k, v, g, b, np.zeros_like(v), s0, cu, 1.0, d_final=dfin)
    M = orc.transition(k, g, b, cu)
    ref = np.einsum("nhij,nhkj->nhik", dfin, M)
    assert np.max(np.abs(ds0 - ref)) <= 1e-12 * (1.0 + np.max(np.abs(ref)))


def test_backward_without_updates_closed_form(orc):
    """beta = 0 and g = 0: S_t = S0 for every t, o_t = scale S0 q_t.  Then dq_t = scale S0^T do_t,
    dv = dk = 0, dS0 = dS_end + scale sum_t do_t q_t^T, and with Sb_t = dS_end + scale
    sum_{s >= t} do_s q_s^T:  dbeta_t = (Sb_t k_t) . (v_t - S0 k_t),  dg_t[j] = sum_i Sb_t[i][j] S0[i][j]."""
    rng = np.random.default_rng(13)
    T, H, dk, dv, scale = 6, 1, 4, 3, 0.5
    q, k, v, _, _, s0, _ = _inputs(rng, [T], H, dk, dv)
    g, b = np.zeros((T, H, dk)), np.zeros((T, H))
    do = rng.standard_normal((T, H, dv))
    dfin = rng.standard_normal(s0.shape)
    dq, dk_, dv_, dg, db, ds0 = orc.kda_tokenloop_bwd(q, k, v, g, b, do, s0, None, scale, d_final=dfin)
    S0 = s0[0, 0]
    assert np.allclose(dq[:, 0], scale * do[:, 0] @ S0, atol=1e-13)
    assert np.all(dk_ == 0) and np.all(dv_ == 0)
    Sb = dfin[0, 0].copy()
    for t in range(T - 1, -1, -1):
        Sb += scale * np.outer(do[t, 0], q[t, 0])
        assert abs(db[t, 0] - (Sb @ k[t, 0]) @ (v[t, 0] - S0 @ k[t, 0])) <= 1e-12
        assert np.allclose(dg[t, 0], np.sum(Sb * S0, axis=0), atol=1e-12)
    assert np.allclose(ds0[0, 0], Sb, atol=1e-12)


def test_backward_is_linear_in_the_upstream_gradients(orc):
    rng = np.random.default_rng(14)
    lengths, H, dk, dv = [9, 4], 2, 6, 5
    q, k, v, g, b, s0, cu = _inputs(rng, lengths, H, dk, dv)
    d1, d2 = rng.standard_normal(v.shape), rng.standard_normal(v.shape)
    f1, f2 = rng.standard_normal(s0.shape), rng.standard_normal(s0.shape)
    g1 = orc.kda_tokenloop_bwd(q, k, v, g, b, d1, s0, cu, 1.0, d_final=f1)
    g2 = orc.kda_tokenloop_bwd(q, k, v, g, b, d2, s0, cu, 1.0, d_final=f2)
    g3 = orc.kda_tokenloop_bwd(q, k, v, g, b, 2.0 * d1 - 3.0 * d2, s0, cu, 1.0, d_final=2.0 * f1 - 3.0 * f2)
    for a, b_, c in zip(g1, g2, g3):
        assert np.allclose(c, 2.0 * a - 3.0 * b_, atol=1e-11)


def test_backward_across_recompute_blocks(orc):
    """A chain of 150 tokens crosses the oracle's 64-token recompute blocks; sampled elements of every
    gradient against central differences."""
    rng = np.random.default_rng(15)
    lengths, H, dk, dv = [150, 70], 1, 4, 3
    q, k, v, g, b, s0, cu = _inputs(rng, lengths, H, dk, dv, decay=0.02)
    Wo = rng.standard_normal((sum(lengths), H, dv))
    Ws = rng.standard_normal(s0.shape)

    def loss(*a):
        o, fs = orc.kda_tokenloop(*a, cu, 1.0)
        return float(np.sum(o * Wo) + np.sum(fs * Ws))

    args = [q, k, v, g, b, s0]
    grads = orc.kda_tokenloop_bwd(q, k, v, g, b, Wo, s0, cu, 1.0, d_final=Ws)
    h = 1e-5
    for a, (x, gx) in enumerate(zip(args, grads)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = list(args), list(args)
            ap[a], am[a] = xp, xm
            num = (loss(*ap) - loss(*am)) / (2 * h)
            assert abs(gx[idx] - num) <= 1e-7 * (1.0 + abs(num)), (a, idx)


@pytest.mark.parametrize("chunk", [1, 5, 16, 64])
def test_chunked_backward_equals_token_loop(orc, chunk):
    """The chunk form's chain rule (the GPU backward's algebra) against reverse mode through the token
    loop: ragged packed sequences (1, 63, 64, 65, 130 tokens and an empty one), decays of both strengths."""
    rng = np.random.default_rng(30 + chunk)
    lengths, H, dk, dv = [1, 63, 0, 64, 65, 130], 2, 8, 6
    for decay in (1.0, 0.05):
        q, k, v, g, b, s0, cu = _inputs(rng, lengths, H, dk, dv, decay=decay)
        do = rng.standard_normal(v.shape)
        dfin = rng.standard_normal(s0.shape)
        ref = orc.kda_tokenloop_bwd(q, k, v, g, b, do, s0, cu, 0.7, d_final=dfin)
        got = orc.kda_chunked_bwd(q, k, v, g, b, do, s0, cu, 0.7, d_final=dfin, chunk=chunk)
        for name, x, r in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, ref):
            assert orc.rel_l2(x, r) < 1e-12, (name, decay)
