"""Pins for the fp64 oracle: it is checked against facts it does not compute itself.

The pins are closed forms the recurrence reduces to (no decay, no update,
one-hot keys, exact recall of a unit key), the product-of-operators form of
the same recurrence, exact rational brute force, structural properties
(linearity, causality, packing), library routines for the front end, and the
numbers the pages print for the state size.  ``test_mutants_are_caught`` plants
a mistake in a copy of the oracle's C source and checks that some pin fails.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import kda_synth as ks

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_inputs(rng, T, H, dk, dv, unit=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, dk))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, b


# ------------------------------------------------------------------------------------------
# pins, written against a token-loop callable so that the mutant test can reuse them
# ------------------------------------------------------------------------------------------

def pin_no_decay_no_update(loop, rng):
    """beta = 0 and g = 0 leave S unchanged, so o_t = S0 q_t."""
    T, H, d = 9, 2, 6
    q, k, v, _, _ = _rand_inputs(rng, T, H, d, d)
    s0 = rng.standard_normal((1, H, d, d))
    o, fs = loop(q, k, v, np.zeros((T, H, d)), np.zeros((T, H)), s0, None, 1.0)
    np.testing.assert_allclose(fs, s0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, np.einsum("hij,thj->thi", s0[0], q), rtol=1e-13, atol=1e-13)


def pin_pure_decay(loop, rng):
    """beta = 0: S_t = S0 Diag(exp(G_t)), G_t the running sum of g; o_t = S0 (exp(G_t) * q_t)."""
    T, H, d = 11, 2, 5
    q, k, v, g, _ = _rand_inputs(rng, T, H, d, d)
    s0 = rng.standard_normal((1, H, d, d))
    scale = 0.37
    o, fs = loop(q, k, v, g, np.zeros((T, H)), s0, None, scale)
    G = np.cumsum(g, axis=0)
    np.testing.assert_allclose(fs[0], s0[0] * np.exp(G[-1])[:, None, :], rtol=1e-12, atol=1e-14)
    ref = scale * np.einsum("hij,thj->thi", s0[0], np.exp(G) * q)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)


def pin_exact_recall(loop, rng):
    """g = 0, beta = 1, ||k_t|| = 1: the update stores v_t under k_t exactly, S_t k_t = v_t.
    With q_t = k_t the output is therefore v_t at every step."""
    T, H, d = 13, 3, 8
    _, k, v, _, _ = _rand_inputs(rng, T, H, d, d)
    s0 = rng.standard_normal((1, H, d, d))
    o, fs = loop(k, k, v, np.zeros((T, H, d)), np.ones((T, H)), s0, None, 1.0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.einsum("hij,hj->hi", fs[0], k[-1]), v[-1], atol=1e-12)


def pin_one_hot_keys(loop, rng):
    """k_t = e_c: column c becomes (1 - beta) alpha_c S[:, c] + beta v_t, every other column j
    is only scaled by alpha_j; o_t = S_t q_t."""
    T, H, dk, dv = 10, 2, 4, 3
    q, _, v, g, b = _rand_inputs(rng, T, H, dk, dv)
    cols = rng.integers(0, dk, size=(T, H))
    k = np.zeros((T, H, dk))
    for t in range(T):
        for h in range(H):
            k[t, h, cols[t, h]] = 1.0
    s0 = rng.standard_normal((1, H, dv, dk))
    scale = 1.3
    o, fs = loop(q, k, v, g, b, s0, None, scale)
    S = s0[0].copy()
    o_ref = np.zeros((T, H, dv))
    for t in range(T):
        for h in range(H):
            a = np.exp(g[t, h])
            c = cols[t, h]
            newS = S[h] * a[None, :]
            newS[:, c] = (1.0 - b[t, h]) * a[c] * S[h][:, c] + b[t, h] * v[t, h]
            S[h] = newS
            o_ref[t, h] = scale * S[h] @ q[t, h]
    np.testing.assert_allclose(fs[0], S, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)


def pin_operator_products(loop, rng):
    """S_t = S_{t-1} M_t + beta_t v_t k_t^T with M_t = Diag(alpha_t)(I - beta_t k_t k_t^T):
    the state after T steps is S0 M_1...M_T + sum_t beta_t v_t k_t^T M_{t+1}...M_T."""
    T, H, dk, dv = 12, 2, 6, 5
    q, k, v, g, b = _rand_inputs(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dv, dk))
    o, fs = loop(q, k, v, g, b, s0, None, 1.0)
    for h in range(H):
        M = [np.diag(np.exp(g[t, h])) @ (np.eye(dk) - b[t, h] * np.outer(k[t, h], k[t, h])) for t in range(T)]
        for t_end in range(1, T + 1):
            P = np.eye(dk)
            acc = np.zeros((dv, dk))
            for t in reversed(range(t_end)):
                acc += b[t, h] * np.outer(v[t, h], k[t, h]) @ P
                P = M[t] @ P
            S = s0[0, h] @ P + acc
            np.testing.assert_allclose(o[t_end - 1, h], S @ q[t_end - 1, h], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(fs[0, h], S, rtol=1e-11, atol=1e-12)


def pin_rational_brute_force(loop, rng):
    """Exact rational arithmetic on tiny shapes (alpha given as a rational, g = ln alpha)."""
    T, dk, dv = 6, 3, 2
    fr = lambda x: Fraction(x).limit_denominator(64)
    alpha = [[fr(rng.uniform(0.05, 1.0)) for _ in range(dk)] for _ in range(T)]
    kk = [[fr(rng.uniform(-1, 1)) for _ in range(dk)] for _ in range(T)]
    qq = [[fr(rng.uniform(-1, 1)) for _ in range(dk)] for _ in range(T)]
    vv = [[fr(rng.uniform(-1, 1)) for _ in range(dv)] for _ in range(T)]
    bb = [fr(rng.uniform(0, 1)) for _ in range(T)]
    S = [[fr(rng.uniform(-1, 1)) for _ in range(dk)] for _ in range(dv)]
    S0 = [row[:] for row in S]
    outs = []
    for t in range(T):
        S = [[S[i][j] * alpha[t][j] for j in range(dk)] for i in range(dv)]
        e = [bb[t] * (vv[t][i] - sum(S[i][j] * kk[t][j] for j in range(dk))) for i in range(dv)]
        S = [[S[i][j] + e[i] * kk[t][j] for j in range(dk)] for i in range(dv)]
        outs.append([sum(S[i][j] * qq[t][j] for j in range(dk)) for i in range(dv)])
    f = lambda m: np.array([[float(x) for x in r] for r in m])
    o, fs = loop(f(qq)[:, None], f(kk)[:, None], f(vv)[:, None], np.log(f(alpha))[:, None],
                 f([bb])[0][:, None], f(S0)[None, None], None, 1.0)
    np.testing.assert_allclose(o[:, 0], f(outs), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(fs[0, 0], f(S), rtol=1e-13, atol=1e-14)


def pin_linearity(loop, rng):
    """For fixed q, k, g, beta the map (S0, V) -> (O, S_T) is linear."""
    T, H, d = 8, 2, 5
    q, k, v1, g, b = _rand_inputs(rng, T, H, d, d)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((1, H, d, d)); s2 = rng.standard_normal((1, H, d, d))
    a1, a2 = 0.7, -1.9
    o1, f1 = loop(q, k, v1, g, b, s1, None, 1.0)
    o2, f2 = loop(q, k, v2, g, b, s2, None, 1.0)
    o3, f3 = loop(q, k, a1 * v1 + a2 * v2, g, b, a1 * s1 + a2 * s2, None, 1.0)
    np.testing.assert_allclose(o3, a1 * o1 + a2 * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f3, a1 * f1 + a2 * f2, rtol=1e-12, atol=1e-12)


PINS = [pin_no_decay_no_update, pin_pure_decay, pin_exact_recall, pin_one_hot_keys, pin_operator_products,
        pin_rational_brute_force, pin_linearity]


def _loop(oracle_mod):
    return lambda q, k, v, g, b, s0, cu, scale: oracle_mod.kda_tokenloop(q, k, v, g, b, s0, cu, scale)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_tokenloop_pins(oracle_mod, pin):
    pin(_loop(oracle_mod), np.random.default_rng(17))


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_chunked_pins(oracle_mod, pin):
    loop = lambda q, k, v, g, b, s0, cu, scale: oracle_mod.kda_chunked(q, k, v, g, b, s0, cu, scale, chunk=4)
    pin(loop, np.random.default_rng(18))


# ------------------------------------------------------------------------------------------
# mutation check: a plausible slip anywhere in the token loop fails at least one pin
# ------------------------------------------------------------------------------------------

MUTANTS = {
    "decay_on_rows": ("S[i * dk + j] *= alpha[j];", "S[i * dk + j] *= alpha[i];"),
    "decay_sign": ("alpha[j] = exp(gt[j]);", "alpha[j] = exp(-gt[j]);"),
    "dropped_beta": ("e[i] = bt * (vt[i] - p);", "e[i] = (vt[i] - p);"),
    "wrong_sign": ("e[i] = bt * (vt[i] - p);", "e[i] = bt * (vt[i] + p);"),
    "transposed_update": ("S[i * dk + j] += e[i] * kt[j];", "S[i * dk + j] += e[j] * kt[i];"),
    "output_reads_key": ("acc += S[i * dk + j] * qt[j];", "acc += S[i * dk + j] * kt[j];"),
    "dropped_scale": ("ot[i] = c->scale * acc;", "ot[i] = acc;"),
}


def _build_mutant(tmp, name, old, new):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "kda_oracle.c")).read()
    # the mutation goes into the token loop's chain function only
    a = src.index("static void tokenloop_chain(")
    z = src.index("\n}\n", a) + 3
    body = src[a:z]
    assert body.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src[:a] + body.replace(old, new) + src[z:])
    so = os.path.join(tmp, f"{name}.so")
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-pthread", "-o", so, path, "-lm"])
    import ctypes
    lib = ctypes.CDLL(so)
    P, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_kda_tokenloop.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, P, P, ctypes.c_int]
    lib.oracle_kda_tokenloop.restype = ctypes.c_int
    return lib


def test_mutants_are_caught(oracle_mod):
    tmp = tempfile.mkdtemp(prefix="kda_mutants_")
    try:
        for name, (old, new) in MUTANTS.items():
            lib = _build_mutant(tmp, name, old, new)
            loop = lambda q, k, v, g, b, s0, cu, scale: oracle_mod._kda(
                lib.oracle_kda_tokenloop, q, k, v, g, b, s0, cu, scale, None, 1)
            caught = []
            for pin in PINS:
                try:
                    pin(loop, np.random.default_rng(17))
                except AssertionError:
                    caught.append(pin.__name__)
            assert caught, f"mutant {name} passed every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


# ------------------------------------------------------------------------------------------
# the two forms, packing, causality, chunk size
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [1, 5, 16, 64])
def test_chunked_equals_tokenloop(oracle_mod, chunk):
    rng = np.random.default_rng(chunk)
    lengths = [1, 63, 64, 65, 130]
    T, H, dk, dv = sum(lengths), 2, 16, 12
    q, k, v, g, b = _rand_inputs(rng, T, H, dk, dv)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    s0 = 0.3 * rng.standard_normal((len(lengths), H, dv, dk))
    o1, f1 = oracle_mod.kda_tokenloop(q, k, v, g, b, s0, cu, 0.5)
    o2, f2 = oracle_mod.kda_chunked(q, k, v, g, b, s0, cu, 0.5, chunk=chunk)
    assert oracle_mod.rel_l2(o2, o1) < 1e-12 and oracle_mod.rel_l2(f2, f1) < 1e-12


def test_packed_equals_separate(oracle_mod):
    rng = np.random.default_rng(3)
    lengths = [5, 17, 1, 9]
    T, H, d = sum(lengths), 2, 8
    q, k, v, g, b = _rand_inputs(rng, T, H, d, d)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    s0 = rng.standard_normal((len(lengths), H, d, d))
    o, fs = oracle_mod.kda_tokenloop(q, k, v, g, b, s0, cu)
    for n in range(len(lengths)):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = oracle_mod.kda_tokenloop(q[sl], k[sl], v[sl], g[sl], b[sl], s0[n:n + 1])
        assert np.array_equal(o1, o[sl]) and np.array_equal(f1[0], fs[n])


def test_causality(oracle_mod):
    rng = np.random.default_rng(4)
    T, H, d = 20, 2, 8
    q, k, v, g, b = _rand_inputs(rng, T, H, d, d)
    o, _ = oracle_mod.kda_tokenloop(q, k, v, g, b)
    t = 11
    k2, v2, g2 = k.copy(), v.copy(), g.copy()
    k2[t:] = rng.standard_normal(k2[t:].shape); v2[t:] += 1.0; g2[t:] *= 0.5
    o2, _ = oracle_mod.kda_tokenloop(q, k2, v2, g2, b)
    assert np.array_equal(o[:t], o2[:t]) and not np.allclose(o[t:], o2[t:])


def test_empty_sequences(oracle_mod):
    rng = np.random.default_rng(5)
    lengths = [0, 4, 0]
    T, H, d = 4, 1, 4
    q, k, v, g, b = _rand_inputs(rng, T, H, d, d)
    s0 = rng.standard_normal((3, H, d, d))
    o, fs = oracle_mod.kda_tokenloop(q, k, v, g, b, s0, np.array([0, 0, 4, 4]))
    assert np.array_equal(fs[0], s0[0]) and np.array_equal(fs[2], s0[2])
    o2, f2 = oracle_mod.kda_chunked(q, k, v, g, b, s0, np.array([0, 0, 4, 4]), chunk=3)
    assert oracle_mod.rel_l2(f2, fs) < 1e-13


def test_state_norm_bound(oracle_mod):
    """alpha <= 1, beta <= 1, ||k|| = 1: ||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t||."""
    rng = np.random.default_rng(6)
    T, H, d = 30, 1, 16
    q, k, v, g, b = _rand_inputs(rng, T, H, d, d)
    s = rng.standard_normal((1, H, d, d))
    for t in range(T):
        _, s_new = oracle_mod.kda_tokenloop(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], s)
        assert np.linalg.norm(s_new) <= np.linalg.norm(s) + b[t, 0] * np.linalg.norm(v[t, 0]) + 1e-12
        s = s_new


def test_state_size_matches_pages(oracle_mod):
    facts = json.load(open(os.path.join(HERE, "golden", "page_facts.json")))
    L, H, d = facts["kda_layers"]["value"], facts["kda_heads"]["value"], facts["kda_head_dim"]["value"]
    n = oracle_mod.state_numel(L, H, d, d)
    assert n == 108_527_616
    assert abs(n / facts["state_values_per_sequence"]["value"] - 1) < facts["state_values_per_sequence"]["rel"]
    assert abs(4 * n / facts["state_bytes_fp32"]["value"] - 1) < facts["state_bytes_fp32"]["rel"]
    assert H * d == facts["inner_width"]["value"]
    assert round(H * d / facts["hidden_size"]["value"], 1) == facts["inner_over_hidden"]["value"]
    # the state does not grow with the context: same size after 3 and after 300 tokens
    rng = np.random.default_rng(7)
    for T in (3, 300):
        q, k, v, g, b = _rand_inputs(rng, T, 1, 8, 8)
        _, fs = oracle_mod.kda_tokenloop(q, k, v, g, b)
        assert fs.shape == (1, 1, 8, 8)


# ------------------------------------------------------------------------------------------
# front end
# ------------------------------------------------------------------------------------------

def _silu(y):
    return y / (1.0 + np.exp(-y))


def test_frontend_matches_numpy_convolve(oracle_mod):
    rng = np.random.default_rng(8)
    T, H, d = 23, 2, 8
    C = H * d
    x = [rng.standard_normal((T, C)) for _ in range(3)]
    w = rng.standard_normal((3 * C, 4))
    q, k, v, cs = oracle_mod.shortconv_silu_l2norm(*x, w, H, d, eps=1e-6)
    outs = []
    for p in range(3):
        a = np.empty((T, C))
        for ch in range(C):
            a[:, ch] = _silu(np.convolve(x[p][:, ch], w[p * C + ch][::-1])[:T])
        outs.append(a.reshape(T, H, d))
    for p, got in ((0, q), (1, k)):
        nrm = np.sqrt((outs[p] ** 2).sum(-1, keepdims=True) + 1e-6)
        np.testing.assert_allclose(got, outs[p] / nrm, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(v, outs[2], rtol=1e-12, atol=1e-14)
    for r in range(3):
        np.testing.assert_array_equal(cs[0, r], np.concatenate([x[0][T - 3 + r], x[1][T - 3 + r], x[2][T - 3 + r]]))


def test_frontend_tap_order_and_silu_value(oracle_mod):
    T, H, d = 6, 1, 2
    C = H * d
    x = np.arange(1.0, T + 1.0)[:, None].repeat(C, 1) / 4.0
    w_old = np.zeros((3 * C, 4)); w_old[:, 0] = 1.0
    w_cur = np.zeros((3 * C, 4)); w_cur[:, 3] = 1.0
    _, _, v_old, _ = oracle_mod.shortconv_silu_l2norm(x, x, x, w_old, H, d)
    _, _, v_cur, _ = oracle_mod.shortconv_silu_l2norm(x, x, x, w_cur, H, d)
    shifted = np.concatenate([np.zeros((3, C)), x[:-3]])
    np.testing.assert_allclose(v_old.reshape(T, C), _silu(shifted), rtol=1e-15)
    np.testing.assert_allclose(v_cur.reshape(T, C), _silu(x), rtol=1e-15)
    one = np.ones((1, C))
    _, _, v1, _ = oracle_mod.shortconv_silu_l2norm(one, one, one, w_cur, H, d)
    assert abs(v1[0, 0, 0] - 0.7310585786300049) < 1e-15   # silu(1) = 1 / (1 + 1/e)


def test_frontend_state_handoff_and_packing(oracle_mod):
    rng = np.random.default_rng(9)
    T, H, d = 19, 2, 4
    C = H * d
    x = [rng.standard_normal((T, C)) for _ in range(3)]
    w = rng.standard_normal((3 * C, 4))
    cs0 = rng.standard_normal((1, 3, 3 * C))
    full = oracle_mod.shortconv_silu_l2norm(*x, w, H, d, conv_state_in=cs0)
    for cut in (1, 2, 3, 7):
        a = oracle_mod.shortconv_silu_l2norm(*(xx[:cut] for xx in x), w, H, d, conv_state_in=cs0)
        b = oracle_mod.shortconv_silu_l2norm(*(xx[cut:] for xx in x), w, H, d, conv_state_in=a[3])
        for i in range(3):
            np.testing.assert_array_equal(np.concatenate([a[i], b[i]]), full[i])
        np.testing.assert_array_equal(b[3], full[3])
    # packed sequences do not see each other's history
    cu = np.array([0, 7, 19])
    cs2 = rng.standard_normal((2, 3, 3 * C))
    packed = oracle_mod.shortconv_silu_l2norm(*x, w, H, d, cu, cs2)
    for n in range(2):
        sl = slice(cu[n], cu[n + 1])
        sep = oracle_mod.shortconv_silu_l2norm(*(xx[sl] for xx in x), w, H, d, conv_state_in=cs2[n:n + 1])
        for i in range(3):
            np.testing.assert_array_equal(sep[i], packed[i][sl])
        np.testing.assert_array_equal(sep[3][0], packed[3][n])


def test_frontend_short_sequence_state(oracle_mod):
    """A sequence shorter than 3 tokens carries part of the incoming state forward."""
    rng = np.random.default_rng(10)
    H, d = 1, 2
    C = H * d
    x = [rng.standard_normal((1, C)) for _ in range(3)]
    w = rng.standard_normal((3 * C, 4))
    cs = rng.standard_normal((1, 3, 3 * C))
    out = oracle_mod.shortconv_silu_l2norm(*x, w, H, d, conv_state_in=cs)[3]
    np.testing.assert_array_equal(out[0, 0], cs[0, 1])
    np.testing.assert_array_equal(out[0, 1], cs[0, 2])
    np.testing.assert_array_equal(out[0, 2], np.concatenate([x[0][0], x[1][0], x[2][0]]))


def test_output_gate_values(oracle_mod):
    o = np.ones((2, 1, 3))
    gate = np.array([[0.0, 50.0, -50.0], [math.log(3.0), 0.0, 0.0]])
    got = oracle_mod.output_gate(o, gate)
    np.testing.assert_allclose(got[0, 0], [0.5, 1.0, 0.0], atol=1e-20)
    assert abs(got[1, 0, 0] - 0.75) < 1e-15


def test_prefill_equals_repeated_decode(oracle_mod):
    """Front end + token loop over T tokens == T decode steps carrying state and conv state."""
    rng = np.random.default_rng(11)
    T, H, d = 7, 2, 4
    C = H * d
    x = [rng.standard_normal((T, C)) for _ in range(3)]
    w = rng.standard_normal((3 * C, 4))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, d))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    s0 = rng.standard_normal((1, H, d, d))
    cs0 = rng.standard_normal((1, 3, 3 * C))
    q, k, v, cs = oracle_mod.shortconv_silu_l2norm(*x, w, H, d, conv_state_in=cs0)
    o, fs = oracle_mod.kda_tokenloop(q, k, v, g, b, s0, None, 0.8)
    s, c = s0, cs0
    for t in range(T):
        ot, s, c = oracle_mod.recurrent_step(x[0][t:t + 1], x[1][t:t + 1], x[2][t:t + 1], w, g[t:t + 1],
                                             b[t:t + 1], s, c, H, d, 0.8)
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(s, fs, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(c, cs)


# ------------------------------------------------------------------------------------------
# the input generator
# ------------------------------------------------------------------------------------------

def test_generator_is_counter_based():
    a = ks.fill(7, 3, ks.NORMAL, (40, 300), "f64")
    b = ks.fill_slice(7, 3, ks.NORMAL, 300, 5, 10, 128, 64, "f64")
    assert np.array_equal(a[5:15, 128:192], b)
    c = ks.fill(7, 3, ks.NORMAL, (40, 300), "f64", threads=1)
    assert np.array_equal(a, c)
    assert abs(a.mean()) < 0.02 and abs(a.std() - 1) < 0.02


def test_generator_distributions():
    z = ks.fill(1, 4, ks.NEG5_SIGMOID, (200, 128), "f32")
    assert z.min() >= -5.0 and z.max() <= 0.0 and abs(z.mean() + 2.5) < 0.05
    z = ks.fill(1, 4, ks.NEG_SOFTPLUS5, (200, 128), "f32")
    assert z.min() >= -5.0 and z.max() <= 0.0
    u = ks.fill(1, 1, ks.UNIT_GROUPS, (10, 4, 128), "f64", p1=128.0)
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, rtol=1e-14)
    bf = ks.fill(1, 1, ks.NORMAL, (10, 64), "bf16")
    f = ks.fill(1, 1, ks.NORMAL, (10, 64), "f32")
    assert np.array_equal(bf, ks.f32_to_bf16(f))
    lens = ks.varlen_lengths(53004, 32)
    assert len(lens) == 32 and min(lens) >= 1024 and max(lens) <= 32768
