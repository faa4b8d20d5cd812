"""GPU parity of kda_chunk_bwd (through its C ABI) against the oracle's reverse mode through the
token loop, on the same seeded inputs.

The backward computes from the same input bits as the oracle (bf16 or fp32 storage) with fp32-level
accuracy: fp32 on the CUDA cores for fp32 inputs; for bf16 inputs on the tensor cores with every fp32
operand split into bf16 pieces (hi + lo, three pieces in the position-pair sums).  Every gradient is held
to rel-L2 <= 1e-4 over the whole tensor, the bound of the fp32 forward; an fp32 emulation of the chunked
algorithm gives 1e-7 .. 3e-6.
"""
import math

import numpy as np
import pytest

import kda_synth as ks

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REL = 1e-4
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as m
    return m


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def dev(a):
    from kda_synth.device import to_device
    return to_device(a)


def host(t):
    from kda_synth.device import to_host_f64
    return to_host_f64(t)


def case(seed, lengths, H, dtype, init_std=0.02, g_kind=ks.NEG5_SIGMOID, with_final=True):
    w = ks.Workload("bwd", "prefill", seed, H=H, lengths=list(lengths), dtype=dtype, g_kind=g_kind,
                    init_state_std=init_std)
    q, k, v, g, b = w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta()
    s0 = w.init_state() if init_std > 0 else None
    do = ks.fill(seed, ks.TID_DO, ks.NORMAL, (w.T, H, 128), dtype)
    dfin = ks.fill(seed, ks.TID_DSTATE, ks.NORMAL, (w.N, H, 128, 128), "f32") if with_final else None
    return w, [q, k, v, g, b, do, s0, dfin]


def run_and_check(kda, orc, w, arrays, scale=1.0):
    q, k, v, g, b, do, s0, dfin = arrays
    cu = w.cu_seqlens() if w.N > 1 else None
    got = kda.kda_chunk_bwd(dev(q), dev(k), dev(v), dev(g), dev(b), dev(do),
                            init_state=None if s0 is None else dev(s0),
                            cu_seqlens=None if cu is None else dev(cu),
                            d_final_state=None if dfin is None else dev(dfin), scale=scale)
    torch.cuda.synchronize()
    ref = orc.kda_tokenloop_bwd(ks.to_f64(q), ks.to_f64(k), ks.to_f64(v), g, b, ks.to_f64(do), s0, cu, scale,
                                d_final=dfin)
    for name, x, r in zip(NAMES, got, ref):
        err = orc.rel_l2(host(x), r)
        assert err <= REL, f"{name}: rel-L2 {err:.3e}"
    assert kda.device_error() == 0
    return got


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_ragged_varlen_with_state_and_scale(kda, orc, dtype):
    """Packed sequences of 1, 63, 64, 65, 130, 0 and 7 tokens (partial chunks, an empty sequence),
    initial states, dL/dS_final, scale d^-1/2."""
    w, arrays = case(201, [1, 63, 64, 65, 130, 0, 7], 3, dtype)
    got = run_and_check(kda, orc, w, arrays, scale=1.0 / math.sqrt(128))
    # the empty sequence passes dL/dS_final straight to dL/dS0
    assert torch.equal(got[5][5], dev(arrays[7])[5])


def test_bwd_packed_sequences_many_chunks(kda, orc):
    """Five packed sequences of 1 to 2,000 tokens with initial states and dL/dS_final (bf16): the chain
    passes store whole chunks by TMA and each sequence's partial last chunk row by row, the reverse pass
    prefetches two chunks ahead through sequences of up to 32 chunks, and the per-chunk kernel runs chunks
    at every position of a sequence."""
    w, arrays = case(5307, [700, 1, 1300, 64, 2000], 4, "bf16")
    run_and_check(kda, orc, w, arrays, scale=1.0 / math.sqrt(128))


def test_bwd_single_sequence_without_state(kda, orc):
    """One sequence of 300 tokens, no initial state, no gradient of the final state."""
    w, arrays = case(202, [300], 2, "bf16", init_std=0.0, with_final=False)
    run_and_check(kda, orc, w, arrays)


@pytest.mark.parametrize("kind", ["no_decay", "floor", "beta0", "beta1"])
def test_bwd_degenerate_gates_and_betas(kda, orc, kind):
    w, arrays = case(203, [200, 64, 1], 2, "f32")
    g, b = arrays[3], arrays[4]
    if kind == "no_decay":
        arrays[3] = np.zeros_like(g)
    elif kind == "floor":
        arrays[3] = np.full_like(g, -5.0)
    elif kind == "beta0":
        arrays[4] = np.zeros_like(b)
    else:
        arrays[4] = np.ones_like(b)
    run_and_check(kda, orc, w, arrays)


def test_bwd_deterministic(kda):
    w, arrays = case(204, [129, 3], 2, "bf16")
    q, k, v, g, b, do, s0, dfin = [dev(a) for a in arrays]
    cu = dev(w.cu_seqlens())
    g1 = kda.kda_chunk_bwd(q, k, v, g, b, do, init_state=s0, cu_seqlens=cu, d_final_state=dfin)
    g2 = kda.kda_chunk_bwd(q, k, v, g, b, do, init_state=s0, cu_seqlens=cu, d_final_state=dfin)
    torch.cuda.synchronize()
    for a, c in zip(g1, g2):
        assert torch.equal(a, c)


def test_bwd_prefill_8k_sampled_heads(kda, orc):
    """The 8K-token, 96-head bf16 prefill's backward as the benchmark launches it; heads 0 and 95
    checked in full against the oracle."""
    w = ks.workload("prefill_8k")
    T, H, d = w.T, w.H, w.d
    from kda_synth.device import fill_device
    fd = lambda tid, kind, shape, dtype, p1=1.0: fill_device(w.seed, tid, kind, shape, dtype, 0.0, p1)
    q = fd(ks.TID_Q, ks.UNIT_GROUPS, (T, H, d), "bf16", float(d))
    k = fd(ks.TID_K, ks.UNIT_GROUPS, (T, H, d), "bf16", float(d))
    v = fd(ks.TID_V, ks.NORMAL, (T, H, d), "bf16")
    g = fd(ks.TID_G, w.g_kind, (T, H, d), "f32")
    b = fd(ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    do = fd(ks.TID_DO, ks.NORMAL, (T, H, d), "bf16")
    got = kda.kda_chunk_bwd(q, k, v, g, b, do)
    torch.cuda.synchronize()
    for x in got[:5]:
        assert torch.isfinite(x).all()
    for h in (0, 95):
        rows = lambda tid, kind, dtype, p1=1.0: w.head_rows(tid, kind, h, dtype, p1=p1)
        qh = ks.to_f64(rows(ks.TID_Q, ks.UNIT_GROUPS, "bf16", float(d)))[:, None]
        kh = ks.to_f64(rows(ks.TID_K, ks.UNIT_GROUPS, "bf16", float(d)))[:, None]
        vh = ks.to_f64(rows(ks.TID_V, ks.NORMAL, "bf16"))[:, None]
        gh = rows(ks.TID_G, w.g_kind, "f32").astype(np.float64)[:, None]
        bh = w.head_beta(h).astype(np.float64)[:, None]
        doh = ks.to_f64(rows(ks.TID_DO, ks.NORMAL, "bf16"))[:, None]
        ref = orc.kda_tokenloop_bwd(qh, kh, vh, gh, bh, doh)
        for name, x, r in zip(NAMES, got, ref):
            err = orc.rel_l2(host(x[:, h:h + 1]), r)
            assert err <= REL, f"head {h} {name}: rel-L2 {err:.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_many_short_sequences(kda, orc, dtype):
    """400 packed sequences of 0 to 70 tokens with initial states and dL/dS_final: the per-chunk kernels'
    slot lookup over many sequences (one or two chunks each, empty ones among them), the chain passes'
    400 x 2 chains; every gradient within 1e-4 of the oracle's reverse mode."""
    rng = np.random.default_rng(121)
    lengths = [int(x) for x in rng.integers(0, 71, size=400)]
    lengths[0], lengths[1], lengths[2] = 0, 64, 65
    w, arrays = case(121, lengths, 2, dtype)
    got = run_and_check(kda, orc, w, arrays)
    # an empty sequence passes dL/dS_final straight through to dL/dS0
    dfin = dev(arrays[7])
    empty = [n for n, L in enumerate(lengths) if L == 0]
    assert len(empty) > 2 and all(torch.equal(got[5][n], dfin[n]) for n in empty)
