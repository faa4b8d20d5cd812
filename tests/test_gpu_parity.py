"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on the same
seeded inputs.

Tolerances (element by element over whole tensors unless noted):
  * bf16 prefill and decode: o rel-L2 <= 5e-3 and max-abs <= 2e-2, state rel-L2 <= 5e-3.
  * fp32 prefill: rel-L2 <= 1e-4 on o and on the final state.
  * conv_state: bit-exact (it is a copy of raw inputs).
  * front end: fp32 outputs rel-L2 <= 1e-5 (fp32 arithmetic on bf16 inputs, a handful
    of roundings per element); bf16 outputs rel-L2 <= 5e-3 and max relative error per
    element <= 2^-8 + 1e-5 (one bf16 rounding, 2^-9, plus fp32 noise).
The oracle consumes exactly the bits the GPU receives, widened to fp64.
"""
import math

import numpy as np
import pytest

import kda_synth as ks

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_O_REL, BF16_O_ABS, BF16_S_REL = 5e-3, 2e-2, 5e-3
F32_REL = 1e-4


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


def small_prefill(seed, lengths, H, dtype, init_std=0.0, g_kind=ks.NEG5_SIGMOID):
    w = ks.Workload("small", "prefill", seed, H=H, lengths=list(lengths), dtype=dtype, g_kind=g_kind,
                    init_state_std=init_std)
    q, k, v, g, b = w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta()
    s0 = w.init_state()
    return w, q, k, v, g, b, s0


def run_chunk(kda, w, q, k, v, g, b, s0, scale=1.0, gate=None):
    cu = dev(w.cu_seqlens()) if w.N > 1 else None
    o, fs = kda.kda_chunk_fwd(dev(q), dev(k), dev(v), dev(g), dev(b), None if s0 is None else dev(s0), cu,
                              scale=scale, out_gate=None if gate is None else dev(gate))
    torch.cuda.synchronize()
    return o, fs


def oracle_chunk(orc, w, q, k, v, g, b, s0, scale=1.0, gate=None):
    cu = w.cu_seqlens() if w.N > 1 else None
    o, fs = orc.kda_tokenloop(ks.to_f64(q), ks.to_f64(k), ks.to_f64(v), g, b, s0, cu, scale)
    if gate is not None:
        o = orc.output_gate(o, ks.to_f64(gate))
    return o, fs


# ------------------------------------------------------------------------------------------
# kda_chunk_fwd
# ------------------------------------------------------------------------------------------

def test_chunk_fp32_tiny_workload(kda, orc):
    """The tiny fp32 workload: H=4, T=256, chunk 64, zero initial state."""
    w = ks.workload("tiny_fp32")
    q, k, v, g, b = w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta()
    o, fs = run_chunk(kda, w, q, k, v, g, b, None)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, None)
    assert orc.rel_l2(host(o), o_ref) <= F32_REL
    assert orc.rel_l2(host(fs), fs_ref) <= F32_REL


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_ragged_varlen_with_state_and_scale(kda, orc, dtype):
    lengths = [1, 63, 64, 65, 130, 0, 7]
    w, q, k, v, g, b, s0 = small_prefill(101, lengths, 3, dtype, init_std=0.02)
    scale = 1.0 / math.sqrt(128)
    o, fs = run_chunk(kda, w, q, k, v, g, b, s0, scale=scale)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0, scale=scale)
    if dtype == "f32":
        assert orc.rel_l2(host(o), o_ref) <= F32_REL and orc.rel_l2(host(fs), fs_ref) <= F32_REL
    else:
        assert orc.rel_l2(host(o), o_ref) <= BF16_O_REL and orc.max_abs(host(o), o_ref) <= BF16_O_ABS
        assert orc.rel_l2(host(fs), fs_ref) <= BF16_S_REL
    # the empty sequence keeps its initial state exactly
    assert torch.equal(fs[5], dev(s0)[5])


def test_chunk_many_short_sequences(kda, orc):
    """1,500 packed sequences of 0 to 70 tokens (bf16, initial states): the chunk offsets' scan runs over
    more than 1,024 sequences (its carry across passes), the state pass runs 3,000 chains in waves, and the
    2,500 or so chunk rows go through the overlapped ranges.  Against the oracle's token loop, and the
    empty sequences keep their initial states exactly."""
    rng = np.random.default_rng(119)
    lengths = [int(x) for x in rng.integers(0, 71, size=1500)]
    lengths[0], lengths[1], lengths[2] = 0, 64, 65
    w, q, k, v, g, b, s0 = small_prefill(119, lengths, 2, "bf16", init_std=0.02)
    assert w.T // 64 + w.N >= 256
    o, fs = run_chunk(kda, w, q, k, v, g, b, s0)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0)
    assert orc.rel_l2(host(o), o_ref) <= BF16_O_REL and orc.max_abs(host(o), o_ref) <= BF16_O_ABS
    assert orc.rel_l2(host(fs), fs_ref) <= BF16_S_REL
    empty = [n for n, L in enumerate(lengths) if L == 0]
    assert len(empty) > 5 and all(torch.equal(fs[n], dev(s0)[n]) for n in empty)
    assert kda.device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_output_gate(kda, orc, dtype):
    w, q, k, v, g, b, s0 = small_prefill(102, [200], 2, dtype, g_kind=ks.NEG_SOFTPLUS5)
    gate = ks.fill(102, ks.TID_GATE, ks.NORMAL, (w.T, w.H * w.d), "bf16")
    o, fs = run_chunk(kda, w, q, k, v, g, b, None, gate=gate)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, None, gate=gate)
    tol = F32_REL if dtype == "f32" else BF16_O_REL
    assert orc.rel_l2(host(o), o_ref) <= tol and orc.rel_l2(host(fs), fs_ref) <= tol


def test_chunk_output_gate_extremes(kda, orc):
    """The bf16 path's gated epilogue, o / (1 + e^-gate) with the fast divide, at gate values whose sigmoid is
    0 to fp32 (-100: the divisor passes 2^126 and the quotient is 0), tiny (-20), 1/2 (0), near 1 (20) and 1
    (100), mixed with N(0, 4) values; packed sequences with whole and partial chunks (both ways the gate
    values are loaded).  Against the oracle's o * sigmoid(gate), elementwise within the bf16 bounds."""
    w, q, k, v, g, b, s0 = small_prefill(118, [200, 64, 37], 2, "bf16", init_std=0.02)
    z = ks.bf16_to_f64(ks.fill(118, ks.TID_GATE, ks.NORMAL, (w.T, w.H * w.d), "bf16")) * 2.0
    special = np.array([-100.0, -20.0, 0.0, 20.0, 100.0])
    pick = (np.arange(z.size).reshape(z.shape) % 7)
    z = np.where(pick < 5, special[np.minimum(pick, 4)], z)
    gate = ks.f32_to_bf16(z.astype(np.float32))
    o, fs = run_chunk(kda, w, q, k, v, g, b, s0, gate=gate)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0, gate=gate)
    assert orc.rel_l2(host(o), o_ref) <= BF16_O_REL and orc.max_abs(host(o), o_ref) <= BF16_O_ABS
    assert orc.rel_l2(host(fs), fs_ref) <= BF16_S_REL
    # where sigma(gate) is 0 to fp32 the output is exactly zero
    o_h = host(o).reshape(w.T, -1)
    assert np.all(o_h[z.reshape(w.T, -1) == -100.0] == 0.0)
    assert kda.device_error() == 0


def test_chunk_final_state_may_alias_initial(kda, orc):
    w, q, k, v, g, b, s0 = small_prefill(103, [70, 5], 2, "f32", init_std=0.02)
    s = dev(s0)
    o, fs = kda.kda_chunk_fwd(dev(q), dev(k), dev(v), dev(g), dev(b), s, dev(w.cu_seqlens()), final_state=s)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0)
    assert orc.rel_l2(host(s), fs_ref) <= F32_REL


def test_chunk_every_output_written_and_deterministic(kda):
    w, q, k, v, g, b, s0 = small_prefill(104, [129, 3], 2, "bf16", init_std=0.02)
    args = [dev(x) for x in (q, k, v, g, b, s0)]
    o1 = torch.full((w.T, w.H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    f1 = torch.full((2, w.H, 128, 128), float("nan"), device="cuda")
    kda.kda_chunk_fwd(*args, dev(w.cu_seqlens()), o=o1, final_state=f1)
    o2, f2 = kda.kda_chunk_fwd(*args, dev(w.cu_seqlens()))
    torch.cuda.synchronize()
    assert not torch.isnan(o1).any() and not torch.isnan(f1).any()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_chunk_causality(kda):
    w, q, k, v, g, b, s0 = small_prefill(105, [150], 2, "bf16")
    o1, _ = run_chunk(kda, w, q, k, v, g, b, None)
    v2 = v.copy()
    v2[90:] = ks.f32_to_bf16(ks.bf16_to_f32(v2[90:]) + 1.0)
    o2, _ = run_chunk(kda, w, q, k, v2, g, b, None)
    assert torch.equal(o1[:90], o2[:90]) and not torch.equal(o1[90:], o2[90:])


def test_chunk_packed_equals_separate(kda):
    lengths = [33, 64, 100]
    w, q, k, v, g, b, s0 = small_prefill(106, lengths, 2, "bf16", init_std=0.02)
    o, fs = run_chunk(kda, w, q, k, v, g, b, s0)
    cu = w.cu_seqlens()
    for n in range(len(lengths)):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = kda.kda_chunk_fwd(dev(q[sl]), dev(k[sl]), dev(v[sl]), dev(g[sl]), dev(b[sl]), dev(s0[n:n + 1]))
        assert torch.equal(o1, o[sl]) and torch.equal(f1[0], fs[n])


DEGENERATE = ("no_decay", "floor", "mixed_channels", "beta0", "beta1", "repeated_key")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", DEGENERATE)
def test_chunk_degenerate_gates_and_betas(kda, orc, case, dtype):
    """The method's limiting cases, each against the oracle on the same bits:
    no_decay (g = 0: the plain delta rule), floor (g = -5 everywhere: a 16-token block spans the
    full e^75 of the split intra-chunk factor), mixed_channels (per key channel g is 0 or -5: some
    channels never forget, the rest forget at once), beta0 (no writes: the state only decays),
    beta1 (full overwrite along k), repeated_key (one key for a whole sequence, beta = 1: every
    off-diagonal entry of A_kk is 1 and T = (I + A_kk)^-1 is bidiagonal)."""
    lengths = [200, 64, 1, 130]
    w, q, k, v, g, b, s0 = small_prefill(110, lengths, 2, dtype, init_std=0.02)
    T, H, d = w.T, w.H, w.d
    cu = w.cu_seqlens()
    if case == "no_decay":
        g = np.zeros_like(g)
    elif case == "floor":
        g = np.full_like(g, -5.0)
    elif case == "mixed_channels":
        mask = (ks.u64(110, ks.TID_G, 0, H * d) & 1).astype(bool).reshape(H, d)
        g = np.broadcast_to(np.where(mask, np.float32(-5.0), np.float32(0.0)), g.shape).copy()
    elif case == "beta0":
        g = np.full_like(g, -0.02)
        b = np.zeros_like(b)
    elif case == "beta1":
        b = np.ones_like(b)
    elif case == "repeated_key":
        g = np.zeros_like(g)
        b = np.ones_like(b)
        k = k.copy()
        for n in range(w.N):
            k[cu[n]:cu[n + 1]] = k[cu[n]]
    o, fs = run_chunk(kda, w, q, k, v, g, b, s0)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0)
    if dtype == "f32":
        assert orc.rel_l2(host(o), o_ref) <= F32_REL and orc.rel_l2(host(fs), fs_ref) <= F32_REL
    else:
        assert orc.rel_l2(host(o), o_ref) <= BF16_O_REL and orc.max_abs(host(o), o_ref) <= BF16_O_ABS
        assert orc.rel_l2(host(fs), fs_ref) <= BF16_S_REL
    assert kda.device_error() == 0


@pytest.mark.parametrize("rows", [1, 3])
def test_chunk_workspace_ranges(kda, orc, rows):
    """A workspace of `rows` chunk rows runs the chunks in ranges; chains that cross a range carry
    their fp32 state through the workspace.  The result is bit-identical to one range and matches
    the oracle."""
    lengths = [130, 1, 0, 257, 64, 5, 0, 70]
    w, q, k, v, g, b, s0 = small_prefill(107, lengths, 3, "bf16", init_std=0.02)
    args = [dev(x) for x in (q, k, v, g, b, s0)] + [dev(w.cu_seqlens())]
    o_full, f_full = kda.kda_chunk_fwd(*args)
    full, least = kda.kda_chunk_fwd_workspace_size(w.N, w.T, w.H)
    per_row = (full - least) // (w.T // 64 + w.N - 1)
    ws = torch.empty(least + (rows - 1) * per_row, dtype=torch.uint8, device="cuda")
    o_r, f_r = kda.kda_chunk_fwd(*args, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o_r, o_full) and torch.equal(f_r, f_full)
    o_ref, fs_ref = oracle_chunk(orc, w, q, k, v, g, b, s0)
    assert orc.rel_l2(host(o_r), o_ref) <= BF16_O_REL and orc.max_abs(host(o_r), o_ref) <= BF16_O_ABS
    assert orc.rel_l2(host(f_r), fs_ref) <= BF16_S_REL
    assert torch.equal(f_r[2], dev(s0)[2]) and torch.equal(f_r[6], dev(s0)[6])
    assert kda.device_error() == 0


@pytest.mark.parametrize("rows", [None, 2])
def test_chunk_frontend_fused_equals_two_passes(kda, orc, rows):
    """kda_chunk_fwd_frontend = kda_shortconv_l2norm (bf16) + kda_chunk_fwd, bit for bit: packed
    sequences (one empty, two shorter than the 3-token history), carried conv state in and out, an
    initial state, the output gate, a row stride wider than H*d; also with a workspace of 2 chunk rows.
    Spot check against the oracle's front end + token loop."""
    H, d = 2, 128
    C = H * d
    lengths = [70, 2, 0, 130, 1, 64]
    T, N = sum(lengths), len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    width = C + 16
    xs = [ks.fill(109, tid, ks.NORMAL, (T, width), "bf16") for tid in (1, 2, 3)]
    cw = ks.fill(109, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25)
    cs = ks.fill(109, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16")
    g = ks.fill(109, ks.TID_G, ks.NEG5_SIGMOID, (T, H, d), "f32")
    b = ks.fill(109, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    s0 = ks.fill(109, ks.TID_STATE, ks.NORMAL, (N, H, d, d), "f32", 0.0, 0.02)
    gate = ks.fill(109, ks.TID_GATE, ks.NORMAL, (T, C), "bf16")
    xd = [dev(x) for x in xs]
    cu_d = dev(cu)
    # two passes
    cs_a = torch.empty((N, 3, 3 * C), dtype=torch.bfloat16, device="cuda")
    q, k, v = kda.kda_shortconv_l2norm(*xd, dev(cw), H, cu_d, dev(cs), cs_a)
    o1, f1 = kda.kda_chunk_fwd(q, k, v, dev(g), dev(b), dev(s0), cu_d, scale=0.5, out_gate=dev(gate))
    # fused
    ws = None
    if rows is not None:
        full, least = kda.kda_chunk_fwd_workspace_size(N, T, H)
        per_row = (full - least) // (T // 64 + N - 1)
        ws = torch.empty(least + (rows - 1) * per_row, dtype=torch.uint8, device="cuda")
    cs_b = dev(cs)  # in place: conv_state_out aliases conv_state_in
    o2, f2 = kda.kda_chunk_fwd_frontend(*xd, dev(cw), dev(g), dev(b), H, dev(s0), cu_d, conv_state_in=cs_b,
                                        conv_state_out=cs_b, scale=0.5, out_gate=dev(gate), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2) and torch.equal(cs_a, cs_b)
    assert kda.device_error() == 0
    # sequence 3 (130 tokens), head 1, against the oracle
    n, h = 3, 1
    t0, t1 = int(cu[n]), int(cu[n + 1])
    sel = lambda x: ks.to_f64(x)[t0:t1, h * d:(h + 1) * d]
    wh = np.concatenate([ks.to_f64(cw)[p * C + h * d: p * C + (h + 1) * d] for p in range(3)])
    csh = np.concatenate([ks.to_f64(cs)[n:n + 1, :, p * C + h * d: p * C + (h + 1) * d] for p in range(3)], axis=2)
    fq, fk, fv = orc.shortconv_silu_l2norm(sel(xs[0]), sel(xs[1]), sel(xs[2]), wh, 1, d, None, csh,
                                           want_state=False)[:3]
    rq, rk, rv = (ks.bf16_to_f64(ks.f32_to_bf16(x.astype(np.float32))) for x in (fq, fk, fv))
    o_ref, f_ref = orc.kda_tokenloop(rq, rk, rv, g[t0:t1, h:h + 1].astype(np.float64),
                                     b[t0:t1, h:h + 1].astype(np.float64), s0[n:n + 1, h:h + 1].astype(np.float64),
                                     None, 0.5)
    o_ref = orc.output_gate(o_ref, ks.to_f64(gate)[t0:t1, h * d:(h + 1) * d])
    assert orc.rel_l2(host(o2[t0:t1, h:h + 1]), o_ref) <= BF16_O_REL
    assert orc.rel_l2(host(f2[n:n + 1, h:h + 1]), f_ref) <= BF16_S_REL


def test_chunk_frontend_fused_packed_overlapped_equals_two_passes(kda):
    """The fused prefill on packed sequences with enough chunk rows for the overlapped ranges (8 sequences,
    20,523 tokens: 325 chunks in at most 328 chunk rows, three ranges whose boundaries cut through
    sequences): the front end of v runs ahead of the state passes on their stream and the state passes
    read v back from o, with carried conv state, initial states and the output gate; the same bits as the
    two passes."""
    H, d = 4, 128
    C = H * d
    lengths = [3000, 5, 4100, 64, 2999, 6000, 1, 4354]
    T, N = sum(lengths), len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    xs = [ks.fill(117, tid, ks.NORMAL, (T, C), "bf16") for tid in (1, 2, 3)]
    cw = ks.fill(117, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25)
    cs = ks.fill(117, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16")
    g = ks.fill(117, ks.TID_G, ks.NEG5_SIGMOID, (T, H, d), "f32")
    b = ks.fill(117, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    s0 = ks.fill(117, ks.TID_STATE, ks.NORMAL, (N, H, d, d), "f32", 0.0, 0.02)
    gate = ks.fill(117, ks.TID_GATE, ks.NORMAL, (T, C), "bf16")
    xd = [dev(x) for x in xs]
    cu_d, cs_d = dev(cu), dev(cs)
    q, k, v = kda.kda_shortconv_l2norm(*xd, dev(cw), H, cu_d, cs_d)
    o1, f1 = kda.kda_chunk_fwd(q, k, v, dev(g), dev(b), dev(s0), cu_d, out_gate=dev(gate))
    o2, f2 = kda.kda_chunk_fwd_frontend(*xd, dev(cw), dev(g), dev(b), H, dev(s0), cu_d, conv_state_in=cs_d,
                                        out_gate=dev(gate))
    torch.cuda.synchronize()
    assert T // 64 + N >= 256   # the overlapped ranges
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    assert kda.device_error() == 0


# ------------------------------------------------------------------------------------------
# kda_shortconv_l2norm
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("out_dtype,lengths", [("f32", [1, 2, 17, 0, 40]), ("bf16", [1, 2, 17, 0, 40]),
                                               ("f32", [130, 1, 37, 200, 8, 3])])
def test_shortconv_varlen_with_state(kda, orc, out_dtype, lengths):
    H, d = 3, 128
    C = H * d
    T, N = sum(lengths), len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    width = C + 8   # a row stride larger than H*d
    xs = [ks.fill(201, tid, ks.NORMAL, (T, width), "bf16") for tid in (1, 2, 3)]
    w = ks.fill(201, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25)
    cs = ks.fill(201, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16")
    tdt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    cs_out = torch.empty((N, 3, 3 * C), dtype=torch.bfloat16, device="cuda")
    q, k, v = kda.kda_shortconv_l2norm(*(dev(x) for x in xs), dev(w), H, dev(cu), dev(cs), cs_out, out_dtype=tdt)
    torch.cuda.synchronize()
    rq, rk, rv, rcs = orc.shortconv_silu_l2norm(*(ks.to_f64(x)[:, :C] for x in xs), ks.to_f64(w), H, d, cu,
                                                ks.to_f64(cs))
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        g64 = host(got)
        if out_dtype == "f32":
            assert orc.rel_l2(g64, ref) <= 1e-5
        else:
            assert orc.rel_l2(g64, ref) <= 5e-3
            assert np.max(np.abs(g64 - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2.0 ** -8 + 1e-5
    assert np.array_equal(cs_out.view(torch.int16).cpu().numpy().view(np.uint16), ks.f32_to_bf16(rcs))


def test_shortconv_state_in_place(kda, orc):
    H, d, C = 2, 128, 256
    lengths = [5, 1]
    T, N = 6, 2
    cu = np.array([0, 5, 6], np.int32)
    xs = [ks.fill(202, tid, ks.NORMAL, (T, C), "bf16") for tid in (1, 2, 3)]
    w = ks.fill(202, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25)
    cs = ks.fill(202, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16")
    cs_dev = dev(cs)
    kda.kda_shortconv_l2norm(*(dev(x) for x in xs), dev(w), H, dev(cu), cs_dev, cs_dev)
    torch.cuda.synchronize()
    _, _, _, rcs = orc.shortconv_silu_l2norm(*(ks.to_f64(x) for x in xs), ks.to_f64(w), H, d, cu, ks.to_f64(cs))
    assert np.array_equal(cs_dev.view(torch.int16).cpu().numpy().view(np.uint16), ks.f32_to_bf16(rcs))


# ------------------------------------------------------------------------------------------
# kda_recurrent_step
# ------------------------------------------------------------------------------------------

def decode_inputs(w):
    xs = [ks.fill(w.seed, tid, ks.NORMAL, (w.N, w.H * w.d), "bf16") for tid in (1, 2, 3)]
    g = ks.fill(w.seed, ks.TID_G, w.g_kind, (w.N, w.H, w.d), "f32")
    b = ks.fill(w.seed, ks.TID_BETA, ks.SIGMOID, (w.N, w.H), "f32")
    return xs, w.conv_w(), g, b, w.init_state(), w.conv_state()


def check_decode(kda, orc, w, scale=1.0, steps=1, gates=None):
    xs, cw, g, b, s0, cs = decode_inputs(w)
    if gates is not None:
        g, b = gates(g, b)
    s_dev, cs_dev = dev(s0), dev(cs)
    s_ref, cs_ref = s0.astype(np.float64), ks.to_f64(cs)
    for step in range(steps):
        if step:  # fresh tokens for later steps
            xs = [ks.fill(w.seed + 1000 * step, tid, ks.NORMAL, (w.N, w.H * w.d), "bf16") for tid in (1, 2, 3)]
        o = kda.kda_recurrent_step(*(dev(x) for x in xs), dev(cw), dev(g), dev(b), s_dev, cs_dev, scale=scale)
        torch.cuda.synchronize()
        o_ref, s_ref, cs_ref = orc.recurrent_step(*(ks.to_f64(x) for x in xs), ks.to_f64(cw), g, b, s_ref, cs_ref,
                                                  w.H, w.d, scale)
        assert orc.rel_l2(host(o), o_ref) <= BF16_O_REL and orc.max_abs(host(o), o_ref) <= BF16_O_ABS
        assert orc.rel_l2(host(s_dev), s_ref) <= BF16_S_REL
        assert np.array_equal(host(cs_dev), cs_ref)   # bf16 widened exactly: bit-exact


def test_decode_small(kda, orc):
    w = ks.Workload("d", "decode", 301, H=3, lengths=[1] * 5, init_state_std=0.02)
    check_decode(kda, orc, w, scale=0.5, steps=8)


@pytest.mark.parametrize("case", ["no_decay_full_write", "floor_no_write", "floor_full_write"])
def test_decode_degenerate_gates(kda, orc, case):
    """g = 0 with beta = 1 (the plain delta rule overwriting along k), g = -5 with beta = 0 (the state
    only decays, by e^-5 a step) and g = -5 with beta = 1, over four chained steps."""
    g_val, b_val = {"no_decay_full_write": (0.0, 1.0), "floor_no_write": (-5.0, 0.0),
                    "floor_full_write": (-5.0, 1.0)}[case]
    w = ks.Workload("d", "decode", 303, H=3, lengths=[1] * 5, init_state_std=0.02)
    check_decode(kda, orc, w, steps=4, gates=lambda g, b: (np.full_like(g, g_val), np.full_like(b, b_val)))


def test_decode_full_workload(kda, orc):
    """64 sequences x 96 heads, fp32 state N(0, 0.02), the whole step checked."""
    check_decode(kda, orc, ks.workload("decode_64"))


def test_prefill_equals_repeated_decode(kda):
    """Front end + chunkwise prefill over T tokens == T fused decode steps (bf16 bounds)."""
    H, C, T = 2, 256, 70
    xs = [ks.fill(302, tid, ks.NORMAL, (T, C), "bf16") for tid in (1, 2, 3)]
    cw = ks.fill(302, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25)
    cs0 = ks.fill(302, ks.TID_CONV_STATE, ks.NORMAL, (1, 3, 3 * C), "bf16")
    g = ks.fill(302, ks.TID_G, ks.NEG5_SIGMOID, (T, H, 128), "f32")
    b = ks.fill(302, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    s0 = ks.fill(302, ks.TID_STATE, ks.NORMAL, (1, H, 128, 128), "f32", 0.0, 0.02)
    xd = [dev(x) for x in xs]
    cs_pre = dev(cs0)
    q, k, v = kda.kda_shortconv_l2norm(*xd, dev(cw), H, None, cs_pre, cs_pre)
    o_pre, fs = kda.kda_chunk_fwd(q, k, v, dev(g), dev(b), dev(s0))
    s, cs = dev(s0), dev(cs0)
    outs = []
    for t in range(T):
        outs.append(kda.kda_recurrent_step(*(x[t:t + 1] for x in xd), dev(cw), dev(g[t:t + 1]), dev(b[t:t + 1]),
                                           s, cs))
    torch.cuda.synchronize()
    o_dec = torch.cat(outs).float()
    rel = (o_dec - o_pre.float()).norm() / o_dec.norm()
    assert rel <= BF16_O_REL
    assert ((s - fs).norm() / s.norm()) <= BF16_S_REL
    assert torch.equal(cs, cs_pre)


# ------------------------------------------------------------------------------------------
# full-size workloads, checked on sampled heads / chains
# ------------------------------------------------------------------------------------------

def fill_dev(w, tid, kind, shape, dtype, p0=0.0, p1=1.0):
    from kda_synth.device import fill_device
    return fill_device(w.seed, tid, kind, shape, dtype, p0, p1)


def head_inputs(w, h, t0, t1):
    """Oracle inputs of head h, tokens [t0, t1): regenerated from the counter-based streams."""
    d, H = w.d, w.H
    q = w.head_rows(ks.TID_Q, ks.UNIT_GROUPS, h, w.dtype, p1=float(d), t0=t0, t1=t1)
    k = w.head_rows(ks.TID_K, ks.UNIT_GROUPS, h, w.dtype, p1=float(d), t0=t0, t1=t1)
    v = w.head_rows(ks.TID_V, ks.NORMAL, h, w.dtype, t0=t0, t1=t1)
    g = w.head_rows(ks.TID_G, w.g_kind, h, "f32", t0=t0, t1=t1)
    b = w.head_beta(h, t0, t1)
    ex = lambda a: ks.to_f64(a)[:, None, :]
    return ex(q), ex(k), ex(v), g.astype(np.float64)[:, None, :], b.astype(np.float64)[:, None]


def test_prefill_8k_sampled_heads(kda, orc):
    """H=96, T=8192 bf16 prefill as the benchmark launches it; heads 0, 37, 95 checked in full."""
    w = ks.workload("prefill_8k")
    T, H, d = w.T, w.H, w.d
    q = fill_dev(w, ks.TID_Q, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    k = fill_dev(w, ks.TID_K, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    v = fill_dev(w, ks.TID_V, ks.NORMAL, (T, H, d), "bf16")
    g = fill_dev(w, ks.TID_G, w.g_kind, (T, H, d), "f32")
    b = fill_dev(w, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    o, fs = kda.kda_chunk_fwd(q, k, v, g, b)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any()
    for h in (0, 37, 95):
        qh, kh, vh, gh, bh = head_inputs(w, h, 0, T)
        o_ref, fs_ref = orc.kda_tokenloop(qh, kh, vh, gh, bh)
        o_h = host(o[:, h:h + 1, :])
        assert orc.rel_l2(o_h, o_ref) <= BF16_O_REL and orc.max_abs(o_h, o_ref) <= BF16_O_ABS
        assert orc.rel_l2(host(fs[:, h:h + 1]), fs_ref) <= BF16_S_REL


def test_prefill_4k_persistent_operand_pass_sampled_heads(kda, orc):
    """4096 tokens x 96 heads with the whole workspace: 64 chunk rows, one range, so the operand
    kernel runs persistently (two CTAs per SM, each taking about 20 (chunk, head) items with the
    next item's loads in flight).  Heads 0, 50 and 95 checked in full against the oracle."""
    w = ks.Workload("prefill_4k", "prefill", 53102, H=96, lengths=[4096])
    T, H, d = w.T, w.H, w.d
    q = fill_dev(w, ks.TID_Q, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    k = fill_dev(w, ks.TID_K, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    v = fill_dev(w, ks.TID_V, ks.NORMAL, (T, H, d), "bf16")
    g = fill_dev(w, ks.TID_G, w.g_kind, (T, H, d), "f32")
    b = fill_dev(w, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    full = kda.kda_chunk_fwd_workspace_size(1, T, H, torch.bfloat16, False)[0]
    ws = torch.empty(full, dtype=torch.uint8, device="cuda")
    o, fs = kda.kda_chunk_fwd(q, k, v, g, b, workspace=ws)
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    for h in (0, 50, 95):
        qh, kh, vh, gh, bh = head_inputs(w, h, 0, T)
        o_ref, fs_ref = orc.kda_tokenloop(qh, kh, vh, gh, bh)
        o_h = host(o[:, h:h + 1, :])
        assert orc.rel_l2(o_h, o_ref) <= BF16_O_REL and orc.max_abs(o_h, o_ref) <= BF16_O_ABS
        assert orc.rel_l2(host(fs[:, h:h + 1]), fs_ref) <= BF16_S_REL


def test_varlen_32_sampled_chains(kda, orc):
    """32 packed sequences (1K..32K tokens), H=96, initial states N(0, 0.02); the shortest,
    a middle and the longest sequence checked in full on heads 0 and 95."""
    w = ks.workload("varlen_32")
    T, H, d, N = w.T, w.H, w.d, w.N
    q = fill_dev(w, ks.TID_Q, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    k = fill_dev(w, ks.TID_K, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d))
    v = fill_dev(w, ks.TID_V, ks.NORMAL, (T, H, d), "bf16")
    g = fill_dev(w, ks.TID_G, w.g_kind, (T, H, d), "f32")
    b = fill_dev(w, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    s0 = fill_dev(w, ks.TID_STATE, ks.NORMAL, (N, H, d, d), "f32", 0.0, w.init_state_std)
    cu = w.cu_seqlens()
    o, fs = kda.kda_chunk_fwd(q, k, v, g, b, s0, dev(cu))
    torch.cuda.synchronize()
    order = np.argsort(w.lengths)
    for n in (int(order[0]), int(order[N // 2]), int(order[-1])):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in (0, 95):
            qh, kh, vh, gh, bh = head_inputs(w, h, t0, t1)
            sh = w.head_state(n, h).astype(np.float64)[None, None]
            o_ref, fs_ref = orc.kda_tokenloop(qh, kh, vh, gh, bh, sh)
            o_h = host(o[t0:t1, h:h + 1, :])
            assert orc.rel_l2(o_h, o_ref) <= BF16_O_REL and orc.max_abs(o_h, o_ref) <= BF16_O_ABS
            assert orc.rel_l2(host(fs[n:n + 1, h:h + 1]), fs_ref) <= BF16_S_REL


def test_long_256k_frontend_gate_sampled_heads(kda, orc):
    """T = 262,144: raw q, k, v -> kda_shortconv_l2norm -> kda_chunk_fwd with the sigmoid
    output gate; heads 0 and 61 checked in full against front end + token loop; the fused
    kda_chunk_fwd_frontend gives the same bits."""
    w = ks.workload("long_256k")
    T, H, d = w.T, w.H, w.d
    C = H * d
    xq = fill_dev(w, ks.TID_Q, ks.NORMAL, (T, C), "bf16")
    xk = fill_dev(w, ks.TID_K, ks.NORMAL, (T, C), "bf16")
    xv = fill_dev(w, ks.TID_V, ks.NORMAL, (T, C), "bf16")
    cw = fill_dev(w, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, w.conv_w_std)
    g = fill_dev(w, ks.TID_G, w.g_kind, (T, H, d), "f32")
    b = fill_dev(w, ks.TID_BETA, ks.SIGMOID, (T, H), "f32")
    gate = fill_dev(w, ks.TID_GATE, ks.NORMAL, (T, C), "bf16")
    q, k, v = kda.kda_shortconv_l2norm(xq, xk, xv, cw, H)
    o, fs = kda.kda_chunk_fwd(q, k, v, g, b, out_gate=gate)
    torch.cuda.synchronize()
    del q, k, v
    # the fused prefill computes the same bits
    o2, fs2 = kda.kda_chunk_fwd_frontend(xq, xk, xv, cw, g, b, H, out_gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(fs2, fs)
    del xq, xk, xv, g, o2, fs2
    cw_h = ks.to_f64(w.conv_w())
    heads = (0, 61)
    fe = []
    for h in heads:
        raw = [ks.to_f64(w.head_rows(tid, ks.NORMAL, h, "bf16")) for tid in (ks.TID_Q, ks.TID_K, ks.TID_V)]
        wh = np.concatenate([cw_h[p * C + h * d: p * C + (h + 1) * d] for p in range(3)])
        fe.append(orc.shortconv_silu_l2norm(*raw, wh, 1, d, want_state=False)[:3])
    qh, kh, vh = (np.concatenate([f[i] for f in fe], axis=1) for i in range(3))   # [T, 2, d]
    gh = np.stack([w.head_rows(ks.TID_G, w.g_kind, h, "f32") for h in heads], axis=1).astype(np.float64)
    bh = np.stack([w.head_beta(h) for h in heads], axis=1).astype(np.float64)
    gt = np.concatenate([ks.to_f64(w.head_rows(ks.TID_GATE, ks.NORMAL, h, "bf16")) for h in heads], axis=1)
    o_h = np.concatenate([host(o[:, h:h + 1, :]) for h in heads], axis=1)
    fs_h = np.concatenate([host(fs[:, h:h + 1]) for h in heads], axis=1)
    # the chunk kernel stores q, k, v in bf16: the oracle rounds its own front-end output the same way
    rq, rk, rv = (ks.bf16_to_f64(ks.f32_to_bf16(x.astype(np.float32))) for x in (qh, kh, vh))
    o_ref, fs_ref = orc.kda_tokenloop(rq, rk, rv, gh, bh)
    o_ref = orc.output_gate(o_ref, gt)
    assert orc.rel_l2(o_h, o_ref) <= BF16_O_REL and orc.max_abs(o_h, o_ref) <= BF16_O_ABS
    assert orc.rel_l2(fs_h, fs_ref) <= BF16_S_REL
    # and against the unrounded fp64 front end
    o_ref2, _ = orc.kda_tokenloop(qh, kh, vh, gh, bh)
    assert orc.rel_l2(o_h, orc.output_gate(o_ref2, gt)) <= BF16_O_REL
