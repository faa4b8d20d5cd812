"""The decay-gate generator: gate = x W_gate^T, g = max(-5, -softplus(x W_a^T W_b^T + a_h)).

The pages give the ingredients (a low-rank projection plus a per-head parameter, floored at -5;
a full-rank output gate) but no formula; the reading above is the library's.  CPU tests pin the
oracle's formula by closed forms (a zero input leaves only the per-head parameter; a one-hot input
picks a weight column; saturation at the floor); GPU tests compare the library with it.

Tolerances (GPU, bf16 inputs, fp32 accumulation, z rounded to bf16 between the two products):
gate rel-L2 <= 5e-3 (one bf16 rounding of the output, 2^-9, dominates); g rel-L2 <= 5e-3 and
max-abs <= 2e-2 (the bf16 rounding of z moves y by about 2^-9 |z| |W_b| per term).
"""
import ctypes

import numpy as np
import pytest

import kda_synth as ks

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def weights(seed, hidden, H, d, rank, a_spread=2.0):
    rng = np.random.default_rng(seed)
    wga = rng.standard_normal((H * d + rank, hidden)) / np.sqrt(hidden)
    wb = rng.standard_normal((H * d, rank)) / np.sqrt(rank)
    a = a_spread * rng.standard_normal(H)
    return wga, wb, a


def test_zero_input_leaves_the_head_parameter(orc):
    H, d, rank, hidden = 3, 8, 4, 16
    wga, wb, a = weights(1, hidden, H, d, rank)
    gate, g = orc.gate_generator(np.zeros((5, hidden)), wga, wb, a, H, d)
    assert np.all(gate == 0)
    for h in range(H):
        np.testing.assert_allclose(g[:, h, :], max(-5.0, -np.log1p(np.exp(a[h]))), rtol=1e-15)


def test_one_hot_input_picks_weight_columns(orc):
    H, d, rank, hidden = 2, 8, 4, 6
    wga, wb, a = weights(2, hidden, H, d, rank)
    gate, g = orc.gate_generator(np.eye(hidden), wga, wb, a, H, d)
    np.testing.assert_array_equal(gate, wga[:H * d].T)      # row i = column i of W_gate
    y = wga[H * d:].T @ wb.T + np.repeat(a, d)               # row i: (W_a column i) W_b^T + a_h
    np.testing.assert_allclose(g.reshape(hidden, H * d), np.maximum(-5, -np.log1p(np.exp(y))), rtol=1e-14)


def test_floor_and_ceiling(orc):
    """A large per-head parameter saturates at the floor -5 exactly; a very negative one gives a
    decay factor just below 1 (g just below 0); g never leaves [-5, 0]."""
    H, d, rank, hidden = 2, 8, 4, 16
    wga, wb, _ = weights(3, hidden, H, d, rank)
    x = np.random.default_rng(4).standard_normal((7, hidden))
    _, g = orc.gate_generator(x, wga, wb, np.array([40.0, -40.0]), H, d)
    assert np.all(g[:, 0, :] == -5.0)
    assert np.all(g[:, 1, :] < 0) and np.all(g[:, 1, :] > -1e-15)
    _, g = orc.gate_generator(x, wga, wb, np.array([0.3, -0.7]), H, d)
    assert np.all((g >= -5.0) & (g <= 0.0))


def test_gate_generator_rejects_bad_arguments():
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    lib = kda.library()
    P = ctypes.c_void_p

    def call(**over):
        a = dict(x=P(4096), T=64, hidden=256, w=P(4096), wb=P(4096), ah=P(4096), H=2, d=128, rank=64, gate=P(4096),
                 g=P(4096), z=P(4096))
        a.update(over)
        return lib.kda_gate_generator(a["x"], a["T"], a["hidden"], a["w"], a["wb"], a["ah"], a["H"], a["d"],
                                      a["rank"], a["gate"], a["g"], a["z"], None)
    assert call(x=None) == 1
    assert call(z=None) == 1
    assert call(w=None) == 1
    assert call(T=0, x=None, gate=None, g=None, z=None) == 0   # nothing to compute
    assert call(g=P(4100)) == 1          # misaligned
    assert call(T=-1) == 1
    assert call(T=1 << 31) == 1
    assert call(hidden=100) == 1         # not a multiple of 8
    assert call(d=64) == 2
    assert call(rank=48) == 1            # not a multiple of 32
    assert call(rank=0) == 1
    assert call(H=0) == 1


# ---------------------------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------------------------

def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def bf16_round(a):
    """fp64 values rounded to bf16 (round to nearest even), as the GPU receives them."""
    f = np.asarray(a, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


@pytest.mark.gpu
@pytest.mark.parametrize("T,hidden,H,rank", [(300, 512, 2, 64), (1000, 1024, 4, 128), (129, 64, 1, 32),
                                             (0, 256, 2, 32)])
def test_gate_generator_matches_oracle(orc, T, hidden, H, rank):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    d = 128
    wga, wb, a = weights(10 + T, hidden, H, d, rank)
    a[0] = 30.0  # one head saturates at the floor
    x = np.random.default_rng(20 + T).standard_normal((T, hidden))
    xq, wgaq, wbq = bf16_round(x), bf16_round(wga), bf16_round(wb)   # the bits the GPU gets
    to = lambda m, dt: torch.from_numpy(np.ascontiguousarray(m)).to(dt).cuda()
    gate, g = kda.kda_gate_generator(to(xq, torch.bfloat16), to(wgaq, torch.bfloat16), to(wbq, torch.bfloat16),
                                     to(a, torch.float32), H, d)
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    if T == 0:
        return
    gate_ref, g_ref = orc.gate_generator(xq, wgaq, wbq, a.astype(np.float32), H, d)
    gh = gate.double().cpu().numpy()
    gg = g.double().cpu().numpy()
    assert rel(gh, gate_ref) <= 5e-3
    assert rel(gg, g_ref) <= 5e-3 and np.abs(gg - g_ref).max() <= 2e-2
    assert np.all(gg[:, 0, :] == -5.0)
    assert np.all((gg >= -5.0) & (gg <= 0.0))


@pytest.mark.gpu
def test_gate_generator_full_size_persistent_tiles(orc):
    """x [8192, 7168] with 96 heads and rank 128, as the benchmark runs it: 64 row tiles x 49 column
    tiles (3,136) in the x-side product and 64 x 48 in the rank product, on at most one CTA per SM, so
    every CTA runs many tiles: the persistent loop past its first tile, both TMEM accumulators and
    their phase flips, and every group of 16 row tiles.  Checked against the oracle on four rows of
    every 128-row tile (one in each 32-lane quarter of the accumulator, at a position that moves from
    tile to tile), over all columns."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as kda
    T, hidden, H, d, rank = 8192, 7168, 96, 128, 128
    rng = np.random.default_rng(53107)
    xq = bf16_round(rng.standard_normal((T, hidden), dtype=np.float32))
    wgaq = bf16_round(rng.standard_normal((H * d + rank, hidden), dtype=np.float32) / np.sqrt(hidden))
    wbq = bf16_round(rng.standard_normal((H * d, rank), dtype=np.float32) / np.sqrt(rank))
    a = 2.0 * rng.standard_normal(H)
    a[7] = 30.0   # one head at the floor
    to = lambda m, dt: torch.from_numpy(np.ascontiguousarray(m)).to(dt).cuda()
    gate, g = kda.kda_gate_generator(to(xq, torch.bfloat16), to(wgaq, torch.bfloat16), to(wbq, torch.bfloat16),
                                     to(a, torch.float32), H, d)
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    mt = T // 128
    rows = np.array([128 * i + 32 * qt + (7 * i + 11 * qt) % 32 for i in range(mt) for qt in range(4)])
    assert len(np.unique(rows // 2048)) == T // 2048          # every group of 16 row tiles
    idx = torch.from_numpy(rows).cuda()
    gh = gate.index_select(0, idx).double().cpu().numpy()
    gg = g.index_select(0, idx).double().cpu().numpy()
    gate_ref, g_ref = orc.gate_generator(xq[rows], wgaq, wbq, a.astype(np.float32), H, d)
    assert rel(gh, gate_ref) <= 5e-3
    assert rel(gg, g_ref) <= 5e-3 and np.abs(gg - g_ref).max() <= 2e-2
    # per tile as well: no 128 x 256 tile of either output is off on its own
    nt = (H * d) // 256
    for i in range(mt):
        for j in range(nt):
            r, c = slice(4 * i, 4 * i + 4), slice(256 * j, 256 * j + 256)
            assert rel(gh[r, c], gate_ref[r, c]) <= 1e-2, (i, j)
            gr = g_ref.reshape(len(rows), H * d)[r, c]
            assert np.abs(gg.reshape(len(rows), H * d)[r, c] - gr).max() <= 2e-2, (i, j)
    assert np.all(gg[:, 7, :] == -5.0)
