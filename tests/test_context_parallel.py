"""Carrying the state across segments of one sequence (context parallelism).

The update is affine in the state, so a segment maps its entering state S to S M + E (M its
transition operator, E its end state from zero).  CPU tests pin the oracle's transition operator
(closed forms and the composition identity against the token loop) and run the exchange logic as two
gloo processes with an fp64 backend; GPU tests check kda_chunk_segment_summary and kda_state_combine
against the oracle and a whole sequence split into segments against one pass.

Tolerances (GPU, against the fp64 oracle): o rel-L2 <= 5e-3 and max-abs <= 2e-2, states and
transition operators rel-L2 <= 5e-3 (the bf16 prefill's); kda_state_combine rel-L2 <= 1e-6 (fp32
products of 128 terms).
"""
import os
import socket

import numpy as np
import pytest

import kda_synth as ks

torch = pytest.importorskip("torch")

BF16_O_REL, BF16_O_ABS, BF16_S_REL = 5e-3, 2e-2, 5e-3


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def rand_inputs(seed, T, H, d, weak=False):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((T, H, d))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, d))))
    if weak:
        g *= 0.01
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


# ---------------------------------------------------------------------------------------------
# oracle pins (CPU)
# ---------------------------------------------------------------------------------------------

def test_transition_without_correction_is_the_decay(orc):
    """beta = 0: every X_t is Diag(alpha_t), so M = Diag(exp(sum_t g_t)) exactly."""
    q, k, v, g, _ = rand_inputs(1, 40, 3, 16)
    M = orc.transition(k, g, np.zeros((40, 3)))
    for h in range(3):
        np.testing.assert_allclose(M[0, h], np.diag(np.exp(g[:, h].sum(0))), rtol=1e-13, atol=1e-300)


def test_transition_of_one_token_without_decay(orc):
    """One token, g = 0: M = I - beta k k^T."""
    _, k, _, _, beta = rand_inputs(2, 1, 2, 8)
    M = orc.transition(k, np.zeros_like(k), beta)
    for h in range(2):
        ref = np.eye(8) - beta[0, h] * np.outer(k[0, h], k[0, h])
        np.testing.assert_allclose(M[0, h], ref, rtol=0, atol=1e-15)


@pytest.mark.parametrize("weak", [False, True])
def test_composition_matches_the_token_loop(orc, weak):
    """The token loop from a random S0 ends in S0 M + E (M by the literal operator product, E by the
    token loop from zero), and splitting a sequence into segments reproduces its outputs."""
    T, H, d = 90, 2, 12
    q, k, v, g, beta = rand_inputs(3, T, H, d, weak)
    S0 = np.random.default_rng(4).standard_normal((1, H, d, d))
    o_full, S_full = orc.kda_tokenloop(q, k, v, g, beta, init_state=S0)
    _, E = orc.kda_tokenloop(q, k, v, g, beta)
    M = orc.transition(k, g, beta)
    scale = np.abs(S_full).max()
    np.testing.assert_allclose(S0 @ M + E, S_full, rtol=0, atol=1e-12 * scale)
    if weak:  # (with the pages' decay M is ~e^-225 here and no test of it can see anything)
        # a planted transposition (M^T) breaks the identity: the pin is sensitive to operand order
        assert np.abs(S0 @ np.swapaxes(M, -1, -2) + E - S_full).max() > 1e-6 * scale
    bounds = [0, 17, 50, 64, T]
    S, outs = S0, []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, S = orc.kda_tokenloop(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], init_state=S)
        outs.append(o)
    np.testing.assert_allclose(np.concatenate(outs), o_full, rtol=0, atol=1e-12 * np.abs(o_full).max())


# ---------------------------------------------------------------------------------------------
# the exchange, two gloo processes with an fp64 backend (CPU)
# ---------------------------------------------------------------------------------------------

def _oracle_ops():
    import oracle
    from gated_delta_rule_53_gb300.context_parallel import Ops

    def summary(q, k, v, g, beta):
        a = [x.numpy() for x in (q, k, v, g, beta)]
        _, E = oracle.kda_tokenloop(*a)
        return torch.from_numpy(E), torch.from_numpy(oracle.transition(a[1], a[3], a[4]))

    def combine(S, M, E):
        return E.clone() if S is None else S @ M + E

    def chunk(q, k, v, g, beta, S, scale):
        a = [x.numpy() for x in (q, k, v, g, beta)]
        o, Sf = oracle.kda_tokenloop(*a, init_state=None if S is None else S.numpy(), scale=scale)
        return torch.from_numpy(o), torch.from_numpy(Sf)

    return Ops(summary, combine, chunk)


def _cp_worker(rank, world, port, bounds, seed):
    import torch.distributed as dist
    from gated_delta_rule_53_gb300.context_parallel import context_parallel_chunk_fwd, torch_all_gather
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, H, d = bounds[-1], 2, 8
        q, k, v, g, beta = rand_inputs(seed, T, H, d, weak=True)
        S0 = np.random.default_rng(seed + 1).standard_normal((1, H, d, d))
        a, b = bounds[rank], bounds[rank + 1]
        seg = [torch.from_numpy(np.ascontiguousarray(x[a:b])) for x in (q, k, v, g, beta)]
        o, S = context_parallel_chunk_fwd(*seg, rank=rank, all_gather=torch_all_gather(),
                                          init_state=torch.from_numpy(S0), scale=0.5, ops=_oracle_ops())
        o_full, S_full = oracle.kda_tokenloop(q, k, v, g, beta, init_state=S0, scale=0.5)
        np.testing.assert_allclose(o.numpy(), o_full[a:b], rtol=0, atol=1e-11 * np.abs(o_full).max())
        if rank == world - 1:
            np.testing.assert_allclose(S.numpy(), S_full, rtol=0, atol=1e-11 * np.abs(S_full).max())
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,bounds", [(2, [0, 37, 80]), (3, [0, 0, 41, 70])])
def test_context_parallel_exchange_gloo(world, bounds):
    """Each rank summarises its segment, all-gathers the summaries, folds those before it and runs
    its segment; every rank's outputs (and the last rank's state) equal one pass over the sequence.
    The second case gives rank 0 an empty segment."""
    import torch.multiprocessing as mp
    mp.start_processes(_cp_worker, args=(world, _free_port(), bounds, 11), nprocs=world, join=True,
                       start_method="spawn")


# ---------------------------------------------------------------------------------------------
# GPU: the library's summary and combine, and a sequence split into segments
# ---------------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_53_gb300 import build
    build.build()
    import gated_delta_rule_53_gb300 as m
    return m


def bf16_inputs(seed, T, H, weak=False, init_std=0.0):
    """Seeded synthetic prefill inputs (bf16 q, k, v as the GPU gets them), g optionally weakened."""
    w = ks.Workload("cp", "prefill", seed, H=H, lengths=[T], init_state_std=init_std)
    q, k, v, g, b = w.qkv("q"), w.qkv("k"), w.qkv("v"), w.g(), w.beta()
    if weak:
        g = (g * np.float32(0.01)).astype(np.float32)
    return q, k, v, g, b, w.init_state()


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def dev(a):
    from kda_synth.device import to_device
    return to_device(a)


def host(t):
    from kda_synth.device import to_host_f64
    return to_host_f64(t)


@pytest.mark.gpu
@pytest.mark.parametrize("T,weak", [(300, True), (1000, False), (64, True)])
def test_segment_summary_matches_oracle(kda, orc, T, weak):
    q, k, v, g, b, _ = bf16_inputs(5300 + T, T, 2, weak)
    E, M = kda.kda_chunk_segment_summary(dev(k), dev(g), dev(b), v=dev(v), q=dev(q))
    torch.cuda.synchronize()
    qf, kf, vf = (ks.to_f64(x) for x in (q, k, v))
    _, E_ref = orc.kda_tokenloop(qf, kf, vf, g, b)
    M_ref = orc.transition(kf, g, b)
    assert rel(host(E), E_ref) <= BF16_S_REL
    if np.linalg.norm(M_ref) > 1e-20:  # with the pages' decay, M underflows after a few dozen tokens
        assert rel(host(M), M_ref) <= BF16_S_REL
    else:
        assert np.abs(host(M)).max() <= 1e-20
    assert kda.device_error() == 0


@pytest.mark.gpu
def test_segment_summary_workspace_paths_agree(kda):
    """Operands computed once for both outputs (full workspace) or once per output in ranges of one
    chunk row (least workspace): the same bits."""
    q, k, v, g, b, _ = bf16_inputs(5401, 700, 3, weak=True)
    args = (dev(k), dev(g), dev(b))
    E1, M1 = kda.kda_chunk_segment_summary(*args, v=dev(v), q=dev(q))
    full, least = kda.kda_chunk_fwd_workspace_size(1, 700, 3, torch.bfloat16, False)
    ws = torch.empty(least, dtype=torch.uint8, device="cuda")
    E2, M2 = kda.kda_chunk_segment_summary(*args, v=dev(v), q=dev(q), workspace=ws)
    _, M3 = kda.kda_chunk_segment_summary(*args, end_state=False)   # transition alone, no v, no q
    torch.cuda.synchronize()
    assert torch.equal(E1, E2) and torch.equal(M1, M2) and torch.equal(M1, M3)


@pytest.mark.gpu
def test_state_combine_matches_fp64(kda):
    rng = np.random.default_rng(7)
    S, M, E = (rng.standard_normal((2, 3, 128, 128)).astype(np.float32) for _ in range(3))
    out = kda.kda_state_combine(dev(S), dev(M), dev(E))
    ref = S.astype(np.float64) @ M.astype(np.float64) + E
    assert rel(host(out), ref) <= 1e-6
    assert torch.equal(kda.kda_state_combine(None, dev(M), dev(E)), dev(E))
    s_d = dev(S)
    kda.kda_state_combine(s_d, dev(M), dev(E), out=s_d)   # in place over S_in
    assert rel(host(s_d), ref) <= 1e-6


@pytest.mark.gpu
@pytest.mark.parametrize("weak", [False, True])
def test_segmented_prefill_matches_oracle(kda, orc, weak):
    """A 2,148-token sequence cut at tokens 700, 1024 and 1500 (not on chunk boundaries), with a
    nonzero initial state: summaries, fold, re-run (simulated ranks on one GPU) against the oracle's
    single pass and against the library's single pass."""
    from gated_delta_rule_53_gb300.context_parallel import segmented_chunk_fwd
    T = 2148
    q, k, v, g, b, s0 = bf16_inputs(5500 + int(weak), T, 2, weak, init_std=0.02)
    tensors = [dev(x) for x in (q, k, v, g, b)]
    o, S = segmented_chunk_fwd(*tensors, bounds=[0, 700, 1024, 1500, T], init_state=dev(s0), scale=0.7)
    o1, S1 = kda.kda_chunk_fwd(*tensors, init_state=dev(s0), scale=0.7)
    torch.cuda.synchronize()
    qf, kf, vf = (ks.to_f64(x) for x in (q, k, v))
    o_ref, S_ref = orc.kda_tokenloop(qf, kf, vf, g, b, init_state=s0, scale=0.7)
    oh, Sh = host(o), host(S)
    assert rel(oh, o_ref) <= BF16_O_REL and np.abs(oh - o_ref).max() <= BF16_O_ABS
    assert rel(Sh, S_ref) <= BF16_S_REL
    assert rel(oh, host(o1)) <= BF16_O_REL and rel(Sh, host(S1)) <= BF16_S_REL
    assert kda.device_error() == 0
