"""Context-parallel chunk_kda: one sequence split into consecutive segments, one per rank.

The update of "Kimi-K3 深度解析", section 三 ("KDA 的关键改进"),
S_t = S_{t-1} Diag(alpha_t)(I - beta_t k_t k_t^T) + beta_t v_t k_t^T, is affine in the state, so a
segment maps whatever state enters it to  S M + E  (M its transition operator, E its end state from a
zero start).  Rank r holds tokens [t_r, t_{r+1}) of the sequence and:

1. summarises its segment: (E_r, M_r)                       -- kda_chunk_segment_summary
2. exchanges summaries with every rank (one all-gather) and folds those of the ranks before it, in
   order, from the sequence's initial state:  S_r = (..((S_0 M_0 + E_0) M_1 + E_1) ..)
                                                              -- kda_state_combine
3. runs its segment from S_r: its outputs o, and (on the last rank) the sequence's final state
                                                              -- kda_chunk_fwd

The arithmetic runs in the library; this module only orders the calls and the exchange.  The compute
backend is a parameter so that the exchange logic can be exercised by CPU processes (``gloo``) with
an fp64 stand-in on hosts without a GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence


@dataclass
class Ops:
    """Compute backend: summary(q, k, v, g, beta) -> (E, M); combine(S or None, M, E) -> S M + E;
    chunk(q, k, v, g, beta, init_state or None, scale) -> (o, final_state)."""
    summary: Callable
    combine: Callable
    chunk: Callable


def library_ops(workspace=None) -> Ops:
    """The library's CUDA kernels (bf16 inputs, one sequence per call)."""
    from . import kda_chunk_fwd, kda_chunk_segment_summary, kda_state_combine

    def summary(q, k, v, g, beta):
        return kda_chunk_segment_summary(k, g, beta, v=v, q=q, workspace=workspace)

    def combine(S, M, E):
        return kda_state_combine(S, M, E)

    def chunk(q, k, v, g, beta, init_state, scale):
        return kda_chunk_fwd(q, k, v, g, beta, init_state=init_state, scale=scale, workspace=workspace)

    return Ops(summary, combine, chunk)


def fold(init_state, ends: Sequence, transitions: Sequence, upto: int, combine: Callable):
    """The state entering segment `upto`: the first `upto` segments' maps applied in order to
    init_state (None = zero)."""
    S = init_state
    for j in range(upto):
        S = combine(S, transitions[j], ends[j])
    return S


def context_parallel_chunk_fwd(q, k, v, g, beta, rank: int, all_gather: Callable[[object], List[object]],
                               init_state=None, scale: float = 1.0, ops: Optional[Ops] = None):
    """This rank's segment [T_r, H, d] of one sequence (all ranks call it together).  all_gather(t)
    returns every rank's t in rank order.  init_state: the sequence's initial state [1, H, d, d] (the
    same on every rank) or None.  Returns (o of this segment, state leaving it); the last rank's state
    is the sequence's final state."""
    ops = ops or library_ops()
    E, M = ops.summary(q, k, v, g, beta)
    ends, transitions = all_gather(E), all_gather(M)
    S = fold(init_state, ends, transitions, rank, ops.combine)
    return ops.chunk(q, k, v, g, beta, S, scale)


def torch_all_gather(group=None) -> Callable:
    """all_gather over a torch.distributed process group (any backend that holds the tensors)."""
    import torch
    import torch.distributed as dist

    def gather(t):
        out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(out, t.contiguous(), group=group)
        return out

    return gather


def segmented_chunk_fwd(q, k, v, g, beta, bounds: Sequence[int], init_state=None, scale: float = 1.0,
                        ops: Optional[Ops] = None):
    """One process plays every rank: segments [bounds[i], bounds[i+1]) of one sequence in turn.
    Returns (o [T, H, d], final state), the same pair one pass over the whole sequence gives."""
    import torch

    ops = ops or library_ops()
    segs = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    if not segs or segs[0][0] != 0 or segs[-1][1] != q.shape[0] or any(a > b for a, b in segs):
        raise ValueError("bounds must run from 0 to T in order")
    cut = lambda x, a, b: x[a:b].contiguous()
    summaries = [ops.summary(cut(q, a, b), cut(k, a, b), cut(v, a, b), cut(g, a, b), cut(beta, a, b))
                 for a, b in segs]
    ends = [s[0] for s in summaries]
    transitions = [s[1] for s in summaries]
    outs, S_in, S = [], init_state, init_state
    for r, (a, b) in enumerate(segs):
        if r:
            S_in = ops.combine(S_in, transitions[r - 1], ends[r - 1])
        o, S = ops.chunk(cut(q, a, b), cut(k, a, b), cut(v, a, b), cut(g, a, b), cut(beta, a, b), S_in, scale)
        outs.append(o)
    return torch.cat(outs, dim=0), S
