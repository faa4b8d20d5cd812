"""Upload synthetic tensors to a CUDA device in bounded host memory.

The values are produced on the host by the counter-based generator of this
package (row block by row block into a pinned staging buffer) and copied to
the device, so a 26 GB tensor never sits in host RAM at once and the values on
the device are bit-identical to what :func:`kda_synth.fill` returns.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _DT, fill_slice

_TORCH = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}


def fill_device(seed: int, tid: int, kind: int, shape, dtype: str = "f32", p0: float = 0.0, p1: float = 1.0,
                device="cuda", block_bytes: int = 1 << 28, out: torch.Tensor | None = None) -> torch.Tensor:
    shape = tuple(int(s) for s in shape)
    last = shape[-1]
    rows = int(np.prod(shape)) // last if last else 0
    _, npdt = _DT[dtype]
    if out is None:
        out = torch.empty(shape, dtype=_TORCH[dtype], device=device)
    flat = out.view(rows, last)
    rows_per = max(1, block_bytes // (last * np.dtype(npdt).itemsize))
    stage = [torch.empty((min(rows_per, rows), last), dtype=_TORCH[dtype], pin_memory=True) for _ in range(2)]
    views = [s.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else s.numpy() for s in stage]
    events = [None, None]
    stream = torch.cuda.current_stream(out.device)
    r0, slot = 0, 0
    while r0 < rows:
        nr = min(rows_per, rows - r0)
        if events[slot] is not None:
            events[slot].synchronize()
        buf = views[slot][:nr]
        fill_slice(seed, tid, kind, last, r0, nr, 0, last, dtype, p0, p1, out=buf)
        flat[r0:r0 + nr].copy_(stage[slot][:nr], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream)
        events[slot] = ev
        r0 += nr
        slot ^= 1
    torch.cuda.synchronize(out.device)
    return out


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """A host array from :mod:`kda_synth` (bf16 as uint16 bits) as a device tensor."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_f64(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> fp64 numpy (bf16 widened exactly)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
