#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300.

One step = one chunkwise prefill (kda_chunk_fwd) of the 8K-token workload:
1 sequence x 8192 tokens x 96 heads x d 128, bf16 q/k/v (q, k L2-normalised),
fp32 g = -5 sigmoid(z) and beta = sigmoid(z), zero initial state; output o
(bf16) and the final fp32 state.  ``value`` is prefill tokens/s (whole job:
sum over ranks).  The same JSON line carries the decode half of the metric:
one fused kda_recurrent_step of 64 sequences x 96 heads, in place on the
403 MB fp32 state, as state GB/s.

The line also times every other configuration at full size: the tiny fp32
prefill (4 heads x 256 tokens), the 32 packed sequences of 1K..32K tokens with
initial states, and the 262,144-token prefill from raw inputs through the fused
front end with the sigmoid output gate; the last key, ``per_config``, repeats
each configuration's figure compactly.

Inputs are synthetic (seeded counter-based generator, kda_synth; the two largest
workloads draw their values on the device with torch's seeded generator, same
distributions) and larger than the 129 MB L2 (1.2 GB per prefill step, 0.84 GB
per decode step), so L2 is not flushed between iterations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica (the path shards by
sequence and head with no exchange); rank 0 prints one JSON line.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=96,d=128) + decode state GB/s, % of roofline"

# prefill: algorithmic bytes per token-head = q, k, v bf16 (3 x 256) + g fp32 (512) + beta (4) + o bf16 (256)
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * 256 + 512 + 4 + 256
# algorithmic flops per token-head at chunk 64: 3 state products (6 d^2) + triangular intra-chunk
# products (~5 C d) + UT solve (~C^2 / 3)
PREFILL_FLOPS_PER_TOKEN_HEAD = 6 * 128 * 128 + 5 * 64 * 128 + (64 * 64) // 3


def prefill_bytes(T, H, N, d=128, init_state=False):
    b = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + N * H * d * d * 4   # + final state out
    if init_state:
        b += N * H * d * d * 4
    return b


def decode_bytes(N, H, d=128):
    C = H * d
    state = 2 * N * H * d * d * 4              # fp32 state read + written
    conv_state = 2 * N * 3 * 3 * C * 2         # bf16 conv state read + written
    x = 3 * N * C * 2                          # raw q, k, v
    g = N * H * d * 4
    o = N * H * d * 2
    w = 3 * C * 4 * 2
    beta = N * H * 4
    return state + conv_state + x + g + o + w + beta


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def bwd_flops_per_token_head(C: int = 64, d: int = 128) -> float:
    """The backward's own products per token and head (no recomputed forward): per chunk 12 C d^2
    (dV' and dS0 from dS_next, dO and dZ: 6 C d^2; dQg, dKg, dKr: 6 C d^2) and 10 C^2 d (the
    triangular products A_qk^T dO, the two solves, dA_qk, dA_kk and the four position-pair sums)."""
    return (12 * C * d * d + 10 * C * C * d) / C


def bwd_bytes_per_token_head(d: int = 128) -> int:
    """What the backward must move per token and head: q, k, v and dL/do in bf16, g and beta in fp32 read; the
    fp32 gradients of q, k, v, g and beta written (the chunk states and tiles its kernels hand to one another
    through the workspace are not counted)."""
    return 4 * d * 2 + d * 4 + 4 + 4 * d * 4 + 4


# The files each entry point's kernels are compiled from (a measured traffic figure stands only while they are unchanged).
FWD_SOURCES = "kda_chunk_tc.cu+kda_tsolve.cuh+kda_frontend.cuh"
BWD_SOURCES = "kda_chunk_bwd.cu+kda_chunk_bwd_tc.cu+kda_bwd_tc.cuh+kda_tsolve.cuh"


def prefill_launches(rows_max: int, rows_fit: int, packed: bool, fused: bool = False) -> int:
    """Kernel launches of one kda_chunk_fwd (fused: kda_chunk_fwd_frontend) call, as the library issues them:
    the chunk-offset kernel (packed sequences only), the front end of v (fused only), then per range of chunk
    rows an operand kernel and a state pass.  Ranges: about eight of at least 128 rows, at most half of what
    the workspace holds, overlapped, once the call and the workspace both hold 256 rows; otherwise as many
    rows as the workspace holds, one range after the other."""
    extra = (1 if packed else 0) + (1 if fused else 0)
    if rows_max <= 0:
        return extra + 1  # no chunk: the state pass alone (initial states pass through)
    rows_fit = max(min(rows_fit, rows_max), 1)
    if rows_fit >= 256 and rows_max >= 256:
        rr = min(max(128, -(-rows_max // 8)), rows_fit // 2)
        nr = -(-rows_max // rr)
    else:
        nr = -(-rows_max // rows_fit)
    return extra + 2 * nr


def fp32_alu_peak_tflops(sms: int = 152, lanes: int = 128, mhz: float = 2070.0) -> float:
    """fp32 FMA rate of the part: SMs x fp32 lanes per SM x 2 flop x the maximum SM clock."""
    return sms * lanes * 2 * mhz * 1e6 / 1e12


def kernel_source_hash(filename: str) -> str:
    """First 16 hex digits of the SHA-256 of a source file, or of several joined by '+' (their bytes in order)."""
    import hashlib
    h = hashlib.sha256()
    for name in filename.split("+"):
        with open(os.path.join(ROOT, "gated_delta_rule_53_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, source: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu capture of `kernel` on `workload`,
    or None when there is none or the kernel's source has changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[f"{kernel}@{workload}"]
    except Exception:
        return None
    if rec.get("workload") != workload or rec.get("source_sha256_16") != kernel_source_hash(source):
        return None
    return rec.get("dram_bytes_per_launch")


def reduce_max(value: float, dist) -> float:
    """Max of a per-rank number over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def smi_index(local_rank: int) -> str:
    """nvidia-smi's name for this process's GPU (CUDA_VISIBLE_DEVICES entries are indices or UUIDs)."""
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if cvd:
        entries = [e.strip() for e in cvd.split(",") if e.strip()]
        if local_rank < len(entries):
            return entries[local_rank]
    return str(local_rank)


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock event reasons, power), so that the
    clocks can be sampled every few milliseconds; None where the library or a call is unavailable."""

    # clock event reason bits of nvml.h
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, gpu_id: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if gpu_id.startswith("GPU-") or gpu_id.startswith("MIG-"):
            rc = self.lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(self.dev))
        else:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(gpu_id)), ctypes.byref(self.dev))
        if rc != 0:
            self.lib.nvmlShutdown()
            raise RuntimeError("no NVML handle for GPU " + gpu_id)
        reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = reasons or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct, u, ull = self.ct, self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(u)) != 0:  # NVML_CLOCK_SM
            return None
        sm = float(u.value)
        smax = float(u.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ct.byref(u)) == 0 else sm
        bits = ull.value if self.reasons_fn(self.dev, ct.byref(ull)) == 0 else 0
        return sm, smax, [name for bit, name in self.REASONS.items() if bits & bit]

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and clock event reasons sampled during the timed region: every 10 ms through NVML's read-only
    queries, or (without NVML) every 50 ms by ``nvidia-smi``, which has to be running before the region starts."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_s: float = 0.01):
        self.gpu_index = gpu_index
        self.period_s = period_s
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []
        self.thread = None
        self.running = False
        self.first = threading.Event()

    def start(self):
        try:
            self.nvml = _Nvml(str(self.gpu_index))
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.running = True
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(self.gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self.first.wait(timeout=5.0)  # nvidia-smi starts in a fraction of a second: begin the region after it

    def _poll(self):
        while self.running:
            s = self.nvml.sample()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.period_s)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.first.set()

    def stop(self):
        if self.nvml is not None:
            self.running = False
            self.thread.join(timeout=2)
            self.nvml.close()
            return self.summarise(self.samples, "nvml")
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summarise(self.parse_smi(self.lines), "nvidia-smi")

    @staticmethod
    def parse_smi(lines):
        """(sm MHz, max sm MHz, [active reasons]) of each nvidia-smi csv line of FIELDS."""
        out = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            out.append((sm, smax, [n for n, val in zip(names, parts[5:9]) if val.lower().startswith("active")]))
        return out

    @staticmethod
    def summarise(samples, source):
        sm = [s[0] for s in samples]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(s[1] for s in samples) if samples else None,
                "reasons": sorted({r for s in samples for r in s[2]}), "samples": len(sm), "source": source}


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def make_prefill_inputs(w, device):
    import kda_synth as ks
    from kda_synth.device import fill_device
    T, H, d = w.T, w.H, w.d
    q = fill_device(w.seed, ks.TID_Q, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d), device=device)
    k = fill_device(w.seed, ks.TID_K, ks.UNIT_GROUPS, (T, H, d), "bf16", 0.0, float(d), device=device)
    v = fill_device(w.seed, ks.TID_V, ks.NORMAL, (T, H, d), "bf16", device=device)
    g = fill_device(w.seed, ks.TID_G, w.g_kind, (T, H, d), "f32", device=device)
    b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (T, H), "f32", device=device)
    return q, k, v, g, b


def make_decode_inputs(w, device):
    import kda_synth as ks
    from kda_synth.device import fill_device
    N, H, d = w.N, w.H, w.d
    C = H * d
    xs = [fill_device(w.seed, t, ks.NORMAL, (N, C), "bf16", device=device) for t in (ks.TID_Q, ks.TID_K, ks.TID_V)]
    cw = fill_device(w.seed, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, w.conv_w_std, device=device)
    g = fill_device(w.seed, ks.TID_G, w.g_kind, (N, H, d), "f32", device=device)
    b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (N, H), "f32", device=device)
    st = fill_device(w.seed, ks.TID_STATE, ks.NORMAL, (N, H, d, d), "f32", 0.0, w.init_state_std, device=device)
    cs = fill_device(w.seed, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16", device=device)
    return xs, cw, g, b, st, cs


def device_draws(shape, kind, dtype, gen, rows_per=1 << 14):
    """A tensor of ``shape`` drawn on the device by torch's seeded generator ``gen``, slice by slice
    (no full-size fp32 temporary): ``kind`` "normal" N(0,1), "unit" rows N(0,1) normalised over the
    last axis, "neg5sig" -5 sigmoid(z), "negsp5" max(-5, -softplus(z)), "sigmoid" sigmoid(z)."""
    import torch
    out = torch.empty(shape, dtype=dtype, device=gen.device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], rows_per):
        r1 = min(shape[0], r0 + rows_per)
        z = torch.randn((r1 - r0,) + tuple(shape[1:]), device=gen.device, generator=gen, dtype=torch.float32)
        if kind == "unit":
            z = z / z.norm(dim=-1, keepdim=True)
        elif kind == "neg5sig":
            z = -5.0 * torch.sigmoid(z)
        elif kind == "negsp5":
            z = torch.clamp(-torch.nn.functional.softplus(z), min=-5.0)
        elif kind == "sigmoid":
            z = torch.sigmoid(z)
        flat[r0:r1] = z.reshape(r1 - r0, -1).to(dtype)
    return out


def timed(fn, steps, warmup, stream, dist=None):
    """Warm-up, then `steps` calls between two barriers + synchronizes, timed with CUDA events
    on `stream`; returns (ms per step over the whole region, mean ms per call, max over ranks)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            fn()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    total_ms = reduce_max(evs[0].elapsed_time(evs[-1]), dist)
    if dist is not None:
        dist.barrier()
    return total_ms / steps, statistics.mean(per), wall


def run_ours(args):
    import torch

    import gated_delta_rule_53_gb300 as kda
    import kda_synth as ks
    from gated_delta_rule_53_gb300 import build as kbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        kbuild.build()
    if dist is not None:
        dist.barrier()
    kda.library()
    hbm_peak, tc_peak, peak_src = load_peaks()
    stream = torch.cuda.Stream(device)

    # ---------------- prefill (the step) ----------------
    w = ks.workload(args.workload)
    q, k, v, g, b = make_prefill_inputs(w, device)
    o = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=device)
    fs = torch.empty((w.N, w.H, w.d, w.d), dtype=torch.float32, device=device)
    # the prefill's workspace (per-chunk operands of the state-independent kernel): all chunks in one range
    ws_full, _ = kda.kda_chunk_fwd_workspace_size(w.N, w.T, w.H, torch.bfloat16, w.N > 1)
    ws = torch.empty(ws_full, dtype=torch.uint8, device=device)
    # per range of chunk rows the operand kernel and the state pass (and the chunk offsets of packed sequences);
    # with the whole workspace the library overlaps ranges of max(128, rows / 8) chunk rows from 256 rows on
    rows = w.T // 64 + (w.N if w.N > 1 else (1 if w.T % 64 else 0))
    launches_per_call = prefill_launches(rows, rows, w.N > 1)
    step = lambda: kda.kda_chunk_fwd(q, k, v, g, b, o=o, final_state=fs, workspace=ws, stream=stream)
    clocks = ClockSampler(smi_index(local))
    clocks.start()
    ms_step, ms_launch, _ = timed(step, args.steps, args.warmup, stream, dist)
    clk = clocks.stop()
    tokens = w.T * world
    value = tokens / (ms_step * 1e-3)
    pbytes = prefill_bytes(w.T, w.H, w.N)
    achieved_gbs = pbytes / (ms_launch * 1e-3) / 1e9
    pflops = w.T * w.H * PREFILL_FLOPS_PER_TOKEN_HEAD
    achieved_tflops = pflops / (ms_launch * 1e-3) / 1e12

    # ---------------- the same sequence cut into 4 segments (context-parallel ranks, played in turn) --------
    # summaries (end state and transition operator, one operand pass for both), the fold by
    # kda_state_combine, and each segment re-run from its entering state, written into o in place
    seg = None
    if w.N == 1:
        nseg = 4
        bnd = [w.T * i // nseg for i in range(nseg + 1)]
        sE = [torch.empty_like(fs) for _ in range(nseg)]
        sM = [torch.empty_like(fs) for _ in range(nseg)]
        sS = [torch.empty_like(fs) for _ in range(nseg)]
        sF = torch.empty_like(fs)   # states leaving the non-last segments (equal to the fold's; unused)

        def summarise(i):
            a, z = bnd[i], bnd[i + 1]
            kda.kda_chunk_segment_summary(k[a:z], g[a:z], b[a:z], v=v[a:z], q=q[a:z], end_state=sE[i],
                                          transition=sM[i], workspace=ws, stream=stream)

        def rerun(i, S_in):
            a, z = bnd[i], bnd[i + 1]
            kda.kda_chunk_fwd(q[a:z], k[a:z], v[a:z], g[a:z], b[a:z], init_state=S_in, o=o[a:z],
                              final_state=fs if i == nseg - 1 else sF, workspace=ws, stream=stream)

        def segmented():
            for i in range(nseg):
                summarise(i)
            S_in = None
            for i in range(nseg):
                if i:
                    S_in = kda.kda_state_combine(S_in, sM[i - 1], sE[i - 1], out=sS[i - 1], stream=stream)
                rerun(i, S_in)

        ssteps = max(3, args.steps // 4)
        ms_seg, _, _ = timed(segmented, ssteps, args.warmup, stream, dist)
        ms_sum, _, _ = timed(lambda: summarise(nseg - 1), ssteps, args.warmup, stream, dist)
        ms_comb, _, _ = timed(lambda: kda.kda_state_combine(sS[0], sM[1], sE[1], out=sS[1], stream=stream), ssteps,
                              args.warmup, stream, dist)
        ms_run, _, _ = timed(lambda: rerun(nseg - 1, sS[nseg - 2]), ssteps, args.warmup, stream, dist)
        seg = {"workload": f"{w.name} cut into {nseg} segments of {w.T // nseg} tokens: context-parallel ranks "
                           "played in turn on one GPU (no exchange between devices timed)",
               "value": w.T / (ms_seg * 1e-3), "unit": "tokens/s", "ms_per_step": ms_seg, "steps": ssteps,
               # per segment: operand kernel + two state passes (summary), operand kernel + state pass (re-run)
               "gpu_launches": ssteps * (nseg * 3 + (nseg - 1) + nseg * 2),
               "segment_summary_ms": ms_sum, "state_combine_ms": ms_comb, "segment_rerun_ms": ms_run,
               "last_rank_ms": ms_sum + (nseg - 1) * ms_comb + ms_run,
               "note": "last_rank_ms: the measured per-call times of the work on the last of the ranks (its "
                       "summary, the fold of the three before it, its re-run), without the all-gather"}
        del sE, sM, sS, sF

    # ---------------- end to end through the API with host buffers ----------------
    # Every step copies its inputs from pinned host memory and reads its result (o and the final
    # state) back.  Steps are pipelined as a serving loop would run them: the next step's
    # host-to-device copy and the previous step's device-to-host read run on their own streams
    # (two copy engines) while the current step computes; two device slots keep them apart.
    host_in = [t.to("cpu").pin_memory() for t in (q, k, v, g, b)]
    del q, k, v, g, b
    slots = [([torch.empty(t.shape, dtype=t.dtype, device=device) for t in host_in],
              torch.empty_like(o), torch.empty_like(fs)) for _ in range(2)]
    host_out = [(torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
                 torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True)) for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {(name, i): torch.cuda.Event() for name in ("h2d", "comp", "d2h") for i in range(2)}
    used = set()

    def e2e_step(i):
        j = i % 2
        dev_in, o_j, fs_j = slots[j]
        with torch.cuda.stream(s_h2d):
            if ("comp", j) in used:
                s_h2d.wait_event(ev[("comp", j)])
            for dst, src in zip(dev_in, host_in):
                dst.copy_(src, non_blocking=True)
            ev[("h2d", j)].record(s_h2d)
        stream.wait_event(ev[("h2d", j)])
        if ("d2h", j) in used:
            stream.wait_event(ev[("d2h", j)])
        kda.kda_chunk_fwd(*dev_in, o=o_j, final_state=fs_j, workspace=ws, stream=stream)
        ev[("comp", j)].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev[("comp", j)])
            host_out[j][0].copy_(o_j, non_blocking=True)
            host_out[j][1].copy_(fs_j, non_blocking=True)
            ev[("d2h", j)].record(s_d2h)
        used.update({("comp", j), ("d2h", j)})

    e2e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    t_end.record(s_d2h)
    torch.cuda.synchronize()
    ms_e2e = reduce_max(t_start.elapsed_time(t_end), dist) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0][0].numel() * host_out[0][0].element_size() + host_out[0][1].numel() * host_out[0][1].element_size()
    del host_in, slots, host_out, ws

    # ---------------- decode (second half of the metric) ----------------
    wd = ks.workload("decode_64")
    xs, cw, gd, bd, st, cs = make_decode_inputs(wd, device)
    od = torch.empty((wd.N, wd.H, wd.d), dtype=torch.bfloat16, device=device)
    dstep = lambda: kda.kda_recurrent_step(*xs, cw, gd, bd, st, cs, o=od, stream=stream)
    dclocks = ClockSampler(smi_index(local))
    dclocks.start()
    # the decode step is ~0.1 ms: time enough of them for the clock sampler to see the region
    _, probe_ms, _ = timed(dstep, 20, args.warmup, stream, dist)
    dsteps = max(args.steps, int(1.0 / max(probe_ms * 1e-3, 1e-6)))
    ms_dec, ms_dec_launch, _ = timed(dstep, dsteps, 0, stream, dist)
    dclk = dclocks.stop()
    dbytes = decode_bytes(wd.N, wd.H)
    dec_gbs = dbytes / (ms_dec_launch * 1e-3) / 1e9

    del xs, cw, gd, bd, st, cs, od

    # ---------------- prefill front end (kda_shortconv_l2norm), a memory-bound pass ----------------
    wf = ks.Workload("frontend_32k", "frontend", 53005, H=96, lengths=[32768])
    Cw = wf.H * wf.d
    from kda_synth.device import fill_device
    xf = [fill_device(wf.seed, t, ks.NORMAL, (wf.T, Cw), "bf16", device=device) for t in (ks.TID_Q, ks.TID_K, ks.TID_V)]
    cwf = fill_device(wf.seed, ks.TID_CONV_W, ks.NORMAL, (3 * Cw, 4), "bf16", 0.0, wf.conv_w_std, device=device)
    outs = [torch.empty((wf.T, wf.H, wf.d), dtype=torch.bfloat16, device=device) for _ in range(3)]
    fstep = lambda: kda.kda_shortconv_l2norm(*xf, cwf, wf.H, q=outs[0], k=outs[1], v=outs[2], stream=stream)
    fsteps = max(20, args.steps // 4)
    ms_fe, ms_fe_launch, _ = timed(fstep, fsteps, args.warmup, stream, dist)
    fe_bytes = 2 * 3 * wf.T * Cw * 2 + 3 * Cw * 4 * 2   # raw in + normalised out (bf16) + weights
    fe_gbs = fe_bytes / (ms_fe_launch * 1e-3) / 1e9

    # ---------------- the gates from the layer input (kda_gate_generator): two tensor-core GEMMs ----------
    # x [8192, 7168] -> output gate [8192, 12288] and, through a rank-128 projection, the decay gate g
    Tg, hid, rk = 8192, 7168, 128
    ggen = torch.Generator(device=device).manual_seed(53007)
    xg = torch.randn(Tg, hid, device=device, generator=ggen).to(torch.bfloat16)
    wga = (torch.randn(w.H * w.d + rk, hid, device=device, generator=ggen) / hid ** 0.5).to(torch.bfloat16)
    wgb = (torch.randn(w.H * w.d, rk, device=device, generator=ggen) / rk ** 0.5).to(torch.bfloat16)
    ah = torch.randn(w.H, device=device, generator=ggen)
    gate_o = torch.empty((Tg, w.H * w.d), dtype=torch.bfloat16, device=device)
    g_o = torch.empty((Tg, w.H, w.d), dtype=torch.float32, device=device)
    z_o = torch.empty((Tg, rk), dtype=torch.bfloat16, device=device)
    gstep = lambda: kda.kda_gate_generator(xg, wga, wgb, ah, w.H, w.d, gate=gate_o, g=g_o, z=z_o, stream=stream)
    gsteps = max(10, args.steps // 4)
    ms_gate, ms_gate_launch, _ = timed(gstep, gsteps, args.warmup, stream, dist)
    gflops = 2 * Tg * hid * (w.H * w.d + rk) + 2 * Tg * rk * w.H * w.d
    gate_tflops = gflops / (ms_gate_launch * 1e-3) / 1e12
    del xg, wga, wgb, ah, gate_o, g_o, z_o

    # ---------------- backward of the prefill (kda_chunk_bwd): bf16 inputs, products on the tensor cores ----------------
    qb, kb, vb, gb, bb = make_prefill_inputs(w, device)
    dob = fill_device(w.seed, ks.TID_DO, ks.NORMAL, (w.T, w.H, w.d), "bf16", device=device)
    wsb = torch.empty(kda.kda_chunk_bwd_workspace_size(1, w.T, w.H), dtype=torch.uint8, device=device)
    bstep = lambda: kda.kda_chunk_bwd(qb, kb, vb, gb, bb, dob, workspace=wsb, stream=stream)
    bsteps = max(5, args.steps // 10)
    ms_bwd, ms_bwd_launch, _ = timed(bstep, bsteps, args.warmup, stream, dist)
    bwd_flops = w.T * w.H * bwd_flops_per_token_head()
    bwd_tflops = bwd_flops / (ms_bwd_launch * 1e-3) / 1e12
    bwd_bytes = w.T * w.H * bwd_bytes_per_token_head()
    bwd_gbs = bwd_bytes / (ms_bwd_launch * 1e-3) / 1e9
    del qb, kb, vb, gb, bb, dob, wsb

    # ---------------- front end + prefill from raw inputs: fused vs two passes (the long workload's path) ----
    gf = fill_device(wf.seed, ks.TID_G, ks.NEG_SOFTPLUS5, (wf.T, wf.H, wf.d), "f32", device=device)
    bf = fill_device(wf.seed, ks.TID_BETA, ks.SIGMOID, (wf.T, wf.H), "f32", device=device)
    of = torch.empty((wf.T, wf.H, wf.d), dtype=torch.bfloat16, device=device)
    fsf = torch.empty((1, wf.H, wf.d, wf.d), dtype=torch.float32, device=device)
    wsf = torch.empty(kda.kda_chunk_fwd_workspace_size(1, wf.T, wf.H, torch.bfloat16, False)[0], dtype=torch.uint8,
                      device=device)
    fused = lambda: kda.kda_chunk_fwd_frontend(*xf, cwf, gf, bf, wf.H, o=of, final_state=fsf, workspace=wsf,
                                               stream=stream)
    def two_pass():
        kda.kda_shortconv_l2norm(*xf, cwf, wf.H, q=outs[0], k=outs[1], v=outs[2], stream=stream)
        kda.kda_chunk_fwd(outs[0], outs[1], outs[2], gf, bf, o=of, final_state=fsf, workspace=wsf, stream=stream)
    lsteps = max(10, args.steps // 10)
    ms_fused, _, _ = timed(fused, lsteps, args.warmup, stream, dist)
    ms_two, _, _ = timed(two_pass, lsteps, args.warmup, stream, dist)
    del xf, outs, gf, bf, of, fsf, wsf

    # ---------------- the same 8K prefill through kda_chunk_fwd_noalloc (static 64 MiB scratch) ----------
    qn, kn, vn, gn, bn = make_prefill_inputs(w, device)
    nsteps = max(5, args.steps // 4)
    ms_na, _, _ = timed(lambda: kda.kda_chunk_fwd_noalloc(qn, kn, vn, gn, bn, o=o, final_state=fs, stream=stream),
                        nsteps, args.warmup, stream, dist)
    del qn, kn, vn, gn, bn

    # ---------------- the tiny fp32 workload (fp32 path on the CUDA cores; latency-bound) ----------------
    wt = ks.workload("tiny_fp32")
    from kda_synth.device import to_device
    tin = [to_device(x) for x in (wt.qkv("q"), wt.qkv("k"), wt.qkv("v"), wt.g(), wt.beta())]
    ot = torch.empty((wt.T, wt.H, wt.d), dtype=torch.float32, device=device)
    fst = torch.empty((1, wt.H, wt.d, wt.d), dtype=torch.float32, device=device)
    tsteps = max(50, args.steps)
    ms_tiny, _, _ = timed(lambda: kda.kda_chunk_fwd(*tin, o=ot, final_state=fst, stream=stream), tsteps,
                          args.warmup, stream, dist)
    tiny_bytes = prefill_bytes(wt.T, wt.H, 1) + wt.T * wt.H * (2 * 3 * 128 + 2 * 128)  # fp32 q, k, v, o
    del tin, ot, fst

    # ---------------- varlen_32 at full size: 32 packed sequences, per-sequence initial states ----------------
    # Values are drawn on the device (torch's seeded generator, the workload's distributions): the host
    # generator would take minutes for 65 GB of inputs; the parity tests check this workload's bits.
    wv = ks.workload("varlen_32")
    gv_ = torch.Generator(device=device).manual_seed(53004)
    Tv, Nv = wv.T, wv.N
    qv = device_draws((Tv, wv.H, wv.d), "unit", torch.bfloat16, gv_)
    kv = device_draws((Tv, wv.H, wv.d), "unit", torch.bfloat16, gv_)
    vv = device_draws((Tv, wv.H, wv.d), "normal", torch.bfloat16, gv_)
    gvv = device_draws((Tv, wv.H, wv.d), "neg5sig", torch.float32, gv_)
    bv = device_draws((Tv, wv.H), "sigmoid", torch.float32, gv_)
    s0v = device_draws((Nv, wv.H, wv.d, wv.d), "normal", torch.float32, gv_) * wv.init_state_std
    cuv = torch.from_numpy(wv.cu_seqlens()).to(device)
    ov = torch.empty((Tv, wv.H, wv.d), dtype=torch.bfloat16, device=device)
    fsv = torch.empty_like(s0v)
    full_v, _ = kda.kda_chunk_fwd_workspace_size(Nv, Tv, wv.H, torch.bfloat16, True)
    wsv = torch.empty(min(full_v, 24 << 30), dtype=torch.uint8, device=device)
    vsteps = max(3, args.steps // 10)
    ms_var, ms_var_launch, _ = timed(lambda: kda.kda_chunk_fwd(qv, kv, vv, gvv, bv, s0v, cuv, o=ov, final_state=fsv,
                                                               workspace=wsv, stream=stream),
                                     vsteps, args.warmup, stream, dist)
    var_bytes = prefill_bytes(Tv, wv.H, Nv, init_state=True)
    var_rows_fit = (wsv.numel() - (2 * wv.H * 128 * 128 * 4 + -(-(Nv + 1) * 4 // 1024) * 1024)) // (wv.H * 82432)
    var_launches = prefill_launches(Tv // 64 + Nv, var_rows_fit, True)
    var_gbs = var_bytes / (ms_var_launch * 1e-3) / 1e9
    del qv, kv, vv, gvv, bv, s0v, cuv, ov, fsv, wsv
    torch.cuda.empty_cache()

    # ---------------- long_256k at full size: raw q, k, v -> front end -> chunk_kda -> sigmoid output gate ----------
    wl = ks.workload("long_256k")
    gl_ = torch.Generator(device=device).manual_seed(53005)
    Tl, Cl = wl.T, wl.H * wl.d
    xl = [device_draws((Tl, Cl), "normal", torch.bfloat16, gl_) for _ in range(3)]
    cwl = (device_draws((3 * Cl, 4), "normal", torch.float32, gl_) * wl.conv_w_std).to(torch.bfloat16)
    gll = device_draws((Tl, wl.H, wl.d), "negsp5", torch.float32, gl_)
    bl = device_draws((Tl, wl.H), "sigmoid", torch.float32, gl_)
    gatel = device_draws((Tl, Cl), "normal", torch.bfloat16, gl_)
    ol = torch.empty((Tl, wl.H, wl.d), dtype=torch.bfloat16, device=device)
    fsl = torch.empty((1, wl.H, wl.d, wl.d), dtype=torch.float32, device=device)
    full_l, _ = kda.kda_chunk_fwd_workspace_size(1, Tl, wl.H, torch.bfloat16, False)
    wsl = torch.empty(full_l, dtype=torch.uint8, device=device)
    lsteps5 = max(3, args.steps // 10)
    ms_long, ms_long_launch, _ = timed(lambda: kda.kda_chunk_fwd_frontend(*xl, cwl, gll, bl, wl.H, out_gate=gatel, o=ol,
                                                                          final_state=fsl, workspace=wsl,
                                                                          stream=stream),
                                       lsteps5, args.warmup, stream, dist)
    qkv_l = [torch.empty((Tl, wl.H, wl.d), dtype=torch.bfloat16, device=device) for _ in range(3)]

    def long_two_pass():
        kda.kda_shortconv_l2norm(*xl, cwl, wl.H, q=qkv_l[0], k=qkv_l[1], v=qkv_l[2], stream=stream)
        kda.kda_chunk_fwd(*qkv_l, gll, bl, out_gate=gatel, o=ol, final_state=fsl, workspace=wsl, stream=stream)
    ms_long2, _, _ = timed(long_two_pass, lsteps5, args.warmup, stream, dist)
    # fused minimum per token: raw q, k, v (3 x 12288 bf16) + g fp32 + beta + gate bf16 + o bf16
    long_bytes_tok = 3 * Cl * 2 + Cl * 4 + wl.H * 4 + Cl * 2 + Cl * 2
    long_bytes = Tl * long_bytes_tok + 3 * Cl * 4 * 2 + wl.H * wl.d * wl.d * 4
    long_gbs = long_bytes / (ms_long_launch * 1e-3) / 1e9
    del xl, cwl, gll, bl, gatel, ol, fsl, wsl, qkv_l
    torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; no dataset or weights involved)",
        "config": {"workload": f"{w.name}: prefill N={w.N} T={w.T} H={w.H} dk=dv={w.d} chunk={w.chunk}, "
                               "bf16 q,k,v (q,k L2-normalised), fp32 g=-5*sigmoid(z), beta=sigmoid(z), S0=0",
                   "global_batch": w.N * world, "seq_len": w.T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1.2 GB per step), no flush"},
        "clocks": clk,
        "e2e": {"value": w.T * world / (ms_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": ms_e2e,
                "note": "pinned host buffers; H2D of step i+1 and D2H of step i-1 overlap step i's kernel"},
        "gpu_launches": args.steps * launches_per_call,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak,
                     "traffic": measured_traffic("kda_chunk_fwd", FWD_SOURCES, w.name),
                     "peak_source": peak_src,
                     "kernel": "kda_chunk_fwd (bf16): chunk_offsets_kernel + chunk_prep_kernel + chunk_state_kernel "
                               "per range of chunk rows, timed as one call", "algorithmic_bytes_per_launch": pbytes,
                     "workspace_bytes": ws_full,
                     "tensor": {"achieved_tflops": achieved_tflops, "peak_tflops": tc_peak,
                                "frac": achieved_tflops / tc_peak,
                                "algorithmic_flops_per_launch": pflops}},
        "decode": {"workload": "decode_64: 64 sequences x 1 token, H=96, d=128, fused ShortConv+SiLU+L2norm, "
                               "in-place fp32 state N(0,0.02)",
                   "value": dec_gbs, "unit": "GB/s", "ms_per_step": ms_dec, "steps": dsteps, "gpu_launches": 2 * dsteps,
                   "algorithmic_bytes_per_launch": dbytes, "clocks": dclk,
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
                                "frac": dec_gbs / hbm_peak,
                                "traffic": measured_traffic("recurrent_step_kernel", "kda_recurrent.cu", wd.name),
                                "peak_source": peak_src}},
        "frontend": {"workload": "frontend_32k: raw q, k, v bf16 [32768, 12288] -> ShortConv(4)+SiLU+L2norm -> "
                                 "bf16 [32768, 96, 128] x 3",
                     "value": fe_gbs, "unit": "GB/s", "ms_per_step": ms_fe, "steps": fsteps, "gpu_launches": fsteps,
                     "algorithmic_bytes_per_launch": fe_bytes,
                     "roofline": {"bound": "hbm", "achieved": fe_gbs, "peak": hbm_peak, "unit": "GB/s",
                                  "frac": fe_gbs / hbm_peak,
                                  "traffic": measured_traffic("shortconv_kernel", "kda_frontend.cu+kda_frontend.cuh", wf.name),
                                  "peak_source": peak_src}},
    }
    if seg is not None:
        line["segmented_prefill"] = seg
    line["gate_generator"] = {
        "workload": f"x bf16 [{Tg}, {hid}] -> output gate bf16 [{Tg}, {w.H * w.d}] and decay gate g = max(-5, "
                    f"-softplus(x W_a^T W_b^T + a_h)) fp32 [{Tg}, {w.H}, {w.d}], rank {rk}; random weights",
        "value": gate_tflops, "unit": "TFLOP/s", "ms_per_step": ms_gate, "steps": gsteps, "gpu_launches": 2 * gsteps,
        "algorithmic_flops_per_launch": gflops,
        "roofline": {"bound": "tensor", "achieved": gate_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": gate_tflops / tc_peak,
                     "traffic": measured_traffic("gemm_gate_kernel", "kda_gate.cu", "gates_8k"), "peak_source": peak_src,
                     "kernel": "gemm_gate_kernel x2 (x [W_gate ; W_a]^T, then the rank product with the gate epilogue)"}}
    bwd_traffic = measured_traffic("kda_chunk_bwd", BWD_SOURCES, w.name)
    line["backward"] = {
        "workload": f"{w.name}: kda_chunk_bwd of the prefill (bf16 q, k, v and dL/do; fp32 gradients of q, k, v, g, "
                    "beta, S0), dL/dS_final = 0",
        "value": w.T * world / (ms_bwd * 1e-3), "unit": "tokens/s", "ms_per_step": ms_bwd, "steps": bsteps,
        "gpu_launches": 5 * bsteps, "algorithmic_bytes_per_launch": bwd_bytes,
        "algorithmic_flops_per_launch": bwd_flops, "products_tflops": bwd_tflops,
        "roofline": {"bound": "hbm", "achieved": bwd_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": bwd_gbs / hbm_peak, "traffic": bwd_traffic,
                     "traffic_GB_s": (bwd_traffic / (ms_bwd_launch * 1e-3) / 1e9) if bwd_traffic else None,
                     "peak_source": peak_src,
                     "kernel": "bwd_prep_tc_kernel + bwd_fwd_state_tc_kernel + bwd_state_tc_kernel + "
                               "bwd_chunk_ab_tc_kernel + bwd_dbeta_kernel, timed as one call"}}
    line["fused_prefill"] = {
        "workload": "frontend_32k raw q, k, v bf16 [32768, 12288] + g = max(-5, -softplus(z)), beta -> "
                    "ShortConv(4)+SiLU+L2norm -> chunk_kda (the long workload's path at 32K tokens)",
        "value": wf.T * world / (ms_fused * 1e-3), "unit": "tokens/s", "ms_per_step": ms_fused, "steps": lsteps,
        "gpu_launches": lsteps * prefill_launches(-(-wf.T // 64), -(-wf.T // 64), False, fused=True),
        "two_pass_value": wf.T * world / (ms_two * 1e-3), "two_pass_ms_per_step": ms_two,
        "note": "kda_chunk_fwd_frontend vs kda_shortconv_l2norm + kda_chunk_fwd; same output bits"}
    line["noalloc_prefill"] = {
        "workload": f"{w.name} through kda_chunk_fwd_noalloc: the library's static 64 MiB scratch, chunk ranges "
                    "of 6 rows one after the other on the caller's stream",
        "value": w.T * world / (ms_na * 1e-3), "unit": "tokens/s", "ms_per_step": ms_na, "steps": nsteps}
    line["varlen_32"] = {
        "workload": f"varlen_32: {Nv} packed sequences (1K..32K tokens, sum {Tv}), H={wv.H}, bf16 q,k,v, fp32 g, beta, "
                    "initial states N(0, 0.02); values drawn on the device with the workload's distributions",
        "value": Tv * world / (ms_var * 1e-3), "unit": "tokens/s", "ms_per_step": ms_var, "steps": vsteps,
        "gpu_launches": vsteps * var_launches, "algorithmic_bytes_per_launch": var_bytes,
        "roofline": {"bound": "hbm", "achieved": var_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": var_gbs / hbm_peak,
                     "traffic": measured_traffic("kda_chunk_fwd", FWD_SOURCES, "varlen_32"),
                     "peak_source": peak_src}}
    line["long_256k"] = {
        "workload": f"long_256k: T={Tl}, raw q,k,v bf16 [{Tl}, {Cl}] -> ShortConv(4)+SiLU+L2norm -> chunk_kda with "
                    "g = max(-5, -softplus(z)) -> o * sigmoid(gate); kda_chunk_fwd_frontend (fused)",
        "value": Tl * world / (ms_long * 1e-3), "unit": "tokens/s", "ms_per_step": ms_long, "steps": lsteps5,
        "gpu_launches": lsteps5 * prefill_launches(-(-Tl // 64), -(-Tl // 64), False, fused=True),
        "algorithmic_bytes_per_launch": long_bytes,
        "two_pass_value": Tl * world / (ms_long2 * 1e-3), "two_pass_ms_per_step": ms_long2,
        "roofline": {"bound": "hbm", "achieved": long_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": long_gbs / hbm_peak,
                     "traffic": measured_traffic("kda_chunk_fwd_frontend", FWD_SOURCES, "long_256k"),
                     "peak_source": peak_src}}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    r3 = lambda x: float(f"{x:.4g}")
    # every configuration's figure, last and compact (it must survive a truncated log tail)
    line["per_config"] = {
        "tiny_fp32": {"tok_s": r3(wt.T * world / (ms_tiny * 1e-3)), "ms": r3(ms_tiny), "bound": "latency",
                      "hbm_frac": r3(tiny_bytes / (ms_tiny * 1e-3) / 1e9 / hbm_peak)},
        "prefill_8k": {"tok_s": r3(value), "ms": r3(ms_step), "hbm_frac": r3(achieved_gbs / hbm_peak),
                       "tensor_frac": r3(achieved_tflops / tc_peak)},
        "decode_64": {"GB_s": r3(dec_gbs), "ms": r3(ms_dec), "hbm_frac": r3(dec_gbs / hbm_peak)},
        "varlen_32": {"tok_s": r3(Tv * world / (ms_var * 1e-3)), "ms": r3(ms_var), "hbm_frac": r3(var_gbs / hbm_peak)},
        "long_256k": {"tok_s": r3(Tl * world / (ms_long * 1e-3)), "ms": r3(ms_long),
                      "hbm_frac": r3(long_gbs / hbm_peak), "two_pass_ms": r3(ms_long2)},
        "noalloc_8k_ms": r3(ms_na), "backward_8k_ms": r3(ms_bwd), "peak_GB_s": hbm_peak}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline leg and --impl reference)
# ------------------------------------------------------------------------------------------------

def oracle_sample(w, heads, t_len):
    import numpy as np

    import kda_synth as ks
    d = w.d
    Hs = len(heads)
    q = np.empty((t_len, Hs, d)); k = np.empty((t_len, Hs, d)); v = np.empty((t_len, Hs, d))
    g = np.empty((t_len, Hs, d)); b = np.empty((t_len, Hs))
    for i, h in enumerate(heads):
        q[:, i] = ks.to_f64(w.head_rows(ks.TID_Q, ks.UNIT_GROUPS, h, w.dtype, p1=float(d), t1=t_len))
        k[:, i] = ks.to_f64(w.head_rows(ks.TID_K, ks.UNIT_GROUPS, h, w.dtype, p1=float(d), t1=t_len))
        v[:, i] = ks.to_f64(w.head_rows(ks.TID_V, ks.NORMAL, h, w.dtype, t1=t_len))
        g[:, i] = w.head_rows(ks.TID_G, w.g_kind, h, "f32", t1=t_len)
        b[:, i] = w.head_beta(h, 0, t_len)
    return q, k, v, g, b


def cpu_baseline(w, budget_s=20.0):
    """The oracle as it stands on this host's cores, on a bounded sample of the workload:
    whole sequences of the first heads, as many heads as fit about half of ``budget_s``."""
    import oracle
    oracle.build()
    cores = oracle.threads()
    heads = min(w.H, max(1, cores))
    t_len = w.T
    while True:
        sample = oracle_sample(w, list(range(heads)), t_len)
        t0 = time.perf_counter()
        oracle.kda_tokenloop(*sample)
        dt = time.perf_counter() - t0
        if heads >= w.H or dt >= 0.25 * budget_s:
            break
        heads = min(w.H, max(heads + 1, int(heads * 0.5 * budget_s / max(dt, 1e-3))))
    token_heads = t_len * heads
    return {"value": token_heads / w.H / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{w.name}: heads 0..{heads - 1} of {w.H}, all {t_len} tokens "
                      f"(fp64 per-token loop, {token_heads} token-heads, {dt:.1f} s); "
                      f"tokens/s = token-heads / {w.H} / seconds"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import kda_synth as ks
    import oracle
    oracle.build()
    w = ks.workload(args.workload)
    cores = oracle.threads()
    heads = list(range(min(w.H, cores)))
    t_len = min(w.T, 256)
    sample = oracle_sample(w, heads, t_len)
    for _ in range(args.warmup):
        oracle.kda_tokenloop(*sample)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.kda_tokenloop(*sample)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    value = t_len * len(heads) / w.H / sec
    desc = (f"{w.name}: heads 0..{len(heads) - 1} of {w.H}, tokens 0..{t_len - 1} per step "
            f"(fp64 per-token loop); tokens/s = token-heads / {w.H} / seconds")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: prefill N={w.N} T={w.T} H={w.H} dk=dv={w.d} (bounded sample per step)",
                   "global_batch": w.N, "seq_len": w.T, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_8k", choices=["prefill_8k"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
