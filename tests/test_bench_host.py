"""Host-side logic of bench.py without a GPU: the max-over-ranks reduction with two gloo
ranks (the replica timing of a multi-GPU run), and the traffic lookup that must go null
once the kernel source no longer matches its ncu capture."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.reduce_max(10.0 + 5.0 * rank, dist)
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"r{r}.json"))["max"] == 15.0


def test_reduce_max_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, None) == 3.5


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    h = bench.kernel_source_hash("kda_recurrent.cu")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"recurrent_step_kernel@decode_64": {
        "workload": "decode_64", "source_sha256_16": h, "dram_bytes_per_launch": 123}}))
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "gated_delta_rule_53_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = open(os.path.join(real_root, "gated_delta_rule_53_gb300", "csrc", "kda_recurrent.cu"), "rb").read()
    (csrc / "kda_recurrent.cu").write_bytes(src)
    assert bench.measured_traffic("recurrent_step_kernel", "kda_recurrent.cu", "decode_64") == 123
    assert bench.measured_traffic("recurrent_step_kernel", "kda_recurrent.cu", "other") is None
    (csrc / "kda_recurrent.cu").write_bytes(src + b"\n// changed\n")
    assert bench.measured_traffic("recurrent_step_kernel", "kda_recurrent.cu", "decode_64") is None


def test_backward_chunk_slots_are_distinct_and_bounded():
    """The backward keeps per-chunk data at slot (bos_n + 64 j) // 64 + n for chunk j of sequence n: over
    random packed batches (empty sequences included) the slots are distinct and below T // 64 + N + 1,
    the size its workspace allocates."""
    import numpy as np
    rng = np.random.default_rng(5)
    for _ in range(200):
        N = int(rng.integers(1, 40))
        lengths = rng.integers(0, 300, size=N) * (rng.random(N) > 0.2)
        bos = np.concatenate([[0], np.cumsum(lengths)])
        T = int(bos[-1])
        slots = [(int(bos[n]) + 64 * j) // 64 + n for n in range(N) for j in range((int(lengths[n]) + 63) // 64)]
        assert len(set(slots)) == len(slots)
        assert all(0 <= s < T // 64 + N + 1 for s in slots)


def test_backward_roofline_constants():
    import bench
    # per chunk of 64 tokens and head: 12 C d^2 + 10 C^2 d flop, per token-head
    assert bench.bwd_flops_per_token_head() == (12 * 64 * 128 * 128 + 10 * 64 * 64 * 128) / 64
    # bytes per token-head: q, k, v, dL/do bf16 (4 x 256) + g fp32 (512) + beta (4) read; dq, dk, dv, dg fp32
    # (4 x 512) + dbeta (4) written
    assert bench.bwd_bytes_per_token_head() == 1024 + 512 + 4 + 2048 + 4
    assert abs(bench.fp32_alu_peak_tflops() - 80.54784) < 1e-9


def test_source_hash_of_several_files():
    import hashlib
    import bench
    csrc = os.path.join(bench.ROOT, "gated_delta_rule_53_gb300", "csrc")
    names = bench.BWD_SOURCES.split("+")
    joined = b"".join(open(os.path.join(csrc, n), "rb").read() for n in names)
    assert bench.kernel_source_hash(bench.BWD_SOURCES) == hashlib.sha256(joined).hexdigest()[:16]
    assert bench.kernel_source_hash(names[0]) == hashlib.sha256(open(os.path.join(csrc, names[0]), "rb").read()).hexdigest()[:16]


def test_clock_sampler_parses_and_summarises():
    sys.path.insert(0, ROOT)
    import bench
    lines = ["0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 1980, 2070, 1380.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "garbage", "0, [N/A], 2070, 0, 0, Not Active, Not Active, Not Active, Not Active"]
    got = bench.ClockSampler.summarise(bench.ClockSampler.parse_smi(lines), "nvidia-smi")
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                   "source": "nvidia-smi"}
    assert bench.ClockSampler.summarise([], "nvml")["sm_mhz"] is None


def test_clock_sampler_polls_nvml_and_falls_back(monkeypatch):
    """The NVML path samples on its own thread until stopped; without NVML and nvidia-smi the line
    says the clocks are unavailable instead of failing."""
    sys.path.insert(0, ROOT)
    import time

    import bench

    class FakeNvml:
        closed = False

        def __init__(self, gpu_id):
            assert gpu_id == "3"

        def sample(self):
            return (1965.0, 2070.0, ["sw_power_cap"])

        def close(self):
            FakeNvml.closed = True

    monkeypatch.setattr(bench, "_Nvml", FakeNvml)
    cs = bench.ClockSampler("3", period_s=0.001)
    cs.start()
    time.sleep(0.05)
    got = cs.stop()
    assert got["source"] == "nvml" and got["samples"] >= 2 and got["sm_mhz"] == 1965.0
    assert got["reasons"] == ["sw_power_cap"] and FakeNvml.closed

    def no_nvml(gpu_id):
        raise OSError("no libnvidia-ml")

    def no_smi(*a, **k):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench, "_Nvml", no_nvml)
    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    cs = bench.ClockSampler("0")
    cs.start()
    assert cs.stop()["sm_mhz"] is None


def test_prefill_launch_count_follows_the_range_rule():
    """gpu_launches of the prefill lines: the chunk-offset kernel only for packed sequences, the front end of
    v only for the fused call, and an operand kernel + a state pass per range (the library's rule: about eight
    overlapped ranges of at least 128 rows from 256 rows on, else ranges of what the workspace holds)."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.prefill_launches(128, 128, False) == 2                 # 8K tokens: one range
    assert bench.prefill_launches(128, 6, False) == 2 * 22              # the 64 MiB scratch: 6 rows per range
    assert bench.prefill_launches(512, 512, False, fused=True) == 9     # 32K fused: 4 ranges of 128 + v
    assert bench.prefill_launches(4096, 4096, False, fused=True) == 17  # 256K fused: 8 ranges of 512 + v
    assert bench.prefill_launches(8172, 3033, True) == 1 + 2 * 8        # packed, capped workspace: 8 of 1022
    assert bench.prefill_launches(300, 200, True) == 1 + 2 * 2          # workspace below 256 rows: serial
    assert bench.prefill_launches(0, 5, False) == 1                     # empty call: the state pass alone
