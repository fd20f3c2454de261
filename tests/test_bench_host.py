"""Host-side pieces of bench.py, on CPU: byte accounting, the max-over-ranks / sum-of-
units aggregation with two gloo ranks, and the profile-summary parser."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from block_quantized_matmul_gq_gb300 import workloads  # noqa: E402


def test_step_bytes_tinyllama():
    nb = bench.step_bytes(workloads.tinyllama_decode_set(), 1, 18)
    assert nb["weights"] == 581_861_376
    assert nb["x"] == 4 * (22 * (6 * 2048 + 5632) + 2048)
    assert nb["y"] == 4 * (22 * (2 * 2048 + 2 * 256 + 2 * 5632 + 2048) + 32000)
    assert nb["total"] == nb["weights"] + nb["x"] + nb["y"]


def test_step_bytes_q4_k_superblocks():
    # 144 bytes per 256 weights: the same 0.5625 bytes per weight as Q4_0
    nb = bench.step_bytes(workloads.tinyllama_decode_set(), 1, 144, 256)
    assert nb["weights"] == 581_861_376


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == (2.0, 300.0)


def test_aggregate_single_rank():
    assert bench.aggregate(0.5, 7.0, 1) == (0.5, 7.0)


def test_profile_summary_requires_current_kernel(tmp_path, monkeypatch):
    p = tmp_path / "summary.md"
    p.write_text(f"traffic_bytes_per_launch: 123\nkernel_source_sha256_16: {bench.kernel_source_hash()}\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(p))
    assert bench.profiled_traffic() == 123
    p.write_text("traffic_bytes_per_launch: 123\nkernel_source_sha256_16: 0000\n")
    assert bench.profiled_traffic() is None


def test_kernel_hash_ignores_comments_only():
    src = "// header\nint f(int a) {\n    /* block\n comment */ return a + 1;  // tail\n}\n"
    same = "int f(int a) {\n\n  return a + 1;\n}\n// a new note\n"
    changed = "int f(int a) {\n    return a + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(changed)


def test_reference_arm_sample_sizes():
    shapes = workloads.tinyllama_decode_set()[:3]
    sample = bench.oracle_sample(shapes, 2, 2)
    assert [r for _, r, _, _ in sample] == [2, 2, 2]
    assert bench.sample_bytes(sample) == sum(2 * 18 * s.K // 32 + 4 * s.K + 8 for s in shapes)


def test_oracle_rows_time_runs_every_slice(monkeypatch):
    """The all-core oracle timing cuts each matrix's rows into one slice per thread and
    runs the unchanged oracle on every slice: together the slices are the matrix."""
    import oracle
    seen = []
    real = oracle.mul_mat

    def spy(t, blocks, M, K, X):
        seen.append((K, blocks.copy()))
        return real(t, blocks, M, K, X)

    monkeypatch.setattr(oracle, "mul_mat", spy)
    step = workloads.tinyllama_decode_set()
    sample = bench.oracle_sample([step[0], step[6]], 7, 2)     # K = 2048 and 5632
    assert bench.oracle_rows_time("q4_0", sample, 3) > 0
    assert len(seen) == 3 * len(sample)
    for blocks, r, K, X in sample:
        parts = [b for k, b in seen if k == K]
        assert sum(len(b) for b in parts) == r
        assert sorted(bytes(row) for b in parts for row in b) == sorted(bytes(row) for row in blocks)
    assert bench.host_cores() >= 1


def test_summarize_keeps_every_workload():
    row = {"N": 1, "us": 3.0, "GBps": 800.0, "frac": 0.12}
    dec = {"single_q4_0_2048x2048": {"per_N": [row], "launch_floor": {"us": 2.0}},
           "tinyllama_decode_q4_0": {"per_N": [dict(row, N=2)]},
           "tinyllama_decode_q8_0": {"per_N": [row]},
           "llama7b_decode_q4_0": {"per_N": [row, dict(row, N=16)]},
           "tinyllama_decode_q4_k": {"per_N": [row, dict(row, N=4)]}}
    pf = {"tinyllama_prefill_n512": {"tflops": 900.0, "frac": 0.46},
          "llama7b_prefill_n2048_q8_0": {"tflops": 1100.0, "frac": 0.56}}
    s = bench.summarize(dec, pf, {"decode_us": {"single_2048x2048_N1": 4.0}}, 6796.9)
    assert s["w1_single_q4_0_2048x2048_N1"] == [3.0, 800.0, 0.12]
    assert s["w1_launch_floor_us"] == 2.0
    assert set(s["w5_llama7b_q4_0"]) == {"N1", "N16"}
    assert set(s["w2_tinyllama_q4_k"]) == {"N1", "N4"}
    assert s["prefill_llama7b_prefill_n2048_q8_0"] == [1100.0, 0.56]
