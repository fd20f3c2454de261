"""Benchmark: the TinyLLaMA-1.1B decode step (155 Q4_0 matrix-vector products, N = 1)
through libgq, as decode mul_mat HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

One step is one pass over the whole weight set: every q/k/v/o/gate/up/down projection of
the 22 layers plus lm_head (581,861,376 bytes of Q4_0 blocks), each against its own
seeded N(0, 1) activation vector, run as one gq_mul_mat_batched launch replayed from a
CUDA graph. The weights (582 MB) are larger than the 129 MB L2, so every step streams
them from HBM. Prints one JSON line (rank 0).

--impl reference times the CPU oracle (oracle/, unchanged, on every host core: each thread
runs it on its own rows of every matrix) on a bounded sample of the same workload: an
R-row slice of every matrix, R sized so the run ends in minutes.
Under torchrun every rank runs an independent replica of the step (the decode step does
not shard across GPUs here: "replicas only"); value sums the ranks' bytes over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode mul_mat HBM GB/s (% of peak); prefill TFLOP/s (% of bf16 peak)"
UNIT = "GB/s"
WORKLOAD_ID = 2
WORKLOAD_NAME = "TinyLLaMA-1.1B decode step, Q4_0 weights, N=1 (155 matmuls: 22 layers x " \
                "q/k/v/o/gate/up/down + lm_head)"
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gemv_stream_tinyllama_decode_q4_0.md")
KERNEL_SOURCES = [os.path.join(ROOT, "block_quantized_matmul_gq_gb300", "csrc", f)
                  for f in ("gq_gemv.cu", "gq_device.cuh")]


# --------------------------------------------------------------------------------------
# helpers (host-side; also exercised by tests/test_bench_host.py on CPU)
# --------------------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(seconds: float, units: float, world: int, device=None):
    """Slowest rank's time and the sum of all ranks' units (replicas: weak scaling)."""
    if world == 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def step_bytes(shapes, N: int, block_bytes: int, block_weights: int = 32) -> dict:
    w = sum(s.M * (s.K // block_weights) * block_bytes for s in shapes)
    x = sum(N * s.K * 4 for s in shapes)
    y = sum(N * s.M * 4 for s in shapes)
    return {"weights": w, "x": x, "y": y, "total": w + x + y}


def replay_median_s(g, dev, replays: int) -> float:
    """Median time of one replay of CUDA graph g over `replays` replays after warm-up
    (seconds). The replays are queued back to back, each bracketed by its own pair of
    CUDA events on the current stream, with one synchronize after the last, so that no
    replay starts on an idle GPU."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(1, replays))]
    for e0, e1 in evs:
        e0.record()
        g.replay()
        e1.record()
    torch.cuda.synchronize(dev)
    times = sorted(e0.elapsed_time(e1) / 1e3 for e0, e1 in evs)
    return times[len(times) // 2]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """The source without comments, blank lines or indentation: what the compiler sees
    (a comment-only edit leaves the kernel, and so its counters, unchanged)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.strip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(units_scale: float = 1.0):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return int(m.group(1)) * units_scale


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


def emit(obj):
    print(json.dumps(obj), flush=True)


# --------------------------------------------------------------------------------------
# reference arm: the CPU oracle on a bounded sample
# --------------------------------------------------------------------------------------
def oracle_sample(shapes, rows: int, seed_workload: int):
    """A `rows`-row slice of every matrix (same shapes, seeds and distribution as the GPU
    arm's inputs, drawn on the CPU), quantized by the oracle; returns [(blocks, r, K, X)]."""
    import oracle
    from block_quantized_matmul_gq_gb300 import workloads
    out = []
    for j, s in enumerate(shapes):
        r = min(rows, s.M)
        W = workloads.weights(r, s.K, workloads.weight_seed(seed_workload, j)).numpy()
        X = workloads.activations(1, s.K, workloads.act_seed(seed_workload, 1, j)).numpy()
        out.append((oracle.quantize("q4_0", W), r, s.K, X))
    return out


def time_oracle(sample, reps: int):
    import oracle
    t0 = time.perf_counter()
    for _ in range(reps):
        for blocks, r, K, X in sample:
            oracle.mul_mat("q4_0", blocks, r, K, X)
    return time.perf_counter() - t0


def sample_bytes(sample) -> int:
    return sum(b.nbytes + X.nbytes + 4 * r * X.shape[0] for b, r, K, X in sample)


def cpu_baseline(shapes, target_s: float = 6.0) -> dict:
    """The oracle as it stands on the TinyLLaMA step, repeated for about target_s seconds:
    at all host cores on a (64 x cores)-row slice of every matrix (each thread runs it on
    its own 64 rows of every matrix), and at one thread on a 64-row slice."""
    cores = host_cores()
    res = {}
    for threads in (cores, 1):
        sample = oracle_sample(shapes, 64 * threads, WORKLOAD_ID)
        nbytes = sample_bytes(sample)
        one = max(oracle_rows_time("q4_0", sample, threads), 1e-3)
        reps = max(1, int(target_s / one))
        dt = sum(oracle_rows_time("q4_0", sample, threads) for _ in range(reps))
        res[threads] = (nbytes * reps / dt / 1e9, reps, dt)
    v, reps, dt = res[cores]
    v1, reps1, dt1 = res[1]
    return {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{64 * cores}-row slice of each of the 155 matrices (N=1; whole matrix "
                      f"where smaller), {reps} passes in {dt:.1f} s on {cores} host threads, "
                      f"64 rows of every matrix per thread",
            "single_core": {"value": round(v1, 4), "unit": UNIT, "cores": 1,
                            "sample": f"64-row slice of each matrix, {reps1} passes in "
                                      f"{dt1:.1f} s"}}


def run_reference(args, shapes):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = host_cores()
    # Per step: an R-row slice of every matrix on all host cores; R sized so the whole
    # run takes about 2 minutes.
    probe = oracle_sample(shapes, 4, WORKLOAD_ID)
    per_row = max(oracle_rows_time("q4_0", probe, 1), 1e-4) / 4 / cores
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(cores, min(4096, budget / per_row)))
    sample = oracle_sample(shapes, rows, WORKLOAD_ID)
    for _ in range(args.warmup):
        oracle_rows_time("q4_0", sample, cores)
    dt = sum(oracle_rows_time("q4_0", sample, cores) for _ in range(args.steps))
    nbytes = sample_bytes(sample)
    value = nbytes * args.steps / dt / 1e9
    desc = (f"{rows}-row slice of each of the 155 matrices per step (N=1), {cores} host "
            f"threads (rows of every matrix split between them)")
    emit({"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": {"workload": WORKLOAD_NAME, "sample": desc},
          "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                           "kind": "oracle", "sample": desc},
          "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


# --------------------------------------------------------------------------------------
# Prefill (tensor-core GEMM): TinyLLaMA gate / down / lm_head at N = 512 and the LLaMA-7B
# shapes at N = 2048, one gq_mul_mat_ws call per matrix, as TFLOP/s (2 M N K / time).
# --------------------------------------------------------------------------------------
PREFILL_SETS = [("tinyllama_prefill_n512", 4, 512), ("llama7b_prefill_n2048", 5, 2048)]


def prefill_measure(dev, reps: int = 10, iters: int = 20, only=None,
                    types=("q4_0", "q8_0", "q4_k"), rotate: bool = True):
    """Each prefill matrix as gq_mul_mat_ws calls replayed from a CUDA graph. Weight copies
    (distinct seeds) are rotated so that every call reads its weights from HBM, not from L2
    (TinyLLaMA gate / down are 6-7 MB, under the 129 MB L2); X and Y stay the same."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    peak_tf = measured_bf16_peak()
    out = {}
    for btype in types:
        for set_name, wl, N in PREFILL_SETS:
            shapes = workloads.tinyllama_prefill_set() if wl == 4 else workloads.llama7b_set()
            rows, tot_flop, tot_s = [], 0.0, 0.0
            for j, sh in enumerate(shapes):
                if only is not None and (set_name, sh.name) != only:
                    continue
                wbytes = sh.M * binding.row_bytes(btype, sh.K)
                copies = min(reps, max(1, -(-4 * L2_BYTES // wbytes))) if rotate else 1
                qs = []
                for c in range(copies):
                    W = workloads.weights(sh.M, sh.K, workloads.weight_seed(wl, j) + 100 * c,
                                          device=dev)
                    qs.append(binding.quantize(W, btype))
                    del W
                X = workloads.activations(N, sh.K, workloads.act_seed(wl, N, j), device=dev)
                Y = torch.empty((N, sh.M), device=dev)
                ws = torch.empty(max(256, binding.workspace_size(btype, sh.M, sh.K, N)),
                                 dtype=torch.uint8, device=dev)
                for c in range(3):
                    binding.mul_mat_ws(qs[c % copies], btype, sh.M, sh.K, X, ws, out=Y)
                torch.cuda.synchronize(dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for r in range(reps):
                        binding.mul_mat_ws(qs[r % copies], btype, sh.M, sh.K, X, ws, out=Y)
                g.replay()
                torch.cuda.synchronize(dev)
                rep_s = replay_median_s(g, dev, iters)
                sec = rep_s / reps
                flop = 2.0 * sh.M * N * sh.K
                tf = flop / sec / 1e12
                rows.append({"matrix": sh.name, "M": sh.M, "K": sh.K, "N": N,
                             "us": round(sec * 1e6, 2), "tflops": round(tf, 1),
                             "frac": round(tf / peak_tf, 4), "weight_copies_rotated": copies})
                tot_flop += flop
                tot_s += sec
                del qs, X, Y, ws, g
            if rows:
                tf = tot_flop / tot_s / 1e12
                key = set_name if btype == "q4_0" else f"{set_name}_{btype}"
                out[key] = {"type": btype, "tflops": round(tf, 1), "frac": round(tf / peak_tf, 4),
                            "matrices": rows}
        if binding.get_last_error() != 0:
            raise RuntimeError("device status word set during the prefill sets")
    return out


# Decode workloads reported beside the headline step (N tokens per call):
# (key, workload id, type, shapes, N values).
DECODE_SETS = [
    ("single_q4_0_2048x2048", 1, "q4_0", "single", (1,)),
    ("tinyllama_decode_q4_0", 2, "q4_0", "tinyllama", (2, 4, 8, 16)),
    ("tinyllama_decode_q8_0", 3, "q8_0", "tinyllama", (1, 2, 4, 8, 16)),
    ("llama7b_decode_q4_0", 5, "q4_0", "llama7b", (1, 16)),
    # the same TinyLLaMA weights (workload 2's seeds) in Q4_K super-blocks
    ("tinyllama_decode_q4_k", 2, "q4_k", "tinyllama", (1, 2, 4, 8, 16)),
]
L2_BYTES = 129 * 2 ** 20
STEPS_PER_GRAPH = 10


def decode_measure(dev, reps: int = 20, iters: int = 20) -> dict:
    """Each decode set as batched calls (one per step) replayed from a CUDA graph; weight
    sets smaller than 4x L2 are copied (distinct seeds) and rotated so every step reads
    its weights from HBM. GB/s counts weights + X + Y once per step."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    peak, _ = measured_peaks()
    out = {}
    for key, wl, btype, which, Ns in DECODE_SETS:
        shapes = {"single": [workloads.MatShape("proj", 2048, 2048)],
                  "tinyllama": workloads.tinyllama_decode_set(),
                  "llama7b": workloads.llama7b_set()}[which]
        bw = 256 if btype == "q4_k" else 32
        nb1 = step_bytes(shapes, 1, binding.block_bytes(btype), bw)
        copies = min(64, max(1, -(-4 * L2_BYTES // nb1["weights"])))
        sets = [QuantizedWeightSet.synthetic(wl if c == 0 else 100 * wl + c, shapes, btype, dev)
                for c in range(copies)]
        rows = []
        for N in Ns:
            nb = step_bytes(shapes, N, binding.block_bytes(btype), bw)
            runs = []
            for c, ws in enumerate(sets):
                xs, ys = ws.make_io(N, wl, dev)
                arrays = ws.problem_arrays(xs, ys)
                work = ws.workspace(arrays, N, dev)
                runs.append((ws, arrays, work, xs, ys))
            for ws, arrays, work, _, _ in runs:
                ws.run(arrays, N, workspace=work)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for r in range(reps):
                    ws, arrays, work, _, _ = runs[r % copies]
                    ws.run(arrays, N, workspace=work)
            g.replay()
            torch.cuda.synchronize(dev)
            rep_s = replay_median_s(g, dev, iters)
            sec = rep_s / reps
            gbs = nb["total"] / sec / 1e9
            rows.append({"N": N, "us": round(sec * 1e6, 2), "GBps": round(gbs, 1),
                         "frac": round(gbs / peak, 4),
                         "path": "CUDA-core decode" if N <= 2 else "tensor-core decode"})
            del runs, g
        if binding.get_last_error() != 0:
            raise RuntimeError("device status word set during the decode sets")
        out[key] = {"type": btype, "matmuls": len(shapes), "weight_bytes": nb1["weights"],
                    "weight_copies_rotated": copies, "per_N": rows}
        if which == "single":
            out[key]["launch_floor"] = launch_floor(dev, reps, iters)
        del sets
    return out


def per_matmul_measure(dev, iters: int = 20) -> dict:
    """Each distinct TinyLLaMA matrix shape alone at N = 1 (gq_mul_mat, one call per
    matrix), in Q4_0 and Q8_0: a graph of R calls, each on its own copy of the blocks so
    that the R copies (>= 4 x L2 together) are read from HBM; the median of `iters`
    replays, per call."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    peak, _ = measured_peaks()
    shapes = {"q_o_proj": (2048, 2048), "k_v_proj": (256, 2048), "gate_up_proj": (5632, 2048),
              "down_proj": (2048, 5632), "lm_head": (32000, 2048)}
    out = {"unit": "GB/s", "peak": peak, "N": 1}
    for btype in ("q4_0", "q8_0"):
        rows = {}
        for name, (M, K) in shapes.items():
            q = binding.quantize(workloads.weights(M, K, 9000 + M, device=dev), btype)
            R = int(min(2048, max(4, -(-4 * L2_BYTES // q.numel()))))
            copies = q.unsqueeze(0).expand(R, *q.shape).contiguous()   # R addresses
            X = workloads.activations(1, K, 9100 + K, device=dev)
            Y = torch.empty((1, M), device=dev)
            for r in range(3):
                binding.mul_mat(copies[r], btype, M, K, X, out=Y)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for r in range(R):
                    binding.mul_mat(copies[r], btype, M, K, X, out=Y)
            g.replay()
            torch.cuda.synchronize(dev)
            sec = replay_median_s(g, dev, iters) / R
            nbytes = q.numel() + 4 * (K + M)
            gbs = nbytes / sec / 1e9
            rows[name] = {"M": M, "K": K, "us": round(sec * 1e6, 2), "GBps": round(gbs, 1),
                          "frac": round(gbs / peak, 4), "copies_rotated": R}
            del g, copies, q
        out[btype] = rows
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set during the per-matmul sets")
    return out


def step_as_calls_measure(dev, ws, xs, ys, N: int, step_bytes_total: int, iters: int = 20,
                          steps: int = 5) -> dict:
    """The decode step as one gq_mul_mat call per matrix (155 launches) instead of one
    batched launch, in a graph of `steps` steps; median of `iters` replays, per step."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding
    peak, _ = measured_peaks()

    def step():
        for m, x, y in zip(ws.mats, xs, ys):
            binding.mul_mat(m.blocks, ws.btype, m.shape.M, m.shape.K, x, out=y)

    step()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(steps):
            step()
    g.replay()
    torch.cuda.synchronize(dev)
    sec = replay_median_s(g, dev, iters) / steps
    gbs = step_bytes_total / sec / 1e9
    return {"calls_per_step": len(ws.mats), "us": round(sec * 1e6, 2), "GBps": round(gbs, 1),
            "frac": round(gbs / peak, 4)}


def launch_floor(dev, reps: int = 20, iters: int = 20) -> dict:
    """The same call on a 1 x 256 matrix (144 bytes of blocks), timed exactly like the
    single 2048 x 2048 product: batched calls on one stream, each a programmatic dependent
    of the one before, replayed from a CUDA graph. What one call costs when it moves
    (almost) nothing: launch, grid start-up, one ring fill and the write of Y."""
    import torch
    from block_quantized_matmul_gq_gb300 import workloads
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    shapes = [workloads.MatShape("tiny", 1, 256)]
    ws = QuantizedWeightSet.synthetic(9, shapes, "q4_0", dev)
    xs, ys = ws.make_io(1, 9, dev)
    arrays = ws.problem_arrays(xs, ys)
    ws.run(arrays, 1)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            ws.run(arrays, 1)
    g.replay()
    torch.cuda.synchronize(dev)
    rep_s = replay_median_s(g, dev, iters)
    return {"M": 1, "K": 256, "us": round(rep_s / reps * 1e6, 2)}


def dense_context_measure(dev, reps: int = 20, iters: int = 20) -> dict:
    """Same-box context, not a target: torch.matmul on dense bf16 weights and bf16 X at the
    workload shapes (the dense path that quantized decode avoids, and the library GEMM
    that prefill competes with). Weight sets under 4x L2 are copied and rotated."""
    import torch
    from block_quantized_matmul_gq_gb300 import workloads
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)

    def mats(shapes, copies):
        return [[torch.randn((s.M, s.K), generator=gen, device=dev, dtype=torch.bfloat16)
                 for s in shapes] for _ in range(copies)]

    def timed(fn):
        fn(0)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in range(reps):
                fn(r)
        g.replay()
        torch.cuda.synchronize(dev)
        rep_s = replay_median_s(g, dev, iters)
        return rep_s / reps * 1e6   # us

    out = {"what": "torch.matmul, bf16 weights and activations, fp32 accumulate (cuBLAS)",
           "decode_us": {}, "prefill": {}}
    sets = [("single_2048x2048", [workloads.MatShape("proj", 2048, 2048)], (1,)),
            ("tinyllama_decode_step", workloads.tinyllama_decode_set(), (1, 16)),
            ("llama7b_set", workloads.llama7b_set(), (1, 16))]
    for name, shapes, Ns in sets:
        wbytes = sum(2 * s.M * s.K for s in shapes)
        copies = min(64, max(1, -(-4 * L2_BYTES // wbytes)))
        Ws = mats(shapes, copies)
        for N in Ns:
            Xs = [torch.randn((N, s.K), generator=gen, device=dev, dtype=torch.bfloat16)
                  for s in shapes]
            Ys = [torch.empty((N, s.M), device=dev, dtype=torch.bfloat16) for s in shapes]

            def step(r, Ws=Ws, Xs=Xs, Ys=Ys):
                for W, X, Y in zip(Ws[r % len(Ws)], Xs, Ys):
                    torch.matmul(X, W.t(), out=Y)
            out["decode_us"][f"{name}_N{N}"] = round(timed(step), 2)
        del Ws
    peak_tf = measured_bf16_peak()
    for set_name, wl, N in PREFILL_SETS:
        shapes = workloads.tinyllama_prefill_set() if wl == 4 else workloads.llama7b_set()
        rows = []
        for s in shapes:
            W = torch.randn((s.M, s.K), generator=gen, device=dev, dtype=torch.bfloat16)
            X = torch.randn((N, s.K), generator=gen, device=dev, dtype=torch.bfloat16)
            Y = torch.empty((N, s.M), device=dev, dtype=torch.bfloat16)
            us = timed(lambda r: torch.matmul(X, W.t(), out=Y))
            tf = 2.0 * s.M * N * s.K / us / 1e6
            rows.append({"matrix": s.name, "us": round(us, 2), "tflops": round(tf, 1),
                         "frac": round(tf / peak_tf, 4)})
            del W, X, Y
        out["prefill"][set_name] = rows
    return out


# --------------------------------------------------------------------------------------
# The oracle per workload, on the host cores: one thread, and all cores (each thread runs
# the unchanged oracle on its own slice of rows; ctypes releases the GIL during the call)
# --------------------------------------------------------------------------------------
ORACLE_ENTRIES = [(1, "q4_0", 1), (2, "q4_0", 1), (3, "q8_0", 1), (3, "q8_0", 2),
                  (3, "q8_0", 4), (3, "q8_0", 8), (3, "q8_0", 16), (4, "q4_0", 512),
                  (5, "q4_0", 1), (5, "q4_0", 16), (5, "q4_0", 2048), (2, "q4_k", 1)]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rows_time(btype, sample, threads: int) -> float:
    """Seconds for the oracle on every (blocks, rows, K, X) of `sample`, the rows of each
    matrix cut into `threads` contiguous slices run on `threads` threads."""
    import concurrent.futures
    import numpy as np
    import oracle
    work = [[] for _ in range(threads)]
    for blocks, r, K, X in sample:
        for i in range(threads):
            a, b = r * i // threads, r * (i + 1) // threads
            if b > a:
                work[i].append((np.ascontiguousarray(blocks[a:b]), b - a, K, X))

    def run(items):
        for blk, r, K, X in items:
            oracle.mul_mat(btype, blk, r, K, X)

    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(run, work))
        return time.perf_counter() - t0


def oracle_per_config(dev, target_s: float = 0.4) -> dict:
    """The oracle (as it stands) timed per workload on a row sample of every matrix, at one
    thread and at all host cores; rates scale to the full workload by its multiply-adds.
    Inputs: the same seeds and shapes as the GPU arm, drawn on the device and copied."""
    import oracle
    from block_quantized_matmul_gq_gb300 import binding, workloads
    cores = host_cores()
    out = {"cores": cores, "entries": []}
    for wl, btype, N in ORACLE_ENTRIES:
        shapes = workloads.WORKLOADS[wl][3]
        full_mac = sum(s.M * s.K * N for s in shapes)
        sum_k = sum(s.K for s in shapes)
        # rows per matrix for about target_s at one thread (about 1e9 multiply-adds per s)
        r1 = max(1, int(target_s * 1e9 / (N * sum_k)))
        ra = r1 * cores
        sample = []
        for j, s in enumerate(shapes):
            r = min(ra, s.M)
            W = workloads.weights(s.M, s.K, workloads.weight_seed(wl, j), device=dev)[:r]
            sample.append((oracle.quantize(btype, W.cpu().numpy()), r, s.K,
                           workloads.activations(N, s.K, workloads.act_seed(wl, N, j),
                                                 device=dev).cpu().numpy()))
            del W
        one = [(b[:min(r1, r)], min(r1, r), K, X) for b, r, K, X in sample]
        t1 = oracle_rows_time(btype, one, 1)
        ta = oracle_rows_time(btype, sample, cores)
        mac1 = sum(r * K * N for _, r, K, _ in one)
        maca = sum(r * K * N for _, r, K, _ in sample)
        s1 = t1 * full_mac / mac1
        sa = ta * full_mac / maca
        e = {"workload": wl, "type": btype, "N": N,
             "rows_per_matrix": {"one_core": r1, "all_cores": ra},
             "full_workload_s": {"one_core": round(s1, 3), "all_cores": round(sa, 3)}}
        if N >= 65:
            e["tflops"] = {"one_core": round(2 * full_mac / s1 / 1e12, 6),
                           "all_cores": round(2 * full_mac / sa / 1e12, 6)}
        else:
            b = step_bytes(shapes, N, binding.block_bytes(btype),
                           256 if btype == "q4_k" else 32)["total"]
            e["GBps"] = {"one_core": round(b / s1 / 1e9, 4), "all_cores": round(b / sa / 1e9, 4)}
        out["entries"].append(e)
        del sample, one
    return out


def q8x_measure(dev, reps: int = 20, iters: int = 20, Ns=(1, 2, 4, 8, 16)) -> dict:
    """The TinyLLaMA Q4_0 decode step through gq_mul_mat_q8x (X quantized per 32-block
    like Q8_0, integer block sums): batched calls replayed from a CUDA graph. GB/s counts
    weights + X + Y once per step, as for the exact path."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    peak, _ = measured_peaks()
    shapes = workloads.tinyllama_decode_set()
    ws = QuantizedWeightSet.synthetic(WORKLOAD_ID, shapes, "q4_0", dev)
    rows = []
    for N in Ns:
        nb = step_bytes(shapes, N, binding.block_bytes("q4_0"))
        xs, ys = ws.make_io(N, WORKLOAD_ID, dev)
        arrays = ws.problem_arrays(xs, ys)
        ws.run_q8x(arrays, N)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                ws.run_q8x(arrays, N)
        g.replay()
        torch.cuda.synchronize(dev)
        rep_s = replay_median_s(g, dev, iters)
        sec = rep_s / reps
        gbs = nb["total"] / sec / 1e9
        rows.append({"N": N, "us": round(sec * 1e6, 2), "GBps": round(gbs, 1),
                     "frac": round(gbs / peak, 4)})
        del g, xs, ys, arrays
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set during the q8x steps")
    return {"workload": "TinyLLaMA-1.1B decode step, Q4_0 weights, X quantized like Q8_0",
            "unit": "GB/s", "per_N": rows}


def fused_measure(dev, reps: int = 20, iters: int = 20, Ns=(1, 2)) -> dict:
    """The fused adjacent steps at decode, each timed from a CUDA graph against the plain
    products it replaces: TinyLLaMA's FFN gate/up pair (2 x 5632 x 2048) through
    gq_mul_mat_swiglu vs two gq_mul_mat calls, and the final RMSNorm into the LM head
    (32000 x 2048) through gq_mul_mat_rmsnorm vs gq_mul_mat alone. Weight copies are
    rotated so every call reads its weights from HBM; GB/s counts weights + X + output once."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    peak, _ = measured_peaks()
    K, Mf, Ml = 2048, 5632, 32000
    rb = binding.row_bytes("q4_0", K)

    def copies(nbytes):
        return min(48, max(1, -(-4 * L2_BYTES // nbytes)))

    def timed(calls):
        for c in calls[:2]:
            c()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in range(reps):
                calls[r % len(calls)]()
        g.replay()
        torch.cuda.synchronize(dev)
        rep_s = replay_median_s(g, dev, iters)
        return rep_s / reps

    out = {"unit": "GB/s", "peak": peak}
    nf = copies(2 * Mf * rb)
    gates = [binding.quantize(workloads.weights(Mf, K, 7000 + c, device=dev), "q4_0") for c in range(nf)]
    ups = [binding.quantize(workloads.weights(Mf, K, 7100 + c, device=dev), "q4_0") for c in range(nf)]
    nl = copies(Ml * rb)
    heads = [binding.quantize(workloads.weights(Ml, K, 7200 + c, device=dev), "q4_0") for c in range(nl)]
    gamma = (1.0 + 0.1 * torch.randn(K, generator=torch.Generator().manual_seed(7300))).to(dev)
    rows_s, rows_r = [], []
    for N in Ns:
        X = workloads.activations(N, K, 7400 + N, device=dev)
        H, G, U = (torch.empty((N, Mf), device=dev) for _ in range(3))
        b = 2 * Mf * rb + N * K * 4 + N * Mf * 4
        fused = timed([lambda c=c: binding.mul_mat_swiglu(gates[c], ups[c], "q4_0", Mf, K, X, out=H)
                       for c in range(nf)])
        plain = timed([lambda c=c: (binding.mul_mat(gates[c], "q4_0", Mf, K, X, out=G),
                                    binding.mul_mat(ups[c], "q4_0", Mf, K, X, out=U))
                       for c in range(nf)])
        rows_s.append({"N": N, "fused_us": round(fused * 1e6, 2), "GBps": round(b / fused / 1e9, 1),
                       "frac": round(b / fused / 1e9 / peak, 4),
                       "two_mul_mat_us (no activation)": round(plain * 1e6, 2)})
        Y = torch.empty((N, Ml), device=dev)
        b = Ml * rb + N * K * 4 + N * Ml * 4
        fused = timed([lambda c=c: binding.mul_mat_rmsnorm(heads[c], "q4_0", Ml, K, X, gamma, 1e-5, out=Y)
                       for c in range(nl)])
        plain = timed([lambda c=c: binding.mul_mat(heads[c], "q4_0", Ml, K, X, out=Y) for c in range(nl)])
        rows_r.append({"N": N, "fused_us": round(fused * 1e6, 2), "GBps": round(b / fused / 1e9, 1),
                       "frac": round(b / fused / 1e9 / peak, 4),
                       "mul_mat_alone_us (no norm)": round(plain * 1e6, 2)})
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set during the fused steps")
    out["swiglu_tinyllama_ffn_gate_up"] = rows_s
    out["rmsnorm_tinyllama_lm_head"] = rows_r
    return out


def profile_decode(spec: str, steps: int) -> dict:
    """For ncu: the TinyLLaMA decode step with N tokens (spec "q8_0/16"), one batched call
    per step with a caller-owned workspace, 3 warm-up steps then `steps` timed ones."""
    import torch
    from block_quantized_matmul_gq_gb300 import binding, workloads
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    btype, n = spec.split("/")
    N = int(n)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = workloads.tinyllama_decode_set()
    ws = QuantizedWeightSet.synthetic(WORKLOAD_ID, shapes, btype, dev)
    xs, ys = ws.make_io(N, WORKLOAD_ID, dev)
    arrays = ws.problem_arrays(xs, ys)
    work = ws.workspace(arrays, N, dev)
    for _ in range(3):
        ws.run(arrays, N, workspace=work)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        ws.run(arrays, N, workspace=work)
    end.record()
    torch.cuda.synchronize(dev)
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set")
    ms = start.elapsed_time(end) / steps
    return {"profile_decode": spec, "ms_per_step": round(ms, 5),
            "weight_GBps": round(ws.weight_bytes / ms / 1e6, 1)}


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


# --------------------------------------------------------------------------------------
# GB300 arm
# --------------------------------------------------------------------------------------
def run_gb300(args, shapes):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from block_quantized_matmul_gq_gb300 import binding
    from block_quantized_matmul_gq_gb300.weightset import QuantizedWeightSet
    from block_quantized_matmul_gq_gb300 import workloads

    N = 1
    ws = QuantizedWeightSet.synthetic(WORKLOAD_ID, shapes, "q4_0", dev)
    nb = step_bytes(shapes, N, binding.block_bytes("q4_0"))
    assert nb["weights"] == ws.weight_bytes

    # Activations and outputs live in two flat buffers (one copy each way per step).
    xs_total = sum(N * s.K for s in shapes)
    ys_total = sum(N * s.M for s in shapes)
    X_flat = torch.empty(xs_total, dtype=torch.float32, device=dev)
    Y_flat = torch.empty(ys_total, dtype=torch.float32, device=dev)
    xs, ys, xo, yo = [], [], 0, 0
    for j, s in enumerate(shapes):
        x = X_flat[xo:xo + N * s.K].view(N, s.K)
        x.copy_(workloads.activations(N, s.K, workloads.act_seed(WORKLOAD_ID, N, j), device=dev))
        xs.append(x)
        ys.append(Y_flat[yo:yo + N * s.M].view(N, s.M))
        xo += N * s.K
        yo += N * s.M
    arrays = ws.problem_arrays(xs, ys)
    launches_per_step = len(arrays)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        ws.run(arrays, N)
    torch.cuda.synchronize(dev)
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set during warm-up")

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ws.run(arrays, N)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    if args.profile:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        ms = start.elapsed_time(end) / args.steps
        if rank == 0:
            emit({"impl": "gb300", "profile_run": True, "ms_per_step": round(ms, 5),
                  "value": round(nb["total"] / ms / 1e6, 2), "unit": UNIT})
        return

    # Timed steps replay a graph of G consecutive steps (as a decode engine replays one
    # graph per step holding this launch among others): no host round trip between steps.
    G = STEPS_PER_GRAPH if args.steps % STEPS_PER_GRAPH == 0 else 1
    graph_g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_g):
        for _ in range(G):
            ws.run(arrays, N)
    graph_g.replay()
    torch.cuda.synchronize(dev)

    # Load phase (about 1 s) so the clock samples see the GPU busy, then the timed steps.
    t_probe = time.perf_counter()
    for _ in range(5):
        graph_g.replay()
    torch.cuda.synchronize(dev)
    per = (time.perf_counter() - t_probe) / (5 * G)
    load_steps = int(min(20000, max(10, 1.0 / max(per, 1e-6))))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        for _ in range(max(1, load_steps // G)):
            graph_g.replay()
        barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(args.steps // G):
            graph_g.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    elapsed = start.elapsed_time(end) / 1e3
    if binding.get_last_error() != 0:
        raise RuntimeError("device status word set during the timed region")
    t_max, bytes_all = aggregate(elapsed, nb["total"] * args.steps, world, dev)
    value = bytes_all / t_max / 1e9
    per_gpu = nb["total"] * args.steps / elapsed / 1e9

    # End to end through the public API with HOST buffers, every step: the step's X in
    # pinned host memory, the batched call given the host X and a pinned host Y (the
    # kernels read X and write Y across NVLink-C2C, include/gq.h), and a host synchronize
    # before the host reads Y and the next step starts. The call is recorded once into a
    # CUDA graph (as a serving loop would), so a step costs one graph launch plus the
    # synchronize. Beside it, the same with explicit copies: pinned X -> device buffer,
    # the call on device buffers, device Y -> pinned host, in one graph.
    X_host = X_flat.cpu().pin_memory()
    Y_host = torch.full((ys_total,), float("nan"), dtype=torch.float32).pin_memory()
    xs_h, ys_h, xo, yo = [], [], 0, 0
    for s in shapes:
        xs_h.append(X_host[xo:xo + N * s.K].view(N, s.K))
        ys_h.append(Y_host[yo:yo + N * s.M].view(N, s.M))
        xo += N * s.K
        yo += N * s.M
    arrays_h = ws.problem_arrays(xs_h, ys_h)
    e2e_steps = max(10, min(args.steps, 2000))

    def e2e_time(record):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            record()
        for _ in range(5):
            g.replay()
            torch.cuda.synchronize(dev)
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            g.replay()
            torch.cuda.synchronize(dev)
        t, b = aggregate(time.perf_counter() - t0, nb["total"] * e2e_steps, world, dev)
        return t, b / t / 1e9

    def explicit_copies():
        X_flat.copy_(X_host, non_blocking=True)
        ws.run(arrays, N)
        Y_host.copy_(Y_flat, non_blocking=True)

    e2e_t, e2e_value = e2e_time(lambda: ws.run(arrays_h, N))
    if not torch.equal(Y_host.view(torch.int32), Y_flat.cpu().view(torch.int32)):
        raise RuntimeError("host-buffer step differs from the device-buffer step")
    e2e_copy_t, e2e_copy_value = e2e_time(explicit_copies)

    # Where an end-to-end step's time goes: each part alone, recorded and replayed the same
    # way with a host synchronize per step.
    def per_step_us(record):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            record()
        for _ in range(5):
            g.replay()
            torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(200):
            g.replay()
            torch.cuda.synchronize(dev)
        return round((time.perf_counter() - t0) / 200 * 1e6, 2)

    e2e_parts = {
        "e2e_step_us": round(e2e_t / e2e_steps * 1e6, 2),
        "kernel_and_sync_us": per_step_us(lambda: ws.run(arrays, N)),
        "explicit_copies": {
            "value": round(e2e_copy_value, 2), "unit": UNIT,
            "step_us": round(e2e_copy_t / e2e_steps * 1e6, 2),
            "h2d_copy_and_sync_us": per_step_us(lambda: X_flat.copy_(X_host, non_blocking=True)),
            "d2h_copy_and_sync_us": per_step_us(lambda: Y_host.copy_(Y_flat, non_blocking=True)),
        },
    }

    peak, peak_src = measured_peaks()
    traffic = profiled_traffic()
    clk = clocks.summary()
    line = {
        "impl": "gb300", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "q4_0 codes x int16 fixed-point activations (dp2a, i32) -> f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "N": N, "matmuls": len(shapes),
                   "weight_bytes": nb["weights"], "algorithmic_bytes_per_step": nb["total"],
                   "l2": "inputs larger than L2: 582 MB of weights streamed per step vs 129 MB L2",
                   "launch": f"{launches_per_step} gq_mul_mat_batched launch per step, "
                             f"CUDA graph of {G} steps replayed",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(per_gpu / peak, 4),
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic,
                     "kernel": "gemv_stream_kernel<Q4_0, 1 token>",
                     "per_launch": "one launch per step: achieved = algorithmic bytes per "
                                   "launch / (CUDA-event step time)"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": nb["x"], "d2h_bytes_per_step": nb["y"],
                "how": "X and Y in pinned host memory passed to gq_mul_mat_batched (read "
                       "and written by the kernels over NVLink-C2C), one graph launch and "
                       "a host synchronize per step",
                "parts": e2e_parts},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        # keys in the order they should be read: the compact per-workload summary first,
        # the details after it
        line["summary"] = None
        line["cpu_baseline"] = None
        step_calls = step_as_calls_measure(dev, ws, xs, ys, N, nb["total"])
        dec = decode_measure(dev)
        per_mm = per_matmul_measure(dev)
        q8x = q8x_measure(dev)
        fused = fused_measure(dev)
        pf = prefill_measure(dev)
        dense = dense_context_measure(dev)
        dec["tinyllama_step_as_155_calls_q4_0"] = step_calls
        line["summary"] = summarize(dec, pf, dense, peak)
        line["decode"] = {"unit": "GB/s", "peak": peak,
                          "peak_source": line["roofline"]["peak_source"], **dec}
        line["decode_per_matmul"] = per_mm
        line["decode_q8x"] = q8x
        line["fused"] = fused
        line["prefill"] = {"unit": "TFLOP/s", "dtype": "bf16 operands, fp32 accumulate",
                           "peak": measured_bf16_peak(),
                           "peak_source": "measured bf16_tflops (MEASURED_PEAKS.json), burst",
                           **pf}
        line["dense_bf16_context"] = dense
        if args.no_cpu_baseline:
            del line["cpu_baseline"]
        else:
            line["cpu_baseline"] = cpu_baseline(shapes)
            line["oracle_per_workload"] = oracle_per_config(dev)
        emit(line)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def summarize(dec: dict, pf: dict, dense: dict, peak: float) -> dict:
    """One short entry per workload (time, rate, fraction of the measured peak), placed
    ahead of the detailed sections of the line."""
    def per_n(key):
        return {f"N{r['N']}": [r["us"], r["GBps"], r["frac"]] for r in dec[key]["per_N"]}


    single = dec["single_q4_0_2048x2048"]
    r1 = single["per_N"][0]
    out = {
        "format": "decode: [us, GB/s, frac of measured HBM]; prefill: [TFLOP/s, frac of "
                  "measured bf16]",
        "w1_single_q4_0_2048x2048_N1": [r1["us"], r1["GBps"], r1["frac"]],
        "w1_launch_floor_us": single["launch_floor"]["us"],
        "w2_tinyllama_q4_0": per_n("tinyllama_decode_q4_0"),
        "w3_tinyllama_q8_0": per_n("tinyllama_decode_q8_0"),
        "w5_llama7b_q4_0": per_n("llama7b_decode_q4_0"),
        "w2_tinyllama_q4_k": per_n("tinyllama_decode_q4_k"),
    }
    calls = dec.get("tinyllama_step_as_155_calls_q4_0")
    if calls:
        out["w2_tinyllama_q4_0_N1_as_155_calls"] = [calls["us"], calls["GBps"], calls["frac"]]
    for key, v in pf.items():
        out["prefill_" + key] = [v["tflops"], v["frac"]]
    ctx = dense.get("decode_us", {})
    if ctx:
        out["dense_bf16_decode_us"] = ctx
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing")
    ap.add_argument("--profile", action="store_true",
                    help="for ncu: warm-up and the timed steps only (no load phase, no e2e, "
                         "no clock sampling, no oracle); prints the device-timed line")
    ap.add_argument("--profile-prefill", metavar="MATRIX", default=None,
                    help="for ncu: time one prefill GEMM only, e.g. llama7b_prefill_n2048/lm_head "
                         "(llama7b_prefill_n2048_q8_0/lm_head for Q8_0, _q4_k for Q4_K)")
    ap.add_argument("--profile-decode", metavar="TYPE/N", default=None,
                    help="for ncu: the TinyLLaMA decode step at N tokens, e.g. q8_0/16")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.profile_decode:
        emit(profile_decode(args.profile_decode, steps=min(args.steps, 20)))
        return
    if args.profile_prefill:
        import torch
        set_name, matrix = args.profile_prefill.split("/")
        btype = "q4_0"
        for suffix in ("_q8_0", "_q4_k"):
            if set_name.endswith(suffix):
                btype, set_name = suffix[1:], set_name[: -len(suffix)]
        emit(prefill_measure(torch.device("cuda", 0), reps=2, iters=1, only=(set_name, matrix),
                             types=(btype,), rotate=False))
        return
    from block_quantized_matmul_gq_gb300 import workloads
    shapes = workloads.tinyllama_decode_set()
    if args.impl == "reference":
        run_reference(args, shapes)
    else:
        run_gb300(args, shapes)


if __name__ == "__main__":
    main()
