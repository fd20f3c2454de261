"""Quantized weights kept resident in HBM, and the batched call over all of them.

The pages' advice is to keep every weight tensor in device memory for the whole run
("No Python! Building an AI Inference Engine Exclusively in C++", section 7.2, after the
cuBLAS listing). A QuantizedWeightSet quantizes each matrix once on the GPU (through
libgq) and then runs every matrix-vector product of a step with one gq_mul_mat_batched
launch (at most GQ_MAX_BATCH = 256 problems per launch).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import binding, workloads


@dataclass
class QuantizedMatrix:
    shape: workloads.MatShape
    blocks: torch.Tensor          # uint8 (M, row_bytes), on the device
    seed: int


@dataclass
class QuantizedWeightSet:
    btype: str
    mats: list[QuantizedMatrix] = field(default_factory=list)

    @property
    def weight_bytes(self) -> int:
        return sum(m.blocks.numel() for m in self.mats)

    @property
    def n_weights(self) -> int:
        return sum(m.shape.M * m.shape.K for m in self.mats)

    @classmethod
    def synthetic(cls, workload: int, shapes, btype: str, device,
                  keep_rows: dict | None = None) -> "QuantizedWeightSet":
        """Draws each matrix N(0, 0.02) with its seed on `device`, quantizes it there and
        drops the fp32 copy. keep_rows maps matrix index -> row indices whose fp32 values
        are copied to the host (for checking sampled outputs against the oracle); the
        copies land in ws.kept[j]."""
        ws = cls(btype)
        ws.kept = {}
        for j, s in enumerate(shapes):
            seed = workloads.weight_seed(workload, j)
            W = workloads.weights(s.M, s.K, seed, device=device)
            blocks = binding.quantize(W, btype)
            if keep_rows and j in keep_rows:
                idx = torch.as_tensor(keep_rows[j], device=device)
                ws.kept[j] = W.index_select(0, idx).cpu()
            del W
            ws.mats.append(QuantizedMatrix(s, blocks, seed))
        return ws

    def make_io(self, N: int, workload: int, device, host_pinned: bool = False):
        """Seeded activations X_j (N, K_j) and output buffers Y_j (N, M_j) per matrix."""
        xs, ys = [], []
        for j, m in enumerate(self.mats):
            X = workloads.activations(N, m.shape.K, workloads.act_seed(workload, N, j),
                                      device=device)
            xs.append(X)
            ys.append(torch.empty((N, m.shape.M), dtype=torch.float32, device=device))
        return xs, ys

    def problem_arrays(self, xs, ys):
        """gq_mul_mat_problem arrays, GQ_MAX_BATCH problems per array."""
        items = [(m.blocks, m.shape.M, m.shape.K, x, y) for m, x, y in zip(self.mats, xs, ys)]
        return [binding.make_problems(items[i:i + binding.MAX_BATCH])
                for i in range(0, len(items), binding.MAX_BATCH)]

    def workspace(self, arrays, N: int, device):
        """A caller-owned workspace big enough for every array (None if none is needed);
        with it, run() allocates nothing and can be recorded into a CUDA graph."""
        need = max([binding.batched_workspace_size(a, self.btype, N) for a in arrays] + [0])
        return torch.empty(need, dtype=torch.uint8, device=device) if need else None

    def run(self, arrays, N: int, stream=None, workspace=None) -> None:
        for arr in arrays:
            if workspace is None:
                binding.mul_mat_batched(arr, self.btype, N, stream=stream)
            else:
                binding.mul_mat_batched_ws(arr, self.btype, N, workspace, stream=stream)

    def run_q8x(self, arrays, N: int, stream=None) -> None:
        """The same products with X quantized per 32-block like Q8_0 (gq_mul_mat_q8x)."""
        for arr in arrays:
            binding.mul_mat_q8x_batched(arr, self.btype, N, stream=stream)
