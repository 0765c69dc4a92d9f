"""Seeded synthetic workloads for the routing plan, dispatch and combine.

This module draws inputs only: router top-k expert ids, router weights and
hidden states.  It contains none of the plan/dispatch/combine arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.

Recipe (the same for every workload):
  * ``numpy.random.default_rng(seed)`` (PCG64);
  * K distinct experts per token by Gumbel-top-K: key[t,e] = log w_e + Gumbel,
    the K largest keys in descending order.  Uniform routing has w_e = 1;
    Zipf routing has w_e proportional to (e+1)^-s;
  * router logits ~ N(0,1) float32 [T,K], softmax over K in float32;
  * hidden states x ~ N(0,1) drawn as float32, rounded to bfloat16 by torch.

The workload shapes follow the pages' scale (hidden 7168, top-6, up to 128
ranks / 256 experts, 16384 tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    P: int          # logical ranks
    E: int          # experts (E/P per rank)
    S: int          # tokens per rank
    H: int          # hidden size
    K: int          # top-k
    A: int          # expert_alignment
    routing: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.2
    seed: int = 0
    fp8: bool = False
    cached_steps: int = 0      # cached-handle dispatches after the fresh one
    expert: str = "identity"   # synthetic expert between dispatch and combine

    @property
    def T(self) -> int:
        return self.P * self.S

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", P=4, E=8, S=64, H=256, K=2, A=1),
    "bf16": Workload("bf16", P=8, E=64, S=2048, H=7168, K=6, A=128),
    "fp8": Workload("fp8", P=16, E=256, S=1024, H=7168, K=6, A=128, fp8=True,
                    expert="dequant"),
    "zipf": Workload("zipf", P=128, E=256, S=128, H=7168, K=6, A=128, routing="zipf",
                     cached_steps=10),
    "rt": Workload("rt", P=32, E=128, S=2048, H=4096, K=8, A=64, expert="scale"),
}


def expert_log_weights(w: Workload) -> np.ndarray:
    if w.routing == "uniform":
        return np.zeros(w.E, np.float64)
    if w.routing == "zipf":
        return -w.zipf_s * np.log(np.arange(1, w.E + 1, dtype=np.float64))
    raise ValueError(w.routing)


def draw_topk(w: Workload, seed: int | None = None):
    """-> (topk_idx [T,K] int64, topk_weights [T,K] float32)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    T, E, K = w.T, w.E, w.K
    logw = expert_log_weights(w)
    idx = np.empty((T, K), np.int64)
    rows = 8192
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        keys = logw[None, :] + rng.gumbel(size=(r1 - r0, E))
        part = np.argpartition(-keys, K - 1, axis=1)[:, :K]
        order = np.argsort(-np.take_along_axis(keys, part, axis=1), axis=1, kind="stable")
        idx[r0:r1] = np.take_along_axis(part, order, axis=1)
    logits = rng.standard_normal((T, K), dtype=np.float32)
    ex = np.exp(logits - logits.max(axis=1, keepdims=True), dtype=np.float32)
    weights = (ex / ex.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return idx, weights


def draw_hidden(T: int, H: int, seed: int) -> np.ndarray:
    """x ~ N(0,1), rounded to bf16 -> [T,H] uint16 bit patterns."""
    rng = np.random.default_rng(seed)
    out = np.empty((T, H), np.uint16)
    rows = max(1, (1 << 24) // max(1, H))
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        f = rng.standard_normal((r1 - r0, H), dtype=np.float32)
        out[r0:r1] = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


def hidden_seed(w: Workload, step: int = 0) -> int:
    """Seed of the hidden states of dispatch number ``step`` (0 = fresh)."""
    return 1_000_003 * (w.seed + 1) + step


def draw_y(n_rows: int, H: int, seed: int) -> np.ndarray:
    """Random expert outputs [n_rows,H] bf16 bits (combine-only parity cases)."""
    return draw_hidden(n_rows, H, seed)


def bits_to_bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bf16_tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
