"""Seeded synthetic inputs for one expert-parallel (EP) layer.

This module is shared by the tests, the bench and the smoke check, and it is
the only code that both the CUDA path and the CPU oracle receive data from.
It draws random numbers and nothing else: it holds none of the layout,
dispatch, descriptor or combine arithmetic.

Workloads (DeepSeek-V3-shaped routing, as the EP articles discuss it: the
UCCL-EP article, section 6 "EP32 dispatch / combine", and the GPU
communication notes, table "EP cross-node MoE: dispatch/combine token"):

  name   R   tokens/rank  hidden  experts  top-k  routing
  tiny   4   16           256     16       2      uniform without replacement
  ll     32  128          7168    256      8      uniform without replacement
  ht     32  4096         7168    256      8      uniform without replacement
  skew   16  8192         2048    64       6      Zipf(s=1.2) popularity, seeded permutation
  small  32  2048         1024    128      4      uniform without replacement

x ~ N(0, 1) rounded to bf16; topk_weights = fp32 softmax of N(0, 1) logits over
the K picks (computed in float64, then rounded once to fp32).  Picks within a
token are distinct and kept in the order they were drawn.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get", "make_routing", "make_x", "make_x_torch",
           "make_expert_out", "make_expert_out_torch", "bf16_bits_from_f32"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_ranks: int
    tokens_per_rank: int
    hidden: int
    num_experts: int
    topk: int
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.2
    seed: int = 0
    # ring settings named by the workload itself (None: the library default)
    channels: int | None = None
    ring_depth: int | None = None
    max_inflight: int | None = None
    rows_per_msg: int | None = None

    @property
    def num_tokens(self) -> int:
        return self.num_ranks * self.tokens_per_rank

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 4, 16, 256, 16, 2, seed=101, channels=8, ring_depth=1024),
    # the low-latency layer's configuration fixes no ring settings: 16 rings
    # (two destination ranks each) make its posting tail shortest
    "ll": Workload("ll", 32, 128, 7168, 256, 8, seed=202, channels=16),
    "ht": Workload("ht", 32, 4096, 7168, 256, 8, seed=303, channels=8),
    "skew": Workload("skew", 16, 8192, 2048, 64, 6, routing="zipf", zipf_s=1.2, seed=404),
    "small": Workload("small", 32, 2048, 1024, 128, 4, seed=505, channels=8, ring_depth=1024,
                      max_inflight=256, rows_per_msg=8),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _topk_of_keys(keys: np.ndarray, k: int) -> np.ndarray:
    """Column indices of the k largest keys per row, largest first."""
    part = np.argpartition(-keys, k - 1, axis=1)[:, :k]
    vals = np.take_along_axis(keys, part, axis=1)
    order = np.argsort(-vals, axis=1, kind="stable")
    return np.take_along_axis(part, order, axis=1)


def make_routing(w: Workload, seed: int | None = None, chunk: int = 16384):
    """topk_idx int32 [T, K] and topk_weights float32 [T, K].

    uniform: K experts drawn uniformly without replacement (the K largest of
    E i.i.d. uniform keys, in decreasing key order).
    zipf: p_i proportional to i^-s over a seeded random permutation of the
    experts; K draws without replacement by successive sampling, done as
    Gumbel-top-K (log p_e + Gumbel noise), which has the same law.
    """
    rng = np.random.default_rng(w.seed if seed is None else seed)
    T, E, K = w.num_tokens, w.num_experts, w.topk
    if w.routing == "zipf":
        perm = rng.permutation(E)
        p = np.arange(1, E + 1, dtype=np.float64) ** (-w.zipf_s)
        logp = np.empty(E)
        logp[perm] = np.log(p / p.sum())
    idx = np.empty((T, K), dtype=np.int32)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        u = rng.random((t1 - t0, E))
        if w.routing == "uniform":
            keys = u
        elif w.routing == "zipf":
            keys = logp[None, :] - np.log(-np.log(np.maximum(u, 1e-300)))
        else:
            raise ValueError(w.routing)
        idx[t0:t1] = _topk_of_keys(keys, K)
    logits = rng.standard_normal((T, K))
    logits -= logits.max(axis=1, keepdims=True)
    ew = np.exp(logits)
    weights = (ew / ew.sum(axis=1, keepdims=True)).astype(np.float32)
    return idx, weights


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) via torch; uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_x(w: Workload, seed: int | None = None, rows: int | None = None) -> np.ndarray:
    """x as bf16 bits (uint16) [T, H], x ~ N(0, 1), generated on the host."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 7919)
    T = w.num_tokens if rows is None else rows
    return bf16_bits_from_f32(rng.standard_normal((T, w.hidden), dtype=np.float32))


def make_expert_out(rows: int, hidden: int, seed: int, chunk_rows: int = 16384) -> np.ndarray:
    """A random expert output as bf16 bits (uint16) [rows, hidden] ~ N(0, 1),
    generated on the host chunk by chunk (for the CPU-only timings)."""
    rng = np.random.default_rng(seed + 15485863)
    out = np.empty((rows, hidden), dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = bf16_bits_from_f32(rng.standard_normal((r1 - r0, hidden), dtype=np.float32))
    return out


def _randn_bf16_torch(rows: int, hidden: int, device, seed: int, chunk_rows: int = 65536):
    """N(0, 1) draws rounded to bf16, generated chunk by chunk on `device`
    from one seeded generator (deterministic for a given device type)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, hidden), generator=g, device=device, dtype=torch.float32)
    return out


def make_x_torch(w: Workload, device, seed: int | None = None):
    """x ~ N(0, 1) as a bf16 tensor generated directly on `device` (for the
    full-size workloads, where a host-side draw would take long)."""
    return _randn_bf16_torch(w.num_tokens, w.hidden, device, (w.seed if seed is None else seed) + 7919)


def make_expert_out_torch(rows: int, hidden: int, device, seed: int):
    """A random bf16 expert output [rows, hidden] ~ N(0, 1) on `device`."""
    return _randn_bf16_torch(rows, hidden, device, seed + 104729)
