"""Seeded synthetic inputs for MoE token dispatch and combine.

This module makes the inputs that both the CUDA path and the CPU oracle are
fed: token hidden rows, top-k routing, routing weights and the per-expert
scales used to fake expert outputs.  It holds none of the dispatch/combine
arithmetic (no counting, no ranking, no quantisation, no reduction); routing
and weights are inputs of the method, not part of it.

Every tensor draws from its own numpy stream, spawned from one SeedSequence
per workload (seed 0 by default), so each tensor is reproducible on its own
and on any machine.

Workloads (shapes of the DeepSeek-V3 MoE layer where named so):
  tiny      T=128,   H=1024, E=16,  k=4, uniform distinct experts, bf16, packed
  decode    T=128,   H=7168, E=256 (32 partitions x 8), k=8, uniform,
            fp8 e4m3 + per-128 scales into a [256, 128, 7168] capacity buffer
  prefill   T=4096,  H=7168, E=256, k=8, uniform, bf16, packed
  skewed    T=8192,  H=7168, E=256 (32 x 8), k=8, Zipf(s=1.2) popularity over
            a seeded permutation, sampled without replacement, fp8, packed
  grouped   T=16384, H=4096, E=128 in 8 groups of 16; top-4 groups by max
            logit, then top-8 experts inside them; bf16, packed
  unbalanced  as skewed with Zipf(s=0.4): max/mean load 1.50 per partition
            (5.59 per expert) with seed 0, the rank imbalance of the second
            Validation table of "Pipeline direct NVLink dispatch with
            triple-buffered prefetch" (DeepEP PR #693)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PACKED = 0
CAPACITY = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    P: int                      # logical partitions of E/P consecutive experts
    routing: str                # "uniform" | "zipf" | "group_limited"
    fp8: bool
    mode: int = PACKED
    capacity: int = 0
    zipf_s: float = 1.2
    groups: int = 1
    topk_groups: int = 1
    description: str = field(default="", compare=False)

    @property
    def R(self) -> int:
        """Rows of the receive buffer."""
        return self.T * self.k if self.mode == PACKED else self.E * self.capacity

    def shrink(self, T: int) -> "Workload":
        """Same workload with fewer tokens (for oracle-sized parity cases)."""
        d = self.__dict__.copy()
        d["T"] = T
        d["name"] = f"{self.name}@T{T}"
        return Workload(**d)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", T=128, H=1024, E=16, k=4, P=1, routing="uniform", fp8=False,
                     description="T=128 H=1024 E=16 top-4, bf16 packed"),
    "decode": Workload("decode", T=128, H=7168, E=256, k=8, P=32, routing="uniform", fp8=True,
                       mode=CAPACITY, capacity=128,
                       description="T=128 H=7168 E=256 (32x8) top-8, fp8 into [256,128,7168]"),
    "prefill": Workload("prefill", T=4096, H=7168, E=256, k=8, P=1, routing="uniform", fp8=False,
                        description="T=4096 H=7168 E=256 top-8, bf16 packed"),
    "skewed": Workload("skewed", T=8192, H=7168, E=256, k=8, P=32, routing="zipf", fp8=True,
                       zipf_s=1.2,
                       description="T=8192 H=7168 E=256 (32x8) top-8 Zipf(1.2), fp8 packed"),
    "grouped": Workload("grouped", T=16384, H=4096, E=128, k=8, P=8, routing="group_limited",
                        fp8=False, groups=8, topk_groups=4,
                        description="T=16384 H=4096 E=128 (8 groups x 16) top-4 groups/top-8, bf16"),
    "unbalanced": Workload("unbalanced", T=8192, H=7168, E=256, k=8, P=32, routing="zipf", fp8=True,
                           zipf_s=0.4,
                           description="T=8192 H=7168 E=256 (32x8) top-8 Zipf(0.4): partition load max/mean 1.5, "
                                       "fp8 packed"),
}

# Independent streams, one per tensor.
_STREAMS = ("x", "routing", "logits", "expert_scale", "expert_out")


def _streams(seed: int) -> dict[str, np.random.Generator]:
    ss = np.random.SeedSequence(seed)
    return {name: np.random.default_rng(s) for name, s in zip(_STREAMS, ss.spawn(len(_STREAMS)))}


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    z = logits - logits.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return (ez / ez.sum(axis=1, keepdims=True)).astype(np.float32)


def routing(wl: Workload, seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """topk_idx [T, k] int32 and topk_w [T, k] float32 for a workload."""
    rs = _streams(seed)
    T, E, k = wl.T, wl.E, wl.k
    if wl.routing == "uniform":
        # k distinct experts per token, uniformly at random.
        idx = np.argsort(rs["routing"].random((T, E)), axis=1, kind="stable")[:, :k]
        w = _softmax_rows(rs["logits"].standard_normal((T, k), dtype=np.float32))
    elif wl.routing == "zipf":
        # Popularity of the expert at rank r is proportional to r^-s; ranks are
        # given to experts by a seeded permutation.  k experts per token are
        # drawn without replacement by Gumbel-top-k (Efraimidis-Spirakis).
        rng = rs["routing"]
        ranks = np.arange(1, E + 1, dtype=np.float64)
        pop_by_rank = ranks ** (-wl.zipf_s)
        pop_by_rank /= pop_by_rank.sum()
        perm = rng.permutation(E)
        pop = np.empty(E, np.float64)
        pop[perm] = pop_by_rank
        keys = np.log(pop)[None, :] + rng.gumbel(size=(T, E))
        idx = np.argsort(-keys, axis=1, kind="stable")[:, :k]
        w = _softmax_rows(rs["logits"].standard_normal((T, k), dtype=np.float32))
    elif wl.routing == "group_limited":
        # Router logits ~ N(0,1); keep the top groups by their best logit, then
        # the top-k experts inside the kept groups; weights = softmax of those
        # k logits.  Ties resolve to the lower index (stable sort).
        logits = rs["logits"].standard_normal((T, E), dtype=np.float32)
        G = wl.groups
        per = E // G
        gmax = logits.reshape(T, G, per).max(axis=2)
        keep = np.argsort(-gmax, axis=1, kind="stable")[:, : wl.topk_groups]
        mask = np.zeros((T, G), bool)
        np.put_along_axis(mask, keep, True, axis=1)
        masked = np.where(np.repeat(mask, per, axis=1), logits, -np.inf)
        idx = np.argsort(-masked, axis=1, kind="stable")[:, :k]
        w = _softmax_rows(np.take_along_axis(logits, idx, axis=1))
    else:
        raise ValueError(wl.routing)
    return np.ascontiguousarray(idx, dtype=np.int32), np.ascontiguousarray(w, dtype=np.float32)


def hidden(wl: Workload, seed: int = 0) -> np.ndarray:
    """x [T, H] as bf16 bit patterns (uint16), bf16 of N(0, 1)."""
    rs = _streams(seed)
    return to_bf16_bits(rs["x"].standard_normal((wl.T, wl.H), dtype=np.float32))


def expert_scales(wl: Workload, seed: int = 0) -> np.ndarray:
    """Per-expert output scale s_e ~ U[0.5, 1.5) for random-scale fake experts."""
    return _streams(seed)["expert_scale"].uniform(0.5, 1.5, size=wl.E).astype(np.float32)


def expert_rows(n_rows: int, H: int, seed: int = 0) -> np.ndarray:
    """n_rows x H independent bf16 N(0,1) rows (stand-in expert outputs)."""
    return to_bf16_bits(_streams(seed)["expert_out"].standard_normal((n_rows, H), dtype=np.float32))


def make(name_or_wl, seed: int = 0) -> dict:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    idx, w = routing(wl, seed)
    return dict(wl=wl, x=hidden(wl, seed), topk_idx=idx, topk_w=w)


def load_stats(wl: Workload, topk_idx: np.ndarray) -> dict:
    """Max/mean load per expert and per partition (describes the input mix)."""
    counts = np.bincount(topk_idx[topk_idx >= 0].ravel(), minlength=wl.E)
    parts = counts.reshape(wl.P, wl.E // wl.P).sum(axis=1)
    return dict(expert_max_over_mean=float(counts.max() / counts.mean()),
                partition_max_over_mean=float(parts.max() / parts.mean()),
                top_expert_tokens=int(counts.max()))
