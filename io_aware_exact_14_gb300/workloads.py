"""Seeded synthetic workloads for exact attention (shared by tests, bench and the oracle's tests).

This module holds the five workload shapes and the recipe that draws their
inputs. It contains none of the attention arithmetic: it only produces
Q, K, V (and the upstream gradient dO) as bf16 tensors on the CPU, so the CUDA
path and the fp64 oracle can be fed bit-identical values.

Recipe (the pages give shapes but no generator; see the design notes):
  * ``torch.Generator('cpu').manual_seed(seed)`` with ``seed = 14 + index``;
  * draw Q, K, V, dO in that order as fp32 ``randn`` of shape [B, H, N, d];
  * multiply Q and K by ``qk_mult`` (3 for the peaky-softmax stress case,
    1 otherwise) and V, dO by 1;
  * round to bf16 (round-to-nearest-even) with ``.to(torch.bfloat16)``.

Shapes follow the workloads the pages discuss: head dims 64/128, sequence
lengths 2K-16K (FlashAttention pages: "GPU memory hierarchy" and "tiling"
sections), causal and non-causal masks.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int                 # 1-based workload number
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: Tuple[bool, ...]   # mask variants the workload runs
    passes: Tuple[str, ...]    # "fwd" and/or "bwd"
    qk_mult: float = 1.0       # multiplier on Q and K before the bf16 cast
    oracle_rows: Optional[int] = None    # rows per head the oracle checks (None: all)
    oracle_slices: Optional[int] = None  # (b, h) slices the oracle checks (None: all)

    @property
    def seed(self) -> int:
        return 14 + self.index

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def shape(self) -> Tuple[int, int, int, int]:
        return (self.B, self.H, self.N, self.d)


WORKLOADS: Dict[int, Workload] = {
    1: Workload(1, "single_head_fwd_B1_H1_N128_d64", 1, 1, 128, 64, (False,), ("fwd",)),
    2: Workload(2, "fwd_bwd_B4_H16_N2048_d128", 4, 16, 2048, 128, (False, True), ("fwd", "bwd")),
    3: Workload(3, "peaky_fwd_B2_H8_N4096_d64_qk_x3", 2, 8, 4096, 64, (False,), ("fwd",),
                qk_mult=3.0),
    4: Workload(4, "long_causal_fwd_B1_H32_N16384_d128", 1, 32, 16384, 128, (True,), ("fwd",),
                oracle_rows=256),
    5: Workload(5, "train_causal_fwd_bwd_B8_H16_N4096_d128", 8, 16, 4096, 128, (True,),
                ("fwd", "bwd"), oracle_slices=2),
}


def make_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0,
                with_grad: bool = True) -> Dict[str, torch.Tensor]:
    """Draw q, k, v (and do) as contiguous bf16 CPU tensors of shape [B, H, N, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    out = {}
    for name in ("q", "k", "v", "do"):
        if name == "do" and not with_grad:
            break
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x = x * qk_mult
        out[name] = x.to(torch.bfloat16).contiguous()
    return out


def make_splitkv_inputs(B: int, H: int, Nq: int, Nk: int, d: int, seed: int) -> Dict[str, torch.Tensor]:
    """Short query blocks against long key sequences: q [B, H, Nq, d], k and v
    [B, H, Nk, d], contiguous bf16 CPU tensors drawn as fp32 N(0, 1) in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    for name, n in (("q", Nq), ("k", Nk), ("v", Nk)):
        out[name] = torch.randn((B, H, n, d), generator=g, dtype=torch.float32).to(torch.bfloat16).contiguous()
    return out


def workload_inputs(w: Workload, with_grad: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    if with_grad is None:
        with_grad = "bwd" in w.passes
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_grad)


def sample_rows(w: Workload, count: int) -> np.ndarray:
    """Query rows the oracle checks per (b, h): shape [B, H, count], sorted.

    Drawn without replacement from ``numpy.random.default_rng(seed)`` per head in
    (b, h) order; rows 0 and N-1 are always included.
    """
    rng = np.random.default_rng(w.seed)
    count = min(count, w.N)
    rows = np.empty((w.B, w.H, count), dtype=np.int64)
    for b in range(w.B):
        for h in range(w.H):
            drawn = rng.choice(w.N, size=count, replace=False).tolist()
            pick = [x for x in drawn if x not in (0, w.N - 1)][: max(count - 2, 0)]
            r = sorted(set([0, w.N - 1] + pick))
            while len(r) < count:  # only reachable for tiny N
                r.append(r[-1])
            rows[b, h] = np.asarray(r[:count])
    return rows


def all_slices(w: Workload) -> list:
    """Every (b, h) slice of the workload, in order."""
    return [(b, h) for b in range(w.B) for h in range(w.H)]


def oracle_slices(w: Workload) -> list:
    """(b, h) slices the oracle checks: the sampled ones, or all of them."""
    return sample_slices(w, w.oracle_slices) if w.oracle_slices else all_slices(w)


def sample_slices(w: Workload, count: int) -> list:
    """(b, h) slices the oracle checks, drawn from ``default_rng(seed + 1000)``."""
    rng = np.random.default_rng(w.seed + 1000)
    flat = rng.choice(w.B * w.H, size=min(count, w.B * w.H), replace=False)
    return [(int(i) // w.H, int(i) % w.H) for i in sorted(flat.tolist())]


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
