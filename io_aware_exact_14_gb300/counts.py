"""Work and traffic counts for exact attention (no attention arithmetic).

FLOP convention (the pages give none): forward 4*B*H*N^2*d (two N x N x d
contractions, S = QK^T and O = PV), backward 2.5x forward (five contractions
counted once: S recomputed, dP, dV, dK, dQ), both halved for a causal mask.

Per-kernel executed work of the backward: the dK/dV kernel runs four
contractions per (query tile, key tile) pair (S^T, dP^T, dV, dK) and the dQ
kernel three (S, dP, dQ), so 14*B*H*N^2*d executed against 10 counted.  For
wide heads (d > 128) dK and dV are two launches that each recompute S^T
(S^T, dV; S^T, dP^T, dK), so the dK/dV step executes five contractions.
"""
from __future__ import annotations


def attn_flops(B: int, H: int, N: int, d: int, causal: bool, pass_: str = "fwd") -> float:
    f = 4.0 * B * H * N * N * d
    if pass_ == "bwd":
        f *= 2.5
    elif pass_ != "fwd":
        raise ValueError(pass_)
    return f / 2 if causal else f


def dkdv_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = (10.0 if d > 128 else 8.0) * B * H * N * N * d
    return f / 2 if causal else f


def dq_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 6.0 * B * H * N * N * d
    return f / 2 if causal else f


def nxn_traffic_bytes(N: int, bytes_per_element: int = 2):
    """(round trip, storage) in bytes of one materialised N x N matrix per (b, h).

    The IO that tiling avoids: writing the score matrix out and reading it
    back costs 2 N^2 elements, holding it costs N^2.
    """
    return 2 * N * N * bytes_per_element, N * N * bytes_per_element


def fwd_min_hbm_bytes(B: int, H: int, N: int, d: int) -> int:
    """Q, K, V read once, O written once (bf16) and LSE written (fp32)."""
    return 4 * B * H * N * d * 2 + 4 * B * H * N


def preprocess_bytes(B: int, H: int, N: int, d: int) -> int:
    """D = rowsum(dO o O): O and dO read (bf16), D written (fp32)."""
    return 2 * B * H * N * d * 2 + 4 * B * H * N
