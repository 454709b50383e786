"""Counting helpers against the figures the pages print (CPU only)."""
import json
import os

from io_aware_exact_14_gb300 import counts

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_io_arithmetic_matches_page():
    with open(os.path.join(GOLDEN, "kernel101_io_arithmetic.json"), encoding="utf-8") as f:
        g = json.load(f)
    rt, st = counts.nxn_traffic_bytes(g["N"], g["bytes_per_element"])
    assert rt / 2**20 == g["printed_round_trip_MiB"]
    assert st / 2**20 == g["printed_storage_MiB"]


def test_flop_convention():
    # forward 4*B*H*N^2*d, backward 2.5x, causal halves
    assert counts.attn_flops(1, 1, 128, 64, False) == 4 * 128 * 128 * 64
    assert counts.attn_flops(8, 16, 4096, 128, True) == 2 * 8 * 16 * 4096**2 * 128
    assert counts.attn_flops(8, 16, 4096, 128, True, "bwd") == 2.5 * counts.attn_flops(8, 16, 4096, 128, True)
    # the two backward kernels execute 14/10 of the counted backward work
    B, H, N, d = 4, 16, 2048, 128
    ex = counts.dkdv_flops(B, H, N, d, False) + counts.dq_flops(B, H, N, d, False)
    assert ex == 1.4 * counts.attn_flops(B, H, N, d, False, "bwd")
    assert counts.fwd_min_hbm_bytes(8, 16, 4096, 128) == 4 * 8 * 16 * 4096 * 128 * 2 + 4 * 8 * 16 * 4096
