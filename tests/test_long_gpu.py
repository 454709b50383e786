"""Long sequences: one head with a million keys through the forward, a 32K-row
causal head through the backward (16K rows for the other head dims and the
non-causal mask), a million-key decode through split-KV.

At these lengths the oracle cannot materialise S, so it is evaluated at
sampled entries (first rows, tile edges, the ragged tail and seeded random
picks): the forward at sampled query rows, the backward at sampled query rows
(dQ) and key rows (dK, dV), with every query row still contributing to the
dK and dV sums.  What this exercises beyond the other tests: offsets and
tensor-map coordinates near 2^20, fp32 row sums and accumulators over 8192
key steps, persistent backward units with 256 query tiles, and split-KV
partitions of very long key ranges.  A last case runs tensors of 2^31
elements (4 GiB each) through the forward and the backward for each kernel
family (d = 64, 128, 256), through split-KV and through the FP8 path: one
seeded block repeated along the batch, so every copy must give the same bits
as the first (which the oracle checks), whatever its offset.
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import make_splitkv_inputs
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu


def _picks(N, n_random, seed):
    fixed = [0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rng = np.random.default_rng(seed)
    r = rng.integers(0, N, n_random)
    return np.unique(np.clip(np.concatenate([fixed, r]), 0, N - 1))


@pytest.mark.parametrize("N,d,causal", [(1 << 20, 128, True), (1 << 20, 128, False), ((1 << 18) - 37, 64, True),
                                        ((1 << 18) + 77, 256, True)])
def test_fwd_long_rows(N, d, causal):
    x, g = device_inputs(1, 1, N, d, seed=5000 + d + causal, with_grad=False)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    rows = _picks(N, 16, 5100 + d)[None, None, :]
    o = f64(o[:, :, rows[0, 0]])
    lse = f64(lse[:, :, rows[0, 0]])
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref_rows(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal, rows)
    assert o_excess_err(o, o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(lse, lse_ref) <= TOL_LSE


@pytest.mark.parametrize("N,d,causal", [(32768 + 77, 128, True), (16384 + 77, 128, False), (16384 - 5, 64, True),
                                        (16384 + 77, 256, True)])
def test_bwd_long_rows(N, d, causal):
    x, g = device_inputs(1, 1, N, d, seed=5200 + d + causal, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], scale, causal)
    rows = _picks(N, 24, 5300 + d)[None, None, :]
    cols = _picks(N, 24, 5400 + d)[None, None, :]
    dq, dk, dv = f64(dq[:, :, rows[0, 0]]), f64(dk[:, :, cols[0, 0]]), f64(dv[:, :, cols[0, 0]])
    assert_no_timeout()
    ref = oracle.attn_bwd_ref_sampled(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal,
                                      rows, cols, group=2048)
    for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = oracle.rel_fro_err(a, r)
        assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"


def test_splitkv_million_keys():
    B, H, Nq, Nk, d = 1, 1, 5, 1 << 20, 128
    x = make_splitkv_inputs(B, H, Nq, Nk, d, seed=5500)
    g = {k: t.cuda() for k, t in x.items()}
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"])
    o, lse = f64(o), f64(lse)
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), 1.0 / np.sqrt(d), False)
    assert o_excess_err(o, o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(lse, lse_ref) <= TOL_LSE


@pytest.mark.parametrize("d", [64, 128, 256])
def test_tensors_of_2_31_elements(d):
    b0, H, N, causal = 8, 64, 512, True
    reps = (1 << 31) // (b0 * H * N * d)          # [8 reps, 64, 512, d]: 2^31 elements
    x, g = device_inputs(b0, H, N, d, seed=5600 + d, with_grad=True)
    big = {n: t.repeat(reps, 1, 1, 1) for n, t in g.items()}
    assert big["q"].numel() == 1 << 31
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(big["q"], big["k"], big["v"], scale, causal)
    grads = fa.fa_bwd(big["q"], big["k"], big["v"], o, lse, big["do"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    for name, t in (("o", o), ("lse", lse)) + tuple(zip(("dq", "dk", "dv"), grads)):
        blocks = t.view(reps, -1)
        assert bool((blocks == blocks[:1]).all()), f"{name}: a repeated block differs from the first"
    # the first block against the oracle on two (b, h) slices
    for b, h in ((0, 0), (b0 - 1, H - 1)):
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        o_ref, lse_ref = oracle.attn_fwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), scale, causal)
        assert o_excess_err(sl(o), o_ref) <= TOL_O
        assert oracle.lse_max_abs_err(sl(lse), lse_ref) <= TOL_LSE
        ref = oracle.attn_bwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), scale, causal)
        for name, a, r in zip(("dq", "dk", "dv"), grads, ref):
            err = oracle.rel_fro_err(sl(a), r)
            assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"


def test_splitkv_keys_of_2_31_elements():
    """Split-KV decode with K and V of 2^31 elements: repeated blocks agree bit
    for bit, and the first matches the oracle."""
    b0, H, Nq, Nk, d = 2, 64, 3, 4096, 128
    reps = (1 << 31) // (b0 * H * Nk * d)
    x = make_splitkv_inputs(b0, H, Nq, Nk, d, seed=5700)
    g = {k: t.cuda().repeat(reps, 1, 1, 1) for k, t in x.items()}
    assert g["k"].numel() == 1 << 31
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"])
    torch.cuda.synchronize()
    assert_no_timeout()
    for name, t in (("o", o), ("lse", lse)):
        blocks = t.view(reps, -1)
        assert bool((blocks == blocks[:1]).all()), f"{name}: a repeated block differs from the first"
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"][:, :2]), f64(x["k"][:, :2]), f64(x["v"][:, :2]),
                                         1.0 / np.sqrt(d), False)
    assert o_excess_err(f64(o[:b0, :2]), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse[:b0, :2]), lse_ref) <= TOL_LSE


def test_fp8_path_on_tensors_of_2_31_elements():
    """The e4m3 quantiser (rotated and transposed) and the FP8 forward on
    tensors of 2^31 elements: repeated blocks give identical codes, descales
    and outputs (the FP8 oracle checks the codes elsewhere)."""
    b0, H, N, d, causal = 8, 64, 512, 128, True
    reps = (1 << 31) // (b0 * H * N * d)
    _, g = device_inputs(b0, H, N, d, seed=5800)
    big = {n: t.repeat(reps, 1, 1, 1) for n, t in g.items()}
    q8, dq = fa.fa_fp8_quantize(big["q"], rotate_seed=11)
    k8, dk = fa.fa_fp8_quantize(big["k"], rotate_seed=11)
    vt8, dv = fa.fa_fp8_quantize(big["v"], transpose=True)
    o, lse = fa.fa_fwd_fp8(q8, k8, vt8, dq, dk, dv, None, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8), ("descale_q", dq), ("descale_v", dv), ("o", o),
                    ("lse", lse)):
        blocks = t.reshape(reps, -1)
        assert bool((blocks == blocks[:1]).all()), f"{name}: a repeated block differs from the first"


def test_strided_views_of_2_31_elements():
    """q, k, v as views of one packed [B, N, 3, H, d] buffer and dq, dk, dv
    written into another, each view of 2^31 elements: repeated blocks agree
    bit for bit and the first matches the oracle."""
    b0, H, N, d, causal = 8, 64, 512, 128, True
    reps = (1 << 31) // (b0 * H * N * d)
    x, g = device_inputs(b0, H, N, d, seed=5900, with_grad=True)
    packed = torch.stack([g[n].transpose(1, 2) for n in ("q", "k", "v")], dim=2).repeat(reps, 1, 1, 1, 1)
    q, k, v = (packed[:, :, i].transpose(1, 2) for i in range(3))   # [B, H, N, d] views
    do = g["do"].repeat(reps, 1, 1, 1)
    assert q.numel() == 1 << 31 and packed.numel() == 3 << 31
    o, lse = fa.fa_fwd_strided(q, k, v, None, causal)
    dpacked = torch.empty_like(packed)
    dq, dk, dv = (dpacked[:, :, i].transpose(1, 2) for i in range(3))
    fa.fa_bwd_strided(q, k, v, o, lse, do, None, causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert_no_timeout()
    for name, t in (("o", o), ("lse", lse), ("dqkv", dpacked)):
        blocks = t.reshape(reps, -1)
        assert bool((blocks == blocks[:1]).all()), f"{name}: a repeated block differs from the first"
    scale = 1.0 / np.sqrt(d)
    b, h = b0 - 1, H - 1
    sl = lambda t: f64(t[b:b + 1, h:h + 1])
    o_ref, lse_ref = oracle.attn_fwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), scale, causal)
    assert o_excess_err(sl(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(sl(lse), lse_ref) <= TOL_LSE
    ref = oracle.attn_bwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), scale, causal)
    for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = oracle.rel_fro_err(sl(a), r)
        assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"
