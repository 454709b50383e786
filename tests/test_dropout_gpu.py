"""Dropout on the probabilities, fused into the CUDA kernels, against the fp64
oracle: the keep mask bit for bit (read back through O and dV with one-hot
inputs), O and LSE, and dQ, dK, dV of the same mask."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import WORKLOADS, sample_slices, workload_inputs
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu

SEED = 0x1234_5678_9ABC_DEF0

SMALL = [
    (1, 1, 128, 64, False, 0.1),
    (1, 2, 200, 128, True, 0.25),
    (2, 1, 384, 128, False, 0.1),
    (1, 3, 129, 64, True, 0.5),
    (1, 1, 17, 128, True, 0.2),
    (2, 2, 1000, 64, True, 0.1),
    (1, 2, 1111, 128, False, 0.15),
    (1, 2, 200, 256, True, 0.25),
    (1, 1, 300, 160, False, 0.1),
    (2, 1, 129, 192, True, 0.5),
    (1, 1, 17, 256, False, 0.2),
    (1, 1, 700, 256, False, 0.15),
]


def _onehot_v(B, H, N, d, kb):
    """V with V[j, c] = 1 where j = 128 kb + c: O[i, c] then isolates key 128 kb + c."""
    v = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    for c in range(min(d, N - 128 * kb)):
        v[:, :, 128 * kb + c, c] = 1.0
    return v


@pytest.mark.parametrize("p,d", [(0.1, 128), (0.5, 128), (0.9, 128), (0.999, 128), (0.1, 256), (0.5, 256)])
def test_forward_mask_bit_exact(p, d):
    """Q = K = 0 makes P uniform (1/N), so with one-hot V each output element is
    keep * scale / N: nonzero exactly where the mask keeps."""
    B, H, N = 2, 3, 384
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    for kb in range((N + 127) // 128):
        v = _onehot_v(B, H, N, d, kb)
        o, _ = fa.fa_fwd_dropout(q, q, v, p, SEED, offset=7, scale=0.125)
        torch.cuda.synchronize()
        assert_no_timeout()
        got = (o.float() != 0).cpu().numpy()
        for b in range(B):
            for h in range(H):
                keep = oracle.dropout_keep(b * H + h, N, N, p, SEED, 7)
                assert np.array_equal(got[b, h, :, :128], keep[:, 128 * kb:128 * kb + 128]), (b, h, kb)


@pytest.mark.parametrize("d", [128, 256])
def test_dkdv_mask_bit_exact(d):
    """dV = (P o M~)^T dO with uniform P and one-hot dO reads the mask through
    the dK/dV kernel's own draw (its threads hold keys, not queries)."""
    B, H, N, p = 1, 2, 256, 0.3
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    v = torch.randn(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fa_fwd_dropout(q, q, v, p, SEED, offset=3, scale=0.125)
    for ib in range(N // 128):
        do = _onehot_v(B, H, N, d, ib)     # dO[i, c] = 1 where i = 128 ib + c
        _, _, dv = fa.fa_bwd_dropout(q, q, v, o, lse, do, p, SEED, offset=3, scale=0.125)
        torch.cuda.synchronize()
        assert_no_timeout()
        got = (dv.float() != 0).cpu().numpy()   # dV[j, c] = keep[128 ib + c, j] * scale / N
        for h in range(H):
            keep = oracle.dropout_keep(h, N, N, p, SEED, 3)
            assert np.array_equal(got[0, h, :, :128], keep[128 * ib:128 * ib + 128, :].T), (h, ib)


@pytest.mark.parametrize("B,H,N,d,causal,p", SMALL)
def test_dropout_forward_parity(B, H, N, d, causal, p):
    x, g = device_inputs(B, H, N, d, seed=500 + N + d + causal)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], p, SEED, offset=N, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_dropout_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal, p,
                                                 SEED, N)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert np.max(np.abs(f64(lse) - lse_ref)) <= TOL_LSE


@pytest.mark.parametrize("B,H,N,d,causal,p", SMALL)
def test_dropout_backward_parity(B, H, N, d, causal, p):
    x, g = device_inputs(B, H, N, d, seed=600 + N + d + causal, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], p, SEED, offset=1, scale=scale, causal=causal)
    dq, dk, dv = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], p, SEED, offset=1, scale=scale,
                                   causal=causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    ref = oracle.attn_bwd_dropout_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal, p,
                                      SEED, 1)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = oracle.rel_fro_err(f64(a), b)
        assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"


def test_dropout_zero_rate_is_plain_and_seeds_differ():
    """p below 1/512 quantises to t = 0 and runs the plain kernels (bitwise the
    same results); another offset draws another mask; reruns are bitwise equal."""
    _, g = device_inputs(1, 2, 300, 128, seed=41, with_grad=True)
    o0, l0 = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    o1, l1 = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], 0.001, SEED, causal=True)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = fa.fa_bwd(g["q"], g["k"], g["v"], o0, l0, g["do"], None, True)
    g1 = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o1, l1, g["do"], 0.0, SEED, causal=True)
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)
    oa, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], 0.2, SEED, offset=0, causal=True)
    ob, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], 0.2, SEED, offset=0, causal=True)
    oc, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], 0.2, SEED, offset=1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and not torch.equal(oa, oc)


def test_dropout_training_workload_sampled_parity():
    """B=8 H=16 N=4096 d=128 causal with p = 0.1: the oracle checks sampled
    (b, h) slices, each with its own head index in the mask counter."""
    w = WORKLOADS[5]
    x = workload_inputs(w, with_grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    p, off = 0.1, 11
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], p, SEED, offset=off, scale=w.scale, causal=True)
    dq, dk, dv = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], p, SEED, offset=off,
                                   scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert_no_timeout()
    for b, h in sample_slices(w, 1):
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        o_ref, lse_ref = oracle.attn_fwd_dropout_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), w.scale, True, p,
                                                     SEED, off, head0=b * w.H + h)
        assert o_excess_err(sl(o), o_ref) <= TOL_O
        assert np.max(np.abs(sl(lse) - lse_ref)) <= TOL_LSE
        ref = oracle.attn_bwd_dropout_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), w.scale, True, p,
                                          SEED, off, head0=b * w.H + h)
        for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            err = oracle.rel_fro_err(sl(a), r)
            assert err <= TOL_GRAD, f"{name} (b={b}, h={h}): relative Frobenius error {err:.3g}"
