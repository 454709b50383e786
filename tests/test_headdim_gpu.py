"""Head dims other than 64 and 128 on the GPU against the fp64 oracle: any
multiple of 8 up to 128 runs in the d = 64 or d = 128 kernels and 136 to 256
in the wide-head (d = 256) kernels, with the tensor maps' true extent, so the
columns past d are zero-filled on load and clipped on store; the sentinel
tests check that no byte past column d of any output row is written."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import make_splitkv_inputs
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu

FWD = [(1, 2, 300, 8, True), (2, 1, 257, 16, False), (1, 3, 200, 32, True), (1, 1, 129, 40, False),
       (2, 2, 384, 48, True), (1, 2, 333, 72, False), (1, 1, 500, 80, True), (2, 2, 256, 96, True),
       (1, 2, 1000, 96, False), (1, 1, 17, 112, True), (1, 2, 640, 120, False),
       # wide heads: one query tile per CTA, K/V moved as d-halves
       (1, 1, 128, 256, False), (1, 2, 300, 256, True), (2, 1, 1000, 256, False), (1, 2, 777, 192, True),
       (1, 1, 1, 256, True), (1, 3, 129, 136, False), (1, 1, 2100, 256, True), (1, 2, 512, 224, False)]
BWD = [(1, 2, 300, 8, True), (1, 3, 200, 32, False), (2, 1, 384, 48, True), (1, 2, 333, 80, False),
       (2, 2, 256, 96, True), (1, 1, 1000, 96, True), (1, 2, 129, 120, False),
       # wide heads: separate dV, dK and dQ launches with 64-row streamed tiles
       (1, 1, 128, 256, False), (1, 2, 300, 256, True), (2, 1, 1000, 192, True), (1, 2, 777, 256, False),
       (1, 1, 1, 256, True), (1, 3, 129, 136, True), (1, 1, 2100, 256, True), (1, 2, 500, 224, False)]


@pytest.mark.parametrize("B,H,N,d,causal", FWD)
def test_fwd_head_dim_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=700 + N + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


@pytest.mark.parametrize("B,H,N,d,causal", BWD)
def test_bwd_head_dim_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=720 + N + d, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    ref = oracle.attn_bwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = oracle.rel_fro_err(f64(a), b)
        assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"


@pytest.mark.parametrize("d", [40, 96, 192])
def test_outputs_leave_columns_past_d_untouched(d):
    """Outputs as [..., :d] views of rows 128 (256) wide filled with a sentinel:
    the kernels' (64, 128 or 256 wide) tile stores must clip at column d."""
    B, H, N, causal = 1, 2, 300, True
    x, g = device_inputs(B, H, N, d, seed=740 + d, with_grad=True)
    o_c, lse_c = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    dq_c, dk_c, dv_c = fa.fa_bwd(g["q"], g["k"], g["v"], o_c, lse_c, g["do"], None, causal)
    width = 128 if d <= 128 else 256
    bufs = [torch.full((B, H, N, width), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    o, dq, dk, dv = (b[..., :d] for b in bufs)
    fa.fa_fwd_strided(g["q"], g["k"], g["v"], None, causal, out=o)
    fa.fa_bwd_strided(g["q"], g["k"], g["v"], o, lse_c, g["do"], None, causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert_no_timeout()
    for b in bufs:
        assert torch.all(b[..., d:] == 7.0)
    assert torch.equal(o, o_c)
    for a, c in zip((dq, dk, dv), (dq_c, dk_c, dv_c)):
        assert torch.equal(a, c)


def test_preprocess_head_dims():
    for d in (8, 40, 96, 200, 256):
        _, g = device_inputs(2, 3, 201, d, seed=750 + d, with_grad=True)
        o = torch.randn_like(g["q"])
        Dvec = fa.fa_bwd_preprocess(o, g["do"])
        torch.cuda.synchronize()
        ref = oracle.bwd_preprocess_ref(f64(o), f64(g["do"]))
        bound = 1e-5 * np.abs(f64(o) * f64(g["do"])).sum(axis=-1) + 1e-6
        assert np.all(np.abs(f64(Dvec) - ref) <= bound), d


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits", [(1, 2, 1, 3000, 96, 0), (2, 1, 40, 1500, 40, 3)])
def test_splitkv_head_dims(B, H, Nq, Nk, d, splits):
    x = make_splitkv_inputs(B, H, Nq, Nk, d, seed=760 + d)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], scale, splits)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, False)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_dropout_head_dim():
    B, H, N, d, p, seed = 1, 2, 300, 80, 0.2, 99
    x, g = device_inputs(B, H, N, d, seed=770, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], p, seed, offset=2, scale=scale, causal=True)
    dq, dk, dv = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], p, seed, offset=2, scale=scale,
                                   causal=True)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_dropout_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, True, p, seed, 2)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE
    ref = oracle.attn_bwd_dropout_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, True, p, seed, 2)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert oracle.rel_fro_err(f64(a), b) <= TOL_GRAD, name


def test_wide_head_forward_leaves_columns_past_d_untouched():
    """d = 192 in the d = 256 kernel: the fourth 64-column box of each O row is
    never stored, and the strided call equals the contiguous one bit for bit."""
    B, H, N, d, causal = 1, 2, 300, 192, True
    _, g = device_inputs(B, H, N, d, seed=780)
    o_c, lse_c = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    buf = torch.full((B, H, N, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[..., :d]
    lse = torch.empty_like(lse_c)
    fa.fa_fwd_strided(g["q"], g["k"], g["v"], None, causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.all(buf[..., d:] == 7.0)
    assert torch.equal(o, o_c) and torch.equal(lse, lse_c)


def test_wide_head_long_rows_sampled():
    """B=2 H=4 N=4096 d=256 causal and not: 64 sampled query rows per head."""
    from io_aware_exact_14_gb300.workloads import Workload, sample_rows
    for causal in (False, True):
        w = Workload(0, "wide", 2, 4, 4096, 256, (causal,), ("fwd",), oracle_rows=64)
        x, g = device_inputs(w.B, w.H, w.N, w.d, seed=790 + causal)
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], w.scale, causal)
        torch.cuda.synchronize()
        assert_no_timeout()
        rows = sample_rows(w, 64)
        o_ref, lse_ref = oracle.attn_fwd_ref_rows(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.scale, causal, rows)
        o_np, l_np = f64(o), f64(lse)
        got_o = np.stack([np.stack([o_np[b, h, rows[b, h]] for h in range(w.H)]) for b in range(w.B)])
        got_l = np.stack([np.stack([l_np[b, h, rows[b, h]] for h in range(w.H)]) for b in range(w.B)])
        assert o_excess_err(got_o, o_ref) <= TOL_O
        assert oracle.lse_max_abs_err(got_l, lse_ref) <= TOL_LSE


def test_wide_head_backward_steps_equal_fused_call():
    """fa_bwd at d = 256 equals fa_bwd_preprocess + fa_bwd_dkdv + fa_bwd_dq, bit for bit,
    and reruns are bitwise identical (no atomics)."""
    _, g = device_inputs(1, 2, 520, 256, seed=795, with_grad=True)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], None, True)
    Dvec = fa.fa_bwd_preprocess(o, g["do"])
    dk2, dv2 = fa.fa_bwd_dkdv(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True)
    dq2 = fa.fa_bwd_dq(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True)
    dq3, dk3, dv3 = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], None, True)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert torch.equal(dq, dq3) and torch.equal(dk, dk3) and torch.equal(dv, dv3)


def test_wide_head_training_shape_sampled_slices():
    """B=2 H=8 N=4096 d=256 causal forward + backward; gradients of two sampled
    (b, h) slices against the oracle."""
    from io_aware_exact_14_gb300.workloads import Workload, sample_slices
    w = Workload(0, "wide_train", 2, 8, 4096, 256, (True,), ("fwd", "bwd"), oracle_slices=2)
    x, g = device_inputs(w.B, w.H, w.N, w.d, seed=797, with_grad=True)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], w.scale, True)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], w.scale, True)
    torch.cuda.synchronize()
    assert_no_timeout()
    for b, h in sample_slices(w, 2):
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        ref = oracle.attn_bwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), w.scale, True)
        for name, a, r in zip(("dq", "dk", "dv"), (dq[b:b + 1, h:h + 1], dk[b:b + 1, h:h + 1],
                                                     dv[b:b + 1, h:h + 1]), ref):
            err = oracle.rel_fro_err(f64(a), r)
            assert err <= TOL_GRAD, f"{name} (b={b}, h={h}): relative Frobenius error {err:.3g}"
