"""Backward parity on the GPU: dQ, dK, dV (and the row term D) from the CUDA
path through the C ABI against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import WORKLOADS, oracle_slices, workload_inputs
from gpu_util import TOL_GRAD, assert_no_timeout, device_inputs, f64

pytestmark = pytest.mark.gpu

SMALL = [
    (1, 1, 128, 64, False),
    (1, 1, 128, 128, True),
    (1, 2, 200, 64, True),
    (1, 2, 200, 128, False),
    (2, 1, 384, 128, True),
    (1, 3, 129, 64, True),
    (1, 1, 640, 128, False),
    (1, 1, 17, 128, True),
    (1, 1, 1, 64, False),
    (2, 2, 1000, 64, True),
    (1, 2, 1111, 128, True),
]


def _grads(g, scale, causal):
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    return o, lse, dq, dk, dv


def _assert_grads(got, ref, where=""):
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        err = oracle.rel_fro_err(f64(a), b)
        assert err <= TOL_GRAD, f"{name}{where}: relative Frobenius error {err:.3g}"


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_bwd_small_full_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=300 + N + d + causal, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    _, _, dq, dk, dv = _grads(g, scale, causal)
    ref = oracle.attn_bwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal)
    _assert_grads((dq, dk, dv), ref)


def test_preprocess_row_term():
    """D_i = sum_c dO_ic O_ic in fp32 against the fp64 product of the same bf16 values."""
    for d in (64, 128):
        _, g = device_inputs(2, 3, 333, d, seed=21, with_grad=True)
        o = torch.randn_like(g["q"])
        Dvec = fa.fa_bwd_preprocess(o, g["do"])
        torch.cuda.synchronize()
        ref = oracle.bwd_preprocess_ref(f64(o), f64(g["do"]))
        bound = 1e-5 * np.abs(f64(o) * f64(g["do"])).sum(axis=-1) + 1e-6
        assert np.all(np.abs(f64(Dvec) - ref) <= bound)


@pytest.mark.parametrize("d,causal", [(128, True), (128, False), (64, True), (96, False), (40, True), (256, True)])
def test_bwd_steps_equal_fused_call(d, causal):
    """fa_bwd equals fa_bwd_preprocess + fa_bwd_dkdv + fa_bwd_dq, bit for bit,
    and leaves the row term D in its workspace."""
    _, g = device_inputs(2, 2, 520, d, seed=22 + d, with_grad=True)
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    o, lse = fa.fa_fwd(q, k, v, None, causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(2, 2, 520, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, None, causal, workspace=ws)
    Dvec = fa.fa_bwd_preprocess(o, do)
    dk2, dv2 = fa.fa_bwd_dkdv(q, k, v, lse, do, Dvec, None, causal)
    dq2 = fa.fa_bwd_dq(q, k, v, lse, do, Dvec, None, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.equal(ws[:Dvec.numel() * 4].view(torch.float32).view_as(Dvec), Dvec)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_bwd_deterministic_and_identities():
    """Bitwise reruns; sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 up to rounding."""
    _, g = device_inputs(2, 2, 768, 64, seed=23, with_grad=True)
    r1 = _grads(g, None, True)
    r2 = _grads(g, None, True)
    for a, b in zip(r1[2:], r2[2:]):
        assert torch.equal(a, b)
    dk, dv = r1[3].double(), r1[4].double()
    do = g["do"].double()
    dv_sum, do_sum = dv.sum(dim=2), do.sum(dim=2)
    assert torch.linalg.vector_norm(dv_sum - do_sum) <= 2e-2 * torch.linalg.vector_norm(do_sum)
    dk_sum = dk.sum(dim=2)
    # each row carries ~1e-2 relative rounding; random errors add up to ~that of ||dK||_F
    assert torch.linalg.vector_norm(dk_sum) <= 2e-2 * torch.linalg.vector_norm(dk)


def test_bwd_no_write_outside_outputs():
    B, H, N, d = 1, 2, 200, 128
    _, g = device_inputs(B, H, N, d, seed=24, with_grad=True)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    pad = 4096
    n = B * H * N * d
    bufs = [torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    views = [b[pad:pad + n].view(B, H, N, d) for b in bufs]
    fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], None, True, dq=views[0], dk=views[1], dv=views[2])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:pad] == 7.0) and torch.all(b[-pad:] == 7.0)


@pytest.mark.parametrize("index", [2, 5])
def test_bwd_workload_parity(index):
    """Full-size backward on the workloads that train.  The oracle checks every
    (b, h) slice of B=4 H=16 N=2048 (both masks) and two sampled slices of the
    B=8 H=16 N=4096 training step."""
    w = WORKLOADS[index]
    x = workload_inputs(w, with_grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    for causal in w.causal:
        _, _, dq, dk, dv = _grads(g, w.scale, causal)
        for t in (dq, dk, dv):
            assert torch.isfinite(t.float()).all()
        for b, h in oracle_slices(w):
            sl = lambda t: f64(t[b:b + 1, h:h + 1])
            ref = oracle.attn_bwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), w.scale, causal)
            _assert_grads((dq[b:b + 1, h:h + 1], dk[b:b + 1, h:h + 1], dv[b:b + 1, h:h + 1]), ref,
                          f" (b={b}, h={h}, causal={causal})")


def test_dq_concurrent_streams_bitwise():
    """The dQ kernel takes work over from not-yet-started CTAs of its own grid:
    two launches running at once on two streams must each give exactly what
    they give alone."""
    _, ga = device_inputs(2, 4, 1500, 128, seed=31, with_grad=True)
    _, gb = device_inputs(2, 4, 1500, 128, seed=32, with_grad=True)
    ref = []
    for g in (ga, gb):
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
        Dvec = fa.fa_bwd_preprocess(o, g["do"])
        torch.cuda.synchronize()
        dq = fa.fa_bwd_dq(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True)
        torch.cuda.synchronize()
        ref.append((lse, Dvec, dq))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out = [torch.empty_like(ref[0][2]), torch.empty_like(ref[1][2])]
    for _ in range(3):
        for g, (lse, Dvec, _), s, dq in zip((ga, gb), ref, (sa, sb), out):
            fa.fa_bwd_dq(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True, dq=dq, stream=s)
        torch.cuda.synchronize()
        assert_no_timeout()
        assert torch.equal(out[0], ref[0][2]) and torch.equal(out[1], ref[1][2])


def test_dkdv_concurrent_streams_bitwise():
    """The dK/dV kernel, like dQ, takes work over from not-yet-started CTAs of
    its own grid: two launches running at once on two streams must each give
    exactly what they give alone."""
    _, ga = device_inputs(2, 4, 1500, 128, seed=33, with_grad=True)
    _, gb = device_inputs(2, 4, 1500, 128, seed=34, with_grad=True)
    ref = []
    for g in (ga, gb):
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
        Dvec = fa.fa_bwd_preprocess(o, g["do"])
        torch.cuda.synchronize()
        dk, dv = fa.fa_bwd_dkdv(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True)
        torch.cuda.synchronize()
        ref.append((lse, Dvec, dk, dv))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out = [(torch.empty_like(r[2]), torch.empty_like(r[3])) for r in ref]
    for _ in range(3):
        for g, (lse, Dvec, _, _), s, (dk, dv) in zip((ga, gb), ref, (sa, sb), out):
            fa.fa_bwd_dkdv(g["q"], g["k"], g["v"], lse, g["do"], Dvec, None, True, dk=dk, dv=dv, stream=s)
        torch.cuda.synchronize()
        assert_no_timeout()
        for (dk, dv), r in zip(out, ref):
            assert torch.equal(dk, r[2]) and torch.equal(dv, r[3])


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 64, 300, 64, True), (2, 96, 256, 128, False)])
def test_bwd_many_short_units_parity(B, H, N, d, causal):
    """Hundreds of one- to three-tile work units, several per persistent CTA:
    the protocols that carry rings, barriers and epilogue stores from one unit
    to the next (and the stores still pending when a CTA runs out of work)."""
    x, g = device_inputs(B, H, N, d, seed=900 + N + d, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    _, _, dq, dk, dv = _grads(g, scale, causal)
    ref = oracle.attn_bwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal)
    _assert_grads((dq, dk, dv), ref)
