"""Strided layouts on the GPU: [B, N, H, d] and packed [B, N, 3, H, d] views go
through the same kernels as the contiguous layout (only the copy engine's
addressing differs), so results must be bitwise those of the contiguous path,
and within tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu


def _bnhd(t):
    """Copy of a contiguous [B, H, N, d] tensor stored as [B, N, H, d], viewed as [B, H, N, d]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 300, 64, True), (1, 4, 257, 128, False), (2, 2, 512, 128, True),
                                             (1, 2, 300, 256, True), (2, 2, 200, 192, False), (1, 3, 700, 40, True)])
def test_fwd_bnhd_bitwise_and_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=610 + N + d)
    o_ref_dev, lse_ref_dev = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    q, k, v = (_bnhd(g[n]) for n in ("q", "k", "v"))
    assert q.stride() == (N * H * d, d, H * d, 1)
    out = torch.empty(B, N, H, d, dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o, lse = fa.fa_fwd_strided(q, k, v, None, causal, out=out)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.equal(o, o_ref_dev) and torch.equal(lse, lse_ref_dev)
    o64, lse64 = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), 1.0 / np.sqrt(d), causal)
    assert o_excess_err(f64(o), o64) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse64) <= TOL_LSE


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 300, 64, True), (1, 2, 384, 128, False), (1, 2, 300, 256, True),
                                             (1, 1, 200, 160, False)])
def test_bwd_packed_qkv_bitwise_and_parity(B, H, N, d, causal):
    """q, k, v read from one [B, N, 3, H, d] buffer and dq, dk, dv written into
    another; o and dO stored as [N, B, H, d]."""
    x, g = device_inputs(B, H, N, d, seed=640 + N + d, with_grad=True)
    o_c, lse_c = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    dq_c, dk_c, dv_c = fa.fa_bwd(g["q"], g["k"], g["v"], o_c, lse_c, g["do"], None, causal)
    qkv = torch.stack([g[n].transpose(1, 2) for n in ("q", "k", "v")], dim=2).contiguous()   # [B, N, 3, H, d]
    q, k, v = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    nbhd = lambda t: t.permute(2, 0, 1, 3).contiguous().permute(1, 2, 0, 3)   # [N, B, H, d] storage
    o, do = nbhd(o_c), nbhd(g["do"])
    dqkv = torch.empty(B, N, 3, H, d, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = (dqkv[:, :, i].transpose(1, 2) for i in range(3))
    fa.fa_bwd_strided(q, k, v, o, lse_c, do, None, causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.equal(dq, dq_c) and torch.equal(dk, dk_c) and torch.equal(dv, dv_c)
    ref = oracle.attn_bwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), 1.0 / np.sqrt(d), causal)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert oracle.rel_fro_err(f64(a), b) <= TOL_GRAD, name


def test_strided_rejects_unaligned_row_stride():
    """A view whose row stride is not 16-byte aligned is refused (FA_ERR_INVALID_ARG)."""
    base = torch.zeros(1, 2, 100, 64 + 4, dtype=torch.bfloat16, device="cuda")
    q = base[..., :64]
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_strided(q, q, q)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
