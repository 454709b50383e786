"""A fixed, seeded sweep of shapes through the forward and the backward
against the fp64 oracle: batch, heads, ragged lengths from 1 to ~700, any
head dim that is a multiple of 8 up to 256, with and without the causal
mask, contiguous or as a strided [B, N, H, d] view.  The hand-picked cases
elsewhere cover each kernel's edges; this sweep covers their combinations
(a short causal row with a wide head, a one-key tail with the four-tile
kernel, strided views of ragged heads, ...)."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from gpu_util import TOL_GRAD, TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 5))
        N = int(rng.choice([int(rng.integers(1, 130)), int(rng.integers(130, 700))]))
        d = 8 * int(rng.integers(1, 33))
        out.append((B, H, N, d, bool(rng.integers(0, 2)), bool(rng.integers(0, 2))))
    return out


CASES = _cases(64, 2026)


def _bnhd(t):
    """The same values as a [B, H, N, d] view of [B, N, H, d] storage."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


@pytest.mark.parametrize("B,H,N,d,causal,strided", CASES)
def test_random_shape_matches_oracle(B, H, N, d, causal, strided):
    x, g = device_inputs(B, H, N, d, seed=3000 + B * 1000 + N + d, with_grad=True)
    scale = 1.0 / np.sqrt(d)
    if strided:
        q, k, v, do = (_bnhd(g[n]) for n in ("q", "k", "v", "do"))
        o, lse = fa.fa_fwd_strided(q, k, v, scale, causal)
        dq, dk, dv = fa.fa_bwd_strided(q, k, v, o, lse, do, scale, causal)
    else:
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
        dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE
    ref = oracle.attn_bwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale, causal)
    for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = oracle.rel_fro_err(f64(a), r)
        assert err <= TOL_GRAD, f"{name}: relative Frobenius error {err:.3g}"
