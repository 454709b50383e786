"""Forward parity on the GPU: the CUDA path through the C ABI against the fp64
oracle on the same seeded bf16 inputs, element by element."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import WORKLOADS, oracle_slices, sample_rows, workload_inputs
from gpu_util import TOL_LSE, TOL_O, assert_no_timeout, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu

# Shapes that span several tiles, ragged tails (N % 128 != 0), an odd count of
# query tiles (the second tile of a CTA absent), N below one tile and N = 1.
SMALL = [
    (1, 1, 128, 64, False),
    (1, 1, 128, 64, True),
    (1, 2, 200, 64, True),
    (1, 2, 200, 128, False),
    (2, 1, 384, 128, True),
    (1, 3, 129, 64, True),
    (1, 1, 640, 128, False),
    (1, 1, 17, 128, True),
    (1, 1, 1, 64, False),
    (1, 1, 1, 128, True),
    (2, 2, 1000, 64, False),
    (1, 2, 1111, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_fwd_small_full_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=100 + N + d + causal)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


# Long rows switch the d = 128 forward to one MMA-issuing warp per query tile
# (at >= 24 key steps per CTA on average): cover that launch path in full,
# with ragged tails, non-causal (25 steps) and causal (25 steps on average).
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 1, 3100, 128, False), (1, 1, 6200, 128, True)])
def test_fwd_two_issuer_full_parity(B, H, N, d, causal):
    x, g = device_inputs(B, H, N, d, seed=500 + N + causal)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_fwd_scale_argument():
    x, g = device_inputs(1, 2, 300, 64, seed=7)
    for scale in (0.02, 0.5):
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], scale, False)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, False)
        assert o_excess_err(f64(o), o_ref) <= TOL_O
        assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_fwd_no_write_outside_outputs():
    """Canaries around O and LSE stay untouched (ragged N: the tail tile is clipped)."""
    B, H, N, d = 1, 2, 200, 128
    _, g = device_inputs(B, H, N, d, seed=11)
    pad = 4096
    o_buf = torch.full((B * H * N * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(g["q"], g["k"], g["v"], None, True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[-pad:] == 7.0)


def test_fwd_deterministic_and_causal_last_row():
    """Bitwise identical reruns; causal row N-1 equals non-causal row N-1."""
    _, g = device_inputs(2, 3, 1024, 128, seed=12)
    o1, l1 = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    o2, l2 = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    o3, l3 = fa.fa_fwd(g["q"], g["k"], g["v"], None, False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1[:, :, -1], o3[:, :, -1])
    assert torch.equal(l1[:, :, -1], l3[:, :, -1])


def _check_rows(w, x, o, lse, causal, rows):
    o_ref, lse_ref = oracle.attn_fwd_ref_rows(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.scale, causal, rows)
    o_np, lse_np = f64(o), f64(lse)
    B, H, R = rows.shape
    got_o = np.stack([np.stack([o_np[b, h, rows[b, h]] for h in range(H)]) for b in range(B)])
    got_l = np.stack([np.stack([lse_np[b, h, rows[b, h]] for h in range(H)]) for b in range(B)])
    assert o_excess_err(got_o, o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(got_l, lse_ref) <= TOL_LSE


def _check_slices(w, x, o, lse, causal, slices):
    for b, h in slices:
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        o_ref, lse_ref = oracle.attn_fwd_ref(sl(x["q"]), sl(x["k"]), sl(x["v"]), w.scale, causal)
        assert o_excess_err(sl(o), o_ref) <= TOL_O, (b, h)
        assert oracle.lse_max_abs_err(sl(lse), lse_ref) <= TOL_LSE, (b, h)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_fwd_workload_parity(index):
    """Each workload at its full size, in the launch configuration the benchmark times.

    The oracle checks every row of every head, slice by slice (bounded host
    memory), except where the workload states a sample: 256 query rows per
    head at N = 16384, two (b, h) slices of the B = 8 training step."""
    w = WORKLOADS[index]
    x = workload_inputs(w, with_grad=False)
    g = {k: t.cuda() for k, t in x.items()}
    for causal in w.causal:
        o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], w.scale, causal)
        torch.cuda.synchronize()
        assert_no_timeout()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        if w.oracle_rows:
            _check_rows(w, x, o, lse, causal, sample_rows(w, w.oracle_rows))
        else:
            _check_slices(w, x, o, lse, causal, oracle_slices(w))
