"""FP8 (e4m3) quantiser and forward on the GPU against the fp64 oracle
(oracle.fp8_ref): quantisation codes and descales bit for bit (both sides do
the same fp32 steps), the forward exactly where the probabilities are powers
of two, within the derived rounding bound elsewhere, and the incoherent
rotation's effect on outlier channels."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import make_splitkv_inputs
from gpu_util import TOL_LSE, assert_no_timeout, device_inputs, f64

pytestmark = pytest.mark.gpu


def _codes_np(t):
    return t.cpu().numpy().astype(np.uint8)


@pytest.mark.parametrize("B,H,N,d,transpose,rotate", [
    (1, 2, 200, 128, False, None), (2, 1, 129, 64, True, None), (1, 3, 300, 96, False, None),
    (1, 1, 77, 32, True, None), (1, 2, 256, 128, False, 1234), (2, 2, 130, 64, True, 99),
    (1, 1, 500, 128, True, 7), (1, 2, 33, 16, False, None),
    (1, 2, 200, 256, False, None), (1, 1, 300, 256, True, 77), (2, 1, 129, 192, True, None),
    (1, 2, 256, 256, False, 4321)])
def test_quantize_bit_exact(B, H, N, d, transpose, rotate):
    x, g = device_inputs(B, H, N, d, seed=800 + N + d)
    xin = g["q"] * 3.0        # a bf16 tensor; both sides quantise exactly these values
    codes, ds = fa.fa_fp8_quantize(xin, transpose=transpose, rotate_seed=rotate)
    torch.cuda.synchronize()
    ref_codes, ref_ds = fp8_ref.fp8_quantize_ref(xin.float().cpu().numpy(), rotate, transpose)
    got = _codes_np(codes)
    if transpose:
        assert got.shape == (B, H, d, fa.fa_fp8_vt_ld(N))
        assert np.all(got[..., N:] == 0)
        got = got[..., :N]
    assert np.array_equal(got, ref_codes)
    assert np.array_equal(ds.cpu().numpy(), ref_ds)


def _quantized(B, H, N, d, seed, qk_mult=1.0, rotate=None):
    x, g = device_inputs(B, H, N, d, seed=seed, qk_mult=qk_mult)
    q8, dq = fa.fa_fp8_quantize(g["q"], rotate_seed=rotate)
    k8, dk = fa.fa_fp8_quantize(g["k"], rotate_seed=rotate)
    vt8, dv = fa.fa_fp8_quantize(g["v"], transpose=True)
    return x, g, (q8, k8, vt8, dq, dk, dv)


def _oracle(args, N, scale, causal):
    q8, k8, vt8, dq, dk, dv = args
    vt = _codes_np(vt8)[..., :N]
    return fp8_ref.attn_fwd_fp8_ref(_codes_np(q8), _codes_np(k8), vt, dq.cpu().numpy(), dk.cpu().numpy(),
                                    dv.cpu().numpy(), scale, causal)


@pytest.mark.parametrize("causal,d", [(False, 128), (True, 128), (False, 256), (True, 256)])
def test_fp8_forward_power_of_two_probabilities_exact(causal, d):
    """Q = e_0, K_j = -a_j e_0 (a_j in 0..8) and scale ln 2 make every
    probability a power of two, which e4m3 holds exactly: O must match the
    oracle to output rounding (any misplaced or misordered P byte shows)."""
    B, H, N = 1, 2, 300
    rng = np.random.default_rng(11)
    q8 = np.zeros((B, H, N, d), dtype=np.uint8)
    q8[..., 0] = fp8_ref.e4m3_encode(np.array([1.0]))[0]
    k8 = np.zeros((B, H, N, d), dtype=np.uint8)
    a = rng.integers(0, 9, (B, H, N))
    k8[..., 0] = fp8_ref.e4m3_encode(-a.astype(np.float64))
    vcodes, dv = fp8_ref.fp8_quantize_ref(rng.standard_normal((B, H, N, d)).astype(np.float32), None, True)
    ld = fa.fa_fp8_vt_ld(N)
    vt8 = np.zeros((B, H, d, ld), dtype=np.uint8)
    vt8[..., :N] = vcodes
    one = np.ones((B, H), dtype=np.float32)
    dev = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    scale = math.log(2.0)
    o, lse = fa.fa_fwd_fp8(dev(q8), dev(k8), dev(vt8), dev(one), dev(one), dev(dv), scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    O, LSE, O8, _ = fp8_ref.attn_fwd_fp8_ref(q8, k8, vcodes, one, one, dv, scale, causal)
    assert np.max(np.abs(O8 - O)) <= 1e-12
    err = np.abs(f64(o) - O) - 2.0 ** -8 * np.abs(O)
    assert np.max(err) <= 1e-5
    assert np.max(np.abs(f64(lse) - LSE)) <= 1e-5


@pytest.mark.parametrize("B,H,N,d,causal,qk", [
    (1, 2, 256, 128, False, 1.0), (2, 1, 333, 128, True, 1.0), (1, 2, 129, 64, True, 3.0),
    (1, 1, 1000, 96, False, 1.0), (2, 2, 200, 32, True, 3.0), (1, 1, 17, 128, True, 1.0),
    (1, 2, 300, 256, True, 1.0), (2, 1, 333, 192, False, 1.0), (1, 1, 1000, 256, False, 1.0),
    (1, 2, 129, 144, True, 3.0)])
def test_fp8_forward_within_rounding_bound(B, H, N, d, causal, qk):
    _, _, args = _quantized(B, H, N, d, seed=820 + N + d, qk_mult=qk)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8(*args, scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    O, LSE, O8, bound = _oracle(args, N, scale, causal)
    excess = np.abs(f64(o) - O) - (1.1 * bound + 2.0 ** -8 * np.abs(O) + 1e-3)
    assert np.max(excess) <= 0, f"max excess {np.max(excess):.3g}"
    assert np.max(np.abs(f64(lse) - LSE)) <= TOL_LSE


@pytest.mark.parametrize("B,H,N,causal,d", [(1, 2, 4096, False, 128), (1, 1, 6400, True, 128),
                                             (1, 1, 3000, True, 256)])
def test_fp8_long_rows(B, H, N, causal, d):
    """Rows of 24-50 key steps per CTA: the ring and barrier phases wrap many times."""
    _, _, args = _quantized(B, H, N, d, seed=870 + N)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8(*args, scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    O, LSE, _, bound = _oracle(args, N, scale, causal)
    assert np.max(np.abs(f64(o) - O) - (1.1 * bound + 2.0 ** -8 * np.abs(O) + 1e-3)) <= 0
    assert np.max(np.abs(f64(lse) - LSE)) <= TOL_LSE


def test_fp8_full_size_sampled():
    """B=8 H=16 N=4096 d=128 causal: sampled heads within the bound."""
    B, H, N, d = 8, 16, 4096, 128
    _, _, args = _quantized(B, H, N, d, seed=830)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8(*args, scale, True)
    torch.cuda.synchronize()
    assert_no_timeout()
    for b, h in ((0, 0), (7, 15), (3, 9)):
        sub = [t[b:b + 1, h:h + 1].contiguous() for t in args[:3]] + [t[b:b + 1, h:h + 1].contiguous() for t in args[3:]]
        O, LSE, _, bound = _oracle(sub, N, scale, True)
        excess = np.abs(f64(o[b:b + 1, h:h + 1]) - O) - (1.1 * bound + 2.0 ** -8 * np.abs(O) + 1e-3)
        assert np.max(excess) <= 0, (b, h)
        assert np.max(np.abs(f64(lse[b:b + 1, h:h + 1]) - LSE)) <= TOL_LSE


def test_incoherent_rotation_helps_with_outlier_channels():
    """With four channels of Q and K 8x larger than the rest, the e4m3 errors of
    those channels' products dominate the score error (about 5% of a score
    unit); rotating first spreads them over all 128 channels (about 1.4%), so
    the FP8 output lands closer to exact bf16-input attention (expected
    relative errors about 7% and 5%)."""
    B, H, N, d = 1, 4, 512, 128
    x, g = device_inputs(B, H, N, d, seed=840)
    q, k = g["q"].clone(), g["k"].clone()
    q[..., :4] *= 8.0
    k[..., :4] *= 8.0
    scale = 1.5 / 128.5       # score std about 1.5
    ref_o, _ = oracle.attn_fwd_ref(f64(q), f64(k), f64(g["v"]), scale, False)
    errs = {}
    for rot in (None, 4321):
        q8, dq = fa.fa_fp8_quantize(q, rotate_seed=rot)
        k8, dk = fa.fa_fp8_quantize(k, rotate_seed=rot)
        vt8, dv = fa.fa_fp8_quantize(g["v"], transpose=True)
        o, _ = fa.fa_fwd_fp8(q8, k8, vt8, dq, dk, dv, scale, False)
        torch.cuda.synchronize()
        errs[rot] = oracle.rel_fro_err(f64(o), ref_o)
    assert errs[4321] < errs[None], errs
    assert errs[4321] <= 0.1, errs


@pytest.mark.parametrize("N,causal,d", [(1, False, 64), (1, True, 64), (130, True, 64), (1, True, 256),
                                         (130, False, 256), (257, True, 160)])
def test_fp8_short_and_ragged_rows(N, causal, d):
    B, H = 2, 2
    _, _, args = _quantized(B, H, N, d, seed=850 + N)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8(*args, scale, causal)
    torch.cuda.synchronize()
    assert_no_timeout()
    O, LSE, _, bound = _oracle(args, N, scale, causal)
    assert np.max(np.abs(f64(o) - O) - (1.1 * bound + 2.0 ** -8 * np.abs(O) + 1e-3)) <= 0
    assert np.max(np.abs(f64(lse) - LSE)) <= TOL_LSE


def test_fp8_all_zero_head():
    """An all-zero Q head quantises to zero codes with descale 1; its scores
    are all 0, so its output is the mean of the (dequantised) values."""
    B, H, N, d = 1, 2, 200, 128
    x, g = device_inputs(B, H, N, d, seed=860)
    q = g["q"].clone()
    q[:, 1] = 0
    q8, dq = fa.fa_fp8_quantize(q)
    k8, dk = fa.fa_fp8_quantize(g["k"])
    vt8, dv = fa.fa_fp8_quantize(g["v"], transpose=True)
    torch.cuda.synchronize()
    assert dq[0, 1].item() == 1.0 and int(q8[:, 1].to(torch.int32).sum()) == 0
    o, lse = fa.fa_fwd_fp8(q8, k8, vt8, dq, dk, dv, None, False)
    torch.cuda.synchronize()
    vt = _codes_np(vt8)[..., :N]
    V = np.swapaxes(fp8_ref.fp8_dequantize(vt, dv.cpu().numpy()), -1, -2)
    mean = V[0, 1].mean(axis=0)
    assert np.max(np.abs(f64(o[0, 1]) - mean[None, :]) - 2.0 ** -8 * np.abs(mean[None, :])) <= 1e-4
    assert np.allclose(f64(lse[0, 1]), math.log(N), atol=1e-4)


# ---------------------------------------------------------------------------
# Split-KV on e4m3 codes (decoding against an e4m3 key/value cache)
# ---------------------------------------------------------------------------

def _quantized_kv(B, H, Nq, Nk, d, seed, rotate=None):
    x = make_splitkv_inputs(B, H, Nq, Nk, d, seed)
    g = {k: t.cuda() for k, t in x.items()}
    q8, dq = fa.fa_fp8_quantize(g["q"], rotate_seed=rotate)
    k8, dk = fa.fa_fp8_quantize(g["k"], rotate_seed=rotate)
    vt8, dv = fa.fa_fp8_quantize(g["v"], transpose=True)
    return (q8, k8, vt8, dq, dk, dv)


def _oracle_kv(args, Nk, scale):
    q8, k8, vt8, dq, dk, dv = args
    vt = _codes_np(vt8)[..., :Nk]
    return fp8_ref.attn_fwd_fp8_ref(_codes_np(q8), _codes_np(k8), vt, dq.cpu().numpy(), dk.cpu().numpy(),
                                    dv.cpu().numpy(), scale, False)


def _within_bound(o, lse, O, LSE, bound):
    excess = np.abs(f64(o) - O) - (1.1 * bound + 2.0 ** -8 * np.abs(O) + 1e-3)
    assert np.max(excess) <= 0, f"max excess {np.max(excess):.3g}"
    assert np.max(np.abs(f64(lse) - LSE)) <= TOL_LSE


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits,rotate", [
    (1, 2, 1, 3000, 128, 0, None),
    (2, 2, 200, 3000, 128, 7, 5),       # two query tiles, ragged key tail, rotated Q and K
    (1, 3, 17, 129, 64, 2, None),       # a one-key last chunk
    (1, 2, 40, 1500, 96, 1, None),      # one chunk
    (1, 2, 64, 128, 32, 5, None),       # more splits wanted than key tiles
    (2, 4, 1, 8192, 128, 0, 11),
    (1, 2, 32, 1000, 128, 0, None),     # the replicated-row path's edge
    (1, 2, 33, 1000, 128, 0, None),
    (1, 2, 1, 3000, 256, 0, None),      # wide heads: width-256 chunks
    (2, 2, 200, 3000, 256, 7, 5),
    (1, 2, 40, 1500, 192, 1, None)])
def test_fp8_splitkv_within_rounding_bound(B, H, Nq, Nk, d, splits, rotate):
    args = _quantized_kv(B, H, Nq, Nk, d, seed=880 + Nq + Nk + d, rotate=rotate)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8_splitkv(*args, scale, splits)
    torch.cuda.synchronize()
    assert_no_timeout()
    O, LSE, _, bound = _oracle_kv(args, Nk, scale)
    _within_bound(o, lse, O, LSE, bound)


def test_fp8_splitkv_chunkings_agree_and_match_the_fp8_forward():
    """Every chunking stays within the bound and reruns are bitwise equal; with
    Nq == Nk the split path lands next to fa_fwd_fp8 (same e4m3 arithmetic per
    chunk, fp32 partials, one merge)."""
    B, H, N, d = 1, 2, 1000, 128
    args = _quantized_kv(B, H, N, N, d, seed=890)
    scale = 1.0 / math.sqrt(d)
    O, LSE, _, bound = _oracle_kv(args, N, scale)
    for splits in (1, 3, 8, 0):
        o, lse = fa.fa_fwd_fp8_splitkv(*args, scale, splits)
        o2, lse2 = fa.fa_fwd_fp8_splitkv(*args, scale, splits)
        torch.cuda.synchronize()
        assert_no_timeout()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        _within_bound(o, lse, O, LSE, bound)
    o1, lse1 = fa.fa_fwd_fp8_splitkv(*args, scale, 1)
    op, lsep = fa.fa_fwd_fp8(*args, scale, False)
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(o1) - f64(op)) - 2.0 ** -7 * np.abs(f64(op))) <= 1e-3
    assert np.max(np.abs(f64(lse1) - f64(lsep))) <= 1e-5


def test_fp8_splitkv_empty_keys_and_short_workspace():
    B, H, Nq, d = 2, 2, 9, 64
    x = make_splitkv_inputs(B, H, Nq, 0, d, 895)
    q8, dq = fa.fa_fp8_quantize(x["q"].cuda())
    k8 = torch.empty(B, H, 0, d, dtype=torch.uint8, device="cuda")
    vt8 = torch.empty(B, H, d, fa.fa_fp8_vt_ld(0), dtype=torch.uint8, device="cuda")
    one = torch.ones(B, H, device="cuda")
    o = torch.full((B, H, Nq, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, Nq, device="cuda")
    fa.fa_fwd_fp8_splitkv(q8, k8, vt8, dq, one, one, None, 0, out=o, lse=lse)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    args = _quantized_kv(1, 2, 16, 2048, 128, seed=896)
    need = fa.fa_fwd_fp8_splitkv_workspace_bytes(1, 2, 16, 2048, 128, 4)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8_splitkv(*args, None, 4, workspace=ws)
    assert e.value.status == fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits", [
    (1, 2, 200, 3000, 128, 7), (1, 2, 17, 1000, 128, 0), (1, 2, 40, 1500, 256, 1), (2, 1, 300, 300, 64, 2)])
def test_fp8_causal_splitkv_within_rounding_bound(B, H, Nq, Nk, d, splits):
    """Causal: query i at position Nk - Nq + i; the oracle runs the FP8
    reference on query codes placed at those positions of an Nk-row array."""
    args = _quantized_kv(B, H, Nq, Nk, d, seed=990 + Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_fp8_splitkv(*args, scale, splits, causal=True)
    torch.cuda.synchronize()
    assert_no_timeout()
    q8, k8, vt8, dq, dk, dv = args
    qp = np.zeros((B, H, Nk, d), dtype=np.uint8)
    qp[:, :, Nk - Nq:] = _codes_np(q8)
    O, LSE, _, bound = fp8_ref.attn_fwd_fp8_ref(qp, _codes_np(k8), _codes_np(vt8)[..., :Nk], dq.cpu().numpy(),
                                                dk.cpu().numpy(), dv.cpu().numpy(), scale, True)
    _within_bound(o, lse, O[:, :, Nk - Nq:], LSE[:, :, Nk - Nq:], bound[:, :, Nk - Nq:])
