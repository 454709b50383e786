"""Split-KV forward (short query blocks against long key sequences) on the GPU
against the fp64 oracle's plain definition, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import make_splitkv_inputs
from gpu_util import TOL_LSE, TOL_O, assert_no_timeout, f64, o_excess_err

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, num_splits (0: the library's choice)
    (1, 1, 1, 1000, 128, 0),
    (2, 3, 5, 4097, 64, 3),
    (1, 2, 128, 8192, 128, 0),
    (2, 2, 200, 3000, 128, 7),      # two query tiles, ragged key tail
    (1, 4, 64, 128, 64, 5),         # more splits wanted than key tiles
    (1, 1, 17, 129, 128, 2),        # a one-key last chunk
    (3, 2, 33, 700, 64, 1),         # one chunk: the plain kernel plus the merge
    # wide heads (the d = 256 kernel's split mode)
    (1, 1, 1, 3000, 256, 0),
    (2, 2, 200, 3000, 256, 7),      # two query tiles, ragged key tail
    (1, 3, 17, 129, 160, 2),        # a one-key last chunk, d below the box width
    (1, 2, 40, 1500, 192, 1),       # one chunk
    (1, 2, 64, 128, 200, 5),        # more splits wanted than key tiles, d not a multiple of 32
    # the replicated-row path (up to 32 query rows at d <= 64) at its edge and just past it
    (2, 2, 32, 2000, 64, 0),
    (2, 2, 33, 2000, 64, 0),
    (1, 3, 31, 700, 40, 3),
    (1, 2, 32, 1500, 256, 2),
]


def _run(B, H, Nq, Nk, d, splits, seed):
    x = make_splitkv_inputs(B, H, Nq, Nk, d, seed)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], scale, splits)
    torch.cuda.synchronize()
    assert_no_timeout()
    return x, g, scale, o, lse


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits", CASES)
def test_splitkv_parity(B, H, Nq, Nk, d, splits):
    x, _, scale, o, lse = _run(B, H, Nq, Nk, d, splits, seed=500 + Nq + Nk + d)
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, False)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


@pytest.mark.parametrize("d", [128, 256])
def test_splitkv_split_counts_agree(d):
    """Every chunking reaches the same exact result, within the forward tolerance
    of the oracle, and the same chunking twice is bitwise the same."""
    B, H, Nq, Nk = 2, 2, 40, 2500
    x = make_splitkv_inputs(B, H, Nq, Nk, d, 77)
    g = {k: t.cuda() for k, t in x.items()}
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), 0.1, False)
    for splits in (1, 2, 5, 20, 0):
        o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], 0.1, splits)
        o2, lse2 = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], 0.1, splits)
        torch.cuda.synchronize()
        assert_no_timeout()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        assert o_excess_err(f64(o), o_ref) <= TOL_O
        assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_splitkv_matches_plain_forward_when_lengths_agree():
    """Nq == Nk, non-causal: the split path and fa_fwd both reach the oracle."""
    B, H, N, d = 1, 3, 1000, 64
    x = make_splitkv_inputs(B, H, N, N, d, 81)
    g = {k: t.cuda() for k, t in x.items()}
    o_s, lse_s = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], None, 4)
    o_p, lse_p = fa.fa_fwd(g["q"], g["k"], g["v"], None, False)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert (o_s.float() - o_p.float()).abs().max().item() <= 2 * TOL_O
    assert (lse_s - lse_p).abs().max().item() <= 2 * TOL_LSE


@pytest.mark.parametrize("d", [64, 256])
def test_splitkv_empty_keys_and_queries(d):
    """Nk == 0: every row has no key, O = 0 and LSE = -inf; Nq == 0 is a no-op."""
    q = torch.randn(2, 2, 9, d, device="cuda").to(torch.bfloat16)
    kv = torch.empty(2, 2, 0, d, device="cuda", dtype=torch.bfloat16)
    o = torch.full_like(q, 7.0)
    lse = torch.zeros(2, 2, 9, device="cuda")
    fa.fa_fwd_splitkv(q, kv, kv, None, 0, out=o, lse=lse)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    q0 = torch.empty(2, 2, 0, d, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(2, 2, 300, d, device="cuda").to(torch.bfloat16)
    o0, lse0 = fa.fa_fwd_splitkv(q0, k, k, None, 0)
    assert o0.numel() == 0 and lse0.numel() == 0


def test_splitkv_rejects_short_workspace():
    """A workspace below fa_fwd_splitkv_workspace_bytes is refused before any launch."""
    B, H, Nq, Nk, d = 1, 2, 16, 2048, 128
    x = make_splitkv_inputs(B, H, Nq, Nk, d, 90)
    g = {k: t.cuda() for k, t in x.items()}
    need = fa.fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, 4)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], None, 4, workspace=ws)
    assert e.value.status == fa.FA_ERR_WORKSPACE


# Causal split-KV: the query block is the last Nq positions of the Nk-long
# sequence (query i at position Nk - Nq + i), the oracle's end-aligned mask.
def _causal_ref(x, scale):
    return oracle.attn_fwd_ref_end_aligned(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale)


CAUSAL_CASES = [
    # B, H, Nq, Nk, d, num_splits
    (1, 2, 1, 3000, 128, 0),        # one query row: sees every key
    (2, 2, 200, 3000, 128, 7),      # two query tiles, early chunks past some rows' positions
    (1, 3, 17, 129, 64, 2),         # replicated rows, a one-key last chunk
    (2, 2, 32, 2000, 64, 0),        # replicated rows at their edge
    (1, 2, 64, 128, 200, 5),        # more splits wanted than key tiles
    (1, 2, 40, 1500, 256, 1),       # wide heads, one chunk
    (1, 1, 500, 700, 96, 0),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,splits", CAUSAL_CASES)
def test_causal_splitkv_parity(B, H, Nq, Nk, d, splits):
    x = make_splitkv_inputs(B, H, Nq, Nk, d, 900 + Nq + Nk + d)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], scale, splits, causal=True)
    torch.cuda.synchronize()
    assert_no_timeout()
    o_ref, lse_ref = _causal_ref(x, scale)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_causal_splitkv_equal_lengths_is_the_square_mask():
    """Nq == Nk: the same result as fa_fwd's causal forward (both within the
    tolerance of the oracle)."""
    B, H, N, d = 1, 2, 700, 128
    x = make_splitkv_inputs(B, H, N, N, d, 950)
    g = {k: t.cuda() for k, t in x.items()}
    o_s, lse_s = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], None, 3, causal=True)
    o_p, lse_p = fa.fa_fwd(g["q"], g["k"], g["v"], None, True)
    torch.cuda.synchronize()
    assert_no_timeout()
    assert (o_s.float() - o_p.float()).abs().max().item() <= 2 * TOL_O
    assert (lse_s - lse_p).abs().max().item() <= 2 * TOL_LSE


def test_causal_splitkv_queries_before_the_first_key():
    """Nq > Nk: the first Nq - Nk queries sit before position 0 and see no key
    (O = 0, LSE = -inf); the rest match the oracle at their positions."""
    B, H, Nq, Nk, d = 1, 2, 300, 200, 64
    x = make_splitkv_inputs(B, H, Nq, Nk, d, 960)
    g = {k: t.cuda() for k, t in x.items()}
    o, lse = fa.fa_fwd_splitkv(g["q"], g["k"], g["v"], None, 2, causal=True)
    torch.cuda.synchronize()
    assert_no_timeout()
    cut = Nq - Nk
    assert torch.all(o[:, :, :cut] == 0) and torch.all(torch.isneginf(lse[:, :, :cut]))
    tail = {"q": x["q"][:, :, cut:], "k": x["k"], "v": x["v"]}
    o_ref, lse_ref = _causal_ref(tail, 1.0 / np.sqrt(d))
    assert o_excess_err(f64(o[:, :, cut:]), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse[:, :, cut:]), lse_ref) <= TOL_LSE
