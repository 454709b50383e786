"""The deadlock guard on the GPU: a bounded wait that runs into its limit.

Every pipeline wait of the kernels gives up after a limit, records a site in
a status word, ends the other waits of its launch and unwinds (copies and
products already issued land, tensor memory is freed).  Here the forward's
copy producer withholds one K/V group (a flag that nothing sets, in effect),
with the waits limited to 20 ms: the tensor-core warp's wait for that group
runs out.  The test checks that the kernel returns, that fa_debug_status
reports FA_ERR_TIMEOUT at a forward site, and that the failure ends only its
own launch: a forward made afterwards, with the failure still recorded,
matches the oracle.  No GPU fault, trap or endless wait is involved.
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from gpu_util import TOL_LSE, TOL_O, device_inputs, f64, o_excess_err

pytestmark = pytest.mark.gpu

LIMIT_US = 20000
SITE_GROUP_WAIT = 0x102     # the forward's wait for a K/V group (tensor-core warp)
SITE_S_WAIT = 0x106         # a softmax warp's wait for its scores


def _forward_matches_oracle(x, g, causal):
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    torch.cuda.synchronize()
    scale = 1.0 / np.sqrt(x["q"].shape[-1])
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_withheld_group_times_out_in_one_cta_and_later_launches_run():
    # one CTA: two query tiles, two key steps (groups 0: K_0, 1: V_0 K_1, 2: V_1)
    x, g = device_inputs(1, 1, 256, 128, seed=31)
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    st = fa.fa_debug_fwd_withhold(g["q"], g["k"], g["v"], withhold_group=1, wait_limit_us=LIMIT_US)
    assert st == fa.FA_OK
    torch.cuda.synchronize()          # the launch ended
    assert fa.fa_debug_status(reset=False) == fa.FA_ERR_TIMEOUT
    # the tensor-core warp starts waiting for group 1 before any softmax warp
    # waits for the scores that need it, so its limit normally runs out first
    assert fa.fa_debug_site() in (SITE_GROUP_WAIT, SITE_S_WAIT), hex(fa.fa_debug_site())
    # the failure is still recorded: later launches must not be cut short by it
    for causal in (False, True):
        _forward_matches_oracle(x, g, causal)
    assert fa.fa_debug_status(reset=True) == fa.FA_ERR_TIMEOUT   # first failure kept until reset
    assert fa.fa_debug_status(reset=False) == fa.FA_OK


def test_withheld_group_ends_every_cta_of_the_launch():
    # 16 CTAs (4 heads x 4 query-tile pairs); every producer withholds group 3
    x, g = device_inputs(2, 2, 1024, 64, seed=32)
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    for causal in (False, True):
        st = fa.fa_debug_fwd_withhold(g["q"], g["k"], g["v"], withhold_group=3, wait_limit_us=LIMIT_US,
                                      causal=causal)
        assert st == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_debug_status(reset=False) == fa.FA_ERR_TIMEOUT
        assert 0x100 <= fa.fa_debug_site() < 0x200, hex(fa.fa_debug_site())
        _forward_matches_oracle(x, g, causal)
        assert fa.fa_debug_status(reset=True) == fa.FA_ERR_TIMEOUT
    assert fa.fa_debug_status(reset=False) == fa.FA_OK


def test_group_past_the_last_withholds_nothing():
    x, g = device_inputs(1, 2, 300, 128, seed=33)
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    o = torch.empty_like(g["q"])
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    st = fa.fa_debug_fwd_withhold(g["q"], g["k"], g["v"], withhold_group=1000, wait_limit_us=LIMIT_US,
                                  out=o, lse=lse)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    o_ref, lse_ref = oracle.attn_fwd_ref(f64(x["q"]), f64(x["k"]), f64(x["v"]), 1.0 / np.sqrt(128), False)
    assert o_excess_err(f64(o), o_ref) <= TOL_O
    assert oracle.lse_max_abs_err(f64(lse), lse_ref) <= TOL_LSE


def test_hook_rejects_bad_arguments():
    _, g = device_inputs(1, 1, 128, 64, seed=34)
    assert fa.fa_debug_fwd_withhold(g["q"], g["k"], g["v"], withhold_group=-1, wait_limit_us=LIMIT_US) \
        == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_fwd_withhold(g["q"], g["k"], g["v"], withhold_group=0, wait_limit_us=0) \
        == fa.FA_ERR_INVALID_ARG
