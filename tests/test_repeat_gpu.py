"""Every kernel family, run many times over: no wait ever gives up, and every
run is bitwise identical to the first.

None of the kernels reduces with atomics or depends on the order in which
CTAs or pipeline roles happen to run, so reruns on the same inputs must give
the same bits; a pipeline race (a barrier phase overtaken by its waiter, a
buffer reused early) shows up as a difference between runs or as a recorded
timeout.  Such races depend on timing, so each case runs REPS times, with
other kernel families launched in between to vary what runs where.  Sizes
span many CTAs, the persistent backward's work stealing and both issue
strategies of the forward.
"""
import pytest
import torch

from io_aware_exact_14_gb300 import fa
from gpu_util import assert_no_timeout, device_inputs

pytestmark = pytest.mark.gpu

REPS = 6


def _fwd(B, H, N, d, causal, seed):
    _, g = device_inputs(B, H, N, d, seed=seed)
    return lambda: fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)


def _bwd(B, H, N, d, causal, seed):
    _, g = device_inputs(B, H, N, d, seed=seed, with_grad=True)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal)
    return lambda: fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], None, causal)


def _dropout(B, H, N, d, causal, seed):
    _, g = device_inputs(B, H, N, d, seed=seed, with_grad=True)

    def run():
        o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], 0.1, 1234, 0, None, causal)
        return (o, lse) + tuple(fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], 0.1, 1234, 0, None,
                                                  causal))
    return run


def _splitkv(B, H, Nq, Nk, d, seed, causal=False):
    _, gq = device_inputs(B, H, Nq, d, seed=seed)
    _, gk = device_inputs(B, H, Nk, d, seed=seed + 1)
    return lambda: fa.fa_fwd_splitkv(gq["q"], gk["k"], gk["v"], causal=causal)


def _fp8_splitkv(B, H, Nq, Nk, d, seed):
    _, gq = device_inputs(B, H, Nq, d, seed=seed)
    _, gk = device_inputs(B, H, Nk, d, seed=seed + 1)
    q8, dq = fa.fa_fp8_quantize(gq["q"])
    k8, dk = fa.fa_fp8_quantize(gk["k"])
    vt8, dv = fa.fa_fp8_quantize(gk["v"], transpose=True)
    return lambda: fa.fa_fwd_fp8_splitkv(q8, k8, vt8, dq, dk, dv)


def _fp8(B, H, N, d, causal, seed):
    _, g = device_inputs(B, H, N, d, seed=seed)

    def run():
        q8, dq = fa.fa_fp8_quantize(g["q"], rotate_seed=5)
        k8, dk = fa.fa_fp8_quantize(g["k"], rotate_seed=5)
        vt8, dv = fa.fa_fp8_quantize(g["v"], transpose=True)
        return (q8, k8, vt8, dq, dk, dv) + tuple(fa.fa_fwd_fp8(q8, k8, vt8, dq, dk, dv, None, causal))
    return run


CASES = {
    "fwd_d128_causal": lambda: _fwd(2, 8, 2048, 128, True, 901),
    "fwd_d128_two_issuers": lambda: _fwd(1, 8, 3200, 128, False, 902),
    "fwd_d64_four_tiles": lambda: _fwd(2, 8, 2048, 64, False, 903),
    "fwd_d96": lambda: _fwd(2, 4, 1500, 96, True, 904),
    "fwd_d256": lambda: _fwd(2, 4, 2048, 256, True, 905),
    "bwd_d128_causal": lambda: _bwd(2, 8, 2048, 128, True, 906),
    "bwd_d128": lambda: _bwd(2, 4, 1536, 128, False, 907),
    "bwd_d64_causal": lambda: _bwd(2, 8, 2048, 64, True, 908),
    "bwd_d256_causal": lambda: _bwd(2, 4, 2048, 256, True, 909),
    "bwd_d192": lambda: _bwd(1, 4, 1100, 192, False, 910),
    "dropout_d128_causal": lambda: _dropout(2, 4, 1024, 128, True, 911),
    "dropout_d256_causal": lambda: _dropout(1, 4, 1024, 256, True, 914),
    "splitkv_d128": lambda: _splitkv(2, 8, 128, 8192, 128, 912),
    "splitkv_d256": lambda: _splitkv(2, 8, 64, 8192, 256, 915),
    "splitkv_d64_decode": lambda: _splitkv(4, 8, 1, 8192, 64, 917),
    "splitkv_d128_causal_chunk": lambda: _splitkv(2, 8, 256, 8192, 128, 918, True),
    "fp8_d128_causal": lambda: _fp8(2, 8, 2048, 128, True, 913),
    "fp8_splitkv_d128": lambda: _fp8_splitkv(2, 8, 16, 8192, 128, 916),
    "fp8_d256_causal": lambda: _fp8(2, 4, 2048, 256, True, 919),
    "fp8_splitkv_d256": lambda: _fp8_splitkv(2, 8, 1, 8192, 256, 920),
}


def _as_tuple(x):
    return x if isinstance(x, tuple) else (x,)


@pytest.mark.parametrize("name", sorted(CASES))
def test_reruns_are_bitwise_identical_and_never_time_out(name):
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    run = CASES[name]()
    # another family between reruns shifts which SM runs which CTA when
    other = CASES["fwd_d128_causal" if name != "fwd_d128_causal" else "bwd_d128"]()
    first = [t.clone() for t in _as_tuple(run())]
    torch.cuda.synchronize()
    assert_no_timeout()
    for rep in range(REPS):
        if rep % 2:
            other()
        again = _as_tuple(run())
        torch.cuda.synchronize()
        assert_no_timeout()
        for i, (a, b) in enumerate(zip(first, again)):
            assert torch.equal(a, b), f"{name}: output {i} differs on rerun {rep + 1}"
