"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: their device memory belongs to a
framework allocator or a fixed budget, or they sit on a latency-critical path
where cudaMalloc's implicit device synchronisation is not acceptable.  For
them fa_bwd_noalloc keeps the backward's row term in scratch built into the
library instead of a caller workspace.  This test calls it through the C ABI
twice in a row (different shapes, so the second call reuses scratch that the
first left behind) and checks each result against fa_bwd, the entry point
with a caller workspace: within the gradient tolerance of the other tests,
and bit for bit, since both run the same deterministic kernels on the same
row term (a stale row left in the scratch would show as a difference).

The file name makes pytest collect it last; it also passes when run alone.
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_14_gb300 import fa
from io_aware_exact_14_gb300.workloads import make_inputs
from gpu_util import TOL_GRAD, f64

pytestmark = pytest.mark.gpu

CASES = [
    (2, 3, 1000, 128, True),    # first call fills the scratch
    (1, 2, 517, 64, False),     # second call: fewer rows, stale rows above stay behind
]


def test_bwd_noalloc_matches_workspace_entry_point():
    for call, (B, H, N, d, causal) in enumerate(CASES):
        x = make_inputs(B, H, N, d, seed=900 + call, with_grad=True)
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        scale = 1.0 / np.sqrt(d)
        o, lse = fa.fa_fwd(q, k, v, scale, causal)
        want = fa.fa_bwd(q, k, v, o, lse, do, scale, causal)
        got = fa.fa_bwd_noalloc(q, k, v, o, lse, do, scale, causal)
        torch.cuda.synchronize()
        assert fa.fa_debug_status(reset=True) == fa.FA_OK
        for name, a, b in zip(("dq", "dk", "dv"), got, want):
            err = oracle.rel_fro_err(f64(a), f64(b))
            assert err <= TOL_GRAD, f"call {call}: {name} differs from fa_bwd by {err:.3g}"
            assert torch.equal(a, b), f"call {call}: {name} is not bitwise equal to fa_bwd's"


def test_bwd_noalloc_at_its_row_limit():
    """B*H*N = 2^21 rows, exactly the built-in scratch: equal to fa_bwd bit
    for bit (every row of the scratch is written and read)."""
    B, H, N, d, causal = 2, 16, 65536, 64, True
    g = torch.Generator(device="cpu")
    g.manual_seed(931)
    q, k, v, do = (torch.randn((B, H, N, d), generator=g).to(torch.bfloat16).cuda() for _ in range(4))
    o, lse = fa.fa_fwd(q, k, v, None, causal)
    want = fa.fa_bwd(q, k, v, o, lse, do, None, causal)
    got = fa.fa_bwd_noalloc(q, k, v, o, lse, do, None, causal)
    torch.cuda.synchronize()
    assert fa.fa_debug_status(reset=True) == fa.FA_OK
    for name, a, b in zip(("dq", "dk", "dv"), got, want):
        assert torch.equal(a, b), f"{name} is not bitwise equal to fa_bwd's at 2^21 rows"


def test_bwd_noalloc_rejects_problems_beyond_its_scratch():
    B, H, N, d = 1, 64, 32769, 64     # 2^21 + 64 rows > the built-in 2^21
    p = [0x100000 * (i + 1) for i in range(9)]
    st = fa.load().fa_bwd_noalloc(*p, B, H, N, d, 0.125, 0, None)
    assert st == 4  # FA_ERR_WORKSPACE
    assert b"exceeds the built-in scratch" in fa.load().fa_last_error_detail()
