"""The training step captured in a CUDA graph and replayed.

Every entry point takes device pointers and launches on the caller's stream;
the kernels get their tensor maps and wait configuration as launch
parameters, so a captured forward + backward replays on whatever the static
buffers hold at replay time.  Each replay, with fresh inputs copied into the
captured buffers, must equal the same calls made eagerly, bit for bit (the
kernels are deterministic).  Covered: the three kernel families (d = 64, 128,
256), both masks, the workspace and the no-allocation backward.
"""
import pytest
import torch

from io_aware_exact_14_gb300 import fa
from gpu_util import assert_no_timeout, device_inputs

pytestmark = pytest.mark.gpu


def _step(t, causal, noalloc):
    fa.fa_fwd(t["q"], t["k"], t["v"], None, causal, out=t["o"], lse=t["lse"])
    if noalloc:
        fa.fa_bwd_noalloc(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], None, causal, dq=t["dq"], dk=t["dk"],
                          dv=t["dv"])
    else:
        fa.fa_bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], None, causal, dq=t["dq"], dk=t["dk"],
                  dv=t["dv"], workspace=t["ws"])


def _buffers(B, H, N, d):
    t = {n: torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
         for n in ("q", "k", "v", "do", "o", "dq", "dk", "dv")}
    t["lse"] = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    t["ws"] = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    return t


@pytest.mark.parametrize("d,causal,noalloc", [(128, True, False), (128, False, True), (64, True, False),
                                              (256, True, False)])
def test_graph_replay_equals_eager_calls(d, causal, noalloc):
    B, H, N = 2, 3, 700
    static = _buffers(B, H, N, d)
    eager = _buffers(B, H, N, d)
    _, first = device_inputs(B, H, N, d, seed=7100 + d, with_grad=True)
    for n in ("q", "k", "v", "do"):
        static[n].copy_(first[n])
    _step(static, causal, noalloc)   # first calls (kernel attributes, scratch lookup) before the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(static, causal, noalloc)
    torch.cuda.synchronize()
    for rep in range(3):
        _, g = device_inputs(B, H, N, d, seed=7200 + 10 * d + rep, with_grad=True)
        for n in ("q", "k", "v", "do"):
            static[n].copy_(g[n])
            eager[n].copy_(g[n])
        graph.replay()
        torch.cuda.synchronize()
        _step(eager, causal, noalloc)
        torch.cuda.synchronize()
        assert_no_timeout()
        for n in ("o", "lse", "dq", "dk", "dv"):
            assert torch.equal(static[n], eager[n]), f"{n} differs on replay {rep}"
