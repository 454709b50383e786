"""The training step captured in a CUDA graph and replayed.

Every entry point takes device pointers and launches on the caller's stream;
the kernels get their tensor maps and wait configuration as launch
parameters, so a captured forward + backward replays on whatever the static
buffers hold at replay time.  Each replay, with fresh inputs copied into the
captured buffers, must equal the same calls made eagerly, bit for bit (the
kernels are deterministic).  Covered: the three kernel families (d = 64, 128,
256), both masks, the workspace and the no-allocation backward; and a
decode step (split-KV on bf16 or e4m3 keys and values, the latter with the
query's quantisation inside the graph).
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


@pytest.mark.parametrize("d,e4m3,causal", [(128, False, False), (64, False, True), (128, True, False),
                                            (256, True, True)])
def test_graph_replay_of_decode_steps(d, e4m3, causal):
    """A decode loop's split-KV call (bf16 or e4m3 keys and values, one
    query row per head) captured once and replayed with new queries equals
    the eager call bit for bit."""
    B, H, Nq, Nk = 2, 4, 4, 3000
    _, kv = device_inputs(B, H, Nk, d, seed=7300 + d)
    q_static = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    outs = {n: (torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda"),
                torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")) for n in ("static", "eager")}
    if e4m3:
        k8, dk = fa.fa_fp8_quantize(kv["k"])
        vt8, dv = fa.fa_fp8_quantize(kv["v"], transpose=True)
        q8 = torch.empty((B, H, Nq, d), dtype=torch.uint8, device="cuda")
        dq = torch.empty((B, H), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(fa.fa_fwd_fp8_splitkv_workspace_bytes(B, H, Nq, Nk, d, 0), 1), dtype=torch.uint8,
                         device="cuda")

        def step(q, out):
            fa.fa_fp8_quantize(q, out=q8, descale=dq)
            fa.fa_fwd_fp8_splitkv(q8, k8, vt8, dq, dk, dv, None, 0, out=out[0], lse=out[1], workspace=ws,
                                  causal=causal)
    else:
        ws = torch.empty(max(fa.fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, 0), 1), dtype=torch.uint8,
                         device="cuda")

        def step(q, out):
            fa.fa_fwd_splitkv(q, kv["k"], kv["v"], None, 0, out=out[0], lse=out[1], workspace=ws, causal=causal)
    _, first = device_inputs(B, H, Nq, d, seed=7400 + d)
    q_static.copy_(first["q"])
    step(q_static, outs["static"])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(q_static, outs["static"])
    torch.cuda.synchronize()
    for rep in range(3):
        _, g = device_inputs(B, H, Nq, d, seed=7500 + 10 * d + rep)
        q_static.copy_(g["q"])
        graph.replay()
        torch.cuda.synchronize()
        step(g["q"], outs["eager"])
        torch.cuda.synchronize()
        assert_no_timeout()
        for i in range(2):
            assert torch.equal(outs["static"][i], outs["eager"][i]), f"output {i} differs on replay {rep}"
