"""Concurrent calls from several host threads, each on its own CUDA stream.

The binding releases the interpreter lock during each C call, so the
library's host state is exercised concurrently: the per-thread tensor-map
cache, the per-context kernel-attribute cache, the per-device SM-count cache
and the per-launch wait epochs.  Every thread runs the forward and the
backward on its own shapes (head dims 64, 96, 128, 256), interleaved, many
times; each result must equal bit for bit the one computed before on the
default stream (the kernels are deterministic)."""
import threading

import pytest
import torch

from io_aware_exact_14_gb300 import fa
from gpu_util import assert_no_timeout, device_inputs

pytestmark = pytest.mark.gpu

SHAPES = [(1, 4, 700, 128, True), (2, 2, 513, 64, False), (1, 3, 300, 256, True), (2, 2, 1000, 96, False)]
ROUNDS = 8


def _step(g, causal, stream):
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], None, causal, stream=stream)
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], None, causal, stream=stream)
    return o, lse, dq, dk, dv


def test_threads_on_their_own_streams_match_serial_results():
    inputs = [device_inputs(B, H, N, d, seed=4000 + i, with_grad=True)[1] for i, (B, H, N, d, _) in enumerate(SHAPES)]
    ref = [tuple(t.clone() for t in _step(g, s[4], None)) for g, s in zip(inputs, SHAPES)]
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            g, causal = inputs[i], SHAPES[i][4]
            for r in range(ROUNDS):
                with torch.cuda.stream(stream):
                    out = _step(g, causal, stream)
                stream.synchronize()
                for k, (a, b) in enumerate(zip(out, ref[i])):
                    if not torch.equal(a, b):
                        errors.append(f"thread {i} round {r} output {k} differs")
                        return
        except Exception as e:   # reported by the main thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(SHAPES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    assert_no_timeout()
