"""Public calls from several host threads at once, each thread on its own CUDA stream.

The calls whose launches size their dynamic shared memory by the call's shape (top-K's
per-SM cap, Finalize, Finalize + RMSNorm, the CUDA-core split-K router) set each
kernel's shared-memory limit to that kernel's largest need, the same for every call, so
that a call from one thread never lowers the limit under another thread's launch. Two
threads with different shapes call them in a loop; every result must equal, bit for
bit, the same call made alone, and no call may fail."""
import threading

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_dev, dev

pytestmark = pytest.mark.gpu

ROUNDS = 25


def _weights(T, K, seed):
    u = synth.rng(seed, synth.WEIGHTS).random((T, K)).astype(np.float32)
    return synth.f32_to_bf16_bits(u / u.sum(1, keepdims=True))


def _work(moe, T, H, E, seed):
    """One thread's inputs and the calls it repeats; returns (inputs, run)."""
    K = synth.K
    logits = dev(synth.normal_f32(seed, 12, (T, synth.E), 2.0))
    bias = dev(synth.correction_bias(seed))
    rows = bf16_dev(synth.expert_rows(T, seed=seed))
    w = bf16_dev(_weights(T, K, seed))
    g = bf16_dev(synth.norm_weight(seed))
    x = bf16_dev(synth.hidden_rows(T, seed=seed, h=H))
    gate = bf16_dev(synth.router_weight(seed, e=E, h=H))
    ws = torch.empty(max(16, moe.router_logits_workspace(T, H, E)), dtype=torch.uint8, device="cuda")

    def run(stream):
        ids, wf, _ = moe.topk_route(logits, bias, K, stream=stream)
        fin = moe.finalize(rows, w, T, K, stream=stream)
        routed, normed = moe.finalize_rmsnorm(rows, w, T, K, g, stream=stream)
        lg = moe.router_logits(x, gate, workspace=ws, algo=moe.ROUTER_SIMT, stream=stream)
        return [ids, wf, fin, routed, normed, lg]

    return run


def _bits(ts):
    return [t.contiguous().view(torch.uint8).cpu() for t in ts]


def test_two_threads_with_different_shapes(moe):
    # (token counts on both sides of every shape-dependent choice: top-K's cap of two or
    # three CTAs per SM, the Finalize + RMSNorm staging for two or three CTAs per SM, the
    # CUDA-core router's K chunk of 1280 or 2048)
    shapes = [(16, 7168, 896, 1), (1300, 2048, 256, 2)]
    runs = [_work(moe, *s) for s in shapes]
    streams = [torch.cuda.Stream() for _ in shapes]
    alone = []
    for run, s in zip(runs, streams):
        with torch.cuda.stream(s):
            out = run(s)
        s.synchronize()
        alone.append(_bits(out))
    errors, results = [], [None] * len(shapes)

    def body(i):
        try:
            with torch.cuda.stream(streams[i]):
                last = None
                for _ in range(ROUNDS):
                    last = runs[i](streams[i])
                streams[i].synchronize()
                results[i] = _bits(last)
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=body, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (a, b) in enumerate(zip(alone, results)):
        for j, (u, v) in enumerate(zip(a, b)):
            assert torch.equal(u, v), f"thread {i}, output {j}"
    assert moe.device_error(clear=True) == 0
