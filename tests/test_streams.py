"""Stream ordering and CUDA-graph capture of the entry points.

Decode and prefill calls of at most 4096 rows run the kv_b product on a second
stream of the library's own, forked from the caller's stream and joined back
into it with events, so a call is ordered on the caller's stream as a whole.
Checked here through the C ABI, bit for bit against the same call on the
default stream (the same kernels in the same configuration on the same
inputs give the same bits):
- calls on a non-default stream, whose outputs are then read by work queued
  on that stream;
- calls captured into a CUDA graph (after one uncaptured call of the same
  host thread, which creates the side stream) and replayed, twice, the second
  time with new inputs written into the captured buffers: a rebuilt-cache
  decode step (B = 64, the side stream), a short prefill (T = 16, the side
  stream) and a latent decode step (one stream throughout);
- a call captured as the first call of its host thread (no side stream is
  created during a capture: the call stays on the capturing stream);
- two host threads calling at the same time on their own streams.
"""
import pytest

import synth
import mla_gb300 as m
from mla_testlib import cuda_weights

pytestmark = pytest.mark.gpu


def _decode_inputs(B, P, cap, seed):
    x = synth.tensor_cuda(seed, "new_x", (B, 7168), synth.X_DIST)
    k = synth.tensor_cuda(seed, "cache_x", (B, 64, cap, 192), (0.0, 1.0))
    v = synth.tensor_cuda(seed + 1, "cache_x", (B, 64, cap, 128), (0.0, 0.5))
    return x, k, v


def test_decode_on_user_stream_matches_default_stream(gpu_available):
    import torch
    W = m.make_weights(cuda_weights(0))
    B, P = 64, 200
    cap = P + 1
    x, k, v = _decode_inputs(B, P, cap, 11)
    ws = m.alloc_workspace(m.MODE_DECODE, B, P)
    k_ref, v_ref, out_ref = k.clone(), v.clone(), torch.empty_like(x)
    m.mla_decode(W, x, P, k_ref, v_ref, out_ref, ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ws2 = m.alloc_workspace(m.MODE_DECODE, B, P)
    k2, v2, out2 = k.clone(), v.clone(), torch.empty_like(x)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):  # repeated steps on the same buffers: each must finish before the next reads
            m.mla_decode(W, x, P, k2, v2, out2, ws2)
        # work on the same stream right after the call sees its finished outputs
        got = out2.clone()
        krow = k2[:, :, P, :].clone()
        vrow = v2[:, :, P, :].clone()
    s.synchronize()
    assert torch.equal(got, out_ref)
    assert torch.equal(krow, k_ref[:, :, P, :]) and torch.equal(vrow, v_ref[:, :, P, :])
    assert torch.equal(k2, k_ref) and torch.equal(v2, v_ref)


def _capture_and_replay(call, refresh, outputs):
    """Capture call() into a graph, replay it, refresh the inputs, replay
    again; returns the outputs after each replay (clones)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    first = [o.clone() for o in outputs]
    refresh()
    g.replay()
    torch.cuda.synchronize()
    second = [o.clone() for o in outputs]
    return first, second


def test_decode_graph_replay_matches_eager(gpu_available):
    import torch
    W = m.make_weights(cuda_weights(0))
    B, P = 64, 120
    cap = P + 1
    x, k, v = _decode_inputs(B, P, cap, 12)
    x_new = synth.tensor_cuda(13, "new_x", (B, 7168), synth.X_DIST)
    ws = m.alloc_workspace(m.MODE_DECODE, B, P)
    # eager references (the first also creates this thread's side stream)
    refs = []
    for xi in (x, x_new):
        kr, vr, orf = k.clone(), v.clone(), torch.empty_like(x)
        m.mla_decode(W, xi, P, kr, vr, orf, ws)
        refs.append((orf, kr, vr))
    torch.cuda.synchronize()
    xs, kg, vg, og = x.clone(), k.clone(), v.clone(), torch.zeros_like(x)
    first, second = _capture_and_replay(lambda: m.mla_decode(W, xs, P, kg, vg, og, ws),
                                        lambda: xs.copy_(x_new), [og, kg, vg])
    for got, (orf, kr, vr) in zip((first, second), refs):
        assert torch.equal(got[0], orf)
        assert torch.equal(got[1], kr) and torch.equal(got[2], vr)


def test_short_prefill_graph_replay_matches_eager(gpu_available):
    import torch
    W = m.make_weights(cuda_weights(0))
    B, T = 1, 16
    x = synth.tensor_cuda(14, "x", (B, T, 7168), synth.X_DIST)
    x_new = synth.tensor_cuda(15, "x", (B, T, 7168), synth.X_DIST)
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    refs = []
    for xi in (x, x_new):
        orf = torch.empty_like(x)
        m.mla_prefill(W, xi, orf, ws)
        refs.append(orf)
    torch.cuda.synchronize()
    xs, og = x.clone(), torch.zeros_like(x)
    first, second = _capture_and_replay(lambda: m.mla_prefill(W, xs, og, ws), lambda: xs.copy_(x_new), [og])
    assert torch.equal(first[0], refs[0])
    assert torch.equal(second[0], refs[1])


def test_latent_decode_graph_replay_matches_eager(gpu_available):
    import torch
    W = m.make_weights(cuda_weights(0))
    B, P = 4, 300
    cap = P + 1
    x = synth.tensor_cuda(16, "new_x", (B, 7168), synth.X_DIST)
    x_new = synth.tensor_cuda(17, "new_x", (B, 7168), synth.X_DIST)
    ckv = synth.tensor_cuda(16, "cache_x", (B, cap, 512), (0.0, 1.0))
    kpe = synth.tensor_cuda(17, "cache_x", (B, cap, 64), (0.0, 1.0))
    ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    refs = []
    for xi in (x, x_new):
        c1, c2, orf = ckv.clone(), kpe.clone(), torch.empty_like(x)
        m.mla_decode_latent(W, xi, P, c1, c2, orf, ws)
        refs.append((orf, c1, c2))
    torch.cuda.synchronize()
    xs, cg1, cg2, og = x.clone(), ckv.clone(), kpe.clone(), torch.zeros_like(x)
    first, second = _capture_and_replay(lambda: m.mla_decode_latent(W, xs, P, cg1, cg2, og, ws),
                                        lambda: xs.copy_(x_new), [og, cg1, cg2])
    for got, (orf, c1, c2) in zip((first, second), refs):
        assert torch.equal(got[0], orf)
        assert torch.equal(got[1], c1) and torch.equal(got[2], c2)


def _in_thread(fn):
    """Run fn() on a new host thread (its own side-stream state) and return
    its result, re-raising what it raised."""
    import threading
    box = {}

    def run():
        import torch
        torch.cuda.set_device(0)
        try:
            box["value"] = fn()
        except BaseException as e:  # handed back to the caller
            box["error"] = e
    t = threading.Thread(target=run)
    t.start()
    t.join()
    if "error" in box:
        raise box["error"]
    return box["value"]


def test_capture_as_first_call_of_a_thread(gpu_available):
    """A thread whose first call is captured: the library creates no stream
    during the capture, so that call stays on the capturing stream; the
    replay still matches the eager call bit for bit."""
    import torch
    W = m.make_weights(cuda_weights(0))
    B, P = 64, 50
    cap = P + 1
    x, k, v = _decode_inputs(B, P, cap, 18)
    ws = m.alloc_workspace(m.MODE_DECODE, B, P)
    kr, vr, orf = k.clone(), v.clone(), torch.empty_like(x)
    m.mla_decode(W, x, P, kr, vr, orf, ws)
    torch.cuda.synchronize()

    def captured_first():
        kg, vg, og = k.clone(), v.clone(), torch.zeros_like(x)
        ws2 = m.alloc_workspace(m.MODE_DECODE, B, P)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            m.mla_decode(W, x, P, kg, vg, og, ws2)
        g.replay()
        torch.cuda.synchronize()
        return og.clone(), kg.clone(), vg.clone()
    og, kg, vg = _in_thread(captured_first)
    assert torch.equal(og, orf)
    assert torch.equal(kg, kr) and torch.equal(vg, vr)


def test_two_threads_on_two_streams(gpu_available):
    """Two host threads, each with its own stream, workspace and side
    stream, run decode steps at the same time: each result equals the
    single-threaded one."""
    import threading
    import torch
    W = m.make_weights(cuda_weights(0))
    B, P = 64, 80
    cap = P + 1
    inputs = [_decode_inputs(B, P, cap, 20 + i) for i in range(2)]
    refs = []
    for x, k, v in inputs:
        kr, vr, orf = k.clone(), v.clone(), torch.empty_like(x)
        m.mla_decode(W, x, P, kr, vr, orf, m.alloc_workspace(m.MODE_DECODE, B, P))
        refs.append((orf, kr, vr))
    torch.cuda.synchronize()
    results = [None, None]
    errors = []
    start = threading.Barrier(2)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            x, k, v = inputs[i]
            s = torch.cuda.Stream()
            kg, vg, og = k.clone(), v.clone(), torch.empty_like(x)
            ws = m.alloc_workspace(m.MODE_DECODE, B, P)
            torch.cuda.synchronize()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(5):
                    m.mla_decode(W, x, P, kg, vg, og, ws)
            s.synchronize()
            results[i] = (og, kg, vg)
        except BaseException as e:
            errors.append(e)
    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for (og, kg, vg), (orf, kr, vr) in zip(results, refs):
        assert torch.equal(og, orf)
        assert torch.equal(kg, kr) and torch.equal(vg, vr)
