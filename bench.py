"""Benchmark of the GB300 MLA sublayer (one JSON line on stdout, rank 0).

Headline step: causal prefill of B=8 sequences of T=4096 tokens (Kimi K2
MLA dims) that also writes both cache forms (rebuilt per-head K/V and the
576-value latent cache), with seeded synthetic inputs already resident in
HBM; metric = tokens/s.  The same line carries the other workloads of the
metric as sub-objects -- prefill B=1 T=2048, prefill B=1 T=16 (weight-bound),
decode on the rebuilt cache B=64 P=1000 and on the latent cache B=128
P=8192 -- and the widened rows (chunked prefill, FP8 weights, ragged and
folded decode, the MLP half, the dense block), a roofline entry for each
dominant kernel, an end-to-end number through the C ABI with host buffers,
the CPU-oracle baseline, the GPU clocks seen during the timed region and the
number of kernel launches.  A compact "summary" of every configuration ends
the line; each configuration's summary is also printed to stderr as it
finishes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--quick]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (sequences are independent, no collective on the data path): value =
all tokens of all ranks / max-over-ranks time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA prefill tokens/s (% bf16 TC peak); decode step µs & HBM GB/s (% of 8 TB/s)"
WORKLOAD = "mla_prefill B=8 T=4096 causal, writes rebuilt K/V and latent caches (Kimi K2 MLA dims)"
NOMINAL_HBM_GBS = 8000.0
D, H, QL, KVL, NOPE, ROPE, QK, V = 7168, 64, 1536, 512, 128, 64, 192, 128
FFN_I = 18432  # SwiGLU MLP width
FFN_WEIGHT_BYTES = 2 * (7168 + 3 * 7168 * FFN_I)
WEIGHT_BYTES = 2 * (7168 + 1536 * 7168 + 1536 + 12288 * 1536 + 576 * 7168 + 512 + 16384 * 512 + 7168 * 8192)


# ---------------------------------------------------------------------------
# algorithmic work (flops count the causal lower triangle, diagonal included)
# ---------------------------------------------------------------------------
def proj_flops_per_token():
    return 2 * (D * (QL + KVL + ROPE) + QL * H * QK + KVL * H * (NOPE + V) + H * V * D)


def prefill_attn_flops(B, T, P0=0):
    """Query t of a chunk after P0 cached positions scores P0 + t + 1 keys."""
    return B * (T * P0 + T * (T + 1) // 2) * 2 * (QK + V) * H


def stage_work(name, mode, B, T_or_P, past=0):
    """(kind, amount) of algorithmic work of one stage launch: ("flop", F) or ("byte", Bytes)."""
    n = B * T_or_P if mode == "prefill" else B
    if name == "a_proj":
        return ("flop", 2 * n * D * (QL + KVL + ROPE))
    if name == "q_b":
        return ("flop", 2 * n * QL * H * QK)
    if name == "kv_b":
        return ("flop", 2 * n * KVL * H * (NOPE + V))
    if name == "o_proj":
        return ("flop", 2 * n * H * V * D)
    if name == "attn" and mode == "prefill":
        return ("flop", prefill_attn_flops(B, T_or_P, past))
    if name == "attn" and mode == "decode":
        L = T_or_P + 1
        return ("byte", B * H * L * (QK + V) * 2)
    if name == "attn" and mode == "latent":
        L = T_or_P + 1
        return ("byte", B * L * (KVL + ROPE) * 2)
    if mode == "ffn":  # MLP half over n = B * T_or_P rows, tensor-bound
        n = B * T_or_P
        if name == "gate_up":
            return ("flop", 2 * n * D * 2 * FFN_I)
        if name == "down":
            return ("flop", 2 * n * FFN_I * D)
    if mode == "ffn_dec":  # few rows: the weights stream once
        n = B * T_or_P
        if name == "gate_up":
            return ("byte", 2 * FFN_I * D * 2 + n * (D + FFN_I) * 2)
        if name == "down":
            return ("byte", FFN_I * D * 2 + n * (FFN_I + 2 * D) * 2)
    return (None, 0)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(v, device=None):
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return v
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank, world, ms_max):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for r in csv.reader(io.StringIO(out)):
            if len(r) >= 9:
                self.rows.append([c.strip() for c in r])
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# The sources each kernel's code and launch configuration come from.
KERNEL_SOURCES = {
    "gemm": ["gemm.cu", "common.cuh", "internal.h"],
    "attn_prefill": ["attn_prefill.cu", "common.cuh", "internal.h"],
    "attn_decode": ["attn_decode.cu", "common.cuh", "internal.h"],
}


def kernel_source_hash(files=None):
    """sha256 (16 hex digits) of the named files under mla_gb300/csrc (all of them by default)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_gb300", "csrc")
    for f in sorted(files if files is not None else os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_stage, config):
    """dram bytes per launch of a stage's kernel from the committed ncu summary,
    only if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{config}:{kernel_stage}")
    if not e or e.get("source_hash") != kernel_source_hash(KERNEL_SOURCES[e["kernel_sources"]]):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
class Runner:
    def __init__(self, device):
        import torch
        import mla_gb300 as m
        import synth
        self.torch, self.m, self.synth = torch, m, synth
        self.dev = device
        self.wt = synth.weights_cuda(0, device=device)
        self.W = m.make_weights(self.wt)
        self.stream = torch.cuda.current_stream()
        self.flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def flush_l2(self):
        """Evict every input from L2: write 512 MB (four times the L2), then
        read it back, so that the lines this writes are also written back to
        HBM here, not during the next timed step."""
        self.flush_buf.zero_()
        self.flush_sum = self.flush_buf.sum()

    def timing(self):
        t = self.m.MlaTiming()
        evs = []
        for i in range(self.m.MAX_STAGES):
            a = self.torch.cuda.Event(enable_timing=True)
            b = self.torch.cuda.Event(enable_timing=True)
            a.record()
            b.record()
            t.start[i] = a.cuda_event
            t.stop[i] = b.cuda_event
            evs.append((a, b))
        return t, evs

    def time_steps(self, step, steps, warmup, flush=True, with_stages=True, stages=None, probe_steps=3,
                   dominant_events=True):
        """Time `steps` calls of step(timing).

        A short instrumented pass first records events around every stage
        (the per-stage breakdown, reported as stage_ms) and picks the
        dominant stage.  The timed region then records events only around
        the whole step and, with dominant_events, around the dominant stage,
        so that the other stages are not separated by event records
        (kernels of one call overlap their start-up with the previous
        kernel's tail).  Without dominant_events the timed steps carry no
        event inside them, and the dominant stage's time is the
        instrumented pass's."""
        torch = self.torch
        for _ in range(warmup):
            step(None)
        torch.cuda.synchronize()
        stage_ms, launches, dom = {}, 0, None
        if with_stages:
            tims = [self.timing() for _ in range(probe_steps)]
            for i in range(probe_steps):
                if flush:
                    self.flush_l2()
                step(tims[i][0])
            torch.cuda.synchronize()
            launches = tims[0][0].n_launches
            for si, name in enumerate(self.m.STAGES):
                if stages is not None and name not in stages:
                    continue  # the library records only the stages its entry point runs
                stage_ms[name] = statistics.mean(evs[si][0].elapsed_time(evs[si][1]) for _, evs in tims)
            dom = max(stage_ms, key=stage_ms.get) if stage_ms else None
            if dom is not None and not dominant_events:
                stage_ms["_dominant_probe"] = (dom, stage_ms[dom])
                dom = None
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        dev_t = []
        for i in range(steps):
            t = None
            if dom is not None:
                t = self.m.MlaTiming()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                b.record()
                si = self.m.STAGES.index(dom)
                t.start[si] = a.cuda_event
                t.stop[si] = b.cuda_event
                dev_t.append((t, a, b))
            if flush:
                self.flush_l2()
            ev[i][0].record()
            step(t)
            ev[i][1].record()
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in ev]
        if dom is not None:
            stage_ms["_dominant_timed"] = (dom, statistics.mean(a.elapsed_time(b) for _, a, b in dev_t))
        return ms, stage_ms, launches

    def time_e2e_pipelined(self, x, out, ws, caches, B, T, steps, warmup):
        """Mean ms per step of mla_prefill through the C ABI with host buffers:
        every step copies its input from pinned host memory (H2D stream),
        runs the call (compute stream) and copies its output back to pinned
        host memory (D2H stream).  Two device buffers of each kind let the
        copies of step i + 1 and i - 1 run while step i computes; events
        order each buffer's reuse.  The timed region runs from before the
        first copy to the end of the last copy back."""
        torch, m = self.torch, self.m
        xh = x.cpu().pin_memory()
        ohs = [torch.empty_like(xh).pin_memory() for _ in range(2)]
        xds = [torch.empty_like(x) for _ in range(2)]
        ods = [out, torch.empty_like(out)]
        comp = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        x_ready, x_free = [ev(), ev()], [ev(), ev()]
        o_ready, o_free = [ev(), ev()], [ev(), ev()]
        for e in x_free + o_free:
            e.record(comp)

        def run(n):
            for i in range(n):
                j = i & 1
                with torch.cuda.stream(h2d):
                    h2d.wait_event(x_free[j])
                    xds[j].copy_(xh, non_blocking=True)
                    x_ready[j].record(h2d)
                comp.wait_event(x_ready[j])
                comp.wait_event(o_free[j])
                m.mla_prefill(self.W, xds[j], ods[j], ws, *caches, T, None, stream=comp)
                x_free[j].record(comp)
                o_ready[j].record(comp)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(o_ready[j])
                    ohs[j].copy_(ods[j], non_blocking=True)
                    o_free[j].record(d2h)
            comp.wait_stream(d2h)
            comp.wait_stream(h2d)

        run(warmup)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        run(steps)
        t1.record(comp)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps

    # ---- prefill ----------------------------------------------------------
    def prefill_setup(self, B, T, with_cache):
        torch, m = self.torch, self.m
        x = self.synth.tensor_cuda(0, "x", (B, T, D), self.synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_PREFILL, B, T, device=self.dev)
        caches = (None,) * 4
        if with_cache:
            caches = (torch.empty((B, H, T, QK), dtype=torch.bfloat16, device=self.dev),
                      torch.empty((B, H, T, V), dtype=torch.bfloat16, device=self.dev),
                      torch.empty((B, T, KVL), dtype=torch.bfloat16, device=self.dev),
                      torch.empty((B, T, ROPE), dtype=torch.bfloat16, device=self.dev))
        return x, out, ws, caches

    def prefill_step_fn(self, x, out, ws, caches, T):
        m = self.m
        cap = T if caches[0] is not None or caches[2] is not None else 0

        def step(timing):
            m.mla_prefill(self.W, x, out, ws, *caches, cap, m.make_params(timing=timing))
        return step

    # ---- the block's MLP half ------------------------------------------------
    def ffn_weights(self):
        if getattr(self, "WF", None) is None:
            self.wft = self.synth.ffn_weights_cuda(0, device=self.dev)
            self.WF = self.m.make_ffn_weights(self.wft)
        return self.WF

    def ffn_step_fn(self, n):
        torch, m, synth = self.torch, self.m, self.synth
        WF = self.ffn_weights()
        x = synth.tensor_cuda(0, "ffn_x", (n, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_FFN, 1, n, device=self.dev)

        def step(timing):
            m.mla_ffn(WF, x, out, ws, m.make_params(timing=timing))
        return step, (x, out, ws)

    def block_step_fn(self, B, T):
        """The dense block: mla_prefill (x -> x') then mla_ffn in place."""
        torch, m = self.torch, self.m
        WF = self.ffn_weights()
        x, mid, ws, caches = self.prefill_setup(B, T, with_cache=False)
        wsf = m.alloc_workspace(m.MODE_FFN, B, T, device=self.dev)

        def step(timing):
            m.mla_prefill(self.W, x, mid, ws, *caches, 0, m.make_params(timing=timing))
            m.mla_ffn(WF, mid, mid, wsf, m.make_params(timing=timing))
        return step, (x, mid, ws, wsf)

    def chunk_step_fn(self, B, P0, T):
        """Chunked prefill of T tokens after P0 positions already in the
        rebuilt cache (written by the library's cache-only prefill of the
        seeded 'cache_x' tokens); every step rewrites rows P0..P0+T-1."""
        torch, m, synth = self.torch, self.m, self.synth
        kc, vc = self.fill_caches(B, P0, P0 + T, rebuilt=True)
        x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_PREFILL, B, T, device=self.dev)

        def step(timing):
            m.mla_prefill_chunk(self.W, x, P0, out, kc, vc, ws, params=m.make_params(timing=timing))
        return step, (kc, vc, x, out, ws)

    def chunk_latent_step_fn(self, B, P0, T):
        """The same chunk against the latent cache (rows 0..P0-1 written by the
        library's cache-only prefill of 'cache_x'); every step rewrites latent
        rows P0..P0+T-1 and rebuilds keys and values of all P0 + T positions."""
        torch, m, synth = self.torch, self.m, self.synth
        ckv, kpe = self.fill_caches(B, P0, P0 + T, rebuilt=False)
        x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_CHUNK_LATENT, B, T, device=self.dev, cap=P0 + T)

        def step(timing):
            m.mla_prefill_chunk_latent(self.W, x, P0, out, ckv, kpe, ws, params=m.make_params(timing=timing))
        return step, (ckv, kpe, x, out, ws)

    def chunk_absorbed_step_fn(self, B, P0, T, absorbed=True):
        """T new tokens per sequence after P0 latent-cache positions, in the
        absorbed form (one latent decode row per token) or, absorbed=False,
        the rebuilt form on the same caches."""
        torch, m, synth = self.torch, self.m, self.synth
        ckv, kpe = self.fill_caches(B, P0, P0 + T, rebuilt=False)
        x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        mode = m.MODE_CHUNK_ABSORBED if absorbed else m.MODE_CHUNK_LATENT
        ws = m.alloc_workspace(mode, B, T, device=self.dev, cap=P0 + T)
        fn = m.mla_prefill_chunk_absorbed if absorbed else m.mla_prefill_chunk_latent

        def step(timing):
            fn(self.W, x, P0, out, ckv, kpe, ws, params=m.make_params(timing=timing))
        return step, (ckv, kpe, x, out, ws)

    # ---- decode -------------------------------------------------------------
    def fill_caches(self, B, P, cap, rebuilt, chunk_tokens=1 << 17):
        """Caches of positions 0..P-1 written by the library's own prefill
        (cache-only mode) from the seeded 'cache_x' tokens."""
        torch, m, synth = self.torch, self.m, self.synth
        if rebuilt:
            c1 = torch.empty((B, H, cap, QK), dtype=torch.bfloat16, device=self.dev)
            c2 = torch.empty((B, H, cap, V), dtype=torch.bfloat16, device=self.dev)
        else:
            c1 = torch.empty((B, cap, KVL), dtype=torch.bfloat16, device=self.dev)
            c2 = torch.empty((B, cap, ROPE), dtype=torch.bfloat16, device=self.dev)
        bs = max(1, min(B, chunk_tokens // max(P, 1)))
        ws = m.alloc_workspace(m.MODE_PREFILL, bs, P, device=self.dev)
        for b0 in range(0, B, bs):
            nb = min(bs, B - b0)
            xc = synth.tensor_cuda(0, "cache_x", (nb, P, D), synth.X_DIST, device=self.dev, row_offset=b0)
            if rebuilt:
                m.mla_prefill(self.W, xc, None, ws, c1[b0:b0 + nb], c2[b0:b0 + nb], None, None, cap)
            else:
                m.mla_prefill(self.W, xc, None, ws, None, None, c1[b0:b0 + nb], c2[b0:b0 + nb], cap)
        torch.cuda.synchronize()
        del ws
        return c1, c2

    def decode_varlen_step_fn(self, B, P_max, rebuilt, lengths):
        """Ragged decode: caches of P_max positions per sequence (the library's
        cache-only prefill), sequence b at position lengths[b]."""
        torch, m, synth = self.torch, self.m, self.synth
        c1, c2 = self.fill_caches(B, P_max, P_max + 1, rebuilt)
        x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        P = torch.tensor(lengths, dtype=torch.int32, device=self.dev)
        ws = m.alloc_workspace(m.MODE_DECODE if rebuilt else m.MODE_DECODE_LATENT, B, P_max, device=self.dev)
        fn = m.mla_decode_varlen if rebuilt else m.mla_decode_latent_varlen

        def step(timing):
            fn(self.W, x, P, P_max, c1, c2, out, ws, m.make_params(timing=timing))
        return step, (c1, c2, x, out, P, ws)

    def decode_folded_step_fn(self, B, P):
        """Latent decode with W_UV folded into o_proj (W_fold built once)."""
        torch, m, synth = self.torch, self.m, self.synth
        wf = torch.empty((D, H * KVL), dtype=torch.bfloat16, device=self.dev)
        m.mla_fold_wuv_into_wo(self.W, wf, m.alloc_workspace(m.MODE_FOLD, 1, 1, device=self.dev))
        c1, c2 = self.fill_caches(B, P, P + 1, False)
        x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P, device=self.dev)

        def step(timing):
            m.mla_decode_latent_folded(self.W, wf, x, P, c1, c2, out, ws, m.make_params(timing=timing))
        return step, (wf, c1, c2, x, out, ws)

    def decode_step_fn(self, B, P, rebuilt):
        torch, m, synth = self.torch, self.m, self.synth
        c1, c2 = self.fill_caches(B, P, P + 1, rebuilt)
        x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST, device=self.dev)
        out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_DECODE if rebuilt else m.MODE_DECODE_LATENT, B, P, device=self.dev)
        fn = m.mla_decode if rebuilt else m.mla_decode_latent

        def step(timing):
            fn(self.W, x, P, c1, c2, out, ws, m.make_params(timing=timing))
        return step, (c1, c2, x, out, ws)


FFN_STAGES = ("ffn_norm", "gate_up", "down")
PREFILL_STAGES = ("input_norm", "a_proj", "latent", "q_b", "kv_b", "attn", "o_proj")
DECODE_STAGES = ("input_norm", "a_proj", "latent", "q_b", "kv_b", "attn", "o_proj")
LATENT_STAGES = ("input_norm", "a_proj", "latent", "q_b", "absorb_q", "attn", "absorb_o", "o_proj")


def varlen_lengths(B, P_max):
    """Seeded per-sequence positions in [1, P_max] (the first P_max, the second 1)."""
    import numpy as np
    lengths = [int(v) for v in np.random.default_rng(7).integers(1, P_max + 1, size=B)]
    lengths[0], lengths[1] = P_max, 1
    return lengths


def roofline_entry(stage_ms, mode, B, TP, pk, config_name, past=0):
    """Roofline of the dominant stage, timed by events around it in every
    timed step."""
    if "_dominant_timed" in stage_ms:
        (name, ms), how = stage_ms["_dominant_timed"], "events around it in every timed step"
    elif "_dominant_probe" in stage_ms:
        (name, ms), how = stage_ms["_dominant_probe"], "events around every stage in a separate instrumented pass"
    else:
        return None
    total = sum(v for k, v in stage_ms.items() if not k.startswith("_"))
    kind, amount = stage_work(name, mode, B, TP, past)
    if kind == "flop":
        ach = amount / (ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"]
        return {"kernel": name, "bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": ncu_traffic(name, config_name), "ms": round(ms, 4),
                "share": round(stage_ms[name] / total, 4), "peak_source": pk["source"] + " (burst)", "timed": how}
    if kind == "byte":
        ach = amount / (ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": ncu_traffic(name, config_name), "ms": round(ms, 4),
                "share": round(stage_ms[name] / total, 4), "peak_source": pk["source"], "timed": how}
    return {"kernel": name, "bound": None, "ms": ms}


def note(summary, key):
    """One configuration's compact numbers on stderr as soon as they exist
    (stdout carries the one JSON line)."""
    print(json.dumps({key: summary[key]}), file=sys.stderr, flush=True)


def _stages_out(stage_ms):
    return {k: round(v, 4) for k, v in stage_ms.items() if not k.startswith("_")}


def cpu_oracle_prefill_sample(n_tokens):
    """The oracle (float64 numpy) on the first n_tokens of sequence 0 of the
    headline B=8, T=4096 workload (causal: those rows are the same
    computation as in the whole step), caches included; returns (tokens/s,
    seconds, threads)."""
    import synth
    from oracle import mla_oracle as om
    names = {"w_in_norm": "g_in", "w_q_a": "w_q_a", "w_q_a_norm": "g_qa", "w_q_b": "w_q_b",
             "w_kv_a": "w_kv_a", "w_kv_a_norm": "g_kva", "w_kv_b": "w_kv_b", "w_o": "w_o"}
    W = {names[n]: synth.bf16_bits_to_f64(b) for n, b in synth.weight_bits(0).items()}
    x = synth.bf16_bits_to_f64(synth.tensor_bits(0, "x", (8, 4096, D), synth.X_DIST, rows=[0]))[:, :n_tokens]
    t0 = time.perf_counter()
    om.prefill(W, x)
    dt = time.perf_counter() - t0
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return n_tokens / dt, dt, threads


def cpu_sample_text(n):
    return (f"the first {n} tokens of sequence 0 of the B=8 T=4096 prefill (causal; its caches included), "
            "float64 numpy oracle")


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return
    n = args.ref_tokens
    times = []
    for _ in range(args.warmup):
        cpu_oracle_prefill_sample(n)
    threads = os.cpu_count()
    for _ in range(args.steps):
        v, dt, threads = cpu_oracle_prefill_sample(n)
        times.append(dt)
    mean_s = statistics.mean(times)
    value = n / mean_s
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 8 * ws, "seq_len": 4096,
                       "parallelism": f"replica{ws}" if ws > 1 else "single"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": cpu_sample_text(n) + " per step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Set up one configuration, run the warm-up steps, then one step between
    cudaProfilerStart and cudaProfilerStop (nothing is timed or reported)."""
    import re
    import torch
    torch.cuda.set_device(0)
    r = Runner("cuda:0")
    keep = None
    mcl = re.fullmatch(r"chunk_latent_b(\d+)_p(\d+)_t(\d+)", args.profile)
    mc = re.fullmatch(r"chunk_b(\d+)_p(\d+)_t(\d+)", args.profile)
    mf = re.fullmatch(r"ffn_n(\d+)", args.profile)
    mt = re.fullmatch(r"(prefill|decode|latent)_b(\d+)_([tp])(\d+)(_cache)?", args.profile)
    m8 = re.fullmatch(r"decode_fp8_b(\d+)_p(\d+)", args.profile)
    if m8:
        B8, P8 = int(m8.group(1)), int(m8.group(2))
        WQ, keepw = r.m.make_weights_fp8(r.wt)
        kc, vc = r.fill_caches(B8, P8, P8 + 1, True)
        x8 = r.synth.tensor_cuda(0, "new_x", (B8, D), r.synth.X_DIST, device=r.dev)
        o8 = torch.empty_like(x8)
        ws8 = r.m.alloc_workspace(r.m.MODE_DECODE, B8, P8, device=r.dev)

        def step(timing):
            r.m.mla_decode_fp8(WQ, x8, P8, kc, vc, o8, ws8, r.m.make_params(timing=timing))
        keep = (WQ, keepw, kc, vc, x8, o8, ws8)
    elif mcl:
        step, keep = r.chunk_latent_step_fn(int(mcl.group(1)), int(mcl.group(2)), int(mcl.group(3)))
    elif mc:
        step, keep = r.chunk_step_fn(int(mc.group(1)), int(mc.group(2)), int(mc.group(3)))
    elif mf:
        step, keep = r.ffn_step_fn(int(mf.group(1)))
    elif not mt:
        raise SystemExit(f"--profile: unknown configuration {args.profile!r}")
    else:
        kind, B, n, cache = mt.group(1), int(mt.group(2)), int(mt.group(4)), bool(mt.group(5))
        if kind == "prefill":
            x, out, ws, caches = r.prefill_setup(B, n, with_cache=cache)
            step = r.prefill_step_fn(x, out, ws, caches, n)
            keep = (x, out, ws, caches)
        else:
            step, keep = r.decode_step_fn(B, n, rebuilt=(kind == "decode"))
    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    step(None)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    print(json.dumps({"profile": args.profile, "warmup": args.warmup, "ok": True}), flush=True)
    del keep


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline prefill only")
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of the headline's sequence 0 the CPU oracle baseline runs (0 = skip)")
    ap.add_argument("--ref-tokens", type=int, default=1024,
                    help="tokens of the headline's sequence 0 each step of --impl reference runs")
    ap.add_argument("--profile", default=None,
                    help="run one step of one configuration for a profiler and exit: prefill_bB_tT[_cache], "
                         "decode_fp8_bB_pP (FP8 weights), "
                         "chunk_bB_pP0_tT / chunk_latent_bB_pP0_tT (chunked prefill on either cache), ffn_nN (MLP half, N rows), "
                         "decode_bB_pP (rebuilt cache) or latent_bB_pP; only that step lies between "
                         "cudaProfilerStart/Stop (ncu --profile-from-start off)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)

    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier_max(v):
        return reduce_max(v, dev)

    pk = peaks()
    r = Runner(dev)
    K, W = args.steps, max(args.warmup, 3)
    summary = {}

    # ---- headline: prefill B=8, T=4096 writing both caches -----------------------
    B, T = 8, 4096
    x, out, ws, caches = r.prefill_setup(B, T, with_cache=True)
    step = r.prefill_step_fn(x, out, ws, caches, T)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        ms, stage_ms, launches = r.time_steps(step, K, W, stages=PREFILL_STAGES)
        wall = time.perf_counter() - wall0
    ms_step = barrier_max(statistics.mean(ms))
    tok = B * T
    value = weak_scaling_value(tok, world, ms_step)
    flops = tok * proj_flops_per_token() + prefill_attn_flops(B, T)
    roof = roofline_entry(stage_ms, "prefill", B, T, pk, "prefill_b8_t4096")

    # end to end: pinned host x -> device, the call (caches stay resident in
    # HBM as a serving engine keeps them), device -> pinned host out; the
    # copies of neighbouring steps overlap the call on their own streams
    e2e_ms = barrier_max(r.time_e2e_pipelined(x, out, ws, caches, B, T, K, W))
    tf = flops / (ms_step * 1e-3) / 1e12
    summary["C5"] = {"cfg": "prefill B=8 T=4096 +caches", "ms": round(ms_step, 4), "tok_s": round(value, 1),
                     "tflops": round(tf, 1), "frac_bf16": round(tf / pk["bf16_tflops"], 4),
                     "e2e_tok_s": round(world * tok / (e2e_ms * 1e-3), 1)}
    note(summary, "C5")

    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded splitmix64 / Box-Muller N(0,1) inputs, N(0,0.02) weights)",
            "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": T,
                       "parallelism": f"replica{world}" if world > 1 else "single",
                       "l2": "inputs (470 MB) larger than L2, and L2 flushed between timed steps "
                             "(512 MB written, then read back)"},
            "tflops": round(tf, 2), "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4),
            "stage_ms": _stages_out(stage_ms),
            "roofline": roof, "gpu_launches": launches * K,
            "stage_ms_note": "per-stage times from a separate instrumented pass (events around every stage)",
            "e2e": {"value": round(world * tok / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
                    "ms_per_step": round(e2e_ms, 4),
                    "how": "pinned host x copied in and out copied back every step, on their own streams "
                           "with two device buffers each, so step i's call overlaps the copies of steps "
                           "i - 1 and i + 1"},
            "clocks": clk.summary(), "wall_s_timed": round(wall, 3)}
    del x, out, ws, caches
    torch.cuda.empty_cache()

    launches_c2 = 0
    if not args.quick:
        ks = max(3, min(K, 10))
        # ---- decode, rebuilt per-head cache: B=64, P=1000 ----------------------
        try:
            B3, P3 = 64, 1000
            step3, keep = r.decode_step_fn(B3, P3, rebuilt=True)
            ms3, st3, l3 = r.time_steps(step3, ks, W, stages=DECODE_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms3)) * 1e3
            byts = B3 * H * (P3 + 1) * (QK + V) * 2 + WEIGHT_BYTES + 2 * B3 * D * 2
            line["decode_rebuilt"] = {
                "workload": "mla_decode B=64 P=1000 (L=1001 keys), rebuilt bf16 K/V cache",
                "us_per_step": round(us, 2), "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_8tbs": round(byts / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "stage_ms": _stages_out(st3),
                "roofline": roofline_entry(st3, "decode", B3, P3, pk, "decode_b64_p1000"), "launches": l3}
            summary["C3"] = {"cfg": "decode B=64 P=1000 rebuilt", "us": round(us, 2),
                             "hbm_gbs": line["decode_rebuilt"]["hbm_gbs"],
                             "frac_8tbs": line["decode_rebuilt"]["frac_8tbs"],
                             "attn_frac_measured": (line["decode_rebuilt"]["roofline"] or {}).get("frac")}
            note(summary, "C3")
            del step3, keep
            torch.cuda.empty_cache()
        except Exception as e:  # report, keep the headline
            line["decode_rebuilt"] = {"error": repr(e)[:300]}
        # ---- decode, latent cache: B=128, P=8192 ---------------------------------
        try:
            B4, P4 = 128, 8192
            step4, keep = r.decode_step_fn(B4, P4, rebuilt=False)
            ms4, st4, l4 = r.time_steps(step4, ks, W, stages=LATENT_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms4)) * 1e3
            byts = B4 * (P4 + 1) * (KVL + ROPE) * 2 + WEIGHT_BYTES + 2 * B4 * D * 2
            line["decode_latent"] = {
                "workload": "mla_decode_latent B=128 P=8192, 576-value latent cache, W_UK/W_UV absorbed",
                "us_per_step": round(us, 2), "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_8tbs": round(byts / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "stage_ms": _stages_out(st4),
                "roofline": roofline_entry(st4, "latent", B4, P4, pk, "latent_b128_p8192"), "launches": l4}
            summary["C4"] = {"cfg": "decode B=128 P=8192 latent", "us": round(us, 2),
                             "hbm_gbs": line["decode_latent"]["hbm_gbs"],
                             "frac_8tbs": line["decode_latent"]["frac_8tbs"],
                             "attn_frac_measured": (line["decode_latent"]["roofline"] or {}).get("frac")}
            note(summary, "C4")
            del step4, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["decode_latent"] = {"error": repr(e)[:300]}
        # ---- latent decode with W_UV folded into o_proj: B=128, P=8192 -----------
        try:
            B4, P4 = 128, 8192
            step4f, keep = r.decode_folded_step_fn(B4, P4)
            ms4f, st4f, l4f = r.time_steps(step4f, ks, W, stages=LATENT_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms4f)) * 1e3
            wbytes = WEIGHT_BYTES - 2 * (7168 * 8192 + 64 * 128 * 512) + 2 * 7168 * 64 * 512
            byts = B4 * (P4 + 1) * (KVL + ROPE) * 2 + wbytes + 2 * B4 * D * 2
            line["decode_latent_folded"] = {
                "workload": "mla_decode_latent_folded B=128 P=8192: W_UV folded into o_proj (470 MB W_fold "
                            "in place of 125 MB of W_UV and W_o)",
                "us_per_step": round(us, 2), "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "stage_ms": _stages_out(st4f), "launches": l4f}
            del step4f, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["decode_latent_folded"] = {"error": repr(e)[:300]}
        # ---- decode with FP8 block-scaled weights: B=64, P=1000 -------------------
        try:
            B3, P3 = 64, 1000
            WQ, keepw = r.m.make_weights_fp8(r.wt)
            kc, vc = r.fill_caches(B3, P3, P3 + 1, True)
            x3 = r.synth.tensor_cuda(0, "new_x", (B3, D), r.synth.X_DIST, device=r.dev)
            o3 = torch.empty_like(x3)
            ws3 = r.m.alloc_workspace(r.m.MODE_DECODE, B3, P3, device=r.dev)

            def step3f(timing):
                r.m.mla_decode_fp8(WQ, x3, P3, kc, vc, o3, ws3, r.m.make_params(timing=timing))
            ms3f, st3f, l3f = r.time_steps(step3f, ks, W, stages=DECODE_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms3f)) * 1e3
            wbytes = sum(t.numel() * t.element_size() for t in keepw.values())
            byts = B3 * H * (P3 + 1) * (QK + V) * 2 + wbytes + 2 * B3 * D * 2
            line["decode_rebuilt_fp8"] = {
                "workload": "mla_decode_fp8 B=64 P=1000, E4M3 weights with power-of-two 128x128 block scales",
                "us_per_step": round(us, 2), "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "weight_bytes": wbytes, "stage_ms": _stages_out(st3f), "launches": l3f}
            summary["C3_fp8"] = {"cfg": "decode B=64 P=1000 rebuilt, FP8 weights", "us": round(us, 2),
                                 "o_proj_us": round(st3f.get("o_proj", 0.0) * 1e3, 1)}
            note(summary, "C3_fp8")
            del WQ, keepw, kc, vc, x3, o3, ws3
            torch.cuda.empty_cache()
        except Exception as e:
            line["decode_rebuilt_fp8"] = {"error": repr(e)[:300]}
        # ---- ragged latent decode: 128 sequences, positions in [1, 8192] ---------
        try:
            B4v, P4v = 128, 8192
            lengths = varlen_lengths(B4v, P4v)
            step4v, keep = r.decode_varlen_step_fn(B4v, P4v, False, lengths)
            ms4v, st4v, l4v = r.time_steps(step4v, ks, W, stages=LATENT_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms4v)) * 1e3
            keys = sum(p + 1 for p in lengths)
            byts = keys * (KVL + ROPE) * 2 + WEIGHT_BYTES + 2 * B4v * D * 2
            line["decode_latent_ragged"] = {
                "workload": f"mla_decode_latent_varlen B=128, seeded positions in [1, 8192] ({keys} keys in all)",
                "us_per_step": round(us, 2), "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_8tbs": round(byts / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "stage_ms": _stages_out(st4v), "launches": l4v}
            del step4v, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["decode_latent_ragged"] = {"error": repr(e)[:300]}
        # ---- prefill B=1, T=2048 (no caches) ------------------------------------------
        try:
            B2, T2 = 1, 2048
            x2, out2, ws2, c2 = r.prefill_setup(B2, T2, with_cache=False)
            step2 = r.prefill_step_fn(x2, out2, ws2, c2, T2)
            ms2, st2, l2 = r.time_steps(step2, ks, W, stages=PREFILL_STAGES, dominant_events=False)
            launches_c2 = l2
            ms2 = barrier_max(statistics.mean(ms2))
            fl2 = B2 * T2 * proj_flops_per_token() + prefill_attn_flops(B2, T2)
            tf2 = fl2 / (ms2 * 1e-3) / 1e12
            line["prefill_b1_t2048"] = {
                "workload": "mla_prefill B=1 T=2048 causal (no caches)",
                "ms_per_step": round(ms2, 4), "tokens_per_s": round(world * B2 * T2 / (ms2 * 1e-3), 1),
                "tflops": round(tf2, 2), "frac_bf16_peak": round(tf2 / pk["bf16_tflops"], 4),
                "stage_ms": _stages_out(st2),
                "roofline": roofline_entry(st2, "prefill", B2, T2, pk, "prefill_b1_t2048"), "launches": l2}
            summary["C2"] = {"cfg": "prefill B=1 T=2048", "ms": round(ms2, 4),
                             "tok_s": line["prefill_b1_t2048"]["tokens_per_s"], "tflops": round(tf2, 1),
                             "frac_bf16": round(tf2 / pk["bf16_tflops"], 4),
                             "attn_ms": round(st2.get("attn", 0.0), 4)}
            note(summary, "C2")
            del x2, out2, ws2, c2
            torch.cuda.empty_cache()
        except Exception as e:
            line["prefill_b1_t2048"] = {"error": repr(e)[:300]}
        # ---- prefill B=1, T=16: the weights stream once (HBM-bound) --------------------
        try:
            B1, T1 = 1, 16
            x1, out1, ws1, c1 = r.prefill_setup(B1, T1, with_cache=False)
            step1 = r.prefill_step_fn(x1, out1, ws1, c1, T1)
            ms1, st1, l1 = r.time_steps(step1, max(ks, 10), W, stages=PREFILL_STAGES, dominant_events=False)
            us1 = barrier_max(statistics.mean(ms1)) * 1e3
            fl1 = B1 * T1 * proj_flops_per_token() + prefill_attn_flops(B1, T1)
            by1 = WEIGHT_BYTES + 2 * B1 * T1 * D * 2
            gbs1 = by1 / (us1 * 1e-6) / 1e9
            tf1 = fl1 / (us1 * 1e-6) / 1e12
            line["prefill_b1_t16"] = {
                "workload": "mla_prefill B=1 T=16 causal (no caches): every weight byte read once for 16 tokens",
                "us_per_step": round(us1, 2), "tokens_per_s": round(world * B1 * T1 / (us1 * 1e-6), 1),
                "hbm_gbs": round(gbs1, 1), "frac_8tbs": round(gbs1 / NOMINAL_HBM_GBS, 4),
                "frac_measured_hbm": round(gbs1 / pk["hbm_gbs"], 4), "algorithmic_bytes": by1,
                "tflops": round(tf1, 2), "frac_bf16_peak": round(tf1 / pk["bf16_tflops"], 4),
                "frac_bf16_peak_note": "meaningless here: 16 flop per weight byte, the step is bound by HBM",
                "stage_ms": _stages_out(st1), "launches": l1}
            summary["C1"] = {"cfg": "prefill B=1 T=16", "us": round(us1, 2),
                             "tok_s": line["prefill_b1_t16"]["tokens_per_s"], "hbm_gbs": round(gbs1, 1),
                             "frac_8tbs": round(gbs1 / NOMINAL_HBM_GBS, 4),
                             "frac_bf16": round(tf1 / pk["bf16_tflops"], 4), "tc_note": "meaningless (HBM-bound)"}
            note(summary, "C1")
            del x1, out1, ws1, c1
            torch.cuda.empty_cache()
        except Exception as e:
            line["prefill_b1_t16"] = {"error": repr(e)[:300]}
        # ---- chunked prefill: B=1, 2048 tokens after 2048 cached positions ----------
        try:
            B6, P6, T6 = 1, 2048, 2048
            step6, keep = r.chunk_step_fn(B6, P6, T6)
            ms6, st6, l6 = r.time_steps(step6, ks, W, stages=PREFILL_STAGES, dominant_events=False)
            ms6 = barrier_max(statistics.mean(ms6))
            fl6 = B6 * T6 * proj_flops_per_token() + prefill_attn_flops(B6, T6, P6)
            line["prefill_chunk"] = {
                "workload": "mla_prefill_chunk B=1 T=2048 after P0=2048 cached positions (rebuilt K/V cache)",
                "ms_per_step": round(ms6, 4), "tokens_per_s": round(world * B6 * T6 / (ms6 * 1e-3), 1),
                "tflops": round(fl6 / (ms6 * 1e-3) / 1e12, 2),
                "frac_bf16_peak": round(fl6 / (ms6 * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "stage_ms": _stages_out(st6),
                "roofline": roofline_entry(st6, "prefill", B6, T6, pk, "chunk_b1_p2048_t2048", past=P6),
                "launches": l6}
            del step6, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["prefill_chunk"] = {"error": repr(e)[:300]}
        try:
            B6, P6, T6 = 1, 2048, 2048
            step6, keep = r.chunk_latent_step_fn(B6, P6, T6)
            ms6, st6, l6 = r.time_steps(step6, ks, W, stages=PREFILL_STAGES, dominant_events=False)
            ms6 = barrier_max(statistics.mean(ms6))
            # algorithmic work as the chunk on the rebuilt cache, plus the kv_b
            # rebuild of the P0 cached positions
            fl6 = (B6 * T6 * proj_flops_per_token() + prefill_attn_flops(B6, T6, P6)
                   + B6 * P6 * 2 * KVL * H * (NOPE + V))
            line["prefill_chunk_latent"] = {
                "workload": "mla_prefill_chunk_latent B=1 T=2048 after P0=2048 positions in the 576-value latent cache",
                "ms_per_step": round(ms6, 4), "tokens_per_s": round(world * B6 * T6 / (ms6 * 1e-3), 1),
                "tflops": round(fl6 / (ms6 * 1e-3) / 1e12, 2),
                "frac_bf16_peak": round(fl6 / (ms6 * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "stage_ms": _stages_out(st6),
                "roofline": roofline_entry(st6, "prefill", B6, T6, pk, "chunk_latent_b1_p2048_t2048", past=P6),
                "launches": l6}
            del step6, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["prefill_chunk_latent"] = {"error": repr(e)[:300]}
        # ---- absorbed chunk: 32 sequences, 4 new tokens after 8188 latent positions ---
        try:
            B8, P8, T8 = 32, 8188, 4
            step8, keep = r.chunk_absorbed_step_fn(B8, P8, T8)
            ms8, st8, l8 = r.time_steps(step8, ks, W, stages=LATENT_STAGES, dominant_events=False)
            us = barrier_max(statistics.mean(ms8)) * 1e3
            keys = B8 * sum(P8 + t + 1 for t in range(T8))
            byts = keys * (KVL + ROPE) * 2 + WEIGHT_BYTES + 2 * B8 * T8 * D * 2
            del step8, keep
            torch.cuda.empty_cache()
            step8r, keep = r.chunk_absorbed_step_fn(B8, P8, T8, absorbed=False)
            ms8r, _, _ = r.time_steps(step8r, max(2, min(ks, 5)), 2, with_stages=False, dominant_events=False)
            us_r = barrier_max(statistics.mean(ms8r)) * 1e3
            del step8r, keep
            torch.cuda.empty_cache()
            line["prefill_chunk_absorbed"] = {
                "workload": "mla_prefill_chunk_absorbed B=32 T=4 after P0=8188 latent-cache positions "
                            "(one latent decode row per new token)",
                "us_per_step": round(us, 2), "tokens_per_s": round(world * B8 * T8 / (us * 1e-6), 1),
                "hbm_gbs": round(byts / (us * 1e-6) / 1e9, 1),
                "frac_measured_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": byts, "stage_ms": _stages_out(st8), "launches": l8,
                "rebuilt_form_us_per_step": round(us_r, 1)}
        except Exception as e:
            line["prefill_chunk_absorbed"] = {"error": repr(e)[:300]}
        # ---- the block's MLP half: 2048 rows (prefill) and 64 rows (decode) ---------
        l_ffn = 0
        try:
            n7 = 2048
            step7, keep = r.ffn_step_fn(n7)
            ms7, st7, l_ffn = r.time_steps(step7, ks, W, stages=FFN_STAGES, dominant_events=False)
            ms7 = barrier_max(statistics.mean(ms7))
            fl7 = 3 * 2 * n7 * D * FFN_I
            line["ffn_prefill"] = {
                "workload": "mla_ffn 2048 rows (post-attention RMSNorm + SwiGLU MLP, I=18432, + residual)",
                "ms_per_step": round(ms7, 4), "tokens_per_s": round(world * n7 / (ms7 * 1e-3), 1),
                "tflops": round(fl7 / (ms7 * 1e-3) / 1e12, 2),
                "frac_bf16_peak": round(fl7 / (ms7 * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "stage_ms": _stages_out(st7),
                "roofline": roofline_entry(st7, "ffn", 1, n7, pk, "ffn_n2048"), "launches": l_ffn}
            del step7, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["ffn_prefill"] = {"error": repr(e)[:300]}
        try:
            n8 = 64
            step8, keep = r.ffn_step_fn(n8)
            ms8, st8, l8 = r.time_steps(step8, ks, W, stages=FFN_STAGES, dominant_events=False)
            us8 = barrier_max(statistics.mean(ms8)) * 1e3
            by8 = FFN_WEIGHT_BYTES + 2 * n8 * D * 2
            line["ffn_decode"] = {
                "workload": "mla_ffn 64 rows (one decode step of 64 sequences): the 793 MB of MLP weights stream once",
                "us_per_step": round(us8, 2), "hbm_gbs": round(by8 / (us8 * 1e-6) / 1e9, 1),
                "frac_measured_hbm": round(by8 / (us8 * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes": by8, "stage_ms": _stages_out(st8),
                "roofline": roofline_entry(st8, "ffn_dec", 1, n8, pk, "ffn_n64"), "launches": l8}
            del step8, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["ffn_decode"] = {"error": repr(e)[:300]}
        # ---- the whole dense block: prefill B=1 T=2048 then the MLP half ----------
        try:
            B9, T9 = 1, 2048
            step9, keep = r.block_step_fn(B9, T9)
            ms9, st9, _ = r.time_steps(step9, ks, W, stages=PREFILL_STAGES + FFN_STAGES,
                                       dominant_events=False)
            ms9 = barrier_max(statistics.mean(ms9))
            fl9 = (B9 * T9 * proj_flops_per_token() + prefill_attn_flops(B9, T9)
                   + 3 * 2 * B9 * T9 * D * FFN_I)
            line["dense_block_prefill"] = {
                "workload": "dense block B=1 T=2048: mla_prefill (causal MLA + residual) then mla_ffn (in place)",
                "ms_per_step": round(ms9, 4), "tokens_per_s": round(world * B9 * T9 / (ms9 * 1e-3), 1),
                "tflops": round(fl9 / (ms9 * 1e-3) / 1e12, 2),
                "frac_bf16_peak": round(fl9 / (ms9 * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                "stage_ms": _stages_out(st9), "launches": launches_c2 + l_ffn}
            del step9, keep
            torch.cuda.empty_cache()
        except Exception as e:
            line["dense_block_prefill"] = {"error": repr(e)[:300]}

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----------------------------------
    if world == 1 and args.cpu_tokens > 0:
        v, dt, threads = cpu_oracle_prefill_sample(args.cpu_tokens)
        line["cpu_baseline"] = {"value": round(v, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": cpu_sample_text(args.cpu_tokens) + f", {dt:.1f} s"}
    # the per-configuration numbers again, compact, at the end of the line
    line["summary"] = summary
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
