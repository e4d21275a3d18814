#!/usr/bin/env python3
"""Throughput of the per-layer inner denoising step of block-wise
diffusion-LLM decoding on GB300.

One step = one pass of the whole hot path for one layer: the fused RMSNorm +
QKV projection + RoPE + paged K/V write of the block rows, the block
attention over [prefix | block | suffix], and the FACache merge of every
invariant row.  The metric is block-query tokens per second per layer-step
(block rows of all sequences / time of one layer-step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config stack|ragged|long|llada_single|tiny]

Headline workload: the LLaDA-8B-shaped 32-layer attention stack (16
sequences, prompt 1024, gen 512, block 32, d_model 4096, 32 heads x 128,
RoPE theta 5e5), every layer with its own weights, paged cache and block
rows: the timed steps walk the 32 layers in order, round after round (the
metric is the mean over the layers).  Synthetic seeded bf16 inputs drawn on
the device (N(0, 1) rows, N(0, 0.02) weights); each layer holds ~1.5 GB, so
no step finds its inputs in the 129 MB L2.  The other LLaDA-shaped workloads
(single layer, long context, ragged batch) are measured the same way on 4
layer instances each and reported under "configs".

Timing: CUDA graphs of 32 layer-steps (two kernels a step, chained by
programmatic dependent launch), replayed back to back between CUDA events on
the launching stream.  Inside the timed region one round of layer-steps in
every 16 (always the first) is replayed call by call with events around each
kernel: those give each kernel's duration for the roofline objects.  The
end-to-end figure calls the public step API with the block rows copied in
from pinned host memory and the block rows' outputs read back to pinned host
memory every step (the read-back on a copy stream, under the next step).

Under torchrun (N > 1) every rank runs its own replica of the workload
(sequences are independent units: weak scaling, no collective on the data
path); the time is the max over ranks.

--impl reference times the fp64 CPU oracle (full recompute of the step, all
heads) on the host cores, one sequence of the workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "stack"
SECONDARY = ("llada_single", "long", "ragged", "llada_single_prefix_only")
METRIC = "block-query tokens/s per layer-step"
UNIT = "tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x: float, ws: int) -> float:
    if ws <= 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}




# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of a
# kernel on a workload, from one ncu capture (summarised under profiles/),
# with the hash of the kernel's sources at capture time: the figure is
# reported only while the sources still hash the same (else null).
KERNEL_SOURCES = {
    "qkv": ("qkv_gemm.cu", "qkv_wide.cu", "norm.cuh", "sm103.cuh", "kernels.cuh", "tmap.cuh"),
    "attention": ("attn_stream.cu", "attn_common.cuh", "sm103.cuh", "kernels.cuh", "tmap.cuh"),
    "lm_head": ("lm_head.cu", "norm.cuh", "sm103.cuh", "kernels.cuh", "tmap.cuh"),
}
TRAFFIC = {
    # (workload, kernel): (DRAM bytes per launch, sources hash); profiles/attn_stream_stack.md,
    # profiles/qkv_wide_stack.md (the DRAM-only capture listed there)
    ("stack", "attention"): (969_189_632, "47432f11b3637cc5"),
    ("stack", "qkv"): (135_171_584, "042ebfe49b5f9368"),
}


def sources_hash(kernel: str) -> str:
    """Hash of the kernel's sources without comments and blank lines: a change of the code
    (not of its comments) makes the recorded DRAM traffic stale."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_wise_kv_gb300", "csrc", f), encoding="utf-8") as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code.strip():
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def traffic_of(workload: str, kernel: str):
    t = TRAFFIC.get((workload, kernel))
    return t[0] if t is not None and t[1] == sources_hash(kernel) else None


def step_bytes_flops(cfg, st):
    """Algorithmic bytes and flops of one layer-step (what the method must
    move and compute), per part: the projection (a1-a4), the block attention
    (a5) and the FACache merge (a6)."""
    D, H, d = cfg.d_model, cfg.n_heads, cfg.head_dim
    HD = H * d
    lay = st.batch.host
    M = int(lay["block_len"].sum())
    N = lay["seq_len"].astype(np.int64)
    B = lay["block_len"].astype(np.int64)
    NU = N - B
    qkv_bytes = 3 * HD * D * 2 + M * D * 2 + 3 * M * HD * 2
    qkv_flops = 6 * M * D * HD
    att_bytes = int((N * HD * 4).sum()) + 2 * M * HD * 2
    att_flops = int((4 * B * N * HD).sum())
    mrg_bytes = int((NU * HD * 6).sum()) + int(NU.sum()) * H * 8  # q, out (bf16), O~/l (fp16); m, l (fp32)
    mrg_flops = int((4 * NU * B * HD).sum())
    return dict(qkv=(qkv_bytes, qkv_flops), attention=(att_bytes, att_flops), merge=(mrg_bytes, mrg_flops))


def describe(cfg, layers: int) -> str:
    """The workload, named by what it is with its sizes."""
    N = np.array([cfg.seq_len(b) for b in range(cfg.batch)], dtype=np.int64)
    M = int(sum(cfg.block))
    seqs = f"batch {cfg.batch}"
    if len(set(cfg.t_prefix)) == 1 and len(set(cfg.gen_len)) == 1 and len(set(cfg.block)) == 1:
        seqs += f", prompt {cfg.t_prefix[0]}, gen {cfg.gen_len[0]}, block {cfg.block[0]}"
    else:
        seqs += f", prompt {min(cfg.t_prefix)}..{max(cfg.t_prefix)}, gen {sorted(set(cfg.gen_len))}, " \
                f"block {sorted(set(cfg.block))}"
    what = f"{cfg.layers}-layer attention stack, layer-steps over all {layers} layers" if cfg.layers > 1 else \
        f"1 layer step ({layers} independent layer instances rotated)"
    return (f"{cfg.name}: {what}, d_model {cfg.d_model}, {cfg.n_heads}x{cfg.head_dim} heads, {seqs} "
            f"(M={M} block rows, N={int(N.sum())} rows)")


def kernel_roofline(name, bytes_, flops, seconds, hbm, tflops_peak, workload, kernel_id):
    """Roofline object of one kernel: bound by HBM or by the tensor pipe,
    whichever gives the longer time at the measured peaks."""
    t_hbm = bytes_ / (hbm * 1e9)
    t_tc = flops / (tflops_peak * 1e12)
    if t_tc > t_hbm:
        achieved = flops / seconds / 1e12
        obj = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 1), "peak": tflops_peak,
               "unit": "TFLOP/s", "frac": round(achieved / tflops_peak, 4), "algorithmic_flops": flops}
    else:
        achieved = bytes_ / seconds / 1e9
        obj = {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
               "frac": round(achieved / hbm, 4)}
    obj["traffic"] = traffic_of(workload, kernel_id)
    obj["algorithmic_bytes"] = bytes_
    obj["t_roof_us"] = round(max(t_hbm, t_tc) * 1e6, 2)
    obj["frac_of_roofline"] = round(max(t_hbm, t_tc) / seconds, 4)
    obj["duration_us"] = round(seconds * 1e6, 2)
    return obj


class Instances:
    """L independent layer instances of a workload (weights, paged cache after
    the block boundary, block rows of one inner step), inputs drawn on the
    device."""

    def __init__(self, cfg, L, dev, seed):
        from block_wise_kv_gb300.inputs import Workload
        from block_wise_kv_gb300.step import LayerStep

        self.cfg = cfg
        wl = Workload(cfg.with_(seed=seed))
        blocks = cfg.block_index
        self.items = []
        for layer in range(L):
            W, g = wl.weights_device(layer, dev)
            st = LayerStep(cfg, layer=layer, weights=(W, g), device=dev)
            del W
            x_full, x_blk = wl.batch_rows_device(layer, 1, blocks, dev)
            st.boundary(x_full)
            self.items.append((st, x_blk, x_full))
        torch.cuda.synchronize()
        for st, _, _ in self.items:
            assert st.batch.error_bits() == 0, "device-side error during the block boundary"

    def __len__(self):
        return len(self.items)


def measure(cfg, L, K, W, P, sample_every, dev, rank, ws, extras=True, e2e_steps=0):
    """Time K layer-steps of workload `cfg` over L layer instances (max over
    ranks), with per-kernel durations sampled inside the timed region; with
    `extras`, also each call alone in steady state, the block-rows-only
    variant, the block boundary, and (e2e_steps > 0) the end-to-end figure."""
    inst = Instances(cfg, L, dev, seed=rank)
    items = inst.items
    M = items[0][0].batch.total_block_rows
    P = max(1, P)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for st, xb, _ in items:
            st.step(xb, stream=stream)
        stream.synchronize()
        # a round: one step of every instance (the projection call, then the block
        # attention and the FACache merge in one launch); a pass: P rounds in one graph
        g_round = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_round, stream=stream):
            for st, xb, _ in items:
                st.step(xb, stream=stream)
        if P > 1:
            g_pass = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_pass, stream=stream):
                for _ in range(P):
                    for st, xb, _ in items:
                        st.step(xb, stream=stream)
        else:
            g_pass = g_round
        g_step, g_qkv, g_att = [], [], []  # per instance: one step; the projection call; the attention call
        for st, xb, _ in items:
            for lst, fn in ((g_step, lambda: st.step(xb, stream=stream)), (g_qkv, lambda: st.qkv(xb, stream=stream)),
                            (g_att, lambda: st.step_attention(stream))):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                lst.append(g)
    torch.cuda.synchronize()

    for i in range(W):
        g_step[i % L].replay()
    torch.cuda.synchronize()
    n_rounds, tail = divmod(K, L)
    n_passes, tail_rounds = divmod(n_rounds, P)
    samples = []

    def call_by_call(j):  # one step of instance j, each kernel between events
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        g_qkv[j].replay()
        e[1].record(stream)
        g_att[j].replay()
        e[2].record(stream)
        samples.append(e)

    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks, torch.cuda.stream(stream):
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        torch.cuda.nvtx.range_push("timed")  # profilers can select the timed launches
        t_start.record(stream)
        for k in range(n_passes):
            if k % sample_every == 0:  # the first round of this pass call by call
                for j in range(L):
                    call_by_call(j)
                for _ in range(P - 1):
                    g_round.replay()
            else:
                g_pass.replay()
        for r in range(tail_rounds):
            if not samples and r == 0:
                for j in range(L):
                    call_by_call(j)
            else:
                g_round.replay()
        for j in range(tail):
            if not samples:
                call_by_call(j)
            else:
                g_step[j].replay()
        t_end.record(stream)
        torch.cuda.nvtx.range_pop()
        stream.synchronize()
        t1 = time.perf_counter()
    torch.cuda.synchronize()
    _barrier(ws)
    total_ms = _max_over_ranks(t_start.elapsed_time(t_end), ws)
    qkv_ms = _max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in samples) / len(samples), ws)
    att_ms = _max_over_ranks(sum(e[1].elapsed_time(e[2]) for e in samples) / len(samples), ws)
    for st, _, _ in items:
        assert st.batch.error_bits() == 0, "device-side error during the timed steps"
    res = {"cfg": cfg, "L": L, "M": M, "st": items[0][0], "K": K, "total_ms": total_ms, "qkv_ms": qkv_ms,
           "att_ms": att_ms, "n_samples": len(samples), "clocks": clocks.summary(), "host_wall_s": t1 - t0,
           "P": P, "sample_every": sample_every}
    if not extras:
        return res

    # each call alone in steady state: a graph of P rounds of one call kind, so
    # consecutive launches of the same kernel overlap as in the step's graphs
    steady = {}
    n_rep = max(2, min(50, (K // (P * L)) or 2))
    with torch.cuda.stream(stream):
        for name, call in (("qkv_rope_write", lambda st, xb: st.qkv(xb, stream=stream)),
                           ("step_attention", lambda st, xb: st.step_attention(stream)),
                           ("block_rows_only", lambda st, xb: (st.qkv(xb, stream=stream), st.attention(stream)))):
            g_one = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_one, stream=stream):
                for _ in range(P):
                    for st, xb, _ in items:
                        call(st, xb)
            for _ in range(2):
                g_one.replay()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(n_rep):
                g_one.replay()
            s1.record(stream)
            s1.synchronize()
            steady[name] = _max_over_ranks(s0.elapsed_time(s1) / (n_rep * P * L), ws)
            del g_one
    res["steady_ms"] = steady

    # the block boundary (cache build: projection of every row, FACache state over
    # U x U), timed apart: once per block, amortised over the block's inner steps
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nb = max(2, min(2 * L, 16))
    b0.record()
    for i in range(nb):
        st, _, x_full = items[i % L]
        st.boundary(x_full)
    b1.record()
    torch.cuda.synchronize()
    res["build_ms"] = _max_over_ranks(b0.elapsed_time(b1) / nb, ws)
    for st, _, _ in items:
        assert st.batch.error_bits() == 0, "device-side error in the block boundary"

    if extras:
        adv = time_advances(cfg, dev, ws)
        if adv is not None:
            res["advance_ms"], res["advances"] = adv
        res["lm_head_ms"] = time_lm_head(cfg, items[0][0], dev, ws)
        res["ffn_ms"] = time_ffn(cfg, items[0][0], dev, ws)

    if e2e_steps > 0:
        res["e2e"] = e2e(items, min(K, e2e_steps), W, ws)
    del g_round, g_pass, g_step, g_qkv, g_att
    return res


def time_advances(cfg, dev, ws, max_adv: int = 8):
    """Mean time of the incremental block boundary (dllm_cache_advance) over a
    sweep of up to max_adv consecutive blocks on one layer instance (prefix
    state pools on), every call timed with events on its stream; None when a
    sequence has no block left to advance to.  Layouts, workspaces and the
    decoded rows are prepared before the timed calls."""
    from block_wise_kv_gb300 import dllm
    from block_wise_kv_gb300.inputs import Workload, layout
    from block_wise_kv_gb300.step import LayerStep

    n_adv = min([max_adv] + [cfg.num_blocks(b) - 1 - cfg.block_index[b] for b in range(cfg.batch)])
    if n_adv < 1:
        return None
    wl = Workload(cfg)
    W, g = wl.weights_device(0, dev)
    st = LayerStep(cfg, layer=0, weights=(W, g), device=dev, pre=True)
    del W
    x_full, _ = wl.batch_rows_device(0, 1, cfg.block_index, dev)
    plan = []
    k_of = list(cfg.block_index)
    prev = st.batch
    for _ in range(n_adv):
        k_of = [k + 1 for k in k_of]
        lay = layout(cfg, k_of)
        new = dllm.BatchLayout(lay["block_table"], lay["seq_len"], lay["block_start"], lay["block_len"], device=dev)
        dec_start = prev.host["block_start"]
        dec = new.with_blocks(dec_start, lay["block_start"] - dec_start)
        wsb = dllm.workspace(dllm.dllm_workspace_size(st.desc, dec.c, dllm.DLLM_OP_CACHE_ADVANCE), dev)
        x_dec = torch.randn(dec.total_block_rows, cfg.d_model, device=dev).to(torch.bfloat16)
        plan.append((new, dec, wsb, x_dec))
        prev = new
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(2):  # the second sweep is timed (the first warms up)
        st.boundary(x_full)
        torch.cuda.synchronize()
        times = []
        for new, dec, wsb, x_dec in plan:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dllm.dllm_cache_advance(st.desc, new.c, dec.c, x_dec, st.gain, st.w_qkv, st.rope, st.rope_max_pos,
                                    st.cache.c, wsb, stream)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
    assert all(new.error_bits() == 0 for new, _, _, _ in plan), "device-side error in the incremental boundary"
    ms = statistics.mean(a.elapsed_time(b) for a, b in times)
    return _max_over_ranks(ms, ws), n_adv


LM_VOCAB = 126464  # the LLaDA-8B vocabulary size (the LM head's weights are synthetic)


def time_lm_head(cfg, st, dev, ws, reps: int = 10):
    """Event-timed dllm_block_lm_head (the block-only epilogue after the layer stack) on the
    workload's block rows with a synthetic LM head of LM_VOCAB entries: mean of `reps`
    calls after a warm-up call, each call timed with events on its stream."""
    from block_wise_kv_gb300 import dllm

    R, D = st.batch.total_seq_rows, cfg.d_model
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    h = torch.randn(R, D, generator=g, device=dev).to(torch.bfloat16)
    W = (torch.randn(LM_VOCAB, D, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    gain = torch.ones(D, dtype=torch.bfloat16, device=dev)
    M = st.batch.total_block_rows
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    pm = torch.empty(M, dtype=torch.float32, device=dev)
    wsb = dllm.workspace(dllm.dllm_lm_head_workspace_size(st.desc, st.batch.c, LM_VOCAB), dev)
    stream = torch.cuda.current_stream()
    call = lambda: dllm.dllm_block_lm_head(st.desc, st.batch.c, LM_VOCAB, h, gain, W, None, lse, am, pm, wsb, stream)
    call()
    torch.cuda.synchronize()
    ev = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0, "device-side error in the LM head"
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del W, h
    return _max_over_ranks(ms, ws)


FFN_DFF = 12288  # the LLaDA-8B FFN width (the weights are synthetic)


def time_ffn(cfg, st, dev, ws, reps: int = 10):
    """Event-timed dllm_block_ffn (the rest of the layer for the block rows: output
    projection + residual, AddNorm with e4m3 quantisation, FP8 gate-up with SwiGLU,
    FP8 down + residual) with random e4m3 weights of the FFN_DFF-wide FFN."""
    from block_wise_kv_gb300 import dllm

    D, HD = cfg.d_model, cfg.n_heads * cfg.head_dim
    R, M = st.batch.total_seq_rows, st.batch.total_block_rows
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    o = (torch.randn(R, HD, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    x = torch.randn(M, D, generator=g, device=dev).to(torch.bfloat16)
    Wo = (torch.randn(D, HD, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    gain = torch.ones(D, dtype=torch.bfloat16, device=dev)

    def codes(rows, cols):  # random e4m3 codes without the NaN pattern
        c = torch.randint(0, 256, (rows, cols), generator=g, device=dev, dtype=torch.int32)
        return torch.where((c & 0x7F) == 0x7F, c & 0x78, c).to(torch.uint8)

    wgu, wd = codes(2 * FFN_DFF, D), codes(D, FFN_DFF)
    sgu = torch.full((2 * FFN_DFF // 128, D // 128), 2e-4, device=dev)
    sd = torch.full((D // 128, FFN_DFF // 128), 2e-4, device=dev)
    y = torch.empty(M, D, dtype=torch.bfloat16, device=dev)
    wsb = dllm.workspace(dllm.dllm_ffn_workspace_size(st.desc, st.batch.c, FFN_DFF), dev)
    stream = torch.cuda.current_stream()
    call = lambda: dllm.dllm_block_ffn(st.desc, st.batch.c, FFN_DFF, o, x, Wo, gain, wgu, sgu, wd, sd, y, wsb, stream)
    call()
    torch.cuda.synchronize()
    ev = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0, "device-side error in the FFN"
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return _max_over_ranks(ms, ws)


def e2e(items, Ke, W, ws):
    """End to end through the public step API: every step copies its block
    rows in from pinned host memory, runs the step and reads the block rows'
    outputs (the rows a sampler consumes) back to pinned host memory.  The
    read-back runs on a copy stream under the next step (another layer); a
    layer's next step waits until its previous read-back is done."""
    L = len(items)
    st0 = items[0][0]
    cu, sb, bl = (st0.batch.host[k] for k in ("cu_seq", "block_start", "block_len"))
    rows = [(int(cu[b] + sb[b]), int(cu[b] + sb[b] + bl[b])) for b in range(st0.batch.batch)]
    x_host = [xb.cpu().pin_memory() for _, xb, _ in items]
    o_host = [torch.empty(st.q_block.shape, dtype=torch.bfloat16).pin_memory() for st, _, _ in items]
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    read_out = [None] * L

    def step(i):
        j = i % L
        st, xb, _ = items[j]
        if read_out[j] is not None:
            main.wait_event(read_out[j])
        xb.copy_(x_host[j], non_blocking=True)
        st.step(xb)
        done = torch.cuda.Event()
        done.record(main)
        copy_stream.wait_event(done)
        with torch.cuda.stream(copy_stream):
            at = 0
            for lo, hi in rows:
                o_host[j][at:at + hi - lo].copy_(st.o_full[lo:hi], non_blocking=True)
                at += hi - lo
        ev = torch.cuda.Event()
        ev.record(copy_stream)
        read_out[j] = ev

    for i in range(min(W, 8)):
        step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for i in range(Ke):
        step(i)
    main.wait_stream(copy_stream)  # the last read-back is inside the timed region
    e1.record(main)
    torch.cuda.synchronize()
    ms = _max_over_ranks(e0.elapsed_time(e1), ws)
    return {"ms": ms, "steps": Ke, "h2d": x_host[0].numel() * x_host[0].element_size(),
            "d2h": o_host[0].numel() * o_host[0].element_size()}


def make_workload(name: str):
    """A named workload; "<name>_prefix_only" is that workload in the prefix-only cache
    mode of the Fast-dLLM page (every row after the prefix recomputed each step)."""
    from block_wise_kv_gb300.inputs import make_config

    if name.endswith("_prefix_only"):
        return make_config(name[: -len("_prefix_only")], prefix_only=True).with_(name=name)
    return make_config(name)


def build_flops(cfg, st):
    """Algorithmic flops of one block boundary: the projection of every row and the
    FACache state of every row of U over the keys of U (Q K^T and P V)."""
    D, HD = cfg.d_model, cfg.n_heads * cfg.head_dim
    lay = st.batch.host
    N = lay["seq_len"].astype(np.int64)
    U = N - lay["block_len"].astype(np.int64)
    return 6 * int(N.sum()) * D * HD + 4 * int((U * U).sum()) * HD


def summarize(res, hbm, tf_burst, ws, tf_sus=None):
    """Throughput, per-kernel durations and roofline objects of one measure()."""
    cfg, st, M = res["cfg"], res["st"], res["M"]
    bf = step_bytes_flops(cfg, st)
    att_bytes = bf["attention"][0] + bf["merge"][0]
    att_flops = bf["attention"][1] + bf["merge"][1]
    q = kernel_roofline("dllm_block_qkv_rope_write (one kernel: RMSNorm, tcgen05 QKV GEMM, RoPE, paged K/V write)",
                        bf["qkv"][0], bf["qkv"][1], res["qkv_ms"] * 1e-3, hbm, tf_burst, cfg.name, "qkv")
    a = kernel_roofline("dllm_step_attention (one kernel: block attention over all keys + FACache merge of "
                        "every invariant row)", att_bytes, att_flops, res["att_ms"] * 1e-3, hbm, tf_burst, cfg.name,
                        "attention")
    out = {"value": round(res["K"] * M * ws / (res["total_ms"] * 1e-3), 1), "ms_per_step": res["total_ms"] / res["K"],
           "qkv_rope_write_us": round(res["qkv_ms"] * 1e3, 2), "step_attention_us": round(res["att_ms"] * 1e3, 2),
           "roofline_kernels": {"qkv_rope_write": q, "step_attention": a},
           "sampled_calls": res["n_samples"]}
    if "steady_ms" in res:
        sd = res["steady_ms"]
        out["steady_state_us"] = {k: round(v * 1e3, 2) for k, v in sd.items()}
        out["steady_state_us"]["how"] = (f"graphs of {res['P'] * res['L']} calls of one kind, replayed back to "
                                         "back (launches overlapped as in the step)")
        out["steady_state_frac"] = {
            "qkv_rope_write": round(q["t_roof_us"] / (sd["qkv_rope_write"] * 1e3), 4),
            "step_attention": round(att_bytes / (sd["step_attention"] * 1e-3) / 1e9 / hbm, 4),
            "how": "qkv: t_roof over the steady-state duration; attention: algorithmic bytes / duration / HBM peak"}
        out["block_rows_only"] = {"value": round(M * ws / (sd["block_rows_only"] * 1e-3), 1), "unit": UNIT,
                                  "us_per_step": round(sd["block_rows_only"] * 1e3, 2)}
    if "build_ms" in res:
        fl = build_flops(cfg, st)
        tf = fl / (res["build_ms"] * 1e-3) / 1e12
        out["cache_build_us"] = {"per_boundary": round(res["build_ms"] * 1e3, 1),
                                 "per_inner_step": round(res["build_ms"] * 1e3 / cfg.steps_per_block, 2),
                                 "roofline": {"bound": "tensor", "achieved": round(tf, 1), "unit": "TFLOP/s",
                                              "flops": fl, "peak": tf_sus or tf_burst,
                                              "frac": round(tf / (tf_sus or tf_burst), 4),
                                              "frac_of_burst": round(tf / tf_burst, 4),
                                              "how": "projection of every row (6 R D HD) + FACache state of U over "
                                                     "U (4 |U|^2 HD per sequence) over the event-timed boundary "
                                                     "(back-to-back boundaries: sustained peak)"}}
        if "lm_head_ms" in res:
            M, D = int(st.batch.total_block_rows), cfg.d_model
            lm_bytes = LM_VOCAB * D * 2 + M * D * 2
            out["block_lm_head"] = kernel_roofline(
                f"dllm_block_lm_head (block rows only: gather + RMSNorm, tcgen05 LM head of {LM_VOCAB} entries with "
                "the softmax summary in its epilogue, ordered merge)", lm_bytes, 2 * M * LM_VOCAB * D,
                res["lm_head_ms"] * 1e-3, hbm, tf_burst, cfg.name, "lm_head")
        if "ffn_ms" in res:
            M, D, HD, F = int(st.batch.total_block_rows), cfg.d_model, cfg.n_heads * cfg.head_dim, FFN_DFF
            fl_bf16, fl_fp8 = 2 * M * D * HD, 2 * M * 2 * F * D + 2 * M * D * F
            by = D * HD * 2 + 2 * F * D + D * F + M * (HD + 2 * D) * 2  # weights, O rows, x, y
            t = res["ffn_ms"] * 1e-3
            t_tc = fl_bf16 / (tf_burst * 1e12) + fl_fp8 / (2 * tf_burst * 1e12)  # e4m3 at twice the bf16 rate
            t_hbm = by / (hbm * 1e9)
            bound = "tensor" if t_tc > t_hbm else "hbm"
            out["block_ffn"] = {
                "kernel": f"dllm_block_ffn (O-projection + residual, AddNorm + e4m3 quantisation, FP8 gate-up + "
                          f"SwiGLU, FP8 down + residual; d_ff {F})",
                "bound": bound, "duration_us": round(t * 1e6, 2), "t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2),
                "frac": round(max(t_tc, t_hbm) / t, 4), "algorithmic_flops": fl_bf16 + fl_fp8,
                "algorithmic_bytes": by, "traffic": None,
                "peak": f"bf16 {tf_burst} TFLOP/s (measured burst), e4m3 twice that (nominal ratio), "
                        f"HBM {hbm} GB/s"}
        if "advance_ms" in res:
            out["cache_build_us"]["advance"] = {
                "per_boundary": round(res["advance_ms"] * 1e3, 1),
                "vs_full_build": round(res["build_ms"] / res["advance_ms"], 2),
                "advances": res["advances"],
                "how": "dllm_cache_advance (only the decoded blocks' rows changed): their projection, the prefix "
                       "state extended by their keys, the state over U rebuilt from it and the suffix keys; mean "
                       "over a sweep of consecutive blocks on one layer instance"}
    return out


def run_ours(args, rank, ws, local):
    from block_wise_kv_gb300 import build, dllm
    from block_wise_kv_gb300.inputs import make_config

    if rank == 0:
        build.build()
    _barrier(ws)
    dllm.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm, tf_burst, tf_sus, peak_kind = _peaks()
    cfg = make_workload(args.config)
    L = cfg.layers if cfg.layers > 1 else args.layers
    P = max(1, 32 // L)  # a graph holds 32 layer-steps
    res = measure(cfg, L, args.steps, args.warmup, P, args.sample_every, dev, rank, ws, extras=True,
                  e2e_steps=args.e2e_steps)
    head = summarize(res, hbm, tf_burst, ws, tf_sus)
    e = res["e2e"]
    M = res["M"]
    clocks, wall = res["clocks"], res["host_wall_s"]
    del res
    torch.cuda.empty_cache()
    configs = {}
    if not args.headline_only and cfg.name == HEADLINE:
        for name in SECONDARY:
            c2 = make_workload(name)
            r2 = measure(c2, args.layers, args.secondary_steps, args.warmup, max(1, 32 // args.layers),
                         args.sample_every, dev, rank, ws, extras=True)
            s2 = summarize(r2, hbm, tf_burst, ws, tf_sus)
            s2["workload"] = describe(c2, args.layers)
            s2["steps"] = args.secondary_steps
            configs[name] = s2
            del r2
            torch.cuda.empty_cache()
    if rank != 0:
        return None
    rk = head["roofline_kernels"]
    dominant = max(rk.values(), key=lambda o: o["duration_us"])
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded, drawn on the device)",
        "config": {"workload": describe(cfg, L),
                   "l2": f"inputs larger than L2: {L} layer instances of ~1-3 GB each, walked in order",
                   "graphs": f"CUDA graphs of {P * L} layer-steps (2 kernels each, chained by programmatic "
                             f"dependent launch); the first round of every {args.sample_every}th graph (always the "
                             "first) replayed call by call with events around each kernel",
                   "parallelism": f"replicas x{ws} (sequences are independent units)"},
        "qkv_rope_write_us": head["qkv_rope_write_us"],
        "step_attention_us": head["step_attention_us"],
        "steady_state_us": head["steady_state_us"],
        "steady_state_frac": head["steady_state_frac"],
        "block_rows_only": head["block_rows_only"],
        "cache_build_us": head["cache_build_us"],
        "block_lm_head": head.get("block_lm_head"),
        "block_ffn": head.get("block_ffn"),
        "roofline": {k: v for k, v in dominant.items()},
        "roofline_kernels": rk,
        "peak_source": f"{peak_kind} MEASURED_PEAKS hbm_gbs / bf16_tflops (burst: each kernel timed alone)",
        "e2e": {"value": round(e["steps"] * M * ws / (e["ms"] * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"], "steps": e["steps"],
                "how": "x_block in from pinned host memory, the step through the public API, the block rows' "
                       "outputs read back to pinned host memory, every step"},
        "gpu_launches": 2 * args.steps,
        "sampled_calls": head["sampled_calls"],
        "host_wall_s": wall,
        "clocks": clocks,
        "configs": configs,
    }
    return line


_ORACLE_INPUTS = {}


def _oracle_inputs(cfg, wl, step):
    """fp64 inputs of the oracle for sequence 0 at the given inner step
    (generated once, outside any timed region)."""
    key = (cfg.name, step)
    if key not in _ORACLE_INPUTS:
        W, g = wl.weights(0)
        x = wl.seq_rows(0, 0, cfg.block_index[0], step).double().numpy()
        _ORACLE_INPUTS[key] = (x, g.double().numpy(), W.double().numpy())
    return _ORACLE_INPUTS[key]


def _oracle_step(cfg, wl, heads, step):
    """The oracle's full-recompute layer step of sequence 0 (every row's output
    for `heads`, None = all: RMSNorm, the projection, RoPE, attention)."""
    import oracle as orc

    x, g, W = _oracle_inputs(cfg, wl, step)
    return orc.layer_step(x, g, W, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps, heads=heads)


def cpu_baseline(cfg, seconds: float):
    """The oracle as it stands, timed on this host's cores on a bounded
    sample: sequence 0's full-recompute step for one head at a time, repeated
    for about `seconds`, scaled to all heads."""
    import oracle as orc
    from block_wise_kv_gb300.inputs import Workload

    wl = Workload(cfg)
    M = cfg.block[0]  # the sample is sequence 0: its block rows per step
    _oracle_step(cfg, wl, [0], 1)  # warm: builds/loads the library, generates the inputs
    n, t = 0, 0.0
    while t < seconds and n < cfg.n_heads:
        t0 = time.perf_counter()
        _oracle_step(cfg, wl, [n % cfg.n_heads], 1)
        t += time.perf_counter() - t0
        n += 1
    per_step = t / n * cfg.n_heads
    return {"value": round(M / per_step, 3), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"full-recompute layer step (fp64) of sequence 0 of {cfg.batch} for {n} of {cfg.n_heads} "
                      f"heads of {cfg.name}, {t:.1f} s, scaled to all heads; rate of that one sequence"}


def run_reference(args, rank, ws):
    if rank != 0:
        return None
    import oracle as orc
    from block_wise_kv_gb300.inputs import Workload, make_config

    cfg = make_config(args.config)
    wl = Workload(cfg)
    M = cfg.block[0]  # each step is sequence 0: its block rows
    _oracle_inputs(cfg, wl, 1)
    K, W = args.steps_ref, args.warmup_ref
    for _ in range(W):
        _oracle_step(cfg, wl, None, 1)
    t0 = time.perf_counter()
    for _ in range(K):
        _oracle_step(cfg, wl, None, 1)
    t = time.perf_counter() - t0
    per_step = t / K
    value = M / per_step
    sample = (f"each step: the full-recompute layer step (fp64, all {cfg.n_heads} heads) of sequence 0 of "
              f"{cfg.batch} of {cfg.name}; value = that sequence's block rows / step time")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
            "steps": K, "warmup": W, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": describe(cfg, cfg.layers if cfg.layers > 1 else 1)},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6400)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--layers", type=int, default=4,
                    help="layer instances of a one-layer workload (the stack uses all of its layers)")
    ap.add_argument("--e2e-steps", type=int, default=512)
    ap.add_argument("--secondary-steps", type=int, default=1024)
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads' figures")
    ap.add_argument("--sample-every", type=int, default=16,
                    help="the first round of every n-th graph (and always of the first) runs call by call")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    rank, ws, local = _dist()
    if args.impl == "reference":
        # each reference step is one sequence's full recompute: keep the run to minutes
        args.steps_ref = max(1, min(args.steps, 8))
        args.warmup_ref = max(1, min(args.warmup, 1))
        line = run_reference(args, rank, ws)
    else:
        if ws != args.gpus and rank == 0:
            print(f"note: --gpus {args.gpus} but WORLD_SIZE {ws}", file=sys.stderr)
        line = run_ours(args, rank, ws, local)
        if line is not None and not args.no_cpu_baseline:
            from block_wise_kv_gb300.inputs import make_config

            line["cpu_baseline"] = cpu_baseline(make_config(args.config), args.cpu_seconds)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
