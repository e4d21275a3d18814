#!/usr/bin/env python3
"""Throughput of the per-layer inner denoising step of block-wise
diffusion-LLM decoding on GB300.

One step = one pass of the whole hot path for one layer: the fused RMSNorm +
QKV projection + RoPE + paged K/V write of the block rows, the block
attention over [prefix | block | suffix], and the FACache merge of every
invariant row.  The metric is block-query tokens per second per layer-step
(block rows of all sequences / step time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: the LLaDA-8B-shaped single layer (batch 1, d_model 4096, 32 heads
x 128, RoPE theta 5e5, prompt 512, gen 256, block 32), synthetic seeded
bf16 inputs and N(0, 0.02) weights.  Steps rotate over several independent
layer instances (about 140 MB each), so no step finds its inputs in the
129 MB L2.  The steps replay CUDA graphs of 32 layer-steps (8 rounds of the
4 instances, as one forward over 32 layers would be; two kernels a step: the
fused RMSNorm + projection + RoPE + K/V write, and the block attention +
FACache merge launch); a sample of the steps (one round in 128) carries CUDA
events around the projection call on its stream, which give its live
duration for the roofline.  The end-to-end figure calls the public step API
with the block rows copied in from pinned host memory and o_full read back to
pinned host memory every step (the read-back on a copy stream, under the next
step).

Under torchrun (N > 1) every rank runs its own replica of the workload
(sequences are independent units: weak scaling, no collective on the data
path); the time is the max over ranks.

--impl reference times the fp64 CPU oracle (full recompute of the step) on
the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llada_single"
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


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one projection
# launch, per workload, from one ncu capture of the kernel as it stands
# (--set full, the launch of an inner step); no entry: not captured.
QKV_TRAFFIC_BYTES = {"llada_single": 103_979_008}


def step_bytes_flops(cfg, st):
    """Algorithmic bytes and flops of one layer-step (what the method must
    move and compute), per part."""
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
    mrg_bytes = int((NU * HD * 8).sum()) + int(NU.sum()) * H * 8
    mrg_flops = int((4 * NU * B * HD).sum())
    return dict(qkv=(qkv_bytes, qkv_flops), attention=(att_bytes, att_flops), merge=(mrg_bytes, mrg_flops))


def describe(cfg) -> str:
    """The workload, named by what it is with its sizes."""
    N = np.array([cfg.seq_len(b) for b in range(cfg.batch)], dtype=np.int64)
    M = int(sum(cfg.block))
    seqs = f"batch {cfg.batch}"
    if len(set(cfg.t_prefix)) == 1 and len(set(cfg.gen_len)) == 1 and len(set(cfg.block)) == 1:
        seqs += f", prompt {cfg.t_prefix[0]}, gen {cfg.gen_len[0]}, block {cfg.block[0]}"
    else:
        seqs += f", prompt {min(cfg.t_prefix)}..{max(cfg.t_prefix)}, gen {sorted(set(cfg.gen_len))}, " \
                f"block {sorted(set(cfg.block))}"
    return (f"{cfg.name}: 1 layer step, d_model {cfg.d_model}, {cfg.n_heads}x{cfg.head_dim} heads, {seqs} "
            f"(M={M} block rows, N={int(N.sum())} rows)")


def run_ours(args, rank, ws, local):
    from block_wise_kv_gb300 import build, dllm
    from block_wise_kv_gb300.inputs import Workload, make_config
    from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of

    if rank == 0:
        build.build()
    _barrier(ws)
    dllm.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = make_config(args.config)
    wl = Workload(cfg.with_(seed=rank))
    blocks = cfg.block_index
    L = args.layers
    inst = []
    for layer in range(L):
        st = LayerStep(cfg, layer=layer)
        st.boundary(full_rows_of(wl, layer, 0, blocks).to(dev))
        xb = block_rows_of(wl, layer, 1, blocks).to(dev)
        inst.append((st, xb))
    torch.cuda.synchronize()
    for st, _ in inst:
        assert st.batch.error_bits() == 0, "device-side error during setup"
    M = inst[0][0].batch.total_block_rows

    # CUDA graphs.  A round is one step of every instance (L steps: the
    # projection call, then the block attention and the FACache merge in one
    # launch); a pass is P rounds in one graph (P L layer-steps, as one
    # forward over the layers of a model would be), so consecutive kernels
    # keep their programmatic-dependent-launch overlap.  In every
    # `sample_every`-th pass the first round replays per-instance pieces
    # instead, with CUDA events around the projection call on its stream:
    # those give the projection's live duration for the roofline, inside the
    # timed region.
    P = max(1, args.rounds_per_graph)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for st, xb in inst:
            st.step(xb, stream=stream)
        stream.synchronize()
        g_round = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_round, stream=stream):
            for st, xb in inst:
                st.step(xb, stream=stream)
        g_pass = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pass, stream=stream):
            for _ in range(P):
                for st, xb in inst:
                    st.step(xb, stream=stream)
        g_step, g_qkv, g_rest = [], [], []  # one step; the projection call; the attention call
        for st, xb in inst:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st.step(xb, stream=stream)
            g_step.append(g)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st.qkv(xb, stream=stream)
            g_qkv.append(g)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st.step_attention(stream)
            g_rest.append(g)
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    sample_every = max(1, args.sample_every)
    for i in range(W):
        g_step[i % L].replay()
    torch.cuda.synchronize()
    n_rounds, tail = divmod(K, L)
    n_passes, tail_rounds = divmod(n_rounds, P)
    qkv_ev = []
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks, torch.cuda.stream(stream):
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        t_start.record(stream)
        for k in range(n_passes):
            if k % sample_every == sample_every - 1:
                for j in range(L):
                    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    e[0].record(stream)
                    g_qkv[j].replay()
                    e[1].record(stream)
                    g_rest[j].replay()
                    e[2].record(stream)
                    qkv_ev.append(e)
                for _ in range(P - 1):
                    g_round.replay()
            else:
                g_pass.replay()
        for _ in range(tail_rounds):
            g_round.replay()
        for j in range(tail):
            g_step[j].replay()
        t_end.record(stream)
        stream.synchronize()
        t1 = time.perf_counter()
    torch.cuda.synchronize()
    _barrier(ws)
    total_ms = t_start.elapsed_time(t_end)
    if not qkv_ev:  # too few rounds to sample: time the projection alone after the region
        with torch.cuda.stream(stream):
            for j in range(L):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(stream)
                g_qkv[j].replay()
                e[1].record(stream)
                g_rest[j].replay()
                e[2].record(stream)
                qkv_ev.append(e)
        torch.cuda.synchronize()
    qkv_ms = sum(e[0].elapsed_time(e[1]) for e in qkv_ev) / len(qkv_ev)
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in qkv_ev) / len(qkv_ev)
    total_ms = _max_over_ranks(total_ms, ws)
    for st, _ in inst:
        assert st.batch.error_bits() == 0, "device-side error during the timed steps"

    # end to end through the public API: pinned host input -> step -> host output.
    # The read-back of a step's o_full runs on a copy stream while the next
    # step (another layer instance) computes; a layer instance's next step
    # waits until its previous o_full has been read out.
    x_host = [xb.cpu().pin_memory() for _, xb in inst]
    o_host = [torch.empty_like(st.o_full, device="cpu").pin_memory() for st, _ in inst]
    x_dev = [torch.empty_like(xb) for _, xb in inst]
    Ke = max(1, min(K, args.e2e_steps))
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    read_out = [None] * L

    def e2e_step(i):
        j = i % L
        st, _ = inst[j]
        if read_out[j] is not None:
            main.wait_event(read_out[j])
        x_dev[j].copy_(x_host[j], non_blocking=True)
        st.step(x_dev[j])
        done = torch.cuda.Event()
        done.record(main)
        copy_stream.wait_event(done)
        with torch.cuda.stream(copy_stream):
            o_host[j].copy_(st.o_full, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(copy_stream)
        read_out[j] = ev

    for i in range(min(W, 8)):
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for i in range(Ke):
        e2e_step(i)
    main.wait_stream(copy_stream)  # the last read-back is inside the timed region
    e1.record(main)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), ws)
    h2d = x_host[0].numel() * x_host[0].element_size()
    d2h = o_host[0].numel() * o_host[0].element_size()

    # secondary: the block rows only (projection + block attention, no FACache
    # merge of the invariant rows: what a DualCache consumer of the block
    # outputs needs), graph-replayed like the main loop
    with torch.cuda.stream(stream):
        g_blk = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_blk, stream=stream):
            for _ in range(P):
                for st, xb in inst:
                    st.qkv(xb, stream=stream)
                    st.attention(stream)
        for _ in range(3):
            g_blk.replay()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_blk = max(1, min(n_passes, 100))
        k0.record(stream)
        for _ in range(n_blk):
            g_blk.replay()
        k1.record(stream)
    torch.cuda.synchronize()
    blk_ms = _max_over_ranks(k0.elapsed_time(k1), ws) / (n_blk * P * L)

    # secondary: each call of the step alone in steady state (a graph of P
    # rounds of that call only, so consecutive launches of the same kernel
    # overlap through programmatic dependent launch as in the step's graphs)
    steady = {}
    with torch.cuda.stream(stream):
        for name, call in (("qkv_rope_write", lambda st, xb: st.qkv(xb, stream=stream)),
                           ("step_attention", lambda st, xb: st.step_attention(stream))):
            g_one = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_one, stream=stream):
                for _ in range(P):
                    for st, xb in inst:
                        call(st, xb)
            for _ in range(3):
                g_one.replay()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_one = max(1, min(n_passes, 100))
            s0.record(stream)
            for _ in range(n_one):
                g_one.replay()
            s1.record(stream)
            s1.synchronize()
            steady[name] = s0.elapsed_time(s1) / (n_one * P * L)
    steady = {k: _max_over_ranks(v, ws) for k, v in steady.items()}

    # the block boundary (cache build: projection of every row, FACache state
    # over U x U), timed apart: once per block, amortised over its inner steps
    x_full = [full_rows_of(wl, layer, 0, blocks).to(dev) for layer in range(L)]
    for j in range(L):
        inst[j][0].boundary(x_full[j])
    torch.cuda.synchronize()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nb = 2 * L
    b0.record()
    for i in range(nb):
        inst[i % L][0].boundary(x_full[i % L])
    b1.record()
    torch.cuda.synchronize()
    build_ms = b0.elapsed_time(b1) / nb

    if rank != 0:
        return None
    hbm, tf_burst, tf_sus, peak_kind = _peaks()
    bf = step_bytes_flops(cfg, inst[0][0])
    qkv_bytes, qkv_flops = bf["qkv"]
    t_qkv = qkv_ms * 1e-3
    achieved = qkv_bytes / t_qkv / 1e9
    value = K * M * ws / (total_ms * 1e-3)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": K,
        "warmup": W,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(cfg),
                   "l2": f"inputs larger than L2: {L} rotating layer instances (~140 MB each)",
                   "graphs": f"one CUDA graph per pass of {P} rounds x {L} steps ({P * L} layer-steps); the first "
                             f"round of every {sample_every}th pass replayed per call with events around the "
                             "projection",
                   "parallelism": f"replicas x{ws} (sequences are independent units)"},
        "qkv_rope_write_us": round(qkv_ms * 1e3, 2),
        "step_attention_us": round(attn_ms * 1e3, 2),
        "step_attention_gbs": round((bf["attention"][0] + bf["merge"][0]) / (attn_ms * 1e-3) / 1e9, 1),
        "steady_state_us": {"qkv_rope_write": round(steady["qkv_rope_write"] * 1e3, 2),
                            "step_attention": round(steady["step_attention"] * 1e3, 2),
                            "how": f"graphs of {P * L} calls of one kind, replayed back to back"},
        "block_rows_only": {"value": round(M * ws / (blk_ms * 1e-3), 1), "unit": UNIT,
                            "us_per_step": round(blk_ms * 1e3, 2)},
        "cache_build_us": {"per_boundary": round(build_ms * 1e3, 1),
                           "per_inner_step": round(build_ms * 1e3 / cfg.steps_per_block, 2)},
        "roofline": {"kernel": "dllm_block_qkv_rope_write (one kernel: RMSNorm, tcgen05 QKV GEMM, RoPE and the "
                               "paged K/V write)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": QKV_TRAFFIC_BYTES.get(cfg.name),
                     "algorithmic_bytes": qkv_bytes, "peak_source": f"{peak_kind} hbm_gbs",
                     "steady_state": {"achieved": round(qkv_bytes / (steady["qkv_rope_write"] * 1e-3) / 1e9, 1),
                                      "frac": round(qkv_bytes / (steady["qkv_rope_write"] * 1e-3) / 1e9 / hbm, 4),
                                      "how": "the same bytes over the per-call duration in graphs of "
                                             f"{P * L} projection calls (launches overlapped as in the step)"}},
        "e2e": {"value": round(Ke * M * ws / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke},
        "gpu_launches": 2 * K,
        "host_wall_s": t1 - t0,
    }
    cl = clocks.summary()
    line["clocks"] = cl
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
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


def _oracle_sample(cfg, wl, heads, step):
    """The oracle's full-recompute layer step restricted to `heads` (every
    row's output for those heads; RMSNorm, K/V of all rows, attention)."""
    import oracle as orc

    x, g, W = _oracle_inputs(cfg, wl, step)
    return orc.layer_step(x, g, W, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps, heads=heads)


def cpu_baseline(cfg, seconds: float):
    """The oracle as it stands, timed on this host's cores on a bounded
    sample: the full step for one head at a time, repeated for about
    `seconds`, scaled to all heads."""
    import oracle as orc
    from block_wise_kv_gb300.inputs import Workload

    wl = Workload(cfg)
    M = cfg.block[0]  # the sample is sequence 0: its block rows per step
    _oracle_sample(cfg, wl, [0], 1)  # warm: builds/loads the library, generates the inputs
    n, t = 0, 0.0
    while t < seconds and n < cfg.n_heads:
        t0 = time.perf_counter()
        _oracle_sample(cfg, wl, [n % cfg.n_heads], 1)
        t += time.perf_counter() - t0
        n += 1
    per_step = t / n * cfg.n_heads
    return {"value": round(M / per_step, 3), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"full-recompute layer step (fp64) of sequence 0 for {n} of {cfg.n_heads} heads of "
                      f"{cfg.name}, {t:.1f} s, scaled to all heads" + ("" if cfg.batch == 1 else
                                                                        " (sequence 0 only)")}


def run_reference(args, rank, ws):
    if rank != 0:
        return None
    import oracle as orc
    from block_wise_kv_gb300.inputs import Workload, make_config

    cfg = make_config(args.config)
    wl = Workload(cfg)
    M = cfg.block[0]  # each step samples sequence 0: its block rows per step
    _oracle_inputs(cfg, wl, 1)
    K, W = args.steps_ref, args.warmup_ref
    for i in range(W):
        _oracle_sample(cfg, wl, [i % cfg.n_heads], 1)
    t0 = time.perf_counter()
    for i in range(K):
        _oracle_sample(cfg, wl, [i % cfg.n_heads], 1)
    t = time.perf_counter() - t0
    per_step = t / K * cfg.n_heads
    value = M / per_step
    sample = (f"each step: full-recompute layer step (fp64) of sequence 0 for one head of {cfg.n_heads}, scaled "
              "to all heads" + ("" if cfg.batch == 1 else "; rate of one sequence"))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
            "steps": K, "warmup": W, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(cfg)},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--layers", type=int, default=4, help="rotating layer instances (inputs larger than L2)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--rounds-per-graph", type=int, default=8,
                    help="rounds of steps (one step of every layer instance each) captured in one graph")
    ap.add_argument("--sample-every", type=int, default=16,
                    help="the first round of every n-th pass carries events around the projection call")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    rank, ws, local = _dist()
    if args.impl == "reference":
        # each reference step is one head's full recompute: keep the run to minutes
        args.steps_ref = max(1, min(args.steps, 32))
        args.warmup_ref = max(1, min(args.warmup, 2))
        line = run_reference(args, rank, ws)
    else:
        if ws != args.gpus and rank == 0:
            print(f"note: --gpus {args.gpus} but WORLD_SIZE {ws}", file=sys.stderr)
        line = run_ours(args, rank, ws, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
