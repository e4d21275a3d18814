"""Run a few inner denoising steps of a named workload through the C ABI,
for profilers (ncu) and quick checks: no timing, no oracle.

    python -m block_wise_kv_gb300.run_steps --config stack --layers 1 --steps 3

Builds `--layers` independent layer instances (weights, paged cache after the
block boundary, block rows), inputs drawn on the device, then runs `--steps`
layer-steps (the projection call, then the attention call: `--split` makes it
the block attention and the FACache merge as two calls) on one stream and
checks the device error word.  `--boundary` also repeats the block boundary
once per instance at the end.  `--ffn K` then calls the rest of the layer
(`dllm_block_ffn`) K times on the first instance's block rows, with random
inputs and random e4m3 weights of width `--d-ff` (the bench's draws).
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import build, dllm
from .inputs import Workload, make_config
from .step import LayerStep


def run_ffn(st: LayerStep, cfg, d_ff: int, calls: int, dev) -> None:
    """`calls` calls of dllm_block_ffn on st's batch: attention output, residual stream,
    W_o and the e4m3 gate-up / down weights drawn like the bench's FFN timing."""
    D, HD = cfg.d_model, cfg.n_heads * cfg.head_dim
    R, M = st.batch.total_seq_rows, st.batch.total_block_rows
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    o = (torch.randn(R, HD, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    x = torch.randn(M, D, generator=g, device=dev).to(torch.bfloat16)
    w_o = (torch.randn(D, HD, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    gain = torch.ones(D, dtype=torch.bfloat16, device=dev)

    def codes(rows, cols):  # random e4m3 codes without the NaN pattern
        c = torch.randint(0, 256, (rows, cols), generator=g, device=dev, dtype=torch.int32)
        return torch.where((c & 0x7F) == 0x7F, c & 0x78, c).to(torch.uint8)

    w_gu, w_dn = codes(2 * d_ff, D), codes(D, d_ff)
    s_gu = torch.full((2 * d_ff // 128, D // 128), 2e-4, device=dev)
    s_dn = torch.full((D // 128, d_ff // 128), 2e-4, device=dev)
    y = torch.empty(M, D, dtype=torch.bfloat16, device=dev)
    ws = dllm.workspace(dllm.dllm_ffn_workspace_size(st.desc, st.batch.c, d_ff), dev)
    stream = torch.cuda.current_stream()
    for _ in range(calls):
        dllm.dllm_block_ffn(st.desc, st.batch.c, d_ff, o, x, w_o, gain, w_gu, s_gu, w_dn, s_dn, y, ws, stream)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--config", default="stack")
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--split", action="store_true")
    ap.add_argument("--boundary", action="store_true")
    ap.add_argument("--ffn", type=int, default=0)
    ap.add_argument("--d-ff", type=int, default=12288)
    args = ap.parse_args(argv)
    build.build()
    dllm.load()
    dev = torch.device("cuda", 0)
    cfg = make_config(args.config)
    wl = Workload(cfg)
    items = []
    for layer in range(args.layers):
        W, g = wl.weights_device(layer, dev)
        st = LayerStep(cfg, layer=layer, weights=(W, g), device=dev)
        del W
        x_full, x_blk = wl.batch_rows_device(layer, 1, cfg.block_index, dev)
        st.boundary(x_full)
        items.append((st, x_blk, x_full))
    torch.cuda.synchronize()
    for i in range(args.steps):
        st, xb, _ = items[i % len(items)]
        st.step(xb, split=args.split)
    if args.boundary:
        for st, _, x_full in items:
            st.boundary(x_full)
    if args.ffn:
        run_ffn(items[0][0], cfg, args.d_ff, args.ffn, dev)
    torch.cuda.synchronize()
    bad = [st.batch.error_bits() for st, _, _ in items]
    if any(bad):
        print(f"device error bits {bad}", file=sys.stderr)
        return 1
    extra = f", {args.ffn} FFN call(s)" if args.ffn else ""
    print(f"{cfg.name}: {args.steps} layer-steps over {len(items)} instance(s){extra} ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
