"""Run a few inner denoising steps of a named workload through the C ABI,
for profilers (ncu) and quick checks: no timing, no oracle.

    python -m block_wise_kv_gb300.run_steps --config stack --layers 1 --steps 3

Builds `--layers` independent layer instances (weights, paged cache after the
block boundary, block rows), inputs drawn on the device, then runs `--steps`
layer-steps (the projection call, then the attention call: `--split` makes it
the block attention and the FACache merge as two calls) on one stream and
checks the device error word.  `--boundary` also repeats the block boundary
once per instance at the end.
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import build, dllm
from .inputs import Workload, make_config
from .step import LayerStep


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--config", default="stack")
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--split", action="store_true")
    ap.add_argument("--boundary", action="store_true")
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
    torch.cuda.synchronize()
    bad = [st.batch.error_bits() for st, _, _ in items]
    if any(bad):
        print(f"device error bits {bad}", file=sys.stderr)
        return 1
    print(f"{cfg.name}: {args.steps} layer-steps over {len(items)} instance(s) ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
