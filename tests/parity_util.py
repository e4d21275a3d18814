"""Shared helpers of the GPU parity tests: run the step through the C ABI and
compare with the fp64 oracle on the same seeded inputs.

Tolerance for bf16 outputs computed with fp32 accumulation: max abs error
<= 2e-2 and relative L2 error <= 5e-3 (over all rows and heads compared).
Intermediates stored as bf16 (q, k, v) may differ from the oracle's rounded
value by one bf16 step (2^-7 relative); elements that cancel to near zero
also carry the absolute difference of the pre-rounding values (the kernel
rounds x^ from fp32 and accumulates in fp32, about 1e-4 here), so the
per-element bound is 2^-7 |ref| + 2e-3 * rms(ref).
"""
import numpy as np
import torch

import oracle as orc
from block_wise_kv_gb300.inputs import Workload

MAX_ABS = 2e-2
REL_L2 = 5e-3


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


def assert_close(got, ref, what, max_abs=MAX_ABS, rel=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref).max() if got.size else 0.0
    r = rel_l2(got, ref)
    assert err <= max_abs and r <= rel, f"{what}: max abs {err:.3e} (<= {max_abs}), rel L2 {r:.3e} (<= {rel})"
    return err, r


def assert_bf16_close(got, ref, what):
    """Per-element: within one bf16 step of the value plus 2e-3 of the RMS."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    bad = np.abs(got - ref) > (2.0 ** -7) * np.abs(ref) + 2e-3 * rms
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} elements off by more than one bf16 step"
    assert rel_l2(got, ref) <= REL_L2, what


def oracle_step(wl: Workload, layer: int, b: int, k: int, step: int, rows=None, W=None, g=None):
    """The oracle's full-recompute layer step for sequence b at (block k, inner step)."""
    cfg = wl.cfg
    if W is None:
        W, g = wl.weights(layer)
    x = wl.seq_rows(layer, b, k, step).double().numpy()
    return orc.layer_step(x, g.double().numpy(), W.double().numpy(), cfg.n_heads, cfg.head_dim, cfg.rope_theta,
                          cfg.rms_eps, rows=rows)


def oracle_cache_state(wl: Workload, layer: int, b: int, k: int, W=None, g=None, step: int = 0):
    """Oracle FACache contents after a cache build of block k of sequence b
    from the rows of inner step `step` (0: the block boundary): (rows of U,
    m, l, O~) over the keys of U."""
    cfg = wl.cfg
    if W is None:
        W, g = wl.weights(layer)
    x = wl.seq_rows(layer, b, k, step).double().numpy()
    ref = orc.layer_step(x, g.double().numpy(), W.double().numpy(), cfg.n_heads, cfg.head_dim, cfg.rope_theta,
                         cfg.rms_eps)
    s = cfg.block_start(b, k)
    e = s + cfg.c_len(b, k)
    U = np.r_[0:s, e:x.shape[0]]
    m, l, Ot = orc.state_build(ref["q"][U], ref["k"], ref["v"], 1.0 / np.sqrt(cfg.head_dim), s, e)
    return U, m, l, Ot


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)
