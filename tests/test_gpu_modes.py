"""GPU parity of the cache modes of the Fast-dLLM page beside DualCache, through
the C ABI, against the fp64 oracle's full recompute of the same rows.

* Prefix-only caching (use_dual_cache = False): every row after the prefix is
  recomputed at every inner step, so the fresh region C is the current block
  and the whole suffix, and the cached invariant rows U are the prefix (the
  prompt and the decoded blocks).  Blocks of more than one page run on the
  128-row query-tile kernels (block rows over every key; rows of U merged with
  their cached state over the keys of C); the cache build keeps the state of U
  over the keys of U as in DualCache.
* Suffix refresh every r inner steps (refresh_interval = r): the cache is
  rebuilt from the rows of steps r, 2r, ...  The exact result of a step is the
  full recompute of the rows the cache was built from, with the block rows of
  the current step: the U rows (prefix and suffix) keep the K, V and state of
  the last rebuild.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from block_wise_kv_gb300 import dllm
from block_wise_kv_gb300.inputs import Config, Workload, make_config
from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of
from parity_util import assert_bf16_close, assert_close, oracle_cache_state, oracle_step, rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_wise_kv_gb300 import build

    build.build()
    dllm.load()
    torch.cuda.init()


def _mini128(**kw) -> Config:
    """head_dim 128 at a small width: 2 heads, d_model 512, prompt 100, gen 192 in blocks of 32."""
    base = dict(name="mini128", d_model=512, n_heads=2, head_dim=128, t_prefix=[100], gen_len=[192], block=[32],
                block_index=[0], embedding=False)
    return make_config("tiny").with_(**{**base, **kw})


def _mini_ragged(**kw) -> Config:
    """Three sequences of different prompts, generation lengths and blocks."""
    base = dict(name="mini_ragged", t_prefix=[70, 200, 64], gen_len=[192, 128, 256], block=[32, 64, 16],
                block_index=[1, 0, 15], embedding=False)
    return make_config("tiny").with_(**{**base, **kw})


def _check_cache(st, wl, layer, k_of, seqs, W, g, step=0):
    for b in seqs:
        U, m, l, Ot = oracle_cache_state(wl, layer, b, k_of[b], W, g, step=step)
        if len(U) == 0:
            continue
        gm = to_np(st.pool_rows(st.cache.m, b))[U]
        gl = to_np(st.pool_rows(st.cache.l, b))[U]
        go = to_np(st.pool_rows(st.cache.o, b))[U]
        assert_close(gm, m, f"cache m seq {b}", max_abs=2e-2, rel=1e-3)
        assert_close(gl / np.exp(m - gm), l, f"cache l seq {b}", max_abs=np.inf, rel=5e-3)
        assert_close(go, Ot / l[..., None], f"cache O~/l seq {b}")


def _run_prefix_only(cfg: Config, steps, layer=0, seqs=None, split=False):
    """Boundary of each sequence's block, then the inner steps; all rows of the
    listed sequences against the oracle's full recompute of the step."""
    assert cfg.prefix_only
    wl = Workload(cfg)
    W, g = wl.weights(layer)
    k_of = cfg.block_index
    st = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g))
    assert st.batch.max_block_len == max(cfg.c_len(b) for b in range(cfg.batch))
    st.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0
    seqs = range(cfg.batch) if seqs is None else seqs
    _check_cache(st, wl, layer, k_of, seqs, W, g)
    for s in steps:
        st.step(block_rows_of(wl, layer, s, k_of).cuda(), split=split)
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        for b in seqs:
            ref = oracle_step(wl, layer, b, k_of[b], s, W=W, g=g)
            what = f"{cfg.name} seq {b} block {k_of[b]} step {s}"
            assert_close(to_np(st.o_full[st.seq_slice(b)]), ref["O"], f"O {what}")
            assert_close(to_np(st.lse[st.seq_slice(b)]), ref["L"], f"LSE {what}", max_abs=2e-2, rel=1e-3)
            c0 = cfg.block_start(b)
            c = slice(c0, c0 + cfg.c_len(b))
            assert_bf16_close(to_np(st.pool_rows(st.cache.k, b))[c], ref["k"][c], f"k rows of C {what}")
            assert_bf16_close(to_np(st.pool_rows(st.cache.v, b))[c], ref["v"][c], f"v rows of C {what}")
            assert_bf16_close(to_np(st.q_block[st.block_slice(b)]), ref["q"][c], f"q_block {what}")
    return st


@pytest.mark.parametrize("k", [0, 3, 7])
def test_prefix_only_tiny(k):
    # C = 256, 160 and 32 rows (the last block has no suffix: one page, the streaming kernel)
    _run_prefix_only(make_config("tiny", prefix_only=True, block_index=[k]), steps=(0, 2))


@pytest.mark.parametrize("k", [0, 2, 5])
def test_prefix_only_head_dim_128(k):
    _run_prefix_only(_mini128(prefix_only=True, block_index=[k]), steps=(0, 1))


def test_prefix_only_ragged_batch():
    # C = 160, 128 and 16 rows: the longest block sets the kernels, short ones ride along
    _run_prefix_only(_mini_ragged(prefix_only=True), steps=(0, 1))


@pytest.mark.parametrize("k", [0, 4])
def test_prefix_only_llada_single(k):
    _run_prefix_only(make_config("llada_single", prefix_only=True, block_index=[k]), steps=(0,))


def test_prefix_only_split_calls_equal_fused():
    """dllm_block_attention + dllm_state_merge as two calls against
    dllm_step_attention, for blocks of more than one page: bit for bit."""
    cfg = _mini_ragged(prefix_only=True)
    wl = Workload(cfg)
    outs = []
    for split in (False, True):
        st = LayerStep(cfg)
        st.boundary(full_rows_of(wl, 0, 0, cfg.block_index).cuda())
        st.step(block_rows_of(wl, 0, 1, cfg.block_index).cuda(), split=split)
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        outs.append((st.o_full.cpu(), st.lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def _run_refresh(cfg: Config, steps, r, layer=0):
    """Inner steps with the cache rebuilt every r steps; returns the relative L2
    distance of each non-refresh step from the full recompute of its own rows."""
    assert cfg.suffix_varies
    wl = Workload(cfg)
    W, g = wl.weights(layer)
    k_of = cfg.block_index
    st = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g))
    st.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
    last = 0  # the step whose rows the cache holds
    stale = []
    Wd, gd = W.double().numpy(), g.double().numpy()
    for s in steps:
        if st.inner_step(s, block_rows_of(wl, layer, s, k_of).cuda(), full_rows_of(wl, layer, s, k_of).cuda(),
                         refresh_interval=r):
            last = s
            torch.cuda.synchronize()
            _check_cache(st, wl, layer, k_of, range(cfg.batch), W, g, step=s)
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        for b in range(cfg.batch):
            c0 = cfg.block_start(b)
            x = wl.seq_rows(layer, b, k_of[b], last).double().numpy()
            x[c0:c0 + cfg.c_len(b)] = wl.block_rows(layer, b, k_of[b], s).double().numpy()
            ref = orc.layer_step(x, gd, Wd, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps)
            what = f"{cfg.name} seq {b} step {s} (cache from step {last})"
            o = to_np(st.o_full[st.seq_slice(b)])
            assert_close(o, ref["O"], f"O {what}")
            assert_close(to_np(st.lse[st.seq_slice(b)]), ref["L"], f"LSE {what}", max_abs=2e-2, rel=1e-3)
            if last != s:
                exact = oracle_step(wl, layer, b, k_of[b], s, W=W, g=g)
                stale.append(rel_l2(o, exact["O"]))
    return stale


def test_refresh_interval_rebuilds_suffix():
    cfg = _mini_ragged(suffix_varies=True, block_index=[1, 0, 3])
    stale = _run_refresh(cfg, steps=range(5), r=2)
    # the steps between refreshes keep the suffix of the last rebuild, which differs from
    # their own rows: the comparison above tells the two apart
    assert len(stale) == 2 * cfg.batch and min(stale) > 1e-2, stale


def test_refresh_every_step_is_full_recompute():
    cfg = _mini128(suffix_varies=True, block_index=[1])
    assert _run_refresh(cfg, steps=range(3), r=1) == []
