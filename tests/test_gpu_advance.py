"""GPU parity of the incremental block boundary (dllm_cache_advance) and of the
prefix state that dllm_cache_build keeps for it, through the C ABI.

After a full build at block k0 and advances to k0+1, k0+2, ... (each with the
final rows of the block just decoded), the cached state of every row of U must
be the oracle's state over the keys of U for the rows of that block boundary
(LaCache §3.3.3), close to a full rebuild on the GPU, and the inner steps that
follow must match the oracle's full recompute (Fast-dLLM DualCache)."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_wise_kv_gb300 import dllm
from block_wise_kv_gb300.inputs import Config, Workload, make_config
from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of
from parity_util import assert_close, oracle_cache_state, oracle_step, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_wise_kv_gb300 import build

    build.build()
    dllm.load()
    torch.cuda.init()


def _mini128(**kw) -> Config:
    base = dict(name="mini128", d_model=512, n_heads=2, head_dim=128, t_prefix=[100], gen_len=[192], block=[32],
                block_index=[0], embedding=False)
    return make_config("tiny").with_(**{**base, **kw})


def _mini_ragged(**kw) -> Config:
    """Three sequences of different prompts, generation lengths and blocks, each with room
    for two more blocks after its current one."""
    base = dict(name="mini_ragged", t_prefix=[70, 200, 64], gen_len=[192, 256, 256], block=[32, 64, 16],
                block_index=[1, 0, 3], embedding=False)
    return make_config("tiny").with_(**{**base, **kw})


def _pools(st, b, U):
    return (to_np(st.pool_rows(st.cache.m, b))[U], to_np(st.pool_rows(st.cache.l, b))[U],
            to_np(st.pool_rows(st.cache.o, b))[U])


def _check_state(st, wl, layer, k_of, W, g, what):
    """The cached state of U against the oracle's for the rows of this boundary."""
    for b in range(wl.cfg.batch):
        U, m, l, Ot = oracle_cache_state(wl, layer, b, k_of[b], W, g)
        if len(U) == 0:
            continue
        gm, gl, go = _pools(st, b, U)
        assert_close(gm, m, f"{what} m seq {b}", max_abs=2e-2, rel=1e-3)
        assert_close(gl / np.exp(m - gm), l, f"{what} l seq {b}", max_abs=np.inf, rel=5e-3)
        assert_close(go, Ot / l[..., None], f"{what} O~/l seq {b}")


def _check_pre(st, wl, layer, k_of, W, g, what):
    """The prefix state of U: the state over the keys before the block."""
    cfg = wl.cfg
    for b in range(cfg.batch):
        x = wl.seq_rows(layer, b, k_of[b], 0).double().numpy()
        ref = orc.layer_step(x, g.double().numpy(), W.double().numpy(), cfg.n_heads, cfg.head_dim, cfg.rope_theta,
                             cfg.rms_eps)
        n, s = x.shape[0], cfg.block_start(b, k_of[b])
        U = np.r_[0:s, s + cfg.c_len(b, k_of[b]):n]
        m, l, Ot = orc.state_build(ref["q"][U], ref["k"], ref["v"], 1.0 / np.sqrt(cfg.head_dim), s, n)
        gm = to_np(st.pool_rows(st.cache.m_pre, b))[U]
        gl = to_np(st.pool_rows(st.cache.l_pre, b))[U]
        go = to_np(st.pool_rows(st.cache.o_pre, b))[U]
        assert_close(gm, m, f"{what} pre m seq {b}", max_abs=2e-2, rel=1e-3)
        assert_close(gl / np.exp(m - gm), l, f"{what} pre l seq {b}", max_abs=np.inf, rel=5e-3)
        assert_close(go, Ot / l[..., None], f"{what} pre O~/l seq {b}")


def _run_advances(cfg: Config, n_adv: int, layer=0, steps=(0,), compare_full=True):
    wl = Workload(cfg)
    W, g = wl.weights(layer)
    k_of = list(cfg.block_index)
    st = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g), pre=True)
    st.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0
    _check_pre(st, wl, layer, k_of, W, g, f"{cfg.name} build block {k_of}")
    last = cfg.steps_per_block - 1
    for _ in range(n_adv):
        x_dec = block_rows_of(wl, layer, last, k_of)  # the current blocks' final rows
        if cfg.prefix_only:  # C holds the suffix too: the decoded rows are the block's own
            x_dec = torch.cat([wl.seq_rows(layer, b, k_of[b], last)[cfg.block_start(b, k_of[b]):
                                                                     cfg.block_start(b, k_of[b]) + cfg.block[b]]
                               for b in range(cfg.batch)], 0).contiguous()
        k_of = [k + 1 for k in k_of]
        st.advance(k_of, x_dec.cuda())
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        what = f"{cfg.name} advanced to block {k_of}"
        _check_state(st, wl, layer, k_of, W, g, what)
        _check_pre(st, wl, layer, k_of, W, g, what)
        if compare_full:  # a full rebuild on the same rows: the same state up to rounding (the decoded
            # rows' q, k, v come from the small-batch projection there, the wide one here)
            fr = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g))
            fr.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
            torch.cuda.synchronize()
            for b in range(cfg.batch):
                n, s = cfg.seq_len(b), cfg.block_start(b, k_of[b])
                U = np.r_[0:s, s + cfg.c_len(b, k_of[b]):n]
                (am, al, ao), (fm, fl, fo) = _pools(st, b, U), _pools(fr, b, U)
                assert_close(am, fm, f"{what} m vs full build seq {b}", max_abs=2e-2, rel=1e-3)
                assert_close(ao, fo, f"{what} O~/l vs full build seq {b}")
        for s_ in steps:
            st.step(block_rows_of(wl, layer, s_, k_of).cuda())
            torch.cuda.synchronize()
            assert st.batch.error_bits() == 0
            for b in range(cfg.batch):
                ref = oracle_step(wl, layer, b, k_of[b], s_, W=W, g=g)
                assert_close(to_np(st.o_full[st.seq_slice(b)]), ref["O"], f"O {what} seq {b} step {s_}")
                assert_close(to_np(st.lse[st.seq_slice(b)]), ref["L"], f"LSE {what} seq {b} step {s_}",
                             max_abs=2e-2, rel=1e-3)
    return st


def test_advance_tiny_every_block():
    # blocks 0 -> 7: the suffix shrinks to nothing at the last block
    _run_advances(make_config("tiny"), n_adv=7, steps=(0, 3))


def test_advance_head_dim_128():
    _run_advances(_mini128(block_index=[1]), n_adv=3, steps=(1,))


def test_advance_ragged_batch():
    _run_advances(_mini_ragged(), n_adv=2, steps=(0,))


def test_advance_prefix_only():
    _run_advances(make_config("tiny", prefix_only=True, block_index=[2]), n_adv=3, steps=(0,))


def test_advance_llada_single():
    _run_advances(make_config("llada_single", block_index=[2]), n_adv=2, steps=(0,))


def test_build_without_prefix_pools_leaves_them_alone():
    """dllm_cache_build without the prefix pools takes the plain state build;
    advancing such a cache is rejected before any launch."""
    cfg = make_config("tiny")
    wl = Workload(cfg)
    st = LayerStep(cfg)
    st.boundary(full_rows_of(wl, 0, 0, cfg.block_index).cuda())
    torch.cuda.synchronize()
    with pytest.raises(dllm.DllmError) as e:
        st.advance([1], block_rows_of(wl, 0, cfg.steps_per_block - 1, cfg.block_index).cuda())
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
