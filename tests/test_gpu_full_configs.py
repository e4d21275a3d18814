"""GPU parity on the full-size LLaDA-8B-shaped configurations, sampled.

The GPU runs the whole batch at full size (every sequence, head and row);
the fp64 oracle recomputes sampled units from scratch: for the 32-layer
stack, layers {0, 31}, sequences {0, last}, blocks {first, middle, last},
inner steps {first, last}; for the long-context batch, sequences {0, last},
the same blocks and steps; for the ragged batch (shuffled physical pages),
every sequence at its own block index, steps {first, last}.  Each sampled
sequence is compared on every row (block rows and invariant rows) for two
heads (one for the ragged batch, rotating over the sequences), together
with the block rows' stored k and v.  Further units compare all 32 heads
(the 32-layer stack and the long-context batch: sequences {0, last}; the
ragged batch: four sequences), and one stack unit runs the attention as the
two separate calls (block attention, then the FACache merge), each with its
own launch plan.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from block_wise_kv_gb300 import dllm
from block_wise_kv_gb300.inputs import Workload, make_config
from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of
from parity_util import assert_bf16_close, assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_wise_kv_gb300 import build

    build.build()
    dllm.load()
    torch.cuda.init()


def _check(cfg, layer, k_of, steps, seqs, heads_of, split=False):
    wl = Workload(cfg)
    W, g = wl.weights(layer)
    st = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g))
    st.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0
    Wd, gd = W.double().numpy(), g.double().numpy()
    for s in steps:
        st.step(block_rows_of(wl, layer, s, k_of).cuda(), split=split)
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        for b in seqs:
            heads = list(heads_of(b))
            x = wl.seq_rows(layer, b, k_of[b], s).double().numpy()
            ref = orc.layer_step(x, gd, Wd, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps,
                                 heads=None if len(heads) == cfg.n_heads else heads)
            what = f"{cfg.name} layer {layer} seq {b} block {k_of[b]} step {s} heads {heads}"
            o = to_np(st.o_full[st.seq_slice(b)][:, heads])
            lse = to_np(st.lse[st.seq_slice(b)][:, heads])
            assert_close(o, ref["O"], f"O {what}")
            assert_close(lse, ref["L"], f"LSE {what}", max_abs=2e-2, rel=1e-3)
            c0 = cfg.block_start(b, k_of[b])
            blk = slice(c0, c0 + cfg.c_len(b, k_of[b]))
            kk = to_np(st.pool_rows(st.cache.k, b))[blk][:, heads]
            vv = to_np(st.pool_rows(st.cache.v, b))[blk][:, heads]
            assert_bf16_close(kk, ref["k"][blk], f"k block rows {what}")
            assert_bf16_close(vv, ref["v"][blk], f"v block rows {what}")


def _first_mid_last(n):
    return sorted({0, n // 2, n - 1})


def test_stack_sampled_layers_sequences_blocks_steps():
    cfg = make_config("stack")
    last = cfg.batch - 1
    for layer in (0, cfg.layers - 1):
        for k in _first_mid_last(cfg.num_blocks(0)):
            _check(cfg, layer, [k] * cfg.batch, (0, cfg.steps_per_block - 1), (0, last),
                   lambda b: (0, cfg.n_heads - 1))


def test_long_context_sampled():
    cfg = make_config("long")
    last = cfg.batch - 1
    for k in _first_mid_last(cfg.num_blocks(0)):
        _check(cfg, 0, [k] * cfg.batch, (0, cfg.steps_per_block - 1), (0, last), lambda b: (b % cfg.n_heads, 31))


def test_ragged_every_sequence():
    cfg = make_config("ragged")
    assert cfg.shuffle_pages
    _check(cfg, 0, list(cfg.block_index), (0, cfg.steps_per_block - 1), range(cfg.batch),
           lambda b: ((7 * b) % cfg.n_heads,))


ALL = lambda b: range(32)  # noqa: E731


def test_stack_all_heads():
    cfg = make_config("stack")
    mid = cfg.num_blocks(0) // 2
    _check(cfg, 0, [mid] * cfg.batch, (cfg.steps_per_block - 1,), (0, cfg.batch - 1), ALL)


def test_stack_split_calls():
    cfg = make_config("stack")
    _check(cfg, cfg.layers - 1, [0] * cfg.batch, (0,), (0, cfg.batch - 1), lambda b: (5, 17), split=True)


def test_long_context_all_heads():
    cfg = make_config("long")
    mid = cfg.num_blocks(0) // 2
    _check(cfg, 0, [mid] * cfg.batch, (cfg.steps_per_block - 1,), (0, cfg.batch - 1), ALL)


def test_ragged_all_heads_four_sequences():
    cfg = make_config("ragged")
    _check(cfg, 0, list(cfg.block_index), (cfg.steps_per_block - 1,), (0, 10, 20, cfg.batch - 1), ALL)
