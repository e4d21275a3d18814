"""GPU parity of the block-only epilogue (dllm_block_lm_head) through the C ABI
against the fp64 oracle (LaCache §3.4, the sampling stage: only the current
block's rows go through the final RMSNorm, the LM head and the softmax).

The hidden states of every row are random, so a kernel that read any row
outside the current blocks would miss the oracle, which is given the block
rows only."""
import numpy as np
import pytest
import torch

import oracle as orc
from block_wise_kv_gb300 import dllm
from block_wise_kv_gb300.inputs import Workload, layout, make_config
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_wise_kv_gb300 import build

    build.build()
    dllm.load()
    torch.cuda.init()


def _run(cfg, vocab, gain_spread=0.0, with_logits=True):
    wl = Workload(cfg)
    h, g, W = wl.lm_inputs(vocab, gain_spread)
    lay = layout(cfg)
    bl = dllm.BatchLayout(lay["block_table"], lay["seq_len"], lay["block_start"], lay["block_len"])
    desc = dllm.layer_desc(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps)
    M = bl.total_block_rows
    dev = "cuda"
    lse = torch.zeros(M, dtype=torch.float32, device=dev)
    am = torch.zeros(M, dtype=torch.int32, device=dev)
    pm = torch.zeros(M, dtype=torch.float32, device=dev)
    logits = torch.zeros(M, vocab, dtype=torch.bfloat16, device=dev) if with_logits else None
    ws = dllm.workspace(dllm.dllm_lm_head_workspace_size(desc, bl.c, vocab), dev)
    dllm.dllm_block_lm_head(desc, bl.c, vocab, h.cuda(), g.cuda(), W.cuda(), logits, lse, am, pm, ws)
    torch.cuda.synchronize()
    assert bl.error_bits() == 0
    # the oracle on the block rows only
    rows = np.concatenate([np.arange(lay["cu_seq"][b] + lay["block_start"][b],
                                     lay["cu_seq"][b] + lay["block_start"][b] + lay["block_len"][b])
                           for b in range(cfg.batch)])
    ref = orc.lm_head(h.double().numpy()[rows], g.double().numpy(), W.double().numpy(), cfg.rms_eps)
    what = f"{cfg.name} vocab {vocab} M {M}"
    assert_close(to_np(lse), ref["lse"], f"lse {what}", max_abs=2e-2, rel=1e-3)
    assert_close(np.log(to_np(pm)), np.log(ref["p_max"]), f"log p_max {what}", max_abs=2e-2, rel=np.inf)
    z = ref["logits"]
    got = to_np(am).astype(np.int64)
    top2 = np.sort(z, axis=1)[:, -2:]
    clear = top2[:, 1] - top2[:, 0] > 0.05
    assert np.array_equal(got[clear], ref["argmax"][clear]), f"argmax {what}"
    # near-ties: the chosen entry is one of the largest logits
    zm = z.max(axis=1)
    assert np.all(zm - z[np.arange(M), got] <= 0.05), f"argmax near-ties {what}"
    if with_logits:
        assert_close(to_np(logits), z, f"logits {what}")
    return clear.mean()


def test_lm_head_tiny():
    _run(make_config("tiny"), 1024)


def test_lm_head_ragged_partial_vocab_tile_and_gain():
    # 2056 entries: the last vocabulary tile holds 8, so its second half is empty
    cfg = make_config("tiny").with_(name="mini_ragged", t_prefix=[70, 200, 64], gen_len=[192, 128, 256],
                                    block=[32, 64, 16], block_index=[1, 0, 15], embedding=False)
    _run(cfg, 2056, gain_spread=0.5)


def test_lm_head_llada_single_without_logits():
    _run(make_config("llada_single"), 32768, with_logits=False)


def test_lm_head_stack_block_rows():
    # 512 block rows (four row tiles of 128) of the 32-layer stack's batch layout
    _run(make_config("stack"), 8192)


def test_lm_head_prefix_only_rows():
    # prefix-only: C (block + suffix, 256 rows) goes to the LM head
    _run(make_config("tiny", prefix_only=True), 1024)
