"""dllm_block_qkv_rope_write_noalloc: the fused projection for callers that
cannot allocate device memory (it uses the library's fixed scratch instead of
a caller workspace).  Its results must match the workspace entry point's on
the same inputs, on two calls in a row.  This file is collected last."""
import numpy as np
import pytest
import torch

from block_wise_kv_gb300 import build, dllm
from block_wise_kv_gb300.inputs import Workload, make_config
from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of
from parity_util import to_np

pytestmark = pytest.mark.gpu


def _call_both(st, xb):
    """(q_block, block K rows, block V rows) from the workspace call and from
    the allocation-free call on the same inputs."""
    out = []
    for noalloc in (False, True):
        st.q_block.zero_()
        if noalloc:
            dllm.dllm_block_qkv_rope_write_noalloc(st.desc, st.batch.c, xb, st.gain, st.w_qkv, st.rope,
                                                  st.rope_max_pos, st.cache.c, st.q_block)
        else:
            st.qkv(xb)
        torch.cuda.synchronize()
        s0 = int(st.batch.host["block_start"][0])
        blk = slice(s0, s0 + int(st.batch.host["block_len"][0]))
        out.append((to_np(st.q_block), to_np(st.pool_rows(st.cache.k, 0))[blk],
                    to_np(st.pool_rows(st.cache.v, 0))[blk]))
    return out


def test_noalloc_matches_workspace_call_twice():
    build.build()
    dllm.load()
    cfg = make_config("llada_single")
    wl = Workload(cfg)
    st = LayerStep(cfg)
    st.boundary(full_rows_of(wl, 0, 0, cfg.block_index).cuda())
    torch.cuda.synchronize()
    for step in (2, 5):  # two calls in a row with different block rows
        (q0, k0, v0), (q1, k1, v1) = _call_both(st, block_rows_of(wl, 0, step, cfg.block_index).cuda())
        # the same kernel on the same inputs: bit for bit, so a stale value left in the
        # scratch by the previous call would show
        assert np.array_equal(q1, q0), f"q_block, call at step {step}"
        assert np.array_equal(k1, k0), f"block K rows, call at step {step}"
        assert np.array_equal(v1, v0), f"block V rows, call at step {step}"
    assert st.batch.error_bits() == 0


def test_noalloc_split_schedule_uses_its_scratch():
    """A small model (6 weight tiles, <= 64 block rows) runs the split
    schedule, whose partial tiles, RMSNorm rows and scales and counters all
    live in the fixed scratch: the results match the workspace call bit for bit,
    call after call (the counters return to zero after each call)."""
    build.build()
    dllm.load()
    cfg = make_config("tiny").with_(d_model=4096, n_heads=2, head_dim=128, t_prefix=[100, 5], gen_len=[96, 40],
                                    block=[32, 20], block_index=[1, 1])
    wl = Workload(cfg)
    st = LayerStep(cfg)
    M = st.batch.total_block_rows
    assert st.ws_step.numel() > 4096 + 512 + M * 4096 * 2  # partial tiles beyond counters, scales and x^ rows
    st.boundary(full_rows_of(wl, 0, 0, cfg.block_index).cuda())
    torch.cuda.synchronize()
    for step in (0, 1, 1):
        (q0, k0, v0), (q1, k1, v1) = _call_both(st, block_rows_of(wl, 0, step, cfg.block_index).cuda())
        assert np.array_equal(q1, q0), f"q_block, step {step}"
        assert np.array_equal(k1, k0), f"block K rows, step {step}"
        assert np.array_equal(v1, v0), f"block V rows, step {step}"
    assert st.batch.error_bits() == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    build.build()
    dllm.load()
    # 1280 block rows of d_model 4096 need 10 MiB of scratch (their x^ rows):
    # more than the fixed 8 MiB
    cfg = make_config("tiny").with_(d_model=4096, n_heads=32, head_dim=128, t_prefix=[64] * 20, gen_len=[64] * 20,
                                    block=[64] * 20, block_index=[0] * 20)
    st = LayerStep(cfg)
    xb = torch.zeros(st.batch.total_block_rows, cfg.d_model, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_qkv_rope_write_noalloc(st.desc, st.batch.c, xb, st.gain, st.w_qkv, st.rope, st.rope_max_pos,
                                              st.cache.c, st.q_block)
    assert e.value.status == dllm.DLLM_ERR_WORKSPACE_TOO_SMALL
