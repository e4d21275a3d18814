"""Host-side logic of the cache modes (no GPU): the batch layout of
prefix-only caching, the rows it feeds the projection, and the suffix refresh
schedule (Fast-dLLM page: "Python API" cache-mode knobs, "Suffix Cache
Refresh")."""
import numpy as np
import pytest
import torch

from block_wise_kv_gb300.inputs import Workload, layout, make_config
from block_wise_kv_gb300.step import refresh_due


def test_prefix_only_layout_covers_block_and_suffix():
    cfg = make_config("tiny").with_(t_prefix=[70, 200], gen_len=[192, 128], block=[32, 64], block_index=[1, 0],
                                    embedding=False, prefix_only=True)
    lay = layout(cfg)
    # C runs from the block start to the end of the sequence
    assert list(lay["block_start"]) == [102, 200]
    assert list(lay["block_len"]) == [262 - 102, 328 - 200]
    assert list(lay["cu_block"]) == [0, 160, 288]
    wl = Workload(cfg)
    for b in range(cfg.batch):
        rows = wl.block_rows(0, b, step=2)
        full = wl.seq_rows(0, b, step=2)
        assert rows.shape == (cfg.c_len(b), cfg.d_model)
        assert torch.equal(rows, full[cfg.block_start(b):])
    # DualCache: C is the block alone
    dual = cfg.with_(prefix_only=False)
    assert list(layout(dual)["block_len"]) == [32, 64]
    assert torch.equal(Workload(dual).block_rows(0, 0, step=2), wl.seq_rows(0, 0, step=2)[102:134])


def test_suffix_rows_vary_by_step_only_when_asked():
    base = make_config("tiny").with_(t_prefix=[64], gen_len=[128], block=[32], block_index=[1], embedding=False)
    s0 = 64 + 64  # first suffix row
    fixed = Workload(base)
    assert torch.equal(fixed.seq_rows(0, 0, step=0)[s0:], fixed.seq_rows(0, 0, step=3)[s0:])
    assert torch.equal(fixed.seq_rows(0, 0, step=0)[s0], fixed.seq_rows(0, 0, step=0)[-1])  # one shared mask row
    vary = Workload(base.with_(suffix_varies=True))
    a, b = vary.seq_rows(0, 0, step=0), vary.seq_rows(0, 0, step=3)
    assert not torch.equal(a[s0:], b[s0:])
    assert torch.equal(a[:64], b[:64])  # the prompt does not change within a block
    assert torch.equal(a, vary.seq_rows(0, 0, step=0))  # seeded


@pytest.mark.parametrize("r,due", [
    (None, []),
    (1, [1, 2, 3, 4, 5, 6, 7]),
    (2, [2, 4, 6]),
    (3, [3, 6]),
    (8, []),
])
def test_refresh_schedule(r, due):
    assert [s for s in range(8) if refresh_due(s, r)] == due


def test_refresh_interval_must_be_positive():
    with pytest.raises(ValueError):
        refresh_due(2, 0)
