"""The bench's algorithmic bytes and flops (the denominators of every roofline
fraction), without a GPU: counted here tensor by tensor for the 32-layer stack
workload and for a ragged layout, against bench.step_bytes_flops."""
from types import SimpleNamespace

import numpy as np

import bench
from block_wise_kv_gb300.inputs import layout, make_config


def _state(cfg):
    return SimpleNamespace(batch=SimpleNamespace(host=layout(cfg)))


def _counted(cfg):
    """Bytes the step must move and flops it must do, one tensor or product at a time."""
    D, H, d = cfg.d_model, cfg.n_heads, cfg.head_dim
    bf16, fp16, fp32 = 2, 2, 4
    seqs = [(cfg.seq_len(b), cfg.c_len(b)) for b in range(cfg.batch)]
    M = sum(B for _, B in seqs)
    qkv = {"W_qkv": 3 * H * d * D * bf16, "x_block": M * D * bf16, "q_block": M * H * d * bf16,
           "k rows": M * H * d * bf16, "v rows": M * H * d * bf16}
    att = {"K pages": sum(N for N, _ in seqs) * H * d * bf16, "V pages": sum(N for N, _ in seqs) * H * d * bf16,
           "q_block": M * H * d * bf16, "O block rows": M * H * d * bf16}
    nu = sum(N - B for N, B in seqs)
    mrg = {"q_pool": nu * H * d * bf16, "O~/l": nu * H * d * fp16, "O rows": nu * H * d * bf16,
           "m": nu * H * fp32, "l": nu * H * fp32}
    flops = {"qkv": 2 * M * D * 3 * H * d,
             "attention": sum(2 * 2 * B * N * H * d for N, B in seqs),  # Q K^T and P V over all N keys
             "merge": sum(2 * 2 * (N - B) * B * H * d for N, B in seqs)}  # U rows over the B block keys
    return {"qkv": (sum(qkv.values()), flops["qkv"]), "attention": (sum(att.values()), flops["attention"]),
            "merge": (sum(mrg.values()), flops["merge"])}


def test_stack_figures():
    cfg = make_config("stack")
    got = bench.step_bytes_flops(cfg, _state(cfg))
    assert got == _counted(cfg)
    assert got["qkv"] == (117_440_512, 51_539_607_552)  # 117.4 MB, 51.5 GF
    assert got["attention"][0] + got["merge"][0] == 1_008_599_040  # a5 + a6: 1.009 GB


def test_ragged_layout():
    cfg = make_config("ragged")
    got = bench.step_bytes_flops(cfg, _state(cfg))
    assert got == _counted(cfg)
    assert np.isclose(got["attention"][0] + got["merge"][0], 3_492_462_336, rtol=0)
