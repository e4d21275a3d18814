"""Device state of one layer for one ragged batch, and the call sequence of
a block boundary and of an inner denoising step through the C ABI.

Nothing here computes: it allocates with torch, fills the C structs and
calls ``dllm_*`` in the order the method defines (Fast-dLLM DualCache,
"Building the Dual Cache Manually": the cache is built at each block
boundary, then every inner step runs on the block rows only).
"""
from __future__ import annotations

import torch

from . import dllm
from .inputs import Config, Workload, layout


class LayerStep:
    """One layer's weights, RoPE table, paged cache, workspaces and outputs
    for the batch layout of `cfg` (block k_b of each sequence)."""

    def __init__(self, cfg: Config, layer: int = 0, blocks=None, device: str = "cuda", cache_fill=None,
                 weights=None, rope_max_pos: int | None = None, pre: bool = False):
        self.cfg = cfg
        self.device = device
        wl = Workload(cfg)
        W, g = weights if weights is not None else wl.weights(layer)
        self.gain = g.to(device).contiguous()
        lay = layout(cfg, blocks)
        self.host_layout = lay
        self.batch = dllm.BatchLayout(lay["block_table"], lay["seq_len"], lay["block_start"], lay["block_len"],
                                      device=device)
        self.desc = dllm.layer_desc(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.rope_theta, cfg.rms_eps)
        # the projection calls read the weight in its tile-packed form
        self.w_qkv = dllm.pack_qkv_weight(self.desc, W.to(device))
        self.rope_max_pos = int(rope_max_pos or self.batch.max_seq_len)
        self.rope = torch.empty(self.rope_max_pos, cfg.head_dim // 2, 2, dtype=torch.float32, device=device)
        dllm.dllm_rope_table_build(self.desc, self.rope_max_pos, self.rope)
        self.cache = dllm.PagedCache(lay["num_pages"], cfg.n_heads, cfg.head_dim, device=device, fill=cache_fill,
                                     pre=pre)
        self.ws_build = dllm.workspace(dllm.dllm_workspace_size(self.desc, self.batch.c, dllm.DLLM_OP_CACHE_BUILD),
                                       device)
        self._block_buffers()
        H, d = cfg.n_heads, cfg.head_dim
        self.o_full = torch.zeros(self.batch.total_seq_rows, H, d, dtype=torch.bfloat16, device=device)
        self.lse = torch.zeros(self.batch.total_seq_rows, H, dtype=torch.float32, device=device)

    def _block_buffers(self) -> None:
        """q_block and the step workspaces, sized for the current blocks."""
        cfg, device = self.cfg, self.device
        self.ws_step = dllm.workspace(
            dllm.dllm_workspace_size(self.desc, self.batch.c, dllm.DLLM_OP_BLOCK_QKV_ROPE_WRITE), device)
        # the attention calls of a step run in order, so one workspace serves all three
        self.ws_attn = dllm.workspace(max(
            dllm.dllm_workspace_size(self.desc, self.batch.c, op)
            for op in (dllm.DLLM_OP_BLOCK_ATTENTION, dllm.DLLM_OP_STATE_MERGE, dllm.DLLM_OP_STEP_ATTENTION)), device)
        self.q_block = torch.zeros(self.batch.total_block_rows, cfg.n_heads, cfg.head_dim, dtype=torch.bfloat16,
                                   device=device)

    # ------------------------------------------------------------ the calls
    def boundary(self, x_full: torch.Tensor, stream=None) -> None:
        dllm.dllm_cache_build(self.desc, self.batch.c, x_full, self.gain, self.w_qkv, self.rope, self.rope_max_pos,
                              self.cache.c, self.ws_build, stream)

    def advance(self, blocks, x_decoded: torch.Tensor, stream=None) -> None:
        """Incremental boundary to the blocks `blocks` (one block index per
        sequence, each starting where the current block ends): the current
        blocks are the decoded ones, x_decoded their final rows.  Needs the
        prefix state pools (pre=True) and a cache built by boundary() and
        advance() calls only."""
        old = self.batch.host
        lay = layout(self.cfg, blocks)
        dec_start = old["block_start"]
        dec_len = lay["block_start"] - dec_start
        if (dec_len <= 0).any():
            raise ValueError("each new block must start after the current one's start")
        new = dllm.BatchLayout(lay["block_table"], lay["seq_len"], lay["block_start"], lay["block_len"],
                               device=self.device)
        dec = new.with_blocks(dec_start, dec_len)
        ws = dllm.workspace(dllm.dllm_workspace_size(self.desc, dec.c, dllm.DLLM_OP_CACHE_ADVANCE), self.device)
        dllm.dllm_cache_advance(self.desc, new.c, dec.c, x_decoded, self.gain, self.w_qkv, self.rope,
                                self.rope_max_pos, self.cache.c, ws, stream)
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        self._advanced = (new, dec, ws)  # alive until the next advance
        self.batch, self.host_layout = new, lay
        self._block_buffers()

    def qkv(self, x_block: torch.Tensor, stream=None) -> None:
        dllm.dllm_block_qkv_rope_write(self.desc, self.batch.c, x_block, self.gain, self.w_qkv, self.rope,
                                       self.rope_max_pos, self.cache.c, self.q_block, self.ws_step, stream)

    def attention(self, stream=None, lse: bool = True) -> None:
        dllm.dllm_block_attention(self.desc, self.batch.c, self.q_block, self.cache.c, self.o_full,
                                  self.lse if lse else None, self.ws_attn, stream)

    def merge(self, stream=None, lse: bool = True) -> None:
        dllm.dllm_state_merge(self.desc, self.batch.c, self.cache.c, self.o_full, self.lse if lse else None,
                              self.ws_attn, stream)

    def step_attention(self, stream=None, lse: bool = True) -> None:
        dllm.dllm_step_attention(self.desc, self.batch.c, self.q_block, self.cache.c, self.o_full,
                                 self.lse if lse else None, self.ws_attn, stream)

    def step(self, x_block: torch.Tensor, stream=None, lse: bool = True, split: bool = False) -> None:
        """One inner denoising step of this layer: fused projection, then the
        block attention and the FACache merge for the invariant rows in one
        launch (`split`: as the two separate calls instead)."""
        self.qkv(x_block, stream)
        if split:
            self.attention(stream, lse)
            self.merge(stream, lse)
        else:
            self.step_attention(stream, lse)

    def inner_step(self, step: int, x_block: torch.Tensor, x_full: torch.Tensor | None = None,
                   refresh_interval: int | None = None, stream=None, lse: bool = True) -> bool:
        """Inner step `step` (0-based) of the current block with the suffix
        refresh schedule of the Fast-dLLM page ("Suffix Cache Refresh"): with
        refresh_interval = r the cache is rebuilt from the rows of this step
        (x_full) before the steps r, 2r, ... of the block; with None only the
        block boundary builds it (the caller's boundary() before step 0).
        Returns whether the cache was rebuilt."""
        due = refresh_due(step, refresh_interval)
        if due:
            if x_full is None:
                raise ValueError(f"inner step {step} refreshes the cache: x_full is needed")
            self.boundary(x_full, stream)
        self.step(x_block, stream, lse)
        return due

    # ---------------------------------------------------------- inspection
    def seq_slice(self, b: int) -> slice:
        cu = self.batch.host["cu_seq"]
        return slice(int(cu[b]), int(cu[b + 1]))

    def block_slice(self, b: int) -> slice:
        cu = self.batch.host["cu_block"]
        return slice(int(cu[b]), int(cu[b + 1]))

    def pool_rows(self, pool: torch.Tensor, b: int) -> torch.Tensor:
        n = int(self.batch.host["seq_len"][b])
        return dllm.gather_rows(pool, self.batch.host["block_table"], b, n)


def refresh_due(step: int, refresh_interval: int | None) -> bool:
    """Whether inner step `step` (> 0) of a block rebuilds the cache first:
    every r-th step for refresh_interval = r, never for None (the block
    boundary, before step 0, always builds it)."""
    if refresh_interval is None:
        return False
    if refresh_interval < 1:
        raise ValueError("refresh_interval must be >= 1 or None")
    return step > 0 and step % refresh_interval == 0


def block_rows_of(wl: Workload, layer: int, step: int, blocks) -> torch.Tensor:
    cfg = wl.cfg
    return torch.cat([wl.block_rows(layer, b, blocks[b], step) for b in range(cfg.batch)], 0).contiguous()


def full_rows_of(wl: Workload, layer: int, step: int, blocks) -> torch.Tensor:
    cfg = wl.cfg
    return torch.cat([wl.seq_rows(layer, b, blocks[b], step) for b in range(cfg.batch)], 0).contiguous()


__all__ = ["LayerStep", "block_rows_of", "full_rows_of", "refresh_due"]
