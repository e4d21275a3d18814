"""Seeded synthetic inputs for the per-layer inner denoising step.

This module is the only piece shared by the CUDA path's tests/bench and the
oracle: it draws numbers and lays out the batch, and holds none of the
method's arithmetic.  Everything the parity checks use is generated on the
CPU with ``torch.Generator`` seeded through SplitMix64, so both sides see
identical bf16 values; the ``*_device`` variants draw the same layout and
distributions on a CUDA device, for throughput measurements only.

Workloads (named after the shapes they have):

* ``tiny``: 1 sequence, d_model 256, 4 heads x 64, RoPE theta 1e4, prompt 64,
  gen 256 = 8 blocks of 32, 4 inner steps per block.  Rows are embeddings of
  token ids (table N(0,1) [1024, 256], mask id 0, prompt ids uniform in
  1..1023, block ids re-drawn every inner step uniform in 0..1023).
* ``llada_single``: LLaDA-8B-shaped layer, 1 sequence, d_model 4096, 32 x 128,
  theta 5e5, prompt 512, gen 256, block 32, 8 inner steps per block.
* ``stack``: 32 independent LLaDA-8B-shaped layers, 16 sequences, prompt
  1024, gen 512, block 32, 16 inner steps.
* ``long``: 4 sequences, prompt 4096, gen 1024, block 64, 32 inner steps.
* ``ragged``: 32 sequences, prompt uniform in [128, 4096], gen in {256, 512},
  block in {16, 32, 64}, each at a random block index, pages shuffled.

Non-embedding workloads draw every row of x from N(0, 1) (bf16): prompt rows
per position, decoded blocks from the seed of their last inner step, the
current block from the seed of the current step, and every suffix row equal
to one shared "mask" row.  Weights are N(0, 0.02) bf16 and the RMSNorm gain
is 1.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np
import torch

_M64 = (1 << 64) - 1
PAGE = 64

# role ids folded into seeds
(_R_WEIGHT, _R_PROMPT, _R_BLOCK, _R_MASK, _R_EMBED, _R_IDS_PROMPT, _R_IDS_BLOCK, _R_SHAPE, _R_PAGES,
 _R_SUFFIX, _R_HIDDEN, _R_LM, _R_FFN) = range(1, 14)


def splitmix64(x: int) -> int:
    """One SplitMix64 output for state x (Steele, Lea & Flood 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & _M64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def derive_seed(*keys: int) -> int:
    s = 0x5EED
    for k in keys:
        s = splitmix64(s ^ (int(k) & _M64))
    return s & ((1 << 63) - 1)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(torch.bfloat16)


@dataclass
class Config:
    name: str
    d_model: int
    n_heads: int
    head_dim: int
    rope_theta: float
    t_prefix: list
    gen_len: list
    block: list
    block_index: list
    steps_per_block: int
    layers: int = 1
    rms_eps: float = 1e-5
    embedding: bool = False
    vocab: int = 1024
    mask_id: int = 0
    shuffle_pages: bool = True
    # Cache modes of the Fast-dLLM page: prefix-only caching recomputes every row after
    # the prefix at every inner step (the fresh region C is the current block and the
    # whole suffix); with suffix_varies the suffix rows change from one inner step to the
    # next (as the hidden states of masked positions do in deeper layers), which a suffix
    # refresh every r inner steps picks up.
    prefix_only: bool = False
    suffix_varies: bool = False
    spare_pages: int = 3
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.t_prefix)

    def seq_len(self, b: int) -> int:
        return self.t_prefix[b] + self.gen_len[b]

    def block_start(self, b: int, k: int | None = None) -> int:
        k = self.block_index[b] if k is None else k
        return self.t_prefix[b] + k * self.block[b]

    def c_len(self, b: int, k: int | None = None) -> int:
        """Rows of the fresh region C of sequence b at block k: the block, or
        (prefix-only) everything from the block start to the end."""
        if self.prefix_only:
            return self.seq_len(b) - self.block_start(b, k)
        return self.block[b]

    def num_blocks(self, b: int) -> int:
        return self.gen_len[b] // self.block[b]

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


def make_config(name: str, **overrides) -> Config:
    """The named workloads.  `overrides` replace fields (e.g. block_index)."""
    if name == "tiny":
        c = Config("tiny", 256, 4, 64, 1e4, [64], [256], [32], [0], 4, embedding=True)
    elif name == "llada_single":
        c = Config("llada_single", 4096, 32, 128, 5e5, [512], [256], [32], [0], 8)
    elif name == "stack":
        c = Config("stack", 4096, 32, 128, 5e5, [1024] * 16, [512] * 16, [32] * 16, [0] * 16, 16, layers=32)
    elif name == "long":
        c = Config("long", 4096, 32, 128, 5e5, [4096] * 4, [1024] * 4, [64] * 4, [0] * 4, 32)
    elif name == "ragged":
        g = np.random.default_rng(derive_seed(_R_SHAPE, 5))
        tp = [int(v) for v in g.integers(128, 4097, size=32)]
        gl = [int(v) for v in g.choice([256, 512], size=32)]
        bl = [int(v) for v in g.choice([16, 32, 64], size=32)]
        bi = [int(g.integers(0, gl[i] // bl[i])) for i in range(32)]
        c = Config("ragged", 4096, 32, 128, 5e5, tp, gl, bl, bi, 8)
    else:
        raise KeyError(name)
    if overrides:
        c = c.with_(**overrides)
    return c


class Workload:
    """Deterministic generator of weights, rows and the paged layout."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        self._embed = None

    # --------------------------------------------------------------- weights
    def weights(self, layer: int = 0):
        """(W_qkv bf16 [3*H*d, D] ~ N(0, 0.02), gain bf16 [D] = 1)."""
        c = self.cfg
        HD = c.n_heads * c.head_dim
        W = randn_bf16((3 * HD, c.d_model), derive_seed(c.seed, _R_WEIGHT, layer), std=0.02)
        g = torch.ones(c.d_model, dtype=torch.bfloat16)
        return W, g

    # ------------------------------------------------------------------ rows
    def _embedding(self) -> torch.Tensor:
        if self._embed is None:
            c = self.cfg
            self._embed = randn_bf16((c.vocab, c.d_model), derive_seed(c.seed, _R_EMBED))
        return self._embed

    def _rows_prompt(self, layer: int, b: int) -> torch.Tensor:
        c = self.cfg
        if c.embedding:
            ids = torch.randint(1, c.vocab, (c.t_prefix[b],), generator=_gen(derive_seed(c.seed, _R_IDS_PROMPT, b)))
            return self._embedding()[ids]
        return randn_bf16((c.t_prefix[b], c.d_model), derive_seed(c.seed, _R_PROMPT, layer, b))

    def _rows_block(self, layer: int, b: int, k: int, step: int) -> torch.Tensor:
        c = self.cfg
        if c.embedding:
            ids = torch.randint(0, c.vocab, (c.block[b],), generator=_gen(derive_seed(c.seed, _R_IDS_BLOCK, b, k, step)))
            return self._embedding()[ids]
        return randn_bf16((c.block[b], c.d_model), derive_seed(c.seed, _R_BLOCK, layer, b, k, step))

    def _row_mask(self, layer: int, b: int) -> torch.Tensor:
        c = self.cfg
        if c.embedding:
            return self._embedding()[c.mask_id:c.mask_id + 1]
        return randn_bf16((1, c.d_model), derive_seed(c.seed, _R_MASK, layer, b))

    def seq_rows(self, layer: int, b: int, k: int | None = None, step: int = 0) -> torch.Tensor:
        """Every row [N_b, D] of sequence b while block k is at inner step
        `step`: prompt | decoded blocks (their last step) | block k (this
        step) | mask rows."""
        c = self.cfg
        k = c.block_index[b] if k is None else k
        parts = [self._rows_prompt(layer, b)]
        for j in range(k):
            parts.append(self._rows_block(layer, b, j, c.steps_per_block - 1))
        parts.append(self._rows_block(layer, b, k, step))
        n_suffix = c.gen_len[b] - (k + 1) * c.block[b]
        if n_suffix > 0:
            parts.append(self._rows_suffix(layer, b, k, step, n_suffix))
        return torch.cat(parts, dim=0).contiguous()

    def _rows_suffix(self, layer: int, b: int, k: int, step: int, n: int) -> torch.Tensor:
        c = self.cfg
        if c.suffix_varies:
            return randn_bf16((n, c.d_model), derive_seed(c.seed, _R_SUFFIX, layer, b, k, step))
        return self._row_mask(layer, b).expand(n, c.d_model)

    def block_rows(self, layer: int, b: int, k: int | None = None, step: int = 0) -> torch.Tensor:
        """The rows of C: the block's rows at this inner step, followed (prefix-only)
        by the suffix rows."""
        c = self.cfg
        k = c.block_index[b] if k is None else k
        if c.prefix_only:
            return self.seq_rows(layer, b, k, step)[c.block_start(b, k):].contiguous()
        return self._rows_block(layer, b, k, step).contiguous()

    def batch_rows(self, layer: int = 0, step: int = 0, blocks=None):
        """(x_full [R, D], x_block [M, D]) packed in sequence order."""
        c = self.cfg
        blocks = c.block_index if blocks is None else blocks
        full = [self.seq_rows(layer, b, blocks[b], step) for b in range(c.batch)]
        blk = [self.block_rows(layer, b, blocks[b], step) for b in range(c.batch)]
        return torch.cat(full, 0).contiguous(), torch.cat(blk, 0).contiguous()

    # ------------------------------------------------- device-drawn variants
    # The same layout and distributions drawn on a CUDA device by a seeded device
    # generator, for throughput measurements at sizes where drawing on the CPU
    # takes minutes (the 32-layer stack holds 25 k rows x 4096 per layer).  The
    # values differ from the CPU draws above, which the parity tests use.
    def weights_device(self, layer: int, device) -> tuple:
        c = self.cfg
        HD = c.n_heads * c.head_dim
        g = torch.Generator(device=device)
        g.manual_seed(derive_seed(c.seed, _R_WEIGHT, layer))
        W = (torch.randn(3 * HD, c.d_model, generator=g, device=device) * 0.02).to(torch.bfloat16)
        return W, torch.ones(c.d_model, dtype=torch.bfloat16, device=device)

    def batch_rows_device(self, layer: int, step: int, blocks, device) -> tuple:
        """(x_full [R, D], x_block [M, D]) on the device, packed in sequence
        order: per sequence prompt | decoded blocks | block (this step) | the
        shared mask row repeated over the suffix."""
        c = self.cfg
        if c.embedding:
            full, blk = self.batch_rows(layer, step, blocks)
            return full.to(device), blk.to(device)
        full, blk = [], []
        for b in range(c.batch):
            g = torch.Generator(device=device)
            g.manual_seed(derive_seed(c.seed, _R_PROMPT, layer, b, blocks[b], step))
            k = blocks[b]
            s0 = c.t_prefix[b] + k * c.block[b]
            head = torch.randn(s0 + c.block[b], c.d_model, generator=g, device=device).to(torch.bfloat16)
            mask = torch.randn(1, c.d_model, generator=g, device=device).to(torch.bfloat16)
            n_suffix = c.gen_len[b] - (k + 1) * c.block[b]
            full.append(torch.cat([head, mask.expand(n_suffix, c.d_model)], 0))
            blk.append(full[-1][s0:] if c.prefix_only else head[s0:])
        return torch.cat(full, 0).contiguous(), torch.cat(blk, 0).contiguous()

    # ------------------------------------------------- block-only epilogue
    def lm_inputs(self, vocab: int, gain_spread: float = 0.0):
        """(h_full [R, D] ~ N(0, 1) bf16: the final hidden states of every row, packed in
        sequence order; final RMSNorm gain bf16 [D] (1, or uniform in 1 +- gain_spread);
        W_lm [vocab, D] ~ N(0, 0.02) bf16: a synthetic LM head)."""
        c = self.cfg
        R = sum(c.seq_len(b) for b in range(c.batch))
        h = randn_bf16((R, c.d_model), derive_seed(c.seed, _R_HIDDEN))
        g = torch.ones(c.d_model)
        if gain_spread > 0:
            u = torch.rand(c.d_model, generator=_gen(derive_seed(c.seed, _R_HIDDEN, 1)))
            g = 1.0 + gain_spread * (2 * u - 1)
        W = randn_bf16((vocab, c.d_model), derive_seed(c.seed, _R_LM, vocab), std=0.02)
        return h, g.to(torch.bfloat16), W

    # ------------------------------------------------- rest of the layer (FFN)
    def ffn_inputs(self, d_ff: int):
        """Inputs of the rest of the layer for the current blocks' rows: o_full [R, H d]
        bf16 ~ N(0, 0.25) (the attention output of every row), x_block [M, D] bf16 ~ N(0, 1)
        (the layer input of the block rows, packed by cu_block), W_o [D, H d] ~ N(0, 0.02)
        bf16, the FFN gain (ones), and the e4m3 weights: W_gate_up codes [2 d_ff, D] (rows
        2j gate, 2j + 1 up) with fp32 scales [2 d_ff / 128, D / 128], W_down codes [D, d_ff]
        with scales [D / 128, d_ff / 128].  Codes are random bytes: random sign, exponent
        field uniform in 1..14 (no NaN code), mantissa uniform; scales uniform in
        [1e-4, 3e-4]."""
        c = self.cfg
        R = sum(c.seq_len(b) for b in range(c.batch))
        M = sum(c.c_len(b) for b in range(c.batch))
        HD, D = c.n_heads * c.head_dim, c.d_model
        o = randn_bf16((R, HD), derive_seed(c.seed, _R_FFN, 1), std=0.5)
        x = randn_bf16((M, D), derive_seed(c.seed, _R_FFN, 2))
        Wo = randn_bf16((D, HD), derive_seed(c.seed, _R_FFN, 3), std=0.02)
        g2 = torch.ones(D, dtype=torch.bfloat16)

        def codes(rows, cols, key):
            gen = _gen(derive_seed(c.seed, _R_FFN, key))
            sign = torch.randint(0, 2, (rows, cols), generator=gen, dtype=torch.int32)
            expo = torch.randint(1, 15, (rows, cols), generator=gen, dtype=torch.int32)
            mant = torch.randint(0, 8, (rows, cols), generator=gen, dtype=torch.int32)
            return ((sign << 7) | (expo << 3) | mant).to(torch.uint8)

        def scales(rows, cols, key):
            return torch.empty(rows // 128, cols // 128).uniform_(1e-4, 3e-4,
                                                                   generator=_gen(derive_seed(c.seed, _R_FFN, key)))

        return dict(o_full=o, x_block=x, w_o=Wo, gain2=g2, w_gu=codes(2 * d_ff, D, 4), gu_scale=scales(2 * d_ff, D, 5),
                    w_down=codes(D, d_ff, 6), down_scale=scales(D, d_ff, 7))

    # ---------------------------------------------------------------- layout
    def page_lists(self):
        """Physical page ids of each sequence (a seeded permutation of the
        pool's pages when shuffle_pages), and the pool size."""
        c = self.cfg
        need = [(c.seq_len(b) + PAGE - 1) // PAGE for b in range(c.batch)]
        total = sum(need) + c.spare_pages
        if c.shuffle_pages:
            perm = np.random.default_rng(derive_seed(c.seed, _R_PAGES)).permutation(total)
        else:
            perm = np.arange(total)
        out, at = [], 0
        for n in need:
            out.append([int(p) for p in perm[at:at + n]])
            at += n
        return out, total


def layout(cfg: Config, blocks=None):
    """Host-side metadata of the batch as int32 numpy arrays: block_table
    [batch, max_pages] (unused entries -1), seq_len, block_start, block_len,
    cu_block, cu_seq, and num_pages."""
    wl = Workload(cfg)
    blocks = cfg.block_index if blocks is None else blocks
    pages, total = wl.page_lists()
    B = cfg.batch
    maxp = max((len(p) for p in pages), default=1)
    bt = np.full((B, max(maxp, 1)), -1, dtype=np.int32)
    for b, pl in enumerate(pages):
        bt[b, :len(pl)] = pl
    seq_len = np.array([cfg.seq_len(b) for b in range(B)], dtype=np.int32)
    bstart = np.array([cfg.block_start(b, blocks[b]) for b in range(B)], dtype=np.int32)
    blen = np.array([cfg.c_len(b, blocks[b]) for b in range(B)], dtype=np.int32)
    cu_block = np.concatenate([[0], np.cumsum(blen)]).astype(np.int32)
    cu_seq = np.concatenate([[0], np.cumsum(seq_len)]).astype(np.int32)
    return dict(block_table=bt, seq_len=seq_len, block_start=bstart, block_len=blen, cu_block=cu_block,
                cu_seq=cu_seq, num_pages=total)
