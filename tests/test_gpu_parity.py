"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle.

Every test runs the block boundary (dllm_cache_build) and inner steps on
seeded synthetic inputs and compares all rows' outputs with the oracle's full
recompute of the same step.  An inner step is dllm_block_qkv_rope_write then
dllm_step_attention (the block attention and the FACache merge in one
launch); test_split_calls_match_oracle_and_fused runs dllm_block_attention
and dllm_state_merge as two separate calls instead, and checks them against
the oracle and bit for bit against the fused call.
"""
import numpy as np
import pytest
import torch

from block_wise_kv_gb300 import dllm
from block_wise_kv_gb300.inputs import Config, Workload, make_config
from block_wise_kv_gb300.step import LayerStep, block_rows_of, full_rows_of
from parity_util import assert_bf16_close, assert_close, oracle_cache_state, oracle_step, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from block_wise_kv_gb300 import build

    build.build()
    dllm.load()
    torch.cuda.init()


def _run_block(cfg: Config, k_of, steps, layer=0, check_cache=True, check_qkv=True, rows_of=None, seqs=None,
               gain=None, split=False):
    """Boundary of the blocks `k_of` (one per sequence) then the given inner
    steps; every listed sequence is compared with the oracle after each step.
    `gain` replaces the workload's RMSNorm gain (all ones); `split` runs the
    attention as the two separate calls."""
    wl = Workload(cfg)
    W, g = wl.weights(layer)
    if gain is not None:
        g = gain
    st = LayerStep(cfg, layer=layer, blocks=k_of, weights=(W, g))
    st.boundary(full_rows_of(wl, layer, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0
    seqs = range(cfg.batch) if seqs is None else seqs
    H, d = cfg.n_heads, cfg.head_dim
    if check_cache:
        for b in seqs:
            U, m, l, Ot = oracle_cache_state(wl, layer, b, k_of[b], W, g)
            if len(U) == 0:
                continue
            gm = to_np(st.pool_rows(st.cache.m, b))[U]
            gl = to_np(st.pool_rows(st.cache.l, b))[U]
            go = to_np(st.pool_rows(st.cache.o, b))[U]
            assert_close(gm, m, f"cache m seq {b}", max_abs=2e-2, rel=1e-3)
            assert_close(gl / np.exp(m - gm), l, f"cache l seq {b}", max_abs=np.inf, rel=5e-3)
            assert_close(go, Ot / l[..., None], f"cache O~/l seq {b}")
    for s in steps:
        st.step(block_rows_of(wl, layer, s, k_of).cuda(), split=split)
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        for b in seqs:
            rows = None if rows_of is None else rows_of(b)
            ref = oracle_step(wl, layer, b, k_of[b], s, rows=rows, W=W, g=g)
            o = to_np(st.o_full[st.seq_slice(b)])
            lse = to_np(st.lse[st.seq_slice(b)])
            sel = slice(None) if rows is None else rows
            assert_close(o[sel], ref["O"], f"O seq {b} block {k_of[b]} step {s}")
            assert_close(lse[sel], ref["L"], f"LSE seq {b} step {s}", max_abs=2e-2, rel=1e-3)
            if check_qkv:
                c0 = cfg.block_start(b, k_of[b])
                blk = slice(c0, c0 + cfg.c_len(b, k_of[b]))
                kk = to_np(st.pool_rows(st.cache.k, b))
                vv = to_np(st.pool_rows(st.cache.v, b))
                assert_bf16_close(kk[blk], ref["k"][blk], f"k block rows seq {b}")
                assert_bf16_close(vv[blk], ref["v"][blk], f"v block rows seq {b}")
                if rows is None:
                    qb = to_np(st.q_block[st.block_slice(b)])
                    assert_bf16_close(qb, ref["q"][blk], f"q_block seq {b}")
    return st


def test_tiny_every_block_every_step():
    cfg = make_config("tiny")
    for k in range(cfg.num_blocks(0)):
        _run_block(cfg, [k], range(cfg.steps_per_block))


def test_rmsnorm_rows_and_scales_in_the_workspace():
    """The fused projection writes, per token row, its RMSNorm scale
    1 / sqrt(mean(x^2) + eps) as a float pair (hi, lo) and the bf16 operand
    x^ into its workspace (after the 1 KB of counters): hi + lo equals the
    fp64 value to ~2^-38, x^ equals the oracle's x^ rounded to bf16 bit for
    bit, and the claim counters are back at zero."""
    import oracle as orc

    cfg = make_config("llada_single")
    wl = Workload(cfg)
    st = LayerStep(cfg)
    for step in (3, 4):
        xb = block_rows_of(wl, 0, step, cfg.block_index)
        st.qkv(xb.cuda())
        torch.cuda.synchronize()
        M, D = xb.shape
        pairs = st.ws_step[4096:4096 + M * 8].view(torch.float32).view(M, 2).double().cpu().numpy()
        x = xb.double().numpy()
        want = 1.0 / np.sqrt((x * x).mean(axis=1) + cfg.rms_eps)
        assert np.max(np.abs((pairs[:, 0] + pairs[:, 1]) / want - 1.0)) < 2.0 ** -38
        off = 4096 + 256 * ((M * 8 + 255) // 256)
        got = st.ws_step[off:off + M * D * 2].view(torch.bfloat16).view(M, D).double().cpu().numpy()
        xh = orc.bf16_round(orc.rmsnorm(x, st.gain.double().cpu().numpy(), cfg.rms_eps))
        assert np.array_equal(got, xh), f"{int((got != xh).sum())} elements of x^ differ"
        assert int(st.ws_step[:4096].view(torch.int32).abs().sum()) == 0, "counters left non-zero"


def test_weight_pack_is_the_documented_permutation():
    """Tile-packed weight: box (t, kb) of 128 rows x 64 columns stored
    contiguously, 2*ceil(D/128) boxes per tile, zeros past d_model; checked
    bit for bit against a host reordering (d_model % 128 == 64 included)."""
    for D, H, d in ((192, 2, 64), (256, 4, 64), (512, 2, 128)):
        desc = dllm.layer_desc(D, H, d, 1e4)
        g = torch.Generator().manual_seed(D)
        W = torch.randn(3 * H * d, D, generator=g).to(torch.bfloat16)
        got = dllm.pack_qkv_weight(desc, W.cuda()).cpu().view(torch.int16).numpy()
        kbp = 2 * ((D + 127) // 128)
        Wp = np.zeros((3 * H * d, kbp * 64), dtype=np.int16)
        Wp[:, :D] = W.view(torch.int16).numpy()
        want = Wp.reshape(3 * H * d // 128, 128, kbp, 64).transpose(0, 2, 1, 3).reshape(-1)
        assert np.array_equal(got, want), (D, H, d)


def test_llada_single_every_block_first_and_last_step():
    cfg = make_config("llada_single")
    for k in range(cfg.num_blocks(0)):
        _run_block(cfg, [k], (0, cfg.steps_per_block - 1), check_cache=(k in (0, 3, cfg.num_blocks(0) - 1)))


def _mini_ragged(**kw):
    # edge cases: empty prefix, last block (empty suffix), page-unaligned
    # blocks, blocks straddling pages, partial last pages, odd block sizes,
    # a sequence made of its block only (no invariant rows).
    return Config("mini_ragged", 256, 4, 64, 1e4,
                  t_prefix=[0, 100, 37, 10, 300, 5, 0, 64],
                  gen_len=[64, 96, 128, 64, 240, 20, 32, 128],
                  block=[32, 32, 16, 64, 48, 20, 32, 64],
                  block_index=[0, 2, 3, 0, 1, 0, 0, 1],
                  steps_per_block=2).with_(**kw)


def test_mini_ragged_edge_cases():
    cfg = _mini_ragged()
    _run_block(cfg, cfg.block_index, (0, 1))


def test_mini_ragged_head_dim_128():
    cfg = _mini_ragged(d_model=512, n_heads=2, head_dim=128, rope_theta=5e5)
    _run_block(cfg, cfg.block_index, (1,))


def test_split_calls_match_oracle_and_fused():
    """dllm_block_attention (block rows) and dllm_state_merge (invariant rows)
    called separately run their own launch plans (every CTA in one role); the
    rows they write match the oracle, and the fused dllm_step_attention on the
    same inputs gives the same bytes (each (sequence, head) and each page is
    computed whole by one CTA in either plan)."""
    cases = [(make_config("tiny"), [2], (1,)), (make_config("tiny"), [7], (3,)),
             (_mini_ragged(), None, (1,)),
             (_mini_ragged(d_model=512, n_heads=2, head_dim=128, rope_theta=5e5), None, (0,)),
             (make_config("llada_single"), [5], (7,))]
    for cfg, k_of, steps in cases:
        k_of = list(cfg.block_index) if k_of is None else k_of
        st = _run_block(cfg, k_of, steps, check_cache=False, check_qkv=False, split=True)
        split_out = (st.o_full.clone(), st.lse.clone())
        st.o_full.zero_()
        st.lse.zero_()
        wl = Workload(cfg)
        st.step(block_rows_of(wl, 0, steps[-1], k_of).cuda())
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        assert torch.equal(split_out[0].view(torch.int16), st.o_full.view(torch.int16)), cfg.name
        assert torch.equal(split_out[1].view(torch.int32), st.lse.view(torch.int32)), cfg.name


def test_rmsnorm_gain_not_one():
    """A random RMSNorm gain (the workloads use g = 1): the fused projection
    applies g[k] to the right K position of every swizzled x tile, also in a
    ragged last K unit (d_model 192 = 1.5 units) and with token tiles of 128,
    64 and 32 rows."""
    for name, d_model, H, d, t_prefix, gen_len, block, k_of in (
            ("gain_ragged_k", 192, 2, 64, [0, 100, 37, 10, 300, 5, 0, 64], [64, 96, 128, 64, 240, 20, 32, 128],
             [32, 32, 16, 64, 48, 20, 32, 64], [0, 2, 3, 0, 1, 0, 0, 1]),
            ("gain_bn64", 512, 2, 128, [100, 5], [96, 40], [32, 20], [1, 1]),
            ("gain_bn32", 1024, 4, 64, [37, 0], [48, 32], [16, 16], [2, 0])):
        cfg = Config(name, d_model, H, d, 1e4, t_prefix=t_prefix, gen_len=gen_len, block=block, block_index=k_of,
                     steps_per_block=2)
        gen = torch.Generator().manual_seed(d_model)
        gain = (0.5 + torch.rand(d_model, generator=gen)).to(torch.bfloat16)
        _run_block(cfg, cfg.block_index, (1,), gain=gain)


def test_split_stream_k_tiles_and_repeatability():
    """Few weight tiles (2 heads x 128 -> 6 tiles) with d_model 4096 and at
    most 64 block rows: the projection splits each tile's K range over
    several CTAs (fp32 partial tiles summed by the last contributor), with
    token tiles of 64 and of 32 rows; the results
    match the oracle, and the same step run again on the same inputs gives
    bit-identical outputs (fixed summation orders)."""
    for name, t_prefix, gen_len, block, k_of in (("split64", [100, 5], [96, 40], [32, 20], [1, 1]),
                                                  ("split32", [37, 0], [48, 32], [16, 16], [2, 0])):
        cfg = Config(name, 4096, 2, 128, 5e5, t_prefix=t_prefix, gen_len=gen_len, block=block, block_index=k_of,
                     steps_per_block=2)
        st = _run_block(cfg, cfg.block_index, (1,))
        M = sum(block)
        plain = 4096 + 256 * ((M * 8 + 255) // 256) + 256 * ((M * 4096 * 2 + 255) // 256)
        assert st.ws_step.numel() > plain, "expected the split schedule (partials)"
        wl = Workload(cfg)
        xb = block_rows_of(wl, 0, 1, cfg.block_index).cuda()
        first = (st.o_full.clone(), st.lse.clone(), st.q_block.clone(), st.cache.k.clone(), st.cache.v.clone())
        for _ in range(3):
            st.step(xb)
            torch.cuda.synchronize()
            again = (st.o_full, st.lse, st.q_block, st.cache.k, st.cache.v)
            for x, y in zip(first, again):
                iv = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
                assert torch.equal(x.view(iv), y.view(iv)), name
        assert int(st.ws_step[:4096].view(torch.int32).abs().sum()) == 0, "arrival counters left non-zero"


def test_placement_is_bit_exact_and_sentinels_survive():
    """A shuffled physical page order (with a consistent block table) gives
    byte-identical outputs and gathered cache contents; pages no sequence
    owns keep their sentinel."""
    outs = []
    for shuffle in (False, True):
        cfg = _mini_ragged(shuffle_pages=shuffle, spare_pages=5)
        wl = Workload(cfg)
        st = LayerStep(cfg, cache_fill=3.0)
        k_of = cfg.block_index
        st.boundary(full_rows_of(wl, 0, 0, k_of).cuda())
        st.step(block_rows_of(wl, 0, 1, k_of).cuda())
        torch.cuda.synchronize()
        assert st.batch.error_bits() == 0
        gathered = {}
        for b in range(cfg.batch):
            n = cfg.seq_len(b)
            s0, e0 = cfg.block_start(b), cfg.block_start(b) + cfg.block[b]
            U = np.r_[0:s0, e0:n]
            for name in ("k", "v"):
                gathered[(name, b)] = st.pool_rows(getattr(st.cache, name), b).cpu()
            for name in ("q", "m", "l", "o"):
                gathered[(name, b)] = st.pool_rows(getattr(st.cache, name), b).cpu()[U]
        used = set(int(p) for p in st.host_layout["block_table"].ravel() if p >= 0)
        spare = [p for p in range(st.cache.num_pages) if p not in used]
        assert len(spare) == 5
        for name in ("k", "v", "q", "m", "l", "o"):
            pool = getattr(st.cache, name)[spare]
            assert torch.all(pool == 3.0), f"spare pages of {name}_pool were written"
        outs.append((st.o_full.cpu(), st.lse.cpu(), st.q_block.cpu(), gathered))
    (o0, l0, q0, g0), (o1, l1, q1, g1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    assert torch.equal(q0.view(torch.int16), q1.view(torch.int16))
    for key in g0:
        a, b = g0[key], g1[key]
        iv = torch.int16 if a.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(a.contiguous().view(iv), b.contiguous().view(iv)), key


def test_bad_block_table_entry_is_reported_not_faulted():
    cfg = _mini_ragged()
    wl = Workload(cfg)
    st = LayerStep(cfg)
    k_of = cfg.block_index
    st.boundary(full_rows_of(wl, 0, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() == 0
    # corrupt one entry on the device: every kernel must skip or clamp it
    st.batch.dev["block_table"][1, 0] = st.cache.num_pages + 7
    st.step(block_rows_of(wl, 0, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() & dllm.DLLM_DEVERR_BAD_PAGE
    # inconsistent metadata: a block that runs past the end of its sequence
    st.batch.error.zero_()
    st.batch.dev["block_table"][1, 0] = int(st.host_layout["block_table"][1, 0])
    st.batch.dev["block_start"][2] = cfg.seq_len(2)
    st.step(block_rows_of(wl, 0, 0, k_of).cuda())
    torch.cuda.synchronize()
    assert st.batch.error_bits() & dllm.DLLM_DEVERR_BAD_SHAPE
    torch.cuda.synchronize()


def test_state_beyond_fp16_range_is_flagged():
    """The cached O~ / l is stored as fp16; it is a convex combination of value
    rows, so only values beyond 65504 in magnitude can take it out of range, and
    the state build flags that instead of storing it silently."""
    cfg = _mini_ragged()
    wl = Workload(cfg)
    W, g = wl.weights(0)
    HD = cfg.n_heads * cfg.head_dim
    for scale, flagged in ((1.0, False), (2.0 ** 24, True)):  # v ~ N(0, (0.02 sqrt(D) scale)^2)
        Ws = W.clone()
        Ws[2 * HD:] *= scale  # exact in bf16
        st = LayerStep(cfg, weights=(Ws, g))
        st.boundary(full_rows_of(wl, 0, 0, cfg.block_index).cuda())
        torch.cuda.synchronize()
        assert bool(st.batch.error_bits() & dllm.DLLM_DEVERR_RANGE) == flagged, scale


def test_host_validation_rejects_before_launch():
    cfg = _mini_ragged()
    st = LayerStep(cfg)
    bad = dllm.layer_desc(cfg.d_model, cfg.n_heads, 96, cfg.rope_theta)
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_attention(bad, st.batch.c, st.q_block, st.cache.c, st.o_full)
    assert e.value.status == dllm.DLLM_ERR_UNSUPPORTED
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_qkv_rope_write(st.desc, st.batch.c, st.q_block, st.gain, st.w_qkv, st.rope, st.rope_max_pos,
                                       st.cache.c, st.q_block, st.ws_step[:16])
    assert e.value.status == dllm.DLLM_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_attention(st.desc, st.batch.c, st.q_block.data_ptr() + 2, st.cache.c, st.o_full)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
