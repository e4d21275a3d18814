"""Host side of the Python binding, without a GPU: the batch metadata the
dllm_batch struct points at, the decoded-blocks batch of an incremental
boundary, the pools' shapes and types (as include/dllm.h states them) and the
row gather the tests use to read the pools."""
import numpy as np
import torch

from block_wise_kv_gb300 import dllm


def _layout(device="cpu"):
    table = np.array([[3, 0, 5, -1], [1, 2, 4, 6]], dtype=np.int32)
    return dllm.BatchLayout(table, seq_len=[150, 256], block_start=[64, 200], block_len=[32, 56], device=device)


def test_batch_layout_prefix_sums_and_bounds():
    lay = _layout()
    h = lay.host
    assert list(h["cu_block"]) == [0, 32, 88]
    assert list(h["cu_seq"]) == [0, 150, 406]
    assert (lay.batch, lay.max_pages) == (2, 4)
    assert (lay.total_block_rows, lay.total_seq_rows) == (88, 406)
    assert (lay.max_block_len, lay.max_seq_len) == (56, 256)
    c = lay.c
    assert (c.batch, c.max_pages_per_seq, c.total_block_rows, c.total_seq_rows, c.max_block_len, c.max_seq_len) == \
        (2, 4, 88, 406, 56, 256)
    # the struct points at the int32 copies of the same values
    for name in ("block_table", "seq_len", "block_start", "block_len", "cu_block", "cu_seq"):
        t = lay.dev[name]
        assert t.dtype == torch.int32 and t.is_contiguous()
        assert getattr(c, name) == t.data_ptr(), name
        np.testing.assert_array_equal(t.numpy(), h[name])
    assert c.error_flag == lay.error.data_ptr() and lay.error_bits() == 0


def test_decoded_blocks_share_the_sequences():
    lay = _layout()
    dec = lay.with_blocks(block_start=[32, 144], block_len=[32, 56])
    c, b = dec.c, lay.c
    # shared with the base: the sequences, their pages and rows, the error word
    for name in ("block_table", "seq_len", "cu_seq", "error_flag"):
        assert getattr(c, name) == getattr(b, name), name
    assert (c.batch, c.max_pages_per_seq, c.total_seq_rows, c.max_seq_len) == (2, 4, 406, 256)
    # its own: the block ranges and their row offsets
    for name in ("block_start", "block_len", "cu_block"):
        assert getattr(c, name) != getattr(b, name), name
    assert list(dec.host["cu_block"]) == [0, 32, 88]
    assert (c.total_block_rows, c.max_block_len) == (88, 56)
    np.testing.assert_array_equal(dec.dev["block_start"].numpy(), [32, 144])


def test_paged_cache_types_match_the_header():
    cache = dllm.PagedCache(num_pages=5, n_heads=3, head_dim=64, device="cpu", fill=3.0, pre=True)
    bf16 = (cache.k, cache.v, cache.q)
    for t in bf16:
        assert t.dtype == torch.bfloat16 and t.shape == (5, 3, dllm.PAGE, 64)
    for t in (cache.m, cache.l, cache.m_pre, cache.l_pre):
        assert t.dtype == torch.float32 and t.shape == (5, 3, dllm.PAGE)
    for t in (cache.o, cache.o_pre):  # the state's O~ / l in fp16
        assert t.dtype == torch.float16 and t.shape == (5, 3, dllm.PAGE, 64)
    assert all(bool(torch.all(t == 3.0)) for t in (*bf16, cache.m, cache.o))
    c = cache.c
    assert (c.k_pool, c.o_pool, c.o_pre, c.num_pages) == (cache.k.data_ptr(), cache.o.data_ptr(),
                                                          cache.o_pre.data_ptr(), 5)
    plain = dllm.PagedCache(num_pages=2, n_heads=1, head_dim=64, device="cpu")
    assert plain.o_pre is None and plain.c.o_pre is None and bool(torch.all(plain.o == 0))


def test_gather_rows_follows_the_block_table():
    H, d = 2, 4
    pool = torch.arange(7 * H * dllm.PAGE * d, dtype=torch.float32).reshape(7, H, dllm.PAGE, d)
    table = np.array([[5, 2, 6]], dtype=np.int32)
    n = 150
    got = dllm.gather_rows(pool, table, 0, n)
    assert got.shape == (n, H, d)
    for r in (0, 63, 64, 100, 128, 149):
        page, slot = table[0][r // dllm.PAGE], r % dllm.PAGE
        assert torch.equal(got[r], pool[page, :, slot]), r
