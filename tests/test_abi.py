"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every entry point include/dllm.h declares, and rejects bad arguments on the
host before any launch (no compute call needs a device here)."""
import ctypes
import os
import re

import pytest

from block_wise_kv_gb300 import build, dllm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return dllm.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "dllm.h")).read()
    return sorted(set(re.findall(r"^\s*(?:dllm_status|const char\*)\s+(dllm_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(dllm.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def _header_constants():
    """Every status code (enum) and #define of include/dllm.h with its value."""
    src = open(os.path.join(ROOT, "include", "dllm.h")).read()
    consts = {n: int(v) for n, v in re.findall(r"^\s*(DLLM_\w+)\s*=\s*(\d+)", src, re.M)}
    consts.update({n: int(v) for n, v in re.findall(r"^#define\s+(DLLM_\w+)\s+(\d+)", src, re.M)})
    return consts


def test_binding_constants_match_the_header():
    consts = _header_constants()
    assert {"DLLM_OK", "DLLM_DEVERR_RANGE", "DLLM_OP_CACHE_ADVANCE"} <= set(consts)
    for name, value in consts.items():
        assert getattr(dllm, name) == value, name


def test_device_error_bits_match_the_header():
    """The kernels OR their own error codes into the caller's word: they are the
    header's DLLM_DEVERR_* bits."""
    src = open(os.path.join(ROOT, "block_wise_kv_gb300", "csrc", "sm103.cuh")).read()
    dev = {n: int(v) for n, v in re.findall(r"^\s*(kErr\w+)\s*=\s*(\d+)", src, re.M)}
    hdr = _header_constants()
    pairs = {"kErrTimeout": "DLLM_DEVERR_TIMEOUT", "kErrBadPage": "DLLM_DEVERR_BAD_PAGE",
             "kErrBadShape": "DLLM_DEVERR_BAD_SHAPE", "kErrRange": "DLLM_DEVERR_RANGE"}
    assert set(dev) == set(pairs)
    for k, h in pairs.items():
        assert dev[k] == hdr[h], (k, h)


def _desc(**kw):
    d = dict(d_model=4096, n_heads=32, head_dim=128, rope_theta=5e5)
    d.update(kw)
    return dllm.layer_desc(**d)


def _batch(batch=2, max_pages=12, M=64, R=1536, max_block=32, max_seq=768):
    fake = 0x10000  # never dereferenced: validation fails or no launch happens in these tests
    return dllm.BatchC(batch, max_pages, M, R, max_block, max_seq, fake, fake, fake, fake, fake, fake, None)


def test_workspace_sizes(lib):
    d, b = _desc(), _batch()
    # 4 KB of counters, one RMSNorm scale pair (8 bytes) per row, the bf16 x^
    # rows (each region 256-byte aligned); 96 weight tiles: no stream-K partials
    assert dllm.dllm_workspace_size(d, b, dllm.DLLM_OP_BLOCK_QKV_ROPE_WRITE) == 4096 + 512 + 64 * 4096 * 2
    # the boundary's 1536 rows take the wide-tile kernel: 96 x 6 output tiles of
    # 128 x 256, fewer than four per SM, so its K chunks are split over the CTAs
    # and fp32 partial tiles of 128 x 256 per tile and contributor follow
    n = dllm.dllm_workspace_size(d, b, dllm.DLLM_OP_CACHE_BUILD)
    base = 4096 + 1536 * 8 + 1536 * 4096 * 2
    assert n > base and (n - base) % (96 * 6 * 128 * 256 * 4) == 0
    # a small model (12 weight tiles) splits each tile's K range over several
    # CTAs: fp32 partial tiles of 128 x 64 per tile and contributor follow
    small = _desc(d_model=1024, n_heads=8, head_dim=64)
    n = dllm.dllm_workspace_size(small, b, dllm.DLLM_OP_BLOCK_QKV_ROPE_WRITE)
    base = 4096 + 512 + 64 * 1024 * 2
    assert n > base and (n - base) % (12 * 128 * 64 * 4) == 0
    for op in (dllm.DLLM_OP_BLOCK_ATTENTION, dllm.DLLM_OP_STATE_MERGE, dllm.DLLM_OP_STEP_ATTENTION):
        assert dllm.dllm_workspace_size(d, b, op) == 0
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_workspace_size(d, b, 17)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT


def test_packed_weight_size_and_host_checks(lib):
    # 2 * ceil(D / 128) boxes of 128 x 64 per 128-row tile of the 3*H*d rows
    assert dllm.dllm_qkv_weight_packed_bytes(_desc()) == 3 * 32 * 128 * 4096 * 2
    assert dllm.dllm_qkv_weight_packed_bytes(_desc(d_model=4032)) == 3 * 32 * 128 * 4096 * 2
    assert dllm.dllm_qkv_weight_packed_bytes(_desc(d_model=192, n_heads=2, head_dim=64)) == 384 * 4 * 64 * 2
    fn = dllm.load().dllm_qkv_weight_pack
    d = _desc()
    n = dllm.dllm_qkv_weight_packed_bytes(d)
    for w, p in ((0x10000, 0x10000 + n // 2), (0x10008, 0x10000000000), (None, 0x10000000000)):
        assert fn(ctypes.byref(d), w, p, None) == dllm.DLLM_ERR_INVALID_ARGUMENT  # overlap, misaligned, NULL


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), dllm.DLLM_ERR_UNSUPPORTED),
    (dict(d_model=4000), dllm.DLLM_ERR_UNSUPPORTED),
    (dict(n_heads=3, head_dim=64), dllm.DLLM_ERR_UNSUPPORTED),
    (dict(rope_theta=0.0), dllm.DLLM_ERR_INVALID_ARGUMENT),
    (dict(rms_eps=-1.0), dllm.DLLM_ERR_INVALID_ARGUMENT),
])
def test_bad_layer_desc(lib, kw, status):
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_workspace_size(_desc(**kw), _batch(), dllm.DLLM_OP_BLOCK_ATTENTION)
    assert e.value.status == status


@pytest.mark.parametrize("kw,status", [
    (dict(batch=-1), dllm.DLLM_ERR_INVALID_ARGUMENT),
    (dict(max_block=769), dllm.DLLM_ERR_INVALID_ARGUMENT),  # a block longer than the longest sequence
    (dict(max_pages=2), dllm.DLLM_ERR_INVALID_ARGUMENT),   # 2 pages cannot hold 768 tokens
    (dict(M=100), dllm.DLLM_ERR_INVALID_ARGUMENT),         # more block rows than batch * max_block_len
    (dict(R=2000), dllm.DLLM_ERR_INVALID_ARGUMENT),        # more rows than batch * max_seq_len
])
def test_bad_batch(lib, kw, status):
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_workspace_size(_desc(), _batch(**kw), dllm.DLLM_OP_BLOCK_ATTENTION)
    assert e.value.status == status


def test_calls_reject_before_launch(lib):
    d = _desc()
    b = _batch()
    cache = dllm.CacheC(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 24)
    # misaligned output pointer
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_attention(d, b, 0x10000, cache, 0x10002, None, None, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
    # workspace too small
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_block_qkv_rope_write(d, b, 0x10000, 0x10000, 0x10000, 0x10000, 1024, cache, 0x10000, 0x10000, 0)
    assert e.value.status == dllm.DLLM_ERR_WORKSPACE_TOO_SMALL
    # RoPE table shorter than the longest sequence
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_cache_build(d, b, 0x10000, 0x10000, 0x10000, 0x10000, 100, cache, 0x10000, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
    # no cache pages
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_state_merge(d, b, dllm.CacheC(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0), 0x10000,
                              None, None, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT


def test_empty_batch_is_a_no_op(lib):
    d = _desc()
    b = _batch(batch=0, M=0, R=0)
    cache = dllm.CacheC(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 24)
    dllm.dllm_block_attention(d, b, 0x10000, cache, 0x10000, None, None, 0)
    dllm.dllm_state_merge(d, b, cache, 0x10000, None, None, 0)


def test_status_strings(lib):
    assert dllm.dllm_status_string(dllm.DLLM_OK) == "ok"
    assert "workspace" in dllm.dllm_status_string(dllm.DLLM_ERR_WORKSPACE_TOO_SMALL)
    assert dllm.dllm_status_string(99) == "unknown status"


def test_cache_advance_rejects_before_launch(lib):
    d = _desc()
    b = _batch()
    fake = 0x10000
    no_pre = dllm.CacheC(fake, fake, fake, fake, fake, fake, 24)
    with_pre = dllm.CacheC(fake, fake, fake, fake, fake, fake, 24, fake, fake, fake)
    # the decoded blocks must describe the same sequences through the same metadata
    other = dllm.BatchC(2, 12, 64, 1536, 32, 768, fake + 256, fake, fake, fake, fake, fake, None)
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_cache_advance(d, b, other, fake, fake, fake, fake, 1024, with_pre, fake, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
    # the prefix state pools are required (all three)
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_cache_advance(d, b, b, fake, fake, fake, fake, 1024, no_pre, fake, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
    half = dllm.CacheC(fake, fake, fake, fake, fake, fake, 24, fake, None, fake)
    with pytest.raises(dllm.DllmError) as e:
        dllm.dllm_cache_build(d, b, fake, fake, fake, fake, 1024, half, fake, 0)
    assert e.value.status == dllm.DLLM_ERR_INVALID_ARGUMENT
    # its workspace is the projection of the decoded rows
    assert dllm.dllm_workspace_size(d, b, dllm.DLLM_OP_CACHE_ADVANCE) == \
        dllm.dllm_workspace_size(d, b, dllm.DLLM_OP_BLOCK_QKV_ROPE_WRITE)


def test_lm_head_rejects_before_launch(lib):
    d = _desc()
    b = _batch()
    fake = 0x10000
    # 2 * ceil(V / 256) half-tile partials (max, sum, argmax) per row and the x^ rows, 256-byte aligned
    n = dllm.dllm_lm_head_workspace_size(d, b, 126464)
    assert n == 64 * 4096 * 2 + 3 * ((2 * 494 * 64 * 4 + 255) // 256 * 256)
    for vocab, kw, status in ((100, {}, dllm.DLLM_ERR_UNSUPPORTED),           # vocab not a multiple of 8
                              (1024, dict(d_model=4032), dllm.DLLM_ERR_UNSUPPORTED),  # d_model not of 128
                              (0, {}, dllm.DLLM_ERR_INVALID_ARGUMENT),
                              (1024, {}, dllm.DLLM_ERR_WORKSPACE_TOO_SMALL)):
        with pytest.raises(dllm.DllmError) as e:
            dllm.dllm_block_lm_head(_desc(**kw), b, vocab, fake, fake, fake, None, fake, fake, fake, None, 0)
        assert e.value.status == status, (vocab, kw)
