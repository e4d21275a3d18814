"""Python binding of the C ABI in include/dllm.h (ctypes).

The functions named ``dllm_*`` marshal arguments only: torch tensors become
device pointers, the current torch stream becomes the cudaStream_t, and a
non-zero status raises ``DllmError``.  Every step of the computation runs in
the CUDA library; there is no fallback.  If the library has not been built
(``python -m block_wise_kv_gb300.build``) importing the binding still works,
but the first call raises.

The helpers below (``LayerDesc``, ``BatchLayout``, ``PagedCache``) only
allocate device memory with torch and fill the C structs.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdllm.so")

DLLM_OK = 0
DLLM_ERR_INVALID_ARGUMENT = 1
DLLM_ERR_UNSUPPORTED = 2
DLLM_ERR_WORKSPACE_TOO_SMALL = 3
DLLM_ERR_CUDA = 4
DLLM_ERR_TIMEOUT = 5

DLLM_DEVERR_TIMEOUT = 1
DLLM_DEVERR_BAD_PAGE = 2
DLLM_DEVERR_BAD_SHAPE = 4
DLLM_DEVERR_RANGE = 8

DLLM_OP_CACHE_BUILD = 0
DLLM_OP_BLOCK_QKV_ROPE_WRITE = 1
DLLM_OP_BLOCK_ATTENTION = 2
DLLM_OP_STATE_MERGE = 3
DLLM_OP_STEP_ATTENTION = 4
DLLM_OP_CACHE_ADVANCE = 5

PAGE = 64

# Every symbol include/dllm.h declares.
EXPORTS = ("dllm_workspace_size", "dllm_rope_table_build", "dllm_qkv_weight_packed_bytes", "dllm_qkv_weight_pack",
           "dllm_cache_build", "dllm_cache_advance", "dllm_block_qkv_rope_write", "dllm_block_qkv_rope_write_noalloc",
           "dllm_block_attention", "dllm_state_merge", "dllm_step_attention", "dllm_lm_head_workspace_size",
           "dllm_block_lm_head", "dllm_ffn_workspace_size", "dllm_block_ffn", "dllm_status_string")


class DllmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({dllm_status_string(status)})")


class LayerDescC(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("softmax_scale", ctypes.c_float)]


class CacheC(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("q_pool", ctypes.c_void_p),
                ("m_pool", ctypes.c_void_p), ("l_pool", ctypes.c_void_p), ("o_pool", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32),
                ("m_pre", ctypes.c_void_p), ("l_pre", ctypes.c_void_p), ("o_pre", ctypes.c_void_p)]


class BatchC(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("total_block_rows", ctypes.c_int32), ("total_seq_rows", ctypes.c_int32),
                ("max_block_len", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("seq_len", ctypes.c_void_p), ("block_start", ctypes.c_void_p),
                ("block_len", ctypes.c_void_p), ("cu_block", ctypes.c_void_p), ("cu_seq", ctypes.c_void_p),
                ("error_flag", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libdllm.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA library not built: {p} is missing "
                                   "(run `python -m block_wise_kv_gb300.build`)")
            lib = ctypes.CDLL(p)
            P = ctypes.POINTER
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            sig = {
                "dllm_workspace_size": [P(LayerDescC), P(BatchC), i32, P(sz)],
                "dllm_rope_table_build": [P(LayerDescC), i32, vp, vp],
                "dllm_qkv_weight_packed_bytes": [P(LayerDescC), P(sz)],
                "dllm_qkv_weight_pack": [P(LayerDescC), vp, vp, vp],
                "dllm_cache_build": [P(LayerDescC), P(BatchC), vp, vp, vp, vp, i32, P(CacheC), vp, sz, vp],
                "dllm_cache_advance": [P(LayerDescC), P(BatchC), P(BatchC), vp, vp, vp, vp, i32, P(CacheC), vp, sz,
                                       vp],
                "dllm_block_qkv_rope_write": [P(LayerDescC), P(BatchC), vp, vp, vp, vp, i32, P(CacheC), vp, vp, sz,
                                              vp],
                "dllm_block_qkv_rope_write_noalloc": [P(LayerDescC), P(BatchC), vp, vp, vp, vp, i32, P(CacheC), vp,
                                                      vp],
                "dllm_block_attention": [P(LayerDescC), P(BatchC), vp, P(CacheC), vp, vp, vp, sz, vp],
                "dllm_state_merge": [P(LayerDescC), P(BatchC), P(CacheC), vp, vp, vp, sz, vp],
                "dllm_step_attention": [P(LayerDescC), P(BatchC), vp, P(CacheC), vp, vp, vp, sz, vp],
                "dllm_lm_head_workspace_size": [P(LayerDescC), P(BatchC), i32, P(sz)],
                "dllm_block_lm_head": [P(LayerDescC), P(BatchC), i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                "dllm_ffn_workspace_size": [P(LayerDescC), P(BatchC), i32, P(sz)],
                "dllm_block_ffn": [P(LayerDescC), P(BatchC), i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            }
            for name, argt in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = argt
                fn.restype = ctypes.c_int
            lib.dllm_status_string.argtypes = [ctypes.c_int]
            lib.dllm_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _nbytes(t) -> int:
    if t is None or isinstance(t, int):
        return 0
    return t.numel() * t.element_size()


def _check(fn: str, status: int) -> None:
    if status != DLLM_OK:
        raise DllmError(fn, status)


# ------------------------------------------------------------ the C ABI ----
def dllm_status_string(status: int) -> str:
    return load().dllm_status_string(int(status)).decode()


def dllm_workspace_size(desc: LayerDescC, batch: BatchC, op: int) -> int:
    out = ctypes.c_size_t(0)
    _check("dllm_workspace_size", load().dllm_workspace_size(ctypes.byref(desc), ctypes.byref(batch), op,
                                                             ctypes.byref(out)))
    return out.value


def dllm_rope_table_build(desc: LayerDescC, max_pos: int, rope_table: torch.Tensor, stream=None) -> None:
    _check("dllm_rope_table_build", load().dllm_rope_table_build(ctypes.byref(desc), int(max_pos), _ptr(rope_table),
                                                                 _stream(stream)))


def dllm_qkv_weight_packed_bytes(desc: LayerDescC) -> int:
    out = ctypes.c_size_t(0)
    _check("dllm_qkv_weight_packed_bytes", load().dllm_qkv_weight_packed_bytes(ctypes.byref(desc), ctypes.byref(out)))
    return out.value


def dllm_qkv_weight_pack(desc: LayerDescC, w_qkv: torch.Tensor, w_packed: torch.Tensor, stream=None) -> None:
    _check("dllm_qkv_weight_pack", load().dllm_qkv_weight_pack(ctypes.byref(desc), _ptr(w_qkv), _ptr(w_packed),
                                                               _stream(stream)))


def pack_qkv_weight(desc: LayerDescC, w_qkv: torch.Tensor, stream=None) -> torch.Tensor:
    """The tile-packed copy of a device bf16 [3*H*d][d_model] weight that the
    projection calls take (allocated here, filled by dllm_qkv_weight_pack)."""
    n = dllm_qkv_weight_packed_bytes(desc)
    out = torch.empty(n // 2, dtype=torch.bfloat16, device=w_qkv.device)
    dllm_qkv_weight_pack(desc, w_qkv.contiguous(), out, stream)
    return out


def dllm_cache_build(desc, batch, x_full, rms_gain, w_packed, rope_table, rope_max_pos, cache, ws, stream=None):
    _check("dllm_cache_build", load().dllm_cache_build(
        ctypes.byref(desc), ctypes.byref(batch), _ptr(x_full), _ptr(rms_gain), _ptr(w_packed), _ptr(rope_table),
        int(rope_max_pos), ctypes.byref(cache), _ptr(ws), _nbytes(ws), _stream(stream)))


def dllm_cache_advance(desc, batch, decoded, x_decoded, rms_gain, w_packed, rope_table, rope_max_pos, cache, ws,
                       stream=None):
    _check("dllm_cache_advance", load().dllm_cache_advance(
        ctypes.byref(desc), ctypes.byref(batch), ctypes.byref(decoded), _ptr(x_decoded), _ptr(rms_gain),
        _ptr(w_packed), _ptr(rope_table), int(rope_max_pos), ctypes.byref(cache), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def dllm_block_qkv_rope_write(desc, batch, x_block, rms_gain, w_packed, rope_table, rope_max_pos, cache, q_block,
                              ws, stream=None):
    _check("dllm_block_qkv_rope_write", load().dllm_block_qkv_rope_write(
        ctypes.byref(desc), ctypes.byref(batch), _ptr(x_block), _ptr(rms_gain), _ptr(w_packed), _ptr(rope_table),
        int(rope_max_pos), ctypes.byref(cache), _ptr(q_block), _ptr(ws), _nbytes(ws), _stream(stream)))


def dllm_block_qkv_rope_write_noalloc(desc, batch, x_block, rms_gain, w_packed, rope_table, rope_max_pos, cache,
                                      q_block, stream=None):
    """dllm_block_qkv_rope_write without a workspace: for callers that cannot
    allocate device memory (the library's fixed 8 MiB scratch is used)."""
    _check("dllm_block_qkv_rope_write_noalloc", load().dllm_block_qkv_rope_write_noalloc(
        ctypes.byref(desc), ctypes.byref(batch), _ptr(x_block), _ptr(rms_gain), _ptr(w_packed), _ptr(rope_table),
        int(rope_max_pos), ctypes.byref(cache), _ptr(q_block), _stream(stream)))


def dllm_block_attention(desc, batch, q_block, cache, o_full, lse=None, ws=None, stream=None):
    _check("dllm_block_attention", load().dllm_block_attention(
        ctypes.byref(desc), ctypes.byref(batch), _ptr(q_block), ctypes.byref(cache), _ptr(o_full), _ptr(lse),
        _ptr(ws), _nbytes(ws), _stream(stream)))


def dllm_state_merge(desc, batch, cache, o_full, lse=None, ws=None, stream=None):
    _check("dllm_state_merge", load().dllm_state_merge(
        ctypes.byref(desc), ctypes.byref(batch), ctypes.byref(cache), _ptr(o_full), _ptr(lse), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def dllm_step_attention(desc, batch, q_block, cache, o_full, lse=None, ws=None, stream=None):
    _check("dllm_step_attention", load().dllm_step_attention(
        ctypes.byref(desc), ctypes.byref(batch), _ptr(q_block), ctypes.byref(cache), _ptr(o_full), _ptr(lse),
        _ptr(ws), _nbytes(ws), _stream(stream)))


def dllm_lm_head_workspace_size(desc, batch, vocab: int) -> int:
    out = ctypes.c_size_t(0)
    _check("dllm_lm_head_workspace_size", load().dllm_lm_head_workspace_size(ctypes.byref(desc), ctypes.byref(batch),
                                                                             int(vocab), ctypes.byref(out)))
    return int(out.value)


def dllm_block_lm_head(desc, batch, vocab, h_full, final_gain, w_lm, logits, lse, argmax, p_max, ws, stream=None):
    _check("dllm_block_lm_head", load().dllm_block_lm_head(
        ctypes.byref(desc), ctypes.byref(batch), int(vocab), _ptr(h_full), _ptr(final_gain), _ptr(w_lm),
        _ptr(logits), _ptr(lse), _ptr(argmax), _ptr(p_max), _ptr(ws), _nbytes(ws), _stream(stream)))


def dllm_ffn_workspace_size(desc, batch, d_ff: int) -> int:
    out = ctypes.c_size_t(0)
    _check("dllm_ffn_workspace_size", load().dllm_ffn_workspace_size(ctypes.byref(desc), ctypes.byref(batch),
                                                                     int(d_ff), ctypes.byref(out)))
    return int(out.value)


def dllm_block_ffn(desc, batch, d_ff, o_full, x_block, w_o, ffn_gain, w_gate_up, w_gate_up_scale, w_down,
                   w_down_scale, y_block, ws, stream=None):
    _check("dllm_block_ffn", load().dllm_block_ffn(
        ctypes.byref(desc), ctypes.byref(batch), int(d_ff), _ptr(o_full), _ptr(x_block), _ptr(w_o), _ptr(ffn_gain),
        _ptr(w_gate_up), _ptr(w_gate_up_scale), _ptr(w_down), _ptr(w_down_scale), _ptr(y_block), _ptr(ws),
        _nbytes(ws), _stream(stream)))


# ---------------------------------------------------- memory / structs ----
def layer_desc(d_model: int, n_heads: int, head_dim: int, rope_theta: float, rms_eps: float = 1e-5,
               softmax_scale: float = 0.0) -> LayerDescC:
    return LayerDescC(d_model, n_heads, head_dim, PAGE, rope_theta, rms_eps, softmax_scale)


class BatchLayout:
    """Device copies of the batch metadata and the dllm_batch struct that
    points at them (the tensors stay alive as long as this object)."""

    def __init__(self, block_table, seq_len, block_start, block_len, device="cuda", error_flag: bool = True):
        bt = np.asarray(block_table, dtype=np.int32)
        self.host = dict(block_table=bt, seq_len=np.asarray(seq_len, np.int32),
                         block_start=np.asarray(block_start, np.int32), block_len=np.asarray(block_len, np.int32))
        h = self.host
        h["cu_block"] = np.concatenate([[0], np.cumsum(h["block_len"])]).astype(np.int32)
        h["cu_seq"] = np.concatenate([[0], np.cumsum(h["seq_len"])]).astype(np.int32)
        self.batch = int(h["seq_len"].shape[0])
        self.dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in h.items()}
        self.error = torch.zeros(1, dtype=torch.int32, device=device) if error_flag else None
        self.max_pages = int(bt.shape[1]) if bt.ndim == 2 and bt.shape[1] > 0 else 1
        self.total_block_rows = int(h["cu_block"][-1])
        self.total_seq_rows = int(h["cu_seq"][-1])
        self.max_block_len = int(h["block_len"].max()) if self.batch else 1
        self.max_seq_len = int(h["seq_len"].max()) if self.batch else 1
        d = self.dev
        self.c = BatchC(self.batch, self.max_pages, self.total_block_rows, self.total_seq_rows, self.max_block_len,
                        self.max_seq_len, _ptr(d["block_table"]), _ptr(d["seq_len"]), _ptr(d["block_start"]),
                        _ptr(d["block_len"]), _ptr(d["cu_block"]), _ptr(d["cu_seq"]), _ptr(self.error))

    def error_bits(self) -> int:
        return 0 if self.error is None else int(self.error.item())

    def with_blocks(self, block_start, block_len) -> "BlockRange":
        """The same sequences with other block ranges (for dllm_cache_advance's
        decoded blocks): the struct shares this layout's block table, seq_len,
        cu_seq and error flag."""
        return BlockRange(self, block_start, block_len)


class BlockRange:
    """A dllm_batch that shares a BatchLayout's sequences and points at its own
    block_start / block_len / cu_block."""

    def __init__(self, base: BatchLayout, block_start, block_len):
        bs = np.asarray(block_start, np.int32)
        bl = np.asarray(block_len, np.int32)
        cu = np.concatenate([[0], np.cumsum(bl)]).astype(np.int32)
        dev = base.dev["seq_len"].device
        self.host = dict(block_start=bs, block_len=bl, cu_block=cu)
        self.dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in self.host.items()}
        self.total_block_rows = int(cu[-1])
        self.max_block_len = int(bl.max()) if bl.size else 1
        d, bd = self.dev, base.dev
        self.c = BatchC(base.batch, base.max_pages, self.total_block_rows, base.total_seq_rows, self.max_block_len,
                        base.max_seq_len, _ptr(bd["block_table"]), _ptr(bd["seq_len"]), _ptr(d["block_start"]),
                        _ptr(d["block_len"]), _ptr(d["cu_block"]), _ptr(bd["cu_seq"]), _ptr(base.error))


class PagedCache:
    """The paged pools of one layer, allocated by torch (zero-filled, or
    filled with `fill` to act as a sentinel)."""

    def __init__(self, num_pages: int, n_heads: int, head_dim: int, device="cuda", fill: float | None = None,
                 pre: bool = False):
        shp = (num_pages, n_heads, PAGE, head_dim)

        def mk(shape, dtype):
            t = torch.zeros(shape, dtype=dtype, device=device)
            if fill is not None:
                t.fill_(fill)
            return t

        self.k = mk(shp, torch.bfloat16)
        self.v = mk(shp, torch.bfloat16)
        self.q = mk(shp, torch.bfloat16)
        self.m = mk(shp[:3], torch.float32)
        self.l = mk(shp[:3], torch.float32)
        self.o = mk(shp, torch.float16)  # the state's O~ / l
        self.num_pages = num_pages
        # the prefix state (for incremental boundaries), when asked for
        self.m_pre = mk(shp[:3], torch.float32) if pre else None
        self.l_pre = mk(shp[:3], torch.float32) if pre else None
        self.o_pre = mk(shp, torch.float16) if pre else None
        self.c = CacheC(_ptr(self.k), _ptr(self.v), _ptr(self.q), _ptr(self.m), _ptr(self.l), _ptr(self.o),
                        num_pages, _ptr(self.m_pre), _ptr(self.l_pre), _ptr(self.o_pre))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Caller-owned scratch of at least nbytes (256-byte aligned by torch's
    allocator), zero-filled."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def gather_rows(pool: torch.Tensor, block_table: np.ndarray, b: int, n: int) -> torch.Tensor:
    """Rows 0..n-1 of sequence b from a pool [P, H, 64, ...] -> [n, H, ...]
    (a torch index operation, for tests and inspection)."""
    pos = torch.arange(n)
    pages = torch.from_numpy(np.asarray(block_table[b], dtype=np.int64))[pos // PAGE].to(pool.device)
    slots = (pos % PAGE).to(pool.device)
    return pool[pages, :, slots]
