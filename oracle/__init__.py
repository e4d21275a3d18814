"""fp64 CPU oracle for one per-layer inner denoising step of block-wise
diffusion-LLM decoding.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library and its Python binding never do; the two sides
share no code (only the seeded input generator feeds both).

All of the arithmetic lives in ``oracle.cpp`` (fp64, OpenMP over independent
outputs), the projection included.  This module loads it with ctypes and composes the plain definition
of the step:

  1. x^ = RMSNorm(x) for every row                  (LaCache §3.3.2, Eq. (1))
  2. [q, k, v] = x^ W_qkv^T                          (LaCache Eq. (1))
  3. RoPE(q, k) at absolute positions 0..N-1         (LaCache Eq. (1); Fast-dLLM
                                                       DualCache "block_start for
                                                       correct RoPE offset")
  4. O = softmax(scale q k^T) v over ALL keys, two-pass, and L = m + ln l
                                                      (Fast-dLLM DualCache,
                                                       "Motivation": the naive
                                                       sampler recomputes the
                                                       full sequence every step)

Readings of points the pages leave open:
scale = 1/sqrt(d_h); rotate-half RoPE pairs (i, i + d/2) with angle
p * theta^(-2i/d); RMSNorm eps = 1e-5 with gain g; the only rounding points
mirrored are the two storage formats of the method: x^ -> bf16 (the GEMM
operand) and q, k, v -> bf16 (the bf16 cache), both round-to-nearest-even.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIBPATH = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64
_f64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_lib/liboracle.so (g++, fp64, OpenMP).

    -ffp-contract=off keeps every multiply and add separately rounded, so the
    x86 and Arm builds produce the same bits."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIBPATH) and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC):
        return _LIBPATH
    tmp = _LIBPATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # DLLM_ORACLE_LIB points the tests' mutation check at a deliberately
            # broken build of oracle.cpp; normally unset.
            path = os.environ.get("DLLM_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            sigs = {
                "orc_num_threads": ([], ctypes.c_int),
                "orc_set_num_threads": ([ctypes.c_int], None),
                "orc_bf16_round": ([_f64], _f64),
                "orc_bf16_round_array": ([_D, _i64], None),
                "orc_rmsnorm": ([_D, _i64, _i64, _D, _f64, _D], None),
                "orc_linear": ([_D, _i64, _i64, _D, _i64, _D], None),
                "orc_rope": ([_D, _i64, _i64, _i64, _I64, _f64], None),
                "orc_attention": ([_D, _i64, _D, _D, _i64, _i64, _i64, _f64, _D, _D], None),
                "orc_attention_online": ([_D, _i64, _D, _D, _i64, _i64, _i64, _f64, _i64, _I64, _D, _D], None),
                "orc_state_build": ([_D, _i64, _D, _D, _i64, _i64, _i64, _f64, _i64, _i64, _i64, _D, _D, _D], None),
                "orc_state_merge": (
                    [_D, _i64, _D, _D, _i64, _i64, _i64, _f64, _i64, _i64, _i64, _D, _D, _D, _D, _D],
                    None,
                ),
                "orc_softmax_stats": ([_D, _i64, _i64, _D, _I64, _D], None),
                "orc_e4m3_decode": ([ctypes.c_int], _f64),
                "orc_e4m3_round": ([_f64], _f64),
                "orc_quant_groups": ([_D, _i64, _i64, _i64, _D, _D], None),
                "orc_dequant_blocks": ([ctypes.c_void_p, _i64, _i64, _i64, _i64, ctypes.c_void_p, _D], None),
                "orc_rmsnorm_f32": ([_D, _i64, _i64, _D, _f64, _D], None),
                "orc_alg1": (
                    [_D, _D, _D, _i64, _i64, _i64, _f64, _i64, _i64, _i64, _i64, ctypes.c_int, _D, _D, _D, _D, _D],
                    None,
                ),
            }
            for name, (argt, rest) in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = argt
                fn.restype = rest
            _lib = lib
    return _lib


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(_D)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ----------------------------------------------------------------- primitives
def bf16_round(a) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even (returned as fp64)."""
    out = np.array(a, dtype=np.float64, copy=True, order="C")
    _load().orc_bf16_round_array(_p(out), out.size)
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x, g = _c(x), _c(g)
    rows, D = x.shape
    out = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), rows, D, _p(g), float(eps), _p(out))
    return out


def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """x [rows, D] times W^T, W stored [nout, D]: the plain C triple loop."""
    x, W = _c(x), _c(W)
    rows, D = x.shape
    nout = W.shape[0]
    assert W.shape[1] == D
    out = np.empty((rows, nout), dtype=np.float64)
    _load().orc_linear(_p(x), rows, D, _p(W), nout, _p(out))
    return out


def rope(t: np.ndarray, pos, theta: float) -> np.ndarray:
    """t [rows, H, d]; returns the rotated copy."""
    out = _c(t).copy()
    rows, H, d = out.shape
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    assert pos.shape == (rows,)
    _load().orc_rope(_p(out), rows, H, d, pos.ctypes.data_as(_I64), float(theta))
    return out


def attention(q, k, v, scale: float):
    """Two-pass full attention.  q [nq,H,d], k/v [nk,H,d] -> (O [nq,H,d], L [nq,H])."""
    q, k, v = _c(q), _c(k), _c(v)
    nq, H, d = q.shape
    nk = k.shape[0]
    O = np.empty((nq, H, d))
    L = np.empty((nq, H))
    _load().orc_attention(_p(q), nq, _p(k), _p(v), nk, H, d, float(scale), _p(O), _p(L))
    return O, L


def attention_online(q, k, v, scale: float, bc: int, order=None):
    q, k, v = _c(q), _c(k), _c(v)
    nq, H, d = q.shape
    nk = k.shape[0]
    O = np.empty((nq, H, d))
    L = np.empty((nq, H))
    optr = None
    if order is not None:
        order = np.ascontiguousarray(order, dtype=np.int64)
        optr = order.ctypes.data_as(_I64)
    _load().orc_attention_online(_p(q), nq, _p(k), _p(v), nk, H, d, float(scale), int(bc), optr, _p(O), _p(L))
    return O, L


def state_build(q_rows, k, v, scale: float, c_lo: int, c_hi: int, bc: int = 64):
    """FACache build over keys outside [c_lo, c_hi).  Returns (m, l, Ot)."""
    q_rows, k, v = _c(q_rows), _c(k), _c(v)
    nr, H, d = q_rows.shape
    nk = k.shape[0]
    m = np.empty((nr, H))
    l = np.empty((nr, H))
    Ot = np.empty((nr, H, d))
    _load().orc_state_build(_p(q_rows), nr, _p(k), _p(v), nk, H, d, float(scale), int(c_lo), int(c_hi), int(bc),
                            _p(m), _p(l), _p(Ot))
    return m, l, Ot


def state_merge(q_rows, k, v, scale: float, c_lo: int, c_hi: int, m, l, Ot, bc: int = 64):
    """FACache reuse: cached state + keys in [c_lo, c_hi).  Returns (O, L)."""
    q_rows, k, v, m, l, Ot = map(_c, (q_rows, k, v, m, l, Ot))
    nr, H, d = q_rows.shape
    nk = k.shape[0]
    O = np.empty((nr, H, d))
    L = np.empty((nr, H))
    _load().orc_state_merge(_p(q_rows), nr, _p(k), _p(v), nk, H, d, float(scale), int(c_lo), int(c_hi), int(bc),
                            _p(m), _p(l), _p(Ot), _p(O), _p(L))
    return O, L


def alg1(q, k, v, scale: float, c_lo: int, c_hi: int, br: int, bc: int, genstep: bool, cache=None):
    """LaCache Algorithm 1 at tile granularity.  cache = (mc, lc, Oc) arrays,
    written when genstep, read otherwise.  Returns (O, L, cache)."""
    q, k, v = _c(q), _c(k), _c(v)
    N, H, d = q.shape
    if cache is None:
        cache = (np.full((N, H), np.nan), np.full((N, H), np.nan), np.full((N, H, d), np.nan))
    mc, lc, Oc = (np.ascontiguousarray(c, dtype=np.float64) for c in cache)
    O = np.empty((N, H, d))
    L = np.empty((N, H))
    _load().orc_alg1(_p(q), _p(k), _p(v), N, H, d, float(scale), int(c_lo), int(c_hi), int(br), int(bc),
                     1 if genstep else 0, _p(mc), _p(lc), _p(Oc), _p(O), _p(L))
    return O, L, (mc, lc, Oc)


def project(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """x [rows, D] times W^T: the projection of the step, `orc_linear`'s plain
    sums in oracle.cpp (pinned against numpy's matmul)."""
    return linear(x, W)


def softmax_stats(z):
    """Per row of logits z [rows, V]: (lse, argmax (lowest index of the max), p_max)."""
    z = _c(z)
    rows, V = z.shape
    lse = np.empty(rows)
    am = np.empty(rows, dtype=np.int64)
    pm = np.empty(rows)
    _load().orc_softmax_stats(_p(z), rows, V, _p(lse), am.ctypes.data_as(_I64), _p(pm))
    return lse, am, pm


def lm_head(h, g, W_lm, eps: float, mirror: bool = True):
    """The block-only epilogue for the given rows (the block rows of the final hidden
    states; LaCache §3.4, the sampling stage): x^ = RMSNorm(h) (rounded to bf16 when
    `mirror`: the GEMM operand), logits = x^ W_lm^T, and the softmax summary.
    Returns dict(logits, lse, argmax, p_max)."""
    xh = rmsnorm(h, g, eps)
    if mirror:
        xh = bf16_round(xh)
    z = linear(xh, W_lm)
    lse, am, pm = softmax_stats(z)
    return dict(logits=z, lse=lse, argmax=am, p_max=pm)


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e4m3_round(x: float) -> float:
    return _load().orc_e4m3_round(float(x))


def quant_groups(x, group: int = 128):
    """LaCache Eq. (7)-(8) per row and group of columns: (dequantised values, scales)."""
    x = _c(x)
    rows, cols = x.shape
    deq = np.empty_like(x)
    sc = np.empty((rows, cols // group))
    _load().orc_quant_groups(_p(x), rows, cols, int(group), _p(deq), _p(sc))
    return deq, sc


def rmsnorm_f32(h, g, eps: float):
    """RMSNorm(h) g as the quantisation's input, in fp32: 1 / rms correctly rounded to fp32,
    then (h * inv) * g with fp32 products (returned as fp64 values)."""
    h, g = _c(h), _c(g)
    rows, D = h.shape
    out = np.empty_like(h)
    _load().orc_rmsnorm_f32(_p(h), rows, D, _p(g), float(eps), _p(out))
    return out


def dequant_blocks(codes, scales, block: int = 128):
    """e4m3 codes [rows][cols] (uint8) times one fp32 scale per block x block."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    rows, cols = codes.shape
    out = np.empty((rows, cols))
    _load().orc_dequant_blocks(codes.ctypes.data, rows, cols, int(block), int(block), scales.ctypes.data, _p(out))
    return out


def ffn(o_rows, x_rows, W_o, g2, wgu_codes, wgu_scale, wd_codes, wd_scale, eps: float, mirror: bool = True):
    """The rest of the layer for the given rows (LaCache §3.4 Mixed precision
    strategy): h1 = x + O W_o^T (rounded to bf16: the residual stream's storage
    point), x2 = RMSNorm(h1) g2 quantised per row and 128 columns (Eq. (7)-(8);
    a quantised code is an integer decided by floating point, so x2 is formed in
    the kernels' fp32 before the decision, see `rmsnorm_f32`), gate / up from the
    e4m3 weights (rows 2j, 2j + 1), a = SiLU(gate) * up quantised the same way,
    y = h1 + a W_down^T.  Returns dict(h1, y)."""
    h1 = x_rows + linear(o_rows, W_o)
    if mirror:
        h1 = bf16_round(h1)
    x2, _ = quant_groups(rmsnorm_f32(h1, g2, eps))
    gu = linear(x2, dequant_blocks(wgu_codes, wgu_scale))
    gate, up = gu[:, 0::2], gu[:, 1::2]
    a = gate / (1.0 + np.exp(-gate)) * up
    aq, _ = quant_groups(a)
    y = h1 + linear(aq, dequant_blocks(wd_codes, wd_scale))
    return dict(h1=h1, y=y)


# ---------------------------------------------------------------- the step
def qkv(x, g, W, n_heads: int, head_dim: int, theta: float, eps: float, pos, mirror: bool = True):
    """Token-wise part of the step (LaCache Eq. (1)) for the given rows:
    returns q, k, v [rows, H, d] after RMSNorm, projection and RoPE at `pos`,
    rounded to bf16 when `mirror` (the bf16 cache is the storage point)."""
    HD = n_heads * head_dim
    xh = rmsnorm(x, g, eps)
    if mirror:
        xh = bf16_round(xh)
    y = project(xh, W)
    rows = y.shape[0]
    q = y[:, :HD].reshape(rows, n_heads, head_dim)
    k = y[:, HD:2 * HD].reshape(rows, n_heads, head_dim)
    v = y[:, 2 * HD:].reshape(rows, n_heads, head_dim)
    q = rope(q, pos, theta)
    k = rope(k, pos, theta)
    if mirror:
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    return q, k, np.ascontiguousarray(v)


def layer_step(x, g, W, n_heads: int, head_dim: int, theta: float, eps: float, scale: float | None = None,
               rows=None, mirror: bool = True, heads=None):
    """The full-recompute definition of one layer step for ONE sequence.

    x [N, D] holds every row of the sequence at this step ([prefix | block |
    suffix]).  Returns dict(q, k, v, O, L) where q, O, L cover `rows` (all rows
    by default) and k, v cover all N rows.  Attention is bidirectional over all
    N keys; positions are 0..N-1.  `heads` restricts the step to a subset of
    heads (their projection rows and their attention), all heads by default."""
    x = np.asarray(x, dtype=np.float64)
    N = x.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(head_dim)
    if rows is None:
        rows = np.arange(N)
    rows = np.asarray(rows, dtype=np.int64)
    d = head_dim
    HD = n_heads * d
    W = np.asarray(W, dtype=np.float64)
    if heads is None:
        heads = np.arange(n_heads)
    sel = np.concatenate([np.arange(h * d, (h + 1) * d) for h in heads])
    Wq, Wk, Wv = W[sel], W[HD + sel], W[2 * HD + sel]
    H = len(heads)
    xh = rmsnorm(x, g, eps)
    if mirror:
        xh = bf16_round(xh)
    # K and V for every row, Q only for the requested rows.
    k = rope(project(xh, Wk).reshape(N, H, d), np.arange(N), theta)
    v = project(xh, Wv).reshape(N, H, d)
    q = rope(project(xh[rows], Wq).reshape(len(rows), H, d), rows, theta)
    if mirror:
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    O, L = attention(q, k, v, scale)
    return dict(q=q, k=k, v=v, O=O, L=L)
