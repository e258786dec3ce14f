"""CPU oracle for INT8-KV-cache attention (test infrastructure).

This package is the slow, plain reference the CUDA library is checked against.  Only
tests/, ``__graft_entry__.smoke()`` and bench.py's ``cpu_baseline`` / ``--impl reference``
legs may import it; the product path never does.  The arithmetic lives in
``kvq_oracle.cpp`` (plain C++, FP64 reference + exact int8 emulation); this module only
marshals numpy arrays into it.

Cache layout (same documented layout the CUDA library uses, read here through the
oracle's own index functions):
    k        int8  [num_blocks][n_kv_heads][head_dim/16][16][16]
    v        int8  [num_blocks][n_kv_heads][head_dim][16]
    k_scale  fp32  [num_blocks][n_kv_heads][16]
    v_scale  fp32  [num_blocks][n_kv_heads][16]
"""
import ctypes
import os

import numpy as np

from . import build as _build

BLOCK_SIZE = 16
PV_TILE = 128

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_kv_bytes_per_token.restype = i64
        lib.oracle_kv_bytes_per_token.argtypes = [i32, i32]
        lib.oracle_bf16_kv_bytes_per_token.restype = i64
        lib.oracle_bf16_kv_bytes_per_token.argtypes = [i32, i32]
        lib.oracle_quant_rows.argtypes = [vp, i64, i32, vp, vp]
        lib.oracle_kv_quant_write.restype = i32
        lib.oracle_kv_quant_write.argtypes = [vp, vp, vp, i32, vp, vp, vp, i32, i32]
        lib.oracle_rope_quant_write.restype = i32
        lib.oracle_rope_quant_write.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, i32, i32, vp, i32, i32,
                                                vp, vp, vp]
        lib.oracle_decode_f64.argtypes = [vp, vp, i32, i32, vp, i32, vp, f64, vp, i32, vp, i32]
        lib.oracle_verify_f64.argtypes = [vp, vp, i32, i32, i32, vp, i32, vp, f64, vp, i32, vp, i32]
        lib.oracle_decode_split_f64.argtypes = [vp, vp, i32, i32, vp, i32, vp, f64, i32, vp, i32]
        lib.oracle_prefill_first_f64.argtypes = [vp, vp, vp, i32, i32, i32, i32, f64, vp, i32, vp, i32]
        lib.oracle_prefill_ref_f64.argtypes = [vp, vp, i32, i32, i32, vp, f64, vp, i32, vp, i32]
        lib.oracle_prefill_qk_int32.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, i32, i32, vp]
        lib.oracle_prefill_qdeq_f64.argtypes = [vp, vp, i32, i32, i32, vp, f64, i32, vp, i32, vp, vp, vp, i32]
        lib.oracle_prefill_int8_emul.argtypes = [vp, vp, i32, i32, i32, vp, ctypes.c_float, i32,
                                                 vp, i32, vp, vp, vp, i32]
        lib.oracle_exp2_det.restype = ctypes.c_float
        lib.oracle_exp2_det.argtypes = [ctypes.c_float]
        lib.oracle_sparse_f64.argtypes = [vp, vp, i32, i32, vp, vp, vp, f64, vp, i32, vp, i32]
        _lib = lib
    return _lib


class _CCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class HostCache:
    """A paged int8 K/V cache in host memory (numpy), in the documented layout."""

    def __init__(self, num_blocks, n_kv_heads, head_dim, block_size=BLOCK_SIZE):
        self.num_blocks, self.n_kv_heads, self.head_dim = num_blocks, n_kv_heads, head_dim
        self.block_size = block_size
        self.k = np.zeros((num_blocks, n_kv_heads, head_dim // 16, block_size, 16), np.int8)
        self.v = np.zeros((num_blocks, n_kv_heads, head_dim, block_size), np.int8)
        self.k_scale = np.zeros((num_blocks, n_kv_heads, block_size), np.float32)
        self.v_scale = np.zeros((num_blocks, n_kv_heads, block_size), np.float32)

    def struct(self):
        s = _CCache(_ptr(self.k), _ptr(self.v), _ptr(self.k_scale), _ptr(self.v_scale),
                    self.num_blocks, self.block_size, self.n_kv_heads, self.head_dim)
        return s


def kv_bytes_per_token(n_kv_heads, head_dim):
    return int(_load().oracle_kv_bytes_per_token(n_kv_heads, head_dim))


def bf16_kv_bytes_per_token(n_kv_heads, head_dim):
    return int(_load().oracle_bf16_kv_bytes_per_token(n_kv_heads, head_dim))


def quant_rows(x_bf16):
    """Per-row absmax int8 quantisation of bf16 rows (uint16 bit patterns, [..., n])."""
    x = _c(x_bf16, np.uint16)
    n = x.shape[-1]
    rows = x.size // n
    codes = np.zeros(x.shape, np.int8)
    scales = np.zeros(x.shape[:-1], np.float32)
    _load().oracle_quant_rows(_ptr(x), rows, n, _ptr(codes), _ptr(scales))
    return codes, scales


def kv_quant_write(cache, k_new, v_new, seq_idx, pos, block_table):
    """Quantise new K/V rows ([T][Hkv][D] bf16 bits) into `cache`; returns #skipped."""
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    seq_idx, pos = _c(seq_idx, np.int32), _c(pos, np.int32)
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt[None, :]
    s = cache.struct()
    return int(_load().oracle_kv_quant_write(ctypes.byref(s), _ptr(k_new), _ptr(v_new),
                                             len(seq_idx), _ptr(seq_idx), _ptr(pos), _ptr(bt),
                                             bt.shape[0], bt.shape[1]))


def rope_quant_write(cache, q, k_new, v_new, seq_idx, pos, block_table, cos_sin, rotary_dim):
    """Fused producer: RoPE on Q and K (table cos_sin [max_pos][rotary_dim] fp32), then the
    quantisation rule; K/V into `cache`.  q: bf16 bits [T][Hq][D] or None.  Returns
    (skipped, q_codes int8 [T][Hq][D], q_scales fp32 [T][Hq], q_rot bf16 bits [T][Hq][D])."""
    k_new, v_new = _c(k_new, np.uint16), _c(v_new, np.uint16)
    seq_idx, pos = _c(seq_idx, np.int32), _c(pos, np.int32)
    cs = _c(cos_sin, np.float32)
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt[None, :]
    T = len(seq_idx)
    D = cache.head_dim
    if q is not None:
        q = _c(q, np.uint16)
        Hq = q.shape[1]
    else:
        Hq = 0
    qc = np.zeros((T, Hq, D), np.int8)
    qs = np.zeros((T, Hq), np.float32)
    qr = np.zeros((T, Hq, D), np.uint16)
    s = cache.struct()
    skipped = int(_load().oracle_rope_quant_write(
        ctypes.byref(s), _ptr(q) if q is not None else None, Hq, _ptr(k_new), _ptr(v_new), T,
        _ptr(seq_idx), _ptr(pos), _ptr(bt), bt.shape[0], bt.shape[1], _ptr(cs), cs.shape[0],
        int(rotary_dim), _ptr(qc), _ptr(qs), _ptr(qr)))
    return skipped, qc, qs, qr


def _units_arg(units):
    if units is None:
        return None, 0
    u = _c(units, np.int64)
    return u, len(u)


def decode_f64(cache, q, block_table, ctx_lens, scale, units=None, n_threads=0):
    """Part A decode: q bf16 bits [B][Hq][D] -> float64 [B][Hq][D] (or [n_units][D])."""
    q = _c(q, np.uint16)
    bt, ctx = _c(block_table, np.int32), _c(ctx_lens, np.int32)
    B, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((B, Hq, D) if u is None else (nu, D), np.float64)
    s = cache.struct()
    _load().oracle_decode_f64(ctypes.byref(s), _ptr(q), B, Hq, _ptr(bt), bt.shape[1], _ptr(ctx),
                              float(scale), _ptr(u), nu, _ptr(out), n_threads)
    return out


def verify_f64(cache, q, block_table, ctx_lens, scale, units=None, n_threads=0):
    """Part A verify decode: q bf16 bits [B][nq][Hq][D] -> float64 [B][nq][Hq][D] (or
    [n_units][D]).  Row i of sequence b sees keys t < ctx_lens[b] - nq + 1 + i."""
    q = _c(q, np.uint16)
    bt, ctx = _c(block_table, np.int32), _c(ctx_lens, np.int32)
    B, nq, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((B, nq, Hq, D) if u is None else (nu, D), np.float64)
    s = cache.struct()
    _load().oracle_verify_f64(ctypes.byref(s), _ptr(q), B, nq, Hq, _ptr(bt), bt.shape[1], _ptr(ctx),
                              float(scale), _ptr(u), nu, _ptr(out), n_threads)
    return out


def decode_split_f64(cache, q, block_table, ctx_lens, scale, split_rows, n_threads=0):
    """Decode through per-split partials and the log-sum-exp merge (FP64)."""
    q = _c(q, np.uint16)
    bt, ctx = _c(block_table, np.int32), _c(ctx_lens, np.int32)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D), np.float64)
    s = cache.struct()
    _load().oracle_decode_split_f64(ctypes.byref(s), _ptr(q), B, Hq, _ptr(bt), bt.shape[1],
                                    _ptr(ctx), float(scale), int(split_rows), _ptr(out),
                                    n_threads)
    return out


def prefill_ref_f64(cache, q, history, bt_row, scale, units=None, n_threads=0):
    """Part A prefill chunk: q bf16 bits [T][Hq][D] -> float64."""
    q = _c(q, np.uint16)
    bt = _c(bt_row, np.int32)
    T, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((T, Hq, D) if u is None else (nu, D), np.float64)
    s = cache.struct()
    _load().oracle_prefill_ref_f64(ctypes.byref(s), _ptr(q), T, Hq, int(history), _ptr(bt),
                                   float(scale), _ptr(u), nu, _ptr(out), n_threads)
    return out


def prefill_qdeq_f64(cache, q, history, bt_row, scale, pv_tile=PV_TILE, units=None, n_threads=0):
    """The method's prefill with exact softmax: Q quantised to its codes and dequantised,
    FP64 attention, no P quantisation.  Returns (out, bound, mag), each float64 [T][Hq][D] (or
    [n_units][D]): bound is the largest change the per-tile P re-quantisation can make to each
    output element, mag = sum_t p_t |v^_t| / l (the scale of fp32 rounding effects)."""
    q = _c(q, np.uint16)
    bt = _c(bt_row, np.int32)
    T, Hq, D = q.shape
    u, nu = _units_arg(units)
    shape = (T, Hq, D) if u is None else (nu, D)
    out, bound, mag = (np.zeros(shape, np.float64) for _ in range(3))
    s = cache.struct()
    _load().oracle_prefill_qdeq_f64(ctypes.byref(s), _ptr(q), T, Hq, int(history), _ptr(bt), float(scale),
                                    int(pv_tile), _ptr(u), nu, _ptr(out), _ptr(bound), _ptr(mag), n_threads)
    return out, bound, mag


def prefill_first_f64(q, k, v, scale, units=None, n_threads=0):
    """The first prefill chunk in high precision: causal attention of q bf16 bits [T][Hq][D] over
    the chunk's own bf16 k, v [T][Hkv][D] (no quantisation) -> float64 [T][Hq][D] (or [n_units][D])."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    T, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((T, Hq, D) if u is None else (nu, D), np.float64)
    _load().oracle_prefill_first_f64(_ptr(q), _ptr(k), _ptr(v), T, Hq, k.shape[1], D, float(scale), _ptr(u), nu,
                                     _ptr(out), n_threads)
    return out


def prefill_int8_emul(cache, q, history, bt_row, scale, pv_tile=PV_TILE, units=None,
                      n_threads=0, want_q_codes=False):
    """Part B prefill chunk (int8 Q, exact integer QK, per-tile int8 P, exact PV)."""
    q = _c(q, np.uint16)
    bt = _c(bt_row, np.int32)
    T, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((T, Hq, D) if u is None else (nu, D), np.float64)
    qc = np.zeros((T, Hq, D), np.int8) if want_q_codes else None
    qs = np.zeros((T, Hq), np.float32) if want_q_codes else None
    s = cache.struct()
    _load().oracle_prefill_int8_emul(ctypes.byref(s), _ptr(q), T, Hq, int(history), _ptr(bt),
                                     float(scale), int(pv_tile), _ptr(u), nu, _ptr(out),
                                     _ptr(qc), _ptr(qs), n_threads)
    return (out, qc, qs) if want_q_codes else out


def exp2_det(x):
    """The deterministic fp32 exp2 the prefill P-code decisions use (scalar)."""
    return float(_load().oracle_exp2_det(float(x)))


def prefill_qk_int32(q_codes, cache, bt_row, q_head, q0, nq, k0, nk):
    """Exact integer QK window [nq][nk] (no mask)."""
    qc = _c(q_codes, np.int8)
    bt = _c(bt_row, np.int32)
    T, Hq, D = qc.shape
    out = np.zeros((nq, nk), np.int32)
    s = cache.struct()
    _load().oracle_prefill_qk_int32(_ptr(qc), T, Hq, ctypes.byref(s), _ptr(bt), int(q_head),
                                    int(q0), int(nq), int(k0), int(nk), _ptr(out))
    return out


def sparse_f64(cache, q, offsets, cells, bt_row, scale, units=None, n_threads=0):
    """Part A sparse attention over per-query cell lists."""
    q = _c(q, np.uint16)
    off, cl, bt = _c(offsets, np.int32), _c(cells, np.int32), _c(bt_row, np.int32)
    N, Hq, D = q.shape
    u, nu = _units_arg(units)
    out = np.zeros((N, Hq, D) if u is None else (nu, D), np.float64)
    s = cache.struct()
    _load().oracle_sparse_f64(ctypes.byref(s), _ptr(q), N, Hq, _ptr(off), _ptr(cl), _ptr(bt),
                              float(scale), _ptr(u), nu, _ptr(out), n_threads)
    return out
