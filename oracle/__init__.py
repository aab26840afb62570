"""The float64 CPU oracle for decode attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may
import this package. The product path (decode_attention_attn_gb300) never does.

Inputs are passed as numpy arrays holding the exact storage bits: float32 arrays for
fp32 data, uint16 arrays for fp16 / bf16 data. Every function wraps one C entry point
of decode_attn_oracle.c; see that file for the passage each one follows.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}

_lib = None


class Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("paged", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("max_seq_len", ctypes.c_int),
        ("num_physical_blocks", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("kv_e4m3", ctypes.c_int),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
    ]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        d = ctypes.c_double
        L.oracle_load.restype = d
        L.oracle_load.argtypes = [ctypes.c_int, P, i64]
        L.oracle_kv_offset.restype = i64
        L.oracle_kv_offset.argtypes = [ctypes.POINTER(Shape), P, ctypes.c_int, ctypes.c_int, i64]
        L.oracle_gather_offsets.restype = ctypes.c_int
        L.oracle_gather_offsets.argtypes = [ctypes.POINTER(Shape), P, P, P]
        L.oracle_decode_attn.restype = ctypes.c_int
        L.oracle_decode_attn.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, d, d, d, d, P,
                                         i64, P, P, P, P, ctypes.c_int]
        L.oracle_split_partial.restype = ctypes.c_int
        L.oracle_split_partial.argtypes = [ctypes.POINTER(Shape), P, P, P, P, ctypes.c_int,
                                           ctypes.c_int, P, i64, d, P, P, P, P]
        L.oracle_lse_merge.restype = ctypes.c_int
        L.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P]
        L.oracle_lse_merge_alpha.restype = ctypes.c_int
        L.oracle_lse_merge_alpha.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P]
        L.oracle_unified_row.restype = ctypes.c_int
        L.oracle_logits.argtypes = [ctypes.POINTER(Shape), P, P, P, P, d, P]
        L.oracle_logits.restype = i64
        L.oracle_unified_row.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, ctypes.c_int,
                                         ctypes.c_int, d, d, d, d, i64, P, P, P, P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a, dtype):
    a = np.ascontiguousarray(a)
    want = {"f32": np.float32, "e4m3": np.uint8}.get(dtype, np.uint16)
    if a.dtype != want:
        raise TypeError(f"oracle expects {np.dtype(want).name} storage for {dtype}, got {a.dtype}")
    return a


def make_shape(*, batch, num_q_heads, num_kv_heads, head_dim, dtype, paged=False, page_size=16,
               max_blocks_per_seq=0, max_seq_len=0, num_physical_blocks=0, kv_dtype=None,
               k_scale=1.0, v_scale=1.0):
    """dtype: q's storage (and K / V's, unless kv_dtype="e4m3": an FP8 cache whose codes
    stand for code * k_scale and code * v_scale)."""
    if kv_dtype not in (None, dtype, "e4m3"):
        raise ValueError("K / V are stored like q or as e4m3")
    fp8 = kv_dtype == "e4m3"
    return Shape(batch, num_q_heads, num_kv_heads, head_dim, int(bool(paged)), page_size,
                 max_blocks_per_seq, max_seq_len, num_physical_blocks, DTYPE_CODES[dtype],
                 int(fp8), k_scale if fp8 else 0.0, v_scale if fp8 else 0.0)


def _dtype_name(shape):
    return {v: k for k, v in DTYPE_CODES.items()}[shape.dtype]


def _kv_dtype_name(shape):
    return "e4m3" if shape.kv_e4m3 else _dtype_name(shape)


def load(dtype, arr, index):
    arr = _bits(arr, dtype)
    return lib().oracle_load(DTYPE_CODES[dtype], _ptr(arr), index)


def decode_attn(shape, q, k, v, block_table, seq_lens, scale, phi=0.0, range_lo=-math.inf,
                range_hi=math.inf, rows=None, nthreads=1):
    """Returns (out [n, d] float64, lse [n], row_flag [n] uint8, margin [n])."""
    dt, kdt = _dtype_name(shape), _kv_dtype_name(shape)
    q, k, v = _bits(q, dt), _bits(k, kdt), _bits(v, kdt)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = shape.batch * shape.num_q_heads if rows_a is None else rows_a.size
    out = np.zeros((n, shape.head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    flag = np.zeros(n, np.uint8)
    margin = np.zeros(n, np.float64)
    rc = lib().oracle_decode_attn(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                                  _ptr(sl), scale, phi, range_lo, range_hi, _ptr(rows_a),
                                  0 if rows_a is None else rows_a.size, _ptr(out), _ptr(lse),
                                  _ptr(flag), _ptr(margin), nthreads)
    if rc:
        raise ValueError("oracle_decode_attn rejected its arguments")
    return out, lse, flag, margin


def gather_offsets(shape, block_table, seq_lens):
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    T = shape.max_blocks_per_seq * shape.page_size if shape.paged else shape.max_seq_len
    offs = np.zeros((shape.batch, shape.num_kv_heads, T), np.int64)
    if lib().oracle_gather_offsets(ctypes.byref(shape), _ptr(bt), _ptr(sl), _ptr(offs)):
        raise ValueError("oracle_gather_offsets rejected its arguments")
    return offs


def logits(shape, q, k, block_table, seq_lens, scale):
    """Every row's scaled logits in row order (b * H_q + h_q), tokens in order: float64."""
    dt, kdt = _dtype_name(shape), _kv_dtype_name(shape)
    q, k = _bits(q, dt), _bits(k, kdt)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros(int(sl.astype(np.int64).sum()) * shape.num_q_heads, np.float64)
    n = lib().oracle_logits(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(bt), _ptr(sl), scale,
                            _ptr(out))
    if n != out.size:
        raise ValueError("oracle_logits rejected its arguments")
    return out


def split_partial(shape, q, k, v, block_table, b, h, tokens, scale):
    """Returns (O_s [d], m_s, l_s, L_s) for the given token indices."""
    dt, kdt = _dtype_name(shape), _kv_dtype_name(shape)
    q, k, v = _bits(q, dt), _bits(k, kdt), _bits(v, kdt)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    o = np.zeros(shape.head_dim, np.float64)
    m, l, L = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    rc = lib().oracle_split_partial(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                                    b, h, _ptr(tok), tok.size, scale, _ptr(o), ctypes.byref(m),
                                    ctypes.byref(l), ctypes.byref(L))
    if rc:
        raise ValueError("oracle_split_partial rejected its arguments")
    return o, m.value, l.value, L.value


def lse_merge(o_s, m_s, l_s):
    o_s = np.ascontiguousarray(o_s, np.float64)
    S, d = o_s.shape
    m_s = np.ascontiguousarray(m_s, np.float64)
    l_s = np.ascontiguousarray(l_s, np.float64)
    o = np.zeros(d, np.float64)
    lse = ctypes.c_double()
    if lib().oracle_lse_merge(S, d, _ptr(o_s), _ptr(m_s), _ptr(l_s), _ptr(o), ctypes.byref(lse)):
        raise ValueError("oracle_lse_merge rejected its arguments")
    return o, lse.value


def lse_merge_alpha(o_s, L_s):
    o_s = np.ascontiguousarray(o_s, np.float64)
    S, d = o_s.shape
    L_s = np.ascontiguousarray(L_s, np.float64)
    o = np.zeros(d, np.float64)
    lse = ctypes.c_double()
    if lib().oracle_lse_merge_alpha(S, d, _ptr(o_s), _ptr(L_s), _ptr(o), ctypes.byref(lse)):
        raise ValueError("oracle_lse_merge_alpha rejected its arguments")
    return o, lse.value


def unified_row(shape, q, k, v, block_table, seq_lens, b, h, scale, phi, range_lo, range_hi,
                split_tokens=0):
    """Returns (out [d], lse, flag, flagged_partitions) of the unified-max form."""
    dt, kdt = _dtype_name(shape), _kv_dtype_name(shape)
    q, k, v = _bits(q, dt), _bits(k, kdt), _bits(v, kdt)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros(shape.head_dim, np.float64)
    lse = ctypes.c_double()
    flag = ctypes.c_uint8()
    nflag = ctypes.c_int64()
    rc = lib().oracle_unified_row(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                                  _ptr(sl), b, h, scale, phi, range_lo, range_hi, split_tokens,
                                  _ptr(out), ctypes.byref(lse), ctypes.byref(flag),
                                  ctypes.byref(nflag))
    if rc:
        raise ValueError("oracle_unified_row rejected its arguments")
    return out, lse.value, flag.value, nflag.value


def host_threads():
    """Host cores this process may use (the oracle's OpenMP thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
