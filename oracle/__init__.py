"""Python access to the plain CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports this module and shares no code with it.

The arithmetic lives in ``oracle.c`` (fp64, closed-form E4M3 decode,
round-to-nearest-even saturating encode, direct masked softmax attention read
through the block table).  This module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _AttnArgs(ctypes.Structure):
    _fields_ = [
        ("q_is_e4m3", ctypes.c_int),
        ("q", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_int),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("seqused_k", ctypes.c_void_p),
        ("batch", ctypes.c_int),
        ("total_q", ctypes.c_int),
        ("num_heads_q", ctypes.c_int),
        ("num_heads_kv", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("q_descale", ctypes.c_float),
        ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p),
        ("descale_batch_stride", ctypes.c_int),
        ("descale_head_stride", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("window_left", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("sinks", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.or_e4m3_decode.restype = ctypes.c_double
            lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.or_e4m3_encode.restype = ctypes.c_uint8
            lib.or_e4m3_encode.argtypes = [ctypes.c_float]
            lib.or_e4m3_encode_array.restype = None
            lib.or_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.or_quantize_q.restype = None
            lib.or_quantize_q.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p]
            lib.or_kv_cache_write.restype = ctypes.c_int64
            lib.or_kv_cache_write.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64,
            ]
            lib.or_lse_combine.restype = None
            lib.or_lse_combine.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
            lib.or_visible_range.restype = ctypes.c_int
            lib.or_visible_range.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int)] * 2
            lib.or_paged_attention.restype = ctypes.c_int
            lib.or_paged_attention.argtypes = [
                ctypes.POINTER(_AttnArgs), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int,
            ]
            lib.or_attention_probs.restype = ctypes.c_int
            lib.or_attention_probs.argtypes = [
                ctypes.POINTER(_AttnArgs), ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p,
            ]
            lib.or_page_size.restype = ctypes.c_int
            _lib = lib
    return _lib


PAGE = 64


def e4m3_decode(codes) -> np.ndarray:
    """Closed-form value of each E4M3 code (float64; NaN for 0x7F / 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.or_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even, saturating E4M3 encode of fp32 values."""
    lib = _load()
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    lib.or_e4m3_encode_array(a.ctypes.data, a.size, out.ctypes.data)
    return out


def quantize_q(q_bf16_bits, q_descale: float) -> np.ndarray:
    """q8 = E4M3_RNE_sat(fl32(q / q_descale)) for bf16 bit patterns (uint16)."""
    lib = _load()
    q = np.ascontiguousarray(q_bf16_bits, dtype=np.uint16)
    out = np.empty(q.shape, dtype=np.uint8)
    lib.or_quantize_q(q.ctypes.data, q.size, float(q_descale), out.ctypes.data)
    return out


def kv_cache_write(key_bits, value_bits, slot_mapping, k_descale: float, v_descale: float, k_cache, v_cache):
    """Quantize and scatter new keys and values into the paged cache, in place.

    key_bits, value_bits: uint16 bf16 bit patterns [T, Hkv, D] (or [T, row] with
    any token stride); slot_mapping: int64 [T]; k_cache, v_cache: uint8
    [num_pages, 64, Hkv, D], modified in place.  Returns the number of slots
    past the cache (skipped)."""
    lib = _load()
    k = np.asarray(key_bits)
    v = np.asarray(value_bits)
    assert k.dtype == np.uint16 and v.dtype == np.uint16
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    num_pages, page, hkv, d = k_cache.shape
    assert page == PAGE and v_cache.shape == k_cache.shape
    T = k.shape[0]
    k2 = k.reshape(T, -1)
    v2 = v.reshape(T, -1)
    assert k2.shape[1] == hkv * d and v2.shape[1] == hkv * d
    # rows may be strided (a view into a wider buffer); elements within a row are contiguous
    assert k2.strides[1] == 2 and v2.strides[1] == 2
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert sm.shape == (T,)
    return int(lib.or_kv_cache_write(k2.ctypes.data, v2.ctypes.data, k2.strides[0] // 2, v2.strides[0] // 2,
                                     sm.ctypes.data, T, hkv, d, float(k_descale), float(v_descale),
                                     k_cache.ctypes.data, v_cache.ctypes.data, num_pages))


def lse_combine(o_parts_bits, lse_parts):
    """Merge attention partials over disjoint key sets by their LSE.

    o_parts_bits: uint16 bf16 patterns [P, total_q, Hq, D]; lse_parts: f32
    [P, Hq, total_q].  Returns (out fp64 [total_q, Hq, D], lse fp64 [Hq, total_q])."""
    lib = _load()
    o = np.ascontiguousarray(o_parts_bits, dtype=np.uint16)
    ls = np.ascontiguousarray(lse_parts, dtype=np.float32)
    P, T, hq, d = o.shape
    assert ls.shape == (P, hq, T)
    out = np.empty((T, hq, d), dtype=np.float64)
    lse = np.empty((hq, T), dtype=np.float64)
    lib.or_lse_combine(o.ctypes.data, ls.ctypes.data, P, T, hq, d, out.ctypes.data, lse.ctypes.data)
    return out, lse


def visible_range(Lq: int, Lk: int, i: int, window_left: int, causal: bool):
    """(lo, hi) key range of query i, or None when it is empty."""
    lib = _load()
    lo, hi = ctypes.c_int(), ctypes.c_int()
    ok = lib.or_visible_range(Lq, Lk, i, window_left, int(bool(causal)), ctypes.byref(lo), ctypes.byref(hi))
    return (lo.value, hi.value) if ok else None


class AttnProblem:
    """The inputs of one paged-attention call, as host numpy arrays.

    q: uint8 E4M3 codes (q_is_e4m3=True) or uint16 bf16 bits, [total_q, Hq, D]
    k_cache, v_cache: uint8 [num_pages, 64, Hkv, D]
    block_table: int32 [batch, max_pages_per_seq]; cu_seqlens_q: int32 [batch+1];
    seqused_k: int32 [batch]; k/v descales: float32 arrays indexed
    b * descale_batch_stride + hk * descale_head_stride.
    """

    def __init__(self, q, q_is_e4m3, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, num_heads_kv,
                 q_descale, k_descale, v_descale, softmax_scale, window_left=-1, causal=True,
                 descale_batch_stride=0, descale_head_stride=0, sinks=None):
        self.q = np.ascontiguousarray(q)
        self.q_is_e4m3 = bool(q_is_e4m3)
        assert self.q.dtype == (np.uint8 if self.q_is_e4m3 else np.uint16)
        self.k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
        self.v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
        self.block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        self.cu_seqlens_q = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.seqused_k = np.ascontiguousarray(seqused_k, dtype=np.int32)
        self.num_heads_kv = int(num_heads_kv)
        self.q_descale = float(q_descale)
        self.k_descale = np.ascontiguousarray(np.atleast_1d(k_descale), dtype=np.float32)
        self.v_descale = np.ascontiguousarray(np.atleast_1d(v_descale), dtype=np.float32)
        self.softmax_scale = float(softmax_scale)
        self.window_left = int(window_left)
        self.causal = bool(causal)
        self.descale_batch_stride = int(descale_batch_stride)
        self.descale_head_stride = int(descale_head_stride)
        # per query head sink logits (natural-log units), or None
        self.sinks = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
        if self.sinks is not None:
            assert self.sinks.shape == (self.q.shape[1],)

    @property
    def total_q(self):
        return self.q.shape[0]

    @property
    def num_heads_q(self):
        return self.q.shape[1]

    @property
    def head_dim(self):
        return self.q.shape[2]

    @property
    def batch(self):
        return self.seqused_k.shape[0]

    def _args(self) -> _AttnArgs:
        a = _AttnArgs()
        a.q_is_e4m3 = int(self.q_is_e4m3)
        a.q = self.q.ctypes.data
        a.k_cache = self.k_cache.ctypes.data
        a.v_cache = self.v_cache.ctypes.data
        a.num_pages = self.k_cache.shape[0]
        a.block_table = self.block_table.ctypes.data
        a.max_pages_per_seq = self.block_table.shape[1]
        a.cu_seqlens_q = self.cu_seqlens_q.ctypes.data
        a.seqused_k = self.seqused_k.ctypes.data
        a.batch = self.batch
        a.total_q = self.total_q
        a.num_heads_q = self.num_heads_q
        a.num_heads_kv = self.num_heads_kv
        a.head_dim = self.head_dim
        a.q_descale = self.q_descale
        a.k_descale = self.k_descale.ctypes.data
        a.v_descale = self.v_descale.ctypes.data
        a.descale_batch_stride = self.descale_batch_stride
        a.descale_head_stride = self.descale_head_stride
        a.softmax_scale = self.softmax_scale
        a.window_left = self.window_left
        a.causal = int(self.causal)
        a.sinks = None if self.sinks is None else self.sinks.ctypes.data
        return a


def paged_attention(prob: AttnProblem, rows=None, threads: int = 0):
    """fp64 attention.  rows=None: every (token, head), returning
    out [total_q, Hq, D] and lse [Hq, total_q].  rows = int array [n, 2] of
    (token, head): returns out [n, D] and lse [n]."""
    lib = _load()
    a = _args_keep = prob._args()
    if rows is None:
        n = prob.total_q * prob.num_heads_q
        out = np.zeros((n, prob.head_dim), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        rc = lib.or_paged_attention(ctypes.byref(a), None, 0, out.ctypes.data, lse.ctypes.data, threads)
        _check(rc)
        return (out.reshape(prob.total_q, prob.num_heads_q, prob.head_dim),
                np.ascontiguousarray(lse.reshape(prob.total_q, prob.num_heads_q).T))
    r = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
    out = np.zeros((r.shape[0], prob.head_dim), dtype=np.float64)
    lse = np.zeros((r.shape[0],), dtype=np.float64)
    rc = lib.or_paged_attention(ctypes.byref(a), r.ctypes.data, r.shape[0], out.ctypes.data, lse.ctypes.data,
                                threads)
    del _args_keep
    _check(rc)
    return out, lse


def attention_probs(prob: AttnProblem, token: int, head: int):
    """(probs over keys 0..Lk-1, out row, lse) for one query row."""
    lib = _load()
    a = prob._args()
    b = int(np.searchsorted(prob.cu_seqlens_q, token, side="right") - 1)
    Lk = int(prob.seqused_k[b])
    probs = np.zeros((max(Lk, 1),), dtype=np.float64)
    o = np.zeros((prob.head_dim,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    rc = lib.or_attention_probs(ctypes.byref(a), token, head, probs.ctypes.data, o.ctypes.data, lse.ctypes.data)
    _check(rc)
    return probs[:Lk], o, float(lse[0])


def _check(rc: int):
    if rc != 0:
        raise ValueError({-1: "block table holds a page id outside the cache",
                          -2: "row names a token outside every sequence",
                          -3: "bad head counts",
                          -4: "bad sequence lengths"}.get(rc, f"oracle error {rc}"))
