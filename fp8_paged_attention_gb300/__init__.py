"""Paged FP8 (E4M3) KV-cache attention for GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/fp8pa.h`` (and the test and
tuning hooks of ``include/fp8pa_testing.h``) (library
``_lib/libfp8pa.so``, built in-tree by ``build()``).  The functions here only
marshal torch tensors into pointers and sizes; every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the library
is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "build", "load_library", "library_path", "quantize_q_fp8", "fp8_paged_attn_fwd", "workspace_size",
    "num_splits", "kernel_launches", "set_timing_events", "set_ctas_per_sm", "set_bf16_dequant_v", "get_device_status", "reset_device_status",
    "kv_cache_write", "DEV_BAD_SLOT", "lse_combine",
    "set_wait_limit", "set_stall_injection", "FP8PA_BF16", "FP8PA_E4M3",
    "DEV_BAD_PAGE", "DEV_TIMEOUT", "DEV_BAD_LENGTH", "PAGE_SIZE", "Fp8paError",
]

FP8PA_BF16 = 0
FP8PA_E4M3 = 1
DEV_BAD_PAGE = 1
DEV_TIMEOUT = 2
DEV_BAD_LENGTH = 4
DEV_BAD_SLOT = 8
PAGE_SIZE = 64

_lock = threading.Lock()
_lib = None


class Fp8paError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"fp8pa status {status}: {message}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force)


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libfp8pa.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _build.up_to_date():
            _build.build()
        lib = ctypes.CDLL(_build.LIB_PATH)
        c = ctypes
        lib.quantize_q_fp8.restype = c.c_int
        lib.quantize_q_fp8.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_longlong, c.c_void_p]
        lib.fp8pa_kv_cache_write.restype = c.c_int
        lib.fp8pa_kv_cache_write.argtypes = [
            c.c_void_p, c.c_void_p, c.c_longlong, c.c_longlong, c.c_void_p, c.c_void_p, c.c_int, c.c_void_p,
            c.c_longlong, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
        ]
        lib.fp8pa_lse_combine.restype = c.c_int
        lib.fp8pa_lse_combine.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_longlong, c.c_int, c.c_int, c.c_void_p,
                                          c.c_void_p, c.c_void_p]
        lib.fp8pa_workspace_size.restype = c.c_size_t
        lib.fp8pa_workspace_size.argtypes = [c.c_int] * 10
        lib.fp8pa_num_splits.restype = c.c_int
        lib.fp8pa_num_splits.argtypes = [c.c_int] * 10
        lib.fp8_paged_attn_fwd.restype = c.c_int
        lib.fp8_paged_attn_fwd.argtypes = [
            c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_void_p, c.c_int, c.c_void_p, c.c_void_p,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_int,
            c.c_int, c.c_float, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_size_t, c.c_void_p, c.c_void_p,
            c.c_void_p,
        ]
        lib.fp8_paged_attn_fwd_sinks.restype = c.c_int
        lib.fp8_paged_attn_fwd_sinks.argtypes = lib.fp8_paged_attn_fwd.argtypes[:-1] + [c.c_void_p, c.c_void_p]
        lib.fp8_paged_attn_fwd_noalloc.restype = c.c_int
        lib.fp8_paged_attn_fwd_noalloc.argtypes = [
            c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_void_p, c.c_int, c.c_void_p, c.c_void_p,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_int,
            c.c_int, c.c_float, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
        ]
        lib.fp8pa_get_device_status.restype = c.c_int
        lib.fp8pa_get_device_status.argtypes = [c.c_void_p, c.c_void_p]
        lib.fp8pa_reset_device_status.restype = c.c_int
        lib.fp8pa_reset_device_status.argtypes = [c.c_void_p]
        lib.fp8pa_last_error.restype = c.c_char_p
        lib.fp8pa_last_error.argtypes = []
        lib.fp8pa_set_wait_limit.restype = None
        lib.fp8pa_set_wait_limit.argtypes = [c.c_uint]
        lib.fp8pa_set_stall_injection.restype = None
        lib.fp8pa_set_stall_injection.argtypes = [c.c_int]
        lib.fp8pa_kernel_launches.restype = c.c_int
        lib.fp8pa_kernel_launches.argtypes = [c.c_int] * 10
        lib.fp8pa_set_bf16_dequant_v.restype = None
        lib.fp8pa_set_bf16_dequant_v.argtypes = [c.c_int]
        lib.fp8pa_set_ctas_per_sm.restype = None
        lib.fp8pa_set_ctas_per_sm.argtypes = [c.c_int]
        lib.fp8pa_set_grid_sms.restype = None
        lib.fp8pa_set_grid_sms.argtypes = [c.c_int]
        lib.fp8pa_set_sm_split.restype = None
        lib.fp8pa_set_sm_split.argtypes = [c.c_int]
        lib.fp8pa_set_prefill_rows.restype = None
        lib.fp8pa_set_prefill_rows.argtypes = [c.c_int]
        lib.fp8pa_set_timing_events.restype = None
        lib.fp8pa_set_timing_events.argtypes = [c.c_void_p, c.c_void_p]
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        msg = load_library().fp8pa_last_error().decode(errors="replace")
        raise Fp8paError(rc, msg)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def workspace_size(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                   window_left=-1, num_splits=0) -> int:
    return int(load_library().fp8pa_workspace_size(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv,
                                                   head_dim, q_dtype, max_pages_per_seq, window_left, num_splits))


def num_splits(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
               window_left=-1, num_splits=0) -> int:
    return int(load_library().fp8pa_num_splits(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim,
                                               q_dtype, max_pages_per_seq, window_left, num_splits))


def kernel_launches(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv, head_dim, q_dtype, max_pages_per_seq,
                    window_left=-1, num_splits=0) -> int:
    """Kernels one fp8_paged_attn_fwd call launches for these sizes."""
    return int(load_library().fp8pa_kernel_launches(batch, total_q, max_seqlen_q, num_heads_q, num_heads_kv,
                                                    head_dim, q_dtype, max_pages_per_seq, window_left, num_splits))


def set_timing_events(start=None, stop=None):
    """Profiling hook (fp8pa_testing.h): record torch.cuda.Event `start`/`stop`
    around the attention kernels of later calls on this thread (None, None: off)."""
    lib = load_library()
    if start is None or stop is None:
        lib.fp8pa_set_timing_events(None, None)
    else:
        if not start.cuda_event or not stop.cuda_event:
            raise ValueError("record the events once before passing them (torch creates them lazily)")
        lib.fp8pa_set_timing_events(start.cuda_event, stop.cuda_event)


def set_ctas_per_sm(ctas: int):
    """Tuning hook (fp8pa_testing.h): force 1 or 2 attention CTAs per SM for
    later calls on this thread (0 = automatic)."""
    load_library().fp8pa_set_ctas_per_sm(int(ctas))


def set_grid_sms(sms: int):
    """Tuning hook (fp8pa_testing.h): attention grids of later calls on this
    thread use at most `sms` SMs (0 = all)."""
    load_library().fp8pa_set_grid_sms(int(sms))


def set_sm_split(sms: int):
    """Tuning hook (fp8pa_testing.h): SMs of the prefill row class when the two
    classes run side by side, for later calls on this thread (0 = estimate)."""
    load_library().fp8pa_set_sm_split(int(sms))


def set_prefill_rows(rows: int):
    """Tuning hook (fp8pa_testing.h): rows per prefill-class tile with BF16 Q
    (32 or 64; 0 = default) for later calls on this thread."""
    load_library().fp8pa_set_prefill_rows(int(rows))


def set_bf16_dequant_v(on: bool):
    """Test hook (fp8pa_testing.h), later calls on this thread: the BF16-Q path
    runs FP8 MMAs with Q split into an exact E4M3 pair, V E4M3 and a hi/lo E4M3
    P (False, default), or the literal form with K dequantized to F16 and V to
    BF16 with a BF16 P (True)."""
    load_library().fp8pa_set_bf16_dequant_v(int(bool(on)))


def quantize_q_fp8(q: torch.Tensor, q_descale: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """E4M3 codes (uint8) of a bf16 tensor: RNE_sat(fl32(q / q_descale))."""
    lib = load_library()
    if q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA bfloat16 tensor")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    _check(lib.quantize_q_fp8(_ptr(q), _ptr(out), _ptr(q_descale), q.numel(), _stream_ptr(stream)))
    return out


def lse_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, out=None, lse=None, stream=None):
    """Merge attention partials over disjoint key shards by their LSE.

    o_parts: bf16 [P, total_q, Hq, D]; lse_parts: f32 [P, Hq, total_q] (each
    part's fp8_paged_attn_fwd out and lse).  Returns (out bf16 [total_q, Hq, D],
    lse f32 [Hq, total_q]).
    """
    lib = load_library()
    if o_parts.dtype != torch.bfloat16 or not o_parts.is_cuda or o_parts.dim() != 4 or not o_parts.is_contiguous():
        raise ValueError("o_parts must be a contiguous CUDA bfloat16 [P, total_q, Hq, D] tensor")
    P, T, hq, d = o_parts.shape
    if lse_parts.dtype != torch.float32 or tuple(lse_parts.shape) != (P, hq, T) or not lse_parts.is_contiguous():
        raise ValueError("lse_parts must be a contiguous float32 [P, Hq, total_q] tensor")
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=o_parts.device)
    _check(lib.fp8pa_lse_combine(_ptr(o_parts), _ptr(lse_parts), P, T, hq, d, _ptr(out), _ptr(lse),
                                 _stream_ptr(stream)))
    return out, lse


def kv_cache_write(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   slot_mapping: torch.Tensor, k_descale: torch.Tensor, v_descale: torch.Tensor, stream=None):
    """Quantize new keys and values to E4M3 and write them into the paged cache.

    key, value: bf16 [T, Hkv, D] CUDA tensors whose rows may be strided (a view
    into a fused QKV buffer); k_cache, v_cache: uint8 [num_pages, 64, Hkv, D];
    slot_mapping: int64 [T] (slot = page * 64 + row, negative = padding);
    descales: one f32 each on the device.  Writes in place; returns nothing.
    """
    lib = load_library()
    for name, t in (("key", key), ("value", value)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3:
            raise ValueError(f"{name} must be a CUDA bfloat16 [T, Hkv, D] tensor")
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{name}: each token row must be contiguous")
    num_pages, page, hkv, d = k_cache.shape
    if page != PAGE_SIZE or tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.dtype != torch.uint8:
        raise ValueError("k_cache / v_cache must be uint8 [num_pages, 64, Hkv, D]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache / v_cache must be contiguous")
    T = key.shape[0]
    if tuple(key.shape) != (T, hkv, d) or tuple(value.shape) != (T, hkv, d):
        raise ValueError("key / value must be [T, Hkv, D] with the cache's Hkv and D")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 tensor of T entries")
    _check(lib.fp8pa_kv_cache_write(_ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(k_cache),
                                    _ptr(v_cache), num_pages, _ptr(slot_mapping), T, hkv, d, _ptr(k_descale),
                                    _ptr(v_descale), _stream_ptr(stream)))


def fp8_paged_attn_fwd(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, max_seqlen_q, q_descale,
                       k_descale, v_descale, softmax_scale, window_left=-1, causal=True, num_splits=0,
                       out=None, lse=None, workspace=None, descale_batch_stride=0, descale_head_stride=0,
                       stream=None, return_lse=True, sinks=None):
    """Attention over a paged E4M3 KV cache.

    q: [total_q, Hq, D] bf16, or uint8 E4M3 codes (FP8-MMA path);
    k_cache, v_cache: uint8 [num_pages, 64, Hkv, D]; block_table int32 [B, max_pages];
    cu_seqlens_q int32 [B+1]; seqused_k int32 [B]; descales: f32 device tensors;
    sinks: optional f32 [Hq] device tensor of per-head sink logits (fp8_paged_attn_fwd_sinks).
    Returns (out bf16 [total_q, Hq, D], lse f32 [Hq, total_q] or None).
    """
    lib = load_library()
    if q.dtype == torch.bfloat16:
        q_dtype = FP8PA_BF16
    elif q.dtype in (torch.uint8, torch.float8_e4m3fn):
        q_dtype = FP8PA_E4M3
    else:
        raise ValueError(f"unsupported q dtype {q.dtype}")
    total_q, hq, d = q.shape
    num_pages, page, hkv, d2 = k_cache.shape
    if page != PAGE_SIZE or d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache must be [num_pages, 64, Hkv, D] with D equal to q's head dim")
    batch, max_pages = block_table.shape
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, total_q), dtype=torch.float32, device=q.device)
    need = workspace_size(batch, total_q, max_seqlen_q, hq, hkv, d, q_dtype, max_pages, window_left, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("block_table", block_table),
                    ("cu_seqlens_q", cu_seqlens_q), ("seqused_k", seqused_k), ("out", out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    args = (_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(block_table), max_pages,
            _ptr(cu_seqlens_q), _ptr(seqused_k), batch, total_q, max_seqlen_q, hq, hkv, d, _ptr(q_descale),
            _ptr(k_descale), _ptr(v_descale), descale_batch_stride, descale_head_stride, float(softmax_scale),
            int(window_left), int(bool(causal)), int(num_splits), _ptr(workspace), workspace.numel(), _ptr(out),
            _ptr(lse))
    if sinks is None:
        _check(lib.fp8_paged_attn_fwd(*args, _stream_ptr(stream)))
    else:
        if sinks.dtype != torch.float32 or not sinks.is_cuda or sinks.numel() != hq or not sinks.is_contiguous():
            raise ValueError("sinks must be a contiguous CUDA float32 tensor of num_heads_q entries")
        _check(lib.fp8_paged_attn_fwd_sinks(*args, _ptr(sinks), _stream_ptr(stream)))
    return out, lse


def get_device_status(stream=None) -> int:
    """Status bits accumulated on the current device (synchronizes the stream)."""
    lib = load_library()
    host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib.fp8pa_get_device_status(host.data_ptr(), _stream_ptr(s)))
    s.synchronize()
    return int(host.item()) & 0xFFFFFFFF


def reset_device_status(stream=None):
    _check(load_library().fp8pa_reset_device_status(_stream_ptr(stream)))


def set_wait_limit(max_iterations: int):
    """Test hook (fp8pa_testing.h): cap every bounded pipeline wait of later
    calls on this thread (0 restores the default)."""
    load_library().fp8pa_set_wait_limit(int(max_iterations))


def set_stall_injection(on: bool):
    """Test hook (fp8pa_testing.h): in later calls on this thread, every
    attention CTA's MMA thread waits on a barrier that nothing arrives on, so
    that the launch takes its bounded-wait timeout path."""
    load_library().fp8pa_set_stall_injection(int(bool(on)))
