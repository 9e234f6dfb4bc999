"""Python binding of libpa: the C-ABI calls with the same names, taking torch
tensors.  Argument marshalling only: every step of the computation runs in
the library's CUDA kernels.  If libpa.so is missing the calls raise; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_DEV_SLOT_RANGE, PA_DEV_BLOCK_RANGE, PA_DEV_QSL, PA_DEV_LENGTHS, PA_DEV_CAPACITY = 1, 2, 4, 8, 16
PA_DEV_TIMEOUT = 32

_DTYPES = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}


class pa_layout(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_size", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("dtype", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class PaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpa error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpa.so (built in-tree by paged_kv_attention_04_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_attention_04_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lp = ctypes.POINTER(pa_layout)
        L.pa_cache_write.argtypes = [vp, vp, vp, i32, vp, vp, lp, vp, vp]
        L.pa_cache_write.restype = i32
        L.pa_forward_workspace_size.argtypes = [lp, i32, i32, i32]
        L.pa_forward_workspace_size.restype = sz
        L.pa_forward.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                 vp, vp, sz, lp, vp, vp]
        L.pa_forward.restype = i32
        L.pa_last_error.argtypes = []
        L.pa_last_error.restype = ctypes.c_char_p
        L.pa_forward_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                         ctypes.c_float, vp, lp, vp, vp]
        L.pa_forward_noalloc.restype = i32
        L.pa_set_profile_events.argtypes = [vp, vp]
        L.pa_set_profile_events.restype = i32
        L.pa_set_prefill_profile_events.argtypes = [vp, vp]
        L.pa_set_prefill_profile_events.restype = i32
        L.pa_set_prefill_overlap.argtypes = [i32]
        L.pa_set_prefill_overlap.restype = i32
        L.pa_version.argtypes = []
        L.pa_version.restype = i32
        _lib = L
    return _lib


def last_error() -> str:
    return lib().pa_last_error().decode()


def _check(rc: int):
    if rc != PA_OK:
        raise PaError(rc, last_error())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _on_one_device(**tensors) -> None:
    """Every tensor argument must be a contiguous CUDA tensor, all on one
    device (a host pointer would reach the kernels unchecked)."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise PaError(PA_ERR_INVALID, f"{name} is not a CUDA tensor")
        if not t.is_contiguous():
            raise PaError(PA_ERR_INVALID, f"{name} is not contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise PaError(PA_ERR_INVALID, f"{name} is on {t.device}, expected {dev}")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_layout(num_q_heads: int, num_kv_heads: int, head_size: int, num_blocks: int,
                dtype, block_size: int = 16, cache_dtype=None, k_scale: float = 1.0,
                v_scale: float = 1.0) -> pa_layout:
    """Layout of a step; cache_dtype defaults to dtype (PA_FP8_E4M3 for an 8-bit cache)."""
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    if cache_dtype is None:
        ccode = code
    elif isinstance(cache_dtype, torch.dtype):
        ccode = PA_FP8_E4M3 if cache_dtype == torch.uint8 else _DTYPES[cache_dtype]
    else:
        ccode = int(cache_dtype)
    return pa_layout(num_q_heads, num_kv_heads, head_size, block_size, num_blocks, code, ccode,
                     float(k_scale), float(v_scale))


def layout_of(k_cache: torch.Tensor, num_q_heads: int, dtype=None, k_scale: float = 1.0,
              v_scale: float = 1.0) -> pa_layout:
    """Layout of a cache tensor [num_blocks][block_size][num_kv_heads][head_size].  A
    uint8 cache holds FP8 (E4M3) codes; then `dtype` (of q/out, default bf16) and the
    scales apply."""
    nb, bs, hkv, d = k_cache.shape
    if k_cache.dtype == torch.uint8:
        return make_layout(num_q_heads, hkv, d, nb, dtype or torch.bfloat16, bs, PA_FP8_E4M3,
                           k_scale, v_scale)
    return make_layout(num_q_heads, hkv, d, nb, k_cache.dtype, bs)


def pa_cache_write(k, v, slot_mapping, k_cache, v_cache, layout: pa_layout,
                   status: torch.Tensor | None = None, stream=None) -> None:
    """Write k[t], v[t] into slot slot_mapping[t] of the caches (in place)."""
    _on_one_device(k=k, v=v, slot_mapping=slot_mapping, k_cache=k_cache, v_cache=v_cache,
                   status=status)
    _check(lib().pa_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]),
                                _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout),
                                _ptr(status), _stream(stream)))


def pa_forward_workspace_size(layout: pa_layout, num_seqs: int, num_tokens: int,
                              max_seq_len: int) -> int:
    n = lib().pa_forward_workspace_size(ctypes.byref(layout), int(num_seqs), int(num_tokens),
                                        int(max_seq_len))
    if n == 0:
        raise PaError(PA_ERR_INVALID, last_error())
    return int(n)


def pa_forward(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
               max_query_len: int, max_seq_len: int, scale: float, out, workspace,
               layout: pa_layout, status: torch.Tensor | None = None, stream=None) -> None:
    """Attention for every row of the flattened step, written into `out`."""
    _on_one_device(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                   seq_lens=seq_lens, query_start_loc=query_start_loc, out=out,
                   workspace=workspace, status=status)
    _check(lib().pa_forward(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            int(block_tables.shape[1]), _ptr(seq_lens), _ptr(query_start_loc),
                            int(seq_lens.shape[0]), int(q.shape[0]), int(max_query_len),
                            int(max_seq_len), float(scale), _ptr(out), _ptr(workspace),
                            int(workspace.numel() * workspace.element_size()),
                            ctypes.byref(layout), _ptr(status), _stream(stream)))


def pa_forward_noalloc(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc,
                       max_query_len: int, max_seq_len: int, scale: float, out,
                       layout: pa_layout, status: torch.Tensor | None = None, stream=None) -> None:
    """pa_forward using the library's built-in device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _on_one_device(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                   seq_lens=seq_lens, query_start_loc=query_start_loc, out=out, status=status)
    _check(lib().pa_forward_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                    int(block_tables.shape[1]), _ptr(seq_lens),
                                    _ptr(query_start_loc), int(seq_lens.shape[0]), int(q.shape[0]),
                                    int(max_query_len), int(max_seq_len), float(scale), _ptr(out),
                                    ctypes.byref(layout), _ptr(status), _stream(stream)))


def _event_handles(start, stop) -> list:
    """CUDA handles of two torch events (None stays None).  torch creates an
    event's handle on its first record, so unrecorded events are recorded once
    here first."""
    handles = []
    for ev in (start, stop):
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:
            ev.record()
        handles.append(ev.cuda_event)
    return handles


def pa_set_profile_events(start: "torch.cuda.Event | None", stop: "torch.cuda.Event | None") -> None:
    """Record `start`/`stop` around the decode-attention kernel of later
    pa_forward calls on this thread (None, None turns it off)."""
    _check(lib().pa_set_profile_events(*_event_handles(start, stop)))


def pa_set_prefill_profile_events(start: "torch.cuda.Event | None",
                                  stop: "torch.cuda.Event | None") -> None:
    """Record `start`/`stop` around the tensor-core prefill kernel of later
    pa_forward calls on this thread, on the stream it runs on (None, None
    turns it off)."""
    _check(lib().pa_set_prefill_profile_events(*_event_handles(start, stop)))


def pa_set_prefill_overlap(on: bool) -> None:
    """True (the default): the prefill kernel runs on a side stream beside the
    decode kernel; False: on the caller's stream before it."""
    _check(lib().pa_set_prefill_overlap(1 if on else 0))


def alloc_workspace(layout: pa_layout, num_seqs: int, num_tokens: int, max_seq_len: int,
                    device="cuda") -> torch.Tensor:
    """Caller-owned workspace for pa_forward (torch's allocator aligns to >= 256 bytes)."""
    n = pa_forward_workspace_size(layout, num_seqs, num_tokens, max_seq_len)
    return torch.empty(n, dtype=torch.uint8, device=device)
