"""ctypes binding of libpkv.so: the C ABI declared in include/pkv.h, one Python
function per C entry point with the same name.

Argument marshalling only: shapes are read off the tensors, pointers and the
current CUDA stream are passed through, return codes become exceptions.  Every
step of the computation runs in the library's kernels.  There is no fallback:
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
PKV_ERR_ARG = -1
PKV_ERR_OOM = -2
PKV_ERR_RANGE = -3
PKV_ERR_UNSUPPORTED = -4
PKV_ERR_CUDA = -5
PKV_ERR_TIMEOUT = -6
PKV_ERR_SHARED = -7
PKV_ERR_WORKSPACE = -8

PKV_STATUS_BAD_SLOT = 1
PKV_STATUS_BAD_BLOCK = 2
PKV_STATUS_BAD_LEN = 4
PKV_STATUS_TIMEOUT = 8
PKV_STATUS_BAD_QSTART = 16
PKV_STATUS_BAD_ITEM = 32

PKV_DECODE_OVERLAP = 1

_c_int, _c_i64, _c_ptr, _c_size, _c_float = (ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_float)

class StepConfig(ctypes.Structure):
    """pkv_step_config."""
    _fields_ = [("num_layers", _c_int), ("max_seqs", _c_int), ("q_len", _c_int), ("num_q_heads", _c_int),
                ("num_kv_heads", _c_int), ("head_dim", _c_int), ("block_size", _c_int), ("num_blocks", _c_int),
                ("max_blocks_per_seq", _c_int), ("partition_size", _c_int), ("scale", _c_float),
                ("use_graph", _c_int)]


class StepLayout(ctypes.Structure):
    """pkv_step_layout (byte offsets and sizes)."""
    _fields_ = [(n, _c_size) for n in ("q_offset", "q_layer_bytes", "k_offset", "v_offset", "kv_layer_bytes",
                                       "slots_offset", "tables_offset", "lens_offset", "stage_bytes",
                                       "out_layer_bytes", "out_bytes", "workspace_bytes", "items_offset")] \
        + [("max_items", _c_int), ("layer_stride", _c_size)]


# name -> (restype, argtypes); mirrors include/pkv.h
SIGNATURES = {
    "pkv_step_layout_of": (_c_int, [ctypes.POINTER(StepConfig), ctypes.POINTER(StepLayout)]),
    "pkv_step_create": (_c_int, [ctypes.POINTER(StepConfig), _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                 _c_ptr, _c_ptr, _c_size, _c_ptr, ctypes.POINTER(_c_ptr)]),
    "pkv_step_destroy": (None, [_c_ptr]),
    "pkv_step_run": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_ptr]),
    "pkv_step_wait": (_c_int, [_c_ptr]),
    "pkv_error_string": (ctypes.c_char_p, [_c_int]),
    "pkv_last_cuda_error": (ctypes.c_char_p, []),
    "pkv_write": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_int,
                           _c_int, _c_ptr, _c_ptr]),
    "pkv_block_copy": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int,
                                _c_ptr, _c_ptr]),
    "paged_attention_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "paged_attention_decode": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int,
                                        _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                        _c_float, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr,
                                        _c_ptr]),
    "paged_attention_decode_ex": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int,
                                           _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                           _c_float, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr,
                                           _c_ptr, _c_ptr]),
    "paged_attention_decode_write": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int,
                                              _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                              _c_float, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr, _c_ptr, _c_ptr]),
    "pkv_decode_items": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr,
                                  _c_int, ctypes.POINTER(_c_int)]),
    "paged_attention_decode_items": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int,
                                              _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                              _c_float, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr,
                                              _c_ptr, _c_ptr, _c_int]),
    "paged_attention_prefill_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "paged_attention_prefill_ex": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int,
                                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                            _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr, _c_ptr]),
    "paged_attention_mixed": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                       _c_ptr, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr, _c_ptr]),
    "pkv_prefill_items": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int,
                                   ctypes.POINTER(_c_int)]),
    "paged_attention_decode_static_scratch": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int,
                                                       _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                       _c_int, _c_float, _c_int, _c_ptr, _c_ptr, _c_ptr]),
    "paged_attention_prefill": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_ptr, _c_ptr,
                                         _c_ptr]),
    "pkv_swap_out": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int,
                              _c_ptr, _c_ptr]),
    "pkv_swap_in": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int,
                             _c_ptr, _c_ptr]),
    "pkv_seq_append_batch": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_int, _c_ptr]),
    "pkv_seq_append_tokens": (_c_int, [_c_ptr, ctypes.c_int64, _c_ptr, _c_int, _c_ptr, ctypes.POINTER(_c_int)]),
    "pkv_prefix_cache_stats": (_c_int, [_c_ptr, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "pkv_seq_swap_out": (_c_int, [_c_ptr, ctypes.c_int64, _c_ptr, _c_int, ctypes.POINTER(_c_int)]),
    "pkv_seq_swap_in": (_c_int, [_c_ptr, ctypes.c_int64, _c_ptr, _c_int, ctypes.POINTER(_c_int)]),
    "pkv_alloc_create": (_c_int, [_c_int, _c_int, ctypes.POINTER(_c_ptr)]),
    "pkv_alloc_destroy": (None, [_c_ptr]),
    "pkv_seq_add": (_c_int, [_c_ptr, _c_i64]),
    "pkv_seq_append": (_c_int, [_c_ptr, _c_i64, _c_int, _c_ptr]),
    "pkv_seq_fork": (_c_int, [_c_ptr, _c_i64, _c_i64]),
    "pkv_seq_cow": (_c_int, [_c_ptr, _c_i64, _c_int, _c_ptr, ctypes.POINTER(_c_int)]),
    "pkv_seq_free": (_c_int, [_c_ptr, _c_i64]),
    "pkv_seq_len": (_c_i64, [_c_ptr, _c_i64]),
    "pkv_block_table": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_ptr, _c_int, _c_ptr]),
    "pkv_num_free": (_c_int, [_c_ptr]),
    "pkv_refcount": (_c_int, [_c_ptr, _c_int]),
}

_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = f"{what} failed: {error_string(code)} ({code})"
        if code == PKV_ERR_CUDA:
            msg += f": {lib().pkv_last_cuda_error().decode()}"
        super().__init__(msg)


def lib():
    """The loaded library; raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_276_gb300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def error_string(code: int) -> str:
    return lib().pkv_error_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != PKV_OK:
        raise PkvError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    """A torch.cuda.Stream, a raw cudaStream_t handle (int), or None for the current stream."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


# --------------------------------------------------------------- kernels
def pkv_write(k, v, slot_mapping, k_cache, v_cache, d_status=None, stream=None):
    """k, v: [T, Hkv, d] bf16; slot_mapping: [T] int64; caches [NB, Hkv, bs, d] bf16 (device)."""
    dev = k_cache.device
    for t, n, dt in ((k, "k", torch.bfloat16), (v, "v", torch.bfloat16), (slot_mapping, "slot_mapping", torch.int64),
                     (k_cache, "k_cache", torch.bfloat16), (v_cache, "v_cache", torch.bfloat16)):
        _need(t, dt, n, dev)
    NB, Hkv, bs, d = k_cache.shape
    T = slot_mapping.shape[0]
    if k.shape != (T, Hkv, d) or v.shape != (T, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between k/v and the caches")
    _check(lib().pkv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, d,
                           _ptr(d_status), _stream(stream, dev)), "pkv_write")


def pkv_block_copy(k_cache, v_cache, src_dst_pairs, d_status=None, stream=None):
    """src_dst_pairs: [n, 2] int32 device tensor of (src, dst) block ids."""
    dev = k_cache.device
    _need(k_cache, torch.bfloat16, "k_cache", dev)
    _need(v_cache, torch.bfloat16, "v_cache", dev)
    _need(src_dst_pairs, torch.int32, "src_dst_pairs", dev)
    NB, Hkv, bs, d = k_cache.shape
    n = src_dst_pairs.numel() // 2
    _check(lib().pkv_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs), n, NB, bs, Hkv, d,
                                _ptr(d_status), _stream(stream, dev)), "pkv_block_copy")


def paged_attention_workspace_size(num_seqs, q_len, num_q_heads, head_dim, max_seq_len, partition_size=0):
    return int(lib().paged_attention_workspace_size(num_seqs, q_len, num_q_heads, head_dim, max_seq_len,
                                                    partition_size))


def paged_attention_decode(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale, out,
                           workspace=None, partition_size=0, d_status=None, stream=None, main_done_event=None):
    """q, out: [B, q_len, Hq, d] bf16; caches [NB, Hkv, bs, d]; tables [B, max_blocks] int32; lens [B] int32.

    main_done_event (a torch.cuda.Event or None): recorded right after the main
    kernel, before the cross-partition merge (paged_attention_decode_ex)."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (out, "out", torch.bfloat16)):
        _need(t, dt, n, dev)
    B, q_len, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or seq_lens.shape != (B,):
        raise ValueError("shape mismatch")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
            int(max_seq_len), q_len, Hq, Hkv, d, bs, NB, float(scale), int(partition_size), _ptr(out),
            _ptr(workspace), ws_bytes, _ptr(d_status), _stream(stream, dev))
    if main_done_event is None:
        _check(lib().paged_attention_decode(*args), "paged_attention_decode")
    else:
        handle = main_done_event.cuda_event
        if not handle:
            raise ValueError("main_done_event: record the torch.cuda.Event once before passing it")
        _check(lib().paged_attention_decode_ex(*args, ctypes.c_void_p(handle)), "paged_attention_decode_ex")


def paged_attention_decode_write(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, seq_lens,
                                 max_seq_len, scale, out, workspace=None, partition_size=0, d_status=None,
                                 stream=None, main_done_event=None):
    """pkv_write of each sequence's newest token + single-token decode, one call.

    q, out: [B, 1, Hq, d] bf16; k_new, v_new: [B, Hkv, d] bf16; slot_mapping: [B] int64 (the newest
    token's slot, or negative); caches [NB, Hkv, bs, d]; tables [B, max_blocks] int32; lens [B] int32."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_new, "k_new", torch.bfloat16), (v_new, "v_new", torch.bfloat16),
                     (slot_mapping, "slot_mapping", torch.int64), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (out, "out", torch.bfloat16)):
        _need(t, dt, n, dev)
    B, q_len, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if q_len != 1 or d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape \
            or k_new.shape != (B, Hkv, d) or v_new.shape != (B, Hkv, d) or slot_mapping.shape != (B,) \
            or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("shape mismatch")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ev = None
    if main_done_event is not None:
        ev = main_done_event.cuda_event
        if not ev:
            raise ValueError("main_done_event: record the torch.cuda.Event once before passing it")
    _check(lib().paged_attention_decode_write(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), B, int(max_seq_len), Hq, Hkv, d, bs, NB, float(scale),
        int(partition_size), _ptr(out), _ptr(workspace), ws_bytes, _ptr(d_status), _stream(stream, dev),
        None if ev is None else ctypes.c_void_p(ev)), "paged_attention_decode_write")


def pkv_decode_items(seq_lens, block_tables, num_kv_heads, block_size, partition_size=0, head_dim=128, out=None):
    """Host work list of a single-token decode batch (numpy int32 lengths [B] and
    tables [B, max_blocks], or None): returns int32 [1 + count, 4], row 0 =
    {count, partition size used, 0, 0}.  partition_size 0: the library picks it.
    ``out`` (int32 [1 + n, 4], C-contiguous) is filled in place when it has room."""
    import numpy as np
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    tbl = None if block_tables is None else np.ascontiguousarray(block_tables, dtype=np.int32)
    B = lens.shape[0]
    if tbl is None:
        maxb = int(-(-int(lens.max(initial=0)) // block_size))
    elif tbl.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    else:
        maxb = tbl.shape[1]
    n = ctypes.c_int(0)
    buf = out if out is not None else np.empty((1, 4), dtype=np.int32)
    for _ in range(2):
        rc = lib().pkv_decode_items(lens.ctypes.data, None if tbl is None else tbl.ctypes.data, maxb, B,
                                    int(num_kv_heads), int(head_dim), int(block_size), int(partition_size),
                                    buf.ctypes.data, buf.shape[0] - 1, ctypes.byref(n))
        if rc == PKV_ERR_RANGE and n.value > buf.shape[0] - 1 and out is None:
            buf = np.empty((1 + n.value, 4), dtype=np.int32)
            continue
        _check(rc, "pkv_decode_items")
        return buf[:1 + n.value]
    raise PkvError(PKV_ERR_RANGE, "pkv_decode_items")


def paged_attention_decode_items(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, seq_lens,
                                 max_seq_len, scale, out, items, grid_items=None, workspace=None, partition_size=0,
                                 d_status=None, stream=None, main_done_event=None, overlap=False):
    """Single-token decode over a work list (device int32 [1 + n, 4] from
    ``pkv_decode_items``); k_new / v_new / slot_mapping all None: no store.
    overlap: PKV_DECODE_OVERLAP (nothing this call reads or stores into is
    touched by the work queued before it, as for the layers of one step)."""
    dev = k_cache.device
    store = k_new is not None or v_new is not None or slot_mapping is not None
    checks = [(q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16), (v_cache, "v_cache", torch.bfloat16),
              (block_tables, "block_tables", torch.int32), (seq_lens, "seq_lens", torch.int32),
              (out, "out", torch.bfloat16), (items, "items", torch.int32)]
    if store:
        checks += [(k_new, "k_new", torch.bfloat16), (v_new, "v_new", torch.bfloat16),
                   (slot_mapping, "slot_mapping", torch.int64)]
    for t, n, dt in checks:
        _need(t, dt, n, dev)
    B, q_len, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if q_len != 1 or d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape \
            or block_tables.shape[0] != B or seq_lens.shape != (B,) or items.dim() != 2 or items.shape[1] != 4:
        raise ValueError("shape mismatch")
    if store and (k_new.shape != (B, Hkv, d) or v_new.shape != (B, Hkv, d) or slot_mapping.shape != (B,)):
        raise ValueError("shape mismatch")
    grid = items.shape[0] - 1 if grid_items is None else int(grid_items)
    if grid > items.shape[0] - 1:
        raise ValueError("grid_items exceeds the rows of items")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ev = None
    if main_done_event is not None:
        ev = main_done_event.cuda_event
        if not ev:
            raise ValueError("main_done_event: record the torch.cuda.Event once before passing it")
    _check(lib().paged_attention_decode_items(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), B, int(max_seq_len), Hq, Hkv, d, bs, NB, float(scale),
        int(partition_size), _ptr(items), grid, _ptr(out), _ptr(workspace), ws_bytes, _ptr(d_status),
        _stream(stream, dev), None if ev is None else ctypes.c_void_p(ev), PKV_DECODE_OVERLAP if overlap else 0),
        "paged_attention_decode_items")


def paged_attention_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_start, scale, out, d_status=None,
                            stream=None):
    """Chunked prefill: q, out [total_q, Hq, 128] bf16; q_start [B + 1] int32 (rows of sequence i are
    q_start[i] .. q_start[i+1]-1, its newest tokens); caches [NB, Hkv, bs, 128]; tables [B, max_blocks]
    int32; lens [B] int32."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (q_start, "q_start", torch.int32),
                     (out, "out", torch.bfloat16)):
        _need(t, dt, n, dev)
    total_q, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    B = seq_lens.shape[0]
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or seq_lens.shape != (B,) or q_start.shape != (B + 1,):
        raise ValueError("shape mismatch")
    _check(lib().paged_attention_prefill(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        _ptr(q_start), B, total_q, Hq, Hkv, d, bs, NB, float(scale), _ptr(out), _ptr(d_status),
        _stream(stream, dev)), "paged_attention_prefill")


def paged_attention_prefill_workspace_size(total_q, num_q_heads, head_dim, max_seq_len, partition_size):
    return int(lib().paged_attention_prefill_workspace_size(int(total_q), int(num_q_heads), int(head_dim),
                                                            int(max_seq_len), int(partition_size)))


def paged_attention_prefill_ex(q, k_cache, v_cache, block_tables, seq_lens, q_start, scale, out, max_seq_len,
                               partition_size, workspace=None, d_status=None, stream=None):
    """paged_attention_prefill with the keys split into partitions of
    ``partition_size`` tokens (0: no split), merged through ``workspace``."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (q_start, "q_start", torch.int32),
                     (out, "out", torch.bfloat16)):
        _need(t, dt, n, dev)
    total_q, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    B = seq_lens.shape[0]
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or seq_lens.shape != (B,) or q_start.shape != (B + 1,):
        raise ValueError("shape mismatch")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().paged_attention_prefill_ex(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        _ptr(q_start), B, total_q, Hq, Hkv, d, bs, NB, float(scale), int(max_seq_len), int(partition_size),
        _ptr(out), _ptr(workspace), ws_bytes, _ptr(d_status), _stream(stream, dev)), "paged_attention_prefill_ex")


def pkv_prefill_items(seq_lens, q_start, total_q, num_q_heads, num_kv_heads, grid):
    """Host work list of a prefill launch of ``grid`` CTAs (numpy int32 lengths
    [B] and q_start [B + 1]): int32 [3 + grid + n] = grid, n, each CTA's range
    offsets [grid + 1], the item indices."""
    import numpy as np
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    B = lens.shape[0]
    if qs.shape != (B + 1,):
        raise ValueError("q_start must be [num_seqs + 1]")
    n = ctypes.c_int(0)
    buf = np.empty(3 + int(grid), dtype=np.int32)
    for _ in range(2):
        rc = lib().pkv_prefill_items(lens.ctypes.data, qs.ctypes.data, B, int(total_q), int(num_q_heads),
                                     int(num_kv_heads), int(grid), buf.ctypes.data, buf.shape[0], ctypes.byref(n))
        if rc == PKV_ERR_RANGE and n.value > buf.shape[0]:
            buf = np.empty(n.value, dtype=np.int32)
            continue
        _check(rc, "pkv_prefill_items")
        return buf[:n.value]
    raise PkvError(PKV_ERR_RANGE, "pkv_prefill_items")


def paged_attention_mixed(q, k_cache, v_cache, block_tables, seq_lens, q_start, scale, out, num_decodes,
                          decode_items, max_decode_len, decode_partition_size=0, workspace=None, prefill_ctas=0,
                          decode_grid=None, d_status=None, stream=None, prefill_items=None):
    """One step of decodes (the first ``num_decodes`` sequences, query rows
    0..num_decodes-1) and prompt chunks (the rest), as paged_attention_prefill
    over the whole batch; ``decode_items`` (device) from pkv_decode_items over the
    decodes' lengths and tables; ``prefill_items`` (device int32, or None) from
    pkv_prefill_items over the chunks with grid ``prefill_ctas``."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (q_start, "q_start", torch.int32),
                     (out, "out", torch.bfloat16), (decode_items, "decode_items", torch.int32)):
        _need(t, dt, n, dev)
    if prefill_items is not None:
        _need(prefill_items, torch.int32, "prefill_items", dev)
    total_q, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    B = seq_lens.shape[0]
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or block_tables.shape[0] != B \
            or seq_lens.shape != (B,) or q_start.shape != (B + 1,) or decode_items.dim() != 2 \
            or decode_items.shape[1] != 4:
        raise ValueError("shape mismatch")
    grid = decode_items.shape[0] - 1 if decode_grid is None else int(decode_grid)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().paged_attention_mixed(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        _ptr(q_start), B, total_q, int(num_decodes), Hq, Hkv, d, bs, NB, float(scale), int(max_decode_len),
        int(decode_partition_size), _ptr(decode_items), grid, int(prefill_ctas), _ptr(prefill_items), _ptr(out),
        _ptr(workspace),
        ws_bytes, _ptr(d_status), _stream(stream, dev)), "paged_attention_mixed")


def _swap_check(k_cache, v_cache, block_ids, host_k, host_v):
    dev = k_cache.device
    for t, n, dt in ((k_cache, "k_cache", torch.bfloat16), (v_cache, "v_cache", torch.bfloat16),
                     (block_ids, "block_ids", torch.int32)):
        _need(t, dt, n, dev)
    for t, n in ((host_k, "host_k"), (host_v, "host_v")):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device.type != "cpu" or not t.is_pinned():
            raise ValueError(f"{n}: contiguous pinned host bf16 tensor expected")
    NB, Hkv, bs, d = k_cache.shape
    n = block_ids.numel()
    if v_cache.shape != k_cache.shape or host_k.shape != (n, Hkv, bs, d) or host_v.shape != host_k.shape:
        raise ValueError("shape mismatch")
    return NB, Hkv, bs, d, n, dev


def pkv_swap_out(k_cache, v_cache, block_ids, host_k, host_v, d_status=None, stream=None):
    """host_k/v[i] = cache[block_ids[i]]; host buffers pinned [n, Hkv, bs, d] bf16."""
    NB, Hkv, bs, d, n, dev = _swap_check(k_cache, v_cache, block_ids, host_k, host_v)
    _check(lib().pkv_swap_out(_ptr(k_cache), _ptr(v_cache), _ptr(block_ids), n, _ptr(host_k), _ptr(host_v), NB, bs,
                              Hkv, d, _ptr(d_status), _stream(stream, dev)), "pkv_swap_out")


def pkv_swap_in(host_k, host_v, block_ids, k_cache, v_cache, d_status=None, stream=None):
    """cache[block_ids[i]] = host_k/v[i]."""
    NB, Hkv, bs, d, n, dev = _swap_check(k_cache, v_cache, block_ids, host_k, host_v)
    _check(lib().pkv_swap_in(_ptr(host_k), _ptr(host_v), _ptr(block_ids), n, _ptr(k_cache), _ptr(v_cache), NB, bs,
                             Hkv, d, _ptr(d_status), _stream(stream, dev)), "pkv_swap_in")


STATIC_SCRATCH_BYTES = 8 << 20  # PKV_STATIC_SCRATCH_BYTES


def paged_attention_decode_static_scratch(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale, out,
                                          partition_size=0, d_status=None, stream=None):
    """paged_attention_decode for callers that cannot allocate: the split-K
    scratch is the library's fixed array (see include/pkv.h)."""
    dev = k_cache.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (seq_lens, "seq_lens", torch.int32), (out, "out", torch.bfloat16)):
        _need(t, dt, n, dev)
    B, q_len, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    _check(lib().paged_attention_decode_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
        int(max_seq_len), q_len, Hq, Hkv, d, bs, NB, float(scale), int(partition_size), _ptr(out),
        _ptr(d_status), _stream(stream, dev)), "paged_attention_decode_static_scratch")


# ------------------------------------------------------------- allocator
class BlockAllocator:
    """Host block manager (pkv_alloc_* / pkv_seq_* in the C ABI)."""

    def __init__(self, num_blocks: int, block_size: int):
        h = ctypes.c_void_p()
        _check(lib().pkv_alloc_create(num_blocks, block_size, ctypes.byref(h)), "pkv_alloc_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            lib().pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def seq_add(self, seq_id: int):
        _check(lib().pkv_seq_add(self._h, seq_id), "pkv_seq_add")

    def seq_append(self, seq_id: int, n_tokens: int, out=None):
        """Returns the n slots (int64 numpy array, or written into ``out``)."""
        import numpy as np
        slots = np.empty(n_tokens, dtype=np.int64) if out is None else out
        _check(lib().pkv_seq_append(self._h, seq_id, n_tokens, slots.ctypes.data if n_tokens else None),
               "pkv_seq_append")
        return slots

    def seq_append_batch(self, seq_ids, n_tokens: int, out=None):
        """Append n_tokens to each listed sequence; returns (or fills ``out`` with)
        the int64 slots, sequence by sequence.  ``seq_ids`` and ``out`` may be
        numpy arrays (``out`` for instance a view of pinned memory)."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        slots = np.empty(len(ids) * n_tokens, dtype=np.int64) if out is None else out
        if slots.dtype != np.int64 or not slots.flags.c_contiguous or slots.size < len(ids) * n_tokens:
            raise ValueError("out: contiguous int64 array of len(seq_ids) * n_tokens expected")
        _check(lib().pkv_seq_append_batch(self._h, ids.ctypes.data, len(ids), n_tokens, slots.ctypes.data),
               "pkv_seq_append_batch")
        return slots

    def seq_append_tokens(self, seq_id: int, token_ids):
        """Append tokens with their ids; returns (slots int64, cached token count).
        Slots of tokens found in the prefix cache are -1."""
        import numpy as np
        toks = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        slots = np.empty(len(toks), dtype=np.int64)
        cached = ctypes.c_int()
        _check(lib().pkv_seq_append_tokens(self._h, seq_id, toks.ctypes.data if len(toks) else None, len(toks),
                                           slots.ctypes.data if len(toks) else None, ctypes.byref(cached)),
               "pkv_seq_append_tokens")
        return slots, cached.value

    def prefix_cache_stats(self):
        """(registered blocks, of which nobody holds)."""
        r, e = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_prefix_cache_stats(self._h, ctypes.byref(r), ctypes.byref(e)), "pkv_prefix_cache_stats")
        return r.value, e.value

    def seq_fork(self, parent: int, child: int):
        _check(lib().pkv_seq_fork(self._h, parent, child), "pkv_seq_fork")

    def seq_cow(self, seq_id: int, logical_block: int = -1):
        pair = (ctypes.c_int32 * 2)()
        copied = ctypes.c_int()
        _check(lib().pkv_seq_cow(self._h, seq_id, logical_block, pair, ctypes.byref(copied)), "pkv_seq_cow")
        return (pair[0], pair[1]) if copied.value else None

    def seq_free(self, seq_id: int):
        _check(lib().pkv_seq_free(self._h, seq_id), "pkv_seq_free")

    def _swap(self, fn, name, seq_id: int, max_blocks: int):
        import numpy as np
        out = np.empty(max(1, max_blocks), dtype=np.int32)
        n = ctypes.c_int()
        _check(fn(self._h, seq_id, out.ctypes.data, max_blocks, ctypes.byref(n)), name)
        return out[:n.value].copy()

    def seq_swap_out(self, seq_id: int, max_blocks: int = 1 << 16):
        """Release the sequence's blocks; returns their ids in logical order (int32)."""
        return self._swap(lib().pkv_seq_swap_out, "pkv_seq_swap_out", seq_id, max_blocks)

    def seq_swap_in(self, seq_id: int, max_blocks: int = 1 << 16):
        """New blocks for a swapped-out sequence, in logical order (int32)."""
        return self._swap(lib().pkv_seq_swap_in, "pkv_seq_swap_in", seq_id, max_blocks)

    def seq_len(self, seq_id: int) -> int:
        n = lib().pkv_seq_len(self._h, seq_id)
        if n < 0:
            raise PkvError(int(n), "pkv_seq_len")
        return int(n)

    def block_table(self, seq_ids, max_blocks: int, table_out=None, lens_out=None):
        """[n, max_blocks] int32 table rows and [n] int32 lengths (or written into
        ``table_out`` / ``lens_out``, e.g. views of pinned memory)."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(list(seq_ids) if not isinstance(seq_ids, np.ndarray) else seq_ids,
                                              dtype=np.int64))
        table = np.empty((len(ids), max_blocks), dtype=np.int32) if table_out is None else table_out
        lens = np.empty(len(ids), dtype=np.int32) if lens_out is None else lens_out
        if (table.dtype != np.int32 or lens.dtype != np.int32 or not table.flags.c_contiguous
                or table.shape != (len(ids), max_blocks) or lens.shape != (len(ids),)):
            raise ValueError("table_out / lens_out: contiguous int32 [n, max_blocks] / [n] expected")
        _check(lib().pkv_block_table(self._h, ids.ctypes.data, len(ids), table.ctypes.data, max_blocks,
                                     lens.ctypes.data), "pkv_block_table")
        return table, lens

    def num_free(self) -> int:
        return int(lib().pkv_num_free(self._h))

    def refcount(self, block: int) -> int:
        rc = lib().pkv_refcount(self._h, block)
        if rc < 0:
            raise PkvError(rc, "pkv_refcount")
        return int(rc)


# --------------------------------------------------------------- step runner
class DecodeStep:
    """pkv_step_*: one decode step of a batch through every layer, one C call.

    Owns the runner's buffers (page-locked staging and output buffers, their
    device twins, the split-K workspace), laid out by ``pkv_step_layout_of``.
    Per step: write the step's queries and new keys / values of rows
    0..n-1 into ``q(l)``, ``k(l)``, ``v(l)`` (host views), call ``run(seq_ids)``,
    then ``wait()``; the outputs are in ``out(l)`` (host views).  The runner
    appends the tokens to the allocator and fills the slots, tables and lengths
    itself; ``slots``, ``tables`` and ``lens`` show them.
    """

    def __init__(self, alloc, k_caches, v_caches, max_seqs, q_len, num_q_heads, max_blocks_per_seq, scale,
                 partition_size=0, use_graph=False, d_status=None):
        k_caches, v_caches = list(k_caches), list(v_caches)
        if not k_caches or len(k_caches) != len(v_caches):
            raise ValueError("one key and one value cache per layer expected")
        dev = k_caches[0].device
        for i, (kc, vc) in enumerate(zip(k_caches, v_caches)):
            _need(kc, torch.bfloat16, f"k_caches[{i}]", dev)
            _need(vc, torch.bfloat16, f"v_caches[{i}]", dev)
            if kc.shape != k_caches[0].shape or vc.shape != kc.shape:
                raise ValueError("every layer's caches must have the same shape")
        NB, Hkv, bs, d = k_caches[0].shape
        self.cfg = StepConfig(len(k_caches), int(max_seqs), int(q_len), int(num_q_heads), Hkv, d, bs, NB,
                              int(max_blocks_per_seq), int(partition_size), float(scale), 1 if use_graph else 0)
        lay = StepLayout()
        _check(lib().pkv_step_layout_of(ctypes.byref(self.cfg), ctypes.byref(lay)), "pkv_step_layout_of")
        self.layout = lay
        self.device = dev
        u8 = torch.uint8
        self.host_stage = torch.empty(lay.stage_bytes, dtype=u8).pin_memory()
        self.dev_stage = torch.empty(lay.stage_bytes, dtype=u8, device=dev)
        self.host_out = torch.empty(lay.out_bytes, dtype=u8).pin_memory()
        self.dev_out = torch.empty(lay.out_bytes, dtype=u8, device=dev)
        self.workspace = torch.empty(max(lay.workspace_bytes, 16), dtype=u8, device=dev)
        self._caches = (k_caches, v_caches)  # kept alive with the runner
        kp = (_c_ptr * len(k_caches))(*[t.data_ptr() for t in k_caches])
        vp = (_c_ptr * len(v_caches))(*[t.data_ptr() for t in v_caches])
        self._alloc = alloc
        h = _c_ptr()
        _check(lib().pkv_step_create(ctypes.byref(self.cfg), alloc._h, kp, vp, _ptr(self.host_stage),
                                     _ptr(self.dev_stage), _ptr(self.dev_out), _ptr(self.host_out),
                                     _ptr(self.workspace), lay.workspace_bytes, _ptr(d_status), ctypes.byref(h)),
               "pkv_step_create")
        self._h = h
        self._run = lib().pkv_step_run
        B, H, ql = int(max_seqs), int(num_q_heads), int(q_len)
        self._q_shape, self._kv_shape = (B, ql, H, d), (B * ql, Hkv, d)
        self.slots = self._view(self.host_stage, lay.slots_offset, torch.int64, (B * ql,))
        self.tables = self._view(self.host_stage, lay.tables_offset, torch.int32, (B, int(max_blocks_per_seq)))
        self.lens = self._view(self.host_stage, lay.lens_offset, torch.int32, (B,))

    @staticmethod
    def _view(buf, off, dtype, shape):
        n = 1
        for x in shape:
            n *= x
        return buf[off:off + n * torch.empty((), dtype=dtype).element_size()].view(dtype).view(shape)

    def q(self, layer):
        return self._view(self.host_stage, self.layout.q_offset + layer * self.layout.layer_stride,
                          torch.bfloat16, self._q_shape)

    def k(self, layer):
        return self._view(self.host_stage, self.layout.k_offset + layer * self.layout.layer_stride,
                          torch.bfloat16, self._kv_shape)

    def v(self, layer):
        return self._view(self.host_stage, self.layout.v_offset + layer * self.layout.layer_stride,
                          torch.bfloat16, self._kv_shape)

    def out(self, layer):
        return self._view(self.host_out, layer * self.layout.out_layer_bytes, torch.bfloat16, self._q_shape)

    def run(self, seq_ids, stream=None):
        """Enqueue one step for ``seq_ids`` (int64 numpy array or sequence); returns at once."""
        import numpy as np
        ids = seq_ids if (isinstance(seq_ids, np.ndarray) and seq_ids.dtype == np.int64
                          and seq_ids.flags.c_contiguous) else np.ascontiguousarray(seq_ids, dtype=np.int64)
        rc = self._run(self._h, ids.ctypes.data, len(ids), _stream(stream, self.device))
        if rc != PKV_OK:
            raise PkvError(rc, "pkv_step_run")

    def wait(self):
        _check(lib().pkv_step_wait(self._h), "pkv_step_wait")

    def close(self):
        if getattr(self, "_h", None):
            lib().pkv_step_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
