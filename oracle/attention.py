"""fp64 CPU oracle for paged attention (ctypes wrapper around pkv_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this module.  It shares no
code with the CUDA path and never imports the product package.

The computation is the plain definition of attention over a block-paged cache:
gather each sequence's blocks in block-table order into contiguous K/V, then
softmax(q K^T * scale) V in fp64 (x321.org "The serving bottleneck is not just
FLOPs", sections "First understand what the KV cache is storing" and
"PagedAttention borrows an operating-system trick").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_paged_attention.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p]
            lib.oracle_set_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Set the OpenMP thread count (n <= 0 keeps it); returns the count in use."""
    return int(_load().oracle_set_threads(int(n)))


def as_bf16_bits(x) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of a torch bf16 tensor or a uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must already hold bf16 bits as uint16")
        return np.ascontiguousarray(x)
    import torch  # local: only for tensors handed in by tests
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, *, num_q_heads,
                    num_kv_heads, head_dim, block_size, scale, q_len=1):
    """fp64 paged attention.

    q: bf16 [B, q_len, Hq, d] (bits or tensor); caches: bf16 [NB, Hkv, bs, d];
    block_tables: int32 [B, max_blocks]; seq_lens: int32 [B].  ``scale`` is the
    fp32 value the kernel receives, widened to fp64.  Returns float64
    [B, q_len, Hq, d].
    """
    qb = as_bf16_bits(q)
    kb = as_bf16_bits(k_cache)
    vb = as_bf16_bits(v_cache)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B = int(sl.shape[0])
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    NB = int(kb.shape[0]) if kb.ndim == 4 else int(kb.size // (num_kv_heads * block_size * head_dim))
    if qb.size != B * q_len * num_q_heads * head_dim:
        raise ValueError("q has the wrong number of elements")
    out = np.zeros((B, q_len, num_q_heads, head_dim), dtype=np.float64)
    rc = _load().oracle_paged_attention(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, bt.ctypes.data,
        int(bt.shape[1]), sl.ctypes.data, B, int(q_len), int(num_q_heads),
        int(num_kv_heads), int(head_dim), int(block_size), NB,
        float(np.float32(scale)), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_paged_attention failed with code {rc}")
    return out


def paged_attention_varlen(q, k_cache, v_cache, block_tables, seq_lens, q_start, *, num_q_heads,
                           num_kv_heads, head_dim, block_size, scale):
    """fp64 paged attention of a chunk of new tokens per sequence (chunked prefill).

    The pages' scheduler splits a long prompt into chunks and runs them in the
    same step as single-token decodes (x321.org "The serving bottleneck is not
    just FLOPs", section "Continuous batching is the other half of the story").
    Sequence i owns query rows q_start[i] .. q_start[i+1]-1 of q (bf16
    [total_q, Hq, d]); they are its newest c_i = q_start[i+1] - q_start[i]
    tokens, so row r < c_i sees keys t < seq_lens[i] - c_i + 1 + r, the causal
    rule of ``paged_attention`` with q_len = c_i.  Each sequence is one call of
    that function on its own rows; rows with no visible key are zero.
    Returns float64 [total_q, Hq, d].
    """
    qb = as_bf16_bits(q)
    qs = np.asarray(q_start, dtype=np.int64).reshape(-1)
    sl = np.asarray(seq_lens, dtype=np.int32).reshape(-1)
    bt = np.asarray(block_tables, dtype=np.int32)
    B = int(sl.shape[0])
    if qs.shape[0] != B + 1 or qs[0] != 0 or np.any(np.diff(qs) < 0):
        raise ValueError("q_start must be [num_seqs + 1], start at 0 and never decrease")
    total = int(qs[-1])
    qb = qb.reshape(-1, num_q_heads, head_dim)
    if qb.shape[0] != total:
        raise ValueError("q must hold q_start[-1] rows")
    out = np.zeros((total, num_q_heads, head_dim), dtype=np.float64)
    for i in range(B):
        lo, hi = int(qs[i]), int(qs[i + 1])
        if hi == lo:
            continue
        out[lo:hi] = paged_attention(qb[lo:hi][None], k_cache, v_cache, bt[i:i + 1], sl[i:i + 1],
                                     num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                                     head_dim=head_dim, block_size=block_size, scale=scale,
                                     q_len=hi - lo)[0]
    return out
