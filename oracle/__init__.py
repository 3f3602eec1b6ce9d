"""Float64 CPU oracle for the attention path -- TEST INFRASTRUCTURE ONLY.

This package is the independent yardstick for the CUDA kernels.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the product package and imports nothing
from it; the product never imports this package.

The arithmetic lives in ``attn_oracle.c`` (plain C, float64, OpenMP over
rows).  This module compiles it with gcc on first use (or via :func:`build`)
and marshals numpy / torch arguments through ctypes.  Every function follows
the article "从零实现 vLLM (1.3)：如何加速 Attention 计算"; the C file cites
the section behind each one.

Inputs that are bf16 on the GPU are passed as their 16-bit patterns (numpy
uint16, or a torch bfloat16 tensor which is reinterpreted), so the oracle sees
exactly the values the kernels see.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()

_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_softmax_naive_f32.argtypes = [_f32p, ctypes.c_int, _f32p]
        lib.oracle_softmax_naive_f64.argtypes = [_f64p, ctypes.c_int, _f64p]
        lib.oracle_softmax_safe.argtypes = [_f64p, ctypes.c_int, _f64p]
        lib.oracle_softmax_online.argtypes = [_f64p, ctypes.c_int, _f64p, _f64p, _f64p]
        lib.oracle_softmax_rows.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int, _f64p, ctypes.c_int]
        lib.oracle_attn_tiled_row.argtypes = [_f64p, _f64p, _f64p, _u8p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_int, _f64p, _f64p, _f64p]
        lib.oracle_attn_varlen.argtypes = [
            _u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _i64p, ctypes.c_int64,
            _f64p, _f64p, ctypes.c_int]
        lib.oracle_attn_varlen.restype = ctypes.c_int
        lib.oracle_decode_paged.argtypes = [
            _u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
            ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
        lib.oracle_decode_paged.restype = ctypes.c_int
        lib.oracle_store_kvcache.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _i64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_store_kvcache.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def as_bits(x) -> np.ndarray:
    """bf16 values as a C-contiguous uint16 array of their bit patterns.

    Accepts a torch bfloat16 tensor (reinterpreted, not converted) or a numpy
    uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must already be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch  # plain CPU use only
    if x.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


# --------------------------------------------------------------------------
# softmax variants
# --------------------------------------------------------------------------

def softmax_naive(x, dtype: str = "f64") -> np.ndarray:
    """e^x / sum e^x with no max shift, in float32 ("f32") or float64 ("f64")."""
    lib = _load()
    if dtype == "f32":
        xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        y = np.empty_like(xa)
        lib.oracle_softmax_naive_f32(_ptr(xa, _f32p), xa.size, _ptr(y, _f32p))
        return y
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty_like(xa)
    lib.oracle_softmax_naive_f64(_ptr(xa, _f64p), xa.size, _ptr(y, _f64p))
    return y


def softmax_safe(x) -> np.ndarray:
    """Three-pass safe softmax (max, shifted sum, normalise)."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty_like(xa)
    lib.oracle_softmax_safe(_ptr(xa, _f64p), xa.size, _ptr(y, _f64p))
    return y


def softmax_online(x):
    """Two-pass online softmax.  Returns (y, m_trace, d_trace)."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.empty_like(xa)
    mt = np.empty_like(xa)
    dt = np.empty_like(xa)
    lib.oracle_softmax_online(_ptr(xa, _f64p), xa.size, _ptr(y, _f64p), _ptr(mt, _f64p), _ptr(dt, _f64p))
    return y, mt, dt


def softmax_rows(x, nthreads: int = 0) -> np.ndarray:
    """Safe softmax of every row of a 2-D array (float64 result).  Accepts
    float32 / float64 arrays and torch tensors (bf16 included, upcast exactly)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if xa.ndim != 2:
        raise ValueError("softmax_rows takes a 2-D array")
    y = np.empty_like(xa)
    _load().oracle_softmax_rows(_ptr(xa, _f64p), xa.shape[0], xa.shape[1], _ptr(y, _f64p), int(nthreads))
    return y


def attn_tiled_row(q, K, V, scale: float, block: int, visible=None):
    """1-pass (m, d', o') recurrence for one query row over key blocks.

    Returns (o [D], m, d')."""
    lib = _load()
    qa = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    Ka = np.ascontiguousarray(np.asarray(K, dtype=np.float64))
    Va = np.ascontiguousarray(np.asarray(V, dtype=np.float64))
    Lk, D = Ka.shape
    o = np.empty(D, dtype=np.float64)
    m = ctypes.c_double()
    d = ctypes.c_double()
    vis = None
    if visible is not None:
        vis = np.ascontiguousarray(np.asarray(visible, dtype=np.uint8))
    lib.oracle_attn_tiled_row(_ptr(qa, _f64p), _ptr(Ka, _f64p), _ptr(Va, _f64p),
                              _ptr(vis, _u8p) if vis is not None else None, Lk, D,
                              float(scale), int(block), _ptr(o, _f64p), ctypes.byref(m), ctypes.byref(d))
    return o, m.value, d.value


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, num_heads_q: int, num_heads_kv: int,
                head_dim: int, softmax_scale: float, causal: bool = True, block_table=None,
                block_size: int = 0, num_blocks: int = 0, rows=None, nthreads: int = 0):
    """Three-step attention over varlen-packed q and contiguous or paged k/v.

    q: [total_q, Hq, D] bf16 bits (any array whose last two dims are Hq, D and
    whose rows are tokens).  k, v: [total_k, Hkv, D] (contiguous) or
    [num_blocks, block_size, Hkv, D] (paged, with block_table [B, max_blocks]).
    rows: optional int64 list of row ids token*Hq + head.
    Returns (out [n, D] float64, lse [n] float64)."""
    lib = _load()
    qb, kb, vb = as_bits(q), as_bits(k), as_bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    B = cq.size - 1
    D = int(head_dim)
    total_q = int(cq[-1])
    n = total_q * num_heads_q if rows is None else len(rows)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    bt = None if block_table is None else _i32(block_table)
    ra = None if rows is None else _i64(rows)
    rc = lib.oracle_attn_varlen(
        _ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p), _ptr(cq, _i32p), _ptr(ck, _i32p), B,
        num_heads_q, num_heads_kv, D, float(softmax_scale), int(bool(causal)),
        _ptr(bt, _i32p) if bt is not None else None, bt.shape[1] if bt is not None else 0,
        int(block_size), int(num_blocks), num_heads_q * D, num_heads_kv * D, num_heads_kv * D,
        _ptr(ra, _i64p) if ra is not None else None, n, _ptr(out, _f64p), _ptr(lse, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_varlen: argument or index outside its storage")
    return out, lse


def decode_paged(q, k_cache, v_cache, cache_seqlens, block_table, num_heads_q: int,
                 num_heads_kv: int, head_dim: int, block_size: int, num_blocks: int,
                 softmax_scale: float, nthreads: int = 0):
    """One query token per sequence through the paged cache.

    q: [B, Hq, D]; caches [num_blocks, block_size, Hkv, D]; returns
    (out [B, Hq, D] float64, lse [B, Hq] float64)."""
    lib = _load()
    qb, kb, vb = as_bits(q), as_bits(k_cache), as_bits(v_cache)
    cs = _i32(cache_seqlens)
    bt = _i32(block_table)
    B = cs.size
    out = np.zeros((B * num_heads_q, head_dim), dtype=np.float64)
    lse = np.zeros(B * num_heads_q, dtype=np.float64)
    rc = lib.oracle_decode_paged(
        _ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p), _ptr(cs, _i32p), _ptr(bt, _i32p),
        bt.shape[1], B, num_heads_q, num_heads_kv, head_dim, int(block_size), int(num_blocks),
        float(softmax_scale), num_heads_q * head_dim, _ptr(out, _f64p), _ptr(lse, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_paged: argument or index outside its storage")
    return out.reshape(B, num_heads_q, head_dim), lse.reshape(B, num_heads_q)


def store_kvcache(k, v, k_cache, v_cache, slot_mapping):
    """Scatter k/v rows into copies of the caches; returns (k_cache', v_cache')
    as uint16 bit arrays with the caches' shapes."""
    lib = _load()
    kb, vb = as_bits(k), as_bits(v)
    kc = as_bits(k_cache).copy()
    vc = as_bits(v_cache).copy()
    sm = _i64(slot_mapping)
    N = sm.size
    Hkv, D = kb.shape[-2], kb.shape[-1]
    num_slots = kc.size // (Hkv * D)
    rc = lib.oracle_store_kvcache(_ptr(kb, _u16p), _ptr(vb, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p),
                                  _ptr(sm, _i64p), N, Hkv, D, Hkv * D, Hkv * D, num_slots)
    if rc != 0:
        raise ValueError("oracle_store_kvcache: slot outside the cache")
    return kc, vc
