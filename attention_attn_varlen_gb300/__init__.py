"""GB300 (sm_103a) varlen / paged attention: thin Python binding of the C ABI.

Every computation runs in the CUDA kernels of ``libattn_varlen.so`` (built
in-tree from ``csrc/`` by :func:`build`).  This module only checks and
marshals arguments: it takes torch CUDA tensors (PyTorch supplies device
memory and streams) and calls the C entry points of ``include/attn_varlen.h``
with their raw pointers on the current stream.  There is no fallback: if the
library is missing or the device is not sm_103 the calls raise.

Entry points (the C ABI's names):
    attn_varlen_fwd         varlen prefill, contiguous or paged K/V (optionally the fp16 V/16 cache)
    attn_varlen_fwd_host    the same prefill for pinned host tensors (copies overlapped by the library)
    attn_decode_paged       single-token decode through the paged cache
    attn_with_kvcache       several new tokens per sequence against the paged cache (attn_kvcache_fwd)
    attn_padded_fwd         a padded [B, S, H, D] batch with per-sequence lengths
    store_kvcache           slot_mapping scatter into the caches (optionally also V/16 in fp16)
    softmax_rows            row softmax (attn_softmax_rows)
    get_last_device_error   the device error word (index, range and timeout checks)
    selftest_bounded_wait   the failure-detection self-test
and the layer-shaped dispatcher in :mod:`attention_attn_varlen_gb300.attention`.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

from ._build import LIB as _LIB_PATH
from ._build import build

__all__ = ["attn_varlen_fwd", "attn_varlen_fwd_host", "host_staging", "attn_decode_paged", "attn_with_kvcache",
           "attn_padded_fwd", "softmax_rows", "store_kvcache", "get_last_device_error", "selftest_bounded_wait",
           "lib", "build", "AttnError", "exported_symbols", "set_kernel_events", "decode_num_splits",
           "decode_workspace_size"]

ATTN_OK = 0
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small", 4: "launch failed",
           5: "device timeout", 6: "device index out of range", 7: "no device", 8: "input value out of range"}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)} (status {status})")


_lib = None
_c = ctypes
_vp, _i32, _i64, _f32, _sz = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_float, _c.c_size_t


def lib():
    """The loaded CUDA library (ctypes.CDLL); raises if it was never built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"CUDA attention library not built ({_LIB_PATH} missing); "
                           "run attention_attn_varlen_gb300.build() on a machine with nvcc")
    L = ctypes.CDLL(_LIB_PATH)
    L.attn_varlen_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32, _i32, _i32, _i32,
                                  _f32, _i32, _vp, _i32, _i32, _i64, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]
    L.attn_varlen_fwd.restype = _i32
    L.attn_varlen_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i64]
    L.attn_varlen_workspace_size.restype = _sz
    L.attn_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _i32,
                                    _f32, _i32, _i64, _i64, _vp, _sz, _vp]
    L.attn_decode_paged.restype = _i32
    L.attn_decode_paged_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                            _i64, _i32, _f32, _i32, _i64, _i64, _vp]
    L.attn_decode_paged_noalloc.restype = _i32
    L.attn_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    L.attn_decode_workspace_size.restype = _sz
    L.attn_decode_num_splits.argtypes = [_i32, _i32, _i32, _i32]
    L.attn_decode_num_splits.restype = _i32
    L.store_kvcache.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, _i64, _i64, _vp]
    L.store_kvcache.restype = _i32
    L.attn_status_string.argtypes = [_i32]
    L.attn_status_string.restype = _c.c_char_p
    L.attn_get_last_device_error.argtypes = [_vp, _c.POINTER(_c.c_uint32)]
    L.attn_get_last_device_error.restype = _i32
    L.attn_abi_version.argtypes = []
    L.attn_abi_version.restype = _i32
    L.attn_selftest_bounded_wait.argtypes = [_vp, _c.POINTER(_c.c_ulonglong)]
    L.attn_selftest_bounded_wait.restype = _i32
    L.attn_kvcache_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _i64, _i32, _f32, _i32, _vp, _vp, _sz, _vp]
    L.attn_kvcache_fwd.restype = _i32
    L.attn_kvcache_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    L.attn_kvcache_workspace_size.restype = _sz
    L.attn_padded_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                                  _vp, _sz, _vp]
    L.attn_padded_fwd.restype = _i32
    L.attn_padded_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    L.attn_padded_workspace_size.restype = _sz
    L.attn_softmax_rows.argtypes = [_vp, _vp, _i64, _i32, _i64, _i64, _i32, _vp]
    L.attn_softmax_rows.restype = _i32
    L.attn_set_kernel_events.argtypes = [_vp, _vp]
    L.attn_set_kernel_events.restype = None
    L.attn_varlen_fwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                                       _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i32, _vp, _vp, _vp, _vp, _vp]
    L.attn_varlen_fwd_host.restype = _i32
    _lib = L
    return L


def exported_symbols() -> list[str]:
    """Function names declared in include/attn_varlen.h."""
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attn_varlen.h")
    src = open(hdr).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _rows(t: torch.Tensor, name: str, heads: int, dim: int) -> int:
    """Row stride (elements) of a [rows, heads, dim] view whose heads and dim are packed."""
    if t.dim() != 3 or t.shape[1] != heads or t.shape[2] != dim:
        raise ValueError(f"{name}: expected [rows, {heads}, {dim}], got {tuple(t.shape)}")
    if t.stride(2) != 1 or t.stride(1) != dim:
        raise ValueError(f"{name}: heads and head_dim must be packed (strides {t.stride()})")
    return t.stride(0) if t.shape[0] > 1 else heads * dim


def _bf16_cuda(*named):
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")


def _int_cuda(name, t, dtype):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


# --------------------------------------------------------------------------
# C-ABI bindings
# --------------------------------------------------------------------------

def attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                    softmax_scale: float | None = None, causal: bool = True, block_table=None,
                    out=None, lse=None, return_lse: bool = False, total_k: int | None = None,
                    workspace=None, stream=None, v16_cache=None):
    """Varlen prefill.  q [total_q, Hq, D]; k/v [total_k, Hkv, D] or, with
    block_table [B, max_blocks] int32, caches [num_blocks, block_size, Hkv, D].
    total_k (paged only): an upper bound of cu_seqlens_k[-1]; defaults to
    B * max_seqlen_k (no device sync).  v16_cache (paged only): the fp16 V / 16
    cache kept by store_kvcache(..., v16_cache=...); the call then converts nothing.
    Returns out [total_q, Hq, D] (and lse [Hq, total_q] float32 if asked)."""
    _bf16_cuda(("q", q), ("k", k), ("v", v), ("out", out))
    if v16_cache is not None:
        if block_table is None:
            raise ValueError("v16_cache goes with a paged cache (block_table)")
        if not v16_cache.is_cuda or v16_cache.dtype != torch.float16 or v16_cache.shape != k.shape \
                or not v16_cache.is_contiguous():
            raise ValueError("v16_cache must be a contiguous float16 CUDA tensor shaped like the caches")
    _int_cuda("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _int_cuda("cu_seqlens_k", cu_seqlens_k, torch.int32)
    total_q, Hq, D = q.shape
    paged = block_table is not None
    if paged:
        _int_cuda("block_table", block_table, torch.int32)
        if k.dim() != 4 or v.shape != k.shape or not k.is_contiguous() or not v.is_contiguous():
            raise ValueError("paged k/v must be contiguous [num_blocks, block_size, Hkv, D]")
        num_blocks, block_size, Hkv, _ = k.shape
        k_stride = v_stride = Hkv * D
        bt_stride = block_table.shape[1]
    else:
        Hkv = k.shape[1]
        k_stride = _rows(k, "k", Hkv, D)
        v_stride = _rows(v, "v", Hkv, D)
        total_k = k.shape[0]
        num_blocks = block_size = bt_stride = 0
    q_stride = _rows(q, "q", Hq, D)
    B = cu_seqlens_q.numel() - 1
    if paged and total_k is None:
        total_k = B * int(max_seqlen_k)
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    out_stride = _rows(out, "out", Hq, D)
    if return_lse and lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    L = lib()
    ws_bytes = L.attn_varlen_workspace_size(B, Hq, Hkv, D, int(max_seqlen_q), 0 if v16_cache is not None
                                            else int(total_k))
    if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws = workspace
    st = L.attn_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                           B, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, scale,
                           1 if causal else 0, _ptr(block_table), bt_stride, block_size, num_blocks, _ptr(v16_cache),
                           q_stride, k_stride, v_stride, out_stride, _ptr(ws), ws.numel() * ws.element_size(),
                           _stream(stream))
    _check(st, "attn_varlen_fwd")
    return (out, lse) if return_lse else out


def decode_num_splits(batch: int, num_heads_kv: int, max_cache_seqlen: int, num_splits: int = 0) -> int:
    return lib().attn_decode_num_splits(batch, num_heads_kv, max_cache_seqlen, num_splits)


def decode_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, max_cache_seqlen, num_splits=0) -> int:
    return lib().attn_decode_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, max_cache_seqlen,
                                            num_splits)


def host_staging(batch: int, total_q: int, total_k: int, num_heads_q: int, num_heads_kv: int, head_dim: int,
                 max_seqlen_q: int, device=None) -> dict:
    """Device buffers, copy streams and events that attn_varlen_fwd_host uses;
    make them once and pass them to every call of the same (or smaller) sizes."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws = lib().attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, int(max_seqlen_q), int(total_k))
    if ws == 0:
        raise ValueError("unsupported sizes for attn_varlen_fwd_host")
    bf = torch.bfloat16
    st = dict(q=torch.empty((total_q, num_heads_q, head_dim), dtype=bf, device=device),
              k=torch.empty((total_k, num_heads_kv, head_dim), dtype=bf, device=device),
              v=torch.empty((total_k, num_heads_kv, head_dim), dtype=bf, device=device),
              out=torch.empty((total_q, num_heads_q, head_dim), dtype=bf, device=device),
              cu=torch.empty(2 * (batch + 1), dtype=torch.int32, device=device),
              ws=torch.empty(ws, dtype=torch.uint8, device=device),
              s_in=torch.cuda.Stream(device), s_out=torch.cuda.Stream(device),
              ev=(torch.cuda.Event(), torch.cuda.Event()))
    for e in st["ev"]:
        e.record(torch.cuda.current_stream(device))   # torch creates the CUDA event on its first record
    return st


def attn_varlen_fwd_host(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                         softmax_scale: float | None = None, causal: bool = True, out=None, chunks: int = 8,
                         device=None, staging=None, synchronize: bool = True):
    """attn_varlen_fwd for host-resident inputs (C entry attn_varlen_fwd_host):
    q, k, v contiguous bf16 CPU tensors (pinned for the copies to overlap),
    cu_seqlens int32 CPU tensors.  The library copies groups of sequences in,
    runs the attention of each group and copies its output back, overlapped on
    three streams.  Returns the output in a pinned CPU tensor (`out` if given);
    with synchronize=True (default) after it has arrived.  `staging` (from
    host_staging) supplies reusable device buffers, streams and events."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous [rows, heads, dim] bf16 CPU tensor")
    cq = torch.as_tensor(cu_seqlens_q)
    ck = torch.as_tensor(cu_seqlens_k)
    for name, t in (("cu_seqlens_q", cq), ("cu_seqlens_k", ck)):
        if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CPU tensor")
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    B = cq.numel() - 1
    if ck.numel() != B + 1 or v.shape != k.shape:
        raise ValueError("cu_seqlens_q / cu_seqlens_k / k / v do not match")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if staging is None:
        staging = host_staging(B, total_q, total_k, Hq, Hkv, D, max_seqlen_q, device)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    elif out.is_cuda or out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 CPU tensor shaped like q")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    main = torch.cuda.current_stream(device)
    ws = staging["ws"]
    ev_a, ev_b = staging["ev"]
    st = lib().attn_varlen_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cq), _ptr(ck), B, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv,
        D, scale, 1 if causal else 0, _ptr(staging["q"]), _ptr(staging["k"]), _ptr(staging["v"]),
        _ptr(staging["out"]), _ptr(staging["cu"]), _ptr(ws), ws.numel(), int(chunks),
        ctypes.c_void_p(main.cuda_stream), ctypes.c_void_p(staging["s_in"].cuda_stream),
        ctypes.c_void_p(staging["s_out"].cuda_stream), ctypes.c_void_p(ev_a.cuda_event),
        ctypes.c_void_p(ev_b.cuda_event))
    _check(st, "attn_varlen_fwd_host")
    if synchronize:
        main.synchronize()
    return out


def attn_decode_paged(q, k_cache, v_cache, cache_seqlens, block_table, softmax_scale: float | None = None,
                      max_cache_seqlen: int | None = None, num_splits: int = 0, out=None, lse=None,
                      return_lse: bool = False, workspace=None, stream=None):
    """Decode: q [B, Hq, D] (or [B, 1, Hq, D]); caches [num_blocks, block_size,
    Hkv, D]; cache_seqlens int32 [B]; block_table int32 [B, max_blocks]; at most
    64 query heads per KV head.  max_cache_seqlen defaults to the block table's
    capacity (no device sync)."""
    if q.dim() == 4:
        if q.shape[1] != 1:
            raise ValueError("attn_decode_paged takes one query token per sequence")
        q = q[:, 0]
    _bf16_cuda(("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out))
    _int_cuda("cache_seqlens", cache_seqlens, torch.int32)
    _int_cuda("block_table", block_table, torch.int32)
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() \
            or not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, D]")
    B, Hq, D = q.shape
    num_blocks, block_size, Hkv, _ = k_cache.shape
    q_stride = _rows(q, "q", Hq, D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    out_stride = _rows(out, "out", Hq, D)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if max_cache_seqlen is None:
        max_cache_seqlen = block_table.shape[1] * block_size
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    L = lib()
    ws_bytes = L.attn_decode_workspace_size(B, Hq, Hkv, D, int(max_cache_seqlen), int(num_splits))
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_have = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = L.attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(cache_seqlens),
                             _ptr(block_table), block_table.shape[1], B, Hq, Hkv, D, block_size, num_blocks,
                             int(max_cache_seqlen), scale, int(num_splits), q_stride, out_stride, _ptr(workspace),
                             ws_have, _stream(stream))
    _check(st, "attn_decode_paged")
    return (out, lse) if return_lse else out


def attn_with_kvcache(q, k_cache, v_cache, cache_seqlens, block_table, softmax_scale: float | None = None,
                      causal: bool = True, max_cache_seqlen: int | None = None, out=None, lse=None,
                      return_lse: bool = False, workspace=None, stream=None, v16_cache=None):
    """Several new tokens per sequence against the paged cache: q [B, Sq, Hq, D]
    (Sq >= 1, all sequences the same Sq); caches [num_blocks, block_size, Hkv, D];
    cache_seqlens int32 [B] counts the cached keys including the Sq new ones.
    Returns out [B, Sq, Hq, D] (and lse [Hq, B*Sq]).  Up to 64 query rows per KV
    head (Sq x Hq/Hkv) run on the split-KV decode kernel, more on the prefill kernel
    (which reads v16_cache, the fp16 V / 16 cache, when given)."""
    if v16_cache is not None and (not v16_cache.is_cuda or v16_cache.dtype != torch.float16
                                  or v16_cache.shape != k_cache.shape or not v16_cache.is_contiguous()):
        raise ValueError("v16_cache must be a contiguous float16 CUDA tensor shaped like the caches")
    if q.dim() != 4:
        raise ValueError("q must be [B, seqlen_q, Hq, D]")
    _bf16_cuda(("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out))
    _int_cuda("cache_seqlens", cache_seqlens, torch.int32)
    _int_cuda("block_table", block_table, torch.int32)
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() \
            or not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, D]")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    B, Sq, Hq, D = q.shape
    num_blocks, block_size, Hkv, _ = k_cache.shape
    if cache_seqlens.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("cache_seqlens / block_table do not match the batch")
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=q.device)
    elif out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if return_lse and lse is None:
        lse = torch.empty((Hq, B * Sq), dtype=torch.float32, device=q.device)
    if max_cache_seqlen is None:
        max_cache_seqlen = block_table.shape[1] * block_size
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    L = lib()
    ws_bytes = L.attn_kvcache_workspace_size(B, Sq, Hq, Hkv, D, int(max_cache_seqlen))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    ws_have = workspace.numel() * workspace.element_size()
    st = L.attn_kvcache_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(cache_seqlens),
                            _ptr(block_table), block_table.shape[1], B, Sq, Hq, Hkv, D, block_size, num_blocks,
                            int(max_cache_seqlen), scale, 1 if causal else 0, _ptr(v16_cache), _ptr(workspace),
                            ws_have, _stream(stream))
    _check(st, "attn_kvcache_fwd")
    return (out, lse) if return_lse else out


def attn_padded_fwd(q, k, v, seqlens_q=None, seqlens_k=None, softmax_scale: float | None = None,
                    causal: bool = True, out=None, lse=None, return_lse: bool = False, workspace=None,
                    stream=None):
    """Padded batch: q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D] (contiguous); only the
    first seqlens_q[b] / seqlens_k[b] rows of sequence b are real (int32 [B],
    None = all).  Returns out [B, Sq, Hq, D] (padding rows are not written) and
    lse [Hq, B*Sq] if asked."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, Sq, Hq, D] and k, v [B, Sk, Hkv, D]")
    _bf16_cuda(("q", q), ("k", k), ("v", v), ("out", out))
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    if k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k does not match q")
    for name, t in (("seqlens_q", seqlens_q), ("seqlens_k", seqlens_k)):
        if t is not None:
            _int_cuda(name, t, torch.int32)
            if t.numel() != B:
                raise ValueError(f"{name} must have one entry per sequence")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if return_lse and lse is None:
        lse = torch.empty((Hq, B * Sq), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    L = lib()
    ws_bytes = L.attn_padded_workspace_size(B, Sq, Sk, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    ws_have = workspace.numel() * workspace.element_size()
    st = L.attn_padded_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seqlens_q), _ptr(seqlens_k), B, Sq,
                           Sk, Hq, Hkv, D, scale, 1 if causal else 0, _ptr(workspace), ws_have, _stream(stream))
    _check(st, "attn_padded_fwd")
    return (out, lse) if return_lse else out


def softmax_rows(x, out=None, stream=None):
    """Softmax along the last dimension of a float32 or bfloat16 CUDA tensor
    (any leading shape; rows may be strided, the last dimension contiguous).
    out: same shape and dtype (may be x)."""
    if not x.is_cuda or x.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("x must be a float32 or bfloat16 CUDA tensor")
    if x.dim() == 0 or x.stride(-1) != 1:
        raise ValueError("the last dimension of x must be contiguous")
    cols = x.shape[-1]
    x2 = x.reshape(-1, cols) if x.dim() != 2 else x
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    if out.shape != x.shape or out.dtype != x.dtype or out.stride(-1) != 1:
        raise ValueError("out must match x in shape and dtype")
    o2 = out.reshape(-1, cols) if out.dim() != 2 else out
    if o2.data_ptr() != out.data_ptr() or x2.data_ptr() != x.data_ptr():
        raise ValueError("x and out must be viewable as [rows, cols]")
    dtype = 1 if x.dtype == torch.bfloat16 else 0
    st = lib().attn_softmax_rows(_ptr(x2), _ptr(o2), x2.shape[0], cols, x2.stride(0) if x2.shape[0] > 1 else cols,
                                 o2.stride(0) if o2.shape[0] > 1 else cols, dtype, _stream(stream))
    _check(st, "attn_softmax_rows")
    return out


def store_kvcache(k, v, k_cache, v_cache, slot_mapping, stream=None, v16_cache=None):
    """Scatter k/v [N, Hkv, D] into caches [num_blocks, block_size, Hkv, D] (or
    any [num_slots, Hkv, D] view) at the flat slots slot_mapping (int64 [N]).
    v16_cache (float16, shaped like the caches): also receives V / 16."""
    _bf16_cuda(("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache))
    if v16_cache is not None and (not v16_cache.is_cuda or v16_cache.dtype != torch.float16
                                  or v16_cache.shape != v_cache.shape or not v16_cache.is_contiguous()):
        raise ValueError("v16_cache must be a contiguous float16 CUDA tensor shaped like the caches")
    _int_cuda("slot_mapping", slot_mapping, torch.int64)
    N, Hkv, D = k.shape
    if not k_cache.is_contiguous() or not v_cache.is_contiguous() or k_cache.shape != v_cache.shape:
        raise ValueError("caches must be contiguous and of the same shape")
    if k_cache.shape[-2:] != (Hkv, D):
        raise ValueError("cache head layout does not match k")
    num_slots = k_cache.numel() // (Hkv * D)
    ks = _rows(k, "k", Hkv, D)
    vs = _rows(v, "v", Hkv, D)
    if slot_mapping.numel() != N:
        raise ValueError("slot_mapping must have one entry per token")
    st = lib().store_kvcache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(v16_cache), _ptr(slot_mapping), N,
                             Hkv, D, ks, vs, num_slots, _stream(stream))
    _check(st, "store_kvcache")


def set_kernel_events(before=None, after=None) -> None:
    """Record two torch.cuda.Event objects (created with enable_timing=True)
    around the main kernel of every later attention call from this thread:
    the prefill's attention kernel or the decode's split-KV kernel.  Call
    with no arguments to switch it off.  Measurement aid for benchmarks."""
    if (before is None) != (after is None):
        raise ValueError("give both events or neither")
    if before is None:
        lib().attn_set_kernel_events(None, None)
        return
    # torch creates the CUDA event on its first record()
    for e in (before, after):
        if not e.cuda_event:
            e.record()
    if not before.cuda_event or not after.cuda_event:
        raise ValueError("events have no CUDA event handle")
    lib().attn_set_kernel_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def selftest_bounded_wait(stream=None) -> dict:
    """Run the library's failure-detection self-test (a bounded wait that runs
    out on purpose; see attn_selftest_bounded_wait).  Returns the two waiters'
    success flags and waited nanoseconds; the device error word then holds the
    timeout."""
    res = (ctypes.c_ulonglong * 4)()
    _check(lib().attn_selftest_bounded_wait(_stream(stream), res), "attn_selftest_bounded_wait")
    return {"first_ok": bool(res[0]), "first_ns": int(res[1]), "second_ok": bool(res[2]), "second_ns": int(res[3])}


def get_last_device_error(stream=None) -> tuple[int, int]:
    """Synchronise the stream and read / clear the device error word.
    Returns (status, raw word)."""
    word = ctypes.c_uint32(0)
    st = lib().attn_get_last_device_error(_stream(stream), ctypes.byref(word))
    return st, word.value
