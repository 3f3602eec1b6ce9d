"""Attention-layer dispatch over the library's calls.

One call per layer and step, following "从零实现 vLLM (1.3)：如何加速 Attention
计算", section "Attention 源码分析": the step's new K/V are first written into the
paged cache (store_kvcache at slot_mapping), then

  * prefill: varlen attention over the packed new tokens; when the step carries
    block tables (prefix cache), K/V are read from the caches instead of the
    step's own k/v;
  * decode: one query token per sequence against the cache (context_lens =
    cache_seqlens, which include the token just stored).  A decode step that
    carries the same number of new tokens for every sequence (speculative
    verification; the page shows one) goes through the kv-cache entry with
    bottom-right causality among the new tokens.

Everything runs in the library's kernels; this module only routes tensors.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import attn_decode_paged, attn_varlen_fwd, attn_with_kvcache, store_kvcache


@dataclass
class AttentionContext:
    """Per-step metadata shared by all attention layers of a forward pass."""
    is_prefill: bool
    slot_mapping: torch.Tensor | None = None     # int64 [N]: flat cache slot of each new token (< 0: skip)
    cu_seqlens_q: torch.Tensor | None = None     # int32 [B+1] (prefill)
    cu_seqlens_k: torch.Tensor | None = None     # int32 [B+1] (prefill)
    max_seqlen_q: int = 0
    max_seqlen_k: int = 0
    context_lens: torch.Tensor | None = None     # int32 [B] (decode): cached keys incl. the new tokens
    block_tables: torch.Tensor | None = None     # int32 [B, max_blocks] (prefix prefill, decode)


class Attention:
    """Causal attention of one layer with a paged KV cache.

    k_cache / v_cache ([num_blocks, block_size, num_kv_heads, head_dim] bf16)
    are bound by the owner (for instance after sizing the pool); until then the
    layer runs without a cache (prefill only).  An optional v16_cache (float16,
    same shape) keeps V / 16 next to the bf16 V: the store fills it and the
    prefix prefill reads it instead of converting the cached V every step."""

    def __init__(self, num_heads: int, head_dim: int, scale: float, num_kv_heads: int):
        if num_heads % num_kv_heads:
            raise ValueError("num_heads must be a multiple of num_kv_heads")
        self.num_heads = num_heads
        self.head_dim = head_dim
        self.scale = float(scale)
        self.num_kv_heads = num_kv_heads
        self.k_cache: torch.Tensor | None = None
        self.v_cache: torch.Tensor | None = None
        self.v16_cache: torch.Tensor | None = None

    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ctx: AttentionContext) -> torch.Tensor:
        """q [N, Hq*D] or [N, Hq, D]; k, v [N, Hkv*D] or [N, Hkv, D].  Returns o
        with q's shape."""
        shape = q.shape
        q = q.view(-1, self.num_heads, self.head_dim)
        k = k.view(-1, self.num_kv_heads, self.head_dim)
        v = v.view(-1, self.num_kv_heads, self.head_dim)
        cached = self.k_cache is not None and self.v_cache is not None and self.k_cache.numel() > 0
        if cached and ctx.slot_mapping is not None and ctx.slot_mapping.numel():
            store_kvcache(k, v, self.k_cache, self.v_cache, ctx.slot_mapping, v16_cache=self.v16_cache)
        if ctx.is_prefill:
            if ctx.block_tables is not None:
                if not cached:
                    raise ValueError("prefix prefill needs the KV cache")
                o = attn_varlen_fwd(q, self.k_cache, self.v_cache, ctx.cu_seqlens_q, ctx.cu_seqlens_k,
                                    ctx.max_seqlen_q, ctx.max_seqlen_k, self.scale, causal=True,
                                    block_table=ctx.block_tables, v16_cache=self.v16_cache)
            else:
                o = attn_varlen_fwd(q, k, v, ctx.cu_seqlens_q, ctx.cu_seqlens_k, ctx.max_seqlen_q,
                                    ctx.max_seqlen_k, self.scale, causal=True)
        else:
            if not cached:
                raise ValueError("decode needs the KV cache")
            if ctx.context_lens is None or ctx.block_tables is None:
                raise ValueError("decode needs context_lens and block_tables")
            batch, n = ctx.context_lens.numel(), q.shape[0]
            if n == batch:
                o = attn_decode_paged(q, self.k_cache, self.v_cache, ctx.context_lens, ctx.block_tables, self.scale,
                                      max_cache_seqlen=ctx.max_seqlen_k or None)
            else:
                if batch == 0 or n % batch:
                    raise ValueError("a decode step carries the same number of new tokens for every sequence")
                sq = n // batch
                o = attn_with_kvcache(q.reshape(batch, sq, self.num_heads, self.head_dim), self.k_cache,
                                      self.v_cache, ctx.context_lens, ctx.block_tables, self.scale, causal=True,
                                      max_cache_seqlen=ctx.max_seqlen_k or None, v16_cache=self.v16_cache)
        return o.view(shape)

    __call__ = forward
