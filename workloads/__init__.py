"""Seeded synthetic inputs for the attention path, shared by the tests, the
smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers, builds index
structures (cu_seqlens, block tables, slot mappings) and counts work.  Both the
CUDA path and the float64 oracle take their inputs from here; neither is
imported by it.

Five workloads, in order (shapes follow the varlen / prefix-cache / decode
examples of "从零实现 vLLM (1.3)：如何加速 Attention 计算", sections "Prefill"
and "Decode"):

  c1_tiny         3 sequences, cu_seqlens_q=[0,5,7,8], cu_seqlens_k=[0,9,16,19],
                  4 heads, head_dim 64, contiguous K/V (the article's own example)
  c2_varlen_gqa   16 sequences, L ~ U{256..4096}, Lq = Lk, GQA 32/8, head_dim 128
  c3_prefix_paged 32 sequences, cached context ~ U{512..8192} plus 1..512 new
                  tokens, paged cache (block_size 256) over a 65,536-block pool,
                  the first 8 sequences sharing their leading prefix blocks
  c4_decode       256 sequences, one query token each, cache_seqlens ~
                  U{128..16384}, block_size 256, pool = total context
  c5_long         2 sequences of 32,768 tokens, MHA 32 heads, head_dim 128;
                  heads 0-15 have Q scaled by 160 before bf16 rounding so the
                  scaled logits reach ~700

Values are N(0, 1) drawn in float32 by numpy's PCG64 and rounded to bf16
(round-to-nearest-even).  Every draw is keyed by (seed, tensor tag, chunk id),
so any subset of a large tensor (a block of the paged cache, a row chunk) can be
regenerated on its own: that is how the oracle gets the inputs of sampled rows
without materialising a multi-gigabyte cache on the host.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 1234
ROW_CHUNK = 256          # tokens per independently seeded chunk of a packed tensor

# tensor tags (part of every seed key)
TAG_Q, TAG_K, TAG_V, TAG_KNEW, TAG_VNEW, TAG_LEN, TAG_PERM, TAG_SAMPLE = range(1, 9)
SHARED = 1 << 20         # "sequence" id used for the shared prefix blocks

CONFIG_NAMES = ["c1_tiny", "c2_varlen_gqa", "c3_prefix_paged", "c4_decode", "c5_long"]


def _nthreads() -> int:
    return max(1, min(32, torch.get_num_threads()))


def normal_bf16(key, n_rows: int, row_elems: int, scale_rows=None) -> torch.Tensor:
    """[n_rows, row_elems] bf16 ~ N(0,1), drawn in chunks of ROW_CHUNK rows,
    chunk c seeded by key + (c,).  scale_rows: optional float32 [row_elems]
    multiplier applied before rounding (used for the overflow-stress heads)."""
    out = torch.empty((n_rows, row_elems), dtype=torch.bfloat16)
    n_chunks = (n_rows + ROW_CHUNK - 1) // ROW_CHUNK

    def job(c):
        r0 = c * ROW_CHUNK
        r1 = min(n_rows, r0 + ROW_CHUNK)
        rng = np.random.default_rng(list(key) + [c])
        x = rng.standard_normal((r1 - r0, row_elems), dtype=np.float32)
        if scale_rows is not None:
            x *= scale_rows[None, :]
        out[r0:r1] = torch.from_numpy(x).to(torch.bfloat16)

    if n_chunks <= 1:
        for c in range(n_chunks):
            job(c)
    else:
        with ThreadPoolExecutor(_nthreads()) as ex:
            list(ex.map(job, range(n_chunks)))
    return out


def block_bf16(key, block_size: int, row_elems: int) -> torch.Tensor:
    """One paged-cache block [block_size, row_elems] bf16 ~ N(0,1) keyed by `key`."""
    rng = np.random.default_rng(list(key))
    x = rng.standard_normal((block_size, row_elems), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def cu_from_lens(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


# --------------------------------------------------------------------------
# workload descriptions (host-side metadata; small)
# --------------------------------------------------------------------------

@dataclass
class Varlen:
    """Contiguous varlen prefill: q [total_q, Hq, D], k/v [total_k, Hkv, D]."""
    name: str
    seed: int
    Hq: int
    Hkv: int
    D: int
    lens_q: np.ndarray
    lens_k: np.ndarray
    causal: bool = True
    q_head_scale: np.ndarray | None = None   # float32 [Hq] or None

    @property
    def batch(self):
        return len(self.lens_q)

    @property
    def cu_q(self):
        return cu_from_lens(self.lens_q)

    @property
    def cu_k(self):
        return cu_from_lens(self.lens_k)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.D)

    def q(self) -> torch.Tensor:
        sr = None
        if self.q_head_scale is not None:
            sr = np.repeat(self.q_head_scale.astype(np.float32), self.D)
        return normal_bf16((self.seed, TAG_Q), int(self.lens_q.sum()), self.Hq * self.D,
                           sr).view(-1, self.Hq, self.D)

    def k(self) -> torch.Tensor:
        return normal_bf16((self.seed, TAG_K), int(self.lens_k.sum()), self.Hkv * self.D).view(-1, self.Hkv, self.D)

    def v(self) -> torch.Tensor:
        return normal_bf16((self.seed, TAG_V), int(self.lens_k.sum()), self.Hkv * self.D).view(-1, self.Hkv, self.D)


@dataclass
class Paged:
    """Paged-cache workload (prefix-cache prefill or decode).

    Sequence b has ctx[b] cached tokens and new[b] new tokens.  For decode
    new = 0 and the one query token of b attends to all cache_seqlens[b] =
    ctx[b] cached keys (its own K/V is taken to be stored already).
    block_table[b] lists physical block ids; logical block i of b holds tokens
    [i*bs, (i+1)*bs)."""
    name: str
    seed: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    ctx: np.ndarray
    new: np.ndarray
    block_table: np.ndarray               # int32 [B, max_blocks] (unused entries = -1)
    shared_blocks: int = 0                # leading logical blocks shared by sequences < n_shared
    n_shared: int = 0
    decode: bool = False

    @property
    def batch(self):
        return len(self.ctx)

    @property
    def lens_k(self):
        return (self.ctx + self.new).astype(np.int64)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.D)

    def block_key(self, tag: int, b: int, i: int):
        if self.n_shared and b < self.n_shared and i < self.shared_blocks:
            return (self.seed, tag, SHARED, i)
        return (self.seed, tag, b, i)

    def block_content(self, tag: int, b: int, i: int) -> torch.Tensor:
        return block_bf16(self.block_key(tag, b, i), self.block_size, self.Hkv * self.D)

    def n_ctx_blocks(self, b: int) -> int:
        return (int(self.ctx[b]) + self.block_size - 1) // self.block_size

    def slot_mapping(self) -> np.ndarray:
        """Flat slots (block_id * block_size + offset) of the new tokens, in
        packed order."""
        out = []
        bs = self.block_size
        for b in range(self.batch):
            j = np.arange(int(self.ctx[b]), int(self.ctx[b] + self.new[b]), dtype=np.int64)
            out.append(self.block_table[b, j // bs].astype(np.int64) * bs + j % bs)
        return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)

    def k_new(self) -> torch.Tensor:
        return normal_bf16((self.seed, TAG_KNEW), int(self.new.sum()), self.Hkv * self.D).view(-1, self.Hkv, self.D)

    def v_new(self) -> torch.Tensor:
        return normal_bf16((self.seed, TAG_VNEW), int(self.new.sum()), self.Hkv * self.D).view(-1, self.Hkv, self.D)

    def q(self) -> torch.Tensor:
        """Prefill: [sum new, Hq, D].  Decode: [B, Hq, D]."""
        n = self.batch if self.decode else int(self.new.sum())
        return normal_bf16((self.seed, TAG_Q), n, self.Hq * self.D).view(-1, self.Hq, self.D)

    def context_blocks(self, seqs=None):
        """Yield (physical block id, logical (b, i), k block, v block) for every
        block that holds cached context of the chosen sequences, shared blocks
        once.  Rows at or beyond ctx[b] inside the last block are returned
        as drawn; callers decide what the cache holds there."""
        seen = set()
        seqs = range(self.batch) if seqs is None else seqs
        for b in seqs:
            for i in range(self.n_ctx_blocks(b)):
                pb = int(self.block_table[b, i])
                if pb in seen:
                    continue
                seen.add(pb)
                yield pb, (b, i), self.block_content(TAG_K, b, i), self.block_content(TAG_V, b, i)

    def ctx_rows_valid(self, b: int, i: int) -> int:
        """How many rows of logical block i of sequence b hold cached context."""
        return int(max(0, min(self.block_size, int(self.ctx[b]) - i * self.block_size)))


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def make(name: str) -> Varlen | Paged:
    idx = CONFIG_NAMES.index(name)
    seed = SEED_BASE + idx
    rng = np.random.default_rng([seed, TAG_LEN])
    if name == "c1_tiny":
        return Varlen(name, seed, 4, 4, 64, np.array([5, 2, 1]), np.array([9, 7, 3]))
    if name == "c2_varlen_gqa":
        L = rng.integers(256, 4096, size=16, endpoint=True)
        return Varlen(name, seed, 32, 8, 128, L.copy(), L.copy())
    if name == "c5_long":
        L = np.array([32768, 32768])
        hs = np.ones(32, dtype=np.float32)
        hs[:16] = 160.0
        return Varlen(name, seed, 32, 32, 128, L, L.copy(), q_head_scale=hs)
    if name == "c3_prefix_paged":
        B, bs, pool = 32, 256, 65536
        ctx = rng.integers(512, 8192, size=B, endpoint=True)
        new = rng.integers(1, 512, size=B, endpoint=True)
        return _paged(name, seed, rng, 32, 8, 128, bs, pool, ctx, new, n_shared=8)
    if name == "c4_decode":
        B, bs = 256, 256
        ctx = rng.integers(128, 16384, size=B, endpoint=True)
        new = np.zeros(B, dtype=np.int64)
        pool = int(sum((int(c) + bs - 1) // bs for c in ctx))
        return _paged(name, seed, rng, 32, 8, 128, bs, pool, ctx, new, decode=True)
    raise KeyError(name)


def _paged(name, seed, rng, Hq, Hkv, D, bs, pool, ctx, new, n_shared=0, decode=False) -> Paged:
    B = len(ctx)
    total = ctx + new
    nblk = [(int(t) + bs - 1) // bs for t in total]
    max_blocks = max(nblk)
    shared_blocks = 0
    if n_shared:
        shared_blocks = int(min(ctx[:n_shared])) // bs
    perm = np.random.default_rng([seed, TAG_PERM]).permutation(pool).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    nxt = 0
    shared_ids = perm[:shared_blocks]
    nxt = shared_blocks
    for b in range(B):
        for i in range(nblk[b]):
            if n_shared and b < n_shared and i < shared_blocks:
                bt[b, i] = shared_ids[i]
            else:
                bt[b, i] = perm[nxt]
                nxt += 1
    assert nxt <= pool, "pool too small"
    return Paged(name, seed, Hq, Hkv, D, bs, pool, np.asarray(ctx, dtype=np.int64),
                 np.asarray(new, dtype=np.int64), bt, shared_blocks, n_shared, decode)


def small_varlen(seed: int, lens_q, lens_k, Hq: int, Hkv: int, D: int, causal: bool = True,
                 q_head_scale=None) -> Varlen:
    """An ad-hoc varlen case for parity tests (same generator, other shapes)."""
    return Varlen(f"varlen_s{seed}", seed, Hq, Hkv, D, np.asarray(lens_q), np.asarray(lens_k), causal,
                  None if q_head_scale is None else np.asarray(q_head_scale, dtype=np.float32))


def small_paged(seed: int, ctx, new, Hq: int, Hkv: int, D: int, block_size: int,
                extra_blocks: int = 3, decode: bool = False, n_shared: int = 0) -> Paged:
    """An ad-hoc paged case: pool = needed blocks + extra_blocks, random table."""
    ctx = np.asarray(ctx, dtype=np.int64)
    new = np.asarray(new, dtype=np.int64)
    need = sum((int(c + n) + block_size - 1) // block_size for c, n in zip(ctx, new))
    rng = np.random.default_rng([seed, TAG_LEN])
    return _paged(f"paged_s{seed}", seed, rng, Hq, Hkv, D, block_size, need + extra_blocks, ctx, new,
                  n_shared=n_shared, decode=decode)


# --------------------------------------------------------------------------
# work accounting (counts, not attention arithmetic)
# --------------------------------------------------------------------------

def visible_pairs(Lq: int, Lk: int, causal: bool = True) -> int:
    """Number of (query, key) pairs left unmasked for one sequence under
    bottom-right causal alignment: query i sees keys j <= Lk - Lq + i, so row i
    has clamp(Lk - Lq + i + 1, 0, Lk) visible keys."""
    if not causal:
        return Lq * Lk
    i = np.arange(Lq, dtype=np.int64)
    return int(np.clip(Lk - Lq + i + 1, 0, Lk).sum())


def prefill_flops(lens_q, lens_k, Hq: int, D: int, causal: bool = True) -> int:
    """4 * D * Hq * sum_b pairs_b: QK^T and PV at 2 flops per multiply-add."""
    pairs = sum(visible_pairs(int(a), int(b), causal) for a, b in zip(lens_q, lens_k))
    return 4 * D * Hq * pairs


def decode_bytes(cache_seqlens, Hq: int, Hkv: int, D: int, block_size: int) -> int:
    """Bytes a decode step must move: K and V of every cached token once per KV
    head (bf16), plus q in, out, and the block-table entries read."""
    L = np.asarray(cache_seqlens, dtype=np.int64)
    kv = int(L.sum()) * Hkv * D * 2 * 2
    B = len(L)
    qo = 2 * B * Hq * D * 2
    bt = int(sum((int(x) + block_size - 1) // block_size for x in L)) * 4
    return kv + qo + bt + B * 4


def store_bytes(num_tokens: int, Hkv: int, D: int, v16: bool = False) -> int:
    """store_kvcache: read k and v rows, write them, read the int64 slots; with
    the fp16 V / 16 cache, write a third row per token."""
    return 2 * num_tokens * Hkv * D * 2 * 2 + 8 * num_tokens + (num_tokens * Hkv * D * 2 if v16 else 0)


def sample_rows(seed: int, n_rows: int, fraction: float = 1 / 64, cap: int | None = None) -> np.ndarray:
    """Deterministic uniform sample of row ids in [0, n_rows), sorted."""
    k = max(1, int(math.ceil(n_rows * fraction)))
    if cap is not None:
        k = min(k, cap)
    rng = np.random.default_rng([seed, TAG_SAMPLE])
    return np.sort(rng.choice(n_rows, size=k, replace=False)).astype(np.int64)


# --------------------------------------------------------------------------
# materialising paged caches (device placement is plain copying)
# --------------------------------------------------------------------------

def _ctx_block_items(cfg: Paged, seqs=None):
    seen, items = set(), []
    for b in (range(cfg.batch) if seqs is None else seqs):
        for i in range(cfg.n_ctx_blocks(b)):
            pb = int(cfg.block_table[b, i])
            if pb not in seen:
                seen.add(pb)
                items.append((pb, b, i))
    return items


def _draw_blocks(cfg: Paged, items):
    """Host tensors [n, bs, Hkv*D] (K and V) for the listed context blocks."""
    n = len(items)
    row = cfg.Hkv * cfg.D
    kh = torch.empty((n, cfg.block_size, row), dtype=torch.bfloat16)
    vh = torch.empty_like(kh)

    def job(t):
        _, b, i = items[t]
        kh[t] = cfg.block_content(TAG_K, b, i)
        vh[t] = cfg.block_content(TAG_V, b, i)

    with ThreadPoolExecutor(_nthreads()) as ex:
        list(ex.map(job, range(n)))
    return kh, vh


def fill_paged_cache(cfg: Paged, k_cache: torch.Tensor, v_cache: torch.Tensor, seqs=None, batch_blocks: int = 512):
    """Write every drawn context block of the chosen sequences into the caches
    ([num_blocks, block_size, Hkv, D], any device) at its physical block id.
    Other blocks are left as they are."""
    items = _ctx_block_items(cfg, seqs)
    kf = k_cache.view(cfg.num_blocks, -1)
    vf = v_cache.view(cfg.num_blocks, -1)
    for s in range(0, len(items), batch_blocks):
        chunk = items[s:s + batch_blocks]
        kh, vh = _draw_blocks(cfg, chunk)
        idx = torch.tensor([pb for pb, _, _ in chunk], dtype=torch.int64, device=k_cache.device)
        if k_cache.is_cuda:
            kh, vh = kh.pin_memory(), vh.pin_memory()
        kf.index_copy_(0, idx, kh.view(len(chunk), -1).to(k_cache.device, non_blocking=True))
        vf.index_copy_(0, idx, vh.view(len(chunk), -1).to(v_cache.device, non_blocking=True))


def compact_paged(cfg: Paged, seqs):
    """A small host-side pool holding only the blocks of `seqs`.

    Returns (k_pool, v_pool, block_table) with pools [n_blocks, bs, Hkv, D]
    bf16 (context blocks drawn, blocks for new tokens zero) and the block
    table of `seqs` renumbered into the pool.  Paging is a pure copy, so
    attention over it equals attention over the full pool."""
    remap = {}
    for b in seqs:
        nb = (int(cfg.lens_k[b]) + cfg.block_size - 1) // cfg.block_size
        for i in range(nb):
            pb = int(cfg.block_table[b, i])
            if pb not in remap:
                remap[pb] = len(remap)
    n = len(remap)
    kp = torch.zeros((n, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    items = _ctx_block_items(cfg, seqs)
    if items:
        kh, vh = _draw_blocks(cfg, items)
        for t, (pb, _, _) in enumerate(items):
            kp[remap[pb]] = kh[t].view(cfg.block_size, cfg.Hkv, cfg.D)
            vp[remap[pb]] = vh[t].view(cfg.block_size, cfg.Hkv, cfg.D)
    width = cfg.block_table.shape[1]
    bt = np.full((len(seqs), width), -1, dtype=np.int32)
    for r, b in enumerate(seqs):
        nb = (int(cfg.lens_k[b]) + cfg.block_size - 1) // cfg.block_size
        for i in range(nb):
            bt[r, i] = remap[int(cfg.block_table[b, i])]
    return kp, vp, bt
