"""Routing of the Attention layer (no GPU): which library call runs, in which
order, with which tensors."""
import pytest
import torch

import attention_attn_varlen_gb300.attention as at


@pytest.fixture
def calls(monkeypatch):
    log = []

    def fake_store(k, v, kc, vc, slots, v16_cache=None):
        log.append(("store", k, kc, slots, v16_cache))

    def fake_varlen(q, k, v, cu_q, cu_k, mq, mk, scale, causal=True, block_table=None, v16_cache=None):
        log.append(("varlen", k, block_table, causal, scale, v16_cache))
        return torch.zeros_like(q)

    def fake_decode(q, kc, vc, lens, bt, scale, max_cache_seqlen=None):
        log.append(("decode", kc, lens, bt, max_cache_seqlen))
        return torch.zeros_like(q)

    monkeypatch.setattr(at, "store_kvcache", fake_store)
    monkeypatch.setattr(at, "attn_varlen_fwd", fake_varlen)
    def fake_kvcache(q, kc, vc, lens, bt, scale, causal=True, max_cache_seqlen=None, v16_cache=None):
        log.append(("kvcache", tuple(q.shape), lens, bt, causal, max_cache_seqlen))
        return torch.zeros_like(q)

    monkeypatch.setattr(at, "attn_decode_paged", fake_decode)
    monkeypatch.setattr(at, "attn_with_kvcache", fake_kvcache)
    return log


def _layer(cache=True):
    layer = at.Attention(num_heads=8, head_dim=16, scale=0.25, num_kv_heads=2)
    if cache:
        layer.k_cache = torch.zeros(4, 16, 2, 16)
        layer.v_cache = torch.zeros(4, 16, 2, 16)
    return layer


def _qkv(n):
    return torch.randn(n, 8 * 16), torch.randn(n, 2 * 16), torch.randn(n, 2 * 16)


def test_prefill_without_cache_uses_the_step_kv(calls):
    layer = _layer(cache=False)
    q, k, v = _qkv(5)
    ctx = at.AttentionContext(is_prefill=True, cu_seqlens_q=torch.tensor([0, 5]), cu_seqlens_k=torch.tensor([0, 5]),
                              max_seqlen_q=5, max_seqlen_k=5)
    o = layer(q, k, v, ctx)
    assert o.shape == q.shape
    assert [c[0] for c in calls] == ["varlen"]
    assert calls[0][1].shape == (5, 2, 16) and calls[0][2] is None and calls[0][3] is True and calls[0][4] == 0.25


def test_store_runs_before_attention_in_prefill(calls):
    layer = _layer()
    q, k, v = _qkv(5)
    slots = torch.arange(5, dtype=torch.int64)
    ctx = at.AttentionContext(is_prefill=True, slot_mapping=slots, cu_seqlens_q=torch.tensor([0, 5]),
                              cu_seqlens_k=torch.tensor([0, 5]), max_seqlen_q=5, max_seqlen_k=5)
    layer(q, k, v, ctx)
    assert [c[0] for c in calls] == ["store", "varlen"]
    assert calls[0][3] is slots
    assert calls[1][2] is None                       # no block table: the step's own k/v
    assert calls[1][1].shape == (5, 2, 16)


def test_prefix_prefill_reads_the_cache(calls):
    layer = _layer()
    q, k, v = _qkv(3)
    bt = torch.zeros(1, 4, dtype=torch.int32)
    ctx = at.AttentionContext(is_prefill=True, slot_mapping=torch.arange(3, dtype=torch.int64),
                              cu_seqlens_q=torch.tensor([0, 3]), cu_seqlens_k=torch.tensor([0, 40]),
                              max_seqlen_q=3, max_seqlen_k=40, block_tables=bt)
    layer(q, k, v, ctx)
    assert [c[0] for c in calls] == ["store", "varlen"]
    assert calls[1][1] is layer.k_cache and calls[1][2] is bt


def test_decode_reads_the_cache_after_the_store(calls):
    layer = _layer()
    q, k, v = _qkv(2)
    lens = torch.tensor([9, 17], dtype=torch.int32)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    ctx = at.AttentionContext(is_prefill=False, slot_mapping=torch.tensor([8, 32]), context_lens=lens,
                              block_tables=bt, max_seqlen_k=17)
    o = layer(q, k, v, ctx)
    assert o.shape == q.shape
    assert [c[0] for c in calls] == ["store", "decode"]
    assert calls[1][1] is layer.k_cache and calls[1][2] is lens and calls[1][3] is bt and calls[1][4] == 17


def test_decode_without_cache_is_refused(calls):
    layer = _layer(cache=False)
    q, k, v = _qkv(1)
    with pytest.raises(ValueError):
        layer(q, k, v, at.AttentionContext(is_prefill=False, context_lens=torch.tensor([1]),
                                           block_tables=torch.zeros(1, 1, dtype=torch.int32)))
    with pytest.raises(ValueError):
        at.Attention(num_heads=6, head_dim=16, scale=1.0, num_kv_heads=4)


def test_multi_token_decode_goes_through_the_kvcache_entry(calls):
    layer = _layer()
    q, k, v = _qkv(6)                               # 2 sequences x 3 new tokens
    lens = torch.tensor([9, 17], dtype=torch.int32)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    ctx = at.AttentionContext(is_prefill=False, slot_mapping=torch.arange(6), context_lens=lens, block_tables=bt,
                              max_seqlen_k=17)
    o = layer(q, k, v, ctx)
    assert o.shape == q.shape
    assert [c[0] for c in calls] == ["store", "kvcache"]
    assert calls[1][1] == (2, 3, 8, 16) and calls[1][2] is lens and calls[1][3] is bt
    assert calls[1][4] is True and calls[1][5] == 17
    with pytest.raises(ValueError):                 # 5 tokens over 2 sequences
        q5, k5, v5 = _qkv(5)
        layer(q5, k5, v5, ctx)



def test_v16_cache_is_filled_by_the_store_and_read_by_the_prefix_prefill(calls):
    layer = _layer()
    layer.v16_cache = torch.zeros(4, 16, 2, 16, dtype=torch.float16)
    q, k, v = _qkv(5)
    bt = torch.zeros(1, 4, dtype=torch.int32)
    ctx = at.AttentionContext(True, slot_mapping=torch.arange(5), cu_seqlens_q=torch.tensor([0, 5]),
                              cu_seqlens_k=torch.tensor([0, 9]), max_seqlen_q=5, max_seqlen_k=9, block_tables=bt)
    layer(q, k, v, ctx)
    assert [c[0] for c in calls] == ["store", "varlen"]
    assert calls[0][4] is layer.v16_cache
    assert calls[1][5] is layer.v16_cache and calls[1][1] is layer.k_cache
