"""attn_with_kvcache (several new tokens per sequence against the paged cache)
on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close, assert_lse_close
from test_gpu_prefill import _paged_device, _paged_oracle, _run_paged, v16_of

pytestmark = pytest.mark.gpu

CASES = [
    # seed, ctx, Sq, Hq, Hkv, D, block_size
    # Sq x G <= 16 query rows per KV head (<= 64 at head_dim 64): the split-KV decode kernel
    (61, [37, 5, 300], 1, 32, 8, 128, 16),
    (62, [1000, 257, 0], 2, 32, 8, 128, 256),
    (63, [511, 2048], 7, 8, 8, 128, 64),
    (68, [254, 3, 1900, 126], 4, 32, 8, 128, 16),    # two n8 column tiles; causal ends straddle split edges
    (69, [30, 1000, 0], 16, 16, 16, 64, 32),         # G = 1, sixteen new tokens
    (70, [500, 77], 2, 64, 8, 128, 64),              # G = 8
    (71, [1200, 5, 64], 1, 32, 2, 128, 16),          # G = 16, one token
    (72, [64, 0, 191], 3, 16, 4, 64, 16),            # twelve live columns of sixteen
    (77, [300, 1500, 7], 8, 32, 8, 128, 64),         # 32 rows at head_dim 128: the one-slot prefill
    (78, [129, 640], 5, 64, 8, 64, 16),              # 40 columns at head_dim 64: three groups, the last one half full
    (79, [2000, 33], 64, 8, 8, 64, 32),              # G = 1, 64 new tokens: four groups
    (80, [400, 1300], 8, 24, 8, 128, 64),            # G = 3, 24 rows: the one-slot prefill (42-token slots)
    # larger Sq x G: the paged varlen prefill (at head_dim 128 up to 128 rows: one slot, V converted in the kernel)
    (81, [129, 640, 3000], 5, 64, 8, 128, 16),       # 40 columns
    (82, [2000, 17, 0, 900], 16, 32, 8, 128, 64),    # 64 columns
    (64, [90, 700, 1], 64, 16, 2, 64, 32),
    (65, [3000, 129], 130, 32, 8, 128, 128),
    (73, [400, 20], 17, 32, 8, 128, 64),
]


@pytest.mark.parametrize("seed,ctx,Sq,Hq,Hkv,D,bs", CASES)
def test_kvcache_with_v16_cache_matches_oracle(seed, ctx, Sq, Hq, Hkv, D, bs):
    """The same calls reading the fp16 V / 16 cache (NaN past every sequence's end):
    the decode route multiplies it by fp16 16 P, the prefill route skips its
    conversion; both against the oracle."""
    cfg = workloads.small_paged(seed, ctx=ctx, new=[Sq] * len(ctx), Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    out, lse = av.attn_with_kvcache(q.cuda().view(cfg.batch, Sq, Hq, D), kc, vc, cs, bt, cfg.scale,
                                    return_lse=True, v16_cache=v16_of(vc))
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out.view(-1, Hq, D), ref.reshape(-1, Hq, D), f"kvcache v16 Sq={Sq}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "kvcache v16 lse")


def _as_kvcache_args(cfg, kc, vc):
    cs = torch.from_numpy(cfg.lens_k.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    return cs, bt


@pytest.mark.parametrize("seed,ctx,Sq,Hq,Hkv,D,bs", CASES)
def test_kvcache_matches_oracle(seed, ctx, Sq, Hq, Hkv, D, bs):
    cfg = workloads.small_paged(seed, ctx=ctx, new=[Sq] * len(ctx), Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    out, lse = av.attn_with_kvcache(q.cuda().view(cfg.batch, Sq, Hq, D), kc, vc, cs, bt, cfg.scale,
                                    return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out.view(-1, Hq, D), ref.reshape(-1, Hq, D), f"kvcache Sq={Sq}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "kvcache lse")


def test_kvcache_equals_paged_varlen_bitexact():
    """Past 64 query columns per KV head (17 tokens x 4 heads) the kv-cache entry
    only derives cu_seqlens on the device; the attention is the paged varlen path,
    bit for bit."""
    cfg = workloads.small_paged(66, ctx=[700, 90, 1500], new=[17, 17, 17], Hq=32, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    out_k, lse_k = av.attn_with_kvcache(q.cuda().view(cfg.batch, 17, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                                        max_cache_seqlen=int(cfg.lens_k.max()), return_lse=True)
    out_v, lse_v = _run_paged(cfg, q, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(out_k.view(-1, cfg.Hq, cfg.D).view(torch.int16), out_v.view(torch.int16))
    assert torch.equal(lse_k, lse_v)
    # the prefill route with the fp16 V / 16 cache: same bits
    out_h, lse_h = av.attn_with_kvcache(q.cuda().view(cfg.batch, 17, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                                        max_cache_seqlen=int(cfg.lens_k.max()), return_lse=True,
                                        v16_cache=v16_of(vc))
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(out_h.view(torch.int16), out_k.view(torch.int16))
    assert torch.equal(lse_h, lse_k)


def test_kvcache_v16_past_one_column_group_runs_the_paged_prefill_bitexact():
    """With the fp16 V / 16 cache, more than 16 query columns per KV head (8 tokens x
    4 heads) go to the paged varlen prefill: the kv-cache entry equals
    attn_varlen_fwd on the same caches bit for bit, and the oracle."""
    cfg = workloads.small_paged(67, ctx=[900, 64, 2100, 8], new=[8, 8, 8, 8], Hq=32, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    v16 = v16_of(vc)
    out_k, lse_k = av.attn_with_kvcache(q.cuda().view(cfg.batch, 8, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                                        max_cache_seqlen=int(cfg.lens_k.max()), return_lse=True, v16_cache=v16)
    out_v, lse_v = _run_paged(cfg, q, kc, vc, v16=v16)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(out_k.view(-1, cfg.Hq, cfg.D).view(torch.int16), out_v.view(torch.int16))
    assert torch.equal(lse_k, lse_v)
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out_k.view(-1, cfg.Hq, cfg.D), ref.reshape(-1, cfg.Hq, cfg.D), "kvcache v16 8 tokens (prefill route)")
    assert_lse_close(lse_k.t().contiguous(), ref_lse.reshape(-1, cfg.Hq), "kvcache v16 8 tokens lse (prefill route)")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Hq,Hkv,D", [(4, 16, 4, 128), (2, 8, 8, 64), (9, 16, 8, 128), (17, 32, 8, 128)])
def test_kvcache_causal_flag(causal, Sq, Hq, Hkv, D):
    """causal=False lets every new token see all cached keys (decode kernel and prefill route)."""
    cfg = workloads.small_paged(74 + Sq, ctx=[300, 64, 5], new=[Sq] * 3, Hq=Hq, Hkv=Hkv, D=D, block_size=32)
    q = cfg.q()
    kc, vc, k_new, v_new = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    av.get_last_device_error()
    out, lse = av.attn_with_kvcache(q.cuda().view(cfg.batch, Sq, Hq, D), kc, vc, cs, bt, cfg.scale,
                                    causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)), causal=causal)
    assert_close(out.view(-1, Hq, D), ref.reshape(-1, Hq, D), f"kvcache causal={causal} Sq={Sq}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "kvcache lse")


@pytest.mark.parametrize("Sq,Hq,Hkv", [(4, 16, 4), (6, 8, 8), (4, 64, 8), (17, 32, 8)])
def test_kvcache_fewer_keys_than_new_tokens(Sq, Hq, Hkv):
    """cache_seqlens[b] < seqlen_q: the first new tokens see no key at all (output
    0, lse -inf) and the rest see a causal prefix of the keys."""
    cfg = workloads.small_paged(80 + Sq, ctx=[0, 150], new=[Sq, Sq], Hq=Hq, Hkv=Hkv, D=128, block_size=16)
    q = cfg.q()
    kc, vc, k_new, v_new = _paged_device(cfg)
    lens = [2, 150 + Sq]
    cs = torch.tensor(lens, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(cfg.block_table).cuda()
    av.get_last_device_error()
    out, lse = av.attn_with_kvcache(q.cuda().view(cfg.batch, Sq, Hq, 128), kc, vc, cs, bt, cfg.scale,
                                    return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, [0, 1], lens_k=lens)
    o = out.view(-1, Hq, 128)
    n_empty = Sq - lens[0]            # token t sees keys j <= L - Sq + t: none for t < Sq - L
    assert torch.equal(o[:n_empty].float().cpu(), torch.zeros(n_empty, Hq, 128))
    assert torch.isneginf(lse.t()[:n_empty]).all()
    assert_close(o, ref.reshape(-1, Hq, 128), f"kvcache short Sq={Sq}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "kvcache short lse")


def test_kvcache_one_token_equals_decode_bitexact():
    """With seqlen_q = 1 the kv-cache entry runs the decode kernel on the same
    split plan as attn_decode_paged: outputs agree bit for bit, lse transposed."""
    cfg = workloads.small_paged(76, ctx=[700, 90, 1500, 3], new=[1] * 4, Hq=32, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    mx = int(cfg.lens_k.max())
    out_k, lse_k = av.attn_with_kvcache(q.cuda().view(cfg.batch, 1, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                                        max_cache_seqlen=mx, return_lse=True)
    out_d, lse_d = av.attn_decode_paged(q.cuda(), kc, vc, cs, bt, cfg.scale, max_cache_seqlen=mx,
                                        return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out_k.view(-1, cfg.Hq, cfg.D).view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(lse_k, lse_d.t())


@pytest.mark.parametrize("Sq,Hq,Hkv", [(4, 8, 8), (4, 64, 8), (17, 32, 8)])
def test_kvcache_seqlen_above_stated_max_is_reported(Sq, Hq, Hkv):
    """A cache_seqlens entry above max_cache_seqlen is clamped and reported, not
    read past (Sq x G = 4 and 32: decode kernel; 68: prefill route)."""
    cfg = workloads.small_paged(67, ctx=[300, 40], new=[Sq, Sq], Hq=Hq, Hkv=Hkv, D=128, block_size=64)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    av.get_last_device_error()
    av.attn_with_kvcache(q.cuda().view(cfg.batch, Sq, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                         max_cache_seqlen=100)
    torch.cuda.synchronize()
    st, word = av.get_last_device_error()
    assert st == 6, (st, hex(word))   # ATTN_ERR_DEVICE_INDEX


def test_kvcache_c4_four_tokens_full_size_sampled():
    """The 4-token kv-cache step at full size (the 256-sequence decode cache; the
    last 4 cached tokens of every sequence are its new ones), in the launch
    configuration the benchmark times; the oracle checks 12 sequences (every
    new token and head)."""
    from test_gpu_decode import poison_tail
    cfg = workloads.make("c4_decode")
    Sq = 4
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    poison_tail(cfg, kc, vc)
    rng = np.random.default_rng(4321)
    q4 = torch.from_numpy(rng.standard_normal((cfg.batch, Sq, cfg.Hq, cfg.D), dtype=np.float32)).to(torch.bfloat16)
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    av.get_last_device_error()
    out, lse = av.attn_with_kvcache(q4.cuda(), kc, vc, cs, bt, cfg.scale, max_cache_seqlen=int(cfg.ctx.max()),
                                    return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    seqs = sorted(np.random.default_rng(45).choice(cfg.batch, 10, replace=False).tolist())
    seqs = sorted(set(seqs) | {int(np.argmax(cfg.ctx)), int(np.argmin(cfg.ctx))})
    kp, vp, btc = workloads.compact_paged(cfg, seqs)
    cu_q = workloads.cu_from_lens(np.full(len(seqs), Sq, dtype=np.int64))
    cu_k = workloads.cu_from_lens(cfg.ctx[seqs])
    ref, ref_lse = oracle.attn_varlen(q4[seqs].reshape(-1, cfg.Hq, cfg.D), kp, vp, cu_q, cu_k, cfg.Hq, cfg.Hkv,
                                      cfg.D, cfg.scale, True, block_table=btc, block_size=cfg.block_size,
                                      num_blocks=kp.shape[0])
    assert_close(out[seqs].reshape(-1, cfg.Hq, cfg.D), ref.reshape(-1, cfg.Hq, cfg.D), "c4 cache, 4 new tokens")
    got_lse = lse.view(cfg.Hq, cfg.batch, Sq)[:, seqs].reshape(cfg.Hq, -1).t().contiguous()
    assert_lse_close(got_lse, ref_lse.reshape(-1, cfg.Hq), "c4 cache, 4 new tokens, lse")
    del kc, vc
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("use16", [False, True])
def test_kvcache_c4_eight_tokens_full_size_sampled(use16):
    """The 8-token kv-cache step at full size (32 query columns per KV head), as
    the benchmark times it: without the fp16 V / 16 cache on the decode kernel in
    two column-group CTAs, with it on the paged prefill; the oracle checks 12
    sequences."""
    from test_gpu_decode import poison_tail
    cfg = workloads.make("c4_decode")
    Sq = 8
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    poison_tail(cfg, kc, vc)
    v16 = v16_of(vc) if use16 else None
    rng = np.random.default_rng(8642)
    q8 = torch.from_numpy(rng.standard_normal((cfg.batch, Sq, cfg.Hq, cfg.D), dtype=np.float32)).to(torch.bfloat16)
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    av.get_last_device_error()
    out, lse = av.attn_with_kvcache(q8.cuda(), kc, vc, cs, bt, cfg.scale, max_cache_seqlen=int(cfg.ctx.max()),
                                    return_lse=True, v16_cache=v16)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    seqs = sorted(np.random.default_rng(46).choice(cfg.batch, 10, replace=False).tolist())
    seqs = sorted(set(seqs) | {int(np.argmax(cfg.ctx)), int(np.argmin(cfg.ctx))})
    kp, vp, btc = workloads.compact_paged(cfg, seqs)
    cu_q = workloads.cu_from_lens(np.full(len(seqs), Sq, dtype=np.int64))
    cu_k = workloads.cu_from_lens(cfg.ctx[seqs])
    ref, ref_lse = oracle.attn_varlen(q8[seqs].reshape(-1, cfg.Hq, cfg.D), kp, vp, cu_q, cu_k, cfg.Hq, cfg.Hkv,
                                      cfg.D, cfg.scale, True, block_table=btc, block_size=cfg.block_size,
                                      num_blocks=kp.shape[0])
    what = "c4 cache, 8 new tokens" + (", v16" if use16 else "")
    assert_close(out[seqs].reshape(-1, cfg.Hq, cfg.D), ref.reshape(-1, cfg.Hq, cfg.D), what)
    got_lse = lse.view(cfg.Hq, cfg.batch, Sq)[:, seqs].reshape(cfg.Hq, -1).t().contiguous()
    assert_lse_close(got_lse, ref_lse.reshape(-1, cfg.Hq), what + ", lse")
    del kc, vc, v16
    torch.cuda.empty_cache()
