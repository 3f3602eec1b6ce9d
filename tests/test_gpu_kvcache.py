"""attn_with_kvcache (several new tokens per sequence against the paged cache)
on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import workloads
from _util import assert_close, assert_lse_close
from test_gpu_prefill import _paged_device, _paged_oracle, _run_paged

pytestmark = pytest.mark.gpu

CASES = [
    # seed, ctx, Sq, Hq, Hkv, D, block_size
    (61, [37, 5, 300], 1, 32, 8, 128, 16),
    (62, [1000, 257, 0], 2, 32, 8, 128, 256),
    (63, [511, 2048], 7, 8, 8, 128, 64),
    (64, [90, 700, 1], 64, 16, 2, 64, 32),
    (65, [3000, 129], 130, 32, 8, 128, 128),
]


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
    """The kv-cache entry only derives cu_seqlens on the device; the attention is
    the paged varlen path, bit for bit."""
    cfg = workloads.small_paged(66, ctx=[700, 90, 1500], new=[5, 5, 5], Hq=32, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    out_k, lse_k = av.attn_with_kvcache(q.cuda().view(cfg.batch, 5, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                                        max_cache_seqlen=int(cfg.lens_k.max()), return_lse=True)
    out_v, lse_v = _run_paged(cfg, q, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(out_k.view(-1, cfg.Hq, cfg.D).view(torch.int16), out_v.view(torch.int16))
    assert torch.equal(lse_k, lse_v)


def test_kvcache_seqlen_above_stated_max_is_reported():
    """A cache_seqlens entry above max_cache_seqlen is clamped and reported, not read past."""
    cfg = workloads.small_paged(67, ctx=[300, 40], new=[4, 4], Hq=8, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    cs, bt = _as_kvcache_args(cfg, kc, vc)
    av.get_last_device_error()
    av.attn_with_kvcache(q.cuda().view(cfg.batch, 4, cfg.Hq, cfg.D), kc, vc, cs, bt, cfg.scale,
                         max_cache_seqlen=100)
    torch.cuda.synchronize()
    st, word = av.get_last_device_error()
    assert st == 6, (st, hex(word))   # ATTN_ERR_DEVICE_INDEX
