"""Paged decode on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def poison_tail(cfg, kc, vc):
    """Fill the cache rows past each sequence's end inside its last block with NaN."""
    bs = cfg.block_size
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=kc.device)
    for b in range(cfg.batch):
        L = int(cfg.lens_k[b])
        if L % bs:
            pb = int(cfg.block_table[b, L // bs])
            kc[pb, L % bs:] = nan
            vc[pb, L % bs:] = nan


def device_cache(cfg, poison=True):
    kc = torch.full((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), float("nan"), dtype=torch.bfloat16,
                    device="cuda")
    vc = torch.full_like(kc, float("nan"))
    workloads.fill_paged_cache(cfg, kc, vc)
    if poison:
        poison_tail(cfg, kc, vc)
    return kc, vc


def oracle_decode(cfg, q, seqs=None):
    seqs = list(range(cfg.batch)) if seqs is None else list(seqs)
    kp, vp, bt = workloads.compact_paged(cfg, seqs)
    return oracle.decode_paged(q[seqs], kp, vp, cfg.ctx[seqs], bt, cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size,
                               kp.shape[0], cfg.scale)


CASES = [
    # seed, lens, Hq, Hkv, D, block_size, num_splits
    (1, [1, 63, 64, 65], 32, 8, 128, 16, 0),
    (2, [300, 1000, 2049], 32, 8, 128, 256, 0),
    (3, [300, 1000, 2049], 32, 8, 128, 256, 1),
    (4, [300, 1000, 2049], 32, 8, 128, 256, 7),
    (5, [0, 77, 1], 8, 8, 128, 32, 0),
    (6, [5, 129, 4096, 700, 33], 16, 2, 64, 64, 0),
    (7, [1000, 513], 4, 4, 128, 128, 3),
    (8, [4097, 31, 2500], 24, 8, 128, 16, 0),
    (9, [300, 2000, 1], 32, 2, 128, 16, 0),     # 16 query heads per KV head: two n8 column tiles
    (10, [700, 65], 48, 3, 64, 32, 5),
    (11, [900, 40, 3000], 64, 2, 128, 64, 0),   # 32 query heads per KV head: two column groups
    (12, [257, 1200], 64, 1, 64, 16, 4),        # 64 heads on one KV head: four column groups
]


@pytest.mark.parametrize("seed,lens,Hq,Hkv,D,bs,splits", CASES)
def test_decode_matches_oracle(seed, lens, Hq, Hkv, D, bs, splits):
    cfg = workloads.small_paged(seed, ctx=lens, new=[0] * len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                                decode=True)
    q = cfg.q()
    kc, vc = device_cache(cfg)
    av.get_last_device_error()
    out, lse = av.attn_decode_paged(q.cuda(), kc, vc, torch.from_numpy(cfg.ctx.astype(np.int32)).cuda(),
                                    torch.from_numpy(cfg.block_table).cuda(), cfg.scale, num_splits=splits,
                                    return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle_decode(cfg, q)
    assert_close(out, ref, f"decode {lens}")
    assert_lse_close(lse, ref_lse, "decode lse")


def test_decode_page_permutation_is_bitexact():
    """The same logical cache under another physical placement gives the same bits."""
    cfg = workloads.small_paged(11, ctx=[900, 1500, 64], new=[0, 0, 0], Hq=32, Hkv=8, D=128, block_size=64,
                                decode=True, extra_blocks=7)
    q = cfg.q().cuda()
    kc, vc = device_cache(cfg, poison=False)
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    o1 = av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, num_splits=4)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(cfg.num_blocks)).cuda()
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    o2 = av.attn_decode_paged(q, kc2, vc2, cs, bt2, cfg.scale, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_decode_split_counts_agree():
    cfg = workloads.small_paged(12, ctx=[3000, 5000], new=[0, 0], Hq=32, Hkv=8, D=128, block_size=256, decode=True)
    q = cfg.q().cuda()
    kc, vc = device_cache(cfg)
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    ref, _ = oracle_decode(cfg, cfg.q())
    for s in (1, 2, 5, 16, 0):
        assert_close(av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, num_splits=s), ref, f"splits={s}")


def test_decode_bad_block_id_is_flagged():
    cfg = workloads.small_paged(13, ctx=[300], new=[0], Hq=8, Hkv=8, D=128, block_size=64, decode=True)
    kc, vc = device_cache(cfg)
    bt = torch.from_numpy(cfg.block_table).cuda()
    bt[0, 1] = cfg.num_blocks + 5
    av.get_last_device_error()
    out = av.attn_decode_paged(cfg.q().cuda(), kc, vc, torch.tensor([300], dtype=torch.int32, device="cuda"), bt,
                               cfg.scale)
    st, word = av.get_last_device_error()
    assert st == 6
    assert torch.isfinite(out.float()).all()


@pytest.mark.slow
def test_decode_c4_full_size_sampled():
    """The 256-sequence workload at full size; the oracle checks 12 sequences."""
    cfg = workloads.make("c4_decode")
    q = cfg.q()
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    poison_tail(cfg, kc, vc)
    out, lse = av.attn_decode_paged(q.cuda(), kc, vc, torch.from_numpy(cfg.ctx.astype(np.int32)).cuda(),
                                    torch.from_numpy(cfg.block_table).cuda(), cfg.scale,
                                    max_cache_seqlen=int(cfg.ctx.max()), return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    seqs = sorted(np.random.default_rng(44).choice(cfg.batch, 12, replace=False).tolist())
    seqs = sorted(set(seqs) | {int(np.argmax(cfg.ctx)), int(np.argmin(cfg.ctx))})
    ref, ref_lse = oracle_decode(cfg, q, seqs)
    assert_close(out[seqs], ref, "c4 decode")
    assert_lse_close(lse[seqs], ref_lse, "c4 decode lse")
    del kc, vc
    torch.cuda.empty_cache()
