"""Varlen prefill (contiguous and paged) on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close, assert_lse_close
from test_gpu_decode import device_cache, poison_tail

pytestmark = pytest.mark.gpu


def run_contig(cfg, q, k, v, causal=True):
    cu_q = torch.from_numpy(cfg.cu_q).cuda()
    cu_k = torch.from_numpy(cfg.cu_k).cuda()
    return av.attn_varlen_fwd(q.cuda() if not q.is_cuda else q, k.cuda() if not k.is_cuda else k,
                              v.cuda() if not v.is_cuda else v, cu_q, cu_k, int(cfg.lens_q.max(initial=0)),
                              int(cfg.lens_k.max(initial=0)), cfg.scale, causal=causal, return_lse=True)


def check_rows(out, lse, ref, ref_lse, rows, Hq, what):
    D = out.shape[-1]
    got = out.reshape(-1, D)[torch.from_numpy(rows).cuda()]
    assert_close(got, ref, what)
    t, h = rows // Hq, rows % Hq
    assert_lse_close(lse[torch.from_numpy(h).cuda(), torch.from_numpy(t).cuda()], ref_lse, what + " lse")


def test_c1_article_example_full():
    cfg = workloads.make("c1_tiny")
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    av.get_last_device_error()
    out, lse = run_contig(cfg, q, k, v)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 4, 4, 64, cfg.scale, True)
    assert_close(out, ref.reshape(out.shape), "c1")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, 4), "c1 lse")


VARLEN_CASES = [
    # seed, lens_q, lens_k, Hq, Hkv, D, causal
    (1, [5, 2, 1], [9, 7, 3], 4, 4, 64, True),
    (2, [1, 17, 128, 129, 300], [1, 17, 128, 129, 300], 8, 2, 128, True),
    (3, [200, 33], [500, 40], 32, 8, 128, True),
    (4, [64, 257], [30, 100], 4, 4, 64, True),
    (5, [0, 100, 0, 3], [5, 100, 0, 3], 16, 2, 128, True),
    (6, [130, 77], [130, 300], 8, 1, 128, False),
    (7, [512, 1000], [512, 1000], 2, 2, 128, True),
    (8, [256], [256], 32, 2, 128, True),
    (9, [700, 45], [700, 45], 32, 8, 64, True),
    (10, [1, 1, 1], [1, 2, 1000], 8, 8, 128, True),
    # groups that do not divide 128: a slot holds 128 // G tokens (126, 125, 126, 96 rows);
    # the rows past them are never stored, and a warp's rows are written row by row
    (11, [1, 42, 43, 300, 85], [1, 42, 43, 300, 90], 24, 8, 128, True),   # G = 3: 42 tokens
    (12, [100, 126, 7, 0], [250, 126, 7, 4], 10, 2, 64, True),             # G = 5: 25 tokens
    (13, [50, 200], [50, 260], 12, 2, 128, False),                          # G = 6: 21 tokens
    (14, [36, 19, 250], [36, 40, 250], 28, 4, 128, True),                   # G = 7: 18 tokens
    (15, [5, 3, 2], [5, 100, 2], 48, 1, 64, True),                          # G = 48: 2 tokens
    (16, [3, 2], [40, 2], 96, 1, 128, True),                                # G = 96: 1 token
]


@pytest.mark.parametrize("seed,lq,lk,Hq,Hkv,D,causal", VARLEN_CASES)
def test_varlen_matches_oracle(seed, lq, lk, Hq, Hkv, D, causal):
    cfg = workloads.small_varlen(seed, lq, lk, Hq, Hkv, D, causal)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    av.get_last_device_error()
    out, lse = run_contig(cfg, q, k, v, causal)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, Hq, Hkv, D, cfg.scale, causal)
    if ref.size:
        assert_close(out, ref.reshape(out.shape), f"varlen {lq}/{lk}")
        assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "varlen lse")


SHORT_Q_CASES = [
    # a few queries per sequence (each <= 128 / G, one query slot) against longer
    # keys: one key tile, odd and even tile counts, rows that see no key (Lq > Lk,
    # causal), an empty sequence
    (96, [1, 5, 32, 0, 17, 32, 9], [1, 130, 4000, 0, 17, 257, 3], 32, 8, 128),
    (97, [64, 3, 64, 1], [64, 640, 1000, 2048], 16, 8, 64),
    (98, [8, 8, 8], [2049, 100, 7000], 32, 8, 128),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed,lq,lk,Hq,Hkv,D", SHORT_Q_CASES)
def test_short_queries_against_long_keys_match_oracle(seed, lq, lk, Hq, Hkv, D, causal):
    """Decode-like varlen calls: every unit has a single active query slot."""
    cfg = workloads.small_varlen(seed, lq, lk, Hq, Hkv, D, causal)
    assert max(lq) * (Hq // Hkv) <= 128
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    av.get_last_device_error()
    out, lse = run_contig(cfg, q, k, v, causal)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, Hq, Hkv, D, cfg.scale, causal)
    assert_close(out, ref.reshape(out.shape), f"short-q varlen {lq}/{lk}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "short-q varlen lse")


def test_unit_order_does_not_change_the_result():
    """Short key ranges take the next unit a whole unit ahead, long ones later: the
    same inputs with max_seqlen_k at the true maximum (1900) and raised past that
    threshold (5000) run the two forms; each unit's result does not depend on
    which CTA computes it or when, so the outputs agree bit for bit."""
    cfg = workloads.small_varlen(95, [300, 1900, 40, 700, 1], [300, 1900, 40, 700, 1], 32, 8, 128, True)
    q, k, v = cfg.q().cuda(), cfg.k().cuda(), cfg.v().cuda()
    cu_q, cu_k = torch.from_numpy(cfg.cu_q).cuda(), torch.from_numpy(cfg.cu_k).cuda()
    av.get_last_device_error()
    o1, l1 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 1900, 1900, cfg.scale, causal=True, return_lse=True)
    o2, l2 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 1900, 5000, cfg.scale, causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_one_pair_launch_takes_units_early_bitexact():
    """With every sequence one query pair the next unit is taken a unit ahead even
    for long keys (a unit has no siblings to share K/V with); raising max_seqlen_q
    past one pair runs the other form on the same units: bit-identical.  With
    max_seqlen_q within one query slot (8 <= 128 / G) slot B's softmax warps share
    slot A's key tiles: its row sums add in another order, so that form is checked
    against the oracle and within a bf16 ulp of the others."""
    lq, lk = [8, 8, 8, 8, 8], [6000, 4500, 130, 5000, 8]
    cfg = workloads.small_varlen(97, lq, lk, 32, 8, 128, True)
    q, k, v = cfg.q().cuda(), cfg.k().cuda(), cfg.v().cuda()
    cu_q, cu_k = torch.from_numpy(cfg.cu_q).cuda(), torch.from_numpy(cfg.cu_k).cuda()
    av.get_last_device_error()
    o1, l1 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 64, 6000, cfg.scale, causal=True, return_lse=True)
    o2, l2 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 200, 6000, cfg.scale, causal=True, return_lse=True)
    o3, l3 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 8, 6000, cfg.scale, causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    ref, ref_lse = oracle.attn_varlen(cfg.q(), cfg.k(), cfg.v(), cfg.cu_q, cfg.cu_k, 32, 8, 128, cfg.scale, True)
    for o, lse, what in ((o1, l1, "one-pair launch"), (o3, l3, "one-slot launch")):
        assert_close(o, ref.reshape(o.shape), what)
        assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, 32), what + " lse")
    d = (o3.float() - o1.float()).abs()
    assert bool((d <= 2.0 ** -7 * o1.float().abs() + 1e-6).all())


ONE_SLOT_CASES = [
    # seed, lens_q, lens_k, Hq, Hkv, causal: every sequence within one 128-row slot (Lq <= 128 / G)
    (71, [128, 1, 0, 77], [900, 1, 5, 77], 16, 16, False),   # MHA: 128 tokens per slot, non-causal
    (72, [128, 60, 3], [128, 2000, 3], 8, 8, True),
    (73, [16, 9, 1, 16], [4000, 9, 300, 17], 32, 4, True),    # G = 8: 16 tokens per slot
    (74, [32, 31, 5], [32, 600, 6000], 32, 8, False),
    (75, [25, 3, 0, 25], [25, 900, 0, 4000], 40, 8, True),   # G = 5: 25 tokens, 125 of 128 rows
]


@pytest.mark.parametrize("seed,lq,lk,Hq,Hkv,causal", ONE_SLOT_CASES)
def test_one_slot_instance_matches_oracle(seed, lq, lk, Hq, Hkv, causal):
    """Launches whose sequences all fit one query slot run the instance in which
    slot B's softmax warps take half of each of slot A's key tiles (the row max and
    row sum exchanged between the two halves).  Against the oracle, and within a
    bf16 ulp of the two-slot kernel (max_seqlen_q raised past one slot)."""
    D = 128
    cfg = workloads.small_varlen(seed, lq, lk, Hq, Hkv, D, causal)
    q, k, v = cfg.q().cuda(), cfg.k().cuda(), cfg.v().cuda()
    cu_q, cu_k = torch.from_numpy(cfg.cu_q).cuda(), torch.from_numpy(cfg.cu_k).cuda()
    mq, mk = int(cfg.lens_q.max()), int(cfg.lens_k.max())
    assert mq <= 128 // (Hq // Hkv)
    av.get_last_device_error()
    o1, l1 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, mq, mk, cfg.scale, causal=causal, return_lse=True)
    o2, l2 = av.attn_varlen_fwd(q, k, v, cu_q, cu_k, 300, mk, cfg.scale, causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle.attn_varlen(cfg.q(), cfg.k(), cfg.v(), cfg.cu_q, cfg.cu_k, Hq, Hkv, D, cfg.scale, causal)
    what = f"one-slot s{seed} Hq{Hq}/{Hkv} causal={causal} {lq}/{lk}"
    assert_close(o1, ref.reshape(o1.shape), what)
    assert_lse_close(l1.t().contiguous(), ref_lse.reshape(-1, Hq), what + " lse")
    d = (o1.float() - o2.float()).abs()
    assert bool((d <= 2.0 ** -7 * o2.float().abs() + 1e-6).all()), what + ": differs from the two-slot kernel"


def test_one_slot_instance_paged_v16_cache():
    """The one-slot instance on the paged cache with the fp16 V / 16 cache (the kv-cache
    route's case): a few new tokens per sequence against long contexts."""
    cfg = workloads.small_paged(75, ctx=[3000, 0, 700, 129], new=[8, 8, 5, 1], Hq=32, Hkv=8, D=128, block_size=64)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    out, lse = _run_paged(cfg, q, kc, vc, v16=v16_of(vc))
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out, ref.reshape(out.shape), "one-slot paged v16")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, 32), "one-slot paged v16 lse")


@pytest.mark.parametrize("lens", [[300, 129], [32, 7, 20]])
def test_varlen_strided_qkv_views(lens):
    """q, k, v as views of one packed [tokens, Hq + 2 Hkv, D] projection (two query
    slots with the conversion pass; one slot, V tiles converted in the kernel)."""
    lens = np.array(lens)
    Hq, Hkv, D = 16, 4, 128
    T = int(lens.sum())
    qkv = workloads.normal_bf16((21, 1), T, (Hq + 2 * Hkv) * D).view(T, Hq + 2 * Hkv, D)
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    cfg = workloads.small_varlen(21, lens, lens, Hq, Hkv, D)
    qkv_d = qkv.cuda()
    out, lse = run_contig(cfg, qkv_d[:, :Hq], qkv_d[:, Hq:Hq + Hkv], qkv_d[:, Hq + Hkv:])
    ref, _ = oracle.attn_varlen(q.contiguous(), k.contiguous(), v.contiguous(), cfg.cu_q, cfg.cu_k, Hq, Hkv, D,
                                cfg.scale, True)
    assert_close(out, ref.reshape(out.shape), "strided")


def test_varlen_overflow_scaled_heads():
    """Half the heads have Q scaled by 160: logits reach hundreds."""
    hs = np.ones(8, dtype=np.float32)
    hs[:4] = 160.0
    cfg = workloads.small_varlen(22, [1000, 300], [1000, 300], 8, 8, 128, q_head_scale=hs)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    out, lse = run_contig(cfg, q, k, v)
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 8, 8, 128, cfg.scale, True)
    assert np.max(ref_lse) > 300
    assert_close(out, ref.reshape(out.shape), "overflow heads")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, 8), "overflow lse")


def _paged_device(cfg):
    """Caches with drawn context blocks, new tokens stored by store_kvcache,
    rows past each sequence poisoned with NaN."""
    kc, vc = device_cache(cfg, poison=False)
    k_new, v_new = cfg.k_new(), cfg.v_new()
    av.store_kvcache(k_new.cuda(), v_new.cuda(), kc, vc, torch.from_numpy(cfg.slot_mapping()).cuda())
    poison_tail(cfg, kc, vc)
    return kc, vc, k_new, v_new


def _paged_oracle(cfg, q, k_new, v_new, seqs, rows_local=None, causal=True, lens_k=None):
    """Oracle on a compact pool of `seqs` after its own store of the new tokens
    (lens_k: attended keys per sequence of `seqs`, default all cached ones)."""
    kp, vp, bt = workloads.compact_paged(cfg, seqs)
    # slots of the new tokens of `seqs` in the compact pool
    bs = cfg.block_size
    slots, tok_idx = [], []
    cu_new = workloads.cu_from_lens(cfg.new)
    for r, b in enumerate(seqs):
        j = np.arange(int(cfg.ctx[b]), int(cfg.ctx[b] + cfg.new[b]))
        slots.append(bt[r, j // bs].astype(np.int64) * bs + j % bs)
        tok_idx.append(np.arange(cu_new[b], cu_new[b + 1]))
    slots = np.concatenate(slots)
    tok_idx = np.concatenate(tok_idx)
    kb, vb = oracle.store_kvcache(k_new[tok_idx], v_new[tok_idx], kp, vp, slots)
    qs = q[torch.from_numpy(tok_idx)]
    cu_q = workloads.cu_from_lens(cfg.new[seqs])
    cu_k = workloads.cu_from_lens(cfg.lens_k[seqs] if lens_k is None else np.asarray(lens_k, dtype=np.int64))
    ref, ref_lse = oracle.attn_varlen(qs, kb.reshape(kp.shape), vb.reshape(vp.shape), cu_q, cu_k, cfg.Hq, cfg.Hkv,
                                      cfg.D, cfg.scale, causal, block_table=bt, block_size=bs,
                                      num_blocks=kp.shape[0], rows=rows_local)
    return ref, ref_lse, tok_idx


def _run_paged(cfg, q, kc, vc, v16=None):
    cu_q = torch.from_numpy(workloads.cu_from_lens(cfg.new)).cuda()
    cu_k = torch.from_numpy(workloads.cu_from_lens(cfg.lens_k)).cuda()
    return av.attn_varlen_fwd(q.cuda(), kc, vc, cu_q, cu_k, int(cfg.new.max()), int(cfg.lens_k.max()), cfg.scale,
                              causal=True, block_table=torch.from_numpy(cfg.block_table).cuda(), return_lse=True,
                              v16_cache=v16)


def v16_of(vc, blocks=None):
    """An fp16 V / 16 cache for the bf16 cache vc, as store_kvcache keeps it (torch's
    round-to-nearest conversion; NaN stays NaN).  blocks: only these block ids, the
    rest NaN."""
    out = torch.full(vc.shape, float("nan"), dtype=torch.float16, device=vc.device)
    idx = torch.arange(vc.shape[0], device=vc.device) if blocks is None else blocks
    for i in range(0, idx.numel(), 256):
        j = idx[i:i + 256]
        out[j] = (vc[j].float() / 16.0).half()
    return out


PAGED_CASES = [
    # seed, ctx, new, Hq, Hkv, D, block_size
    (31, [37, 5, 300], [6, 1, 90], 32, 8, 128, 16),
    (32, [1000, 257, 0], [200, 1, 64], 32, 8, 128, 256),
    (33, [511, 2048], [129, 3], 8, 8, 128, 64),
    (34, [90, 700], [40, 333], 16, 2, 64, 32),
    (35, [300, 17, 1000], [50, 3, 130], 40, 8, 128, 16),   # G = 5
]


@pytest.mark.parametrize("seed,ctx,new,Hq,Hkv,D,bs", PAGED_CASES)
def test_paged_prefill_v16_cache_is_bitexact(seed, ctx, new, Hq, Hkv, D, bs):
    """Reading V / 16 from an fp16 cache kept beside the bf16 one gives the bits
    of the call that converts V itself; the V' cache rows past every sequence
    hold NaN (they must be zeroed before the P V product)."""
    cfg = workloads.small_paged(seed, ctx=ctx, new=new, Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    v16 = v16_of(vc)
    av.get_last_device_error()
    out_a, lse_a = _run_paged(cfg, q, kc, vc)
    out_b, lse_b = _run_paged(cfg, q, kc, vc, v16)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.isfinite(out_b.float()).all()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)


ONE_SLOT_PAGED_CASES = [
    # seed, ctx, new, Hq, Hkv, block_size: head_dim 128, every sequence's new tokens within one slot
    (36, [37, 900, 0, 300], [8, 8, 8, 1], 32, 8, 16),
    (37, [5000, 129], [32, 3], 32, 8, 64),
    (38, [700, 20, 3000], [25, 25, 2], 40, 8, 256),   # G = 5: 25-token slots
]


@pytest.mark.parametrize("seed,ctx,new,Hq,Hkv,bs", ONE_SLOT_PAGED_CASES)
def test_one_slot_converts_v_in_the_kernel(seed, ctx, new, Hq, Hkv, bs):
    """One-slot launches without a V / 16 cache load each bf16 V tile and convert it
    to V / 16 in shared memory (no conversion pass, no V' copy): the oracle's
    values, and for groups dividing 128 the bits of the call reading the fp16 V / 16
    cache, although the bf16 cache slots past every sequence hold NaN (the converted
    tile's rows past the sequence are zeroed)."""
    cfg = workloads.small_paged(seed, ctx=ctx, new=new, Hq=Hq, Hkv=Hkv, D=128, block_size=bs)
    assert max(new) <= 128 // (Hq // Hkv)
    q = cfg.q()
    kc, vc, k_new, v_new = _paged_device(cfg)
    assert torch.isnan(vc.float()).any()
    av.get_last_device_error()
    out_a, lse_a = _run_paged(cfg, q, kc, vc)
    out_b, lse_b = _run_paged(cfg, q, kc, vc, v16_of(vc))
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out_a, ref.reshape(out_a.shape), f"one-slot in-kernel V' {ctx}+{new}")
    assert_lse_close(lse_a.t().contiguous(), ref_lse.reshape(-1, Hq), "one-slot in-kernel V' lse")
    if 128 % (Hq // Hkv) == 0:
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(lse_a, lse_b)
    else:   # with the V / 16 cache such a group runs the two-slot instance (other row-sum order)
        assert_close(out_b, ref.reshape(out_b.shape), f"one-slot V' cache {ctx}+{new}")


@pytest.mark.parametrize("seed,ctx,new,Hq,Hkv,D,bs", PAGED_CASES)
def test_paged_prefill_matches_oracle(seed, ctx, new, Hq, Hkv, D, bs):
    cfg = workloads.small_paged(seed, ctx=ctx, new=new, Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    out, lse = _run_paged(cfg, q, kc, vc)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    assert_close(out, ref.reshape(out.shape), f"paged {ctx}+{new}")
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), "paged lse")


def test_paged_equals_contiguous_bitexact():
    """Paging is pure addressing: the same K/V, paged or packed, gives the same bits."""
    cfg = workloads.small_paged(41, ctx=[700, 90], new=[300, 60], Hq=32, Hkv=8, D=128, block_size=128)
    q = cfg.q()
    kc, vc, k_new, v_new = _paged_device(cfg)
    out_p, lse_p = _run_paged(cfg, q, kc, vc)
    # gather the logical K/V rows into packed tensors (torch indexing on the device)
    bs = cfg.block_size
    rows = []
    for b in range(cfg.batch):
        j = np.arange(int(cfg.lens_k[b]))
        rows.append(cfg.block_table[b, j // bs].astype(np.int64) * bs + j % bs)
    rows = torch.from_numpy(np.concatenate(rows)).cuda()
    kk = kc.view(-1, cfg.Hkv, cfg.D)[rows].contiguous()
    vv = vc.view(-1, cfg.Hkv, cfg.D)[rows].contiguous()
    cu_q = torch.from_numpy(workloads.cu_from_lens(cfg.new)).cuda()
    cu_k = torch.from_numpy(workloads.cu_from_lens(cfg.lens_k)).cuda()
    out_c, lse_c = av.attn_varlen_fwd(q.cuda(), kk, vv, cu_q, cu_k, int(cfg.new.max()), int(cfg.lens_k.max()),
                                      cfg.scale, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse_p, lse_c)


def test_decode_equals_last_row_of_paged_prefill():
    cfg = workloads.small_paged(42, ctx=[500, 1200], new=[40, 1], Hq=32, Hkv=8, D=128, block_size=256)
    q = cfg.q()
    kc, vc, _, _ = _paged_device(cfg)
    out, _ = _run_paged(cfg, q, kc, vc)
    cu_new = workloads.cu_from_lens(cfg.new)
    last = torch.from_numpy(cu_new[1:] - 1).cuda()
    dec = av.attn_decode_paged(q.cuda()[last], kc, vc, torch.from_numpy(cfg.lens_k.astype(np.int32)).cuda(),
                               torch.from_numpy(cfg.block_table).cuda(), cfg.scale)
    d = (dec.float() - out[last].float()).abs().max().item()
    assert d <= 1e-2


@pytest.mark.slow
def test_c2_full_size_sampled():
    cfg = workloads.make("c2_varlen_gqa")
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    av.get_last_device_error()
    out, lse = run_contig(cfg, q, k, v)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    rows = workloads.sample_rows(cfg.seed, q.shape[0] * cfg.Hq)
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D, cfg.scale, True,
                                      rows=rows)
    check_rows(out, lse, ref, ref_lse, rows, cfg.Hq, "c2")


@pytest.mark.slow
def test_c5_long_overflow_sampled():
    cfg = workloads.make("c5_long")
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    out, lse = run_contig(cfg, q, k, v)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.isfinite(out.float()).all()
    # 4 (sequence, head) pairs: two overflow-stress heads, two plain ones; 1/64 of their rows
    rng = np.random.default_rng(cfg.seed + 5)
    rows = []
    for b, h in [(0, 3), (1, 12), (0, 20), (1, 31)]:
        i = np.sort(rng.choice(32768, 512, replace=False))
        rows.append((int(cfg.cu_q[b]) + i) * cfg.Hq + h)
    rows = np.concatenate(rows).astype(np.int64)
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D, cfg.scale, True,
                                      rows=rows)
    assert np.max(ref_lse) > 500
    check_rows(out, lse, ref, ref_lse, rows, cfg.Hq, "c5")


@pytest.mark.slow
def test_c3_prefix_paged_full_size_sampled():
    cfg = workloads.make("c3_prefix_paged")
    q = cfg.q()
    av.get_last_device_error()
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    k_new, v_new = cfg.k_new(), cfg.v_new()
    av.store_kvcache(k_new.cuda(), v_new.cuda(), kc, vc, torch.from_numpy(cfg.slot_mapping()).cuda())
    poison_tail(cfg, kc, vc)
    out, lse = _run_paged(cfg, q, kc, vc)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    # oracle: 6 sequences (3 of them sharing the prefix), 1/16 of their rows
    seqs = [0, 3, 7, 12, 20, 31]
    Hq = cfg.Hq
    n_local = int(cfg.new[seqs].sum()) * Hq
    rows_local = workloads.sample_rows(cfg.seed, n_local, 1 / 16)
    ref, ref_lse, tok_idx = _paged_oracle(cfg, q, k_new, v_new, seqs, rows_local)
    rows = tok_idx[rows_local // Hq] * Hq + rows_local % Hq
    check_rows(out, lse, ref, ref_lse, rows, Hq, "c3")
    # the same step with the fp16 V / 16 cache (referenced blocks only; the rest NaN)
    used = torch.from_numpy(np.unique(cfg.block_table[cfg.block_table >= 0]).astype(np.int64)).cuda()
    v16 = v16_of(vc, used)
    out16, lse16 = _run_paged(cfg, q, kc, vc, v16)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(out.view(torch.int16), out16.view(torch.int16))
    assert torch.equal(lse, lse16)
    del kc, vc, v16
    torch.cuda.empty_cache()


@pytest.mark.parametrize("vscale", [1e5, 1e-3])
def test_value_scale_of_v(vscale):
    """PV runs in fp16 on 16 P and V / 16: large and small V keep their
    relative accuracy (the metrics are scale-free)."""
    cfg = workloads.small_varlen(52, [300, 77], [300, 77], 8, 2, 128)
    q, k = cfg.q(), cfg.k()
    v = (cfg.v().float() * vscale).to(torch.bfloat16)
    out, lse = run_contig(cfg, q, k, v)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, _ = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 8, 2, 128, cfg.scale, True)
    g = out.float().cpu().double().numpy().reshape(ref.shape)
    rel = np.sqrt(((g - ref) ** 2).sum() / (ref ** 2).sum())
    assert rel <= 2e-3, rel


@pytest.mark.parametrize("L", [100, 300])
def test_v_beyond_fp16_range_is_reported(L):
    """|v| >= 2^20 is clamped and reported: by the one-slot kernel's own conversion
    (100 tokens) and by the conversion pass (300 tokens, two slots)."""
    cfg = workloads.small_varlen(53, [L], [L], 4, 4, 128)
    q, k, v = cfg.q(), cfg.k(), cfg.v().clone()
    v[5, 0, 3] = 3.0e6
    av.get_last_device_error()
    out, _ = run_contig(cfg, q, k, v)
    st, word = av.get_last_device_error()
    assert st == 8 and word & 4
    assert torch.isfinite(out.float()).all()


def test_kernel_event_hook_times_the_attention_kernel_only():
    """attn_set_kernel_events: the span recorded around the attention kernel is
    positive and lies inside the span of the whole call."""
    cfg = workloads.small_varlen(5, [300, 900, 17], [300, 900, 17], 8, 2, 128)
    q, k, v = cfg.q().cuda(), cfg.k().cuda(), cfg.v().cuda()
    run_contig(cfg, q, k, v)   # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    av.set_kernel_events(ka, kb)
    try:
        a.record()
        out, _ = run_contig(cfg, q, k, v)
        b.record()
    finally:
        av.set_kernel_events()
    torch.cuda.synchronize()
    call_ms, kern_ms = a.elapsed_time(b), ka.elapsed_time(kb)
    assert 0.0 < kern_ms <= call_ms
    assert a.elapsed_time(ka) >= 0.0 and kb.elapsed_time(b) >= 0.0
    with pytest.raises(ValueError):
        av.set_kernel_events(ka, None)


def test_paged_prefill_ignores_stale_workspace():
    """With a block table the fp16 V' buffer is sized by an upper bound of the
    key count; a workspace full of NaN bit patterns must not reach the output."""
    cfg = workloads.small_paged(35, ctx=[90, 700, 1], new=[64, 64, 64], Hq=16, Hkv=2, D=64, block_size=32)
    q = cfg.q()
    kc, vc, k_new, v_new = _paged_device(cfg)
    B = cfg.batch
    total_k = B * int(cfg.lens_k.max()) + 300
    ws_bytes = av.lib().attn_varlen_workspace_size(B, cfg.Hq, cfg.Hkv, cfg.D, int(cfg.new.max()), total_k)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    cu_q = torch.from_numpy(workloads.cu_from_lens(cfg.new)).cuda()
    cu_k = torch.from_numpy(workloads.cu_from_lens(cfg.lens_k)).cuda()
    av.get_last_device_error()
    out = av.attn_varlen_fwd(q.cuda(), kc, vc, cu_q, cu_k, int(cfg.new.max()), int(cfg.lens_k.max()), cfg.scale,
                             block_table=torch.from_numpy(cfg.block_table).cuda(), total_k=total_k, workspace=ws)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, _, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(B)))
    assert_close(out, ref.reshape(out.shape), "paged, stale workspace")


@pytest.mark.parametrize("chunks", [1, 3, 8])
def test_host_pipelined_prefill_equals_device_call(chunks):
    """attn_varlen_fwd_host (C entry: host buffers in and out, copies of one
    sequence group overlapped with the attention of another) returns the device
    call's bits, and matches the oracle on sampled rows."""
    cfg = workloads.small_varlen(36, [700, 5, 1300, 64, 129, 900], [700, 5, 1300, 64, 129, 900], 32, 8, 128)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    ref = av.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cfg.cu_q).cuda(),
                             torch.from_numpy(cfg.cu_k).cuda(), 1300, 1300, cfg.scale)
    av.get_last_device_error()
    got = av.attn_varlen_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), torch.from_numpy(cfg.cu_q),
                                  torch.from_numpy(cfg.cu_k), 1300, 1300, cfg.scale, chunks=chunks)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert not got.is_cuda
    assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16))
    rows = workloads.sample_rows(cfg.seed + chunks, q.shape[0] * cfg.Hq, 1 / 16)
    oref, _ = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D, cfg.scale, True, rows=rows)
    assert_close(got.reshape(-1, cfg.D)[torch.from_numpy(rows)], oref, f"host pipeline, {chunks} groups")


def test_host_pipelined_prefill_rejects_bad_offsets():
    """The host entry reads cu_seqlens on the host and refuses offsets that are
    not monotone or exceed the stated maxima, before any copy."""
    cfg = workloads.small_varlen(37, [100, 50], [100, 50], 8, 2, 64)
    q, k, v = cfg.q().pin_memory(), cfg.k().pin_memory(), cfg.v().pin_memory()
    bad = torch.tensor([0, 120, 150], dtype=torch.int32)   # lengths 120, 30 on 150 rows
    with pytest.raises(av.AttnError) as e:
        av.attn_varlen_fwd_host(q, k, v, bad, torch.from_numpy(cfg.cu_k), 100, 100, cfg.scale)
    assert e.value.status == 1
    dec = torch.tensor([0, 100, 90], dtype=torch.int32)
    with pytest.raises((av.AttnError, ValueError)):
        av.attn_varlen_fwd_host(q, k, v, dec, torch.from_numpy(cfg.cu_k), 100, 100, cfg.scale)
