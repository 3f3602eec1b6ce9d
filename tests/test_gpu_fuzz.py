"""Randomised parity sweep: shapes drawn from seeded generators (batch sizes, lengths
including empty sequences and Lq > Lk, GQA groups, head dims, causal or not, block
sizes, new-token counts, with and without the fp16 V/16 cache, softmax row lengths
across every kernel's range), each call compared with the float64 oracle.  The
hand-picked cases of the other files pin known edges; this file looks for the
unknown ones."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close, assert_lse_close
from test_gpu_decode import device_cache, oracle_decode
from test_gpu_prefill import _paged_device, _paged_oracle, _run_paged, run_contig, v16_of

pytestmark = pytest.mark.gpu


def _heads(rng):
    """(Hq, Hkv) with a group of up to 8 heads (every entry takes it), some not dividing 128."""
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while G * Hkv > 32:
        Hkv //= 2
    return G * Hkv, max(Hkv, 1)


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_varlen(seed):
    rng = np.random.default_rng(5000 + seed)
    Hq, Hkv = _heads(rng)
    D = int(rng.choice([64, 128]))
    causal = bool(rng.random() < 0.7)
    B = int(rng.integers(1, 7))
    lq = rng.integers(0, 400, B)
    lk = np.empty(B, dtype=np.int64)
    for b in range(B):
        r = rng.random()
        lk[b] = lq[b] if r < 0.4 else (lq[b] + rng.integers(0, 700) if r < 0.8 else rng.integers(0, lq[b] + 1))
    if lq.sum() == 0:
        lq[0] = 1
        lk[0] = max(lk[0], 1)
    cfg = workloads.small_varlen(7000 + seed, lq.tolist(), lk.tolist(), Hq, Hkv, D, causal)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    av.get_last_device_error()
    out, lse = run_contig(cfg, q, k, v, causal)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, Hq, Hkv, D, cfg.scale, causal)
    what = f"fuzz varlen s{seed} Hq{Hq}/{Hkv} D{D} causal={causal} {lq.tolist()}/{lk.tolist()}"
    assert_close(out, ref.reshape(out.shape), what)
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), what + " lse")


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_paged_prefill(seed):
    rng = np.random.default_rng(6000 + seed)
    Hq, Hkv = _heads(rng)
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 64, 256]))
    B = int(rng.integers(1, 6))
    ctx = rng.integers(0, 2000, B)
    new = rng.integers(1, 200, B)
    cfg = workloads.small_paged(8000 + seed, ctx=ctx.tolist(), new=new.tolist(), Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    use16 = bool(rng.random() < 0.5)
    out, lse = _run_paged(cfg, q, kc, vc, v16=v16_of(vc) if use16 else None)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)))
    what = f"fuzz paged s{seed} Hq{Hq}/{Hkv} D{D} bs{bs} v16={use16} {ctx.tolist()}+{new.tolist()}"
    assert_close(out, ref.reshape(out.shape), what)
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), what + " lse")


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_kvcache(seed):
    rng = np.random.default_rng(6500 + seed)
    Hq, Hkv = _heads(rng)
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 64, 256]))
    B = int(rng.integers(1, 6))
    Sq = int(rng.integers(1, 25))
    ctx = rng.integers(0, 3000, B)
    cfg = workloads.small_paged(8500 + seed, ctx=ctx.tolist(), new=[Sq] * B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs)
    q = cfg.q()
    av.get_last_device_error()
    kc, vc, k_new, v_new = _paged_device(cfg)
    cs = torch.from_numpy(cfg.lens_k.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    use16 = bool(rng.random() < 0.5)
    causal = bool(rng.random() < 0.8)
    out, lse = av.attn_with_kvcache(q.cuda().view(B, Sq, Hq, D), kc, vc, cs, bt, cfg.scale, causal=causal,
                                    return_lse=True, v16_cache=v16_of(vc) if use16 else None)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse, _ = _paged_oracle(cfg, q, k_new, v_new, list(range(cfg.batch)), causal=causal)
    what = f"fuzz kvcache s{seed} Hq{Hq}/{Hkv} D{D} bs{bs} Sq{Sq} v16={use16} causal={causal} ctx={ctx.tolist()}"
    assert_close(out.view(-1, Hq, D), ref.reshape(-1, Hq, D), what)
    assert_lse_close(lse.t().contiguous(), ref_lse.reshape(-1, Hq), what + " lse")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_decode_splits(seed):
    rng = np.random.default_rng(6800 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))   # the decode kernel takes any group
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 64, 256]))
    B = int(rng.integers(1, 9))
    ctx = rng.integers(0, 5000, B)
    cfg = workloads.small_paged(8800 + seed, ctx=ctx.tolist(), new=[0] * B, Hq=G * Hkv, Hkv=Hkv, D=D,
                                block_size=bs, decode=True)
    kc, vc = device_cache(cfg)
    qh = cfg.q()
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    splits = int(rng.choice([0, 1, 3, 7]))
    av.get_last_device_error()
    out, lse = av.attn_decode_paged(qh.cuda(), kc, vc, cs, bt, cfg.scale, num_splits=splits, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, ref_lse = oracle_decode(cfg, qh)
    what = f"fuzz decode s{seed} G{G} Hkv{Hkv} D{D} bs{bs} splits={splits} ctx={ctx.tolist()}"
    assert_close(out, ref, what)
    assert_lse_close(lse, ref_lse, what + " lse")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_softmax_rows(seed):
    rng = np.random.default_rng(6900 + seed)
    # row lengths across the warp, ring, register-row, cluster and two-pass kernels
    cols = int(rng.choice([rng.integers(1, 1025), rng.integers(1025, 4097), rng.integers(4097, 16385),
                           rng.integers(16385, 70000), rng.integers(131073, 140000)]))
    rows = int(rng.integers(1, max(2, min(3000, 4_000_000 // cols))))
    bf16 = bool(rng.random() < 0.5)
    pad = int(rng.choice([0, 0, 8, 13]))   # a row stride past the row (13: element accesses)
    x = (rng.standard_normal((rows, cols)) * 25.0).astype(np.float32)
    xt = torch.from_numpy(x)
    if bf16:
        xt = xt.to(torch.bfloat16)
    wide = torch.zeros(rows, cols + pad, dtype=xt.dtype)
    wide[:, :cols] = xt
    xd = wide.cuda()[:, :cols]
    y = av.softmax_rows(xd)
    torch.cuda.synchronize()
    ref = oracle.softmax_rows(xt)
    got = y.float().cpu().double().numpy()
    rel = 2.0 ** -8 + 1e-4 if bf16 else 1e-4
    err = np.abs(got - ref)
    bad = err > rel * np.abs(ref) + 1e-7
    assert not bad.any(), f"softmax {rows}x{cols} bf16={bf16} pad={pad}: max err {err.max():.3e}"
