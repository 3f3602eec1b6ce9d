"""Padded-batch prefill (attn_padded_fwd) on the GPU: bit-identical to the varlen
path on the real rows, whatever the padding holds, and against the oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _pad(packed, cu, S, fill=float("nan")):
    """[total, H, D] varlen rows -> [B, S, H, D] with `fill` in the padding."""
    B = len(cu) - 1
    out = torch.full((B, S) + tuple(packed.shape[1:]), fill, dtype=packed.dtype)
    for b in range(B):
        out[b, :cu[b + 1] - cu[b]] = packed[cu[b]:cu[b + 1]]
    return out


def _real_rows(padded, cu):
    return torch.cat([padded[b, :cu[b + 1] - cu[b]] for b in range(len(cu) - 1)])


CASES = [
    # seed, lens_q, lens_k, Hq, Hkv, D, causal
    (81, [5, 300, 1, 129], [5, 300, 1, 129], 32, 8, 128, True),
    (82, [40, 7, 200], [300, 7, 1000], 16, 2, 64, True),
    (83, [64, 3], [100, 900], 8, 8, 128, False),
]


@pytest.mark.parametrize("seed,lq,lk,Hq,Hkv,D,causal", CASES)
def test_padded_equals_varlen_and_oracle(seed, lq, lk, Hq, Hkv, D, causal):
    cfg = workloads.small_varlen(seed, lq, lk, Hq, Hkv, D, causal=causal)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    Sq, Sk = int(max(lq)) + 13, int(max(lk)) + 70
    qp, kp, vp = _pad(q, cfg.cu_q, Sq).cuda(), _pad(k, cfg.cu_k, Sk).cuda(), _pad(v, cfg.cu_k, Sk).cuda()
    sq = torch.tensor(lq, dtype=torch.int32).cuda()
    sk = torch.tensor(lk, dtype=torch.int32).cuda()
    av.get_last_device_error()
    out_p, lse_p = av.attn_padded_fwd(qp, kp, vp, sq, sk, cfg.scale, causal=causal, return_lse=True)
    cu_q = torch.from_numpy(cfg.cu_q).cuda()
    cu_k = torch.from_numpy(cfg.cu_k).cuda()
    out_v, lse_v = av.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), cu_q, cu_k, max(lq), max(lk), cfg.scale,
                                      causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    got = _real_rows(out_p, cfg.cu_q)
    assert torch.equal(got.view(torch.int16), out_v.view(torch.int16))
    rows = torch.cat([torch.arange(b * Sq, b * Sq + lq[b]) for b in range(len(lq))]).cuda()
    assert torch.equal(lse_p[:, rows], lse_v)
    ref, ref_lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, Hq, Hkv, D, cfg.scale, causal)
    assert_close(got, ref.reshape(got.shape), "padded")
    assert_lse_close(lse_v.t().contiguous(), ref_lse.reshape(-1, Hq), "padded lse")


def test_padded_without_lengths_is_full_rows():
    cfg = workloads.small_varlen(84, [96, 96], [96, 96], 8, 2, 128)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    out_p = av.attn_padded_fwd(q.view(2, 96, 8, 128).cuda(), k.view(2, 96, 2, 128).cuda(),
                               v.view(2, 96, 2, 128).cuda(), softmax_scale=cfg.scale)
    out_v = av.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cfg.cu_q).cuda(),
                               torch.from_numpy(cfg.cu_k).cuda(), 96, 96, cfg.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(-1, 8, 128).view(torch.int16), out_v.view(torch.int16))


def test_padded_length_beyond_padding_is_reported():
    cfg = workloads.small_varlen(85, [10, 20], [10, 20], 8, 8, 64)
    qp = _pad(cfg.q(), cfg.cu_q, 24, 0.0).cuda()
    kp = _pad(cfg.k(), cfg.cu_k, 24, 0.0).cuda()
    vp = _pad(cfg.v(), cfg.cu_k, 24, 0.0).cuda()
    av.get_last_device_error()
    av.attn_padded_fwd(qp, kp, vp, torch.tensor([10, 30], dtype=torch.int32).cuda(),
                       torch.tensor([10, 20], dtype=torch.int32).cuda(), cfg.scale)
    torch.cuda.synchronize()
    st, word = av.get_last_device_error()
    assert st == 6, (st, hex(word))   # ATTN_ERR_DEVICE_INDEX


@pytest.mark.slow
def test_padded_c2_full_size_equals_varlen():
    """The benchmark's padded batch: c2_varlen_gqa as [16, 4096, H, D] with the
    per-sequence lengths and NaN in the padding; the real rows equal the varlen
    call on the packed tensors bit for bit (that call is checked against the
    oracle at this size by the prefill tests)."""
    cfg = workloads.make("c2_varlen_gqa")
    S = 4096
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    qp, kp, vp = _pad(q, cfg.cu_q, S).cuda(), _pad(k, cfg.cu_k, S).cuda(), _pad(v, cfg.cu_k, S).cuda()
    sq = torch.from_numpy(cfg.lens_q.astype(np.int32)).cuda()
    sk = torch.from_numpy(cfg.lens_k.astype(np.int32)).cuda()
    av.get_last_device_error()
    out_p = av.attn_padded_fwd(qp, kp, vp, sq, sk, cfg.scale)
    out_v = av.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cfg.cu_q).cuda(),
                               torch.from_numpy(cfg.cu_k).cuda(), int(cfg.lens_q.max()), int(cfg.lens_k.max()),
                               cfg.scale)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert torch.equal(_real_rows(out_p, cfg.cu_q).view(torch.int16), out_v.view(torch.int16))
    del qp, kp, vp, out_p, out_v
    torch.cuda.empty_cache()
