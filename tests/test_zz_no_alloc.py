"""The allocation-free decode entry point, called through the C ABI.

attn_decode_paged_noalloc serves callers that cannot allocate device memory
while they decode (for instance a serving loop that gave every free byte to
its KV-cache pool at start-up, or a hot path where cudaMalloc could
synchronise the device).  It keeps its split partials in a scratch array the
library reserves statically.  This file checks, against the float64 oracle and
against attn_decode_paged (caller-provided workspace):
  - two calls in a row that share the same scratch;
  - a batch whose automatic split count needs more partials than the scratch
    holds, so the entry point lowers it (the result must equal
    attn_decode_paged with the lowered count, bit for bit);
  - an explicit split count too large for the scratch, which is refused.
It is named so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import workloads
from _util import assert_close, assert_lse_close
from test_gpu_decode import device_cache, oracle_decode

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20   # ATTN_DECODE_NOALLOC_SCRATCH_BYTES


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, q, kc, vc, out, lse, cs, bt, cfg, max_len, splits):
    return L.attn_decode_paged_noalloc(_p(q), _p(kc), _p(vc), _p(out), _p(lse), _p(cs), _p(bt), bt.shape[1],
                                       cfg.batch, cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size, cfg.num_blocks, max_len,
                                       cfg.scale, splits, 0, 0,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _partial_bytes(batch, Hq, D, splits):
    return batch * Hq * splits * (D + 1) * 4


def test_noalloc_decode_matches_oracle_and_workspace_decode_twice():
    L = av.lib()
    cfg = workloads.small_paged(91, ctx=[4000, 129, 2500, 64, 7000, 1, 3333, 800], new=[0] * 8, Hq=32, Hkv=8,
                                D=128, block_size=256, decode=True)
    kc, vc = device_cache(cfg)
    qh = cfg.q()
    q = qh.cuda()
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    max_len = int(cfg.ctx.max())
    av.get_last_device_error()
    ref, ref_lse = av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=max_len, return_lse=True)
    torch.cuda.synchronize()
    oref, oref_lse = oracle_decode(cfg, qh)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _noalloc(L, q, kc, vc, out, lse, cs, bt, cfg, max_len, 0)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from the workspace call"
        assert_close(out, oref, f"no-alloc decode vs oracle, call {call}")
        assert_lse_close(lse, oref_lse, f"no-alloc lse vs oracle, call {call}")
    assert av.get_last_device_error()[0] == 0


def test_noalloc_lowers_the_automatic_split_count_to_fit():
    """192 sequences, 32 query heads, a stated max length of 65,536 keys: the
    automatic plan (16 splits) needs 50.7 MB of partials, more than the 32 MiB
    scratch, so the entry point runs the largest count that fits."""
    L = av.lib()
    rng = np.random.default_rng(93)
    ctx = rng.integers(1, 2000, size=192, endpoint=True)
    ctx[5], ctx[40] = 65536, 20000
    cfg = workloads.small_paged(93, ctx=ctx.tolist(), new=[0] * 192, Hq=32, Hkv=8, D=128, block_size=256, decode=True)
    max_len = 65536
    auto = L.attn_decode_num_splits(cfg.batch, cfg.Hkv, max_len, 0)
    assert _partial_bytes(cfg.batch, cfg.Hq, cfg.D, auto) > SCRATCH_BYTES
    fit = SCRATCH_BYTES // _partial_bytes(cfg.batch, cfg.Hq, cfg.D, 1)
    assert 2 <= fit < auto
    kc, vc = device_cache(cfg)
    qh = cfg.q()
    q = qh.cuda()
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    av.get_last_device_error()
    out = torch.full((cfg.batch, cfg.Hq, cfg.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((cfg.batch, cfg.Hq), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(L, q, kc, vc, out, lse, cs, bt, cfg, max_len, 0) == 0
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    # the lowered plan is attn_decode_paged's plan for `fit` splits
    ref = av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=max_len, num_splits=int(fit))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    oref, oref_lse = oracle_decode(cfg, qh)
    assert_close(out, oref, "no-alloc decode, lowered split count")
    assert_lse_close(lse, oref_lse, "no-alloc lse, lowered split count")


def test_noalloc_refuses_explicit_splits_beyond_its_scratch():
    L = av.lib()
    cfg = workloads.small_paged(92, ctx=[5000] * 64, new=[0] * 64, Hq=32, Hkv=8, D=128, block_size=256,
                                decode=True)
    kc = torch.zeros((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    q = cfg.q().cuda()
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    out = torch.empty_like(q)
    lse = torch.empty((cfg.batch, cfg.Hq), dtype=torch.float32, device="cuda")
    # 64 sequences x 32 heads x 64 splits x 129 floats = 67.6 MB > 32 MiB
    assert _partial_bytes(64, 32, 128, 64) > SCRATCH_BYTES
    assert _noalloc(L, q, kc, kc, out, lse, cs, bt, cfg, 5000, 64) == 3
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
