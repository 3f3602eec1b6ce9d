"""The allocation-free decode entry point, called through the C ABI.

attn_decode_paged_noalloc serves callers that cannot allocate device memory
while they decode (for instance a serving loop that gave every free byte to
its KV-cache pool at start-up, or a hot path where cudaMalloc could
synchronise the device).  It keeps its split partials in a scratch array the
library reserves statically.  This file checks that it returns what
attn_decode_paged (caller-provided workspace) returns, on two calls in a row
that share the same scratch, and that a split count too large for the scratch
is refused.  It is named so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import workloads
from _util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, q, kc, vc, out, lse, cs, bt, cfg, max_len, splits):
    return L.attn_decode_paged_noalloc(_p(q), _p(kc), _p(vc), _p(out), _p(lse), _p(cs), _p(bt), bt.shape[1],
                                       cfg.batch, cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size, cfg.num_blocks, max_len,
                                       cfg.scale, splits, 0, 0,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_decode_twice():
    L = av.lib()
    cfg = workloads.small_paged(91, ctx=[4000, 129, 2500, 64, 7000, 1, 3333, 800], new=[0] * 8, Hq=32, Hkv=8,
                                D=128, block_size=256, decode=True)
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    q = cfg.q().cuda()
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).cuda()
    bt = torch.from_numpy(cfg.block_table).cuda()
    max_len = int(cfg.ctx.max())
    ref, ref_lse = av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=max_len, return_lse=True)
    torch.cuda.synchronize()
    ref64 = ref.float().double().cpu().numpy()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _noalloc(L, q, kc, vc, out, lse, cs, bt, cfg, max_len, 0)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert_close(out, ref64, f"no-alloc decode, call {call}")
        assert_lse_close(lse, ref_lse.double().cpu().numpy(), f"no-alloc lse, call {call}")
    assert av.get_last_device_error()[0] == 0


def test_noalloc_refuses_splits_beyond_its_scratch():
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
    assert _noalloc(L, q, kc, kc, out, lse, cs, bt, cfg, 5000, 64) == 3
    assert _noalloc(L, q, kc, kc, out, lse, cs, bt, cfg, 5000, 0) == 0
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
