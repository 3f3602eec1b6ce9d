"""The Attention layer through an engine-like sequence of steps (prefill, two
decode steps, a three-token decode step, a prefix-cache prefill) on one paged cache, each step against the
float64 oracle over the whole history."""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_varlen_gb300.attention import Attention, AttentionContext
from _util import assert_close

pytestmark = pytest.mark.gpu

Hq, Hkv, D, BS = 8, 2, 128, 16


def _rand(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


def _cu(lens):
    return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)


@pytest.mark.parametrize("v16", [False, True])
def test_engine_steps_match_oracle(v16):
    """v16: the layer also keeps the fp16 V / 16 cache (filled by the store, read
    by the prefix prefill and the kv-cache entry's prefill route)."""
    gen = torch.Generator().manual_seed(77)
    rng = np.random.default_rng(77)
    prompts = np.array([37, 300, 5])
    B = len(prompts)
    max_blocks = 32
    num_blocks = B * max_blocks + 4
    tables = rng.permutation(num_blocks)[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    layer = Attention(Hq, D, D ** -0.5, Hkv)
    layer.k_cache = torch.full((num_blocks, BS, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    layer.v_cache = torch.full_like(layer.k_cache, float("nan"))
    if v16:
        layer.v16_cache = torch.full(layer.k_cache.shape, float("nan"), dtype=torch.float16, device="cuda")
    hist_k = [torch.empty(0, Hkv, D, dtype=torch.bfloat16) for _ in range(B)]
    hist_v = [torch.empty(0, Hkv, D, dtype=torch.bfloat16) for _ in range(B)]
    lens = np.zeros(B, dtype=np.int64)
    bt = torch.from_numpy(tables).cuda()

    def slots_for(new):
        s = []
        for b in range(B):
            j = np.arange(lens[b], lens[b] + new[b])
            s.append(tables[b, j // BS].astype(np.int64) * BS + j % BS)
        return torch.from_numpy(np.concatenate(s)).cuda()

    def step(new, kind):
        new = np.asarray(new)
        n = int(new.sum())
        q, k, v = _rand(gen, n, Hq, D), _rand(gen, n, Hkv, D), _rand(gen, n, Hkv, D)
        cu_new = np.concatenate([[0], np.cumsum(new)])
        for b in range(B):
            hist_k[b] = torch.cat([hist_k[b], k[cu_new[b]:cu_new[b + 1]]])
            hist_v[b] = torch.cat([hist_v[b], v[cu_new[b]:cu_new[b + 1]]])
        slots = slots_for(new)
        total = lens + new
        if kind == "prefill":
            ctx = AttentionContext(True, slots, _cu(new).cuda(), _cu(total).cuda(), int(new.max()), int(total.max()))
        elif kind == "prefix":
            ctx = AttentionContext(True, slots, _cu(new).cuda(), _cu(total).cuda(), int(new.max()), int(total.max()),
                                   block_tables=bt)
        else:
            ctx = AttentionContext(False, slots, context_lens=torch.from_numpy(total.astype(np.int32)).cuda(),
                                   block_tables=bt, max_seqlen_k=int(total.max()))
        o = layer(q.cuda().reshape(n, Hq * D), k.cuda(), v.cuda(), ctx)
        torch.cuda.synchronize()
        lens[:] = total
        ref, _ = oracle.attn_varlen(q, torch.cat(hist_k), torch.cat(hist_v), _cu(new).numpy(), _cu(total).numpy(),
                                    Hq, Hkv, D, D ** -0.5, True)
        assert_close(o.view(n, Hq, D), ref.reshape(n, Hq, D), kind)

    step(prompts, "prefill")
    step([1, 1, 1], "decode")
    step([1, 1, 1], "decode")
    step([3, 3, 3], "decode")        # three new tokens per sequence (the kv-cache entry)
    step([20, 3, 40], "prefix")
    step([17, 17, 17], "decode")     # 17 x 4 query rows per KV head: the kv-cache entry's prefill route
