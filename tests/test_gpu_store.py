"""store_kvcache on the GPU against the oracle's copy loop: bit-exact."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("Hkv,D,strided", [(8, 128, False), (8, 128, True), (4, 64, False), (2, 96, False),
                                            (2, 3, False)])
def test_store_kvcache_bitexact(Hkv, D, strided):
    rng = np.random.default_rng(100 + D)
    N, num_slots = 300, 1024
    slots = rng.permutation(num_slots)[:N].astype(np.int64)
    slots[::17] = -1                                       # skipped tokens
    if strided:
        # k and v as views of a packed qkv-like buffer: token stride 3*Hkv*D
        big = workloads.normal_bf16((7, 1), N, 3 * Hkv * D).view(N, 3 * Hkv, D)
        k_h, v_h = big[:, Hkv:2 * Hkv], big[:, 2 * Hkv:]
    else:
        k_h = workloads.normal_bf16((7, 2), N, Hkv * D).view(N, Hkv, D)
        v_h = workloads.normal_bf16((7, 3), N, Hkv * D).view(N, Hkv, D)
    # caches start as a sentinel bit pattern (including NaN encodings)
    sentinel = torch.from_numpy(rng.integers(0, 1 << 16, size=(num_slots, Hkv, D), dtype=np.uint16).view(np.int16))
    kc_h = sentinel.view(torch.bfloat16).clone()
    vc_h = sentinel.view(torch.bfloat16).clone()
    exp_k, exp_v = oracle.store_kvcache(k_h.contiguous(), v_h.contiguous(), kc_h, vc_h, slots)

    if strided:
        big_d = big.cuda()
        k_d, v_d = big_d[:, Hkv:2 * Hkv], big_d[:, 2 * Hkv:]
    else:
        k_d, v_d = k_h.cuda(), v_h.cuda()
    kc_d, vc_d = kc_h.cuda(), vc_h.cuda()
    av.store_kvcache(k_d, v_d, kc_d, vc_d, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kc_d), exp_k.reshape(num_slots, Hkv, D))
    assert np.array_equal(_bits(vc_d), exp_v.reshape(num_slots, Hkv, D))
    assert av.get_last_device_error()[0] == 0


def test_store_kvcache_bad_slot_is_flagged_not_written():
    N, Hkv, D, num_slots = 4, 2, 64, 16
    k = torch.ones((N, Hkv, D), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((num_slots, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    av.get_last_device_error()
    av.store_kvcache(k, k, kc, vc, torch.tensor([0, 99, -1, 3], dtype=torch.int64, device="cuda"))
    st, word = av.get_last_device_error()
    assert st == 6 and word & 1
    assert kc[0].float().eq(1).all() and kc[3].float().eq(1).all()
    assert kc[1].float().eq(0).all() and kc[2].float().eq(0).all()
    assert av.get_last_device_error()[0] == 0          # the word was cleared


@pytest.mark.parametrize("Hkv,D,strided", [(8, 128, False), (8, 128, True), (2, 96, False), (2, 3, False)])
def test_store_kvcache_fp16_v_over_16(Hkv, D, strided):
    """With v16_cache the store also writes V / 16 as fp16 at the same slots
    (round to nearest, torch's conversion as the reference); other slots keep
    their sentinel bits, and K/V are written exactly as without it."""
    rng = np.random.default_rng(200 + D)
    N, num_slots = 257, 700
    slots = rng.permutation(num_slots)[:N].astype(np.int64)
    slots[::13] = -1
    if strided:
        big = workloads.normal_bf16((8, 1), N, 3 * Hkv * D).view(N, 3 * Hkv, D)
        k_h, v_h = big[:, Hkv:2 * Hkv], big[:, 2 * Hkv:]
    else:
        k_h = workloads.normal_bf16((8, 2), N, Hkv * D).view(N, Hkv, D)
        v_h = (workloads.normal_bf16((8, 3), N, Hkv * D).float() * 300.0).to(torch.bfloat16).view(N, Hkv, D)
    sentinel = torch.from_numpy(rng.integers(0, 1 << 16, size=(num_slots, Hkv, D), dtype=np.uint16).view(np.int16))
    kc_h = sentinel.view(torch.bfloat16).clone()
    vc_h = sentinel.view(torch.bfloat16).clone()
    v16_h = sentinel.view(torch.float16).clone()
    exp_k, exp_v = oracle.store_kvcache(k_h.contiguous(), v_h.contiguous(), kc_h, vc_h, slots)
    exp_16 = v16_h.clone()
    keep = slots >= 0
    exp_16[torch.from_numpy(slots[keep])] = (v_h.contiguous()[torch.from_numpy(keep)].float() / 16.0).half()
    if strided:
        big_d = big.cuda()
        k_d, v_d = big_d[:, Hkv:2 * Hkv], big_d[:, 2 * Hkv:]
    else:
        k_d, v_d = k_h.cuda(), v_h.cuda()
    kc_d, vc_d, v16_d = kc_h.cuda(), vc_h.cuda(), v16_h.cuda()
    av.get_last_device_error()
    av.store_kvcache(k_d, v_d, kc_d, vc_d, torch.from_numpy(slots).cuda(), v16_cache=v16_d)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    assert np.array_equal(_bits(kc_d), exp_k.reshape(num_slots, Hkv, D))
    assert np.array_equal(_bits(vc_d), exp_v.reshape(num_slots, Hkv, D))
    assert torch.equal(v16_d.cpu().view(torch.int16), exp_16.view(torch.int16))


def test_store_kvcache_v_beyond_fp16_range_is_reported():
    N, Hkv, D, num_slots = 4, 2, 64, 16
    v = torch.ones((N, Hkv, D), dtype=torch.bfloat16, device="cuda")
    v[2, 1, 5] = 3.0e6
    kc = torch.zeros((num_slots, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vc, v16 = torch.zeros_like(kc), torch.zeros((num_slots, Hkv, D), dtype=torch.float16, device="cuda")
    av.get_last_device_error()
    av.store_kvcache(v, v, kc, vc, torch.tensor([0, 1, 2, 3], dtype=torch.int64, device="cuda"), v16_cache=v16)
    st, word = av.get_last_device_error()
    assert st == 8 and word & 4
    assert torch.isfinite(v16.float()).all() and v16[2, 1, 5].item() == 65504.0


@pytest.mark.slow
def test_store_kvcache_bench_8x_tokens():
    """The benchmark's 8x store: 8 x the c3 step's new tokens (68,024) into random
    distinct slots, with the V/16 cache, the launch configuration the benchmark
    times (its grid follows the token count); a smaller pool than the benchmark's
    65,536 blocks keeps the test's memory down.  Every written slot is compared
    with the oracle's copy bit for bit, on a sample of slots."""
    cfg = workloads.make("c3_prefix_paged")
    n = 8 * int(cfg.new.sum())
    Hkv, D, num_slots = cfg.Hkv, cfg.D, 1 << 20
    slots = np.random.default_rng(cfg.seed + 14).choice(num_slots, n, replace=False).astype(np.int64)
    k_h = workloads.normal_bf16((9, 1), n, Hkv * D).view(n, Hkv, D)
    v_h = workloads.normal_bf16((9, 2), n, Hkv * D).view(n, Hkv, D)
    kc = torch.zeros((num_slots, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    v16 = torch.zeros((num_slots, Hkv, D), dtype=torch.float16, device="cuda")
    av.get_last_device_error()
    av.store_kvcache(k_h.cuda(), v_h.cuda(), kc, vc, torch.from_numpy(slots).cuda(), v16_cache=v16)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    pick = np.sort(np.random.default_rng(3).choice(n, 4096, replace=False))
    sl = torch.from_numpy(slots[pick])
    # the oracle's copy loop on the sampled tokens into a compact pool of their slots
    ref_k, ref_v = oracle.store_kvcache(k_h[pick].contiguous(), v_h[pick].contiguous(),
                                        torch.zeros((len(pick), Hkv, D), dtype=torch.bfloat16),
                                        torch.zeros((len(pick), Hkv, D), dtype=torch.bfloat16),
                                        np.arange(len(pick), dtype=np.int64))
    assert np.array_equal(_bits(kc[sl.cuda()]), ref_k.reshape(len(pick), Hkv, D))
    assert np.array_equal(_bits(vc[sl.cuda()]), ref_v.reshape(len(pick), Hkv, D))
    assert torch.equal(v16[sl.cuda()].cpu().view(torch.int16),
                       (v_h[pick].float() / 16.0).half().view(torch.int16))
    del kc, vc, v16
    torch.cuda.empty_cache()
