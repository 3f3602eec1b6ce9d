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
