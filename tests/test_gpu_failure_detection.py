"""Failure detection on the GPU without a fault: a bounded mbarrier wait runs out
on purpose (nothing ever completes the barrier), the kernel records the timeout
in the device error word and returns, a second waiter gives up on the abort flag
the first one raised, and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle
import workloads
from _util import assert_close

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 1 << 1
SRC_SELFTEST = 1 << 13
STATUS_DEVICE_TIMEOUT = 5


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    av.get_last_device_error()
    r = av.selftest_bounded_wait()
    # the first waiter ran out after about the wait limit (one second)
    assert not r["first_ok"]
    assert 0.9e9 <= r["first_ns"] <= 3.0e9, r
    # the second started half a limit later and gave up on the abort flag, before its own limit
    assert not r["second_ok"]
    assert r["second_ns"] < 0.9e9, r
    st, word = av.get_last_device_error()
    assert st == STATUS_DEVICE_TIMEOUT
    assert word & ERR_TIMEOUT and word & SRC_SELFTEST, hex(word)
    # the word is cleared by that read, and the device still runs the library's kernels
    assert av.get_last_device_error()[0] == 0
    cfg = workloads.small_varlen(99, [40, 7], [300, 7], 8, 2, 128, True)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    out = av.attn_varlen_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cfg.cu_q).cuda(),
                             torch.from_numpy(cfg.cu_k).cuda(), 40, 300, cfg.scale)
    torch.cuda.synchronize()
    assert av.get_last_device_error()[0] == 0
    ref, _ = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 8, 2, 128, cfg.scale, True)
    assert_close(out, ref.reshape(out.shape), "after the self-test")
