"""Host-side checks of the seeded input generators and the work accounting."""
import numpy as np
import torch

import workloads


def test_generators_are_seeded_and_chunk_reproducible():
    a = workloads.normal_bf16((1, 2), 700, 16)
    b = workloads.normal_bf16((1, 2), 700, 16)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # a prefix of rows regenerates the same values chunk by chunk
    c = workloads.normal_bf16((1, 2), 300, 16)
    assert torch.equal(c[:256].view(torch.int16), a[:256].view(torch.int16))
    d = workloads.normal_bf16((1, 3), 700, 16)
    assert not torch.equal(a, d)
    assert abs(float(a.float().mean())) < 0.1 and abs(float(a.float().std()) - 1) < 0.1


def test_visible_pairs_bruteforce():
    for Lq in range(0, 7):
        for Lk in range(0, 9):
            for causal in (True, False):
                n = sum(1 for i in range(Lq) for j in range(Lk) if (not causal) or j <= Lk - Lq + i)
                assert workloads.visible_pairs(Lq, Lk, causal) == n


def test_article_example_flops():
    c = workloads.make("c1_tiny")
    # pairs = 5*9 - 10 + 2*7 - 1 + 1*3 = 51
    assert workloads.prefill_flops(c.lens_q, c.lens_k, 4, 64) == 4 * 64 * 4 * 51


def test_paged_workloads_are_consistent():
    c3 = workloads.make("c3_prefix_paged")
    assert c3.num_blocks == 65536 and c3.block_size == 256 and c3.batch == 32
    used = c3.block_table[c3.block_table >= 0]
    # shared prefix blocks are the only repeated ids
    ids, counts = np.unique(used, return_counts=True)
    assert set(ids[counts > 1]) == set(c3.block_table[0, : c3.shared_blocks])
    assert np.all(counts[counts > 1] == c3.n_shared)
    sm = c3.slot_mapping()
    assert len(sm) == c3.new.sum() and len(np.unique(sm)) == len(sm)
    c4 = workloads.make("c4_decode")
    assert c4.batch == 256 and c4.ctx.min() >= 128 and c4.ctx.max() <= 16384
    used = c4.block_table[c4.block_table >= 0]
    assert len(np.unique(used)) == len(used) == c4.num_blocks


def test_sample_rows_deterministic():
    a = workloads.sample_rows(5, 10000)
    b = workloads.sample_rows(5, 10000)
    assert np.array_equal(a, b) and len(a) == 157 and np.all(np.diff(a) > 0)
