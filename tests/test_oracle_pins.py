"""Pins of the float64 oracle against what the article and mathematics fix.

Nothing here needs a GPU.  Each test checks the oracle against something other
than itself: the article's worked examples (tests/golden/article_examples.json,
each entry citing its section of "从零实现 vLLM (1.3)：如何加速 Attention 计算"),
closed forms, invariants, special cases that reduce to textbook results, or an
independent library computation (numpy / scipy) on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp
from scipy.special import softmax as sp_softmax

import oracle
import workloads

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "article_examples.json")))


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.float().double().numpy()


def scipy_attention(q, k, v, lens_q, lens_k, Hq, Hkv, scale, causal=True):
    """Independent library statement: numpy matmul + scipy softmax/logsumexp on
    each sequence and head, padded-free.  q [Tq,Hq,D], k/v [Tk,Hkv,D] float64."""
    G = Hq // Hkv
    cq = np.concatenate([[0], np.cumsum(lens_q)])
    ck = np.concatenate([[0], np.cumsum(lens_k)])
    D = q.shape[-1]
    out = np.zeros((q.shape[0], Hq, D))
    lse = np.full((q.shape[0], Hq), -np.inf)
    for b in range(len(lens_q)):
        Lq, Lk = lens_q[b], lens_k[b]
        for h in range(Hq):
            Q = q[cq[b]:cq[b + 1], h]
            K = k[ck[b]:ck[b + 1], h // G]
            V = v[ck[b]:ck[b + 1], h // G]
            X = scale * (Q @ K.T)
            if causal:
                i = np.arange(Lq)[:, None]
                j = np.arange(Lk)[None, :]
                X = np.where(j <= Lk - Lq + i, X, -np.inf)
            for r in range(Lq):
                if np.all(np.isneginf(X[r])):
                    continue
                out[cq[b] + r, h] = sp_softmax(X[r]) @ V
                lse[cq[b] + r, h] = logsumexp(X[r])
    return out, lse


# --------------------------------------------------------------------------
# softmax pins
# --------------------------------------------------------------------------

def test_online_softmax_worked_example():
    """[10, 0, 8, 12, 5]: the running max and the proxy denominator d'_i =
    sum_{j<=i} e^{x_j - m_i} (its definition, evaluated directly), and the
    2-pass result equal to the 3-pass safe softmax."""
    x = GOLDEN["online_softmax_example"]["x"]
    y, mt, dt = oracle.softmax_online(x)
    assert list(mt) == [10, 10, 10, 12, 12]
    for i in range(len(x)):
        m_i = max(x[: i + 1])
        d_def = math.fsum(math.exp(xj - m_i) for xj in x[: i + 1])
        assert abs(dt[i] - d_def) <= 1e-15 * d_def
    # numbers quoted in the design notes for the lost table
    np.testing.assert_allclose(dt, [1.0, 1.0000453999, 1.1353806832, 1.1536570663, 1.1545689483], rtol=1e-10)
    ys = oracle.softmax_safe(x)
    np.testing.assert_allclose(y, ys, rtol=0, atol=1e-15)
    closed = np.array([math.exp(xi - 12) for xi in x]) / math.fsum(math.exp(xi - 12) for xi in x)
    np.testing.assert_allclose(ys, closed, rtol=1e-14)
    np.testing.assert_allclose(ys, [0.1172171514, 5.32165044e-6, 0.0158636164, 0.8661241076, 7.898029536e-4],
                               rtol=1e-8)


def test_overflow_example_700_710_705():
    x = GOLDEN["overflow_example"]["x"]
    ys = oracle.softmax_safe(x)
    assert np.all(np.isfinite(ys))
    den = 1 + math.exp(-5) + math.exp(-10)
    np.testing.assert_allclose(ys, [math.exp(-10) / den, 1 / den, math.exp(-5) / den], rtol=1e-14)
    with np.errstate(all="ignore"):
        y32 = oracle.softmax_naive(x, "f32")        # e^700.. overflow float32: inf/inf
        y64 = oracle.softmax_naive(x, "f64")        # only e^710 overflows float64
    assert not np.any(np.isfinite(y32))
    assert np.isnan(y64[1]) and y64[0] == 0.0 and y64[2] == 0.0


def test_fp16_overflow_threshold():
    """The article's float16 overflow point: e^11 still fits, e^12 does not."""
    assert GOLDEN["fp16_threshold"]["overflow_at_or_above"] == 11
    with np.errstate(over="ignore"):
        assert np.isfinite(np.exp(np.float16(11)))
        assert np.isinf(np.exp(np.float16(12)))


def test_library_example_weights():
    g = GOLDEN["library_scores"]
    ys = oracle.softmax_safe(g["scores"])
    np.testing.assert_allclose(ys, g["weights"], atol=0.01)
    assert abs(ys.sum() - 1) < 1e-15
    np.testing.assert_allclose(ys, sp_softmax(np.array(g["scores"])), rtol=1e-14)


# --------------------------------------------------------------------------
# attention pins
# --------------------------------------------------------------------------

def _one_head(q, k, v, causal=True, scale=1.0):
    """Single sequence, single head, through the oracle; arrays float32-valued."""
    Lq, D = q.shape
    Lk = k.shape[0]
    qb = bf16(q).view(Lq, 1, D)
    kb = bf16(k).view(Lk, 1, D)
    vb = bf16(v).view(Lk, 1, D)
    return oracle.attn_varlen(qb, kb, vb, [0, Lq], [0, Lk], 1, 1, D, scale, causal)


def test_weighted_sum_of_values():
    """Step 3 of the article: the output row is sum_j a_j v_j with a =
    softmax of the logits.  One query, keys that give logits exactly the
    library example's scores (bf16-exact), one-hot values -> the weights."""
    s = np.array([10.0, 0.10009765625, 8.5])         # 0.1 rounded to bf16
    D = 3
    q = np.zeros((1, D)); q[0, 0] = 1.0
    k = np.zeros((3, D)); k[:, 0] = s
    v = np.eye(3)
    out, lse = _one_head(q, k, v, causal=False)
    np.testing.assert_allclose(out[0], sp_softmax(s), rtol=1e-14)
    np.testing.assert_allclose(out[0], GOLDEN["weighted_sum"]["weights"], atol=0.01)
    np.testing.assert_allclose(lse[0], logsumexp(s), rtol=1e-15)
    # linearity in V: random V gives weights @ V
    rng = np.random.default_rng(0)
    v2 = rng.standard_normal((3, 5)).astype(np.float32)
    q2 = np.zeros((1, 5)); q2[0, 0] = 1.0
    k2 = np.zeros((3, 5)); k2[:, 0] = s
    out2, _ = _one_head(q2, k2, v2, causal=False)
    np.testing.assert_allclose(out2[0], sp_softmax(s) @ f64(bf16(v2)), rtol=1e-13)


def test_rows_sum_to_one():
    """With V = 1 everywhere the output is the row sum of A, which is 1."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((7, 16)) * 3
    k = rng.standard_normal((11, 16)) * 3
    v = np.ones((11, 16))
    for causal in (True, False):
        out, _ = _one_head(q, k, v, causal=causal, scale=0.25)
        np.testing.assert_allclose(out, 1.0, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(2)
    Lq, Lk, D = 4, 9, 8
    q = np.zeros((Lq, D))
    k = rng.standard_normal((Lk, D))
    v = rng.standard_normal((Lk, D))
    out, _ = _one_head(q, k, v, causal=True)
    vv = f64(bf16(v))
    for i in range(Lq):
        nvis = Lk - Lq + i + 1                       # bottom-right alignment
        np.testing.assert_allclose(out[i], vv[:nvis].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(3)
    D = 8
    q = rng.standard_normal((5, D)) * 4
    k = rng.standard_normal((5, D))
    v = rng.standard_normal((5, D))
    out, _ = _one_head(q, k, v, causal=True)        # Lq = Lk: query 0 sees key 0 only
    np.testing.assert_array_equal(out[0], f64(bf16(v))[0])
    out1, _ = _one_head(q[:1], k[:1], v[:1], causal=True)
    np.testing.assert_array_equal(out1[0], f64(bf16(v))[0])


def test_causal_is_bottom_right_aligned():
    """One-hot values expose the weights: query i sees exactly keys
    j <= Lk - Lq + i."""
    rng = np.random.default_rng(4)
    for Lq, Lk in [(3, 8), (5, 5), (1, 6), (6, 4)]:
        D = Lk
        q = rng.standard_normal((Lq, D))
        k = rng.standard_normal((Lk, D))
        out, lse = _one_head(q, k, np.eye(Lk), causal=True)
        for i in range(Lq):
            last = Lk - Lq + i
            if last < 0:
                assert np.all(out[i] == 0) and np.isneginf(lse[i])
                continue
            assert np.all(out[i][last + 1:] == 0)
            assert np.all(out[i][: last + 1] > 0)
            assert abs(out[i].sum() - 1) < 1e-12


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq/Hkv): values constant per KV head."""
    Hq, Hkv, D, L = 8, 2, 4, 6
    rng = np.random.default_rng(5)
    q = bf16(rng.standard_normal((L, Hq, D)))
    k = bf16(rng.standard_normal((L, Hkv, D)))
    v = np.zeros((L, Hkv, D), dtype=np.float32)
    for g in range(Hkv):
        v[:, g, :] = g + 1
    out, _ = oracle.attn_varlen(q, k, bf16(v), [0, L], [0, L], Hq, Hkv, D, 0.5, True)
    out = out.reshape(L, Hq, D)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], h // (Hq // Hkv) + 1, rtol=1e-14)


def test_tiled_recurrence_equals_untiled():
    """The 1-pass (m, d', o') recurrence over key blocks equals the three-step
    result: the article's 4-key / 2-block toy, then every block size on random
    tiny inputs."""
    rng = np.random.default_rng(6)
    cases = [(4, 2, [2])] + [(Lk, D, list(range(1, Lk + 1))) for Lk, D in [(7, 5), (13, 8), (1, 3)]]
    for Lk, D, blocks in cases:
        q = f64(bf16(rng.standard_normal(D) * 2))
        K = f64(bf16(rng.standard_normal((Lk, D)) * 2))
        V = f64(bf16(rng.standard_normal((Lk, D))))
        ref, lse = _one_head(q[None], K, V, causal=False, scale=0.7)
        for blk in blocks:
            o, m, d = oracle.attn_tiled_row(q, K, V, 0.7, blk)
            np.testing.assert_allclose(o, ref[0], rtol=1e-12, atol=1e-14)
            assert abs(m + math.log(d) - lse[0]) < 1e-12


def test_varlen_example_slicing():
    """The article's cu_seqlens example: packed result equals each sequence on
    its own slice, and equals padded batches with the padding masked."""
    g = GOLDEN["varlen_example"]
    cfg = workloads.make("c1_tiny")
    assert list(cfg.cu_q) == g["cu_seqlens_q"] and list(cfg.cu_k) == g["cu_seqlens_k"]
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    assert q.shape[0] == 8                           # not the article's "[7, ...]"
    out, lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 4, 4, 64, cfg.scale, True)
    out = out.reshape(8, 4, 64)
    for (q0, q1), (k0, k1) in zip(g["q_slices"], g["k_slices"]):
        o1, _ = oracle.attn_varlen(q[q0:q1], k[k0:k1], v[k0:k1], [0, q1 - q0], [0, k1 - k0], 4, 4, 64,
                                   cfg.scale, True)
        np.testing.assert_array_equal(out[q0:q1], o1.reshape(q1 - q0, 4, 64))
    # padded form: pad every sequence to the longest (5 queries, 9 keys), mask padding
    Pq, Pk = max(cfg.lens_q), max(cfg.lens_k)
    assert [Pq] * 3 == g["padded_lengths"]
    qf, kf, vf = f64(q), f64(k), f64(v)
    for b, ((q0, q1), (k0, k1)) in enumerate(zip(g["q_slices"], g["k_slices"])):
        Qp = np.zeros((Pq, 4, 64)); Qp[: q1 - q0] = qf[q0:q1]
        Kp = np.zeros((Pk, 4, 64)); Kp[: k1 - k0] = kf[k0:k1]
        Vp = np.zeros((Pk, 4, 64)); Vp[: k1 - k0] = vf[k0:k1]
        Lq, Lk = q1 - q0, k1 - k0
        X = np.einsum("ihd,jhd->hij", Qp, Kp) * cfg.scale
        i = np.arange(Pq)[:, None]
        j = np.arange(Pk)[None, :]
        ok = (j < Lk) & (j <= Lk - Lq + i)
        X = np.where(ok[None], X, -np.inf)
        A = sp_softmax(X[:, :Lq], axis=-1)
        O = np.einsum("hij,jhd->ihd", A, Vp)
        np.testing.assert_allclose(out[q0:q1], O, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_against_library_bruteforce(causal):
    rng = np.random.default_rng(7)
    lens_q = np.array([3, 1, 6, 0, 5])
    lens_k = np.array([7, 4, 6, 2, 5]) if causal else np.array([2, 9, 6, 3, 1])
    Hq, Hkv, D = 6, 2, 16
    q = bf16(rng.standard_normal((lens_q.sum(), Hq, D)))
    k = bf16(rng.standard_normal((lens_k.sum(), Hkv, D)))
    v = bf16(rng.standard_normal((lens_k.sum(), Hkv, D)))
    out, lse = oracle.attn_varlen(q, k, v, workloads.cu_from_lens(lens_q), workloads.cu_from_lens(lens_k),
                                  Hq, Hkv, D, 0.3, causal)
    ref, ref_lse = scipy_attention(f64(q), f64(k), f64(v), lens_q, lens_k, Hq, Hkv, 0.3, causal)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(ref_lse.shape), ref_lse, rtol=1e-13)


def test_row_subset_matches_full():
    cfg = workloads.small_varlen(11, [9, 4], [9, 12], 4, 2, 32)
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    full, lse = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 4, 2, 32, cfg.scale, True)
    rows = np.array([0, 5, 17, 40, 51])
    sub, lse_s = oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, 4, 2, 32, cfg.scale, True, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(lse_s, lse[rows])


def test_overflow_scale_heads_stay_finite():
    """Logits near 700: the max-shift keeps everything finite and equal to the
    library's shifted softmax."""
    rng = np.random.default_rng(8)
    L, H, D = 40, 2, 32
    hs = np.array([160.0, 1.0], dtype=np.float32)
    q = bf16(rng.standard_normal((L, H, D)).astype(np.float32) * hs[None, :, None])
    k = bf16(rng.standard_normal((L, H, D)))
    v = bf16(rng.standard_normal((L, H, D)))
    scale = 1 / math.sqrt(D)
    out, lse = oracle.attn_varlen(q, k, v, [0, L], [0, L], H, H, D, scale, True)
    assert np.all(np.isfinite(out))
    X = scale * np.einsum("id,jd->ij", f64(q)[:, 0], f64(k)[:, 0])
    assert np.max(np.abs(X)) > 100
    ref, ref_lse = scipy_attention(f64(q), f64(k), f64(v), [L], [L], H, H, scale, True)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-11, atol=1e-12)


def test_paged_gather_equals_contiguous():
    """Paging is a pure copy: the oracle through a random block table equals the
    contiguous layout bit for bit."""
    cfg = workloads.small_paged(21, ctx=[37, 5, 64], new=[6, 1, 9], Hq=4, Hkv=2, D=16, block_size=16)
    bs, Hkv, D = cfg.block_size, cfg.Hkv, cfg.D
    kc = torch.zeros((cfg.num_blocks * bs, Hkv, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    contig_k, contig_v = [], []
    rng = np.random.default_rng(22)
    for b in range(cfg.batch):
        Lk = int(cfg.lens_k[b])
        kk = bf16(rng.standard_normal((Lk, Hkv, D)))
        vv = bf16(rng.standard_normal((Lk, Hkv, D)))
        for j in range(Lk):
            r = int(cfg.block_table[b, j // bs]) * bs + j % bs
            kc[r] = kk[j]
            vc[r] = vv[j]
        contig_k.append(kk)
        contig_v.append(vv)
    q = bf16(rng.standard_normal((int(cfg.new.sum()), 4, D)))
    cu_q = workloads.cu_from_lens(cfg.new)
    cu_k = workloads.cu_from_lens(cfg.lens_k)
    paged, lp = oracle.attn_varlen(q, kc, vc, cu_q, cu_k, 4, Hkv, D, cfg.scale, True,
                                   block_table=cfg.block_table, block_size=bs, num_blocks=cfg.num_blocks)
    cont, lc = oracle.attn_varlen(q, torch.cat(contig_k), torch.cat(contig_v), cu_q, cu_k, 4, Hkv, D,
                                  cfg.scale, True)
    np.testing.assert_array_equal(paged, cont)
    np.testing.assert_array_equal(lp, lc)


def test_decode_equals_last_row_of_prefill():
    cfg = workloads.small_paged(31, ctx=[20, 33, 1], new=[0, 0, 0], Hq=4, Hkv=2, D=16, block_size=16,
                                decode=True)
    bs, Hkv, D = cfg.block_size, cfg.Hkv, cfg.D
    kc = torch.zeros((cfg.num_blocks, bs, Hkv, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for pb, (b, i), kb, vb in cfg.context_blocks():
        kc[pb] = kb.view(bs, Hkv, D)
        vc[pb] = vb.view(bs, Hkv, D)
    q = cfg.q()
    out, lse = oracle.decode_paged(q, kc, vc, cfg.ctx, cfg.block_table, 4, Hkv, D, bs, cfg.num_blocks,
                                   cfg.scale)
    cu_q = np.arange(cfg.batch + 1, dtype=np.int32)
    o2, l2 = oracle.attn_varlen(q, kc, vc, cu_q, workloads.cu_from_lens(cfg.ctx), 4, Hkv, D, cfg.scale,
                                True, block_table=cfg.block_table, block_size=bs, num_blocks=cfg.num_blocks)
    np.testing.assert_array_equal(out.reshape(-1, D), o2)
    np.testing.assert_array_equal(lse.reshape(-1), l2)


def test_decode_shapes_of_the_article():
    g = GOLDEN["decode_shapes"]
    q = torch.zeros(g["q"])
    assert list(q.unsqueeze(1).shape) == g["q_unsqueezed"]


def test_store_kvcache_copy_loop():
    rng = np.random.default_rng(9)
    N, Hkv, D, slots = 6, 2, 8, 20
    k = bf16(rng.standard_normal((N, Hkv, D)))
    v = bf16(rng.standard_normal((N, Hkv, D)))
    kc = torch.full((slots, Hkv, D), 7.0, dtype=torch.bfloat16)   # sentinel
    vc = torch.full((slots, Hkv, D), -3.0, dtype=torch.bfloat16)
    sm = np.array([4, -1, 19, 0, 7, -5])
    k2, v2 = oracle.store_kvcache(k, v, kc, vc, sm)
    ek = oracle.as_bits(kc).copy()
    ev = oracle.as_bits(vc).copy()
    keep = sm >= 0
    ek[sm[keep]] = oracle.as_bits(k)[keep]
    ev[sm[keep]] = oracle.as_bits(v)[keep]
    np.testing.assert_array_equal(k2, ek)
    np.testing.assert_array_equal(v2, ev)
    untouched = np.setdiff1d(np.arange(slots), sm[keep])
    assert np.all(k2[untouched] == oracle.as_bits(kc)[untouched])
    with pytest.raises(ValueError):
        oracle.store_kvcache(k, v, kc, vc, np.array([0, 1, 2, 3, 4, 20]))


def test_empty_and_no_visible_rows():
    """Lk = 0 or a query that sees no key: output 0 and lse = -inf."""
    q = bf16(np.ones((3, 1, 4)))
    k = bf16(np.ones((1, 1, 4)))
    out, lse = oracle.attn_varlen(q, k, k, [0, 2, 3], [0, 0, 1], 1, 1, 4, 1.0, True)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:2]))
    np.testing.assert_array_equal(out[2], 1.0)


def test_softmax_rows_pins():
    """oracle.softmax_rows: every row equals scipy's softmax, sums to 1, and the
    overflow row [700, 710, 705] keeps its closed form."""
    from scipy.special import softmax as sp_softmax
    rng = np.random.default_rng(5)
    x = rng.normal(size=(37, 301)) * 30.0
    x[3] = -1e3
    y = oracle.softmax_rows(x)
    np.testing.assert_allclose(y, sp_softmax(x, axis=1), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-12)
    z = oracle.softmax_rows(np.array([[700.0, 710.0, 705.0]]))[0]
    e = np.exp(np.array([-10.0, 0.0, -5.0]))
    np.testing.assert_allclose(z, e / e.sum(), rtol=1e-14)
