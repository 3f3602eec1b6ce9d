"""Row softmax (online two-pass kernel) on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_attn_varlen_gb300 as av
import oracle

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (3, 7), (33, 31), (64, 128), (17, 1000), (8, 2048), (5, 2049), (9, 4096), (4, 4097),
          (2, 100003), (700, 512),
          (6, 16384), (3, 12296), (2, 32768),   # long rows: a CTA per row (in registers up to 64 KB)
          (1000, 3000), (400, 9000),            # more rows than CTAs: each CTA loads its next row early
          (20000, 1500),                        # rows streamed through shared memory, the ring wraps often
          (3, 40000), (3, 65536), (200, 20000),  # a cluster of CTAs per row: 5, 8, 3 slices of 32 KB
          (2, 131072), (40, 200000),            # fp32 8 / bf16 7 slices of 64 KB
          (2, 200000)]                          # fp32 beyond 8 slices of 64 KB: two passes


def _inputs(seed, rows, cols, scale=30.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, cols)) * scale).astype(np.float32)
    if rows > 1 and cols >= 3:
        x[1, :3] = [700.0, 710.0, 705.0]   # large logits: no overflow with the running max
    return x


def _check(y, ref, bf16):
    y = y.float().cpu().double().numpy()
    assert np.all(np.isfinite(y))
    rel = 2.0 ** -8 + 1e-4 if bf16 else 1e-4
    err = np.abs(y - ref)
    bad = err > rel * np.abs(ref) + 1e-7
    assert not bad.any(), f"max err {err.max():.3e} at {np.argwhere(bad)[0]}"
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=(2e-2 if bf16 else 1e-4))


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("bf16", [False, True])
def test_softmax_rows_matches_oracle(rows, cols, bf16):
    x = torch.from_numpy(_inputs(rows * 7 + cols, rows, cols))
    if bf16:
        x = x.to(torch.bfloat16)
    ref = oracle.softmax_rows(x)
    y = av.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    _check(y, ref, bf16)


def test_softmax_rows_strided_inplace_and_unaligned():
    x = torch.from_numpy(_inputs(91, 40, 3001))
    wide = torch.zeros(40, 3100, dtype=torch.float32)
    wide[:, :3001] = x
    wide = wide.cuda()
    view = wide[:, :3001]                      # row stride 3100
    ref = oracle.softmax_rows(x)
    y = av.softmax_rows(view)
    _check(y, ref, False)
    av.softmax_rows(view, out=view)            # in place
    _check(view, ref, False)
    assert torch.equal(wide[:, 3001:], torch.zeros(40, 99, device="cuda"))
    # bf16 rows with a partial last 16-byte vector (5003 = 625 * 8 + 3), stride 5008
    xb = torch.from_numpy(_inputs(93, 30, 5003)).to(torch.bfloat16)
    wb = torch.zeros(30, 5008, dtype=torch.bfloat16)
    wb[:, :5003] = xb
    wb = wb.cuda()
    _check(av.softmax_rows(wb[:, :5003]), oracle.softmax_rows(xb), True)
    # fp32 rows of 3 cluster slices with a partial last vector, stride 40004
    xc = torch.from_numpy(_inputs(94, 5, 40001))
    wc = torch.zeros(5, 40004, dtype=torch.float32)
    wc[:, :40001] = xc
    wc = wc.cuda()
    _check(av.softmax_rows(wc[:, :40001]), oracle.softmax_rows(xc), False)
    # a view that starts 4 bytes past a 16-byte boundary (element accesses)
    buf = torch.zeros(40 * 301 + 1, dtype=torch.float32, device="cuda")
    xu = buf[1:].view(40, 301)
    x2 = torch.from_numpy(_inputs(92, 40, 301))
    xu.copy_(x2.cuda())
    _check(av.softmax_rows(xu), oracle.softmax_rows(x2), False)


def test_softmax_rows_online_recurrence_on_the_article_example():
    """[10, 0, 8, 12, 5]: the kernel's result equals the online recurrence's."""
    x = torch.tensor([[10.0, 0.0, 8.0, 12.0, 5.0]])
    y = av.softmax_rows(x.cuda()).cpu().double().numpy()[0]
    ref, m_trace, _ = oracle.softmax_online(x.numpy()[0])
    np.testing.assert_allclose(y, ref, rtol=1e-5)
    assert m_trace[-1] == 12.0


@pytest.mark.slow
@pytest.mark.parametrize("rows,cols,dt", [(32768, 8192, "f32"), (262144, 1024, "bf16"), (4096, 65536, "f32")])
def test_softmax_bench_shapes_sampled_rows(rows, cols, dt):
    """The bench's three shapes at full size (the kernels it times: a CTA per row, a
    warp per row, a cluster per row), 64 sampled rows against the oracle."""
    g = torch.Generator(device="cuda").manual_seed(1234 + rows)
    x = torch.randn(rows, cols, device="cuda", generator=g) * 30.0
    if dt == "bf16":
        x = x.to(torch.bfloat16)
    y = av.softmax_rows(x)
    torch.cuda.synchronize()
    pick = torch.from_numpy(np.sort(np.random.default_rng(rows).choice(rows, 64, replace=False))).cuda()
    xs = x[pick].cpu()
    _check(y[pick], oracle.softmax_rows(xs), dt == "bf16")
    del x, y
    torch.cuda.empty_cache()
