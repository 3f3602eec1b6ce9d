"""Shared helpers for the parity tests (comparison metrics, device placement)."""
import json
import os

import numpy as np
import torch

# Tolerance for bf16 inputs / fp32 accumulation / bf16 output against the
# float64 oracle: relative RMS <= 2e-3 over the compared outputs, and per
# element |err| <= 1e-2 + 2^-8 |ref|.  The second term is the bf16 output's own
# rounding bound (8 significant bits, round-to-nearest: half an ulp is at most
# 2^-8 of the value); without it no bf16 result could meet 1e-2 once |ref| >= 4.
# lse (float32) is compared with a relative bound.
MAX_ABS = 1e-2
OUT_ROUND = 2.0 ** -8
REL_RMS = 2e-3
LSE_ABS = 2e-3


def errors(got, ref, raw: bool = False):
    """(max over elements of |err| - 2^-8 |ref|, relative RMS) of got
    (bf16/float tensor or array) vs ref (float64); with raw=True also the plain
    max |err| and the largest |ref| (third and fourth entries)."""
    g = got.float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    g = g.reshape(r.shape)
    d = g - r
    max_abs = float(np.max(np.abs(d) - OUT_ROUND * np.abs(r))) if d.size else 0.0
    den = float(np.sqrt(np.sum(r * r)))
    rel = float(np.sqrt(np.sum(d * d)) / den) if den > 0 else float(np.sqrt(np.sum(d * d)))
    if not raw:
        return max_abs, rel
    return max_abs, rel, float(np.max(np.abs(d))) if d.size else 0.0, float(np.max(np.abs(r))) if r.size else 0.0


def _log_parity(what, max_abs, rel, raw_max=None, ref_max=None):
    """With ATTN_PARITY_LOG=<file> set, append each comparison's metrics to that
    file (one JSON object per line) so a run of the parity tests can be tabulated:
    the plain max |err|, the max of |err| - 2^-8 |ref| (the bf16 output's own
    rounding taken out), the largest |ref| and the relative RMS."""
    path = os.environ.get("ATTN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "max_abs_err": raw_max, "max_abs_minus_rounding": max_abs,
                                "max_abs_ref": ref_max, "rel_rms": rel}) + "\n")


def assert_close(got, ref, what=""):
    g = got.float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    max_abs, rel, raw_max, ref_max = errors(got, ref, raw=True)
    _log_parity(what, max_abs, rel, raw_max, ref_max)
    assert max_abs <= MAX_ABS and rel <= REL_RMS, f"{what}: max|err|={max_abs:.3e} relRMS={rel:.3e}"
    return max_abs, rel


def assert_lse_close(got, ref, what=""):
    g = got.float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: lse finiteness differs"
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), f"{what}: lse -inf pattern differs"
    if fin.any():
        err = np.max(np.abs(g[fin] - r[fin]) / np.maximum(1.0, np.abs(r[fin])))
        assert err <= LSE_ABS, f"{what}: lse err {err:.3e}"


def cuda(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()
