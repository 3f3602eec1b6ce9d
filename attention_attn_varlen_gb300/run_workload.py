"""Run one operation of the attention path on a named synthetic workload.

    python -m attention_attn_varlen_gb300.run_workload --workload c2_varlen_gqa --op prefill --iters 3

A plain driver for profilers and quick checks: it builds the inputs on the
device, runs the chosen call `--iters` times on the current stream and exits
with the device error status.  No timing, no comparison.

  --op prefill  attn_varlen_fwd (contiguous workloads c1, c2, c5; paged c3)
  --op store    store_kvcache of the new tokens (c3)
  --op decode   attn_decode_paged (c4)
  --op kvcache  attn_with_kvcache with --sq new query tokens per sequence (c4 cache)
  --op softmax  attn_softmax_rows on a seeded [--rows, --cols] matrix (--dtype f32 | bf16;
                --workload is ignored)
  --seqs N      keep only the first N sequences (smaller captures)
  --v16         paged prefill / store / kvcache: keep the fp16 V / 16 cache beside
                the bf16 one (filled for the blocks in use, then by the store)
  --compact-pool  paged workloads: a pool of just the blocks the block table
                uses, ids randomly permuted (same block size, lengths and
                shared-prefix blocks; for profiler captures of a few GB at most)
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import attention_attn_varlen_gb300 as av  # noqa: E402
import workloads  # noqa: E402


def _trim(cfg, n):
    if n is None or n >= cfg.batch:
        return cfg
    if isinstance(cfg, workloads.Varlen):
        cfg.lens_q = cfg.lens_q[:n]
        cfg.lens_k = cfg.lens_k[:n]
        return cfg
    cfg.ctx = cfg.ctx[:n]
    cfg.new = cfg.new[:n]
    cfg.block_table = cfg.block_table[:n]
    return cfg


def _compact_pool(cfg, seed=7):
    """Renumber the referenced blocks into a pool of exactly that many blocks
    (random order); contents are keyed by logical (sequence, block), so the
    workload is unchanged apart from the physical ids."""
    bt = cfg.block_table
    ids = np.unique(bt[bt >= 0])
    perm = np.random.default_rng(seed).permutation(len(ids)).astype(np.int32)
    remap = np.full(int(ids.max()) + 1, -1, dtype=np.int32)
    remap[ids] = perm
    cfg.block_table = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    cfg.num_blocks = len(ids)
    return cfg


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c2_varlen_gqa", choices=workloads.CONFIG_NAMES)
    ap.add_argument("--op", required=True, choices=["prefill", "store", "decode", "kvcache", "softmax"])
    ap.add_argument("--rows", type=int, default=262144)
    ap.add_argument("--cols", type=int, default=1024)
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="bf16")
    ap.add_argument("--sq", type=int, default=4, help="new query tokens per sequence (--op kvcache)")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seqs", type=int, default=None)
    ap.add_argument("--compact-pool", action="store_true")
    ap.add_argument("--v16", action="store_true")
    a = ap.parse_args(argv)
    av.lib()
    dev = torch.device("cuda", 0)
    if a.op == "softmax":
        g = torch.Generator(device=dev).manual_seed(1)
        x = torch.randn(a.rows, a.cols, device=dev, generator=g) * 30.0
        x = x.to(torch.bfloat16 if a.dtype == "bf16" else torch.float32)
        y = torch.empty_like(x)
        for _ in range(a.iters):
            av.softmax_rows(x, out=y)
        torch.cuda.synchronize()
        st, word = av.get_last_device_error()
        print(f"softmax {a.rows}x{a.cols} {a.dtype} x{a.iters}: device status {st} word {word:#x}")
        return 0 if st == 0 else 1
    cfg = _trim(workloads.make(a.workload), a.seqs)
    if a.compact_pool and isinstance(cfg, workloads.Paged):
        cfg = _compact_pool(cfg)
    if isinstance(cfg, workloads.Varlen):
        if a.op != "prefill":
            raise SystemExit("contiguous workloads only have --op prefill")
        q, k, v = cfg.q().to(dev), cfg.k().to(dev), cfg.v().to(dev)
        cu_q = torch.from_numpy(cfg.cu_q).to(dev)
        cu_k = torch.from_numpy(cfg.cu_k).to(dev)
        out = torch.empty_like(q)
        for _ in range(a.iters):
            av.attn_varlen_fwd(q, k, v, cu_q, cu_k, int(cfg.lens_q.max()), int(cfg.lens_k.max()), cfg.scale, out=out)
    else:
        kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        workloads.fill_paged_cache(cfg, kc, vc)
        bt = torch.from_numpy(np.ascontiguousarray(cfg.block_table)).to(dev)
        q = cfg.q().to(dev)
        if a.op == "decode":
            cs = torch.from_numpy(cfg.ctx.astype(np.int32)).to(dev)
            out = torch.empty_like(q)
            for _ in range(a.iters):
                av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=int(cfg.ctx.max()), out=out)
        elif a.op == "kvcache":
            # the last --sq cached tokens of each sequence are its new ones
            cs = torch.from_numpy(cfg.ctx.astype(np.int32)).to(dev)
            g = torch.Generator(device=dev).manual_seed(4321)
            qn = torch.randn(cfg.batch, a.sq, cfg.Hq, cfg.D, device=dev, generator=g).to(torch.bfloat16)
            out = torch.empty_like(qn)
            v16 = None
            if a.v16:
                v16 = torch.empty(kc.shape, dtype=torch.float16, device=dev)
                for i in range(0, cfg.num_blocks, 256):
                    v16[i:i + 256] = (vc[i:i + 256].float() / 16.0).half()
            for _ in range(a.iters):
                av.attn_with_kvcache(qn, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=int(cfg.ctx.max()), out=out,
                                     v16_cache=v16)
        else:
            k_new, v_new = cfg.k_new().to(dev), cfg.v_new().to(dev)
            slots = torch.from_numpy(cfg.slot_mapping()).to(dev)
            cu_q = torch.from_numpy(workloads.cu_from_lens(cfg.new)).to(dev)
            cu_k = torch.from_numpy(workloads.cu_from_lens(cfg.lens_k)).to(dev)
            out = torch.empty_like(q)
            v16 = None
            if a.v16:
                v16 = torch.empty(kc.shape, dtype=torch.float16, device=dev)
                used = torch.from_numpy(np.unique(cfg.block_table[cfg.block_table >= 0]).astype(np.int64)).to(dev)
                for i in range(0, used.numel(), 256):
                    j = used[i:i + 256]
                    v16[j] = (vc[j].float() / 16.0).half()
            for _ in range(a.iters):
                av.store_kvcache(k_new, v_new, kc, vc, slots, v16_cache=v16)
                if a.op == "prefill":
                    av.attn_varlen_fwd(q, kc, vc, cu_q, cu_k, int(cfg.new.max()), int(cfg.lens_k.max()), cfg.scale,
                                       block_table=bt, out=out, v16_cache=v16)
    st, word = av.get_last_device_error()
    print(f"{a.workload} {a.op} x{a.iters}: device status {st} word {word:#x}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
