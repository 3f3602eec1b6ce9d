"""Throughput of the attention hot path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Main line: varlen causal prefill, 16 sequences with L ~ U{256..4096} (Lq = Lk),
GQA 32/8, head_dim 128, bf16 (the prefill half of the metric), in TFLOP/s of
algorithmic work (4 * D * Hq * visible pairs).  One step = one attn_varlen_fwd
call over the batch.  L2 is flushed (a 512 MB write) between timed steps,
outside the timed events.  The same line carries every other workload as an
extra object with its roofline and the oracle timed on a sample of it:
  tiny_prefill    the article's 3-sequence example (launch-bound)
  decode          256-sequence paged decode (KV GB/s, the decode half of the
                  metric) and 4 / 8 new tokens per sequence on the same cache
  prefix_prefill  store_kvcache + paged prefix-cache prefill
  long_prefill    2 x 32k tokens with logits ~700 on half the heads
  row_softmax, padded_prefill
Each roofline is the dominant kernel's algorithmic work per launch over its
own device time (events the library records around that launch), against the
measured peaks of MEASURED_PEAKS.json: the bf16 burst figure for every
prefill (each kernel is timed by itself at full clocks), the copy bandwidth
for the HBM-bound kernels.
  cpu_baseline  the float64 oracle on a bounded sample of the main workload,
                timed on this host's cores (rank 0, N = 1 only)
  e2e           the same metric through the C entry attn_varlen_fwd_host with
                host buffers: pinned host -> device copies of q, k, v and
                cu_seqlens, the kernels, and the device -> host copy of the
                output, all inside the events
  clocks        nvidia-smi samples taken while the measurements ran
  summary       (last key) one compact entry per workload: step value, kernel
                value, roofline fraction, oracle value

Under torchrun (N > 1) every rank runs its own independent batch (replicas,
weak scaling: the units never need another rank's data); the timing is
bracketed by barriers and the maximum over ranks is reported.

--impl reference times the oracle itself as the reference arm (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "prefill TFLOP/s & decode KV GB/s at 1 GB300; % of tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


# --------------------------------------------------------------------------
# distributed plumbing (host side only; no collective on the data path)
# --------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(
        os.environ.get("WORLD_SIZE", "1"))


def dist_init(backend: str):
    import torch.distributed as dist
    if dist.is_available() and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def dist_max(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, max_seconds: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------------------
# peaks, clocks, profile data
# --------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi -lms sampling in the background while measurements run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        pw = np.array([r[2] for r in rows])
        loaded = [r for r in rows if r[2] >= 0.5 * pw.max()] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in loaded])), "sm_max_mhz": float(max(r[1] for r in rows)),
                "reasons": reasons, "samples": len(loaded), "power_w_max": float(pw.max())}


def src_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "prefill": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "prefill_paged": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "decode": ["attention_attn_varlen_gb300/csrc/decode.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "decode_sq4": ["attention_attn_varlen_gb300/csrc/decode.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "decode_sq8": ["attention_attn_varlen_gb300/csrc/decode.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "kvcache_sq4_v16": ["attention_attn_varlen_gb300/csrc/decode.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "kvcache_sq8_v16": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "kvcache_sq8": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "kvcache_sq16": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "kvcache_sq16_v16": ["attention_attn_varlen_gb300/csrc/prefill.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "store": ["attention_attn_varlen_gb300/csrc/store_kvcache.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "softmax_warp": ["attention_attn_varlen_gb300/csrc/softmax.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "softmax_cta_reg": ["attention_attn_varlen_gb300/csrc/softmax.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
    "softmax_cluster": ["attention_attn_varlen_gb300/csrc/softmax.cu", "attention_attn_varlen_gb300/csrc/common.cuh"],
}


def ncu_traffic(kernel: str, units: float):
    """DRAM bytes per launch from the committed ncu summary, scaled to `units`
    (profiles/dram_traffic.txt stores bytes per unit of work and the source
    digest of the kernel it was taken on); None if absent or the kernel
    changed since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kernel:
            if f[1] != src_digest(KERNEL_SOURCES[kernel]):
                return None
            return float(f[2]) * units
    return None


# --------------------------------------------------------------------------
# timing helpers
# --------------------------------------------------------------------------

def time_steps(fn, steps: int, flush=None, kernel: bool = False):
    """Per-step CUDA-event times (ms) on the current stream; `flush` runs
    between steps outside the events.  With kernel=True also returns the
    per-step device time of the call's main kernel alone (events the library
    records around that launch on the same stream)."""
    import torch
    import attention_attn_varlen_gb300 as av
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    try:
        for (a, b), (ka, kb) in zip(evs, kev):
            if flush is not None:
                flush()
            if kernel:
                av.set_kernel_events(ka, kb)
            a.record()
            fn()
            b.record()
    finally:
        if kernel:
            av.set_kernel_events()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    if not kernel:
        return ms
    return ms, [a.elapsed_time(b) for a, b in kev]


# --------------------------------------------------------------------------
# workloads on the device
# --------------------------------------------------------------------------

def varlen_inputs(cfg, device):
    import torch
    return dict(q=cfg.q().to(device), k=cfg.k().to(device), v=cfg.v().to(device),
                cu_q=torch.from_numpy(cfg.cu_q).to(device), cu_k=torch.from_numpy(cfg.cu_k).to(device),
                mq=int(cfg.lens_q.max()), mk=int(cfg.lens_k.max()))


def bench_varlen(av, cfg, inp, steps, warmup, flush):
    import torch
    out = torch.empty_like(inp["q"])

    def step():
        av.attn_varlen_fwd(inp["q"], inp["k"], inp["v"], inp["cu_q"], inp["cu_k"], inp["mq"], inp["mk"], cfg.scale,
                           out=out)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist_barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ms, kms = time_steps(step, steps, flush, kernel=True)
    torch.cuda.synchronize()
    dist_barrier()
    wall = time.perf_counter() - t0
    return ms, wall, kms


def bench_varlen_e2e(av, cfg, inp, steps, warmup, flush):
    """Host buffers in, host buffer out, through the C entry attn_varlen_fwd_host
    (the library copies one group of sequences in while it runs the attention of
    the previous group and copies an earlier group's output back)."""
    import torch
    hq, hk, hv = (inp[n].cpu().pin_memory() for n in ("q", "k", "v"))
    hcq, hck = inp["cu_q"].cpu().pin_memory(), inp["cu_k"].cpu().pin_memory()
    hout = torch.empty(hq.shape, dtype=hq.dtype).pin_memory()
    staging = av.host_staging(cfg.batch, hq.shape[0], hk.shape[0], cfg.Hq, cfg.Hkv, cfg.D, inp["mq"])

    def step():
        av.attn_varlen_fwd_host(hq, hk, hv, hcq, hck, inp["mq"], inp["mk"], cfg.scale, out=hout, staging=staging)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = time_steps(step, steps, flush)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hcq, hck))
    d2h = hout.numel() * hout.element_size()
    del staging
    return ms, h2d, d2h


def oracle_timed(fn, min_seconds: float = 0.0):
    """Run fn() (an oracle call) until at least min_seconds have passed; returns
    (seconds per call, calls)."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        t = time.perf_counter() - t0
        if t >= min_seconds:
            return t / n, n


def oracle_line(value, unit, sample, seconds):
    return {"value": value, "unit": unit, "cores": os.cpu_count(), "kind": "oracle", "sample": sample,
            "seconds": seconds}


def bench_decode(av, device, steps, warmup, flush, peaks, with_oracle=True):
    import torch
    cfg = workloads.make("c4_decode")
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    qh = cfg.q()
    q = qh.to(device)
    cs = torch.from_numpy(cfg.ctx.astype(np.int32)).to(device)
    bt = torch.from_numpy(cfg.block_table).to(device)
    out = torch.empty_like(q)
    mx = int(cfg.ctx.max())
    ws_bytes = av.decode_workspace_size(cfg.batch, cfg.Hq, cfg.Hkv, cfg.D, mx, 0)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    splits = av.decode_num_splits(cfg.batch, cfg.Hkv, mx, 0)

    def step():
        av.attn_decode_paged(q, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=mx, out=out, workspace=ws)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms, kms = time_steps(step, steps, flush, kernel=True)
    t = float(np.mean(ms)) / 1e3
    tk = float(np.mean(kms)) / 1e3
    nbytes = workloads.decode_bytes(cfg.ctx, cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size)
    gbs = nbytes / t / 1e9
    res = {"workload": "c4_decode: 256 seqs x 1 token, cache_seqlens U{128..16384}, GQA 32/8, D128, "
                       "block_size 256, random block table",
           "value": gbs, "unit": "GB/s", "ms_per_step": t * 1e3, "num_splits": splits,
           "algorithmic_bytes": nbytes,
           "roofline": {"bound": "hbm", "kernel": "attn_decode_split_kernel", "achieved": nbytes / tk / 1e9,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": nbytes / tk / 1e9 / peaks["hbm_gbs"],
                        "kernel_ms": tk * 1e3,
                        "traffic": ncu_traffic("decode", float(cfg.ctx.sum()) * cfg.Hkv)},
           "launches_per_step": 2 if splits > 1 else 1}
    # the same cache, Sq new query tokens per sequence (multi-token decode through
    # attn_with_kvcache; the last Sq cached tokens are the new ones)
    g = torch.Generator(device=device).manual_seed(4321)
    # the fp16 V / 16 cache the store would keep beside the bf16 one (here converted once,
    # outside the timing); the multi-token lines are also measured reading it
    v16 = torch.empty(kc.shape, dtype=torch.float16, device=device)
    for i in range(0, cfg.num_blocks, 256):
        v16[i:i + 256] = (vc[i:i + 256].float() / 16.0).half()
    for Sq in (4, 8, 16):
        qn = torch.randn(cfg.batch, Sq, cfg.Hq, cfg.D, device=device, generator=g).to(torch.bfloat16)
        wsn = torch.empty(av.lib().attn_kvcache_workspace_size(cfg.batch, Sq, cfg.Hq, cfg.Hkv, cfg.D, mx),
                          dtype=torch.uint8, device=device)
        outn = torch.empty_like(qn)

        def stepn():
            av.attn_with_kvcache(qn, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=mx, out=outn, workspace=wsn)
        for _ in range(warmup):
            stepn()
        torch.cuda.synchronize()
        msn, kmsn = time_steps(stepn, steps, flush, kernel=True)
        tn = float(np.mean(msn)) / 1e3
        tkn = float(np.mean(kmsn)) / 1e3
        fln = workloads.prefill_flops(np.full(cfg.batch, Sq), cfg.ctx, cfg.Hq, cfg.D)
        nbn = nbytes + 2 * cfg.batch * (Sq - 1) * cfg.Hq * cfg.D * 2    # the extra query and output rows
        # past 16 query rows per KV head (head_dim 128) the entry runs the one-slot
        # paged prefill, which converts the bf16 V tiles in shared memory
        rows = Sq * cfg.Hq // cfg.Hkv
        on_prefill_n = rows > 16
        res[f"kvcache_{Sq}_tokens"] = {
            "workload": f"c4_decode cache, {Sq} new query tokens per sequence (attn_with_kvcache: " +
                        ("one-slot paged prefill (tcgen05), V tiles converted in shared memory"
                         if on_prefill_n else "split-KV decode kernel") +
                        f", {rows} query rows per KV head, bottom-right causal)",
            "value": nbn / tn / 1e9, "unit": "GB/s", "tflops": fln / tn / 1e12, "ms_per_step": tn * 1e3,
            "algorithmic_bytes": nbn,
            "roofline": {"bound": "hbm", "kernel": "attn_prefill_kernel" if on_prefill_n else "attn_decode_split_kernel",
                         "achieved": nbn / tkn / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": nbn / tkn / 1e9 / peaks["hbm_gbs"],
                         "kernel_ms": tkn * 1e3,
                         "traffic": ncu_traffic(f"kvcache_sq{Sq}" if on_prefill_n else f"decode_sq{Sq}",
                                                float(cfg.ctx.sum()) * cfg.Hkv)},
            "launches_per_step": 3 if on_prefill_n else (2 if splits > 1 else 1)}

        def stepv():
            av.attn_with_kvcache(qn, kc, vc, cs, bt, cfg.scale, max_cache_seqlen=mx, out=outn, workspace=wsn,
                                 v16_cache=v16)
        for _ in range(warmup):
            stepv()
        torch.cuda.synchronize()
        msv, kmsv = time_steps(stepv, steps, flush, kernel=True)
        tv, tkv = float(np.mean(msv)) / 1e3, float(np.mean(kmsv)) / 1e3
        # with the V/16 cache, more than 16 query rows per KV head run on the paged prefill
        on_prefill = Sq * cfg.Hq // cfg.Hkv > 16
        res[f"kvcache_{Sq}_tokens_v16"] = {
            "workload": (f"the same {Sq}-token step reading the fp16 V/16 cache: " +
                         ("the paged varlen prefill (tcgen05), no conversion pass" if on_prefill else
                          "split-KV decode kernel, PV on one fp16 term 16 P")),
            "value": nbn / tv / 1e9, "unit": "GB/s", "ms_per_step": tv * 1e3, "algorithmic_bytes": nbn,
            "roofline": {"bound": "hbm", "kernel": "attn_prefill_kernel" if on_prefill else "attn_decode_split_kernel",
                         "achieved": nbn / tkv / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": nbn / tkv / 1e9 / peaks["hbm_gbs"],
                         "kernel_ms": tkv * 1e3,
                         "traffic": ncu_traffic(f"kvcache_sq{Sq}_v16", float(cfg.ctx.sum()) * cfg.Hkv)},
            # prefill route: cu_seqlens kernel, scheduling pre-pass, attention
            "launches_per_step": 3 if on_prefill else (2 if splits > 1 else 1)}
        del qn, wsn, outn
    del kc, vc, v16
    torch.cuda.empty_cache()
    if with_oracle:
        # the oracle on 48 of the 256 sequences, every query row
        seqs = sorted(np.random.default_rng(cfg.seed + 11).choice(cfg.batch, 48, replace=False).tolist())
        kp, vp, btc = workloads.compact_paged(cfg, seqs)
        qs = qh[torch.tensor(seqs)]
        import oracle
        oracle.build()
        sec, n = oracle_timed(lambda: oracle.decode_paged(qs, kp, vp, cfg.ctx[seqs], btc, cfg.Hq, cfg.Hkv, cfg.D,
                                                          cfg.block_size, kp.shape[0], cfg.scale), 1.0)
        ob = workloads.decode_bytes(cfg.ctx[seqs], cfg.Hq, cfg.Hkv, cfg.D, cfg.block_size)
        res["oracle"] = oracle_line(ob / sec / 1e9, "GB/s", f"48 of 256 sequences, all their query rows "
                                    f"({int(cfg.ctx[seqs].sum())} cached tokens), mean of {n} calls; float64, "
                                    f"OpenMP", sec)
    return res


def bench_prefix(av, device, steps, warmup, flush, peaks, with_oracle=True):
    import torch
    cfg = workloads.make("c3_prefix_paged")
    kc = torch.empty((cfg.num_blocks, cfg.block_size, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    workloads.fill_paged_cache(cfg, kc, vc)
    qh, k_new_h, v_new_h = cfg.q(), cfg.k_new(), cfg.v_new()
    q = qh.to(device)
    k_new, v_new = k_new_h.to(device), v_new_h.to(device)
    slots = torch.from_numpy(cfg.slot_mapping()).to(device)
    cu_q = torch.from_numpy(workloads.cu_from_lens(cfg.new)).to(device)
    cu_k = torch.from_numpy(workloads.cu_from_lens(cfg.lens_k)).to(device)
    bt = torch.from_numpy(cfg.block_table).to(device)
    out = torch.empty_like(q)
    mq, mk = int(cfg.new.max()), int(cfg.lens_k.max())
    # the fp16 V / 16 cache beside the bf16 one: earlier steps' stores filled it for
    # the cached context (here: converted once, outside the timing, for the blocks in use)
    v16 = torch.empty(kc.shape, dtype=torch.float16, device=device)
    used = torch.from_numpy(np.unique(cfg.block_table[cfg.block_table >= 0]).astype(np.int64)).to(device)
    for i in range(0, used.numel(), 256):
        j = used[i:i + 256]
        v16[j] = (vc[j].float() / 16.0).half()

    def store():
        av.store_kvcache(k_new, v_new, kc, vc, slots, v16_cache=v16)

    def attn():
        av.attn_varlen_fwd(q, kc, vc, cu_q, cu_k, mq, mk, cfg.scale, block_table=bt, out=out, v16_cache=v16)

    def step():
        store()
        attn()

    def step_convert():   # the same step without the V' cache: each call converts the V it reads
        av.store_kvcache(k_new, v_new, kc, vc, slots)
        av.attn_varlen_fwd(q, kc, vc, cu_q, cu_k, mq, mk, cfg.scale, block_table=bt, out=out)
    for _ in range(warmup):
        step()
        step_convert()
    torch.cuda.synchronize()
    ms = time_steps(step, steps, flush)
    ms_conv = time_steps(step_convert, steps, flush)
    ms_attn, kms_attn = time_steps(attn, steps, flush, kernel=True)
    ms_store, kms_store = time_steps(store, steps, flush, kernel=True)
    flops = workloads.prefill_flops(cfg.new, cfg.lens_k, cfg.Hq, cfg.D)
    sbytes = workloads.store_bytes(int(cfg.new.sum()), cfg.Hkv, cfg.D, v16=True)
    # the attention call's algorithmic bytes: q and out once, every distinct cache row
    # the block tables reach read once as K (bf16) and V / 16 (fp16)
    rows_used = {}
    for b in range(cfg.batch):
        lk = int(cfg.lens_k[b])
        for i in range((lk + cfg.block_size - 1) // cfg.block_size):
            blk = int(cfg.block_table[b, i])
            rows_used[blk] = max(rows_used.get(blk, 0), min(cfg.block_size, lk - i * cfg.block_size))
    distinct_rows = sum(rows_used.values())
    abytes = (2 * int(cfg.new.sum()) * cfg.Hq * cfg.D * 2) + distinct_rows * cfg.Hkv * cfg.D * 2 * 2
    t = float(np.mean(ms)) / 1e3
    ta = float(np.mean(ms_attn)) / 1e3
    tk = float(np.mean(kms_attn)) / 1e3
    ts = float(np.mean(ms_store)) / 1e3
    tks = float(np.mean(kms_store)) / 1e3
    tc = float(np.mean(ms_conv)) / 1e3
    # the same scatter at 8x the tokens (random distinct slots of the pool), to
    # separate the kernel's fixed cost from its bandwidth
    n8 = 8 * int(cfg.new.sum())
    kb8, vb8 = k_new.repeat(8, 1, 1), v_new.repeat(8, 1, 1)
    sl8 = torch.from_numpy(np.random.default_rng(cfg.seed + 14).choice(cfg.num_blocks * cfg.block_size, n8,
                                                                       replace=False).astype(np.int64)).to(device)

    def store8():
        av.store_kvcache(kb8, vb8, kc, vc, sl8, v16_cache=v16)
    for _ in range(warmup):
        store8()
    ms_s8, kms_s8 = time_steps(store8, steps, flush, kernel=True)
    sb8 = workloads.store_bytes(n8, cfg.Hkv, cfg.D, v16=True)
    t8, tk8 = float(np.mean(ms_s8)) / 1e3, float(np.mean(kms_s8)) / 1e3
    del kb8, vb8, sl8
    res = {"workload": "c3_prefix_paged: 32 seqs, context U{512..8192} + 1..512 new tokens, GQA 32/8, D128, "
                       "block_size 256, 65536-block pool, 8 seqs share prefix blocks; step = store_kvcache + "
                       "paged prefill, with the fp16 V/16 cache the store keeps",
           "value": flops / t / 1e12, "unit": "TFLOP/s", "ms_per_step": t * 1e3,
           "attn_ms": ta * 1e3, "store_ms": ts * 1e3,
           "without_v16_cache": {"value": flops / tc / 1e12, "ms_per_step": tc * 1e3},
           "roofline": {"bound": "tensor", "kernel": "attn_prefill_kernel", "achieved": flops / tk / 1e12,
                        "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": flops / tk / 1e12 / peaks["bf16_tflops"], "kernel_ms": tk * 1e3,
                        "traffic": ncu_traffic("prefill_paged", float(cfg.new.sum()))},
           # C3 has both bounds: the HBM side of the same kernel time, and t_min / t with
           # t_min = max(FLOPs / bf16 peak, bytes / copy bandwidth)
           "hbm": {"algorithmic_bytes": abytes, "distinct_cache_rows": distinct_rows,
                   "achieved": abytes / tk / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": abytes / tk / 1e9 / peaks["hbm_gbs"]},
           "roofline_tmin_frac": max(flops / (peaks["bf16_tflops"] * 1e12), abytes / (peaks["hbm_gbs"] * 1e9)) / tk,
           "store_kvcache": {"workload": "the step's 8503 new tokens: K, V and the fp16 V/16 row of each",
                             "value": sbytes / ts / 1e9, "unit": "GB/s", "ms_per_step": ts * 1e3,
                             "algorithmic_bytes": sbytes,
                             "roofline": {"bound": "hbm", "kernel": "store_kvcache_kernel",
                                          "achieved": sbytes / tks / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                          "frac": sbytes / tks / 1e9 / peaks["hbm_gbs"], "kernel_ms": tks * 1e3,
                                          "traffic": ncu_traffic("store", float(cfg.new.sum()))},
                             "tokens": int(cfg.new.sum())},
           "store_kvcache_8x": {"workload": f"{n8} tokens (the step's new tokens 8 times over) into random distinct "
                                            "slots of the pool, K, V and V/16 rows",
                                "value": sb8 / t8 / 1e9, "unit": "GB/s", "ms_per_step": t8 * 1e3,
                                "algorithmic_bytes": sb8,
                                "roofline": {"bound": "hbm", "kernel": "store_kvcache_kernel",
                                             "achieved": sb8 / tk8 / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                             "frac": sb8 / tk8 / 1e9 / peaks["hbm_gbs"], "kernel_ms": tk8 * 1e3}},
           "launches_per_step": 3}
    del kc, vc, v16
    torch.cuda.empty_cache()
    if with_oracle:
        # the oracle on 6 sequences (3 of them sharing the prefix), 1/16 of their query rows,
        # after its own store of their new tokens into a compact pool
        import oracle
        oracle.build()
        seqs = [0, 3, 7, 12, 20, 31]
        kp, vp, btc = workloads.compact_paged(cfg, seqs)
        bs = cfg.block_size
        cu_new = workloads.cu_from_lens(cfg.new)
        sl, tok = [], []
        for r, b in enumerate(seqs):
            j = np.arange(int(cfg.ctx[b]), int(cfg.ctx[b] + cfg.new[b]))
            sl.append(btc[r, j // bs].astype(np.int64) * bs + j % bs)
            tok.append(np.arange(cu_new[b], cu_new[b + 1]))
        sl, tok = np.concatenate(sl), np.concatenate(tok)
        kb, vb = oracle.store_kvcache(k_new_h[tok], v_new_h[tok], kp, vp, sl)
        kb, vb = kb.reshape(kp.shape), vb.reshape(vp.shape)
        qs = qh[torch.from_numpy(tok)]
        lq, lk = cfg.new[seqs], cfg.lens_k[seqs]
        cq, ckk = workloads.cu_from_lens(lq), workloads.cu_from_lens(lk)
        rows = workloads.sample_rows(cfg.seed + 12, len(tok) * cfg.Hq, 1 / 16)
        sec, n = oracle_timed(lambda: oracle.attn_varlen(qs, kb, vb, cq, ckk, cfg.Hq, cfg.Hkv, cfg.D, cfg.scale, True,
                                                         block_table=btc, block_size=bs, num_blocks=kp.shape[0],
                                                         rows=rows), 1.0)
        fl = rows_flops_lens(lq, lk, cfg.Hq, cfg.D, rows)
        res["oracle"] = oracle_line(fl / sec / 1e12, "TFLOP/s", f"{len(rows)} query rows (1/16) of 6 of the 32 "
                                    f"sequences, paged through a compact pool; {fl / 1e9:.1f} GFLOP, mean of {n} "
                                    f"calls; float64, OpenMP", sec)
    return res


def bench_padded(av, device, steps, warmup, flush, peaks):
    """c2_varlen_gqa as a padded batch [16, 4096, H, D] with per-sequence lengths."""
    import torch
    cfg = workloads.make("c2_varlen_gqa")
    S = 4096
    B = cfg.batch
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    qp = torch.zeros(B, S, cfg.Hq, cfg.D, dtype=torch.bfloat16)
    kp = torch.zeros(B, S, cfg.Hkv, cfg.D, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    for b in range(B):
        qp[b, :cfg.lens_q[b]] = q[cfg.cu_q[b]:cfg.cu_q[b + 1]]
        kp[b, :cfg.lens_k[b]] = k[cfg.cu_k[b]:cfg.cu_k[b + 1]]
        vp[b, :cfg.lens_k[b]] = v[cfg.cu_k[b]:cfg.cu_k[b + 1]]
    qp, kp, vp = qp.to(device), kp.to(device), vp.to(device)
    sq = torch.from_numpy(cfg.lens_q.astype(np.int32)).to(device)
    sk = torch.from_numpy(cfg.lens_k.astype(np.int32)).to(device)
    out = torch.empty_like(qp)
    ws = torch.empty(av.lib().attn_padded_workspace_size(B, S, S, cfg.Hq, cfg.Hkv, cfg.D), dtype=torch.uint8,
                     device=device)

    def step():
        av.attn_padded_fwd(qp, kp, vp, sq, sk, cfg.scale, out=out, workspace=ws)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = time_steps(step, steps, flush)
    t = float(np.mean(ms)) / 1e3
    flops = workloads.prefill_flops(cfg.lens_q, cfg.lens_k, cfg.Hq, cfg.D)
    del qp, kp, vp, out, ws
    torch.cuda.empty_cache()
    return {"workload": "c2_varlen_gqa as a padded batch [16, 4096, 32|8, 128] with per-sequence lengths",
            "value": flops / t / 1e12, "unit": "TFLOP/s", "ms_per_step": t * 1e3,
            "frac": flops / t / 1e12 / peaks["bf16_tflops"], "launches_per_step": 3}


def bench_softmax(av, device, steps, warmup, flush, peaks):
    """Row softmax (online two-pass kernel): algorithmic bytes = one read and one
    write of the matrix."""
    import torch
    res = {}
    for name, rows, cols, dt, kern in (("f32_32768x8192", 32768, 8192, torch.float32, "softmax_cta_reg"),
                                       ("bf16_262144x1024", 262144, 1024, torch.bfloat16, "softmax_warp"),
                                       ("f32_4096x65536", 4096, 65536, torch.float32, "softmax_cluster")):
        g = torch.Generator(device=device).manual_seed(1234 + rows)
        x = (torch.randn(rows, cols, device=device, generator=g) * 30.0).to(dt)
        y = torch.empty_like(x)

        def step():
            av.softmax_rows(x, out=y)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        ms = time_steps(step, steps, flush)
        t = float(np.mean(ms)) / 1e3
        nbytes = 2 * x.numel() * x.element_size()
        gbs = nbytes / t / 1e9
        res[name] = {"value": gbs, "unit": "GB/s", "ms_per_step": t * 1e3, "algorithmic_bytes": nbytes,
                     "roofline": {"bound": "hbm", "kernel": {"softmax_cta_reg": "softmax_rows_cta_reg_kernel",
                                                             "softmax_warp": "softmax_rows_warp_kernel",
                                                             "softmax_cluster": "softmax_rows_cta_reg_kernel (cluster of 8)"}[kern],
                                  "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gbs / peaks["hbm_gbs"], "traffic": ncu_traffic(kern, x.numel())},
                     "launches_per_step": 1}
        del x, y
    torch.cuda.empty_cache()
    res["workload"] = ("row softmax, N(0, 30^2) logits, each row read once and held in registers: fp32 32768 x 8192 "
                       "(a CTA per row), bf16 262144 x 1024 (a warp per row), fp32 4096 x 65536 (a cluster of 8 CTAs "
                       "per row)")
    return res


def bench_contig(av, name, device, steps, warmup, flush, peaks, with_oracle=True):
    """A contiguous varlen workload (c1_tiny, c5_long) through attn_varlen_fwd,
    with the oracle on the whole workload (c1) or 4 (sequence, head) pairs (c5)."""
    import torch
    cfg = workloads.make(name)
    qh, kh, vh = cfg.q(), cfg.k(), cfg.v()
    inp = dict(q=qh.to(device), k=kh.to(device), v=vh.to(device), cu_q=torch.from_numpy(cfg.cu_q).to(device),
               cu_k=torch.from_numpy(cfg.cu_k).to(device), mq=int(cfg.lens_q.max()), mk=int(cfg.lens_k.max()))
    ms, _, kms = bench_varlen(av, cfg, inp, steps, warmup, flush)
    flops = workloads.prefill_flops(cfg.lens_q, cfg.lens_k, cfg.Hq, cfg.D)
    t = float(np.mean(ms)) / 1e3
    tk = float(np.mean(kms)) / 1e3
    desc = {"c1_tiny": "c1_tiny: the article's example, cu_seqlens_q [0,5,7,8], cu_seqlens_k [0,9,16,19], 4 heads, "
                       "D64 (launch-bound: 52 kFLOP)",
            "c5_long": "c5_long: 2 x 32768 tokens, MHA 32 heads, D128, heads 0-15 with Q x160 (logits ~700)"}[name]
    res = {"workload": desc, "value": flops / t / 1e12, "unit": "TFLOP/s", "ms_per_step": t * 1e3,
           "algorithmic_flops": flops,
           "roofline": {"bound": "tensor", "kernel": "attn_prefill_kernel", "achieved": flops / tk / 1e12,
                        "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": flops / tk / 1e12 / peaks["bf16_tflops"], "kernel_ms": tk * 1e3,
                        "traffic": None, "peak_source": "measured bf16 burst"},
           "launches_per_step": 2}
    del inp
    torch.cuda.empty_cache()
    if with_oracle:
        import oracle
        oracle.build()
        if name == "c1_tiny":
            sec, n = oracle_timed(lambda: oracle.attn_varlen(qh, kh, vh, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D,
                                                             cfg.scale, True), 0.5)
            res["oracle"] = oracle_line(flops / sec / 1e12, "TFLOP/s", f"the whole workload (32 query rows), mean "
                                        f"of {n} calls; float64, OpenMP", sec)
        else:
            rng = np.random.default_rng(cfg.seed + 13)
            rows = []
            for b, h in [(0, 3), (1, 12), (0, 20), (1, 31)]:
                i = np.sort(rng.choice(int(cfg.lens_q[b]), 256, replace=False))
                rows.append((int(cfg.cu_q[b]) + i) * cfg.Hq + h)
            rows = np.concatenate(rows).astype(np.int64)
            sec, n = oracle_timed(lambda: oracle.attn_varlen(qh, kh, vh, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D,
                                                             cfg.scale, True, rows=rows), 1.0)
            fl = rows_flops_lens(cfg.lens_q, cfg.lens_k, cfg.Hq, cfg.D, rows)
            res["oracle"] = oracle_line(fl / sec / 1e12, "TFLOP/s", f"{len(rows)} query rows: 256 of each of 4 "
                                        f"(sequence, head) pairs, two with logits ~700; {fl / 1e9:.1f} GFLOP, mean "
                                        f"of {n} calls; float64, OpenMP", sec)
    return res


# --------------------------------------------------------------------------
# the oracle on this host (CPU baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_sample_run(cfg, q, k, v, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.attn_varlen(q, k, v, cfg.cu_q, cfg.cu_k, cfg.Hq, cfg.Hkv, cfg.D, cfg.scale, True, rows=rows)
    return time.perf_counter() - t0


def rows_flops_lens(lens_q, lens_k, Hq, D, rows):
    """Algorithmic flops of sampled query rows (row id = token * Hq + head of a
    varlen packing with these lengths): 4 * D * visible keys each."""
    lens_q = np.asarray(lens_q, dtype=np.int64)
    lens_k = np.asarray(lens_k, dtype=np.int64)
    cu = workloads.cu_from_lens(lens_q)
    t = np.asarray(rows, dtype=np.int64) // Hq
    b = np.searchsorted(cu, t, side="right") - 1
    i = t - cu[b]
    vis = np.clip(lens_k[b] - lens_q[b] + i + 1, 0, lens_k[b])
    return float(4 * D * vis.sum())


def rows_flops(cfg, rows):
    return rows_flops_lens(cfg.lens_q, cfg.lens_k, cfg.Hq, cfg.D, rows)


def cpu_baseline(cfg, q, k, v, target_s: float = 8.0):
    import oracle
    oracle.build()
    n_rows = q.shape[0] * cfg.Hq
    cal = workloads.sample_rows(cfg.seed + 77, n_rows, 1.0, cap=2000)
    t_cal = oracle_sample_run(cfg, q, k, v, cal)
    rate = rows_flops(cfg, cal) / max(t_cal, 1e-6)
    per_row = rows_flops(cfg, cal) / len(cal)
    n = int(min(n_rows, max(2000, target_s * rate / per_row)))
    rows = workloads.sample_rows(cfg.seed + 78, n_rows, 1.0, cap=n)
    t = oracle_sample_run(cfg, q, k, v, rows)
    fl = rows_flops(cfg, rows)
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(rows)} of {n_rows} query rows (uniform over sequence, head, position) of "
                      f"{cfg.name}; {fl / 1e9:.1f} GFLOP in {t:.1f} s; float64 three-step attention, OpenMP",
            "seconds": t}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = workloads.make("c2_varlen_gqa")
    q, k, v = cfg.q(), cfg.k(), cfg.v()
    import oracle
    oracle.build()
    n_rows = q.shape[0] * cfg.Hq
    # each step: a bounded sample (about 2 s of host time)
    cal = workloads.sample_rows(cfg.seed + 90, n_rows, 1.0, cap=1000)
    t_cal = oracle_sample_run(cfg, q, k, v, cal)
    n = int(min(n_rows, max(500, 2.0 / max(t_cal, 1e-6) * len(cal))))
    for w in range(args.warmup):
        oracle_sample_run(cfg, q, k, v, workloads.sample_rows(cfg.seed + 100 + w, n_rows, 1.0, cap=n))
    times, flops = [], []
    for s in range(args.steps):
        rows = workloads.sample_rows(cfg.seed + 200 + s, n_rows, 1.0, cap=n)
        times.append(oracle_sample_run(cfg, q, k, v, rows))
        flops.append(rows_flops(cfg, rows))
    value = sum(flops) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "c2_varlen_gqa", "global_batch": 16, "seq_len": "U{256..4096}",
                       "sample_rows_per_step": n},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{n} query rows per step of c2_varlen_gqa"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _r(x, nd=4):
    """Round for the compact summary (significant digits)."""
    if x is None or not isinstance(x, (int, float)) or x == 0 or not math.isfinite(x):
        return x
    return float(f"{x:.{nd}g}")


def summary(line, peaks, peak_src):
    """Compact per-workload table: step value, dominant-kernel value, roofline
    fraction (against the measured peaks) and the oracle's value, one entry per
    workload, so that the end of the line carries every number."""
    out = {}

    def put(key, d, oracle=None, extra=None):
        if not d:
            return
        rf = d.get("roofline", {})
        e = {"value": _r(d.get("value")), "unit": d.get("unit"), "kernel": _r(rf.get("achieved")),
             "frac": _r(rf.get("frac", d.get("frac")), 3), "ms": _r(d.get("ms_per_step"))}
        if oracle:
            e["oracle"] = _r(oracle.get("value"))
        if extra:
            e.update(extra)
        out[key] = {k: v for k, v in e.items() if v is not None}

    main = {"value": line["value"], "unit": "TFLOP/s", "roofline": line["roofline"], "ms_per_step": line["ms_per_step"]}
    put("c2", main, line.get("cpu_baseline"), {"step_frac": _r(line["value"] / peaks["bf16_tflops"], 3),
                                               "e2e": _r(line["e2e"]["value"])})
    put("c1", line.get("tiny_prefill"), (line.get("tiny_prefill") or {}).get("oracle"))
    c3 = line.get("prefix_prefill")
    if c3:
        put("c3", c3, c3.get("oracle"), {"step_frac": _r(c3["value"] / peaks["bf16_tflops"], 3),
                                         "no_v16": _r(c3["without_v16_cache"]["value"]),
                                         "hbm_frac": _r(c3["hbm"]["frac"], 3),
                                         "tmin_frac": _r(c3["roofline_tmin_frac"], 3)})
        put("c3_store", c3["store_kvcache"])
        put("store_8x", c3.get("store_kvcache_8x"))
    c4 = line.get("decode")
    if c4:
        put("c4", c4, c4.get("oracle"))
        put("c4_sq4", c4.get("kvcache_4_tokens"))
        put("c4_sq8", c4.get("kvcache_8_tokens"))
        put("c4_sq4_v16", c4.get("kvcache_4_tokens_v16"))
        put("c4_sq8_v16", c4.get("kvcache_8_tokens_v16"))
        put("c4_sq16", c4.get("kvcache_16_tokens"))
        put("c4_sq16_v16", c4.get("kvcache_16_tokens_v16"))
    c5 = line.get("long_prefill")
    if c5:
        put("c5", c5, c5.get("oracle"), {"step_frac": _r(c5["value"] / peaks["bf16_tflops"], 3)})
    sm = line.get("row_softmax")
    if sm:
        put("softmax_f32", sm.get("f32_32768x8192"))
        put("softmax_bf16", sm.get("bf16_262144x1024"))
        put("softmax_f32_long", sm.get("f32_4096x65536"))
    put("padded", line.get("padded_prefill"))
    out["peaks"] = {"bf16_burst_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"], "source": peak_src}
    return out


# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only-main", action="store_true", help="skip the extra workloads")
    ap.add_argument("--no-oracle", action="store_true", help="skip the oracle timings")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    rank, local_rank, world = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist_init("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    import attention_attn_varlen_gb300 as av
    av.build()
    av.lib()
    peaks, peak_src = load_peaks()
    with_oracle = rank == 0 and world == 1 and not args.no_oracle

    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def flush():
        flush_buf.zero_()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()

    cfg = workloads.make("c2_varlen_gqa")
    if rank:
        # an independent batch per rank (same shapes, other values)
        cfg.seed += 1000 * rank
    inp = varlen_inputs(cfg, device)
    flops = workloads.prefill_flops(cfg.lens_q, cfg.lens_k, cfg.Hq, cfg.D)
    ms, wall, kms = bench_varlen(av, cfg, inp, args.steps, args.warmup, flush)
    ms_mean = float(np.mean(ms))
    ms_max = dist_max(ms_mean, device)
    value = aggregate(flops, ms_max / 1e3, world) / 1e12
    kernel_ms = float(np.mean(kms))
    achieved = flops / (kernel_ms / 1e3) / 1e12
    e2e_ms, h2d, d2h = bench_varlen_e2e(av, cfg, inp, args.steps, args.warmup, flush)
    e2e_max = dist_max(float(np.mean(e2e_ms)), device)
    del inp
    torch.cuda.empty_cache()

    extras = {}
    if not args.only_main:
        extras["tiny_prefill"] = bench_contig(av, "c1_tiny", device, args.steps, args.warmup, flush, peaks,
                                              with_oracle)
        extras["decode"] = bench_decode(av, device, args.steps, args.warmup, flush, peaks, with_oracle)
        extras["prefix_prefill"] = bench_prefix(av, device, args.steps, args.warmup, flush, peaks, with_oracle)
        extras["long_prefill"] = bench_contig(av, "c5_long", device, max(3, args.steps // 3), args.warmup, flush,
                                              peaks, with_oracle)
        extras["row_softmax"] = bench_softmax(av, device, args.steps, args.warmup, flush, peaks)
        extras["padded_prefill"] = bench_padded(av, device, args.steps, args.warmup, flush, peaks)
    clocks = sampler.stop()

    status, word = av.get_last_device_error()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "c2_varlen_gqa: varlen causal prefill, 16 seqs, L ~ U{256..4096} (Lq = Lk), "
                               "GQA 32/8, head_dim 128, bf16, packed by cu_seqlens",
                   "global_batch": 16 * world, "seq_len": "U{256..4096}", "total_tokens": int(cfg.lens_q.sum()),
                   "algorithmic_flops": flops, "l2": "flushed between timed steps (512 MB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "attn_prefill_kernel", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "kernel_ms": kernel_ms,
                     "traffic": ncu_traffic("prefill", float(cfg.lens_q.sum())),
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 1.9 PFLOP/s"},
        "e2e": {"value": aggregate(flops, e2e_max / 1e3, world) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_max,
                "path": "C entry attn_varlen_fwd_host: pinned host q/k/v in, host out, 8 overlapped groups"},
        # per step: the pre-pass (unit list + fp16 V') and the attention kernel
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
        "device_status": status,
    }
    line.update(extras)
    if with_oracle:
        line["cpu_baseline"] = cpu_baseline(cfg, cfg.q(), cfg.k(), cfg.v())
    line["summary"] = summary(line, peaks, peak_src)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist_barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
