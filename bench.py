#!/usr/bin/env python3
"""Benchmark of the KIVI decode hot path on GB300.

One step = one decode step of the whole path for every sequence of the
batch: kivi_append_flush appends one new K/V token per sequence (quantizing
and packing a G-token group whenever the residual window overflows), then
kivi_decode_attn runs split-K decode attention over the packed cache.

Default workload: Llama-3-8B GQA decode layer shape, 64 sequences, 32 query
heads over 8 kv heads, head_dim 128, 32768 cached tokens per sequence, bf16
inputs, 2-bit codes, G = 32, R = 128 (--bits, --k-bits, --v-bits, --group and
--residual select the other settings). Inputs are synthetic and seeded; the
cache (about 1.64 GB) is larger than L2, so no flush is needed between steps.

Prints one JSON line. value = KV tokens attended per second over the timed
steps (sum over sequences of kv_len, per step, divided by the step time).
The roofline object is for the decode-attention kernel, from its own CUDA
event timings inside the timed region.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the only CPU-side arm; there is no other implementation).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-tokens/s and achieved HBM GB/s (% of GB300 peak), 2-bit KIVI cache"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- workload
WORKLOAD_NAMES = {0: "tiny decode", 1: "Llama-2-7B MHA decode step", 2: "Llama-3-8B GQA decode step",
                  3: "streaming append + decode step", 4: "long varlen (Mistral-7B shape) decode step"}


def workload_spec(args):
    import synth
    wl = synth.workload(getattr(args, "workload", 2))
    if args.batch:
        wl = wl.replace(batch=args.batch, lengths=(args.context or wl.lengths[0],) * args.batch)
    if args.context:
        wl = wl.replace(lengths=(args.context,) * wl.batch)
    if args.bits:
        wl = wl.replace(bits=args.bits)
    if args.group:
        wl = wl.replace(group=args.group)
    if args.residual:
        wl = wl.replace(residual=args.residual)
    if getattr(args, "q_heads", 0):
        if args.q_heads % wl.num_kv_heads:
            raise SystemExit(f"--q-heads must be a multiple of the {wl.num_kv_heads} kv heads")
        wl = wl.replace(num_q_heads=args.q_heads)
    return wl


def kv_bits(args, wl):
    """Key and value code widths: --k-bits / --v-bits where given, else the workload's."""
    return (getattr(args, "k_bits", 0) or wl.bits), (getattr(args, "v_bits", 0) or wl.bits)


def attn_bytes(wl, lengths, kb, vb):
    """Algorithmic bytes one decode launch must read: per packed (token, kv head) the key
    and value codes (D kb / 8 + D vb / 8 B) and the fp16 scale and zero shares of keys and
    values (2 * 2 * 2 * D / G B): 96 B at 2 bits and G = 32 (32 + 16 + 32 + 16), 160 B at
    4 bits; 512 B per residual token (fp16/bf16 K and V)."""
    R, G, D, H = wl.residual, wl.group, wl.head_dim, wl.num_kv_heads
    per_packed = (D * kb // 8 + D * vb // 8) + 2 * 2 * 2 * D // G
    total = 0
    for L in lengths:
        npk = G * (max(L - R, 0) // G)
        total += H * (npk * per_packed + (L - npk) * 2 * D * 2)
    return total


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per (token, kv head) of one
# decode launch, from ncu captures of the kernels in their current version on the 8-sequence
# case of the Llama-3-8B GQA workload (2-bit, bf16): 209.11 MB for 8 x 8 x 32772 units at
# query group 4, and 415.19 MB for 16 x 8 x 32772 units at query group 8 (64 query heads).
# Keyed by (kernel, k_bits, v_bits, G, R, query group, input dtype); a configuration without
# an entry reports traffic as null.
NCU_TRAFFIC_BYTES_PER_UNIT = {
    ("decode_mma_kernel", 2, 2, 32, 128, 4, "bf16"): 209_112_832 / (8 * 8 * 32772),
    ("decode_mma_kernel", 2, 2, 32, 128, 8, "bf16"): 415_185_408 / (16 * 8 * 32772),
}


def reduce_max(x: float, device=None) -> float:
    """Max of x over the ranks of the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job rate under weak scaling: every rank processed units_per_rank in at most max_ms."""
    return units_per_rank * world / (max_ms / 1e3)


def prefill_io_bytes(wl, L, kb, vb):
    """Algorithmic bytes of appending L tokens to an empty sequence: the K and V inputs read,
    the packed codes and fp16 scale/zero written for n_packed(L) tokens, the ring rows written."""
    R, G, D, H = wl.residual, wl.group, wl.head_dim, wl.num_kv_heads
    npk = G * (max(L - R, 0) // G)
    read = 2 * L * D * 2
    written = npk * (D * kb // 8 + D * vb // 8 + 2 * 2 * 2 * D // G) + (L - npk) * 2 * D * 2
    return H * (read + written)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ---------------------------------------------------------------- GPU arm
def smi_id(device) -> str:
    """nvidia-smi --id of a torch device: its PCI bus id when torch reports one."""
    import torch
    p = torch.cuda.get_device_properties(device)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return str(device.index or 0)


def gen_sequence_kv(wl, b, L, device):
    """K, V of sequence b for all kv heads, [Hkv][L][D], drawn on the GPU."""
    import torch
    import synth
    K = torch.stack([synth.torch_kv_head_major(wl, b, h, 0, L, "k", device) for h in range(wl.num_kv_heads)])
    V = torch.stack([synth.torch_kv_head_major(wl, b, h, 0, L, "v", device) for h in range(wl.num_kv_heads)])
    return K, V


def step_inputs(wl, L0s, n_steps, device):
    """New K/V tokens ([steps][B][Hkv][1][D]) at positions L0s[b] + s and queries ([steps][B][Hq][D])."""
    import torch
    import synth
    B, H, D = wl.batch, wl.num_kv_heads, wl.head_dim
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    kn = torch.empty((n_steps, B, H, 1, D), dtype=tdt, device=device)
    vn = torch.empty_like(kn)
    for b in range(B):
        for h in range(H):
            kn[:, b, h, 0] = synth.torch_kv_head_major(wl, b, h, L0s[b], n_steps, "k", device)
            vn[:, b, h, 0] = synth.torch_kv_head_major(wl, b, h, L0s[b], n_steps, "v", device)
    q = torch.stack([torch.from_numpy(wl.query(s).view(np.int16)).view(tdt) for s in range(n_steps)]).to(device)
    return kn, vn, q


def run_gpu(args, rank, world, local_rank, full=True):
    """The timed decode steps of one workload. full=False (the per-workload lines) skips the
    end-to-end leg."""
    import torch
    import bit_asymmetric_kv_kivi_gb300 as kivi

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workload_spec(args)
    B, Hq, H, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    kb, vb = kv_bits(args, wl)
    L0s = list(wl.lengths)
    L0 = max(L0s)
    n_steps = args.warmup + args.steps
    G = wl.group
    cap = ((L0 + n_steps + args.steps + G - 1) // G) * G   # decode steps of both timed legs
    cfg = kivi.Config(k_bits=kb, v_bits=vb, group=G, residual=wl.residual, head_dim=D, num_q_heads=Hq,
                      num_kv_heads=H, dtype=kivi.BF16 if wl.dtype == "bf16" else kivi.F16)
    cache = kivi.KVCache(cfg, B, cap, device, paged=args.paged, page_seed=1)

    # prefill (outside the timed steps): every sequence's K and V drawn on the GPU, then one
    # append call for the whole batch, timed on its own for the prefill line of the report.
    # The first call loads the kernels; the cache is then emptied and the same call timed.
    ks, vs = [], []
    for b in range(B):
        K, V = gen_sequence_kv(wl, b, L0s[b], device)
        ks.append(K)
        vs.append(V)
    kp = torch.tensor([k.data_ptr() for k in ks], dtype=torch.int64, device=device)
    vp = torch.tensor([v.data_ptr() for v in vs], dtype=torch.int64, device=device)
    nn = torch.tensor(L0s, dtype=torch.int32, device=device)
    cache.append_ptrs(kp, vp, nn, L0)
    torch.cuda.synchronize()
    cache.kv_len.zero_()
    cache.max_len = 0
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record()
    cache.append_ptrs(kp, vp, nn, L0)
    pe1.record()
    torch.cuda.synchronize()
    prefill_ms = pe0.elapsed_time(pe1)
    prefill_bytes = sum(prefill_io_bytes(wl, L, kb, vb) for L in L0s)
    del ks, vs
    torch.cuda.synchronize()
    cache.max_len = L0
    assert int(cache.status.item()) == 0, cache.status.item()

    kn, vn, q = step_inputs(wl, L0s, n_steps, device)
    ones = torch.ones(B, dtype=torch.int32, device=device)
    kptr = [torch.tensor([kn[s, b].data_ptr() for b in range(B)], dtype=torch.int64, device=device)
            for s in range(n_steps)]
    vptr = [torch.tensor([vn[s, b].data_ptr() for b in range(B)], dtype=torch.int64, device=device)
            for s in range(n_steps)]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
    max_len_final = L0 + n_steps
    ws = cache.workspace(max_len_final)
    stream = torch.cuda.current_stream(device)

    # caches smaller than twice the 129 MB L2 are flushed (a 512 MB write) before every
    # step, outside the per-step timing
    cache_bytes = attn_bytes(wl, L0s, kb, vb)
    flush = cache_bytes < 256 << 20
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=device) if flush else None
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

    def step(s, ev_a=None, ev_b=None):
        cache.append_ptrs(kptr[s], vptr[s], ones, 1)
        if ev_a is not None:
            ev_a.record(stream)
        cache.decode(q[s], out, wl.softmax_scale, max_kv_len=max_len_final)
        if ev_b is not None:
            ev_b.record(stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    attn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(smi_id(device)) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            if flush:
                flush_buf.zero_()
            step_ev[i][0].record(stream)
            step(args.warmup + i, *attn_ev[i])
            step_ev[i][1].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = sum(a.elapsed_time(b) for a, b in step_ev) if flush else ev0.elapsed_time(ev1)
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    assert int(cache.status.item()) == 0, cache.status.item()

    lens_per_step = [[L + args.warmup + i + 1 for L in L0s] for i in range(args.steps)]
    kv_tokens = sum(sum(ls) for ls in lens_per_step)
    bytes_per_step = [attn_bytes(wl, ls, kb, vb) for ls in lens_per_step]
    units_per_step = [wl.num_kv_heads * sum(ls) for ls in lens_per_step]

    # ------------------------------------------------------------ end to end through the public API
    e2e = run_e2e(args, cache, wl, device, [L + n_steps for L in L0s], max_len_final + args.steps, out) if full \
        else None

    res = {
        "total_ms": total_ms, "attn_ms": attn_ms, "kv_tokens": kv_tokens, "attn_bytes": bytes_per_step,
        "attn_units": units_per_step,
        "clocks": clk.summary(), "e2e": e2e, "cap": cap, "flush": flush,
        # the one-launch append, then decode_mma_kernel and its merge kernel (query groups 1, 2,
        # 4 and 8) or decode_multi_kernel (other groups)
        "launches_per_step": 1 + (2 if Hq // H in (1, 2, 4, 8) else 1),
        "prefill": {"ms": prefill_ms, "algorithmic_bytes": prefill_bytes,
                    "GBps": prefill_bytes / (prefill_ms / 1e3) / 1e9 if prefill_ms > 0 else None},
    }
    return res, wl


def run_gpu_multi(args, rank, world, local_rank):
    """Verification steps (--n-query N): each step appends N tokens per sequence (the draft
    tokens of a speculative decoder) and runs kivi_decode_multi_attn for their N queries,
    each attending causally to the cache. Returns the JSON line's fields."""
    import torch
    import synth
    import bit_asymmetric_kv_kivi_gb300 as kivi

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = workload_spec(args)
    B, Hq, H, D, N = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, args.n_query
    kb, vb = kv_bits(args, wl)
    G = wl.group
    L0s = list(wl.lengths)
    n_steps = args.warmup + args.steps
    max_len = max(L0s) + n_steps * N
    cap = ((max_len + G - 1) // G) * G
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    cfg = kivi.Config(k_bits=kb, v_bits=vb, group=G, residual=wl.residual, head_dim=D, num_q_heads=Hq,
                      num_kv_heads=H, dtype=kivi.BF16 if wl.dtype == "bf16" else kivi.F16)
    cache = kivi.KVCache(cfg, B, cap, device, paged=args.paged, page_seed=1)
    ks, vs = zip(*(gen_sequence_kv(wl, b, L0s[b], device) for b in range(B)))
    cache.append(list(ks), list(vs))
    del ks, vs
    # each step's N new tokens per sequence, contiguous [Hkv][N][D], and its queries [B][N][Hq][D]
    kst, vst = [], []
    for b in range(B):
        kall = torch.stack([synth.torch_kv_head_major(wl, b, h, L0s[b], n_steps * N, "k", device) for h in range(H)])
        vall = torch.stack([synth.torch_kv_head_major(wl, b, h, L0s[b], n_steps * N, "v", device) for h in range(H)])
        kst.append([kall[:, s * N:(s + 1) * N].contiguous() for s in range(n_steps)])
        vst.append([vall[:, s * N:(s + 1) * N].contiguous() for s in range(n_steps)])
    kptr = [torch.tensor([kst[b][s].data_ptr() for b in range(B)], dtype=torch.int64, device=device)
            for s in range(n_steps)]
    vptr = [torch.tensor([vst[b][s].data_ptr() for b in range(B)], dtype=torch.int64, device=device)
            for s in range(n_steps)]
    q = [torch.from_numpy(np.stack([wl.query(s * N + i) for i in range(N)], axis=1).view(np.int16)).view(tdt).to(device)
         for s in range(n_steps)]
    nn = torch.full((B,), N, dtype=torch.int32, device=device)
    out = torch.empty((B, N, Hq, D), dtype=torch.float32, device=device)
    cache.decode_multi(q[0], out, wl.softmax_scale, max_kv_len=max_len)    # sizes the workspace
    stream = torch.cuda.current_stream(device)
    cache_bytes = attn_bytes(wl, L0s, kb, vb)
    flush = cache_bytes < 256 << 20
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=device) if flush else None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(s, e=None):
        if e is not None:
            e[0].record(stream)
        cache.append_ptrs(kptr[s], vptr[s], nn, N)
        if e is not None:
            e[1].record(stream)
        cache.decode_multi(q[s], out, wl.softmax_scale, max_kv_len=max_len)
        if e is not None:
            e[2].record(stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    with ClockSampler(smi_id(device)) as clk:
        for i in range(args.steps):
            if flush:
                flush_buf.zero_()
            step(args.warmup + i, ev[i])
        torch.cuda.synchronize()
    assert int(cache.status.item()) == 0, cache.status.item()
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    attn_ms = [e[1].elapsed_time(e[2]) for e in ev]
    lens = [[L + (args.warmup + i + 1) * N for L in L0s] for i in range(args.steps)]
    pairs = [sum(N * L - N * (N - 1) // 2 for L in ls) for ls in lens]      # (query, visible token) pairs
    nbytes = [attn_bytes(wl, ls, kb, vb) for ls in lens]
    total_ms = sum(step_ms)
    value = sum(pairs) * world / (total_ms / 1e3)
    avg_ms = sum(attn_ms) / len(attn_ms)
    achieved = sum(nbytes) / len(nbytes) / (avg_ms / 1e3) / 1e9
    # one query at query groups 1, 2, 4 and 8, several queries at groups 4 and 8, and two queries
    # at groups 1 and 2 run on the decode kernel
    on_mma = (N == 1 and Hq // H in (1, 2, 4, 8)) or (N > 1 and Hq // H in (4, 8)) or (N == 2 and Hq // H in (1, 2))
    peak, peak_kind = measured_hbm_peak()
    return {
        "metric": f"verification step ({N} queries per sequence): query x KV-token pairs/s", "value": value,
        "unit": "query-KV-pairs/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD_NAMES[args.workload]} with {N} draft tokens appended and verified per step: "
                               f"{B} sequences from {L0s[0]} tokens, {Hq} query / {H} kv heads, {kb}/{vb}-bit K/V, "
                               f"G={G}, R={wl.residual}, {wl.dtype}", "n_query": N,
                   "l2": "flushed before every step" if flush else "no flush: the cache is larger than L2",
                   "layout": "paged" if args.paged else "contiguous"},
        "roofline": {"bound": "hbm", "kernel": "decode_mma_kernel" if on_mma else "decode_multi_kernel",
                     "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "avg_launch_ms": avg_ms,
                     "algorithmic_bytes_per_launch": sum(nbytes) / len(nbytes), "traffic": None},
        "attn_pairs_per_s": sum(pairs) / (sum(attn_ms) / 1e3),
        # the append (one launch up to G new tokens, three beyond), then decode_mma_kernel and its
        # merge kernel, or decode_multi_kernel
        "gpu_launches": ((1 if N <= wl.group else 3) + (2 if on_mma else 1)) * args.steps, "clocks": clk.summary(),
    }


def run_e2e(args, cache, wl, device, L_start, max_len, out_dev):
    """Same step through the public API, with every step's inputs copied host -> device from
    pinned memory and its attention output copied back, inside the timed region. The copies
    run on two copy streams (in and out) and overlap the compute of the neighbouring steps:
    inputs and outputs are double-buffered, and events order each buffer's copy-in, use and
    copy-out."""
    import torch
    B, Hq, H, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    n = min(args.steps, 50)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    kn, vn, q = step_inputs(wl, L_start, n, device)
    kh, vh, qh = kn.cpu().pin_memory(), vn.cpu().pin_memory(), q.cpu().pin_memory()
    out_h = torch.empty((n, B, Hq, D), dtype=torch.float32).pin_memory()
    kd = [torch.empty((B, H, 1, D), dtype=tdt, device=device) for _ in range(2)]
    vd = [torch.empty_like(kd[0]) for _ in range(2)]
    qd = [torch.empty((B, Hq, D), dtype=tdt, device=device) for _ in range(2)]
    od = [out_dev, torch.empty_like(out_dev)]
    kptr = [torch.tensor([kd[i][b].data_ptr() for b in range(B)], dtype=torch.int64, device=device) for i in range(2)]
    vptr = [torch.tensor([vd[i][b].data_ptr() for b in range(B)], dtype=torch.int64, device=device) for i in range(2)]
    ones = torch.ones(B, dtype=torch.int32, device=device)
    compute = torch.cuda.current_stream(device)
    cin, cout = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer i copied in
    ev_used = [torch.cuda.Event() for _ in range(2)]    # buffer i's step done (inputs read, output written)
    ev_out = [torch.cuda.Event() for _ in range(2)]     # output of buffer i copied out

    def copy_in(s):
        i = s & 1
        with torch.cuda.stream(cin):
            if s >= 2:
                cin.wait_event(ev_used[i])              # step s - 2 has read kd/vd/qd[i]
            kd[i].copy_(kh[s], non_blocking=True)
            vd[i].copy_(vh[s], non_blocking=True)
            qd[i].copy_(qh[s], non_blocking=True)
            ev_in[i].record(cin)

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    copy_in(0)
    for s in range(n):
        i = s & 1
        compute.wait_event(ev_in[i])
        if s >= 2:
            compute.wait_event(ev_out[i])               # step s - 2's output has left od[i]
        cache.append_ptrs(kptr[i], vptr[i], ones, 1)
        cache.decode(qd[i], od[i], wl.softmax_scale, max_kv_len=max_len)
        ev_used[i].record(compute)
        if s + 1 < n:
            copy_in(s + 1)                              # overlaps this step's compute
        with torch.cuda.stream(cout):
            cout.wait_event(ev_used[i])
            out_h[s].copy_(od[i], non_blocking=True)
            ev_out[i].record(cout)
    cout.wait_stream(compute)
    cout.wait_stream(cin)
    e1.record(cout)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    kv_tokens = sum(sum(L + s + 1 for L in L_start) for s in range(n))
    h2d = (kd[0].numel() + vd[0].numel() + qd[0].numel()) * 2
    d2h = out_dev.numel() * 4
    return {"value": kv_tokens / (ms / 1e3), "unit": "KV-tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / n, "kv_tokens": kv_tokens, "steps": n,
            "copies": "copy-in and copy-out streams overlapping compute, double-buffered inputs and outputs"}


# ---------------------------------------------------------------- every workload in one line
# The sub-lines of the default run: each workload's decode steps (append + attention) timed
# as in the headline, fewer steps, no end-to-end leg. Workload 3 runs its 512 decode steps
# after the 16384-token prefill, at 2 and 4 bits.
SUB_WORKLOADS = (("0 tiny decode", 0, 0, 200), ("1 Llama-2-7B MHA", 1, 0, 200),
                 ("3 streaming 2-bit", 3, 2, 507), ("3 streaming 4-bit", 3, 4, 507),
                 ("4 long varlen", 4, 0, 100))


def run_workloads(args, rank, world, local_rank):
    import torch
    lines = {}
    for name, wi, bits, steps in SUB_WORKLOADS:
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup = wi, steps, 5
        sub.batch = sub.context = sub.q_heads = sub.group = sub.residual = sub.k_bits = sub.v_bits = 0
        sub.bits, sub.paged = bits, False
        res, wl = run_gpu(sub, rank, world, local_rank, full=False)
        kb, vb = kv_bits(sub, wl)
        avg_ms = sum(res["attn_ms"]) / len(res["attn_ms"])
        avg_bytes = sum(res["attn_bytes"]) / len(res["attn_bytes"])
        peak, peak_kind = measured_hbm_peak()
        gbps = avg_bytes / (avg_ms / 1e3) / 1e9
        lines[name] = {
            "workload": f"{WORKLOAD_NAMES[wi]}: {wl.batch} sequences, {wl.num_q_heads} query / {wl.num_kv_heads} kv "
                        f"heads, {kb}/{vb}-bit K/V, G={wl.group}, R={wl.residual}, {wl.dtype}",
            "steps": steps, "kv_tokens_per_s": res["kv_tokens"] / (res["total_ms"] / 1e3),
            "ms_per_step": res["total_ms"] / steps, "attn_kv_tokens_per_s": (res["kv_tokens"] / steps) / (avg_ms / 1e3),
            "attn_GBps": gbps, "frac": gbps / peak, "peak": peak, "peak_kind": peak_kind,
            "avg_launch_ms": avg_ms, "algorithmic_bytes_per_launch": avg_bytes,
            "l2": "flushed before every step" if res["flush"] else "no flush: the cache is larger than L2"}
        del res
        torch.cuda.empty_cache()
    return lines


# ---------------------------------------------------------------- CPU oracle arm
def oracle_sample(wl, n_steps, kb, vb, budget_s=20.0):
    """The oracle on a bounded sample of the workload: one sequence (all kv and query
    heads) prefilled to the workload's context, then n_steps decode steps of
    append + attention. Returns (KV-tokens/s, threads, description)."""
    import oracle
    oracle.build()
    L0 = wl.lengths[0]
    ocfg = oracle.Cfg(k_bits=kb, v_bits=vb, group=wl.group, residual=wl.residual, num_q_heads=wl.num_q_heads,
                      num_kv_heads=wl.num_kv_heads, dtype=oracle.BF16 if wl.dtype == "bf16" else oracle.F16)
    cap = ((L0 + n_steps + wl.group - 1) // wl.group) * wl.group
    seq = oracle.SeqCache(ocfg, cap)
    K, V = wl.kv_seq(0, 0, L0)
    assert seq.append(K, V) == oracle.OK
    Kn, Vn = wl.kv_seq(0, L0, n_steps)
    t0 = time.perf_counter()
    tokens = 0
    done = 0
    for s in range(n_steps):
        assert seq.append(np.ascontiguousarray(Kn[:, s:s + 1]), np.ascontiguousarray(Vn[:, s:s + 1])) == oracle.OK
        seq.decode(wl.query(s, 0), wl.softmax_scale)
        tokens += seq.L
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"oracle (C, fp32 codec + fp64 attention, OpenMP over query heads) on sequence 0 of the workload: "
            f"prefill {L0} tokens untimed, then {done} timed decode steps of append + attention "
            f"({wl.num_q_heads} query heads over {wl.num_kv_heads} kv heads)")
    return tokens / dt, threads, desc, dt


def oracle_parts(wl, kb, vb, runs=3, quant_tokens=2048):
    """The oracle timed in its two parts on sequence 0 of the workload, median of `runs`
    each: quantization (one append of `quant_tokens` tokens, every kv head, to an empty
    cache: codec, packing and the ring) and fp64 decode attention (every query head over the
    workload's context, prefilled untimed). Threads as the process runs them (OpenMP)."""
    import oracle
    oracle.build()
    L0 = wl.lengths[0]
    ocfg = oracle.Cfg(k_bits=kb, v_bits=vb, group=wl.group, residual=wl.residual, num_q_heads=wl.num_q_heads,
                      num_kv_heads=wl.num_kv_heads, dtype=oracle.BF16 if wl.dtype == "bf16" else oracle.F16)
    nq = min(quant_tokens, L0)
    Kq, Vq = wl.kv_seq(0, 0, nq)
    quant = []
    for _ in range(runs):
        seq = oracle.SeqCache(ocfg, ((nq + wl.group - 1) // wl.group) * wl.group)
        t0 = time.perf_counter()
        assert seq.append(Kq, Vq) == oracle.OK
        quant.append(time.perf_counter() - t0)
    cap = ((L0 + wl.group - 1) // wl.group) * wl.group
    seq = oracle.SeqCache(ocfg, cap)
    K, V = wl.kv_seq(0, 0, L0)
    assert seq.append(K, V) == oracle.OK
    attn = []
    for r in range(runs):
        t0 = time.perf_counter()
        seq.decode(wl.query(r, 0), wl.softmax_scale)
        attn.append(time.perf_counter() - t0)
    return statistics.median(quant), nq, statistics.median(attn), L0


def cpu_baseline(args, wl, kb, vb):
    """The cpu_baseline object of the JSON line (the oracle, as it stands, on this host)."""
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    v, _, desc, _ = oracle_sample(wl, 4, kb, vb, budget_s=20.0)
    quant_s, nq, attn_s, L0 = oracle_parts(wl, kb, vb)
    out = {"value": v, "unit": "KV-tokens/s", "cores": threads, "kind": "oracle", "sample": desc,
           "threads": threads, "runs": 3,
           "quant_s": quant_s, "quant_tokens": nq, "quant_tokens_per_s": nq / quant_s,
           "attn_s": attn_s, "attn_context": L0, "attn_kv_tokens_per_s": L0 / attn_s,
           "parts": "median of 3: quant_s = one append of quant_tokens tokens (all kv heads) to an empty cache; "
                    "attn_s = one fp64 decode of every query head over attn_context tokens"}
    if args.workload in (0, 1):
        # single-threaded leg, in a child process whose OpenMP runtime starts with one thread
        code = ("import json,sys; sys.path.insert(0, %r); import bench, synth; wl = synth.workload(%d); "
                "print(json.dumps(bench.oracle_parts(wl, %d, %d)))" % (ROOT, args.workload, kb, vb))
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
        if r.returncode == 0:
            q1, n1, a1, l1 = json.loads(r.stdout.strip().splitlines()[-1])
            out["single_thread"] = {"threads": 1, "quant_s": q1, "quant_tokens": n1, "attn_s": a1,
                                    "attn_kv_tokens_per_s": l1 / a1}
    return out


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kivi", choices=["kivi", "reference"])
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--context", type=int, default=0)
    ap.add_argument("--bits", type=int, default=0, help="code width of keys and values (default: 2)")
    ap.add_argument("--k-bits", type=int, default=0, help="key code width (overrides --bits)")
    ap.add_argument("--v-bits", type=int, default=0, help="value code width (overrides --bits)")
    ap.add_argument("--group", type=int, default=0, help="G: 32 (default) or 64")
    ap.add_argument("--residual", type=int, default=0, help="R: a multiple of G (default 128)")
    ap.add_argument("--q-heads", type=int, default=0,
                    help="query heads per sequence, a multiple of the workload's kv heads (64 over 8: query group 8)")
    ap.add_argument("--workload", type=int, default=2, choices=[0, 1, 2, 3, 4],
                    help="0 tiny, 1 Llama-2-7B MHA, 2 Llama-3-8B GQA (default), 3 streaming, 4 long varlen")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-query", type=int, default=0,
                    help="time verification steps instead: append N tokens per sequence, then multi-query attention")
    ap.add_argument("--paged", action="store_true",
                    help="packed cache in shared G-token pages behind block tables (random page order)")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the per-workload lines (workloads 0, 1, 3 at 2 and 4 bits, 4) of the default run")
    args = ap.parse_args()
    if any((args.batch, args.context, args.bits, args.k_bits, args.v_bits, args.group, args.residual, args.q_heads,
            args.paged, args.workload != 2)):
        args.workloads = False    # the sub-lines belong to the default headline run only

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    wl = workload_spec(args)
    kb, vb = kv_bits(args, wl)
    widths = f"{kb}-bit" if kb == vb else f"{kb}-bit key / {vb}-bit value"
    ctx = (f"{wl.lengths[0]} cached tokens" if len(set(wl.lengths)) == 1 else
           f"{min(wl.lengths)}..{max(wl.lengths)} cached tokens (mean {sum(wl.lengths) / len(wl.lengths):.0f})")
    config = {
        "workload": (f"{WORKLOAD_NAMES[args.workload]}: {wl.batch} sequences x {ctx}, "
                     f"{wl.num_q_heads} query / {wl.num_kv_heads} kv heads, head_dim {wl.head_dim}, "
                     f"{widths} KIVI (G={wl.group}, R={wl.residual}), {wl.dtype} inputs"),
        "batch": wl.batch, "context": wl.lengths[0] if len(set(wl.lengths)) == 1 else "varlen",
        "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads,
        "head_dim": wl.head_dim, "bits": wl.bits if kb == vb else None, "k_bits": kb, "v_bits": vb,
        "group": wl.group, "residual": wl.residual, "input_dtype": wl.dtype,
        "step": f"append 1 token/sequence (+ group flush every {wl.group} steps) + decode attention",
        "l2": ("flushed before every step (512 MB write, outside the step timing): the cache is smaller than L2"
               if attn_bytes(wl, list(wl.lengths), kb, vb) < 256 << 20 else
               "no flush: the packed cache is larger than L2 (129 MB)"),
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "layout": f"paged: {wl.group}-token pages of one shared pool in random order" if args.paged else "contiguous",
    }
    if args.impl == "reference":
        if rank != 0:
            return
        v, threads, desc, dt = oracle_sample(wl, args.warmup + args.steps, kb, vb, budget_s=60.0)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "KV-tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / (args.warmup + args.steps), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": "KV-tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "KV-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.n_query:
        line = run_gpu_multi(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line))
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    res, wl = run_gpu(args, rank, world, local_rank)

    dev = torch.device("cuda", local_rank)
    total_ms = reduce_max(res["total_ms"], dev)
    e2e_ms = reduce_max(res["e2e"]["ms_per_step"], dev)
    res["e2e"]["value"] = job_throughput(res["e2e"]["kv_tokens"], world, e2e_ms * res["e2e"]["steps"])
    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    value = job_throughput(res["kv_tokens"], world, total_ms)
    attn_ms = res["attn_ms"]
    avg_attn_ms = sum(attn_ms) / len(attn_ms)
    avg_bytes = sum(res["attn_bytes"]) / len(res["attn_bytes"])
    achieved = avg_bytes / (avg_attn_ms / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    # the decode kernel the library picks: the persistent tensor-core kernel for query groups of
    # 1, 2, 4 and 8, the multi-query kernel (one query) for any other group
    group = config["q_heads"] // config["kv_heads"]
    kernel = "decode_mma_kernel" if group in (1, 2, 4, 8) else "decode_multi_kernel"
    per_unit = None if args.paged else NCU_TRAFFIC_BYTES_PER_UNIT.get(
        (kernel, kb, vb, wl.group, wl.residual, group, config["input_dtype"]))
    traffic = per_unit * sum(res["attn_units"]) / len(res["attn_units"]) if per_unit else None
    line = {
        "metric": METRIC, "value": value, "unit": "KV-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": avg_bytes, "avg_launch_ms": avg_attn_ms,
                     "traffic": traffic,
                     "traffic_source": "ncu capture at 8 sequences, scaled by (token, kv head) units" if per_unit else None},
        "attn_kv_tokens_per_s": (res["kv_tokens"] / args.steps) / (avg_attn_ms / 1e3),
        "e2e": {k: res["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "copies")},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "prefill": res["prefill"],
        "clocks": res["clocks"],
    }
    if args.workloads and args.n_query == 0:
        line["workloads"] = run_workloads(args, rank, world, local_rank)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, wl, kb, vb)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
