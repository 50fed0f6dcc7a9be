#!/usr/bin/env python
"""Benchmark of the hybrid-head attention path on GB300.

One JSON line on stdout (rank 0).  Metric: hybrid-attention prefill useful
TFLOP/s (only unmasked (query, key) pairs count, 4*d flops each), with decode
GB/s of the kept KV-cache bytes reported beside it.

  step      one pass of the prefill path over one batch: the planner (visited
            tiles, longest-first work queue) and the fused FA/SSA/BLOCK
            attention kernel, on the workload named by --workload (default: the
            Llama-3.1-8B-shaped 32K layer, 6 of 8 KV heads SSA).
  value     useful TFLOP/s of the whole step, inputs resident in HBM; L2 is
            flushed (256 MB memset) before every timed step, outside the
            events.
  e2e       the same metric through the C ABI with pinned host buffers: Q/K/V
            and the mode mask copied in, O and LSE copied out, every step, by
            one ea_hybrid_attn_prefill_host call (chunks of query blocks, so
            the copies overlap the attention); the unpipelined time is given
            beside it.
  decode    B=32 x 128K-token cache, 2 FA + 6 SSA KV heads: kept K/V bytes per
            step / step time.
  roofline  the attention kernel alone (CUDA events around its launch):
            visited-tile flops / its duration against the measured bf16 peak.
  xa256k_seeded_mask, routed64k_36_layers
            the other two prefill workloads, each with its own clock record:
            the 256K XA-SSA layer (2 BLOCK heads on the seeded density-0.2
            block mask, 6 SSA heads at 128/4096) and the Qwen3-8B-shaped
            36-layer 64K stack whose modes come from the router pre-pass.

--impl reference runs the fp64 CPU oracle (the only independent implementation
of this method here) on a bounded row sample of the same workload.
"""
import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-attn prefill useful TFLOP/s (% bf16 peak); decode GB/s (% HBM)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
BLOCK_MODE = 2


# ------------------------------------------------------------------ counting
def kept_pairs_per_kv_head(mode, S, sink, window, bm_head=None, T=128):
    """Unmasked causal (query, key) pairs of one KV head (closed forms)."""
    if mode == 0:
        return S * (S + 1) // 2
    if mode == 1:
        i = np.arange(S, dtype=np.int64)
        return int((np.minimum(i + 1, window) + np.clip(np.minimum(sink, i + 1 - window), 0, None)).sum())
    nB = (S + T - 1) // T
    rows = np.full(nB, T, dtype=np.int64)
    rows[-1] = S - (nB - 1) * T
    below = np.tril(bm_head.astype(np.int64), -1).sum(axis=1)
    diag = bm_head.diagonal().astype(np.int64)
    return int((rows * below * T).sum() + (diag * rows * (rows + 1) // 2).sum())


def visited_tiles_per_kv_head(mode, S, sink, window, bm_head=None, T=128):
    nB = (S + T - 1) // T
    if mode == 0:
        return nB * (nB + 1) // 2
    if mode == 1:
        w_tiles = (window - 1 + T - 1) // T
        s_tiles = (sink + T - 1) // T
        tot = 0
        for qb in range(nB):
            lo = max(0, qb - w_tiles)
            tot += min(s_tiles, lo) + (qb - lo + 1)
        return tot
    return int(np.tril(bm_head != 0).sum())


def prefill_work(cfg, m, bm):
    """(useful flops, visited-tile flops) of one layer."""
    g = cfg.Hq // cfg.Hkv
    useful = visited = 0
    for b in range(cfg.B):
        for h in range(cfg.Hkv):
            mode = int(m[b, h])
            bmh = None if bm is None else bm[b, h]
            useful += kept_pairs_per_kv_head(mode, cfg.S, cfg.sink, cfg.window, bmh) * g
            visited += visited_tiles_per_kv_head(mode, cfg.S, cfg.sink, cfg.window, bmh) * g
    return 4 * cfg.d * useful, 4 * cfg.d * 128 * 128 * visited


def decode_kept_bytes(cfg, m, rows=None):
    """K+V bytes of the kept cache entries (read once, shared by the group).
    rows: the decode rows [B, Hkv, nB] of the block mask, for BLOCK heads."""
    keys = 0
    for b in range(cfg.B):
        for h in range(cfg.Hkv):
            L = cfg.L
            mode = int(m[b, h])
            if mode == 1:
                ns = min(cfg.sink, L)
                keys += ns + (L - max(L - cfg.window, ns))
            elif mode == BLOCK_MODE:
                qb = (L - 1) // 128
                kept = np.nonzero(np.asarray(rows[b, h, :qb + 1]))[0]
                keys += int(sum(min(128, L - 128 * int(kb)) for kb in kept))
            else:
                keys += L
    return keys * 2 * cfg.d * 2


def job_throughput(local_ms, world, work_per_rank_step, steps, device):
    """Whole-job throughput of N replicas: the timed region is the slowest
    rank's (max over ranks), the work is every rank's (weak scaling, each rank
    processes its own batch).  Returns (max ms, work units per second / 1e12)."""
    if world > 1:
        t = torch.tensor([local_ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        local_ms = float(t.item())
    return local_ms, world * work_per_rank_step * steps / (local_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ environment
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
           "bf16_tflops_sustained": None, "source": "fallback"}
    try:
        with open(path) as f:
            d = json.load(f)
        flat = {}

        def walk(x, pre=""):
            if isinstance(x, dict):
                for k, v in x.items():
                    walk(v, pre + k + ".")
            elif isinstance(x, (int, float)):
                flat[pre[:-1]] = float(x)
        walk(d)
        for k, v in flat.items():
            kl = k.lower()
            if "hbm" in kl and "gbs" in kl:
                out["hbm_gbs"] = v
            elif "bf16" in kl and "sustained" in kl:
                out["bf16_tflops_sustained"] = v
            elif "bf16" in kl and "tflops" in kl:
                out["bf16_tflops"] = v
        out["source"] = "measured"
    except (OSError, ValueError):
        pass
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def profile_traffic(name, src):
    """DRAM traffic per launch recorded by an ncu summary under profiles/, if the
    kernel source has not changed since (else None)."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_sha256")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != digest or "traffic_bytes_per_launch" not in vals:
        return None
    return float(vals["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ workloads
def get_cfg(name):
    from sparse_head_attention_gb300 import workloads as wl
    table = {"llama32k": wl.LLAMA_32K, "tiny": wl.TINY, "xa256k": wl.XA_SSA_256K}
    return table[name]


def make_prefill_inputs(cfg, dev):
    from sparse_head_attention_gb300 import workloads as wl
    Q, K, V = wl.qkv(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=cfg.seed, device=dev)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, cfg.fa_impl, cfg.sa_impl)
    bm = None
    if cfg.fa_impl == 2 or cfg.sa_impl == 2:
        bm = wl.block_mask(cfg.B, cfg.Hkv, cfg.S, density=cfg.block_density, seed=cfg.seed)
    return Q, K, V, m, bm


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, dev):
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl

    cfg = get_cfg(args.workload)
    Q, K, V, m_cpu, bm_cpu = make_prefill_inputs(cfg, dev)
    m = m_cpu.to(dev)
    bm = None if bm_cpu is None else bm_cpu.to(dev)
    useful_flops, tile_flops = prefill_work(cfg, m_cpu.numpy(), None if bm_cpu is None else bm_cpu.numpy())
    O = torch.empty_like(Q)
    LSE = torch.empty(cfg.B, cfg.Hq, cfg.S, dtype=torch.float32, device=dev)
    ws = ea.prefill_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        ea.ea_prefill_plan(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, m, sink=cfg.sink, window=cfg.window,
                           block_mask=bm, workspace=ws)
        if ev is not None:
            ev[0].record(stream)
        ea.ea_prefill_attend(Q, K, V, m, sink=cfg.sink, window=cfg.window, block_mask=bm,
                             O=O, LSE=LSE, workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev_s[i].record(stream)
        step(ev_k[i])
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = sum(s.elapsed_time(e) for s, e in zip(ev_s, ev_e))
    kern_ms = [a.elapsed_time(b) for a, b in ev_k]
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error during the timed steps")
    step_ms, value = job_throughput(step_ms, world, useful_flops, args.steps, dev)
    ms_per_step = step_ms / args.steps

    peaks = measured_peaks()
    k_ms = statistics.mean(kern_ms)
    achieved = tile_flops / (k_ms * 1e-3) / 1e12
    # the committed ncu summary covers the 32K layer only; other workloads carry no traffic figure
    traffic = None
    if cfg.name == "llama3_8b_layer_prefill_s32k_fa_ssa":
        traffic = profile_traffic("prefill_attention_llama32k.md",
                                  os.path.join(ROOT, "sparse_head_attention_gb300", "csrc", "ea_prefill.cu"))
    roofline = {"bound": "tensor", "kernel": "hybrid_prefill_kernel", "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic, "peak_source": peaks["source"],
                "work": "visited-tile flops 4*d*128*128 per tile per query head = %.4e per launch" % tile_flops,
                "kernel_ms": round(k_ms, 4)}

    # ---- end to end through the C ABI with pinned host buffers: one
    # ea_hybrid_attn_prefill_host call per step (Q/K/V/m[/mask] copied in,
    # O and LSE copied back, chunked so that copies overlap the attention)
    e2e = None
    if not args.no_e2e:
        hQ = Q.cpu().pin_memory()
        hK = K.cpu().pin_memory()
        hV = V.cpu().pin_memory()
        hm = m_cpu.pin_memory()
        hbm = None if bm is None else bm.cpu().pin_memory()
        hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
        hL = torch.empty(LSE.shape, dtype=LSE.dtype, pin_memory=True)
        buf = ea.prefill_host_buffer(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, with_block_mask=hbm is not None,
                                     device=dev)

        def e2e_step():
            ea.ea_hybrid_attn_prefill_host(hQ, hK, hV, hm, sink=cfg.sink, window=cfg.window,
                                           block_mask=hbm, O=hO, LSE=hL, device_buffer=buf,
                                           n_chunks=args.e2e_chunks, stream=stream)

        def serial_step():
            # the same step without the overlap, for comparison: whole tensors
            # up, one fused launch, whole outputs back
            dQ.copy_(hQ, non_blocking=True)
            dK.copy_(hK, non_blocking=True)
            dV.copy_(hV, non_blocking=True)
            dm.copy_(hm, non_blocking=True)
            ea.ea_hybrid_attn_prefill(dQ, dK, dV, dm, sink=cfg.sink, window=cfg.window, block_mask=bm,
                                      O=O, LSE=LSE, workspace=ws)
            hO.copy_(O, non_blocking=True)
            hL.copy_(LSE, non_blocking=True)

        def time_steps(fn, n):
            # median per-step time: the host link is shared, and a step that
            # meets a burst of someone else's traffic would skew a mean
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            per_step = []
            for _ in range(n):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                per_step.append(a.elapsed_time(b))
            return statistics.median(per_step)

        n_e2e = max(5, min(args.steps, 10))
        if world > 1:
            torch.distributed.barrier()
        e_ms = time_steps(e2e_step, n_e2e)
        if world > 1:
            # whole-job figure: the slowest replica's step
            t = torch.tensor([e_ms], dtype=torch.float64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e_ms = float(t.item())
        if ea.ea_check_errors(buf) != 0:
            raise RuntimeError("device error in the end-to-end prefill")
        dQ, dK, dV, dm = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V), torch.empty_like(m)
        s_ms = time_steps(serial_step, n_e2e)
        h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hm) + ((hbm,) if hbm is not None else ()))
        d2h = sum(t.numel() * t.element_size() for t in (hO, hL))
        e2e = {"value": round(world * useful_flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms, 3), "estimator": "median of %d steps" % n_e2e,
               "call": "ea_hybrid_attn_prefill_host (chunked copies overlapped with the attention, "
                       "%s chunks)" % (args.e2e_chunks or "10"),
               "serial_ms_per_step": round(s_ms, 3)}
        del hQ, hK, hV, dQ, dK, dV, buf

    # ---- decode
    decode = None
    if not args.no_decode:
        decode = run_decode(args, dev, peaks, flush)

    # ---- a variable-length serving batch in one launch
    varlen = run_varlen(args, dev, peaks, flush)

    # ---- router latency (36-layer 64K shape: 8 KV heads, 128 -> 64 -> 2)
    router = run_router(dev)

    # ---- XA block-mask estimation and the XA-SSA layer that uses it (256K)
    xa = None
    if not args.no_xa:
        xa = run_xa(args, dev, peaks, flush)

    # ---- the other two prefill workloads: the 256K XA-SSA layer on the seeded
    # block mask, and the 36-layer router-driven 64K stack
    xa256k = None
    if not args.no_xa256k and cfg.name != get_cfg("xa256k").name:
        xa256k = run_seeded_layer(args, dev, peaks, flush, "xa256k")
    routed = None
    if not args.no_routed:
        routed = run_routed_layers(args, dev, peaks, flush)
    multi = None
    if not args.no_multi_layer:
        multi = run_multi_layer(args, dev, peaks, flush)

    # ---- sparsity ratios of the timed layer (host)
    msr, esr = ea.ea_sparsity_ratios(
        (m_cpu.numpy() == cfg.sa_impl).astype(np.uint8), m_cpu.numpy(), cfg.S, sink=cfg.sink,
        window=cfg.window, block_masks=None if bm_cpu is None else [bm_cpu.numpy()[0]])

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V; seeded SA-head choice)",
        "config": {"workload": cfg.name, "B": cfg.B, "seq_len": cfg.S, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                   "d": cfg.d, "sa_heads": cfg.sa_heads, "sink": cfg.sink, "window": cfg.window,
                   "omega_msr": msr, "omega_esr": round(esr, 6),
                   "useful_flops_per_step": useful_flops, "visited_tile_flops_per_step": tile_flops,
                   "pct_of_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
                   "l2": "flushed before every timed step (256 MB memset, outside the events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "decode": decode,
        "varlen": varlen,
        "router": router,
        "xa": xa,
        "xa256k_seeded_mask": xa256k,
        "routed64k_36_layers": routed,
        "multi_layer_launch": multi,
    }
    # the CPU baseline is reported by rank 0 of a single-GPU run only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, Q, K, V, m_cpu, bm_cpu, args)
    return line


def run_decode(args, dev, peaks, flush):
    import dataclasses

    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    cfg = wl.DECODE_128K
    if args.decode_batch != cfg.B:
        cfg = dataclasses.replace(cfg, B=args.decode_batch, name="%s_b%d" % (cfg.name, args.decode_batch))
    q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev)
    _, m_cpu = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
    m = m_cpu.to(dev)
    nbytes = decode_kept_bytes(cfg, m_cpu.numpy())
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, device=dev)
    O = torch.empty_like(q)
    LSE = torch.empty(cfg.B, cfg.Hq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m, sink=cfg.sink, window=cfg.window, O=O, LSE=LSE,
                                 workspace=ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    # The cache (2 x 8.6 GB at B = 32) is far larger than L2 and every step
    # streams its kept rows in order, so no L2 flush is needed between steps
    # (a flush would also leave L2 full of dirty lines whose write-back lands
    # in the next timed step).
    n = max(args.steps, 20)
    ms = []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m, sink=cfg.sink, window=cfg.window, O=O, LSE=LSE,
                                 workspace=ws)
        b.record(stream)
        ms.append((a, b))
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in decode")
    t = statistics.mean(a.elapsed_time(b) for a, b in ms)
    gbs = nbytes / (t * 1e-3) / 1e9

    # XA-SSA routing of the same cache: the two FA heads become BLOCK heads
    # reading the kept blocks of their decode row (L - 1) / 128 of a block mask
    # (each block kept with probability 0.2, the first and the query's own block
    # always; only the decode rows are drawn, the other rows stay empty)
    nBd = (cfg.L + 127) // 128
    _, m_xa_cpu = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, BLOCK_MODE, 1)
    rows = torch.rand((cfg.B, cfg.Hkv, nBd), generator=torch.Generator().manual_seed(7)) < 0.2
    rows[..., 0] = True
    rows[..., (cfg.L - 1) // 128] = True
    rows[..., (cfg.L - 1) // 128 + 1:] = False
    bm_xa = torch.zeros((cfg.B, cfg.Hkv, nBd, nBd), dtype=torch.uint8, device=dev)
    bm_xa[:, :, (cfg.L - 1) // 128, :] = rows.to(torch.uint8).to(dev)
    m_xa = m_xa_cpu.to(dev)
    xbytes = decode_kept_bytes(cfg, m_xa_cpu.numpy(), rows.numpy())

    def xa_step():
        ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m_xa, sink=cfg.sink, window=cfg.window, O=O,
                                 LSE=LSE, workspace=ws, block_mask=bm_xa)

    for _ in range(args.warmup):
        xa_step()
    torch.cuda.synchronize()
    xms = []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        xa_step()
        b.record(stream)
        xms.append((a, b))
    torch.cuda.synchronize()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in the XA-SSA decode")
    tx = statistics.mean(a.elapsed_time(b) for a, b in xms)
    del bm_xa
    xa_ssa = {"routing": "2 BLOCK (decode rows of a 0.2-density block mask) + 6 SSA KV heads",
              "value": round(xbytes / (tx * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(tx, 4),
              "frac": round(xbytes / (tx * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
              "kept_kv_bytes_per_step": xbytes,
              "gpu_launches_per_step": 4}

    # the same step over a paged cache: 256-row pages of all sequences
    # scattered through one pool by a random permutation
    page_size = 256
    per_seq = cfg.L // page_size
    perm = torch.randperm(cfg.B * per_seq, generator=torch.Generator().manual_seed(3)).to(dev)
    table = perm.view(cfg.B, per_seq).to(torch.int32)
    Kp = torch.empty(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d, dtype=torch.bfloat16, device=dev)
    Kp[perm] = Kc.view(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d)
    del Kc
    Vp = torch.empty_like(Kp)
    Vp[perm] = Vc.view(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d)
    del Vc

    def paged_step():
        ea.ea_hybrid_attn_decode_paged(q, Kp, Vp, table, sl, m, sink=cfg.sink, window=cfg.window, O=O,
                                       LSE=LSE, workspace=ws)

    for _ in range(args.warmup):
        paged_step()
    torch.cuda.synchronize()
    pms = []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        paged_step()
        b.record(stream)
        pms.append((a, b))
    torch.cuda.synchronize()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in paged decode")
    tp = statistics.mean(a.elapsed_time(b) for a, b in pms)
    del Kp, Vp
    paged = {"page_size": page_size, "value": round(nbytes / (tp * 1e-3) / 1e9, 1), "unit": "GB/s",
             "ms_per_step": round(tp, 4), "frac": round(nbytes / (tp * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
             "layout": "pages of all sequences permuted through one pool; block table [B, L/256]"}
    return {"workload": cfg.name, "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(t, 4),
            "l2": "inputs larger than L2 (%.1f GB of K/V cache), no flush between steps"
                  % (2 * cfg.B * cfg.L * cfg.Hkv * cfg.d * 2 / 1e9),
            "paged": paged,
            "xa_ssa": xa_ssa,
            "kept_kv_bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "kernel": "decode_plan_kernel + decode_split_kernel + decode_merge_kernel",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": profile_traffic("decode_split_b4_l128k.md", os.path.join(
                             ROOT, "sparse_head_attention_gb300", "csrc", "ea_decode.cu"))
                         if cfg.B == 32 else None,
                         "peak_source": peaks["source"]},
            "gpu_launches_per_step": 3, "clocks": clk,
            "small_batch": run_decode_small(args, dev, peaks) if cfg.B == 32 else None}


def run_decode_small(args, dev, peaks):
    """Decode at serving batch sizes B = 1 and 4 (the 128K cache, heads and
    routing of the B = 32 line): the step through the public call, timed eager
    (host argument handling and three launches inside the events) and replayed
    from a CUDA graph (device time of the same launches), as a serving loop
    that captures its decode step runs it."""
    import dataclasses

    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.current_stream()
    for B in (1, 4):
        cfg = dataclasses.replace(wl.DECODE_128K, B=B, name="%s_b%d" % (wl.DECODE_128K.name, B))
        q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev)
        _, m_cpu = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
        m = m_cpu.to(dev)
        nbytes = decode_kept_bytes(cfg, m_cpu.numpy())
        ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, device=dev)
        O = torch.empty_like(q)
        LSE = torch.empty(cfg.B, cfg.Hq, dtype=torch.float32, device=dev)

        def step():
            ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m, sink=cfg.sink, window=cfg.window, O=O, LSE=LSE,
                                     workspace=ws)

        def timed(fn, n=200):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n

        t_eager = timed(step)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        t_graph = timed(g.replay)
        if ea.ea_check_errors(ws) != 0:
            raise RuntimeError("device error in the small-batch decode")
        out["b%d" % B] = {
            "kept_kv_bytes_per_step": nbytes,
            "us_per_step_eager": round(t_eager * 1e3, 2),
            "us_per_step_graph": round(t_graph * 1e3, 2),
            "frac_eager": round(nbytes / (t_eager * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "frac_graph": round(nbytes / (t_graph * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        del q, Kc, Vc, ws, g
    out["timing"] = ("200 back-to-back steps between two events (the cache is larger than L2); "
                     "eager: the Python call each step; graph: one captured call replayed")
    return out


def run_varlen(args, dev, peaks, flush):
    """A serving-like prefill batch in one ea_hybrid_attn_prefill_varlen launch:
    128 sequences of 256..8192 tokens (seeded uniform), packed back to back,
    heads and routing of the 32K layer (32/8 heads, 2 FA + 6 SSA, 128/2048).
    Work is counted per sequence with the same closed forms as the 32K line."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    cfg = wl.LLAMA_32K
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(256, 8193, size=128)][:args.varlen_seqs]
    total = sum(lens)
    Q = wl.randn_bf16((total, cfg.Hq, cfg.d), seed=21, device=dev)
    K = wl.randn_bf16((total, cfg.Hkv, cfg.d), seed=22, device=dev)
    V = wl.randn_bf16((total, cfg.Hkv, cfg.d), seed=23, device=dev)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
    _, m1 = wl.routing_from_sa_heads(1, cfg.Hkv, cfg.sa_heads, cfg.fa_impl, cfg.sa_impl)
    m_cpu = m1.repeat(len(lens), 1)
    m = m_cpu.to(dev)
    g = cfg.Hq // cfg.Hkv
    useful = tile = 0
    for L in lens:
        for h in range(cfg.Hkv):
            mode = int(m_cpu[0, h])
            useful += kept_pairs_per_kv_head(mode, L, cfg.sink, cfg.window) * g
            tile += visited_tiles_per_kv_head(mode, L, cfg.sink, cfg.window) * g
    useful *= 4 * cfg.d
    tile *= 4 * cfg.d * 128 * 128
    ws = ea.prefill_varlen_workspace(len(lens), total, max(lens), cfg.Hq, cfg.Hkv, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(cfg.Hq, total, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ea.ea_hybrid_attn_prefill_varlen(Q, K, V, cu, m, max_seqlen=max(lens), sink=cfg.sink,
                                         window=cfg.window, O=O, LSE=LSE, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(5, min(args.steps, 20))):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in the variable-length prefill")
    ms = statistics.median(x.elapsed_time(y) for x, y in ts)
    return {"workload": "%d sequences of 256..8192 tokens (%d in all), 32/8 heads, 2 FA + 6 SSA" % (len(lens), total),
            "ms_per_step": round(ms, 4),
            "useful_tflops": round(useful / (ms * 1e-3) / 1e12, 1),
            "visited_tile_tflops": round(tile / (ms * 1e-3) / 1e12, 1),
            "frac": round(tile / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "step": "setup + planner + fused kernel, one launch for all sequences",
            "l2": "flushed before every timed step (256 MB memset, outside the events)"}


def run_xa(args, dev, peaks, flush):
    """XA block-mask estimation on the 256K XA-SSA layer (2 BLOCK + 6 SSA KV heads,
    32 query heads), inputs with planted hot key blocks; then the whole XA-SSA
    layer step: estimation of the BLOCK heads' masks followed by the fused prefill
    (planner + kernel) that consumes them.  Estimation work: 2 * 16 * 128 flops per
    causal 16 x 16 cell per query head (the antidiagonal's 16 dot products), or per
    computed cell of the 128 x 256 cell tiles."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    cfg = wl.XA_SSA_256K
    if args.xa_seq != cfg.S:
        cfg = dataclasses.replace(cfg, name="xa_ssa_prefill_s%d" % args.xa_seq, S=args.xa_seq)
    Q, K = wl.xa_planted_qk(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=0, device=dev)
    V = wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=2, device=dev)
    _, m_cpu = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, cfg.fa_impl, cfg.sa_impl)
    m = m_cpu.to(dev)
    units = int((m_cpu == BLOCK_MODE).sum())
    g = cfg.Hq // cfg.Hkv
    nB = cfg.S // 128
    nA = cfg.S // 16
    useful = nA * (nA + 1) // 2 * 4096 * g * units
    n_rt = (nA + 127) // 128
    tile = sum(rt // 2 + 1 for rt in range(n_rt)) * 128 * 256 * 4096 * g * units
    xws = ea.xa_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, units, device=dev)
    bm = torch.zeros(cfg.B, cfg.Hkv, nB, nB, dtype=torch.uint8, device=dev)
    pws = ea.prefill_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(cfg.B, cfg.Hq, cfg.S, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def estimate():
        ea.ea_xa_estimate(Q, K, m, max_units=units, block_mask=bm, workspace=xws)

    def layer():
        estimate()
        ea.ea_hybrid_attn_prefill(Q, K, V, m, sink=cfg.sink, window=cfg.window, block_mask=bm,
                                  O=O, LSE=LSE, workspace=pws)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(5, min(args.steps, 10))):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) for x, y in ts)

    est_ms = timed(estimate)
    layer_ms = timed(layer)
    if ea.ea_check_errors(xws) != 0 or ea.ea_check_errors(pws) != 0:
        raise RuntimeError("device error in the XA estimation step")
    bm_cpu = bm.cpu()
    dens = []
    pf_tile = 0
    for h in range(cfg.Hkv):
        mode = int(m_cpu[0, h])
        head = bm_cpu[0, h].numpy() if mode == BLOCK_MODE else None
        if head is not None:
            dens.append(round(float(head.sum()) / (nB * (nB + 1) / 2), 4))
        pf_tile += visited_tiles_per_kv_head(mode, cfg.S, cfg.sink, cfg.window, head) * g
    pf_tile *= 4 * cfg.d * 128 * 128
    del Q, K, V, O, LSE, xws, pws
    return {"workload": "%s: 2 BLOCK + 6 SSA KV heads, 32 query heads, planted hot key blocks (5 %%); "
                        "stride 16, threshold 0.9" % cfg.name,
            "estimate_ms": round(est_ms, 4),
            "estimate_useful_tflops": round(useful / (est_ms * 1e-3) / 1e12, 1),
            "estimate_tile_tflops": round(tile / (est_ms * 1e-3) / 1e12, 1),
            "estimate_frac": round(tile / (est_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "estimate_step": "unit list + antidiagonal score pass + threshold selection (3 launches)",
            "block_density": dens,
            "layer_ms": round(layer_ms, 4),
            "layer_step": "estimation + planner + fused prefill on the estimated masks (5 launches)",
            "layer_prefill_tile_tflops": round(pf_tile / ((layer_ms - est_ms) * 1e-3) / 1e12, 1),
            "l2": "flushed before every timed step (256 MB memset, outside the events)"}


def run_router(dev):
    """Router pre-pass timings: all 36 layers of the 64K workload in one
    ea_route_layers launch (the form the pre-pass takes when a model's K states
    are at hand), the same 36 layers as 36 ea_route launches, and one layer at
    S = 4K / 64K / 1M to show that the cost does not grow with length."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    cfg = wl.QWEN_64K_36L
    L = cfg.layers
    # the router reads only the boundary tokens, so one resident K serves
    # every layer; each layer has its own weights
    K = wl.randn_bf16((1, cfg.S, cfg.Hkv, cfg.d), seed=1, device=dev)
    wb = [wl.router_weights(l, d=cfg.d, hidden=64, device=dev) for l in range(L)]
    Ks = [K] * L
    r = torch.empty(L, 1, cfg.Hkv, dtype=torch.uint8, device=dev)
    mm = torch.empty_like(r)
    lg = torch.empty(L, 1, cfg.Hkv, 2, dtype=torch.float64, device=dev)

    def timed(fn, n=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        e.record()
        torch.cuda.synchronize()
        return 1000 * a.elapsed_time(e) / n

    def one_launch():
        ea.ea_route_layers(Ks, [w for w, _ in wb], [b for _, b in wb], r_out=r, m_out=mm,
                           logits_out=lg)

    def per_layer():
        for l in range(L):
            ea.ea_route(K, *wb[l], r_out=r[l], m_out=mm[l], logits_out=lg[l])

    def graphed(fn):
        # device time alone: the calls replayed from a CUDA graph
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return timed(g.replay)

    us_all = timed(one_launch)
    us_per = timed(per_layer)
    us_all_dev = graphed(one_launch)
    us_per_dev = graphed(per_layer)
    by_len = {}
    for S in (4096, 65536, 1 << 20):
        Kl = wl.randn_bf16((1, S, cfg.Hkv, cfg.d), seed=2, device=dev)
        by_len[str(S)] = round(timed(lambda: ea.ea_route(Kl, *wb[0], r_out=r[0], m_out=mm[0],
                                                         logits_out=lg[0])), 2)
        del Kl
    return {"workload": "router pre-pass, 8 KV heads, boundary 100+100 tokens, MLP 128-64-2",
            "us_36_layers_one_launch": round(us_all, 2),
            "us_36_layers_per_layer_launches": round(us_per, 2),
            "us_36_layers_one_launch_graph": round(us_all_dev, 2),
            "us_36_layers_per_layer_launches_graph": round(us_per_dev, 2),
            "us_one_layer_by_seq_len": by_len,
            "note": "eager figures include the host-side call (argument marshalling); "
                    "graph figures are device time of the same calls replayed from a CUDA graph"}


# ------------------------------------------------------------------ oracle
def _oracle_rows(cfg, m_cpu, bm_cpu, offset, n_rows_per_head):
    """A bounded row sample: one query head of every KV head, rows spread evenly
    over the sequence (shifted by `offset` so repeated samples differ), with the
    useful flops of those rows."""
    g = cfg.Hq // cfg.Hkv
    idx = (np.linspace(0, cfg.S - 1, n_rows_per_head).astype(np.int64) + offset) % cfg.S
    rows = np.array([[0, h * g, i] for h in range(cfg.Hkv) for i in idx], dtype=np.int64)
    flops = 0
    for h in range(cfg.Hkv):
        mode = int(m_cpu[0, h])
        bmh = None if bm_cpu is None else bm_cpu[0, h]
        for i in idx:
            if mode == 0:
                kept = i + 1
            elif mode == 1:
                kept = min(i + 1, cfg.window) + max(0, min(cfg.sink, i + 1 - cfg.window))
            else:
                qb = i // 128
                kept = int(bmh[qb, :qb].sum()) * 128 + (int(i % 128) + 1) * int(bmh[qb, qb])
            flops += 4 * cfg.d * kept
    return rows, flops


def cpu_baseline(cfg, Q, K, V, m_cpu, bm_cpu, args, budget_s=10.0):
    """The fp64 oracle on this machine's cores over a time-bounded row sample."""
    import oracle
    Qc, Kc, Vc = Q.cpu(), K.cpu(), V.cpu()
    bm = None if bm_cpu is None else bm_cpu.numpy()
    oracle.lib()
    t0 = time.perf_counter()
    done_rows = done_flops = 0
    k = 0
    while time.perf_counter() - t0 < budget_s and k < 64:
        rows, flops = _oracle_rows(cfg, m_cpu, bm, 7919 * k, 256)
        oracle.prefill_rows(Qc, Kc, Vc, m_cpu, rows, sink=cfg.sink, window=cfg.window, block_mask=bm)
        done_rows += len(rows)
        done_flops += flops
        k += 1
    dt = time.perf_counter() - t0
    return {"value": done_flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d query rows of %s (%d batches of 256 evenly spaced rows per KV head), "
                      "%.3g useful flops in %.1f s" % (done_rows, cfg.name, k, done_flops, dt)}


def run_reference(args):
    import oracle
    cfg = get_cfg(args.workload)
    Q, K, V, m_cpu, bm_cpu = make_prefill_inputs(cfg, "cpu")
    bm = None if bm_cpu is None else bm_cpu.numpy()
    rows, flops = _oracle_rows(cfg, m_cpu, bm, 0, 64)
    oracle.lib()
    for _ in range(args.warmup):
        oracle.prefill_rows(Q, K, V, m_cpu, rows[:8], sink=cfg.sink, window=cfg.window, block_mask=bm)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.prefill_rows(Q, K, V, m_cpu, rows, sink=cfg.sink, window=cfg.window, block_mask=bm)
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    sample = ("%d query rows (64 per KV head, evenly spaced) of %s per step, %.3g useful flops"
              % (len(rows), cfg.name, flops))
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V)", "impl": "reference",
            "config": {"workload": cfg.name, "B": cfg.B, "seq_len": cfg.S, "Hq": cfg.Hq,
                       "Hkv": cfg.Hkv, "d": cfg.d},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ------------------------------------------------------------------ 36-layer routed workload
def run_routed_layers(args, dev, peaks=None, flush=None):
    """Qwen3-8B-shaped attention stack: 36 layers, S=65536, 32/8 heads, SSA
    128/2048.  One step = for every layer: the router pre-pass on that layer's K
    (pool -> 128-64-2 MLP -> argmax -> mode), the planner and the fused prefill
    driven by those modes.  The output bias beta of the router is set once,
    before timing, by bisection on the device so that the model-level share of
    SA heads is 0.75 (the pages report 0.63-0.85 at test time).  Every layer has
    its own resident Q/K/V (36 x 768 MB); L2 is flushed before every timed
    step.  The attention kernels are also timed alone (CUDA events around each
    layer's launch) for the roofline fraction."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    cfg = wl.QWEN_64K_36L
    peaks = peaks or measured_peaks()
    L = cfg.layers if args.layers is None else args.layers
    layers = []
    for l in range(L):
        K = wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=3 * (cfg.seed + l) + 1, device=dev)
        layers.append(K)
    # beta: bisect on the device router so that 75% of the L*8 decisions are SA
    def sa_share(beta):
        wb = [wl.router_weights(l, d=cfg.d, hidden=64, seed=cfg.seed, beta=beta, device=dev)
              for l in range(L)]
        r, _, _ = ea.ea_route_layers(layers, [w for w, _ in wb], [b for _, b in wb])
        return int(r.sum().item()) / (L * cfg.Hkv)
    lo, hi = -0.05, 0.05
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if sa_share(mid) < 0.75:
            lo = mid
        else:
            hi = mid
    beta = hi
    weights = [wl.router_weights(l, d=cfg.d, hidden=64, seed=cfg.seed, beta=beta, device=dev) for l in range(L)]
    Qs, Vs = [], []
    for l in range(L):
        Qs.append(wl.randn_bf16((cfg.B, cfg.S, cfg.Hq, cfg.d), seed=3 * (cfg.seed + l), device=dev))
        Vs.append(wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=3 * (cfg.seed + l) + 2, device=dev))
    O = torch.empty_like(Qs[0])
    LSE = torch.empty(cfg.B, cfg.Hq, cfg.S, dtype=torch.float32, device=dev)
    ws = ea.prefill_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, device=dev)
    r_buf = [torch.empty(cfg.B, cfg.Hkv, dtype=torch.uint8, device=dev) for _ in range(L)]
    m_buf = [torch.empty(cfg.B, cfg.Hkv, dtype=torch.uint8, device=dev) for _ in range(L)]
    stream = torch.cuda.current_stream()

    def step(kev=None):
        for l in range(L):
            W, b = weights[l]
            ea.ea_route(layers[l], W, b, r_out=r_buf[l], m_out=m_buf[l])
            ea.ea_prefill_plan(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, m_buf[l], sink=cfg.sink,
                               window=cfg.window, workspace=ws)
            if kev is not None:
                kev[l][0].record(stream)
            ea.ea_prefill_attend(Qs[l], layers[l], Vs[l], m_buf[l], sink=cfg.sink, window=cfg.window,
                                 O=O, LSE=LSE, workspace=ws)
            if kev is not None:
                kev[l][1].record(stream)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in the routed workload")
    m_all = torch.stack([m.cpu()[0] for m in m_buf]).numpy()
    r_all = torch.stack([r.cpu()[0] for r in r_buf]).numpy()
    useful = tile = 0
    for l in range(L):
        u, t = prefill_work(cfg, m_all[l:l + 1], None)
        useful += u
        tile += t
    msr, esr = ea.ea_sparsity_ratios(r_all, m_all, cfg.S, sink=cfg.sink, window=cfg.window)
    ranges = [(a, min(a + 12, L)) for a in range(0, L, 12)]
    msr_ranges = {"layers %d-%d" % (a, b - 1): ea.ea_sparsity_ratios(r_all[a:b], m_all[a:b], cfg.S,
                                                                    sink=cfg.sink, window=cfg.window)[0]
                  for a, b in ranges}
    if flush is None:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    n_steps = max(3, min(args.steps // 6, 5))
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    ts, kts = [], []
    for _ in range(n_steps):
        flush.zero_()
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(kev)
        e.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(e))
        kts.append(sum(x.elapsed_time(y) for x, y in kev))
    clk = clocks.stop()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in the routed workload")
    ms = statistics.median(ts)
    kms = statistics.median(kts)
    del Qs, Vs, layers, O, LSE
    return {"workload": cfg.name, "layers": L, "ms_per_step": round(ms, 3),
            "steps_timed": n_steps, "estimator": "median of %d steps" % n_steps,
            "useful_tflops": round(useful / (ms * 1e-3) / 1e12, 1),
            "visited_tile_tflops": round(tile / (ms * 1e-3) / 1e12, 1),
            "frac_of_bf16_peak": round(tile / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "kernels_ms_per_step": round(kms, 3),
            "kernels_visited_tile_tflops": round(tile / (kms * 1e-3) / 1e12, 1),
            "kernels_frac_of_bf16_peak": round(tile / (kms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "useful_flops_per_step": useful, "visited_tile_flops_per_step": tile,
            "omega_msr": msr, "omega_msr_by_layers": msr_ranges, "omega_esr": round(esr, 4),
            "router_output_bias_beta": beta,
            "step": "per layer: ea_route -> ea_prefill_plan -> ea_prefill_attend (fused kernel)",
            "gpu_launches_per_step": 4 * L,
            "l2": "flushed before every timed step (256 MB memset, outside the events)",
            "clocks": clk}


def run_seeded_layer(args, dev, peaks, flush, name):
    """One prefill layer of another benchmark workload (planner + fused kernel
    per step, inputs resident, L2 flushed before every timed step), with its own
    clock record: the 256K XA-SSA layer on the seeded density-0.2 block mask."""
    import sparse_head_attention_gb300 as ea
    cfg = get_cfg(name)
    Q, K, V, m_cpu, bm_cpu = make_prefill_inputs(cfg, dev)
    m = m_cpu.to(dev)
    bm = None if bm_cpu is None else bm_cpu.to(dev)
    useful, tile = prefill_work(cfg, m_cpu.numpy(), None if bm_cpu is None else bm_cpu.numpy())
    O = torch.empty_like(Q)
    LSE = torch.empty(cfg.B, cfg.Hq, cfg.S, dtype=torch.float32, device=dev)
    ws = ea.prefill_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        ea.ea_prefill_plan(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, m, sink=cfg.sink, window=cfg.window,
                           block_mask=bm, workspace=ws)
        if ev is not None:
            ev[0].record(stream)
        ea.ea_prefill_attend(Q, K, V, m, sink=cfg.sink, window=cfg.window, block_mask=bm,
                             O=O, LSE=LSE, workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    n = max(5, min(args.steps, 10))
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    evs = []
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        a.record(stream)
        step(k)
        b.record(stream)
        evs.append((a, b, k))
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ea.ea_check_errors(ws) != 0:
        raise RuntimeError("device error in the %s layer" % name)
    ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    kms = statistics.mean(k[0].elapsed_time(k[1]) for _, _, k in evs)
    msr, esr = ea.ea_sparsity_ratios(
        (m_cpu.numpy() == cfg.sa_impl).astype(np.uint8), m_cpu.numpy(), cfg.S, sink=cfg.sink,
        window=cfg.window, block_masks=None if bm_cpu is None else [bm_cpu.numpy()[0]])
    dens = None
    if bm_cpu is not None:
        nB = (cfg.S + 127) // 128
        dens = [round(float(np.tril(bm_cpu[0, h].numpy()).sum()) / (nB * (nB + 1) / 2), 4)
                for h in range(cfg.Hkv) if int(m_cpu[0, h]) == BLOCK_MODE]
    del Q, K, V, O, LSE
    return {"workload": cfg.name, "B": cfg.B, "seq_len": cfg.S, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
            "sink": cfg.sink, "window": cfg.window, "block_density_seeded": cfg.block_density,
            "block_density_kept": dens, "steps_timed": n,
            "ms_per_step": round(ms, 4), "useful_tflops": round(useful / (ms * 1e-3) / 1e12, 1),
            "kernel_ms": round(kms, 4),
            "visited_tile_tflops": round(tile / (kms * 1e-3) / 1e12, 1),
            "frac_of_bf16_peak": round(tile / (kms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "useful_flops_per_step": useful, "visited_tile_flops_per_step": tile,
            "omega_msr": msr, "omega_esr": round(esr, 6),
            "step": "ea_prefill_plan + ea_prefill_attend (2 launches)",
            "l2": "flushed before every timed step (256 MB memset, outside the events)",
            "clocks": clk}


def run_multi_layer(args, dev, peaks, flush):
    """36 layers of the Llama-3.1-8B-shaped layer (32/8 heads, SSA 128/2048, per
    layer a seeded choice of about 6 SSA KV heads of 8) at S = 4K and 16K:
    the per-layer loop (ea_hybrid_attn_prefill per layer: planner + launch, and
    the pipeline drains at every layer's end) against one
    ea_hybrid_attn_prefill_layers call (one planner and one launch whose
    longest-first queue mixes every layer's items)."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    L = 36
    out = {"workload": "36 layers, B=1, Hq=32, Hkv=8, d=128, SSA 128/2048, seeded modes per layer",
           "l2": "flushed before every timed step (256 MB memset, outside the events)"}
    stream = torch.cuda.current_stream()
    for S in (4096, 16384):
        cfg = dataclasses.replace(wl.LLAMA_32K, S=S, name="llama_s%d" % S)
        Qs = [wl.randn_bf16((1, S, 32, 128), seed=3 * l, device=dev) for l in range(L)]
        Ks = [wl.randn_bf16((1, S, 8, 128), seed=3 * l + 1, device=dev) for l in range(L)]
        Vs = [wl.randn_bf16((1, S, 8, 128), seed=3 * l + 2, device=dev) for l in range(L)]
        g = torch.Generator().manual_seed(S)
        m_cpu = [(torch.rand(1, 8, generator=g) < 0.75).to(torch.uint8) for _ in range(L)]
        ms = [m.to(dev) for m in m_cpu]
        tile = sum(prefill_work(cfg, m.numpy(), None)[1] for m in m_cpu)
        Os = [torch.empty_like(Qs[0]) for _ in range(L)]
        LSEs = [torch.empty(1, 32, S, dtype=torch.float32, device=dev) for _ in range(L)]
        ws1 = ea.prefill_workspace(1, S, 32, 8, device=dev)
        wsl = ea.prefill_layers_workspace(L, 1, S, 32, 8, device=dev)

        def per_layer():
            for l in range(L):
                ea.ea_hybrid_attn_prefill(Qs[l], Ks[l], Vs[l], ms[l], sink=128, window=2048, O=Os[l],
                                          LSE=LSEs[l], workspace=ws1)

        def one_launch():
            ea.ea_hybrid_attn_prefill_layers(Qs, Ks, Vs, ms, sink=128, window=2048, Os=Os, LSEs=LSEs,
                                             workspace=wsl)

        def timed(fn):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            return statistics.median(x.elapsed_time(y) for x, y in ts)

        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        t_loop = timed(per_layer)
        t_one = timed(one_launch)
        clk = clocks.stop()
        if ea.ea_check_errors(ws1) != 0 or ea.ea_check_errors(wsl) != 0:
            raise RuntimeError("device error in the multi-layer prefill")
        out["s%d" % S] = {
            "per_layer_loop_ms": round(t_loop, 3), "one_launch_ms": round(t_one, 3),
            "speedup": round(t_loop / t_one, 3),
            "one_launch_visited_tile_tflops": round(tile / (t_one * 1e-3) / 1e12, 1),
            "one_launch_frac_of_bf16_peak": round(tile / (t_one * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "per_layer_visited_tile_tflops": round(tile / (t_loop * 1e-3) / 1e12, 1),
            "visited_tile_flops": tile, "gpu_launches": {"per_layer_loop": 3 * L, "one_launch": 3},
            "clocks": clk}
        del Qs, Ks, Vs, Os, LSEs, ws1, wsl
    return out


# ------------------------------------------------------------------ Algorithm 1(a) comparison
def serial_dispatch(ea, Q, K, V, m_cpu, sink, window, O, LSE, ws_fa, ws_sa):
    """Serial Dispatch ("Paper Reading - Elastic Attention" (English notes),
    §04 Deployment, Algorithm 1(a)): split the KV heads into the FA and the SA
    group, copy each group's Q/K/V into tensors of their own, run one
    single-mode attention launch per group, and copy the outputs back into
    place.  Same kernels as the fused path; only the dispatch differs."""
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    g = Hq // Hkv
    dev = Q.device
    for mode, ws in ((0, ws_fa), (1, ws_sa)):
        kv = [h for h in range(Hkv) if int(m_cpu[0, h]) == mode]
        if not kv:
            continue
        kv_t = torch.tensor(kv, device=dev)
        q_t = torch.tensor([h * g + j for h in kv for j in range(g)], device=dev)
        Qs = Q.index_select(2, q_t)
        Ks = K.index_select(2, kv_t)
        Vs = V.index_select(2, kv_t)
        ms = torch.full((B, len(kv)), mode, dtype=torch.uint8, device=dev)
        Os, Ls = ea.ea_hybrid_attn_prefill(Qs, Ks, Vs, ms, sink=sink, window=window, workspace=ws)
        O.index_copy_(2, q_t, Os)
        LSE.index_copy_(1, q_t, Ls)


def run_serial_sweep(args, dev):
    """Fused single launch vs Serial Dispatch over the layer sparsity ratio
    (1..7 of 8 KV heads SSA, sink 128 / window 2048) and sequence length, on
    the Llama-3.1-8B attention shape; one JSON line per point."""
    import sparse_head_attention_gb300 as ea
    from sparse_head_attention_gb300 import workloads as wl
    B, Hq, Hkv, d, sink, window = 1, 32, 8, 128, 128, 2048
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for S in args.serial_lengths:
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=0, device=dev)
        O = torch.empty_like(Q)
        LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
        ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
        ws_fa = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
        ws_sa = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
        for n_sa in range(1, Hkv):
            sa = wl.sa_heads_randperm(Hkv, n_sa, 0)
            _, m_cpu = wl.routing_from_sa_heads(B, Hkv, sa)
            m = m_cpu.to(dev)
            runs = {
                "fused": lambda: ea.ea_hybrid_attn_prefill(Q, K, V, m, sink=sink, window=window,
                                                           O=O, LSE=LSE, workspace=ws),
                "serial": lambda: serial_dispatch(ea, Q, K, V, m_cpu, sink, window, O, LSE,
                                                  ws_fa, ws_sa),
            }
            res = {}
            for name, fn in runs.items():
                for _ in range(2):
                    fn()
                torch.cuda.synchronize()
                ts = []
                for _ in range(max(3, args.steps // 5)):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b))
                res[name] = statistics.median(ts)
            print(json.dumps({"comparison": "fused vs serial dispatch", "seq_len": S,
                              "omega_msr_layer": n_sa / Hkv, "fused_ms": round(res["fused"], 4),
                              "serial_ms": round(res["serial"], 4),
                              "speedup": round(res["serial"] / res["fused"], 3)}), flush=True)
        print(json.dumps({"comparison": "fused vs serial dispatch", "seq_len": S,
                          "clocks": clocks.stop()}), flush=True)
        del Q, K, V, O, LSE


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama32k", choices=["llama32k", "tiny", "xa256k"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="chunks of the end-to-end pipelined call (0 = the library's choice)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-xa", action="store_true", help="skip the XA estimation line")
    ap.add_argument("--xa-only", action="store_true",
                    help="time only the XA estimation (profiling helper; prints its object)")
    ap.add_argument("--xa-seq", type=int, default=262144,
                    help="sequence length of the XA line (262144 is the benchmark workload)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode workload (profiling helper; prints its object)")
    ap.add_argument("--routed-layers", action="store_true",
                    help="time the 36-layer router-driven 64K workload instead of the benchmark")
    ap.add_argument("--layers", type=int, default=None, help="layers of --routed-layers (default 36)")
    ap.add_argument("--no-routed", action="store_true", help="skip the 36-layer routed 64K line")
    ap.add_argument("--no-multi-layer", action="store_true",
                    help="skip the 36-layer one-launch vs per-layer comparison (4K and 16K)")
    ap.add_argument("--no-xa256k", action="store_true",
                    help="skip the 256K XA-SSA layer on the seeded block mask")
    ap.add_argument("--serial-sweep", action="store_true",
                    help="fused single launch vs Serial Dispatch (Algorithm 1(a)) sweep instead of the benchmark")
    ap.add_argument("--serial-lengths", type=int, nargs="+", default=[16384, 32768, 65536, 131072])
    ap.add_argument("--varlen-seqs", type=int, default=128,
                    help="the first N sequences of the variable-length batch (a smaller case for ncu)")
    ap.add_argument("--decode-batch", type=int, default=32,
                    help="decode batch (32 is the benchmark workload; smaller for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from sparse_head_attention_gb300 import build as ea_build
    ea_build.build()
    if args.routed_layers:
        if rank == 0:
            print(json.dumps(run_routed_layers(args, dev, measured_peaks())), flush=True)
        return 0
    if args.serial_sweep:
        if rank == 0:
            run_serial_sweep(args, dev)
        return 0
    if args.xa_only:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        if rank == 0:
            print(json.dumps(run_xa(args, dev, measured_peaks(), flush)), flush=True)
        return 0
    if args.decode_only:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        if rank == 0:
            print(json.dumps(run_decode(args, dev, measured_peaks(), flush)), flush=True)
        return 0
    line = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
