"""Benchmark: exact causal attention prefill (TFLOP/s) and KV-cache decode (GB/s) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--prefill NAME] [--only prefill|decode|paged|window|backward|rope]
                    [--no-cpu-baseline] [--no-e2e]

One step = one pass of the whole hot path over synthetic bf16 inputs that are
already resident in device memory: a causal GQA prefill (B=1, Hq=64, Hkv=8,
N=16384, d=128), a decode step (B=16, Hq=32, Hkv=8, d=128, cache lengths
uniform on [1024, 8192]), the same decode over a paged cache (64-token
pages) with the new token appended, the prefill again with a 4096-key
causal sliding window, and the backward pass of the causal prefill (dQ, dK,
dV from the o and lse that step's prefill wrote and a seeded dO) and the prefill
with rotary position embedding (base 10000) in a second loop. L2 is flushed (a 256 MiB write) before each
of the two launches, outside their CUDA-event brackets, followed by a 256 MiB
read so the timed kernel does not pay for writing back the flush's dirty lines.
Prints one JSON line.

``value`` is prefill TFLOP/s (4*B*Hq*Nq*Nk*d, halved for causal) over the
prefill launches; the decode result sits in ``decode`` (GB/s of the cache
rows actually read, sum(seqlens)*Hkv*d*2*2 bytes, plus q, o and lse).
Under torchrun every rank runs the same workload (replicas; weak scaling)
and rank 0 prints the aggregate over the max-over-ranks time.

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample
of the same workload per step, on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_scaled_dot_03_b300 import workloads as W  # noqa: E402

METRIC = "attn fwd TFLOP/s (bf16, causal) and decode GB/s; % of B300 roofline"
PREFILL = {w.name: w for w in W.PREFILL_WORKLOADS}
L2_FLUSH_BYTES = 256 << 20
WINDOW = 4096  # local-window width of the sliding-window prefill measured beside the full one


# ---------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "exact_scaled_dot_03_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name, files):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since the counters were taken (else None)."""
    p = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("source_sha", "dram_bytes_per_launch")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_sha") != kernel_source_hash(files):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle arm
def oracle_prefill_sample(w, q, k, v, h, r0, r1):
    """Time the oracle on query rows [r0, r1) of head h; return (useful flops, seconds)."""
    import oracle
    from exact_scaled_dot_03_b300.workloads import bf16_bits
    hk = h // (w.Hq // w.Hkv)
    qd = oracle.bf16_bits_to_f64(bf16_bits(q[:1, h:h + 1]))
    kd = oracle.bf16_bits_to_f64(bf16_bits(k[:1, hk:hk + 1]))
    vd = oracle.bf16_bits_to_f64(bf16_bits(v[:1, hk:hk + 1]))
    rows = np.arange(r0, r1)
    t0 = time.perf_counter()
    oracle.attention_forward(qd, kd, vd, w.scale, w.causal, rows=rows)
    dt = time.perf_counter() - t0
    visible = (np.minimum(rows + (w.Nk - w.Nq), w.Nk - 1) + 1).clip(0).sum() if w.causal else rows.size * w.Nk
    return 4.0 * w.d * float(visible), dt


def oracle_decode_sample(w, q, kc, vc, sl, bs):
    import oracle
    from exact_scaled_dot_03_b300.workloads import bf16_bits
    sel = list(bs)
    qd = oracle.bf16_bits_to_f64(bf16_bits(q[sel]))
    kd = oracle.bf16_bits_to_f64(bf16_bits(kc[sel]))
    vd = oracle.bf16_bits_to_f64(bf16_bits(vc[sel]))
    t0 = time.perf_counter()
    oracle.attention_decode(qd, kd, vd, sl[sel].numpy(), w.scale)
    dt = time.perf_counter() - t0
    nbytes = int(sl[sel].sum()) * w.Hkv * w.d * 2 * 2
    return nbytes, dt


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, q, k, v, budget_s=12.0):
    """The oracle on a bounded sample: 512-row blocks from the last (heaviest)
    rows of successive heads until the time budget is used."""
    flops, secs, blocks = 0.0, 0.0, []
    h, r1 = 0, w.Nq
    while secs < budget_s and len(blocks) < 64:
        r0 = max(0, r1 - 512)
        f, dt = oracle_prefill_sample(w, q, k, v, h, r0, r1)
        flops += f
        secs += dt
        blocks.append((h, r0, r1))
        h = (h + 1) % w.Hq
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{len(blocks)} blocks of 512 query rows (the last rows, heaviest under the causal mask) "
                      f"of heads 0..{len(blocks) - 1} of {w.name}; {secs:.1f} s of fp64 numpy on the host"}


def run_reference(args, w, wd):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    q, k, v = W.prefill_inputs(w)
    dq, kc, vc, sl = W.decode_inputs(wd)
    times, flops = [], []
    dec_bytes, dec_secs = 0, 0.0
    for step in range(args.warmup + args.steps):
        h = step % w.Hq
        f, dt = oracle_prefill_sample(w, q, k, v, h, w.Nq - 512, w.Nq)
        nb, ddt = oracle_decode_sample(wd, dq, kc, vc, sl, [step % wd.B])
        if step >= args.warmup:
            times.append(dt)
            flops.append(f)
            dec_bytes += nb
            dec_secs += ddt
    value = sum(flops) / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "decode_workload": wd.name,
                   "sample_per_step": "512 heaviest query rows of one head (prefill) + one sequence (decode)"},
        "decode": {"value": dec_bytes / dec_secs / 1e9, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"per step: query rows [{w.Nq - 512}, {w.Nq}) of one head of {w.name}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- replicas
def max_over_ranks(totals: dict, device) -> dict:
    """Per-part timed totals (ms), element-wise max over all ranks: the job
    is as fast as its slowest replica. Identity on a single process."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return dict(totals)
    names = sorted(totals)
    t = torch.tensor([totals[n] for n in names], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(names, t.tolist()))


def job_rate(work_per_step: float, steps: int, world: int, total_ms: float) -> float:
    """Whole-job throughput: the work every replica did (each rank runs the
    same workload: weak scaling) over the slowest rank's timed total."""
    return world * work_per_step * steps / (total_ms / 1e3)


# ---------------------------------------------------------------- GPU arm
def run_ours(args, w, wd):
    from exact_scaled_dot_03_b300 import binding
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    do_pre = args.only in (None, "prefill")
    do_dec = args.only in (None, "decode")
    do_pag = args.only in (None, "paged")
    do_win = args.only in (None, "window")
    do_bwd = args.only in (None, "backward")
    do_rope = args.only in (None, "rope")

    parts = []  # (name, launch function)
    kernels = {"prefill": 1, "decode": 1, "window": 1, "paged": 1, "backward": 3, "rope": 3}  # our launches per call
    if do_pre or do_bwd or do_rope:
        q_h, k_h, v_h = W.prefill_inputs(w)
        q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32, device=dev)
        if do_pre:
            parts.append(("prefill", lambda: binding.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)))
    if do_dec:
        dq_h, kc_h, vc_h, sl_h = W.decode_inputs(wd)
        dq, kc, vc, sl = dq_h.to(dev), kc_h.to(dev), vc_h.to(dev), sl_h.to(dev)
        do = torch.empty_like(dq)
        dlse = torch.empty(wd.B, wd.Hq, dtype=torch.float32, device=dev)
        ws = binding.decode_workspace(wd.B, wd.Hq, wd.Hkv, wd.Lmax, wd.d, device=dev)
        parts.append(("decode", lambda: binding.decode(dq, kc, vc, sl, scale=wd.scale, workspace=ws, out=do,
                                                       lse=dlse)))
    if do_win:
        ww = W.CAUSAL_GQA_16384
        if not do_pre:
            q_h, k_h, v_h = W.prefill_inputs(ww)
            q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
            o = torch.empty_like(q)
            lse = torch.empty(ww.B, ww.Hq, ww.Nq, dtype=torch.float32, device=dev)
        parts.append(("window", lambda: binding.fwd(q, k, v, causal=True, scale=ww.scale, out=o, lse=lse,
                                                    window=WINDOW)))
    if do_pag:
        wp = W.DECODE_GQA_PAGED
        pq_h, pkn_h, pvn_h, pkp_h, pvp_h, pbt_h, psl_h = W.paged_decode_inputs(wp)
        pq, pkn, pvn, pkp, pvp, pbt, psl = (t.to(dev) for t in (pq_h, pkn_h, pvn_h, pkp_h, pvp_h, pbt_h, psl_h))
        po = torch.empty_like(pq)
        plse = torch.empty(wp.B, wp.Hq, dtype=torch.float32, device=dev)
        pws = torch.zeros(int(binding.lib().attn_decode_paged_workspace_size(wp.B, wp.Hq, wp.Hkv, pbt.shape[1],
                                                                             wp.page_size, wp.d)),
                          dtype=torch.uint8, device=dev)
        # Every call appends at position seqlens[b] (the same slot each time: the
        # lengths are not advanced between timed calls, so the work is identical).
        parts.append(("paged", lambda: binding.decode_paged(pq, pkp, pvp, pbt, psl, pkn, pvn, scale=wp.scale,
                                                            workspace=pws, out=po, lse=plse)))
    if do_bwd:
        dout = W.backward_inputs(w)[3].to(dev)   # Q, K, V are the prefill's draw; dO follows them
        binding.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)  # o, lse (rewritten each step)
        bws = torch.empty(max(1, int(binding.lib().attn_bwd_workspace_size(w.B, w.Hq, w.Nq))), dtype=torch.uint8,
                          device=dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        parts.append(("backward", lambda: binding.bwd(q, k, v, o, lse, dout, causal=w.causal, scale=w.scale,
                                                      workspace=bws, dq=gq, dk=gk, dv=gv)))
    if do_rope:
        rws = torch.empty(int(binding.lib().attn_fwd_rope_workspace_size(w.B, w.Hkv, w.Nq, w.Nk, w.d)),
                          dtype=torch.uint8, device=dev)
        ro = torch.empty_like(q)
        rlse = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32, device=dev)
        parts.append(("rope", lambda: binding.fwd_rope(q, k, v, causal=w.causal, scale=w.scale, base=10000.0,
                                                       workspace=rws, out=ro, lse=rlse)))
    # The backward and RoPE prefill are timed in their own loop after the
    # others: their seconds of full tensor load would otherwise hold the part
    # at its power cap while the prefill is timed.
    later = ("backward", "rope")
    groups = [[p for p in parts if p[0] not in later], [p for p in parts if p[0] in later]]
    groups = [g for g in groups if g]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2 (evicts the inputs), then read another
        # one so that no dirty line is left for the timed kernel to write back.
        flush.zero_()
        torch.sum(clean, dim=0, out=clean_sum)

    for _ in range(args.warmup):
        for _, fn in parts:
            flush_l2()
            fn()
    torch.cuda.synchronize()
    code, detail = binding.device_status()
    if code != binding.OK:
        raise RuntimeError(f"device status after warm-up: {code} {detail}")

    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ms = {}
    t_wall = 0.0
    for gi, group in enumerate(groups):
        if gi > 0:  # the later group gets its own warm-up
            for _ in range(args.warmup):
                for _, fn in group:
                    flush_l2()
                    fn()
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in group]
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        # Keep the device busy while the host queues the timed launches, so no
        # event bracket contains host launch latency (that is the e2e number's job).
        torch.cuda._sleep(int(2e9 * (0.01 + 0.0004 * args.steps * len(group))))
        t0 = time.perf_counter()
        for step in ev:
            for (e0, e1), (_, fn) in zip(step, group):
                flush_l2()           # outside the event bracket
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        t_wall += time.perf_counter() - t0
        ms.update({name: [step[i][0].elapsed_time(step[i][1]) for step in ev] for i, (name, _) in enumerate(group)})
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    launches = sum(kernels[name] for name, _ in parts) * args.steps
    code, detail = binding.device_status()
    if code != binding.OK:
        raise RuntimeError(f"device status after the timed steps: {code} {detail}")

    tot = max_over_ranks({name: sum(v) for name, v in ms.items()}, dev)
    peaks = measured_peaks()

    roofline = dec_block = None
    value = unit = None
    if do_pre:
        flops = w.flops()
        value = job_rate(flops, args.steps, world, tot["prefill"]) / 1e12
        unit = "TFLOP/s"
        achieved = flops / (statistics.mean(ms["prefill"]) / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"],
                    "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"]
                                          if peaks.get("bf16_tflops_sustained") else None),
                    "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                    "traffic": profiled_traffic("attn_fwd_kernel_causal_gqa_traffic.txt",
                                                ("fwd_kernel.cuh", "ptx.cuh")),
                    "algorithmic_flops_per_launch": flops, "kernel": "attn_fwd_kernel<128>"}
    if do_dec:
        dec_bytes = int(sl_h.sum()) * wd.Hkv * wd.d * 2 * 2 + 2 * wd.B * wd.Hq * wd.d * 2 + 4 * wd.B * wd.Hq
        dec_value = job_rate(dec_bytes, args.steps, world, tot["decode"]) / 1e9
        dec_achieved = dec_bytes / (statistics.mean(ms["decode"]) / 1e3) / 1e9
        dec_roof = {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": dec_achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} copy bandwidth",
                    "traffic": profiled_traffic("attn_decode_kernel_gqa_traffic.txt",
                                                ("decode_kernel.cuh", "ptx.cuh")),
                    "algorithmic_bytes_per_launch": dec_bytes, "kernel": "attn_decode_kernel<128,4>"}
        dec_block = {"metric": "decode GB/s (cache rows read + q/o/lse)", "value": dec_value, "unit": "GB/s",
                     "ms": tot["decode"] / args.steps, "roofline": dec_roof}
        if not do_pre:   # decode alone: its numbers are the line's
            value, unit, roofline = dec_value, "GB/s", dec_roof
    win_block = None
    if do_win:
        # FLOPs of the pairs that are actually visible: row i sees min(i+1, WINDOW) keys
        pairs = sum(min(i + 1, WINDOW) for i in range(ww.Nq))
        win_flops = 4.0 * ww.B * ww.Hq * ww.d * pairs
        win_value = job_rate(win_flops, args.steps, world, tot["window"]) / 1e12
        win_achieved = win_flops / (statistics.mean(ms["window"]) / 1e3) / 1e12
        win_roof = {"bound": "tensor", "achieved": win_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": win_achieved / peaks["bf16_tflops"], "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                    "traffic": None, "algorithmic_flops_per_launch": win_flops,
                    "kernel": "attn_fwd_kernel<128, window>"}
        win_block = {"metric": "causal sliding-window prefill TFLOP/s (visible pairs only)",
                     "workload": f"{ww.name}_window{WINDOW}", "value": win_value, "unit": "TFLOP/s",
                     "ms": tot["window"] / args.steps, "roofline": win_roof}
        if not (do_pre or do_dec or do_pag):
            value, unit, roofline = win_value, "TFLOP/s", win_roof
    pag_block = None
    if do_pag:
        pag_bytes = ((int(psl_h.sum()) + wp.B) * wp.Hkv * wp.d * 2 * 2 + 2 * wp.B * wp.Hq * wp.d * 2
                     + 4 * wp.B * wp.Hq + 2 * wp.B * wp.Hkv * wp.d * 2 * 2)
        pag_value = job_rate(pag_bytes, args.steps, world, tot["paged"]) / 1e9
        pag_achieved = pag_bytes / (statistics.mean(ms["paged"]) / 1e3) / 1e9
        pag_roof = {"bound": "hbm", "achieved": pag_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": pag_achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} copy bandwidth",
                    "traffic": None, "algorithmic_bytes_per_launch": pag_bytes,
                    "kernel": "attn_decode_kernel<128,4> (paged, append)"}
        pag_block = {"metric": "paged decode + append GB/s (cache rows read incl. the new token, q/o/lse, "
                               "appended rows read and written)", "workload": wp.name, "value": pag_value,
                     "unit": "GB/s", "ms": tot["paged"] / args.steps, "roofline": pag_roof}
        if not do_pre and not do_dec:
            value, unit, roofline = pag_value, "GB/s", pag_roof

    bwd_block = None
    if do_bwd:
        # The usual convention for the backward: 2.5x the forward's FLOPs (five
        # products of the forward's size: S, dP, dV, dK, dQ); the recomputation
        # of S and dP in the dQ kernel is not counted.
        bwd_flops = 2.5 * w.flops()
        bwd_value = job_rate(bwd_flops, args.steps, world, tot["backward"]) / 1e12
        bwd_achieved = bwd_flops / (statistics.mean(ms["backward"]) / 1e3) / 1e12
        bwd_roof = {"bound": "tensor", "achieved": bwd_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": bwd_achieved / peaks["bf16_tflops"],
                    "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
                    "traffic": profiled_traffic("attn_bwd_causal_gqa_traffic.txt", ("bwd_kernel.cuh", "ptx.cuh")),
                    "traffic_note": "DRAM bytes of one backward call (dK/dV + dQ kernels), from the ncu capture",
                    "algorithmic_flops_per_launch": bwd_flops,
                    "kernel": "bwd_prep_kernel<128> + attn_bwd_dkdv_kernel<128> + attn_bwd_dq_kernel<128>"}
        bwd_block = {"metric": "causal attention backward TFLOP/s (2.5x forward FLOPs)", "workload": w.name,
                     "value": bwd_value, "unit": "TFLOP/s", "ms": tot["backward"] / args.steps,
                     "roofline": bwd_roof}
        if not (do_pre or do_dec or do_pag or do_win):
            value, unit, roofline = bwd_value, "TFLOP/s", bwd_roof

    rope_block = None
    if do_rope:
        # The pre-pass (table + rotated K) is inside the timed call; FLOPs are the prefill's.
        rflops = w.flops()
        rope_value = job_rate(rflops, args.steps, world, tot["rope"]) / 1e12
        rope_achieved = rflops / (statistics.mean(ms["rope"]) / 1e3) / 1e12
        rope_roof = {"bound": "tensor", "achieved": rope_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": rope_achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)", "traffic": None,
                     "algorithmic_flops_per_launch": rflops,
                     "kernel": "rope_table_kernel<128> + rope_k_kernel<128> + attn_fwd_kernel<128> (RoPE on Q)"}
        rope_block = {"metric": "causal prefill with RoPE TFLOP/s (prefill FLOPs; table and K rotation included)",
                      "workload": f"{w.name}_rope10000", "value": rope_value, "unit": "TFLOP/s",
                      "ms": tot["rope"] / args.steps, "roofline": rope_roof}
        if args.only == "rope":
            value, unit, roofline = rope_value, "TFLOP/s", rope_roof

    e2e = None
    if do_pre and not args.no_e2e:   # every rank measures its own replica; rank 0 reports the aggregate
        e2e = measure_e2e(args, w, q_h, k_h, v_h, dev)
        e2e["value"] *= world

    cpu = None
    if do_pre and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q_h, k_h, v_h)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sum(tot.values()) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": (w.name if do_pre else wd.name if do_dec else W.DECODE_GQA_PAGED.name if do_pag
                                    else f"{W.CAUSAL_GQA_16384.name}_window{WINDOW}" if do_win
                                    else f"{w.name}_backward" if do_bwd else f"{w.name}_rope10000"),
                       "l2": "flushed before every timed launch: 256 MiB written, then 256 MiB read (no dirty lines left)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        }
        if do_pre and do_dec:
            line["config"]["decode_workload"] = wd.name
        if do_pre:
            line["prefill_ms"] = tot["prefill"] / args.steps
        line["per_step_ms"] = {name: [round(x, 4) for x in v] for name, v in ms.items()}
        if do_pre and do_dec:
            line["decode"] = dec_block
        if pag_block is not None and (do_pre or do_dec):
            line["decode_paged"] = pag_block
        if win_block is not None and (do_pre or do_dec or do_pag):
            line["prefill_window"] = win_block
        if bwd_block is not None and (do_pre or do_dec or do_pag or do_win):
            line["backward"] = bwd_block
        if rope_block is not None and args.only != "rope":
            line["prefill_rope"] = rope_block
        line.update({"roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * world,
                     "clocks": clocks, "wall_s_timed_region": t_wall})
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(args, w, q_h, k_h, v_h, dev):
    """Prefill through the public API from pinned host buffers: per step the
    H2D copy of q, k, v, the launch, and the D2H copy of o and lse."""
    from exact_scaled_dot_03_b300 import binding as B
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty_like(q_h).pin_memory()
    lp = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32).pin_memory()
    qd, kd, vd = torch.empty_like(qp, device=dev), torch.empty_like(kp, device=dev), torch.empty_like(vp, device=dev)
    od = torch.empty_like(qd)
    ld = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32, device=dev)
    steps = max(1, min(args.steps, 10))

    def step():
        qd.copy_(qp, non_blocking=True)
        kd.copy_(kp, non_blocking=True)
        vd.copy_(vp, non_blocking=True)
        B.fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld)
        op.copy_(od, non_blocking=True)
        lp.copy_(ld, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    h2d = (qp.numel() + kp.numel() + vp.numel()) * 2
    d2h = op.numel() * 2 + lp.numel() * 4
    return {"value": w.flops() / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill", default=W.CAUSAL_GQA_16384.name, choices=sorted(PREFILL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["prefill", "decode", "paged", "window", "backward", "rope"], default=None,
                    help="time one kernel alone (profiling); the JSON line then carries only its numbers")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    w = PREFILL[args.prefill]
    wd = W.DECODE_GQA
    if args.impl == "reference":
        run_reference(args, w, wd)
    else:
        run_ours(args, w, wd)


if __name__ == "__main__":
    main()
