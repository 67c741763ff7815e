"""Benchmark: exact attention prefill (TFLOP/s) and KV-cache decode (GB/s) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--prefill NAME] [--only PART] [--no-cpu-baseline] [--no-e2e]

One step = one pass of the whole hot path over synthetic bf16 inputs that are
already resident in device memory, one timed launch per part:
  prefill         causal GQA prefill B=1 Hq=64 Hkv=8 N=16384 d=128 (the line's value)
  decode          B=16 Hq=32 Hkv=8 d=128, cache lengths uniform on [1024, 8192]
  c1_single_head  B=1 H=1 N=128 d=64, non-causal
  c2_mha_d64      B=4 H=12 N=2048 d=64, non-causal
  c3_causal_mha   B=2 H=32 N=4096 d=128, causal
  paged           the decode over a paged cache (64-token pages), new token appended
and, in a second loop (their full tensor load would otherwise keep the part at
its power cap while the prefill is timed), the causal GQA prefill with a
4096-key sliding window, the backward pass of the causal GQA prefill (dQ, dK,
dV from the o and lse its prefill wrote and a seeded dO) and that prefill with
rotary position embedding (base 10000). L2 is flushed before every timed
launch, outside its CUDA-event bracket: a 256 MiB write, then a 256 MiB read
so the timed kernel does not pay for writing back the flush's dirty lines.
Prints one JSON line.

``value`` is the causal GQA prefill's TFLOP/s (4*B*Hq*Nq*Nk*d, halved for
causal); every other part has its own block with its own roofline (decode:
GB/s of the cache rows actually read, sum(seqlens)*Hkv*d*2*2 bytes, plus q, o
and lse). Each roofline gives the fraction of the measured peak and of the
nominal B300 peak. The decode block also carries, as context, the rate of a
plain device copy moving the same number of bytes, timed after the timed
region the same way. Under torchrun every rank runs the same workload
(replicas; weak scaling) and rank 0 prints the aggregate over the
max-over-ranks time.

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
# The other prefill workloads, each timed as its own part of the step.
EXTRA_PREFILL = (("c1_single_head", W.SINGLE_HEAD), ("c2_mha_d64", W.MHA_2048),
                 ("c3_causal_mha", W.CAUSAL_MHA_4096))
# Nominal B300 figures the stated targets are written against (dense bf16 tensor
# rate, HBM3e bandwidth): every roofline block also reports its fraction of these.
SPEC_BF16_TFLOPS = 2250.0
SPEC_HBM_GBS = 8000.0
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
    # Not a measurement of this GPU: an earlier B300 reading, used only when the
    # measured file is missing, and labelled as such in every block.
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "FALLBACK (not measured on this GPU)"}


def tensor_roof(achieved, peaks, flops, kernel, traffic=None, **extra):
    """Roofline block of a tensor-bound kernel: TFLOP/s against the measured
    cuBLAS bf16 burst peak and against the nominal dense bf16 rate."""
    r = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
         "frac": achieved / peaks["bf16_tflops"],
         "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"]
                               if peaks.get("bf16_tflops_sustained") else None),
         "frac_of_spec": achieved / SPEC_BF16_TFLOPS, "spec_peak": SPEC_BF16_TFLOPS,
         "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)", "traffic": traffic,
         "algorithmic_flops_per_launch": flops, "kernel": kernel}
    r.update(extra)
    return r


def hbm_roof(achieved, peaks, nbytes, kernel, traffic=None, **extra):
    """Roofline block of an HBM-bound kernel: GB/s against the measured copy
    bandwidth and against the nominal HBM3e bandwidth."""
    r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": achieved / peaks["hbm_gbs"], "frac_of_spec": achieved / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
         "peak_source": f"{peaks['source']} copy bandwidth", "traffic": traffic,
         "algorithmic_bytes_per_launch": nbytes, "kernel": kernel}
    r.update(extra)
    return r


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
    on = lambda name: args.only in (None, name)  # noqa: E731
    do_pre, do_dec, do_pag, do_win, do_bwd, do_rope = (on(n) for n in
                                                      ("prefill", "decode", "paged", "window", "backward", "rope"))
    extra = [(name, wx) for name, wx in EXTRA_PREFILL if on(name)]

    parts = []  # (name, launch function)
    # our kernel launches per call
    kernels = {"prefill": 1, "decode": 1, "window": 1, "paged": 1, "backward": 3, "rope": 3,
               **{name: 1 for name, _ in EXTRA_PREFILL}}
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
    for name, wx in extra:
        xq, xk, xv = (t.to(dev) for t in W.prefill_inputs(wx))
        xo = torch.empty_like(xq)
        xl = torch.empty(wx.B, wx.Hq, wx.Nq, dtype=torch.float32, device=dev)
        parts.append((name, lambda wx=wx, xq=xq, xk=xk, xv=xv, xo=xo, xl=xl:
                      binding.fwd(xq, xk, xv, causal=wx.causal, scale=wx.scale, out=xo, lse=xl)))
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
    # The backward, the RoPE prefill and the sliding-window prefill are timed
    # in their own loop after the others: their full tensor load (each a
    # multi-millisecond launch per step) would otherwise hold the part at its
    # power cap while the prefill is timed.
    later = ("backward", "rope", "window")
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
    copy_ctx = None
    if do_dec:
        # Context for the decode's roofline, outside the timed region: a plain
        # device copy moving the same number of bytes (half read, half written).
        nb = int(sl_h.sum()) * wd.Hkv * wd.d * 2 * 2 + 2 * wd.B * wd.Hq * wd.d * 2 + 4 * wd.B * wd.Hq
        src = torch.empty(nb // 2, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        cts = []
        for r in range(args.warmup + args.steps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src)
            e1.record(stream)
            torch.cuda.synchronize()
            if r >= args.warmup:
                cts.append(e0.elapsed_time(e1))
        cms = statistics.median(cts)
        copy_ctx = {"value": 2 * (nb // 2) / (cms / 1e3) / 1e9, "unit": "GB/s", "ms": cms,
                    "what": "torch copy_ of half the decode's bytes into a second buffer (the same bytes moved), "
                            "L2 flushed, median; context for the decode's roofline fraction, not a peak"}
        del src, dst
    mean_s = lambda name: statistics.mean(ms[name]) / 1e3  # noqa: E731  (seconds per launch)

    blocks = {}  # name -> block, in the order they are printed
    headline = None
    if do_pre:
        flops = w.flops()
        blocks["prefill"] = {
            "metric": "causal prefill TFLOP/s", "workload": w.name,
            "value": job_rate(flops, args.steps, world, tot["prefill"]) / 1e12, "unit": "TFLOP/s",
            "ms": tot["prefill"] / args.steps,
            "roofline": tensor_roof(flops / mean_s("prefill") / 1e12, peaks, flops, "attn_fwd_kernel<128>",
                                    profiled_traffic("attn_fwd_kernel_causal_gqa_traffic.txt",
                                                     ("fwd_kernel.cuh", "ptx.cuh")))}
    if do_dec:
        dec_bytes = int(sl_h.sum()) * wd.Hkv * wd.d * 2 * 2 + 2 * wd.B * wd.Hq * wd.d * 2 + 4 * wd.B * wd.Hq
        blocks["decode"] = {
            "metric": "decode GB/s (cache rows read + q/o/lse)", "workload": wd.name,
            "value": job_rate(dec_bytes, args.steps, world, tot["decode"]) / 1e9, "unit": "GB/s",
            "ms": tot["decode"] / args.steps,
            "roofline": hbm_roof(dec_bytes / mean_s("decode") / 1e9, peaks, dec_bytes, "attn_decode_kernel<128,4>",
                                 profiled_traffic("attn_decode_kernel_gqa_traffic.txt",
                                                  ("decode_kernel.cuh", "ptx.cuh"))),
            "device_copy_same_bytes": copy_ctx}
    for name, wx in extra:
        f = wx.flops()
        blk = {"metric": f"{'causal ' if wx.causal else ''}prefill TFLOP/s", "workload": wx.name,
               "value": job_rate(f, args.steps, world, tot[name]) / 1e12, "unit": "TFLOP/s",
               "ms": tot[name] / args.steps, "us_per_launch": 1e6 * mean_s(name),
               "roofline": tensor_roof(f / mean_s(name) / 1e12, peaks, f, f"attn_fwd_kernel<{wx.d}>")}
        if name == "c1_single_head":
            blk["note"] = "one CTA: latency-bound by construction; the fraction is reported, not a target"
        blocks[name] = blk
    if do_win:
        # FLOPs of the pairs that are actually visible: row i sees min(i+1, WINDOW) keys
        pairs = sum(min(i + 1, WINDOW) for i in range(ww.Nq))
        win_flops = 4.0 * ww.B * ww.Hq * ww.d * pairs
        blocks["prefill_window"] = {
            "metric": "causal sliding-window prefill TFLOP/s (visible pairs only)",
            "workload": f"{ww.name}_window{WINDOW}",
            "value": job_rate(win_flops, args.steps, world, tot["window"]) / 1e12, "unit": "TFLOP/s",
            "ms": tot["window"] / args.steps,
            "roofline": tensor_roof(win_flops / mean_s("window") / 1e12, peaks, win_flops,
                                    "attn_fwd_kernel<128, window>")}
    if do_pag:
        pag_bytes = ((int(psl_h.sum()) + wp.B) * wp.Hkv * wp.d * 2 * 2 + 2 * wp.B * wp.Hq * wp.d * 2
                     + 4 * wp.B * wp.Hq + 2 * wp.B * wp.Hkv * wp.d * 2 * 2)
        blocks["decode_paged"] = {
            "metric": "paged decode + append GB/s (cache rows read incl. the new token, q/o/lse, "
                      "appended rows read and written)", "workload": wp.name,
            "value": job_rate(pag_bytes, args.steps, world, tot["paged"]) / 1e9, "unit": "GB/s",
            "ms": tot["paged"] / args.steps,
            "roofline": hbm_roof(pag_bytes / mean_s("paged") / 1e9, peaks, pag_bytes,
                                 "attn_decode_kernel<128,4> (paged, append)")}
    if do_bwd:
        # The usual convention for the backward: 2.5x the forward's FLOPs (five
        # products of the forward's size: S, dP, dV, dK, dQ); the recomputation
        # of S and dP in the dQ kernel is not counted.
        bwd_flops = 2.5 * w.flops()
        blocks["backward"] = {
            "metric": "causal attention backward TFLOP/s (2.5x forward FLOPs)", "workload": w.name,
            "value": job_rate(bwd_flops, args.steps, world, tot["backward"]) / 1e12, "unit": "TFLOP/s",
            "ms": tot["backward"] / args.steps,
            "roofline": tensor_roof(bwd_flops / mean_s("backward") / 1e12, peaks, bwd_flops,
                                    "bwd_prep_kernel<128> + attn_bwd_dkdv_kernel<128> + attn_bwd_dq_kernel<128>",
                                    profiled_traffic("attn_bwd_causal_gqa_traffic.txt", ("bwd_kernel.cuh", "ptx.cuh")),
                                    traffic_note="DRAM bytes of one backward call (dK/dV + dQ kernels), "
                                                 "from the ncu capture")}
    if do_rope:
        # The pre-pass (table + rotated K) is inside the timed call; FLOPs are the prefill's.
        rflops = w.flops()
        blocks["prefill_rope"] = {
            "metric": "causal prefill with RoPE TFLOP/s (prefill FLOPs; table and K rotation included)",
            "workload": f"{w.name}_rope10000",
            "value": job_rate(rflops, args.steps, world, tot["rope"]) / 1e12, "unit": "TFLOP/s",
            "ms": tot["rope"] / args.steps,
            "roofline": tensor_roof(rflops / mean_s("rope") / 1e12, peaks, rflops,
                                    "rope_table_kernel<128> + rope_k_kernel<128> + attn_fwd_kernel<128> (RoPE on Q)")}
    # The line's own value: the causal GQA prefill, else the one part timed alone.
    head_name = "prefill" if do_pre else next(iter(blocks))
    headline = blocks.pop(head_name)

    e2e = None
    if do_pre and not args.no_e2e:   # every rank measures its own replica; rank 0 reports the aggregate
        e2e = measure_e2e(args, w, q_h, k_h, v_h, dev)
        e2e["value"] *= world

    cpu = None
    if do_pre and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q_h, k_h, v_h)

    if rank == 0:
        line = {
            "metric": METRIC, "value": headline["value"], "unit": headline["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(tot.values()) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": headline["workload"],
                       "l2": "flushed before every timed launch: 256 MiB written, then 256 MiB read (no dirty lines left)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": headline["roofline"],
            "peaks_used": {"bf16_tflops": peaks["bf16_tflops"], "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                           "hbm_gbs": peaks["hbm_gbs"], "source": peaks["source"],
                           "spec_bf16_tflops": SPEC_BF16_TFLOPS, "spec_hbm_gbs": SPEC_HBM_GBS},
        }
        if head_name == "prefill":
            line["prefill_ms"] = headline["ms"]
        if headline.get("device_copy_same_bytes") is not None:
            line["device_copy_same_bytes"] = headline["device_copy_same_bytes"]
        # Short blocks first (the five workloads), the longer ones after.
        line.update(blocks)
        line.update({"cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * world,
                     "clocks": clocks, "wall_s_timed_region": t_wall,
                     "median_ms": {name: round(statistics.median(v), 4) for name, v in ms.items()}})
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(args, w, q_h, k_h, v_h, dev):
    """Prefill through the public host-buffer API (attn_fwd_host) from pinned
    host memory: every step copies q, k, v in and o, lse out, pipelined per
    (batch, KV head) chunk against the kernels; the step ends when the last
    copy out has landed."""
    from exact_scaled_dot_03_b300 import binding as B
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty_like(q_h).pin_memory()
    lp = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32).pin_memory()
    ws = torch.empty(B.fwd_host_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d), dtype=torch.uint8, device=dev)
    steps = max(1, min(args.steps, 10))

    def step():
        B.fwd_host(qp, kp, vp, causal=w.causal, scale=w.scale, out=op, lse=lp, workspace=ws)

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
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps, "api": "attn_fwd_host"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill", default=W.CAUSAL_GQA_16384.name, choices=sorted(PREFILL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["prefill", "decode", "paged", "window", "backward", "rope",
                                       *(name for name, _ in EXTRA_PREFILL)], default=None,
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
