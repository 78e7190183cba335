"""Benchmark of the jagged flash attention hot path (forward + backward).

One step = jfa_fwd + jfa_bwd over one batch of the jagged self-attention
workload (B=64 sequences, lengths uniform in [16, 2048], H=8, D=128, bf16,
non-causal).  value = useful TFLOPS on true lengths: (4 + 10) * H * D * pairs
per step.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the fp64 CPU oracle on the host cores (bounded
sample of the same workload); there is no GPU reference implementation.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import jfa_workloads as W  # noqa: E402

METRIC = "JFA fwd and bwd useful TFLOPS (bf16) and % of GB300 tensor peak"
DEFAULT_WORKLOAD = "jagged_self"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _flops(x):
    p = W.pairs(x["lengths"], x["causal"], x["q_len"], x["broadcast_q"])
    f = 4.0 * x["H"] * x["D"] * p
    return f, 2.5 * f, p


# Algorithmic tensor-core FLOPs of one launch of each product kernel, per
# head and query-key pair (2 * D per product): forward S and PV; dK/dV pass
# S^T, dP^T, dV, dK; dQ pass S, dP, dQ; broadcast-Q backward all five.
KERNEL_FLOPS_PER_PAIR_D = {"fwd": 4.0, "bwd_kv": 8.0, "bwd_q": 6.0, "bwd_fused": 10.0}
KERNEL_DESC = {
    "fwd": "forward (S = QK^T, O += PV)",
    "bwd_kv": "backward dK/dV pass (S^T, dP^T, dV += P^T dO, dK += dS^T Q)",
    "bwd_q": "backward dQ pass (S, dP, dQ += dS K)",
    "bwd_fused": "broadcast-Q backward (five products)",
}
# DRAM bytes (read + write) per launch from one ncu capture of the kernels
# as they are now, on the jagged self-attention workload (B=64, H=8, D=128;
# profiles/dram_jagged_self.md has the command and the split); to be reset
# to {} whenever one of these kernels changes.
KERNEL_TRAFFIC = {
    "jagged_self": {"fwd": 449209856 + 120235520, "bwd_kv": 606568448 + 253562112,
                    "bwd_q": 627318528 + 126046720},
}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, ws, device="cpu"):
    """The job's figure for a per-rank time: its maximum over all ranks (one
    all-reduce, which every rank calls; it also orders the ranks like a
    barrier).  One rank: the value itself."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ws, step_flops, ms_per_step):
    """Whole-job TFLOPS: each of the ws ranks runs one replica of the step,
    and the step takes ms_per_step (the slowest rank's time)."""
    return ws * step_flops / (ms_per_step * 1e-3) / 1e12


def _oracle_sample(x, budget_s, max_seqs=None):
    """Time the fp64 oracle (fwd + bwd) on the workload's sequences, in order,
    until `budget_s` seconds of CPU work; returns (flops, seconds, n_seqs)."""
    from oracle import jfa_oracle as orc
    f64 = lambda t: t.float().numpy().astype(np.float64)
    off = x["offsets"]
    L = x["lengths"]
    tot_f, tot_t, n = 0.0, 0.0, 0
    order = range(len(L)) if max_seqs is None else range(min(max_seqs, len(L)))
    for b in order:
        s0, s1 = int(off[b]), int(off[b + 1])
        if x["broadcast_q"]:
            q = f64(x["q"])
            do = f64(x["dout"][b:b + 1])
        else:
            q = f64(x["q"][s0:s1])
            do = f64(x["dout"][s0:s1])
        k, v = f64(x["k"][s0:s1]), f64(x["v"][s0:s1])
        sub = [0, s1 - s0]
        t0 = time.perf_counter()
        orc.forward(q, k, v, sub, x["scale"], x["causal"], x["broadcast_q"])
        orc.backward(q, k, v, sub, do, x["scale"], x["causal"], x["broadcast_q"])
        tot_t += time.perf_counter() - t0
        p = W.pairs([s1 - s0], x["causal"], x["q_len"], x["broadcast_q"])
        tot_f += 14.0 * x["H"] * x["D"] * p
        n += 1
        if tot_t >= budget_s:
            break
    return tot_f, tot_t, n


def run_reference(args, x, wname):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    for _ in range(args.warmup):
        _oracle_sample(x, 0.0, max_seqs=1)
    per_step = []
    flops = []
    nseq = 0
    for _ in range(args.steps):
        f, t, n = _oracle_sample(x, args.ref_step_seconds)
        per_step.append(t)
        flops.append(f)
        nseq = n
    tf = sum(flops) / sum(per_step) / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(per_step) / len(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wname, **_cfg(x, wname)},
        "cpu_baseline": {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"first {nseq} sequences (all heads) per step, fwd+bwd"},
        "e2e": {"value": tf, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _cfg(x, wname):
    return {"B": int(x["B"]), "H": x["H"], "D": x["D"], "T": x["T"], "causal": x["causal"],
            "broadcast_q": x["broadcast_q"], "q_len": x["q_len"], "max_len": x["max_len"],
            "lengths": W.WORKLOADS[wname].lengths_desc, "seed": W.WORKLOADS[wname].seed}


def run_ours(args, x, wname):
    import torch
    import jagged_flash_attention_gb300 as jfa

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    jfa.lib()
    peak, peak_sus, hbm, peak_src = _peaks()
    fwd_f, bwd_f, pairs = _flops(x)
    step_f = fwd_f + bwd_f
    B, H, D, Lq = x["B"], x["H"], x["D"], x["q_len"]
    bq, causal, scale, max_len = x["broadcast_q"], x["causal"], x["scale"], x["max_len"]

    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    out, lse = jfa.forward(q, k, v, off, max_len, causal=causal, broadcast_q=bq, scale=scale)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    stream = torch.cuda.current_stream()

    def fwd():
        jfa.forward(q, k, v, off, max_len, causal=causal, broadcast_q=bq, scale=scale, out=out,
                    lse=lse)

    def bwd():
        jfa.backward(q, k, v, off, max_len, out, lse, do, causal=causal, broadcast_q=bq,
                     scale=scale, dq=dq, dk=dk, dv=dv)

    for _ in range(args.warmup):
        fwd()
        bwd()
    jfa.jfa_sync_and_check()
    jfa.profile_read()  # discard anything recorded before the timed region

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = jfa.launch_count()
    jfa.profile_enable(True)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    jfa.profile_enable(False)
    launches = jfa.launch_count() - launches0
    kprof = jfa.profile_read()
    if ws > 1:
        torch.distributed.barrier()
    jfa.jfa_sync_and_check()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), ws, dev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_per_step = total_ms / args.steps
    value = job_value(ws, step_f, ms_per_step)

    # End to end through the public API: every step copies its inputs from
    # pinned host memory to the device, makes the two calls and copies every
    # result (out, lse, dq, dk, dv) back to pinned host memory.  Steps are
    # pipelined the way a streaming caller runs them: host->device copies,
    # compute and device->host copies on three streams with two device buffer
    # sets, so step i+1's inputs move in and step i-1's results move out while
    # step i computes.  The timed region spans the first input copy to the
    # last result copy.
    hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "dout"))
    hoff = torch.from_numpy(x["offsets"]).pin_memory()
    ho, hl = torch.empty_like(out, device="cpu").pin_memory(), torch.empty_like(lse, device="cpu").pin_memory()
    hdq, hdk, hdv = (torch.empty_like(t, device="cpu").pin_memory() for t in (dq, dk, dv))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hoff))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl, hdq, hdk, hdv))
    e2e_steps = max(3, min(args.steps, 10))
    sets = [dict(q=q, k=k, v=v, do=do, off=off, out=out, lse=lse, dq=dq, dk=dk, dv=dv)]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(cmp_done[i % 2])  # step i-2 has consumed this set's inputs
            for h, n in ((hq, "q"), (hk, "k"), (hv, "v"), (hdo, "do"), (hoff, "off")):
                b[n].copy_(h, non_blocking=True)
            in_done[i % 2].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(in_done[i % 2])
            if i >= 2:
                s_cmp.wait_event(out_done[i % 2])  # step i-2's results have left this set
            jfa.forward(b["q"], b["k"], b["v"], b["off"], max_len, causal=causal, broadcast_q=bq,
                        scale=scale, out=b["out"], lse=b["lse"])
            jfa.backward(b["q"], b["k"], b["v"], b["off"], max_len, b["out"], b["lse"], b["do"],
                         causal=causal, broadcast_q=bq, scale=scale, dq=b["dq"], dk=b["dk"],
                         dv=b["dv"])
            cmp_done[i % 2].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[i % 2])
            for n, h in (("out", ho), ("lse", hl), ("dq", hdq), ("dk", hdk), ("dv", hdv)):
                h.copy_(b[n], non_blocking=True)
            out_done[i % 2].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(2, 2 + e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    jfa.jfa_sync_and_check()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    e2e_val = job_value(ws, step_f, e2e_ms)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        f, t, n = _oracle_sample(x, args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": "TFLOPS", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"first {n} of {B} sequences, all {H} heads, fwd+bwd in fp64 "
                         f"({t:.1f} s)"}
    bwd_tf = bwd_f / (bwd_ms * 1e-3) / 1e12
    fwd_tf = fwd_f / (fwd_ms * 1e-3) / 1e12
    # Per-kernel device time over the timed region (events on the launching
    # stream, recorded by the library); roofline of the dominant kernel.
    kernels = {k: {"ms_per_launch": t / n, "launches": n, "share": 0.0}
               for k, (t, n) in kprof.items() if n > 0}
    tot = sum(t for t, n in kprof.values())
    for k, (t, n) in kprof.items():
        if n > 0:
            kernels[k]["share"] = t / tot
    dom = max((k for k in kernels if k in KERNEL_FLOPS_PER_PAIR_D),
              key=lambda k: kprof[k][0])
    dom_flops = KERNEL_FLOPS_PER_PAIR_D[dom] * H * D * pairs
    dom_tf = dom_flops / (kernels[dom]["ms_per_launch"] * 1e-3) / 1e12
    for k, v in kernels.items():
        if k in KERNEL_FLOPS_PER_PAIR_D:
            v["tflops"] = KERNEL_FLOPS_PER_PAIR_D[k] * H * D * pairs / (v["ms_per_launch"] * 1e-3) / 1e12
        tr = KERNEL_TRAFFIC.get(wname, {}).get(k)
        if tr is not None:
            v["dram_bytes"] = tr
            v["dram_gbs"] = tr / (v["ms_per_launch"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wname, **_cfg(x, wname), "pairs": pairs,
                   "l2": "inputs larger than L2 (q,k,v,dout,out each "
                         f"{x['q'].numel() * 2 / 1e6:.0f} MB); no flush",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "frac_of_peak": value / peak,
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak},
        "roofline": {"bound": "tensor", "kernel": KERNEL_DESC[dom],
                     "algorithmic_tflop_per_launch": dom_flops / 1e12,
                     "ms_per_launch": kernels[dom]["ms_per_launch"],
                     "achieved": dom_tf, "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "traffic": KERNEL_TRAFFIC.get(wname, {}).get(dom),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)"},
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "schedule": "every step copies all inputs in and all results out; input "
                            "copies, compute and result copies pipelined on three streams "
                            "with two device buffer sets"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.ORDER)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="draw this many sequences instead of the workload's B "
                         "(same length distribution; for profiling captures)")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    lengths = None if args.batch is None else W.sample_lengths(w, B=args.batch)
    x = W.make_inputs(w, lengths=lengths)
    if args.impl == "reference":
        run_reference(args, x, args.workload)
    else:
        run_ours(args, x, args.workload)


if __name__ == "__main__":
    main()
