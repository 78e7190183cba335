"""Benchmark of the jagged flash attention hot path (forward + backward).

One step = jfa_fwd + jfa_bwd over one batch of a workload.  The headline
workload is the jagged self-attention batch (B=64 sequences, lengths uniform
in [16, 2048], H=8, D=128, bf16, non-causal); value = useful TFLOPS on true
lengths: (4 + 10) * H * D * pairs per step.  The same JSON line carries, under
`workloads`, the other four workloads (tiny self-attention, broadcast-Q,
causal self-attention, skewed broadcast-Q), each device-timed with its
per-kernel roofline fractions.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--only]

--only times the named workload alone (no `workloads` object).
--impl reference times the fp64 CPU oracle on the host cores (bounded sample
of the same workload); there is no GPU reference implementation.
"""
import argparse
import contextlib
import datetime
import hashlib
import json
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
L2_BYTES = 129 * 2 ** 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _pairs(x):
    return W.pairs(x["lengths"], x["causal"], x["q_len"], x["broadcast_q"],
                   x.get("window", (-1, -1)))


def _flops(x):
    p = _pairs(x)
    f = 4.0 * x["H"] * x["D"] * p
    return f, 2.5 * f, p


KERNEL_DESC = {
    "sched": "forward work-list scheduler",
    "fwd": "forward (S = QK^T, O += PV)",
    "prep": "backward pre-pass (work lists, LSE*log2e, Delta = rowsum(dO*O))",
    "bwd_kv": "backward dK/dV pass (S^T, dP^T, dV += P^T dO, dK += dS^T Q)",
    "bwd_q": "self-attention backward dQ pass (S, dP, dQ += dS K)",
    "bwd_qb": "broadcast-Q backward dQ pass (S, dP, dQ += dS K over key-tile chunks)",
    "finalize": "broadcast-Q dQ: sum of the chunk partials, bf16",
    "bwd_bs": "broadcast-Q backward in one pass (short dense Q): dK, dV and dQ partials",
    "fwd_combine": "broadcast-Q forward: merge of split sequences",
    "sparse_pool": "block-sparse selection: K-block and Q-block means",
    "sparse_select": "block-sparse selection: scores and top-k per Q block",
    "bwd_kv_pair": "backward dK/dV pass on CTA pairs (cta_group::2 products over two key blocks)",
    "sparse_check": "block-sparse forward: check of every block list",
}


def kernel_model(x):
    """Algorithmic work of one launch of each kernel kind on workload x:
    {kind: (tensor FLOPs, DRAM bytes)}.  FLOPs count true (query, key) pairs
    (2 * D per pair and product); bytes count each tensor the kernel must
    read or write once: Q rows are T (self) or q_len (broadcast), O / dO rows
    T or B * q_len, K / V rows T (with H_kv heads); bf16 tensors, fp32 LSE
    and statistics (8 bytes per row and head; self-attention keeps four
    copies).  A window counts only the pairs inside the band."""
    H, D, T, B, Lq = x["H"], x["D"], x["T"], x["B"], x["q_len"]
    bq = x["broadcast_q"]
    pairs = _pairs(x)
    row, rkv = H * D * 2, x.get("Hkv", H) * D * 2
    qrows, orows = (Lq, B * Lq) if bq else (T, T)
    stat = 8 * H * orows
    m = {
        "sched": (0.0, 4.0 * (B + 1)),
        "fwd": (4.0 * H * D * pairs, (qrows + orows) * row + 2 * T * rkv + 4 * H * orows),
        "prep": (0.0, 2 * orows * row + 4 * H * orows + (stat if bq else 4 * stat)),
        "bwd_kv": (8.0 * H * D * pairs, (qrows + orows) * row + 4 * T * rkv + stat),
    }
    m["bwd_kv_pair"] = m["bwd_kv"]
    if bq:
        m["bwd_qb"] = (6.0 * H * D * pairs,
                       (qrows + orows) * row + 2 * T * rkv + stat + 4 * Lq * H * D)
        m["finalize"] = (0.0, 6 * Lq * H * D)
        # one-pass backward of a short dense Q: Q, K, V, dO read, dK, dV written once
        m["bwd_bs"] = (10.0 * H * D * pairs,
                       (qrows + orows) * row + 4 * T * rkv + stat + 4 * Lq * H * D)
        m["fwd_combine"] = (0.0, 0.0)
    else:
        m["bwd_q"] = (6.0 * H * D * pairs, 3 * T * row + 2 * T * rkv + stat)
    # block-sparse selection: K and Q read once (the means are small)
    m["sparse_pool"] = (0.0, T * rkv + T * row)
    m["sparse_select"] = (0.0, 0.0)
    m["sparse_check"] = (0.0, 0.0)
    return m


def step_model(x):
    """(FLOPs, bytes) of the forward and of the backward step: the method's
    useful FLOPs (fwd 4, bwd 10 * H * D * pairs) and the bytes each tensor
    needs once: fwd Q, K, V, O, LSE; bwd Q, K, V, O (for Delta), dO (twice),
    LSE, Delta, and dQ, dK, dV written."""
    H, D, T, B, Lq = x["H"], x["D"], x["T"], x["B"], x["q_len"]
    fwd_f, bwd_f, _ = _flops(x)
    row, rkv = H * D * 2, x.get("Hkv", H) * D * 2
    qrows, orows = (Lq, B * Lq) if x["broadcast_q"] else (T, T)
    fwd_b = (qrows + orows) * row + 2 * T * rkv + 4 * H * orows
    bwd_b = (2 * qrows + 3 * orows) * row + 4 * T * rkv + 8 * H * orows
    return (fwd_f, fwd_b), (bwd_f, bwd_b)


def _roof(flops, nbytes, seconds, peak_tf, hbm_gbs):
    """Roofline fraction max(flops / peak, bytes / bandwidth) / time, and the
    bound that sets it."""
    tf, tb = flops / (peak_tf * 1e12), nbytes / (hbm_gbs * 1e9)
    return (max(tf, tb) / seconds if seconds > 0 else 0.0), ("tensor" if tf >= tb else "hbm")


# DRAM bytes (read + write) per launch measured by ncu, with the sha256 of
# the sources the kernel was built from; bench.py reports a record only while
# those sources are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
KERNEL_SOURCES = {
    "fwd": ["fwd.cu"], "bwd_kv": ["bwd_kv.cu"], "bwd_q": ["bwd_q.cu"], "bwd_qb": ["bwd_qb.cu"],
    "prep": ["aux.cu"], "finalize": ["aux.cu"], "sched": ["aux.cu"], "bwd_bs": ["bwd_bs.cu"],
    "fwd_combine": ["fwd_bs.cu"], "sparse_pool": ["sparse.cu"], "sparse_select": ["sparse.cu"],
    "bwd_kv_pair": ["bwd_kv.cu"], "sparse_check": ["aux.cu"],
}


def source_hash(kind):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "jagged_flash_attention_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kind, []) + ["common.cuh", "ptx.cuh"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_record(kind, wname):
    try:
        with open(TRAFFIC_FILE) as f:
            recs = json.load(f)["records"]
    except Exception:
        return None
    for r in recs:
        if r["kernel"] == kind and r["workload"] == wname:
            return r["bytes_per_launch"] if r["sha256"] == source_hash(kind) else None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, with host timestamps, for
    the whole measurement session; summaries over any time window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []

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
        out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        for l in out.splitlines():
            f = [v.strip() for v in l.split(",")]
            if len(f) < 10:
                continue
            try:
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            try:
                t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None  # unknown time: counted in every window
            reasons = {n for n, v in zip(self.NAMES, f[6:10]) if v.lower() == "active"}
            self.samples.append((t, sm, mx, reasons))

    def summary(self, windows=None):
        """Samples inside any of the (t0, t1) host-time windows (all samples
        if windows is None)."""
        sel = [s for s in self.samples
               if windows is None or s[0] is None or any(t0 <= s[0] <= t1 for t0, t1 in windows)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set().union(*(s[3] for s in sel))
        return {"sm_mhz": statistics.median(s[1] for s in sel),
                "sm_max_mhz": max(s[2] for s in sel), "reasons": sorted(reasons),
                "samples": len(sel)}


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
        win = x.get("window", (-1, -1))
        orc.forward(q, k, v, sub, x["scale"], x["causal"], x["broadcast_q"], window=win)
        orc.backward(q, k, v, sub, do, x["scale"], x["causal"], x["broadcast_q"], window=win)
        tot_t += time.perf_counter() - t0
        p = W.pairs([s1 - s0], x["causal"], x["q_len"], x["broadcast_q"], win)
        tot_f += 14.0 * x["H"] * x["D"] * p
        n += 1
        if tot_t >= budget_s:
            break
    return tot_f, tot_t, n


def _l2_note(x):
    big = x["k"].numel() * 2
    if big > L2_BYTES:
        return f"inputs larger than L2 (k, v {big / 1e6:.0f} MB each); no flush"
    return "inputs fit in L2: a 256 MB buffer is written between timed steps (flush)"


def _workload_def(wname):
    if wname in W.WORKLOADS:
        return W.WORKLOADS[wname]
    if wname in PAIR_VARIANTS:  # the base workload; only the dK/dV pass differs
        return W.WORKLOADS[PAIR_VARIANTS[wname]]
    if wname in SPARSE_VARIANTS:
        return W.WORKLOADS[SPARSE_VARIANTS[wname]]
    return W.variant(wname)


def _config(x, wname, ws=1):
    """The workload description both arms print (same keys)."""
    w = _workload_def(wname)
    return {"workload": wname, "B": int(x["B"]), "H": x["H"], "H_kv": x.get("Hkv", x["H"]),
            "D": x["D"], "T": x["T"], "causal": x["causal"], "broadcast_q": x["broadcast_q"],
            "q_len": x["q_len"], "window": list(x.get("window", (-1, -1))),
            "max_len": x["max_len"], "lengths": w.lengths_desc, "seed": w.seed,
            "pairs": _pairs(x), "l2": _l2_note(x),
            "parallelism": "replicas" if ws > 1 else "single GPU"}


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
        "config": _config(x, wname, args.gpus),
        "cpu_baseline": {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"first {nseq} sequences (all heads) per step, fwd+bwd"},
        "e2e": {"value": tf, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _kernels_entry(x, kprof, peak, hbm, wname):
    """Per kernel kind: mean device time per launch, launches, share, and its
    roofline fraction on the algorithmic work of kernel_model."""
    model = kernel_model(x)
    tot = sum(t for t, n in kprof.values())
    out = {}
    for k, (t, n) in kprof.items():
        if n == 0:
            continue
        ms = t / n
        f, b = model.get(k, (0.0, 0.0))
        frac, bound = _roof(f, b, ms * 1e-3, peak, hbm)
        e = {"ms_per_launch": ms, "launches": n, "share": t / tot if tot else 0.0,
             "tflops": f / (ms * 1e-3) / 1e12, "gbs": b / (ms * 1e-3) / 1e9,
             "bound": bound, "roofline_frac": frac}
        tr = traffic_record(k, wname)
        if tr is not None:
            e["dram_bytes"] = tr
        out[k] = e
    return out


def _breakdown(jfa, torch, x, run_steps, n):
    """Runs n steps with every launch bracketed by a CUDA event pair and
    returns that per-kernel profile; then selects, for the timed region that
    follows, events around the dominant kernel's launches only (by device
    time, among kernels with algorithmic FLOPs): events around every launch
    would add about 1.5% to a step."""
    jfa.profile_read()
    jfa.profile_select(None)
    torch.cuda.synchronize()
    jfa.profile_enable(True)
    run_steps(n)
    torch.cuda.synchronize()
    jfa.profile_enable(False)
    kp = jfa.profile_read()
    model = kernel_model(x)
    ran = [k for k, (t, c) in kp.items() if c > 0]
    cands = [k for k in ran if model.get(k, (0, 0))[0] > 0] or ran
    jfa.profile_select([max(cands, key=lambda k: kp[k][0])])
    return kp


def _time_steps(jfa, torch, x, steps, warmup, stream, dev, min_seconds=0.15):
    """Device-timed fwd / bwd steps of workload x through the public API;
    returns (fwd ms per step, bwd ms per step, kernel profile of the
    breakdown window, launches, host time window of the timed steps)."""
    B, H, D = x["B"], x["H"], x["D"]
    bq, causal, scale, max_len = x["broadcast_q"], x["causal"], x["scale"], x["max_len"]
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    out, lse = jfa.forward(q, k, v, off, max_len, causal=causal, broadcast_q=bq, scale=scale,
                           window=x.get("window", (-1, -1)))
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    flush = None
    if x["k"].numel() * 2 <= L2_BYTES:
        flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    win = x.get("window", (-1, -1))

    def fwd():
        jfa.forward(q, k, v, off, max_len, causal=causal, broadcast_q=bq, scale=scale, out=out,
                    lse=lse, window=win)

    def bwd():
        jfa.backward(q, k, v, off, max_len, out, lse, do, causal=causal, broadcast_q=bq,
                     scale=scale, dq=dq, dk=dk, dv=dv, window=win)

    for _ in range(warmup):
        fwd()
        bwd()
    jfa.jfa_sync_and_check()
    # enough steps for a timed region of about min_seconds (clock samples)
    torch.cuda.synchronize()
    t_probe = time.time()
    fwd()
    bwd()
    torch.cuda.synchronize()
    per_step = max(time.time() - t_probe, 1e-6)
    steps = int(min(max(steps, round(min_seconds / per_step)), 500))

    def run(n):
        for _ in range(n):
            if flush is not None:
                flush.zero_()
            fwd()
            bwd()

    kprof = _breakdown(jfa, torch, x, run, max(3, steps // 4))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    n0 = jfa.launch_count()
    t0 = time.time()
    jfa.profile_enable(True)
    for i in range(steps):
        if flush is not None:
            flush.zero_()  # torch's kernel, outside this step's events
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    jfa.profile_enable(False)
    t1 = time.time()
    launches = jfa.launch_count() - n0
    jfa.profile_read()  # the dominant kernel's launches (the breakdown window has them all)
    jfa.profile_select(None)
    jfa.jfa_sync_and_check()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    return fwd_ms, bwd_ms, kprof, launches, (t0, t1), steps


def _sparse_pairs(lengths, H, bl, ct, causal, window):
    """Computed (query, key) pairs of the block-sparse forward, summed over
    the heads: per (sequence, head, Q block) and listed K block, the keys of
    the block inside each row's band (all of them without a local mask)."""
    big = 1 << 40
    wl = big if window is None or window[0] is None or window[0] < 0 else window[0]
    wr = big if window is None or window[1] is None or window[1] < 0 else window[1]
    if causal:
        wr = min(wr, 0)
    pairs = 0
    for b, n in enumerate(np.asarray(lengths).tolist()):
        for i in range(-(-n // 256)):
            rows = np.arange(256 * i, min(n, 256 * i + 256))[:, None]
            for h in range(H):
                sel = bl[b, h, i, :ct[b, h, i]].astype(np.int64)[None, :]
                lo = np.maximum(sel * 128, rows - wl)
                hi = np.minimum(np.minimum(sel * 128 + 127, n - 1), rows + wr)
                pairs += int(np.clip(hi - lo + 1, 0, None).sum())
    return pairs


def _time_sparse(jfa, torch, x, permille, steps, warmup, stream, dev, min_seconds=0.15):
    """Block-sparse forward (selection + attention over the selected blocks)
    of workload x (with its causal mask and window, if any), device-timed;
    returns (ms per step, kernel profile of the breakdown window, computed
    (query, key) pairs summed over the heads, host window, steps)."""
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    ml, scale = x["max_len"], x["scale"]
    causal, window = bool(x["causal"]), x.get("window")
    blocks, counts = jfa.block_select(q, k, off, ml, permille, causal=causal, window=window)
    out, lse = jfa.forward_sparse(q, k, v, off, ml, blocks, counts, scale=scale, causal=causal,
                                  window=window)

    def step():
        jfa.block_select(q, k, off, ml, permille, blocks=blocks, counts=counts, causal=causal,
                         window=window)
        jfa.forward_sparse(q, k, v, off, ml, blocks, counts, scale=scale, out=out, lse=lse,
                           causal=causal, window=window)

    for _ in range(warmup):
        step()
    jfa.jfa_sync_and_check()
    torch.cuda.synchronize()
    t_probe = time.time()
    step()
    torch.cuda.synchronize()
    steps = int(min(max(steps, round(min_seconds / max(time.time() - t_probe, 1e-6))), 500))

    def run(n):
        for _ in range(n):
            step()

    kprof = _breakdown(jfa, torch, x, run, max(3, steps // 4))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    jfa.profile_enable(True)
    h0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    jfa.profile_enable(False)
    win = (h0, time.time())
    jfa.profile_read()
    jfa.profile_select(None)
    jfa.jfa_sync_and_check()
    pairs = _sparse_pairs(x["lengths"], x["H"], blocks.cpu().numpy(), counts.cpu().numpy(),
                          causal, window)
    return e0.elapsed_time(e1) / steps, kprof, pairs, win, steps


# The dK/dV pass on pairs of CTAs (cta_group::2 products over two key
# blocks; the library runs it under JFA_KV_PAIR=1): name -> workload.
PAIR_VARIANTS = {"jagged_self_kv_pair": "jagged_self", "broadcast_q_kv_pair": "broadcast_q"}


class _kv_pair:
    """JFA_KV_PAIR=1 inside the block (the library reads it on every call)."""

    def __enter__(self):
        self.old = os.environ.get("JFA_KV_PAIR")
        os.environ["JFA_KV_PAIR"] = "1"

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop("JFA_KV_PAIR", None)
        else:
            os.environ["JFA_KV_PAIR"] = self.old


# Block-sparse variants of the bench line: name -> the workload they run on.
SPARSE_VARIANTS = {"jagged_self_block_sparse500": "jagged_self",
                   "causal_self_block_sparse500": "causal_self"}


def _sparse_entry(xs, base, sname, sp_ms, sp_prof, sp_pairs, sp_steps, peak, hbm, dense_fwd_ms):
    """Bench entry of a block-sparse variant: selection + attention per step;
    the attention kernel's work is the computed pairs."""
    kern = _kernels_entry(xs, sp_prof, peak, hbm, sname)
    fl = 4.0 * xs["D"] * sp_pairs  # sp_pairs counts every head
    if "fwd" in kern:
        ms = kern["fwd"]["ms_per_launch"]
        kern["fwd"]["tflops"] = fl / (ms * 1e-3) / 1e12
        kern["fwd"]["roofline_frac"] = kern["fwd"]["tflops"] / peak
    dense_pairs = W.pairs(xs["lengths"], xs["causal"], xs["q_len"], xs["broadcast_q"],
                          xs.get("window", (-1, -1)))
    return {
        "config": {k: v for k, v in _config(xs, base).items()
                   if k not in ("parallelism",)} | {"permille": 500},
        "steps": sp_steps,
        "fwd": {"ms": sp_ms, "tflops": fl / (sp_ms * 1e-3) / 1e12,
                "selected_fraction": sp_pairs / (xs["H"] * dense_pairs),
                "dense_fwd_ms": dense_fwd_ms,
                "speedup_vs_dense": (dense_fwd_ms / sp_ms) if dense_fwd_ms else None},
        "kernels": kern,
    }


def _workload_entry(x, wname, fwd_ms, bwd_ms, kprof, peak, hbm, clk, window, steps):
    fwd_f, bwd_f, pairs = _flops(x)
    (ff, fb), (bf, bb) = step_model(x)
    fwd_frac, fwd_bound = _roof(ff, fb, fwd_ms * 1e-3, peak, hbm)
    bwd_frac, bwd_bound = _roof(bf, bb, bwd_ms * 1e-3, peak, hbm)
    kernels = _kernels_entry(x, kprof, peak, hbm, wname)
    work = [k for k in kernels if k not in ("sched", "finalize")]
    dom = max(work, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches"])
    return {
        "config": {k: v for k, v in _config(x, wname).items() if k not in ("parallelism",)},
        "steps": steps,
        "value": (fwd_f + bwd_f) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12, "unit": "TFLOPS",
        "fwd": {"ms": fwd_ms, "tflops": fwd_f / (fwd_ms * 1e-3) / 1e12,
                "frac_of_peak": fwd_f / (fwd_ms * 1e-3) / 1e12 / peak,
                "roofline_frac": fwd_frac, "bound": fwd_bound, "algorithmic_bytes": fb},
        "bwd": {"ms": bwd_ms, "tflops": bwd_f / (bwd_ms * 1e-3) / 1e12,
                "frac_of_peak": bwd_f / (bwd_ms * 1e-3) / 1e12 / peak,
                "roofline_frac": bwd_frac, "bound": bwd_bound, "algorithmic_bytes": bb},
        "kernels": kernels,
        "dominant": {"kernel": dom, "desc": KERNEL_DESC.get(dom, dom),
                     "bound": kernels[dom]["bound"], "frac": kernels[dom]["roofline_frac"]},
        "clocks": clk.summary([window]),
    }


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
    B, H, D = x["B"], x["H"], x["D"]
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
    clk = ClockSampler(local)
    clk.__enter__()
    windows = []
    # Per-kernel breakdown (`kernels`): a shorter window in which every
    # launch is bracketed by a CUDA event pair on its stream.  The timed
    # region after it brackets only the dominant kernel, whose mean launch
    # time the roofline reports: events around every launch would add about
    # 2% to the step.
    n_brk = max(3, args.steps // 4)
    jfa.profile_select(None)
    b_start, b_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    jfa.profile_enable(True)
    hb0 = time.time()
    b_start.record(stream)
    for _ in range(n_brk):
        fwd()
        bwd()
    b_end.record(stream)
    torch.cuda.synchronize()
    brk_window = (hb0, time.time())
    jfa.profile_enable(False)
    kprof_all = jfa.profile_read()
    model = kernel_model(x)
    dom = max((k for k, (t, n) in kprof_all.items() if n > 0 and model.get(k, (0, 0))[0] > 0),
              key=lambda k: kprof_all[k][0])
    brk_ms = b_start.elapsed_time(b_end) / n_brk
    jfa.profile_select([dom])
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = jfa.launch_count()
    jfa.profile_enable(True)
    h0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    windows.append((h0, time.time()))
    windows.append(brk_window)
    jfa.profile_enable(False)
    launches = jfa.launch_count() - launches0
    kprof = jfa.profile_read()  # the dominant kernel's launches only
    jfa.profile_select(None)
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
    del sets, hq, hk, hv, hdo, ho, hl, hdq, hdk, hdv

    # The other workloads (rank 0 of a single-GPU run, unless --only): each
    # device-timed over a few steps through the same public API.
    workloads, variants = {}, {}
    sparse_entries = {}
    if ws == 1 and not args.only:
        workloads[wname] = (x, fwd_ms, bwd_ms, kprof_all, windows[0], args.steps)
        for other in W.ORDER:
            if other == wname:
                continue
            xo = W.make_inputs(W.WORKLOADS[other])
            steps = max(3, min(args.steps, args.workload_steps))
            f_ms, b_ms, kp, _, win, steps = _time_steps(jfa, torch, xo, steps,
                                                        max(3, args.warmup), stream, dev)
            windows.append(win)
            workloads[other] = (xo, f_ms, b_ms, kp, win, steps)
            del xo
            torch.cuda.empty_cache()
        # block-sparse forward at a 0.5 selection ratio, against the dense
        # forward of the same workload (causal_self: with its causal mask)
        for sname, base in SPARSE_VARIANTS.items():
            xs = W.make_inputs(W.WORKLOADS[base])
            sp_ms, sp_prof, sp_pairs, win, sp_steps = _time_sparse(
                jfa, torch, xs, 500, max(3, min(args.steps, args.workload_steps)),
                max(3, args.warmup), stream, dev)
            windows.append(win)
            sparse_entries[sname] = (base, sp_ms, sp_prof, sp_pairs, win, sp_steps, xs)
            del xs
            torch.cuda.empty_cache()
        # GQA and sliding-window variants, the same way
        for vname in W.VARIANTS:
            xo = W.make_inputs(W.variant(vname))
            steps = max(3, min(args.steps, args.workload_steps))
            f_ms, b_ms, kp, _, win, steps = _time_steps(jfa, torch, xo, steps,
                                                        max(3, args.warmup), stream, dev)
            windows.append(win)
            variants[vname] = (xo, f_ms, b_ms, kp, win, steps)
            del xo
            torch.cuda.empty_cache()
        # the dK/dV pass on CTA pairs (cta_group::2), the same way
        for vname, base in PAIR_VARIANTS.items():
            xo = W.make_inputs(W.WORKLOADS[base])
            steps = max(3, min(args.steps, args.workload_steps))
            with _kv_pair():
                f_ms, b_ms, kp, _, win, steps = _time_steps(jfa, torch, xo, steps,
                                                            max(3, args.warmup), stream, dev)
            windows.append(win)
            variants[vname] = (xo, f_ms, b_ms, kp, win, steps)
            del xo
            torch.cuda.empty_cache()
    clk.__exit__(None, None, None)
    for sname, (base, sp_ms, sp_prof, sp_pairs, win, sp_steps, xs) in sparse_entries.items():
        dense_fwd_ms = workloads[base][1]  # (x, fwd ms, ...) of the dense run
        variants[sname] = _sparse_entry(xs, base, sname, sp_ms, sp_prof, sp_pairs, sp_steps,
                                        peak, hbm, dense_fwd_ms) | {"clocks": clk.summary([win])}
    sparse_entries.clear()
    for group in (workloads, variants):
        for other, entry in list(group.items()):
            if isinstance(entry, tuple):
                xo, f_ms, b_ms, kp, win, steps = entry
                group[other] = _workload_entry(xo, other, f_ms, b_ms, kp, peak, hbm, clk, win,
                                               steps)

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
    kernels = _kernels_entry(x, kprof_all, peak, hbm, wname)
    dom_flops = model[dom][0]
    dom_ms = kprof[dom][0] / kprof[dom][1]  # over the timed region
    dom_tf = dom_flops / (dom_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(x, wname, ws),
        "frac_of_peak": value / peak,
        # the same against the measured sustained (seconds-long, power-capped)
        # bf16 rate, for reference; the timed region here is milliseconds long
        "frac_of_sustained_peak": (value / peak_sus) if peak_sus else None,
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak},
        "roofline": {"bound": "tensor", "kernel": KERNEL_DESC[dom],
                     "algorithmic_tflop_per_launch": dom_flops / 1e12,
                     "ms_per_launch": dom_ms, "launches": kprof[dom][1],
                     "achieved": dom_tf, "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "peak_sustained": peak_sus,
                     "frac_of_sustained": (dom_tf / peak_sus) if peak_sus else None,
                     "traffic": traffic_record(dom, wname),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)"},
        "kernels": kernels,
        "kernels_window": {"steps": n_brk, "ms_per_step": brk_ms,
                           "events": "every launch bracketed (the timed region: the "
                                     "dominant kernel's launches only)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "schedule": "every step copies all inputs in and all results out; input "
                            "copies, compute and result copies pipelined on three streams "
                            "with two device buffer sets"},
        "gpu_launches": launches,
        "clocks": clk.summary(windows),
        "clocks_headline": clk.summary(windows[:1]),
    }
    if workloads:
        line["workloads"] = workloads
    if variants:
        line["variants"] = variants
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_variant(args):
    """One variant alone, device-timed like the bench line's `variants`
    entries (the block-sparse forward: selection + attention per step)."""
    import torch
    import jagged_flash_attention_gb300 as jfa
    dev = torch.device("cuda")
    jfa.lib()
    peak, _, hbm, _ = _peaks()
    stream = torch.cuda.current_stream()
    steps, warmup = max(3, args.steps), max(3, args.warmup)
    if args.variant in SPARSE_VARIANTS:
        base = SPARSE_VARIANTS[args.variant]
        w = W.WORKLOADS[base]
        lengths = None if args.batch is None else W.sample_lengths(w, B=args.batch)
        x = W.make_inputs(w, lengths=lengths)
        ms, kprof, pairs, _, steps = _time_sparse(jfa, torch, x, 500, steps, warmup, stream, dev)
        entry = _sparse_entry(x, base, args.variant, ms, kprof, pairs, steps, peak, hbm, None)
    else:
        pair = args.variant in PAIR_VARIANTS
        w = W.WORKLOADS[PAIR_VARIANTS[args.variant]] if pair else W.variant(args.variant)
        lengths = None if args.batch is None else W.sample_lengths(w, B=args.batch)
        x = W.make_inputs(w, lengths=lengths)
        with (_kv_pair() if pair else contextlib.nullcontext()):
            f_ms, b_ms, kprof, _, _, steps = _time_steps(jfa, torch, x, steps, warmup, stream,
                                                         dev)
        fwd_f, bwd_f, _ = _flops(x)
        entry = {"fwd": {"ms": f_ms, "tflops": fwd_f / (f_ms * 1e-3) / 1e12},
                 "bwd": {"ms": b_ms, "tflops": bwd_f / (b_ms * 1e-3) / 1e12},
                 "kernels": _kernels_entry(x, kprof, peak, hbm, args.variant)}
    print(json.dumps({"variant": args.variant, "steps": steps, "B": int(x["B"]), **entry}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.ORDER)
    ap.add_argument("--only", action="store_true",
                    help="time the named workload alone (no `workloads` object)")
    ap.add_argument("--workload-steps", type=int, default=10,
                    help="timed steps of each other workload (at least 3)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default=None,
                    choices=list(W.VARIANTS) + list(SPARSE_VARIANTS) + list(PAIR_VARIANTS),
                    help="time one GQA / window / block-sparse variant alone (one JSON line "
                         "with that variant's entry; for profiling captures)")
    ap.add_argument("--batch", type=int, default=None,
                    help="draw this many sequences instead of the workload's B "
                         "(same length distribution; for profiling captures)")
    args = ap.parse_args()
    if args.variant is not None:
        run_variant(args)
        return
    w = W.WORKLOADS[args.workload]
    lengths = None if args.batch is None else W.sample_lengths(w, B=args.batch)
    x = W.make_inputs(w, lengths=lengths)
    if args.impl == "reference":
        run_reference(args, x, args.workload)
    else:
        run_ours(args, x, args.workload)


if __name__ == "__main__":
    main()
