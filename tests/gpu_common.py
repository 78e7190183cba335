"""Shared helpers of the GPU parity tests: run the CUDA library through the
C ABI, run the fp64 oracle on the same seeded bf16 inputs, compare."""
import dataclasses

import numpy as np
import torch

import jfa_workloads as W
from oracle import jfa_oracle as orc

# Acceptance bars: O max-abs 2e-2 and rel-L2 1e-2; dQ/dK/dV rel-L2 1e-2;
# LSE abs 1e-3.
O_MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_ABS = 1e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def workload(name, **over):
    return dataclasses.replace(W.WORKLOADS[name], **over)


def inputs(name, lengths=None, **over):
    return W.make_inputs(workload(name, **over), lengths=lengths)


def run_gpu(x, stream=None, bwd=True):
    import jagged_flash_attention_gb300 as jfa
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    res = {}
    win = x.get("window", (-1, -1))
    out, lse = jfa.forward(q, k, v, off, x["max_len"], causal=x["causal"],
                           broadcast_q=x["broadcast_q"], scale=x["scale"], stream=stream,
                           window=win)
    if bwd:
        dq, dk, dv = jfa.backward(q, k, v, off, x["max_len"], out, lse, do, causal=x["causal"],
                                  broadcast_q=x["broadcast_q"], scale=x["scale"], stream=stream,
                                  window=win)
    jfa.jfa_sync_and_check(stream)
    res["out"], res["lse"] = f64(out), f64(lse)
    if bwd:
        res["dq"], res["dk"], res["dv"] = f64(dq), f64(dk), f64(dv)
    return res


def run_oracle(x, seqs=None, heads=None, bwd=True):
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    win = x.get("window", (-1, -1))
    out, lse = orc.forward(q, k, v, x["offsets"], x["scale"], x["causal"], x["broadcast_q"],
                           seqs=seqs, heads=heads, window=win)
    res = {"out": out, "lse": lse}
    if bwd:
        res["dq"], res["dk"], res["dv"] = orc.backward(q, k, v, x["offsets"], do, x["scale"],
                                                       x["causal"], x["broadcast_q"],
                                                       seqs=seqs, heads=heads, window=win)
    return res


def compare(g, r, what=("out", "lse", "dq", "dk", "dv")):
    """Element-wise comparison on the entries the oracle computed (non-NaN)."""
    report = {}
    for n in what:
        ref = r[n]
        sel = ~np.isnan(ref)
        a, b = g[n][sel], ref[sel]
        if n == "lse":
            inf = np.isinf(b)
            assert np.array_equal(np.isinf(a) & (a < 0), inf), "LSE -inf pattern"
            err = float(np.abs(a[~inf] - b[~inf]).max()) if (~inf).any() else 0.0
            report[n] = err
            assert err <= LSE_ABS, f"LSE abs err {err}"
            continue
        assert np.isfinite(a).all(), f"{n}: non-finite values"
        rl = rel_l2(a, b) if np.linalg.norm(b) > 0 else float(np.abs(a).max())
        report[n] = rl
        assert rl <= REL_L2, f"{n}: rel-L2 {rl}"
        if n == "out":
            ma = float(np.abs(a - b).max())
            report["out_max_abs"] = ma
            assert ma <= O_MAX_ABS, f"O max-abs {ma}"
    return report
