"""The allocation-free forward entry point (jfa_fwd_bq_noalloc).

It serves callers that must not allocate device memory while the library
runs, for example code whose device memory is owned and pre-partitioned by a
host framework that forbids allocation during execution.  Its scratch is a
fixed device array inside the library, shared by every call.  These tests
call it through the C ABI twice in a row (the second call reuses what the
first left in that array) and compare each result with the fp64 oracle at
the tolerances of the other parity tests, and with the allocating forward
entry point.  All buffers are allocated by the test before the call.  One
case runs in a fresh process in which this entry point is the first call
into the library (so its one-time device set-up runs there), repeats it, and
checks that the device's free memory does not change across the repeats.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from tests.gpu_common import LSE_ABS, O_MAX_ABS, REL_L2, compare, f64, inputs, rel_l2, run_oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    "self_ragged": dict(name="jagged_self", lengths=[1, 127, 128, 129, 700, 3], H=2),
    "causal": dict(name="causal_self", lengths=[300, 17, 513], H=2),
    "broadcast_with_empty": dict(name="broadcast_q", lengths=[0, 130, 5, 0, 600], H=3, q_len=200),
    "d64_broadcast": dict(name="skewed_broadcast_q", lengths=[9, 0, 1000, 64], H=2),
}


def _close(out, lse, out_ref, lse_ref):
    a, b = f64(out), f64(out_ref)
    assert np.isfinite(a).all()
    assert np.abs(a - b).max() <= O_MAX_ABS
    assert rel_l2(a, b) <= REL_L2
    la, lb = f64(lse), f64(lse_ref)
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    fin = np.isfinite(lb)
    assert np.abs(la[fin] - lb[fin]).max(initial=0.0) <= LSE_ABS


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_noalloc_forward_matches_oracle_twice(case):
    import jagged_flash_attention_gb300 as jfa
    spec = dict(CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    ref = run_oracle(x, bwd=False)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    B, H, D, Lq = x["B"], x["H"], x["D"], x["q_len"]
    bq, causal, scale, max_len = x["broadcast_q"], x["causal"], x["scale"], x["max_len"]
    out_ref, lse_ref = jfa.forward(q, k, v, off, max_len, causal=causal, broadcast_q=bq,
                                   scale=scale)
    jfa.jfa_sync_and_check()
    for _ in range(2):
        out = torch.full_like(out_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        jfa.jfa_fwd_bq_noalloc(q, k, v, off, B, H, D, max_len, Lq, bq, causal, scale, out, lse)
        jfa.jfa_sync_and_check()
        compare({"out": f64(out), "lse": f64(lse)}, ref, ["out", "lse"])
        _close(out, lse, out_ref, lse_ref)


_FRESH = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import jagged_flash_attention_gb300 as jfa
from tests.gpu_common import compare, f64, inputs, run_oracle
x = inputs("broadcast_q", [0, 130, 5, 0, 600, 257], H=3, q_len=200)
ref = run_oracle(x, bwd=False)
dev = torch.device("cuda")
q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
off = torch.from_numpy(x["offsets"]).to(dev)
B, H, D, Lq = x["B"], x["H"], x["D"], x["q_len"]
outs = [torch.full((B, Lq, H, D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(4)]
lses = [torch.full((B, H, Lq), float("nan"), device=dev) for _ in range(4)]
torch.cuda.synchronize()
assert jfa.launch_count() == 0  # nothing of the library has run in this process
free = []
for i in range(4):
    jfa.jfa_fwd_bq_noalloc(q, k, v, off, B, H, D, x["max_len"], Lq, 1, 0, x["scale"],
                           outs[i], lses[i])
    jfa.jfa_sync_and_check()
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
for i in range(4):
    compare({"out": f64(outs[i]), "lse": f64(lses[i])}, ref, ["out", "lse"])
o2, l2 = jfa.forward(q, k, v, off, x["max_len"], broadcast_q=True, scale=x["scale"])
jfa.jfa_sync_and_check()
same = bool(torch.equal(o2, outs[3]) and torch.equal(l2, lses[3]))
print(json.dumps({"free": free, "same_as_allocating": same}))
"""


def test_noalloc_first_call_in_fresh_process_allocates_nothing():
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    free = res["free"]
    # the first call may load the library's device code; later calls allocate nothing
    assert free[1] == free[2] == free[3], free
    assert res["same_as_allocating"]


def test_noalloc_rejects_problems_beyond_its_scratch():
    import jagged_flash_attention_gb300 as jfa
    with pytest.raises(jfa.JfaError) as ei:
        # 16 heads * 4096 sequences * 64 tiles = 4M work items > 1 MiB of scratch
        jfa.jfa_fwd_bq_noalloc(16, 16, 16, 16, 4096, 16, 128, 8192, 0, 0, 0, 0.1, 16, 16,
                               stream=0)
    assert ei.value.status == 5 and "static scratch" in str(ei.value)
