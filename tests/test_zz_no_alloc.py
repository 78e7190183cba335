"""The allocation-free forward entry point (jfa_fwd_bq_noalloc).

It serves callers that must not allocate device memory while the library
runs, for example code whose device memory is owned and pre-partitioned by a
host framework that forbids allocation during execution.  Its scratch is a
fixed device array inside the library, shared by every call.  These tests
call it through the C ABI twice in a row (the second call reuses what the
first left in that array) and compare each result with the allocating
forward entry point, at the tolerances of the other parity tests.  All
buffers are allocated by the test before the call.
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import LSE_ABS, O_MAX_ABS, REL_L2, f64, inputs, rel_l2

pytestmark = pytest.mark.gpu

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
def test_noalloc_forward_matches_allocating_forward_twice(case):
    import jagged_flash_attention_gb300 as jfa
    spec = dict(CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
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
        _close(out, lse, out_ref, lse_ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import jagged_flash_attention_gb300 as jfa
    with pytest.raises(jfa.JfaError) as ei:
        # 16 heads * 4096 sequences * 64 tiles = 4M work items > 1 MiB of scratch
        jfa.jfa_fwd_bq_noalloc(16, 16, 16, 16, 4096, 16, 128, 8192, 0, 0, 0, 0.1, 16, 16,
                               stream=0)
    assert ei.value.status == 5 and "static scratch" in str(ei.value)
