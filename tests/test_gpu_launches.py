"""The library's launch accounting on the GPU: one self-attention forward
plus backward enqueues exactly the kernels the design names (a scheduler and
the forward; the pre-pass that builds both backward work lists and the row
statistics, the dK/dV pass and the dQ pass), and the event timer sees each
of them on the launching stream."""
import pytest
import torch

from tests.gpu_common import inputs

pytestmark = pytest.mark.gpu


def test_self_attention_launches_and_kernel_times():
    import jagged_flash_attention_gb300 as jfa
    x = inputs("tiny_self")
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    out, lse = jfa.forward(q, k, v, off, x["max_len"])
    torch.cuda.synchronize()
    jfa.profile_read()
    n0 = jfa.launch_count()
    jfa.profile_enable(True)
    try:
        out, lse = jfa.forward(q, k, v, off, x["max_len"])
        jfa.backward(q, k, v, off, x["max_len"], out, lse, do)
        torch.cuda.synchronize()
    finally:
        jfa.profile_enable(False)
    assert jfa.launch_count() - n0 == 5
    prof = jfa.profile_read()
    counts = {k: n for k, (t, n) in prof.items() if n}
    assert counts == {"sched": 1, "fwd": 1, "prep": 1, "bwd_kv": 1, "bwd_q": 1}
    for kind in counts:
        assert prof[kind][0] > 0.0, kind
    # With a kind selection only the selected launches get events; every
    # launch is still counted.
    n0 = jfa.launch_count()
    jfa.profile_select(["bwd_kv"])
    jfa.profile_enable(True)
    try:
        out, lse = jfa.forward(q, k, v, off, x["max_len"])
        jfa.backward(q, k, v, off, x["max_len"], out, lse, do)
        torch.cuda.synchronize()
    finally:
        jfa.profile_enable(False)
        jfa.profile_select(None)
    assert jfa.launch_count() - n0 == 5
    prof = jfa.profile_read()
    assert {kind: n for kind, (t, n) in prof.items() if n} == {"bwd_kv": 1}
    assert prof["bwd_kv"][0] > 0.0
    jfa.jfa_sync_and_check()


def test_broadcast_launches():
    """Broadcast-Q forward + backward: the scheduler and the forward, then the
    pre-pass (both backward work lists and the padded row statistics), the
    dK/dV pass, the chunked dQ pass and the finalize that sums its partials."""
    import jagged_flash_attention_gb300 as jfa
    x = inputs("broadcast_q", [0, 130, 5, 600], H=2, q_len=200)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    out, lse = jfa.forward(q, k, v, off, x["max_len"], broadcast_q=True)
    torch.cuda.synchronize()
    jfa.profile_read()
    n0 = jfa.launch_count()
    jfa.profile_enable(True)
    try:
        out, lse = jfa.forward(q, k, v, off, x["max_len"], broadcast_q=True)
        jfa.backward(q, k, v, off, x["max_len"], out, lse, do, broadcast_q=True)
        torch.cuda.synchronize()
    finally:
        jfa.profile_enable(False)
    assert jfa.launch_count() - n0 == 6
    counts = {k: n for k, (t, n) in jfa.profile_read().items() if n}
    assert counts == {"sched": 1, "fwd": 1, "prep": 1, "bwd_kv": 1, "bwd_qb": 1, "finalize": 1}
    jfa.jfa_sync_and_check()


def test_broadcast_short_q_one_pass_launches():
    """Broadcast-Q with D = 64 and q_len <= 128: the backward is the pre-pass
    (dQ-pass list and statistics only), one pass for dK, dV and the dQ
    partials, and the finalize."""
    import jagged_flash_attention_gb300 as jfa
    x = inputs("skewed_broadcast_q", [0, 130, 5, 600], H=2)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    out, lse = jfa.forward(q, k, v, off, x["max_len"], broadcast_q=True)
    torch.cuda.synchronize()
    jfa.profile_read()
    jfa.profile_enable(True)
    try:
        jfa.backward(q, k, v, off, x["max_len"], out, lse, do, broadcast_q=True)
        torch.cuda.synchronize()
    finally:
        jfa.profile_enable(False)
    counts = {k: n for k, (t, n) in jfa.profile_read().items() if n}
    assert counts == {"prep": 1, "bwd_bs": 1, "finalize": 1}
    jfa.jfa_sync_and_check()
