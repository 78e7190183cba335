"""The C ABI under CUDA graph capture: every entry point enqueues its kernels
and its stream-ordered scratch on the caller's stream and never synchronises,
so a forward + backward step can be captured once and replayed (the way a
launch-bound loop of small calls runs).  A replay on new inputs copied into
the captured buffers gives the same bytes as eager calls on those inputs:
every kernel is deterministic (no floating-point atomics; broadcast-Q dQ
partials are summed in a fixed order)."""
import numpy as np
import pytest
import torch

from tests.gpu_common import inputs

pytestmark = pytest.mark.gpu

CASES = {
    "self_d128": dict(name="jagged_self", lengths=[1, 127, 300, 700, 129], H=2),
    "self_causal_gqa": dict(name="causal_self", lengths=[5, 400, 260], H=4, Hkv=2),
    "bcast_q256": dict(name="broadcast_q", lengths=[0, 3, 300, 129], H=2, q_len=256),
    "bcast_short_d64": dict(name="skewed_broadcast_q", lengths=[1, 500, 0, 70], H=2),
    "gqa_window_d128": dict(name="jagged_self", lengths=[3, 400, 129, 700], H=4, Hkv=2,
                            window=(200, 50)),
}


def _bufs(x, dev):
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    return q, k, v, do, off


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_graph_replay_equals_eager(case):
    import jagged_flash_attention_gb300 as jfa
    spec = dict(CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    dev = torch.device("cuda")
    bq, causal, ml = x["broadcast_q"], x["causal"], x["max_len"]
    win = x.get("window", (-1, -1))
    q, k, v, do, off = _bufs(x, dev)
    out = torch.empty((x["B"], x["q_len"], x["H"], x["D"]) if bq else q.shape, dtype=q.dtype,
                      device=dev)
    lse = torch.empty((x["B"], x["H"], x["q_len"]) if bq else (x["H"], k.shape[0]),
                      dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step(stream=None):
        jfa.forward(q, k, v, off, ml, causal=causal, broadcast_q=bq, scale=x["scale"], out=out,
                    lse=lse, stream=stream, window=win)
        jfa.backward(q, k, v, off, ml, out, lse, do, causal=causal, broadcast_q=bq,
                     scale=x["scale"], dq=dq, dk=dk, dv=dv, stream=stream, window=win)

    # eager warm-up (the library's per-device state exists before capture)
    step()
    jfa.jfa_sync_and_check()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    # new values in the captured input buffers, same shapes and offsets
    gen = torch.Generator().manual_seed(1234)
    for t in (q, k, v, do):
        t.copy_(torch.randn(t.shape, generator=gen).to(t.dtype))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    jfa.jfa_sync_and_check()
    got = [t.clone() for t in (out, lse, dq, dk, dv)]
    # eager on the same inputs
    step()
    torch.cuda.synchronize()
    jfa.jfa_sync_and_check()
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), got, (out, lse, dq, dk, dv)):
        assert torch.equal(a, b), name
    assert torch.isfinite(got[0]).all()


SPARSE_CASES = {
    "jagged_d128": dict(name="jagged_self", lengths=[1, 600, 257, 1000, 129], H=2),
    "causal_d128": dict(name="causal_self", lengths=[5, 700, 300], H=2),
    "bcast_q256": dict(name="broadcast_q", lengths=[0, 3, 600, 129], H=2, q_len=256),
}


@pytest.mark.parametrize("case", list(SPARSE_CASES), ids=list(SPARSE_CASES))
def test_sparse_graph_replay_equals_eager(case):
    """Selection (pooling, scoring, list check) and the sparse forward,
    captured once and replayed on new inputs, equal eager calls."""
    import jagged_flash_attention_gb300 as jfa
    spec = dict(SPARSE_CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    dev = torch.device("cuda")
    bq, causal, ml = x["broadcast_q"], x["causal"], x["max_len"]
    q, k, v, do, off = _bufs(x, dev)
    bl, ct = jfa.block_select(q, k, off, ml, 500, broadcast_q=bq, causal=causal)
    out, lse = jfa.forward_sparse(q, k, v, off, ml, bl, ct, scale=x["scale"], broadcast_q=bq,
                                  causal=causal)

    def step(stream=None):
        jfa.block_select(q, k, off, ml, 500, blocks=bl, counts=ct, stream=stream,
                         broadcast_q=bq, causal=causal)
        jfa.forward_sparse(q, k, v, off, ml, bl, ct, scale=x["scale"], out=out, lse=lse,
                           stream=stream, broadcast_q=bq, causal=causal)

    step()
    jfa.jfa_sync_and_check()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    gen = torch.Generator().manual_seed(4321)
    for t in (q, k, v):
        t.copy_(torch.randn(t.shape, generator=gen).to(t.dtype))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    jfa.jfa_sync_and_check()
    got = [t.clone() for t in (bl, ct, out, lse)]
    step()
    torch.cuda.synchronize()
    jfa.jfa_sync_and_check()
    for name, a, b in zip(("blocks", "counts", "out", "lse"), got, (bl, ct, out, lse)):
        assert torch.equal(a, b), name
    assert int(got[1].sum()) > 0
    assert torch.isfinite(got[2]).all()
