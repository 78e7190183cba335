"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle on
identical seeded bf16 inputs.  Small cases compare every output element;
the full-size workloads compare sampled (sequence, head) pairs (and the
whole batch-summed dQ in broadcast mode)."""
import numpy as np
import pytest
import torch

import jfa_workloads as W
from tests.gpu_common import compare, inputs, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

EDGE = [1, 127, 128, 129, 255, 256, 257, 2, 64]

SMALL = {
    "tiny_self": dict(name="tiny_self"),
    "self_d128_edges": dict(name="jagged_self", lengths=EDGE, H=2),
    "self_d64_edges": dict(name="tiny_self", lengths=EDGE, H=3),
    "causal_d128_edges": dict(name="causal_self", lengths=[1, 128, 129, 300, 513, 17], H=2),
    "causal_d64_edges": dict(name="causal_self", lengths=[5, 128, 257, 64, 190], H=2, D=64),
    "self_total_below_tile": dict(name="jagged_self", lengths=[3, 5, 20], H=2),
    "causal_total_below_tile": dict(name="causal_self", lengths=[7, 30], H=3),
    "self_one_long": dict(name="jagged_self", lengths=[1000], H=1),
    "bcast_d128_ragged_q": dict(name="broadcast_q", lengths=[0, 1, 130, 0, 300, 5, 128], H=3,
                                q_len=200),
    "bcast_d64": dict(name="skewed_broadcast_q", lengths=[0, 7, 129, 1, 500], H=2),
    "bcast_three_q_tiles": dict(name="broadcast_q", lengths=[40, 256, 1], H=2, q_len=300),
    "bcast_all_empty_but_one": dict(name="broadcast_q", lengths=[0, 0, 3, 0], H=1, q_len=17),
    # D = 64: q_len <= 128 takes the one-pass backward, longer q_len two passes
    "bcast_d64_q128_one_pass": dict(name="skewed_broadcast_q", lengths=[130, 0, 1, 257, 128],
                                    H=3, q_len=128),
    "bcast_d64_q1_one_pass": dict(name="skewed_broadcast_q", lengths=[5, 300, 0, 2], H=2,
                                  q_len=1),
    "bcast_d64_q200_two_pass": dict(name="skewed_broadcast_q", lengths=[3, 0, 300, 129, 1], H=2,
                                    q_len=200),
    # q_len <= 128: the streamed forward; chunk boundaries split sequences
    # into pieces that the combine kernel merges
    "bcast_stream_split_one_long": dict(name="skewed_broadcast_q", lengths=[3000], H=2),
    "bcast_stream_split_d128": dict(name="broadcast_q", lengths=[0, 900, 5, 1300, 0, 77], H=2,
                                    q_len=100),
    # q_len <= 64: the queries spread over the four TMEM lane quadrants
    "bcast_stream_spread_d128_q40": dict(name="broadcast_q", lengths=[0, 900, 5, 1300, 129], H=2,
                                         q_len=40),
    "bcast_stream_spread_d64_q17": dict(name="skewed_broadcast_q", lengths=[3000, 1, 0, 129, 64],
                                        H=2, q_len=17),
    "bcast_stream_spread_d64_q49": dict(name="skewed_broadcast_q", lengths=[700, 2, 300], H=3,
                                        q_len=49),
    "jagged_self_B6": dict(name="jagged_self", lengths=W.sample_lengths(
        W.WORKLOADS["jagged_self"], B=6)),
    "broadcast_q_B16": dict(name="broadcast_q", lengths=W.sample_lengths(
        W.WORKLOADS["broadcast_q"], B=16)),
    "causal_self_B2_H2": dict(name="causal_self", lengths=[3000, 777], H=2),
    "skewed_bq_B64": dict(name="skewed_broadcast_q", lengths=np.concatenate(
        [W.sample_lengths(W.WORKLOADS["skewed_broadcast_q"], B=62), [8192, 4097]])),
}


@pytest.mark.parametrize("case", list(SMALL), ids=list(SMALL))
def test_small_parity(case):
    spec = dict(SMALL[case])
    x = inputs(spec.pop("name"), spec.pop("lengths", None), **spec)
    g = run_gpu(x)
    r = run_oracle(x)
    rep = compare(g, r)
    print(case, rep)


FULL = ["jagged_self", "broadcast_q", "causal_self", "skewed_broadcast_q"]


def _sample(lengths, rng, k=4):
    order = np.argsort(lengths)
    pick = {int(order[0]), int(order[-1])}
    while len(pick) < min(k, len(lengths)):
        pick.add(int(rng.integers(0, len(lengths))))
    return sorted(pick)


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full workload sizes, in the launch configuration the benchmark times;
    the oracle computes sampled (sequence, head) pairs."""
    x = W.make_inputs(W.WORKLOADS[name])
    g = run_gpu(x)
    rng = np.random.default_rng(99)
    seqs = _sample(x["lengths"], rng)
    heads = sorted({0, x["H"] - 1})
    r = run_oracle(x, seqs=seqs, heads=heads)
    what = ["out", "lse", "dk", "dv"] + ([] if x["broadcast_q"] else ["dq"])
    rep = compare(g, r, what)
    if x["broadcast_q"]:
        # dQ sums over every sequence: check it against the full oracle sum.
        full = run_oracle(x, heads=heads)
        rep.update(compare(g, {"dq": full["dq"]}, ["dq"]))
    print(name, seqs, rep)


def test_length_one_closed_form():
    """Length-1 sequences: O is the V row, dV = dO, dQ = dK = 0."""
    x = inputs("jagged_self", [1] * 37, H=3)
    g = run_gpu(x)
    v, do = x["v"].float().numpy(), x["dout"].float().numpy()
    assert np.array_equal(g["out"], v)
    assert np.array_equal(g["dv"], do)
    assert np.abs(g["dq"]).max() < 1e-3 and np.abs(g["dk"]).max() < 1e-3
    lse_ref = x["scale"] * np.einsum("thd,thd->ht", x["q"].double().numpy(), x["k"].double().numpy())
    assert np.abs(g["lse"] - lse_ref).max() < 1e-3


def test_constant_v_and_onehot_rows_sum_to_one():
    x = inputs("tiny_self", [5, 64, 33, 1, 60], H=2)
    T = x["T"]
    c = torch.linspace(-2, 2, 64).to(torch.bfloat16)
    x["v"] = c.view(1, 1, 64).expand(T, 2, 64).contiguous()
    g = run_gpu(x)
    assert np.abs(g["out"] - c.float().numpy()[None, None, :]).max() < 2e-2
    # dQ = dK = 0 up to the bf16 rounding of O that enters Delta
    assert np.abs(g["dq"]).max() < 5e-2 and np.abs(g["dk"]).max() < 5e-2
    # one-hot V rows (L <= D): O exposes P, whose rows sum to 1
    v = torch.zeros(T, 2, 64)
    off = x["offsets"]
    for b in range(len(off) - 1):
        for j in range(off[b], off[b + 1]):
            v[j, :, j - off[b]] = 1.0
    x["v"] = v.to(torch.bfloat16)
    g = run_gpu(x, bwd=False)
    assert np.abs(g["out"].sum(-1) - 1.0).max() < 2e-2
    r = run_oracle(x, bwd=False)
    compare(g, r, ["out", "lse"])


def test_forward_is_deterministic_and_stream_ordered():
    x = inputs("jagged_self", [300, 1, 129, 700], H=2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = run_gpu(x, stream=s, bwd=False)
    b = run_gpu(x, bwd=False)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_outputs_stay_inside_their_rows():
    """Canary rows after the packed outputs are never written."""
    import jagged_flash_attention_gb300 as jfa
    x = inputs("jagged_self", [130, 7, 255], H=2)
    dev = torch.device("cuda")
    T, H, D = x["k"].shape
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    sentinel = torch.tensor(12345.0, dtype=torch.bfloat16)
    big = lambda: torch.full((T + 200, H, D), float(sentinel), dtype=torch.bfloat16, device=dev)
    out, dq, dk, dv = big(), big(), big(), big()
    lse = torch.full((H, T + 64), 777.0, device=dev)
    jfa.jfa_fwd(q, k, v, off, 3, H, D, x["max_len"], 0, 0, x["scale"], out, lse)
    jfa.jfa_bwd(q, k, v, off, 3, H, D, x["max_len"], 0, 0, x["scale"], out, lse, do, dq, dk, dv)
    jfa.jfa_sync_and_check()
    for t in (out, dq, dk, dv):
        assert torch.all(t[T:] == sentinel)
        assert torch.all(torch.isfinite(t[:T].float()))


@pytest.mark.parametrize("bad", ["first_not_zero", "too_long", "decreasing"])
def test_bad_offsets_reported_by_device(bad):
    import jagged_flash_attention_gb300 as jfa
    x = inputs("jagged_self", [100, 50, 80], H=2)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    off = x["offsets"].copy()
    max_len = x["max_len"]
    if bad == "first_not_zero":
        off[0] = 1
    elif bad == "too_long":
        max_len = 60
    else:
        off[2] = off[1] - 1
    offd = torch.from_numpy(off).to(dev)
    out = torch.full_like(q, 3.0)
    lse = torch.full((2, x["T"]), 5.0, device=dev)
    jfa.jfa_fwd(q, k, v, offd, 3, 2, 128, max_len, 0, 0, x["scale"], out, lse)
    with pytest.raises(jfa.JfaError) as ei:
        jfa.jfa_sync_and_check()
    assert ei.value.status == 1
    assert torch.all(out == 3.0) and torch.all(lse == 5.0)
    # the library stays usable and the error word was cleared
    g = run_gpu(x, bwd=False)
    assert np.isfinite(g["out"]).all()


def test_zero_max_len_broadcast():
    import jagged_flash_attention_gb300 as jfa
    dev = torch.device("cuda")
    B, H, D, Lq = 3, 2, 64, 5
    q = torch.randn(Lq, H, D, device=dev).to(torch.bfloat16)
    k = torch.zeros(0, H, D, device=dev, dtype=torch.bfloat16)
    off = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    kk = torch.zeros(8, H, D, device=dev, dtype=torch.bfloat16)  # non-null pointer for K/V
    out = torch.full((B, Lq, H, D), 9.0, device=dev, dtype=torch.bfloat16)
    lse = torch.zeros(B, H, Lq, device=dev)
    jfa.jfa_fwd_bq(q, kk, kk, off, B, H, D, 0, Lq, 1, 0, 0.125, out, lse)
    jfa.jfa_sync_and_check()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    del k


@pytest.mark.parametrize("name", ["jagged_self", "tiny_self"])
def test_buffers_aligned_to_16_bytes_only(name):
    """Every tensor starts 16 bytes into a larger allocation (16-byte but not
    32-byte aligned), so the kernels' 32-byte load and store paths must take
    their 16-byte fallbacks; results match the oracle as for aligned buffers."""
    import jagged_flash_attention_gb300 as jfa
    x = inputs(name, EDGE, H=2)
    dev = torch.device("cuda")

    def shifted(shape, dtype=torch.bfloat16, src=None):
        n = int(np.prod(shape))
        buf = torch.zeros(n + 8, dtype=dtype, device=dev)
        view = buf[8:].view(*shape)
        assert view.data_ptr() % 32 == 16
        if src is not None:
            view.copy_(src.to(dev))
        return view

    q, k, v, do = (shifted(tuple(x[n].shape), src=x[n]) for n in ("q", "k", "v", "dout"))
    off = torch.from_numpy(x["offsets"]).to(dev)
    T, H, D = q.shape
    out = shifted((T, H, D))
    lse = torch.empty(H, T, dtype=torch.float32, device=dev)
    jfa.forward(q, k, v, off, x["max_len"], scale=x["scale"], out=out, lse=lse)
    dq, dk, dv = (shifted((T, H, D)) for _ in range(3))
    jfa.backward(q, k, v, off, x["max_len"], out, lse, do, scale=x["scale"], dq=dq, dk=dk,
                 dv=dv)
    jfa.jfa_sync_and_check()
    g = {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    g = {n: t.detach().float().cpu().numpy().astype(np.float64) for n, t in g.items()}
    compare(g, run_oracle(x))
