"""GPU parity of the GQA and sliding-window variants (jfa_fwd_ex /
jfa_bwd_ex) against the fp64 oracle on identical seeded bf16 inputs.

GQA: query head h reads K/V head h / (H / H_kv); dK / dV sum over the
group.  Windows keep keys [i - left, i + right] of query i; the cases put
band edges inside tiles, across tile boundaries and on ragged tails, with
bands narrower than a tile and wider than a sequence.  Broadcast-Q cases
run GQA through the streamed forward (q_len <= 128), the two-pass backward
(which GQA takes for every q_len) and the general forward."""
import numpy as np
import pytest

from tests.gpu_common import compare, inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

EDGE = [1, 127, 128, 129, 255, 256, 257, 2, 64]

CASES = {
    # GQA, self-attention
    "gqa_self_d128": dict(name="jagged_self", lengths=EDGE, H=4, Hkv=2),
    "gqa_self_d64_one_kv_head": dict(name="tiny_self", lengths=EDGE, H=3, Hkv=1),
    "gqa_causal_d128": dict(name="causal_self", lengths=[1, 128, 129, 300, 513, 17], H=4, Hkv=2),
    # sliding windows
    "window_causal_d128": dict(name="causal_self", lengths=[1, 129, 300, 700, 1000], H=2,
                               window=(200, -1)),
    "window_causal_narrow_d64": dict(name="causal_self", lengths=[300, 5, 257, 128], H=2, D=64,
                                     window=(50, -1)),
    "window_two_sided_d128": dict(name="jagged_self", lengths=[1, 200, 700, 129], H=2,
                                  window=(150, 90)),
    "window_right_only_d128": dict(name="jagged_self", lengths=[300, 40, 129], H=2,
                                   window=(-1, 70)),
    "window_wider_than_sequences": dict(name="jagged_self", lengths=[100, 37, 250], H=2,
                                        window=(400, 400)),
    "window_tile_aligned_d128": dict(name="causal_self", lengths=[512, 384], H=2,
                                     window=(128, -1)),
    "window_gqa_d64": dict(name="tiny_self", lengths=[400, 3, 129, 260], H=4, Hkv=2,
                           window=(100, 30)),
    "window_gqa_causal_d128": dict(name="causal_self", lengths=[1000, 64, 333], H=6, Hkv=2,
                                   window=(300, -1)),
    # broadcast-Q with GQA
    "bcast_gqa_d128_general": dict(name="broadcast_q", lengths=[0, 1, 130, 300, 5], H=4, Hkv=2,
                                   q_len=200),
    "bcast_gqa_d64_stream": dict(name="skewed_broadcast_q", lengths=[0, 7, 129, 1, 500, 3000],
                                 H=4, Hkv=2),
    "bcast_gqa_d128_stream": dict(name="broadcast_q", lengths=[900, 0, 77], H=4, Hkv=1,
                                  q_len=100),
}


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_variant_parity(case):
    spec = dict(CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths", None), **spec)
    g = run_gpu(x)
    r = run_oracle(x)
    rep = compare(g, r)
    print(case, rep)


def test_zero_window_closed_form():
    """Window (0, 0): each query sees only its own key, so O = V, dV = dO
    (summed over the group's query heads), dQ = dK = 0."""
    x = inputs("jagged_self", [1, 130, 257], H=4, Hkv=2, window=(0, 0))
    g = run_gpu(x)
    v = x["v"].float().numpy()
    do = x["dout"].float().numpy().astype(np.float64)
    hk = np.arange(4) // 2
    assert np.array_equal(g["out"], v[:, hk, :])
    T = x["T"]
    np.testing.assert_allclose(g["dv"], do.reshape(T, 2, 2, -1).sum(2), atol=2e-2, rtol=1e-2)
    assert np.abs(g["dq"]).max() < 1e-3 and np.abs(g["dk"]).max() < 1e-3


def test_window_gqa_medium_sampled():
    """A larger windowed GQA case (H = 16 over 4 K/V heads, sequences up to
    6000, a 1024-key causal band), sampled (sequence, head) pairs."""
    x = inputs("causal_self", [6000, 1, 2500, 4097, 700], H=16, Hkv=4, window=(1024, -1))
    g = run_gpu(x)
    r = run_oracle(x, seqs=[0, 1, 3], heads=[0, 5, 15])
    rep = compare(g, r)
    print(rep)
