"""GPU parity of the dK/dV pass on pairs of CTAs ("Optimizing Jagged Flash
Attention with TLX", "2-CTA collaborative MMA (backward)"): with
JFA_KV_PAIR=1 the library runs the dK/dV pass as clusters of two CTAs whose
cta_group::2 products (M = 256) cover two adjacent key blocks.  The cases
against the fp64 oracle put the second CTA of a pair on a missing block (an
odd number of key blocks), on ragged blocks and on one-key sequences; GQA
sums dK / dV over the group inside the pair; broadcast-Q runs it in the
two-pass backward with q_len not a multiple of the 64-row half tiles.  The
pair and single-CTA passes are also compared with each other: both compute
every dK / dV element from the same bf16 operands in the same K order."""
import numpy as np
import pytest

import jfa_workloads as W
from tests.gpu_common import compare, inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

EDGE = [1, 127, 128, 129, 255, 256, 257, 383, 700, 2]

CASES = {
    "self_d128_edges": dict(name="jagged_self", lengths=EDGE, H=2),
    "self_d128_gqa": dict(name="jagged_self", lengths=[129, 640, 1, 385, 1000], H=4, Hkv=2),
    "self_d128_many_items": dict(name="jagged_self", lengths=None, H=2, B=12),
    "bcast_d128_q256": dict(name="broadcast_q", lengths=[0, 1, 130, 300, 700, 257], H=4,
                            q_len=256),
    "bcast_d128_q200_gqa": dict(name="broadcast_q", lengths=[5, 129, 0, 900], H=4, Hkv=2,
                                q_len=200),
    "bcast_d128_q300": dict(name="broadcast_q", lengths=[383, 1, 64, 1200], H=2, q_len=300),
}


def _run(x, pair, monkeypatch):
    """Forward + backward, and which dK/dV kernel ran."""
    import jagged_flash_attention_gb300 as jfa
    monkeypatch.setenv("JFA_KV_PAIR", "1" if pair else "0")
    jfa.profile_read()
    jfa.profile_enable(True)
    res = run_gpu(x)
    jfa.profile_enable(False)
    counts = {k: n for k, (_, n) in jfa.profile_read().items() if n}
    assert counts.get("bwd_kv_pair", 0) == (1 if pair else 0), counts
    assert counts.get("bwd_kv", 0) == (0 if pair else 1), counts
    return res


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_pair_backward_parity(case, monkeypatch):
    spec = dict(CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    g = _run(x, True, monkeypatch)
    single = _run(x, False, monkeypatch)
    r = run_oracle(x)
    print(case, compare(g, r))
    for n in ("dk", "dv", "dq", "out", "lse"):
        a, b = g[n], single[n]
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin), n
        err = float(np.abs(a[fin] - b[fin]).max()) if fin.any() else 0.0
        scale = float(np.abs(b[fin]).max()) if fin.any() else 1.0
        print(f"  {n}: pair vs single max abs {err:.3g} (of {scale:.3g})")
        assert err <= 1e-2 * max(scale, 1e-6), n


@pytest.mark.parametrize("name", ["jagged_self", "broadcast_q"])
def test_pair_full_size_equals_single(name, monkeypatch):
    """Full workload sizes, in the launch configuration the benchmark times
    (its `*_kv_pair` variants): the pair pass's dK and dV equal the
    single-CTA pass's bit for bit, and the kernel that ran is the pair one."""
    x = W.make_inputs(W.WORKLOADS[name])
    g = _run(x, True, monkeypatch)
    single = _run(x, False, monkeypatch)
    for n in ("dk", "dv"):
        assert np.array_equal(g[n], single[n]), n
