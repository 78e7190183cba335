"""The seeded workload generators: deterministic, and with the length
distributions each workload names."""
import numpy as np

import jfa_workloads as W


def test_lengths_are_deterministic_and_in_range():
    for name in W.ORDER:
        w = W.WORKLOADS[name]
        a, b = W.sample_lengths(w), W.sample_lengths(w)
        np.testing.assert_array_equal(a, b)
        assert a.size == w.B and a.min() >= 1
    L = W.sample_lengths(W.WORKLOADS["tiny_self"])
    assert L.max() <= 64
    L = W.sample_lengths(W.WORKLOADS["jagged_self"])
    assert L.min() >= 16 and L.max() <= 2048 and abs(L.mean() - 1032) < 150
    L = W.sample_lengths(W.WORKLOADS["broadcast_q"])
    assert L.max() <= 4096 and 380 < np.median(L) < 680
    L = W.sample_lengths(W.WORKLOADS["causal_self"])
    assert L.min() >= 256 and L.max() <= 8192
    L = W.sample_lengths(W.WORKLOADS["skewed_broadcast_q"])
    assert (L == 8192).sum() >= 41 and L.max() <= 8192 and 170 < L[L < 8192].mean() < 230


def test_offsets_and_pairs():
    off = W.offsets_from_lengths([3, 0, 5])
    assert off.dtype == np.int32 and list(off) == [0, 3, 3, 8]
    assert W.pairs([3, 0, 5]) == 9 + 25
    assert W.pairs([3, 5], causal=True) == 6 + 15
    assert W.pairs([3, 5], q_len=7, broadcast_q=True) == 56


def test_values_deterministic_bf16():
    import torch
    x = W.make_inputs(W.WORKLOADS["tiny_self"])
    y = W.make_inputs(W.WORKLOADS["tiny_self"])
    assert x["q"].dtype == torch.bfloat16
    assert torch.equal(x["q"], y["q"]) and torch.equal(x["dout"], y["dout"])
    assert x["q"].shape == (x["T"], 2, 64)
    b = W.make_inputs(W.WORKLOADS["broadcast_q"], lengths=[3, 4])
    assert b["q"].shape == (256, 4, 128) and b["dout"].shape == (2, 256, 4, 128)


def test_sparse_pair_count_by_enumeration():
    """The block-sparse bench's computed-pair count equals the number of
    (row, key) entries of the block mask AND the band, enumerated."""
    import bench
    rng = np.random.default_rng(5)
    lengths = np.array([1, 300, 700, 129])
    for causal, window in ((False, (-1, -1)), (True, (-1, -1)), (False, (100, 40)),
                           (True, (300, -1))):
        bl, ct = W.random_block_lists(lengths, 2, 700, seed=int(rng.integers(100)), p_keep=0.5)
        wl = None if window[0] < 0 else window[0]
        wr = None if window[1] < 0 else window[1]
        want = 0
        for b, n in enumerate(lengths.tolist()):
            for h in range(2):
                for r in range(n):
                    i = r // 256
                    listed = set(bl[b, h, i, :ct[b, h, i]].tolist())
                    for c in range(n):
                        ok = (c // 128 in listed and (not causal or c <= r)
                              and (wl is None or c >= r - wl) and (wr is None or c <= r + wr))
                        want += ok
        assert bench._sparse_pairs(lengths, 2, bl, ct, causal, window) == want


def test_every_bench_variant_resolves_to_a_workload():
    """Every name the bench line reports under `variants` maps to a workload
    definition (the GQA / window variants, the block-sparse and the CTA-pair
    ones)."""
    import bench
    names = list(W.VARIANTS) + list(bench.SPARSE_VARIANTS) + list(bench.PAIR_VARIANTS)
    for n in names:
        w = bench._workload_def(n)
        assert w.name in W.WORKLOADS, n


def test_breakdown_selects_the_dominant_flop_kernel():
    """bench's breakdown window: every kind profiled, then events only around
    the kernel with the most device time among those with algorithmic FLOPs
    (the pre-pass, FLOP-free, is never chosen even when it is slow)."""
    import types

    import bench

    calls = []
    prof = {"sched": (0.1, 3), "fwd": (0.9, 3), "prep": (5.0, 3), "bwd_kv": (1.6, 3),
            "bwd_q": (1.3, 3)}
    reads = iter([{}, prof])
    fake = types.SimpleNamespace(
        profile_read=lambda: next(reads),
        profile_select=lambda kinds=None: calls.append(("select", kinds)),
        profile_enable=lambda on: calls.append(("enable", on)))
    torch_ = types.SimpleNamespace(cuda=types.SimpleNamespace(synchronize=lambda: None))
    ran = []
    x = W.make_inputs(W.WORKLOADS["tiny_self"])
    got = bench._breakdown(fake, torch_, x, ran.append, 4)
    assert got == prof and ran == [4]
    assert calls == [("select", None), ("enable", True), ("enable", False),
                     ("select", ["bwd_kv"])]


def test_window_pairs_by_brute_force():
    """The useful-work count behind every TFLOPS figure, against an explicit
    mask: query i keeps key j iff i - left <= j <= i + right (causal: right
    = 0; -1: unbounded)."""
    lengths = [1, 7, 20, 0, 33]
    for causal, win in [(False, (3, 2)), (False, (0, -1)), (False, (-1, 4)), (True, (5, -1)),
                        (True, (-1, -1)), (False, (-1, -1)), (False, (0, 0))]:
        want = 0
        for n in lengths:
            for i in range(n):
                for j in range(n):
                    lo = i - win[0] if win[0] >= 0 else -10**9
                    hi = i + (0 if causal else (win[1] if win[1] >= 0 else 10**9))
                    if causal and win[1] >= 0:
                        hi = min(hi, i + win[1])
                    want += lo <= j <= hi
        assert W.pairs(lengths, causal=causal, window=win) == want, (causal, win)


def test_bench_work_model_products():
    """Tensor FLOPs per launch in the bench's model: 2*D per pair and
    product (forward 2 products, dK/dV pass 4, dQ pass 3: S and dP again,
    then dS K); the method's backward counts 5."""
    import bench
    for name, lengths in (("tiny_self", None), ("broadcast_q", [0, 5, 300])):
        x = W.make_inputs(W.WORKLOADS[name], lengths=lengths)
        p = bench._pairs(x)
        unit = 2.0 * x["H"] * x["D"] * p
        m = bench.kernel_model(x)
        fwd_f, bwd_f, _ = bench._flops(x)
        assert m["fwd"][0] == 2 * unit and fwd_f == 2 * unit
        assert m["bwd_kv"][0] == 4 * unit and bwd_f == 5 * unit
        assert m["bwd_qb" if x["broadcast_q"] else "bwd_q"][0] == 3 * unit
    frac, bound = bench._roof(1e12, 1e9, 1e-3, 1000.0, 1000.0)
    assert bound == "tensor" and abs(frac - 1.0) < 1e-12
