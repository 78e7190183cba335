"""GPU parity of the block-sparse variant ("Optimizing Jagged Flash Attention
with TLX", section 3, "Block-sparse attention") against the fp64 oracle.

* Stage 2 (jfa_fwd_sparse) on seeded random block lists drawn by the input
  generator, element by element: ragged sequences, lists with one block, all
  blocks, none (O = 0, LSE = -inf), D = 64 and 128, GQA.
* Stage 1 (jfa_block_select): counts exactly; the selected set equals the
  oracle's wherever the oracle's scores separate the k-th and (k+1)-th best
  by more than the fp32 rounding of the GPU's scores, and is valid (no
  unselected block scores clearly higher than a selected one) everywhere;
  unused slots hold -1.
* Both stages together against the oracle's own selection and forward, on
  inputs whose selections are unambiguous.
* A bad list is caught on the device and nothing is written.
"""
import numpy as np
import pytest
import torch

import jfa_workloads as W
from oracle import jfa_oracle as orc
from tests.gpu_common import compare, f64, inputs

pytestmark = pytest.mark.gpu

GAP = 1e-4  # fp32 score rounding is far below this


def _dev(x):
    dev = torch.device("cuda")
    return ((x[n].to(dev) for n in ("q", "k", "v")), torch.from_numpy(x["offsets"]).to(dev))


def _gpu_sparse(x, blocks, counts):
    import jagged_flash_attention_gb300 as jfa
    (q, k, v), off = _dev(x)
    bl = torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.int32)).cuda()
    ct = torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).cuda()
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], bl, ct, scale=x["scale"])
    jfa.jfa_sync_and_check()
    return {"out": f64(out), "lse": f64(lse)}


def _oracle_sparse(x, blocks, counts):
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out, lse = orc.forward_sparse(q, k, v, x["offsets"], x["scale"], blocks, counts)
    return {"out": out, "lse": lse}


LIST_CASES = {
    "d128_edges_half": (dict(name="jagged_self", lengths=[1, 127, 128, 129, 255, 256, 257, 700],
                             H=2), 0.5, 0.0),
    "d128_one_block": (dict(name="jagged_self", lengths=[300, 1000, 40], H=2), 0.0, 0.0),
    "d128_all_blocks": (dict(name="jagged_self", lengths=[513, 2], H=2), 1.0, 0.0),
    "d128_some_empty": (dict(name="jagged_self", lengths=[600, 260, 5], H=2), 0.4, 0.3),
    "d64_gqa": (dict(name="tiny_self", lengths=[900, 3, 385], H=4, Hkv=2), 0.5, 0.1),
    "d128_gqa_long": (dict(name="jagged_self", lengths=[3000, 129], H=4, Hkv=1), 0.3, 0.0),
}


@pytest.mark.parametrize("case", list(LIST_CASES), ids=list(LIST_CASES))
def test_sparse_forward_on_given_lists(case):
    spec, p_keep, p_empty = LIST_CASES[case]
    spec = dict(spec)
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    blocks, counts = W.random_block_lists(x["lengths"], x["H"], x["max_len"], seed=7,
                                          p_keep=p_keep, p_empty=p_empty)
    g = _gpu_sparse(x, blocks, counts)
    r = _oracle_sparse(x, blocks, counts)
    print(case, compare(g, r, ("out", "lse")))


def _gpu_select(x, permille):
    import jagged_flash_attention_gb300 as jfa
    (q, k, _), off = _dev(x)
    blocks, counts = jfa.block_select(q, k, off, x["max_len"], permille)
    jfa.jfa_sync_and_check()
    return blocks.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("permille,spec", [
    (500, dict(name="jagged_self", lengths=[1, 300, 1000, 129, 2048], H=4, Hkv=2)),
    (250, dict(name="tiny_self", lengths=[700, 64, 1500], H=3)),
    (1000, dict(name="jagged_self", lengths=[500, 130], H=2)),
    (1, dict(name="jagged_self", lengths=[900, 17], H=2)),
])
def test_block_select(permille, spec):
    spec = dict(spec)
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    gb, gc = _gpu_select(x, permille)
    rb, rc, rs = orc.block_select(f64(x["q"]), f64(x["k"]), x["offsets"], permille)
    np.testing.assert_array_equal(gc, rc)
    exact = 0
    for b in range(gc.shape[0]):
        for h in range(gc.shape[1]):
            for i in range(gc.shape[2]):
                c = int(gc[b, h, i])
                assert np.all(gb[b, h, i, c:] == -1)
                if c == 0:
                    continue
                sel = gb[b, h, i, :c]
                assert np.all(np.diff(sel) > 0)
                sc = rs[b, h, i]
                nk = int(np.sum(~np.isnan(sc)))
                assert sel.min() >= 0 and sel.max() < nk
                unsel = np.setdiff1d(np.arange(nk), sel)
                if unsel.size:  # valid: nothing left out scores clearly above a kept block
                    assert sc[unsel].max() <= sc[sel].min() + GAP
                srt = np.sort(sc[:nk])[::-1]
                if c == nk or srt[c - 1] - srt[c] > GAP:
                    np.testing.assert_array_equal(sel, rb[b, h, i, :c])
                    exact += 1
    assert exact > 0
    print(permille, "exactly compared lists:", exact)


def test_select_then_forward_matches_oracle():
    """Stage 1 then stage 2 on the GPU against the oracle's own selection and
    sparse forward (inputs whose selections are unambiguous)."""
    import jagged_flash_attention_gb300 as jfa
    x = inputs("jagged_self", [1500, 700, 257], H=2)
    q64, k64 = f64(x["q"]), f64(x["k"])
    rb, rc, rs = orc.block_select(q64, k64, x["offsets"], 500)
    # the seeded inputs separate the k-th and (k+1)-th scores clearly
    for idx in np.ndindex(rc.shape):
        c = int(rc[idx])
        if c == 0:
            continue
        srt = np.sort(rs[idx][~np.isnan(rs[idx])])[::-1]
        assert c == srt.size or srt[c - 1] - srt[c] > GAP, idx
    (q, k, v), off = _dev(x)
    blocks, counts = jfa.block_select(q, k, off, x["max_len"], 500)
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], blocks, counts, scale=x["scale"])
    jfa.jfa_sync_and_check()
    g = {"out": f64(out), "lse": f64(lse)}
    r = _oracle_sparse(x, rb, rc)
    print(compare(g, r, ("out", "lse")))


def test_full_selection_equals_dense():
    x = inputs("jagged_self", [1000, 129, 3], H=2)
    blocks, counts = W.random_block_lists(x["lengths"], 2, x["max_len"], seed=1, p_keep=1.0)
    g = _gpu_sparse(x, blocks, counts)
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out, lse = orc.forward(q, k, v, x["offsets"], x["scale"])
    compare(g, {"out": out, "lse": lse}, ("out", "lse"))


def test_bad_list_is_caught_on_the_device():
    import jagged_flash_attention_gb300 as jfa
    x = inputs("jagged_self", [600, 300], H=2)
    blocks, counts = W.random_block_lists(x["lengths"], 2, x["max_len"], seed=3, p_keep=1.0)
    blocks[0, 1, 1, :2] = [3, 2]  # not ascending
    (q, k, v), off = _dev(x)
    bl = torch.from_numpy(blocks).cuda()
    ct = torch.from_numpy(counts).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((2, x["T"]), 7.0, device="cuda")
    jfa.jfa_fwd_sparse(q, k, v, off, 2, 2, 2, 128, x["max_len"], 0, 0, x["scale"], bl, ct, out,
                       lse)
    with pytest.raises(jfa.JfaError, match="block-sparse list"):
        jfa.jfa_sync_and_check()
    assert torch.isnan(out).all() and (lse == 7.0).all()
    # a count above the sequence's K blocks
    blocks, counts = W.random_block_lists(x["lengths"], 2, x["max_len"], seed=3, p_keep=1.0)
    counts[1, 0, 0] = 4  # sequence 1 has 3 K blocks
    blocks[1, 0, 0, 3] = 3
    bl = torch.from_numpy(blocks).cuda()
    ct = torch.from_numpy(counts).cuda()
    jfa.jfa_fwd_sparse(q, k, v, off, 2, 2, 2, 128, x["max_len"], 0, 0, x["scale"], bl, ct, out,
                       lse)
    with pytest.raises(jfa.JfaError, match="block-sparse list"):
        jfa.jfa_sync_and_check()
    # the library still works afterwards
    blocks, counts = W.random_block_lists(x["lengths"], 2, x["max_len"], seed=4)
    compare(_gpu_sparse(x, blocks, counts), _oracle_sparse(x, blocks, counts), ("out", "lse"))


# ------------------------------------------------------------ broadcast-Q

def _gpu_sparse_bq(x, blocks, counts):
    import jagged_flash_attention_gb300 as jfa
    (q, k, v), off = _dev(x)
    bl = torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.int32)).cuda()
    ct = torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).cuda()
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], bl, ct, scale=x["scale"],
                                  broadcast_q=True)
    jfa.jfa_sync_and_check()
    return {"out": f64(out), "lse": f64(lse)}


def _oracle_sparse_bq(x, blocks, counts):
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out, lse = orc.forward_sparse(q, k, v, x["offsets"], x["scale"], blocks, counts,
                                  broadcast_q=True)
    return {"out": out, "lse": lse}


BQ_CASES = {
    "bq_d128_q300_gqa": dict(name="broadcast_q", lengths=[0, 1, 300, 700, 129], H=4, Hkv=2,
                             q_len=300),
    "bq_d64_q64": dict(name="skewed_broadcast_q", lengths=[1000, 0, 5, 257], H=2),
}


@pytest.mark.parametrize("case", list(BQ_CASES), ids=list(BQ_CASES))
def test_broadcast_sparse_forward_on_given_lists(case):
    spec = dict(BQ_CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    blocks, counts = W.random_block_lists(x["lengths"], x["H"], x["max_len"], seed=9,
                                          p_keep=0.5, p_empty=0.1, q_len=x["q_len"])
    print(case, compare(_gpu_sparse_bq(x, blocks, counts), _oracle_sparse_bq(x, blocks, counts),
                        ("out", "lse")))


@pytest.mark.parametrize("case", list(BQ_CASES), ids=list(BQ_CASES))
def test_broadcast_select_then_forward(case):
    """Both stages on the GPU against the oracle's selection and forward, where
    the oracle's scores separate the boundary; the lists valid everywhere."""
    import jagged_flash_attention_gb300 as jfa
    spec = dict(BQ_CASES[case])
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    (q, k, v), off = _dev(x)
    blocks, counts = jfa.block_select(q, k, off, x["max_len"], 500, broadcast_q=True)
    jfa.jfa_sync_and_check()
    gb, gc = blocks.cpu().numpy(), counts.cpu().numpy()
    rb, rc, rs = orc.block_select(f64(x["q"]), f64(x["k"]), x["offsets"], 500, broadcast_q=True)
    np.testing.assert_array_equal(gc, rc)
    same = True
    for idx in np.ndindex(gc.shape):
        c = int(gc[idx])
        if c == 0:
            continue
        sel = gb[idx][:c]
        sc = rs[idx]
        nk = int(np.sum(~np.isnan(sc)))
        assert np.all(np.diff(sel) > 0) and sel.max() < nk
        unsel = np.setdiff1d(np.arange(nk), sel)
        if unsel.size:
            assert sc[unsel].max() <= sc[sel].min() + GAP
        srt = np.sort(sc[:nk])[::-1]
        if c == nk or srt[c - 1] - srt[c] > GAP:
            np.testing.assert_array_equal(sel, rb[idx][:c])
        else:
            same = False
    g = _gpu_sparse_bq(x, gb, gc)  # the GPU's own lists, through the public call
    if same:  # every list is the oracle's: compare the outputs with the oracle's stages
        print(case, compare(g, _oracle_sparse_bq(x, rb, rc), ("out", "lse")))


# ------------------------------------------- causal and sliding-window masks

def _gpu_sparse_local(x, blocks, counts, causal, window):
    import jagged_flash_attention_gb300 as jfa
    (q, k, v), off = _dev(x)
    bl = torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.int32)).cuda()
    ct = torch.from_numpy(np.ascontiguousarray(counts, dtype=np.int32)).cuda()
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], bl, ct, scale=x["scale"],
                                  causal=causal, window=window)
    jfa.jfa_sync_and_check()
    return {"out": f64(out), "lse": f64(lse)}


def _oracle_sparse_local(x, blocks, counts, causal, window):
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out, lse = orc.forward_sparse(q, k, v, x["offsets"], x["scale"], blocks, counts,
                                  causal=causal, window=window)
    return {"out": out, "lse": lse}


LOCAL_CASES = {
    "causal_d128_edges": (dict(name="causal_self", lengths=[1, 127, 128, 129, 255, 256, 257, 700],
                               H=2), True, None, 0.5),
    "causal_d128_sparse_lists": (dict(name="causal_self", lengths=[1500, 300], H=2), True, None,
                                 0.25),
    "window_d64_gqa": (dict(name="tiny_self", lengths=[900, 3, 385], H=4, Hkv=2), False, (64, 0),
                       0.5),
    "window_d128_two_sided": (dict(name="jagged_self", lengths=[1000, 129, 600], H=2), False,
                              (300, 200), 0.6),
    "window_d128_right_only": (dict(name="jagged_self", lengths=[700, 260], H=2), False, (0, 130),
                               0.7),
}


@pytest.mark.parametrize("case", list(LOCAL_CASES), ids=list(LOCAL_CASES))
def test_local_sparse_forward_on_given_lists(case):
    """Random lists (also with blocks outside the band, and causal rows left
    without a listed admissible key) under a causal mask or a window."""
    spec, causal, window, p_keep = LOCAL_CASES[case]
    spec = dict(spec)
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    blocks, counts = W.random_block_lists(x["lengths"], x["H"], x["max_len"], seed=11,
                                          p_keep=p_keep, p_empty=0.1)
    r = _oracle_sparse_local(x, blocks, counts, causal, window)
    g = _gpu_sparse_local(x, blocks, counts, causal, window)
    print(case, compare(g, r, ("out", "lse")),
          "rows without a key:", int(np.isinf(r["lse"]).sum()))


@pytest.mark.parametrize("case", list(LOCAL_CASES)[1:4], ids=list(LOCAL_CASES)[1:4])
def test_local_select_and_forward(case):
    """Stage 1 under a local mask: counts exact, every list inside the
    candidates (the oracle's full selection), valid against the oracle's
    scores and equal to the oracle's list where the boundary is separated;
    then stage 2 on the GPU's lists against the oracle's forward on them."""
    import jagged_flash_attention_gb300 as jfa
    spec, causal, window, _ = LOCAL_CASES[case]
    spec = dict(spec)
    x = inputs(spec.pop("name"), spec.pop("lengths"), **spec)
    (q, k, v), off = _dev(x)
    blocks, counts = jfa.block_select(q, k, off, x["max_len"], 400, causal=causal, window=window)
    jfa.jfa_sync_and_check()
    gb, gc = blocks.cpu().numpy(), counts.cpu().numpy()
    q64, k64 = f64(x["q"]), f64(x["k"])
    rb, rc, rs = orc.block_select(q64, k64, x["offsets"], 400, causal=causal, window=window)
    cb, cc, _ = orc.block_select(q64, k64, x["offsets"], 1000, causal=causal, window=window)
    np.testing.assert_array_equal(gc, rc)
    exact = 0
    for idx in np.ndindex(gc.shape):
        c = int(gc[idx])
        assert np.all(gb[idx][c:] == -1)
        if c == 0:
            continue
        sel = gb[idx][:c]
        cand = cb[idx][:int(cc[idx])]
        assert np.all(np.diff(sel) > 0) and np.isin(sel, cand).all(), idx
        sc = rs[idx]
        unsel = np.setdiff1d(cand, sel)
        if unsel.size:
            assert sc[unsel].max() <= sc[sel].min() + GAP
        srt = np.sort(sc[cand])[::-1]
        if c == cand.size or srt[c - 1] - srt[c] > GAP:
            np.testing.assert_array_equal(sel, rb[idx][:c])
            exact += 1
    assert exact > 0
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], blocks, counts, scale=x["scale"],
                                  causal=causal, window=window)
    jfa.jfa_sync_and_check()
    r = _oracle_sparse_local(x, gb, gc, causal, window)
    print(case, "exact lists:", exact, compare({"out": f64(out), "lse": f64(lse)}, r,
                                               ("out", "lse")))


def test_local_full_selection_equals_dense_local():
    x = inputs("causal_self", [1000, 129, 3], H=2)
    blocks, counts = W.random_block_lists(x["lengths"], 2, x["max_len"], seed=1, p_keep=1.0)
    g = _gpu_sparse_local(x, blocks, counts, True, (300, None))
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out, lse = orc.forward(q, k, v, x["offsets"], x["scale"], True, window=(300, None))
    compare(g, {"out": out, "lse": lse}, ("out", "lse"))


# ------------------------------------------------------------- full size

@pytest.mark.parametrize("name", ["jagged_self", "causal_self"])
def test_sparse_full_size_sampled(name):
    """Full workload sizes at 500 permille, in the launch configuration the
    benchmark times (jagged_self_block_sparse500, causal_self_block_sparse500;
    causal_self with its causal mask): the GPU's lists and forward on every
    sequence, the oracle on sampled sequences and heads, following the GPU's
    lists (the forward) and its own (the selection, compared where the
    oracle's scores separate the boundary, valid everywhere)."""
    import jagged_flash_attention_gb300 as jfa
    x = W.make_inputs(W.WORKLOADS[name])
    causal = bool(x["causal"])
    (q, k, v), off = _dev(x)
    blocks, counts = jfa.block_select(q, k, off, x["max_len"], 500, causal=causal)
    out, lse = jfa.forward_sparse(q, k, v, off, x["max_len"], blocks, counts, scale=x["scale"],
                                  causal=causal)
    jfa.jfa_sync_and_check()
    gb, gc = blocks.cpu().numpy(), counts.cpu().numpy()
    g_out, g_lse = f64(out), f64(lse)
    rng = np.random.default_rng(17)
    L = x["lengths"]
    order = np.argsort(L)
    seqs = sorted({int(order[-1]), int(order[len(L) // 2]), int(rng.integers(0, len(L)))})
    heads = sorted({0, x["H"] - 1})
    offs = x["offsets"]
    exact = 0
    for b in seqs:
        s0, s1 = int(offs[b]), int(offs[b + 1])
        sub_off = np.array([0, s1 - s0], dtype=np.int64)
        for h in heads:
            hk = h // (x["H"] // x["Hkv"])
            qs = f64(x["q"][s0:s1, h:h + 1])
            ks = f64(x["k"][s0:s1, hk:hk + 1])
            vs = f64(x["v"][s0:s1, hk:hk + 1])
            bl = gb[b:b + 1, h:h + 1]
            ct = gc[b:b + 1, h:h + 1]
            r_out, r_lse = orc.forward_sparse(qs, ks, vs, sub_off, x["scale"], bl, ct, causal=causal)
            got = {"out": g_out[s0:s1, h:h + 1], "lse": g_lse[h:h + 1, s0:s1]}
            compare(got, {"out": r_out, "lse": r_lse}, ("out", "lse"))
            rb, rc, rs = orc.block_select(qs, ks, sub_off, 500, causal=causal)
            cb, cc, _ = orc.block_select(qs, ks, sub_off, 1000, causal=causal)
            nq = rc.shape[2]  # the sequence's Q blocks; the GPU's lists past them are empty
            np.testing.assert_array_equal(ct[:, :, :nq], rc)
            assert not ct[:, :, nq:].any()
            for i in range(nq):
                c = int(ct[0, 0, i])
                if c == 0:
                    continue
                sel = bl[0, 0, i, :c]
                cand = cb[0, 0, i, :int(cc[0, 0, i])]
                assert np.all(np.diff(sel) > 0) and np.isin(sel, cand).all()
                sc = rs[0, 0, i]
                unsel = np.setdiff1d(cand, sel)
                if unsel.size:
                    assert sc[unsel].max() <= sc[sel].min() + GAP
                srt = np.sort(sc[cand])[::-1]
                if c == cand.size or srt[c - 1] - srt[c] > GAP:
                    np.testing.assert_array_equal(sel, rb[0, 0, i, :c])
                    exact += 1
    assert exact > 0
    print(name, seqs, heads, "exact lists:", exact)
