"""Pins for the oracle's GQA and sliding-window readings.  CPU only.

GQA ("Optimizing Jagged Flash Attention with TLX", sections 3 and 4 name it
as a supported variant): query head h reads K/V head h // (H / H_kv), and
dK / dV of a K/V head sum over its query heads.  Sliding window (same
sections): key j is kept for query i iff i - wl <= j <= i + wr, causal being
wr = 0.  The pins:

* library routes: torch's float64 scaled_dot_product_attention with
  `enable_gqa` (its own head grouping) and with a band mask built by torch's
  tril / triu, plus its autograd, on padded sequences;
* special cases: GQA equals multi-head attention on K/V heads repeated per
  group (dK / dV then summed per group); a window wider than every sequence
  is no window; a zero window keeps only the diagonal, so O = V, LSE =
  scale q_i.k_i, dV = dO and dQ = dK = 0; wl = 0 with causal is the same;
* brute force: explicit loops over admissible keys on a tiny case;
* finite differences of the windowed GQA loss;
* planted slips (head mapping h % H_kv, dK overwritten instead of summed
  over the group, an off-by-one or swapped window bound) that these catch.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import jfa_oracle


def _case(lengths, H, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(off[-1])
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((T, Hkv, D))
    v = rng.standard_normal((T, Hkv, D))
    do = rng.standard_normal((T, H, D))
    return q, k, v, do, off


def _torch_padded(q, k, v, do, off, scale, causal=False, window=None):
    """Padded [B, H, Lmax, D] float64 SDPA (enable_gqa when K/V have fewer
    heads) with a key-padding and band mask, + autograd.  Written without the
    oracle: the band comes from torch's tril / triu diagonals."""
    B = len(off) - 1
    L = np.diff(off)
    Lm = int(L.max())
    pad = lambda x: torch.stack([
        torch.nn.functional.pad(torch.from_numpy(x[off[b]:off[b + 1]]).permute(1, 0, 2),
                                (0, 0, 0, Lm - int(L[b]))) for b in range(B)])
    Q, K, V, dO = (pad(x).clone().requires_grad_(True) for x in (q, k, v, do))
    wl, wr = (None, None) if window is None else window
    if causal:
        wr = 0
    mask = torch.zeros(B, 1, Lm, Lm, dtype=torch.bool)
    ones = torch.ones(Lm, Lm, dtype=torch.bool)
    for b in range(B):
        n = int(L[b])
        m = torch.zeros(Lm, Lm, dtype=torch.bool)
        m[:, :n] = True
        if wr is not None:
            m &= ones.tril(wr)    # j - i <= wr
        if wl is not None:
            m &= ones.triu(-wl)   # j - i >= -wl
        m[n:, :] = True  # padded query rows: anything finite, dropped below
        mask[b, 0] = m
    gqa = K.shape[1] != Q.shape[1]
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                                         enable_gqa=gqa)
    (O * dO.detach()).sum().backward()
    unpad = lambda X: np.concatenate([X[b, :, :int(L[b])].permute(1, 0, 2).detach().numpy()
                                      for b in range(B)])
    return unpad(O), unpad(Q.grad), unpad(K.grad), unpad(V.grad)


def _check_vs_torch(H, Hkv, causal, window, seed, lengths=(1, 17, 5, 33, 2, 40)):
    D, scale = 8, 0.3
    q, k, v, do, off = _case(list(lengths), H, Hkv, D, seed)
    out, _ = oracle.forward(q, k, v, off, scale, causal, window=window)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal, window=window)
    O, dQ, dK, dV = _torch_padded(q, k, v, do, off, scale, causal, window)
    np.testing.assert_allclose(out, O, atol=1e-12)
    np.testing.assert_allclose(dq, dQ, atol=1e-11)
    np.testing.assert_allclose(dk, dK, atol=1e-11)
    np.testing.assert_allclose(dv, dV, atol=1e-11)


@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (4, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_torch_enable_gqa(H, Hkv, causal):
    _check_vs_torch(H, Hkv, causal, None, seed=31)


@pytest.mark.parametrize("window,causal", [((3, 5), False), ((7, 0), False), ((None, 2), False),
                                           ((4, None), False), ((6, None), True), ((0, 3), False)])
def test_window_equals_torch_band_mask(window, causal):
    _check_vs_torch(2, 2, causal, window, seed=32)


def test_window_and_gqa_equal_torch():
    _check_vs_torch(4, 2, True, (9, None), seed=33)
    _check_vs_torch(6, 3, False, (5, 2), seed=34)


def test_gqa_equals_repeated_kv():
    """GQA = multi-head attention on K/V heads repeated per group; dK / dV of
    a K/V head = the sum of the repeated heads' gradients."""
    H, Hkv, D, scale = 6, 2, 8, 0.4
    q, k, v, do, off = _case([4, 0, 11, 7], H, Hkv, D, seed=35)
    g = H // Hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    for causal, window in ((False, None), (True, None), (False, (2, 3))):
        out, lse = oracle.forward(q, k, v, off, scale, causal, window=window)
        out_r, lse_r = oracle.forward(q, kr, vr, off, scale, causal, window=window)
        np.testing.assert_array_equal(out, out_r)
        np.testing.assert_array_equal(lse, lse_r)
        dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal, window=window)
        dq_r, dk_r, dv_r = oracle.backward(q, kr, vr, off, do, scale, causal, window=window)
        np.testing.assert_allclose(dq, dq_r, atol=1e-13)
        T = k.shape[0]
        np.testing.assert_allclose(dk, dk_r.reshape(T, Hkv, g, D).sum(2), atol=1e-13)
        np.testing.assert_allclose(dv, dv_r.reshape(T, Hkv, g, D).sum(2), atol=1e-13)


def test_broadcast_gqa_equals_repeated_kv():
    H, Hkv, D, scale, Lq = 4, 2, 8, 0.3, 5
    rng = np.random.default_rng(36)
    lengths = [3, 0, 9, 2]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, B = int(off[-1]), len(lengths)
    q = rng.standard_normal((Lq, H, D))
    k, v = rng.standard_normal((T, Hkv, D)), rng.standard_normal((T, Hkv, D))
    do = rng.standard_normal((B, Lq, H, D))
    g = H // Hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    out, lse = oracle.forward(q, k, v, off, scale, broadcast_q=True)
    out_r, lse_r = oracle.forward(q, kr, vr, off, scale, broadcast_q=True)
    np.testing.assert_array_equal(out, out_r)
    np.testing.assert_array_equal(lse, lse_r)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, broadcast_q=True)
    dq_r, dk_r, dv_r = oracle.backward(q, kr, vr, off, do, scale, broadcast_q=True)
    np.testing.assert_allclose(dq, dq_r, atol=1e-13)
    np.testing.assert_allclose(dk, dk_r.reshape(T, Hkv, g, D).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(T, Hkv, g, D).sum(2), atol=1e-13)


def test_wide_window_is_no_window():
    H, D, scale = 2, 8, 0.5
    q, k, v, do, off = _case([5, 12, 1], H, H, D, seed=37)
    # (causal, window): the longest sequence has 12 keys, so |i - j| <= 11
    for causal, window in ((False, (12, 12)), (True, (11, None)), (False, (100, None))):
        windowed = oracle.forward(q, k, v, off, scale, causal, window=window)
        plain = oracle.forward(q, k, v, off, scale, causal)
        for x, y in zip(windowed, plain):
            np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal,window", [(False, (0, 0)), (True, (0, None))])
def test_zero_window_keeps_the_diagonal(causal, window):
    """Only key i for query i: O = V row, LSE = scale q_i.k_i, dV = dO (summed
    over the group's heads), dQ = dK = 0."""
    H, Hkv, D, scale = 4, 2, 8, 0.45
    q, k, v, do, off = _case([3, 1, 8], H, Hkv, D, seed=38)
    g = H // Hkv
    out, lse = oracle.forward(q, k, v, off, scale, causal, window=window)
    hk = np.arange(H) // g
    np.testing.assert_allclose(out, v[:, hk, :], atol=1e-14)
    np.testing.assert_allclose(lse, scale * np.einsum("thd,thd->ht", q, k[:, hk, :]), atol=1e-13)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal, window=window)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    T = k.shape[0]
    np.testing.assert_allclose(dv, do.reshape(T, Hkv, g, D).sum(2), atol=1e-14)


def test_window_brute_force():
    """Every output row by explicit sums over the admissible keys."""
    H, Hkv, D, scale = 4, 2, 4, 0.6
    lengths = [6, 9]
    q, k, v, do, off = _case(lengths, H, Hkv, D, seed=39)
    wl, wr = 2, 1
    out, lse = oracle.forward(q, k, v, off, scale, window=(wl, wr))
    g = H // Hkv
    for b in range(len(lengths)):
        s0, s1 = int(off[b]), int(off[b + 1])
        for h in range(H):
            for i in range(s0, s1):
                keys = [j for j in range(s0, s1) if i - wl <= j <= i + wr]
                e = [math.exp(scale * float(np.dot(q[i, h], k[j, h // g]))) for j in keys]
                den = sum(e)
                o = sum(w * v[j, h // g] for w, j in zip(e, keys)) / den
                np.testing.assert_allclose(out[i, h], o, atol=1e-13)
                assert abs(lse[h, i] - math.log(den)) < 1e-13


def test_window_gqa_finite_differences():
    H, Hkv, D, scale = 4, 2, 3, 0.7
    q, k, v, do, off = _case([4, 6], H, Hkv, D, seed=40)
    window = (2, 1)

    def loss(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, off, scale, window=window)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, window=window)
    eps = 1e-6
    rng = np.random.default_rng(41)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**{n + "_": a for n, a in args_p.items()}) -
                  loss(**{n + "_": a for n, a in args_m.items()})) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


# ------------------------------------------------------ planted slips caught

def _mutant_module(replace_from, replace_to):
    import importlib.util
    import inspect
    src = inspect.getsource(jfa_oracle)
    if replace_from not in src:  # a stale slip must not pass as a caught one
        raise LookupError(replace_from)
    spec = importlib.util.spec_from_loader("jfa_oracle_variant_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(replace_from, replace_to), "jfa_oracle_variant_mutant", "exec"),
         mod.__dict__)
    return mod


def _check_module(mod, H, Hkv, causal, window, seed=42):
    D, scale = 8, 0.3
    q, k, v, do, off = _case([1, 17, 5, 33, 2, 40], H, Hkv, D, seed)
    out, _ = mod.forward(q, k, v, off, scale, causal, window=window)
    dq, dk, dv = mod.backward(q, k, v, off, do, scale, causal, window=window)
    O, dQ, dK, dV = _torch_padded(q, k, v, do, off, scale, causal, window)
    np.testing.assert_allclose(out, O, atol=1e-12)
    np.testing.assert_allclose(dq, dQ, atol=1e-11)
    np.testing.assert_allclose(dk, dK, atol=1e-11)
    np.testing.assert_allclose(dv, dV, atol=1e-11)


def test_unmutated_copy_passes():
    _check_module(_mutant_module("", ""), 4, 2, False, (3, 5))


@pytest.mark.parametrize("slip", [
    ("kb, vb = k[s0:s1, h // group, :], v[s0:s1, h // group, :]\n        qb = q",
     "kb, vb = k[s0:s1, h % Hkv, :], v[s0:s1, h % Hkv, :]\n        qb = q"),
    ("dk[s0:s1, h // group, :] += dkb", "dk[s0:s1, h // group, :] = dkb"),
    ("dv[s0:s1, h // group, :] += dvb", "dv[s0:s1, h // group, :] = dvb"),
    ("s = np.where(j < i - wl, -np.inf, s)", "s = np.where(j <= i - wl, -np.inf, s)"),
    ("s = np.where(j > i + wr, -np.inf, s)", "s = np.where(j > i + wr + 1, -np.inf, s)"),
    ("wl, wr = (None, None) if window is None else window",
     "wr, wl = (None, None) if window is None else window"),
])
def test_planted_variant_slips_are_caught(slip):
    mod = _mutant_module(*slip)
    with pytest.raises(AssertionError):
        _check_module(mod, 4, 2, False, (3, 5))
