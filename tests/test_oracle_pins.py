"""Pins for the fp64 oracle: closed forms, brute force, a library special
case, finite differences and invariants.  CPU only.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
flipped causal mask, a transposed product, a wrong sign in dS, a missing
Delta term, a wrong layout index) fails at least one test; the mutation tests
at the end plant such slips in the oracle and check that they are caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import jfa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _self_case(lengths, H, D, seed, scale_in=1.0):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(off[-1])
    q, k, v, do = (_rand((T, H, D), rng, scale_in) for _ in range(4))
    return q, k, v, do, off


def _bq_case(lengths, Lq, H, D, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, B = int(off[-1]), len(lengths)
    q = _rand((Lq, H, D), rng)
    k, v = _rand((T, H, D), rng), _rand((T, H, D), rng)
    do = _rand((B, Lq, H, D), rng)
    return q, k, v, do, off


# ---------------------------------------------------------------- closed forms

def _golden_cases():
    with open(os.path.join(GOLDEN, "closed_form_two_keys.json")) as f:
        return json.load(f)["cases"]


def _arr(x):
    return np.array(x, dtype=object).astype(float) if "-inf" in json.dumps(x) \
        else np.array(x, dtype=np.float64)


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    bq = case.get("broadcast_q", False)
    q, k, v, do = (_arr(case[n]) for n in ("q", "k", "v", "dout"))
    out, lse = oracle.forward(q, k, v, case["offsets"], case["scale"], case["causal"], bq)
    dq, dk, dv = oracle.backward(q, k, v, case["offsets"], do, case["scale"], case["causal"], bq)
    np.testing.assert_allclose(out, _arr(case["out"]), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(_arr(case["lse"])))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], _arr(case["lse"])[fin], rtol=0, atol=1e-12)
    for got, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        np.testing.assert_allclose(got, _arr(case[name]), rtol=0, atol=1e-12, err_msg=name)


def test_length_one_sequences():
    """A length-1 sequence returns its V row; LSE = scale q.k; dQ = dK = 0; dV = dO."""
    H, D, scale = 3, 8, 0.37
    q, k, v, do, off = _self_case([1] * 5, H, D, seed=11)
    out, lse = oracle.forward(q, k, v, off, scale)
    np.testing.assert_allclose(out, v, atol=1e-14)
    np.testing.assert_allclose(lse, scale * np.einsum("thd,thd->ht", q, k), atol=1e-13)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv, do, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(causal):
    """Constant V rows c give O = c, dQ = dK = 0 and dV_j = sum_i P_ij dO_i."""
    H, D, scale = 2, 4, 0.5
    lengths = [3, 1, 6]
    q, k, v, do, off = _self_case(lengths, H, D, seed=12)
    c = np.array([[0.5, -1.0, 2.0, 0.25], [1.5, 0.0, -0.75, 3.0]])
    v = np.broadcast_to(c[None], v.shape).copy()
    out, _ = oracle.forward(q, k, v, off, scale, causal)
    np.testing.assert_allclose(out, np.broadcast_to(c[None], out.shape), atol=1e-13)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    # dV by brute force with explicit python loops over i, j
    for b in range(len(lengths)):
        s0, s1 = off[b], off[b + 1]
        for h in range(H):
            for j in range(s0, s1):
                acc = np.zeros(D)
                for i in range(s0, s1):
                    if causal and j > i:
                        continue
                    p = _brute_prob(q, k, i, j, s0, s1, h, scale, causal)
                    acc += p * do[i, h]
                np.testing.assert_allclose(dv[j, h], acc, atol=1e-12)


def _brute_prob(q, k, i, j, s0, s1, h, scale, causal, qrow=None):
    """softmax probability of key j for query i by explicit sums (math.exp)."""
    qi = q[i, h] if qrow is None else qrow
    keys = [jj for jj in range(s0, s1) if not (causal and jj - s0 > i - s0)]
    den = sum(math.exp(scale * float(np.dot(qi, k[jj, h]))) for jj in keys)
    return math.exp(scale * float(np.dot(qi, k[j, h]))) / den


def test_rows_sum_to_one_onehot_v():
    """With one-hot V rows (L <= D) O exposes P: rows sum to 1 and O[i, j] = P_ij."""
    H, D, scale = 2, 16, 0.25
    lengths = [5, 16, 1, 9]
    q, k, _, _, off = _self_case(lengths, H, D, seed=13)
    T = off[-1]
    v = np.zeros((T, H, D))
    for b in range(len(lengths)):
        for j in range(off[b], off[b + 1]):
            v[j, :, j - off[b]] = 1.0
    for causal in (False, True):
        out, _ = oracle.forward(q, k, v, off, scale, causal)
        np.testing.assert_allclose(out.sum(-1), 1.0, atol=1e-13)
        for b in range(len(lengths)):
            s0, s1 = off[b], off[b + 1]
            for h in range(H):
                for i in range(s0, s1):
                    for j in range(s0, s1):
                        p = 0.0 if (causal and j > i) else \
                            _brute_prob(q, k, i, j, s0, s1, h, scale, causal)
                        assert abs(out[i, h, j - s0] - p) < 1e-13


def test_lse_direct_sum():
    """LSE equals log(sum exp(S)) computed without the max shift (small S)."""
    H, D, scale = 2, 4, 0.3
    lengths = [7, 2, 12]
    q, k, v, _, off = _self_case(lengths, H, D, seed=14, scale_in=0.5)
    for causal in (False, True):
        _, lse = oracle.forward(q, k, v, off, scale, causal)
        for b in range(len(lengths)):
            s0, s1 = off[b], off[b + 1]
            for h in range(H):
                for i in range(s0, s1):
                    tot = 0.0
                    for j in range(s0, s1):
                        if causal and j > i:
                            continue
                        tot += math.exp(scale * float(np.dot(q[i, h], k[j, h])))
                    assert abs(lse[h, i] - math.log(tot)) < 1e-13


# ------------------------------------------------- library special case (torch)

def _torch_padded_self(q, k, v, do, off, scale, causal):
    """Padded [B, H, Lmax, D] float64 SDPA with a key-padding mask + autograd.
    Written independently of the oracle (pad, mask, library attention)."""
    B = len(off) - 1
    L = np.diff(off)
    Lm = int(L.max())
    H, D = q.shape[1], q.shape[2]
    pad = lambda x: torch.stack([
        torch.nn.functional.pad(torch.from_numpy(x[off[b]:off[b + 1]]).permute(1, 0, 2),
                                (0, 0, 0, Lm - int(L[b]))) for b in range(B)])
    Q, K, V, dO = (pad(x).clone().requires_grad_(True) for x in (q, k, v, do))
    mask = torch.zeros(B, 1, Lm, Lm, dtype=torch.bool)
    for b in range(B):
        n = int(L[b])
        m = torch.zeros(Lm, Lm, dtype=torch.bool)
        m[:, :n] = True
        if causal:
            m &= torch.ones(Lm, Lm, dtype=torch.bool).tril()
        m[n:, :] = True  # padded query rows: anything finite, dropped below
        mask[b, 0] = m
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    (O * dO.detach()).sum().backward()
    unpad = lambda X: np.concatenate([X[b, :, :int(L[b])].permute(1, 0, 2).detach().numpy()
                                      for b in range(B)])
    return unpad(O), unpad(Q.grad), unpad(K.grad), unpad(V.grad)


@pytest.mark.parametrize("causal", [False, True])
def test_jagged_equals_padded_dense_torch(causal):
    H, D, scale = 3, 16, 0.2
    lengths = [1, 17, 5, 33, 2, 64]
    q, k, v, do, off = _self_case(lengths, H, D, seed=15)
    out, _ = oracle.forward(q, k, v, off, scale, causal)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal)
    O, dQ, dK, dV = _torch_padded_self(q, k, v, do, off, scale, causal)
    np.testing.assert_allclose(out, O, atol=1e-12)
    np.testing.assert_allclose(dq, dQ, atol=1e-11)
    np.testing.assert_allclose(dk, dK, atol=1e-11)
    np.testing.assert_allclose(dv, dV, atol=1e-11)


def test_broadcast_equals_stacked_torch():
    """Broadcast-Q = per-sequence cross attention stacked; dQ = sum of dQ_b."""
    H, D, scale, Lq = 2, 8, 0.35, 5
    lengths = [3, 0, 9, 1, 4]
    q, k, v, do, off = _bq_case(lengths, Lq, H, D, seed=16)
    out, lse = oracle.forward(q, k, v, off, scale, broadcast_q=True)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, broadcast_q=True)
    dq_sum = np.zeros_like(q)
    for b, n in enumerate(lengths):
        s0, s1 = off[b], off[b + 1]
        if n == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            assert np.all(dk[s0:s1] == 0)
            continue
        Q = torch.from_numpy(q).permute(1, 0, 2).clone().requires_grad_(True)
        K = torch.from_numpy(k[s0:s1]).permute(1, 0, 2).clone().requires_grad_(True)
        V = torch.from_numpy(v[s0:s1]).permute(1, 0, 2).clone().requires_grad_(True)
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)
        (O * torch.from_numpy(do[b]).permute(1, 0, 2)).sum().backward()
        np.testing.assert_allclose(out[b], O.permute(1, 0, 2).detach().numpy(), atol=1e-12)
        lse_ref = torch.logsumexp(scale * Q.detach() @ K.detach().transpose(1, 2), -1)
        np.testing.assert_allclose(lse[b], lse_ref.numpy(), atol=1e-12)
        np.testing.assert_allclose(dk[s0:s1], K.grad.permute(1, 0, 2).numpy(), atol=1e-11)
        np.testing.assert_allclose(dv[s0:s1], V.grad.permute(1, 0, 2).numpy(), atol=1e-11)
        dq_sum += Q.grad.permute(1, 0, 2).numpy()
    np.testing.assert_allclose(dq, dq_sum, atol=1e-11)


# ------------------------------------------------------- finite differences

def _loss(q, k, v, do, off, scale, causal, bq):
    out, _ = oracle.forward(q, k, v, off, scale, causal, bq)
    return float(np.sum(out * do))


@pytest.mark.parametrize("mode", ["self", "causal", "broadcast"])
def test_gradients_finite_differences(mode):
    H, D, scale = 1, 4, 0.7
    causal, bq = mode == "causal", mode == "broadcast"
    if bq:
        q, k, v, do, off = _bq_case([3, 5], 4, H, D, seed=17)
    else:
        q, k, v, do, off = _self_case([2, 5], H, D, seed=17)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, causal, bq)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = dict(q=q, k=k, v=v)
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, off, scale, causal, bq)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, off, scale, causal, bq)
            fd[idx] = (lp - lm) / (2 * eps)
        rel = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert rel < 1e-6, (name, rel)


# ------------------------------------------------------------ invariants

def test_sequence_permutation_permutes_outputs():
    H, D, scale = 2, 8, 0.4
    lengths = [4, 9, 1, 6]
    q, k, v, do, off = _self_case(lengths, H, D, seed=18)
    perm = [2, 0, 3, 1]
    idx = np.concatenate([np.arange(off[b], off[b + 1]) for b in perm])
    off_p = np.concatenate([[0], np.cumsum([lengths[b] for b in perm])])
    out, lse = oracle.forward(q, k, v, off, scale)
    out_p, lse_p = oracle.forward(q[idx], k[idx], v[idx], off_p, scale)
    np.testing.assert_allclose(out_p, out[idx], atol=1e-13)
    np.testing.assert_allclose(lse_p, lse[:, idx], atol=1e-13)
    g = oracle.backward(q, k, v, off, do, scale)
    gp = oracle.backward(q[idx], k[idx], v[idx], off_p, do[idx], scale)
    for a, b in zip(g, gp):
        np.testing.assert_allclose(b, a[idx], atol=1e-12)


def test_key_permutation_within_sequence():
    """Non-causal: permuting keys (with their values) leaves O unchanged and
    permutes dK, dV; dQ is unchanged."""
    H, D, scale, Lq = 2, 8, 0.4, 3
    lengths = [6, 4]
    q, k, v, do, off = _bq_case(lengths, Lq, H, D, seed=19)
    perm = np.array([3, 0, 5, 1, 4, 2, 7, 9, 6, 8])
    out, lse = oracle.forward(q, k, v, off, scale, broadcast_q=True)
    out_p, lse_p = oracle.forward(q, k[perm], v[perm], off, scale, broadcast_q=True)
    np.testing.assert_allclose(out_p, out, atol=1e-13)
    np.testing.assert_allclose(lse_p, lse, atol=1e-13)
    dq, dk, dv = oracle.backward(q, k, v, off, do, scale, broadcast_q=True)
    dqp, dkp, dvp = oracle.backward(q, k[perm], v[perm], off, do, scale, broadcast_q=True)
    np.testing.assert_allclose(dqp, dq, atol=1e-12)
    np.testing.assert_allclose(dkp, dk[perm], atol=1e-12)
    np.testing.assert_allclose(dvp, dv[perm], atol=1e-12)


def test_delta_equals_rowsum_p_dp():
    """rowsum(dO * O) equals sum_j P_ij dP_ij (the Delta used by the backward)."""
    H, D, scale = 2, 8, 0.4
    q, k, v, do, off = _self_case([5, 3], H, D, seed=20)
    out, _ = oracle.forward(q, k, v, off, scale)
    d = oracle.delta_rowsum(out, do)
    for b in range(2):
        s0, s1 = off[b], off[b + 1]
        for h in range(H):
            for i in range(s0, s1):
                tot = sum(_brute_prob(q, k, i, j, s0, s1, h, scale, False)
                          * float(np.dot(do[i, h], v[j, h])) for j in range(s0, s1))
                assert abs(d[h, i] - tot) < 1e-12


def test_sampling_matches_full():
    H, D, scale = 3, 8, 0.4
    q, k, v, do, off = _self_case([5, 7, 2], H, D, seed=21)
    out, lse = oracle.forward(q, k, v, off, scale)
    out_s, lse_s = oracle.forward(q, k, v, off, scale, seqs=[1], heads=[0, 2])
    sl = slice(off[1], off[2])
    np.testing.assert_array_equal(out_s[sl][:, [0, 2]], out[sl][:, [0, 2]])
    assert np.all(np.isnan(out_s[sl][:, 1])) and np.all(np.isnan(out_s[: off[1]]))


# -------------------------------------------- planted mistakes are caught

def _mutant_scores_no_scale(qc, kb, scale, causal, row0, window=None):
    return _orig_scores(qc, kb, 1.0, causal, row0, window)


def _mutant_scores_flipped_causal(qc, kb, scale, causal, row0, window=None):
    s = scale * (qc @ kb.T)
    if causal:
        i = np.arange(row0, row0 + qc.shape[0])[:, None]
        j = np.arange(kb.shape[0])[None, :]
        s = np.where(j < i, -np.inf, s)
    return s


_orig_scores = jfa_oracle._scores


@pytest.mark.parametrize("mutant", [_mutant_scores_no_scale, _mutant_scores_flipped_causal])
def test_planted_mistakes_in_scores_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(jfa_oracle, "_scores", mutant)
    with pytest.raises(AssertionError):
        test_jagged_equals_padded_dense_torch(causal=True)


def _mutant_ds_no_delta(p, dp):
    return p * dp


def _mutant_ds_wrong_sign(p, dp):
    return p * (np.sum(p * dp, axis=1)[:, None] - dp)


@pytest.mark.parametrize("mutant", [_mutant_ds_no_delta, _mutant_ds_wrong_sign])
def test_planted_mistakes_in_backward_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(jfa_oracle, "_grad_scores", mutant)
    with pytest.raises(AssertionError):
        test_gradients_finite_differences("self")
    with pytest.raises(AssertionError):
        test_jagged_equals_padded_dense_torch(causal=False)


def test_planted_row_index_slip_is_caught(monkeypatch):
    """Flip the sign of every other query row of dS (an index slip)."""
    orig = jfa_oracle._grad_scores

    def mutant(p, dp):
        return orig(p, dp) * np.where(np.arange(p.shape[0])[:, None] % 2 == 0, 1.0, -1.0)
    monkeypatch.setattr(jfa_oracle, "_grad_scores", mutant)
    with pytest.raises(AssertionError):
        test_gradients_finite_differences("broadcast")
