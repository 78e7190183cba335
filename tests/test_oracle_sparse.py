"""Pins for the oracle's block-sparse variant ("Optimizing Jagged Flash
Attention with TLX", section 3, "Block-sparse attention"): block scores from
mean-pooled Q (256-row) and K (128-key) blocks, top-k K blocks per Q block,
and attention over the selected blocks only.  CPU only.

* a full selection (permille = 1000) is dense attention;
* the sparse forward equals torch's float64 scaled_dot_product_attention with
  a boolean mask expanded (by torch) from the block list;
* brute force: selection by explicit loops (pooled sums, dot products, a
  sort keyed on (-score, index)); attention rows by explicit sums;
* invariants: a positive scale of Q, a constant added to every key row (the
  scores of one Q block all move by the same amount only for means, not for
  sums over ragged blocks), a permutation of rows inside a K block;
* the count rule k = max(1, ceil(permille * n / 1000));
* planted slips (sum for mean, lowest scores kept, 128-row Q blocks, head
  map h % H_kv) that these catch;
* with a causal mask or a sliding window: a full selection is dense local
  attention; candidates found by testing every (row, key) pair; the forward
  against SDPA with the block mask AND a torch.tril / torch.triu band; a
  causal row whose listed blocks hold no admissible key (O = 0, LSE =
  -inf); slips (band ignored by the candidates or the attention, k counted
  from all blocks) caught.
"""
import math

import numpy as np
import pytest
import torch

from oracle import jfa_oracle

QB, KB = 256, 128


def _case(lengths, H, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(off[-1])
    return (rng.standard_normal((T, H, D)), rng.standard_normal((T, Hkv, D)),
            rng.standard_normal((T, Hkv, D)), off)


def test_count_rule():
    for n in (1, 2, 3, 7, 16, 64, 65):
        for p in (1, 100, 333, 500, 999, 1000):
            assert jfa_oracle.sparse_k_count(n, p) == min(n, max(1, math.ceil(p * n / 1000)))
    assert jfa_oracle.sparse_k_count(0, 500) == 0


def test_full_selection_is_dense():
    q, k, v, off = _case([300, 1, 513, 129], 4, 2, 8, seed=51)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 1000)
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.3, blocks, counts)
    ref_out, ref_lse = jfa_oracle.forward(q, k, v, off, 0.3)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def _torch_block_masked(q, k, v, off, scale, blocks, counts):
    """Per sequence: SDPA (enable_gqa) with a mask expanded by torch from the
    block-level selection matrix."""
    out = np.zeros(q.shape)
    H = q.shape[1]
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        nqb, nkb = -(-n // QB), -(-n // KB)
        sel = torch.zeros(H, nqb, nkb, dtype=torch.bool)
        for h in range(H):
            for i in range(nqb):
                for j in blocks[b, h, i, :counts[b, h, i]]:
                    sel[h, i, int(j)] = True
        mask = sel.repeat_interleave(QB, dim=1)[:, :n].repeat_interleave(KB, dim=2)[:, :, :n]
        Q = torch.from_numpy(q[s0:s1]).permute(1, 0, 2)
        K = torch.from_numpy(k[s0:s1]).permute(1, 0, 2)
        V = torch.from_numpy(v[s0:s1]).permute(1, 0, 2)
        O = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=scale, enable_gqa=K.shape[0] != Q.shape[0])
        out[s0:s1] = O.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("permille", [250, 500, 750])
def test_sparse_forward_equals_torch_block_mask(permille):
    q, k, v, off = _case([700, 129, 1000, 5], 4, 2, 8, seed=52)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, permille)
    out, _ = jfa_oracle.forward_sparse(q, k, v, off, 0.25, blocks, counts)
    ref = _torch_block_masked(q, k, v, off, 0.25, blocks, counts)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_sparse_forward_brute_force_rows():
    q, k, v, off = _case([600], 2, 1, 4, seed=53)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 400)
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.5, blocks, counts)
    rng = np.random.default_rng(0)
    for i in rng.choice(600, 12, replace=False):
        for h in range(2):
            keys = [j for j in range(600) if j // KB in set(blocks[0, h, i // QB, :counts[0, h, i // QB]].tolist())]
            e = [math.exp(0.5 * float(np.dot(q[i, h], k[j, 0]))) for j in keys]
            den = sum(e)
            o = sum(w * v[j, 0] for w, j in zip(e, keys)) / den
            np.testing.assert_allclose(out[i, h], o, atol=1e-12)
            assert abs(lse[h, i] - math.log(den)) < 1e-12


def _select_by_loops(q, k, off, permille, group):
    """Selection written with explicit loops and a sort keyed on (-score, j)."""
    res = {}
    H, D = q.shape[1], q.shape[2]
    for b in range(len(off) - 1):
        s0, n = int(off[b]), int(off[b + 1] - off[b])
        nk = -(-n // KB)
        kk = 0 if nk == 0 else min(nk, max(1, -(-(permille * nk) // 1000)))
        for h in range(H):
            kbar = []
            for j in range(nk):
                rows = range(s0 + j * KB, s0 + min(n, (j + 1) * KB))
                kbar.append([sum(k[r, h // group, d] for r in rows) / len(rows) for d in range(D)])
            for i in range(-(-n // QB)):
                rows = range(s0 + i * QB, s0 + min(n, (i + 1) * QB))
                qbar = [sum(q[r, h, d] for r in rows) / len(rows) for d in range(D)]
                sc = [sum(a * c for a, c in zip(qbar, kbar[j])) for j in range(nk)]
                best = sorted(range(nk), key=lambda j: (-sc[j], j))[:kk]
                res[(b, h, i)] = sorted(best)
    return res


def test_selection_brute_force():
    q, k, v, off = _case([300, 1, 700, 129], 4, 2, 6, seed=54)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 500)
    ref = _select_by_loops(q, k, off, 500, 2)
    for (b, h, i), sel in ref.items():
        assert list(blocks[b, h, i, :counts[b, h, i]]) == sel, (b, h, i)


def test_selection_invariants():
    q, k, v, off = _case([900, 333, 1025], 2, 2, 8, seed=55)
    base, counts, _ = jfa_oracle.block_select(q, k, off, 400)
    # a positive scale of Q keeps the order of every score row
    b2, _, _ = jfa_oracle.block_select(3.5 * q, k, off, 400)
    np.testing.assert_array_equal(base, b2)
    # a constant added to every key row moves all scores of a Q block alike
    c = np.random.default_rng(1).standard_normal(8) * 5
    b3, _, _ = jfa_oracle.block_select(q, k + c, off, 400)
    np.testing.assert_array_equal(base, b3)
    # rows permuted inside each K block
    perm = np.arange(k.shape[0])
    for b in range(3):
        s0, s1 = off[b], off[b + 1]
        for j0 in range(s0, s1, KB):
            seg = perm[j0:min(s1, j0 + KB)]
            perm[j0:min(s1, j0 + KB)] = seg[::-1]
    b4, _, _ = jfa_oracle.block_select(q, k[perm], off, 400)
    np.testing.assert_array_equal(base, b4)


# ------------------------------------------------------ planted slips caught

def _mutant_module(replace_from, replace_to):
    import importlib.util
    import inspect
    src = inspect.getsource(jfa_oracle)
    if replace_from not in src:  # a stale slip must not pass as a caught one
        raise LookupError(replace_from)
    spec = importlib.util.spec_from_loader("jfa_oracle_sparse_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(replace_from, replace_to), "jfa_oracle_sparse_mutant", "exec"),
         mod.__dict__)
    return mod


def _check(mod):
    q, k, v, off = _case([300, 1, 700, 129], 4, 2, 6, seed=54)
    blocks, counts, _ = mod.block_select(q, k, off, 500)
    ref = _select_by_loops(q, k, off, 500, 2)
    for (b, h, i), sel in ref.items():
        assert list(blocks[b, h, i, :counts[b, h, i]]) == sel, (b, h, i)
    # the invariant that separates means from sums over ragged blocks
    c = np.full(6, 3.0)
    b3, _, _ = mod.block_select(q, k + c, off, 500)
    np.testing.assert_array_equal(blocks, b3)
    out, _ = mod.forward_sparse(q, k, v, off, 0.25, blocks, counts)
    np.testing.assert_allclose(out, _torch_block_masked(q, k, v, off, 0.25, blocks, counts),
                               atol=1e-12)


def test_unmutated_copy_passes():
    _check(_mutant_module("", ""))


@pytest.mark.parametrize("slip", [
    ("h // group, :].mean(axis=0) for j in range(nk)", "h // group, :].sum(axis=0) for j in range(nk)"),
    ("order = cand[np.argsort(-sc[cand]", "order = cand[np.argsort(sc[cand]"),
    ("keep = np.isin(kblock, blocks[b, h, i, :counts[b, h, i]])",
     "keep = np.isin(kblock, blocks[b, h, min(i * 2, blocks.shape[2] - 1), :counts[b, h, i]])"),
    ("h // group, :].mean(axis=0) for j in range(nk)", "h % Hkv, :].mean(axis=0) for j in range(nk)"),
])
def test_planted_sparse_slips_are_caught(slip):
    with pytest.raises(AssertionError):
        _check(_mutant_module(*slip))


# ------------------------------------------------------------ broadcast-Q

def _bq_case(lengths, Lq, H, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(off[-1])
    return (rng.standard_normal((Lq, H, D)), rng.standard_normal((T, Hkv, D)),
            rng.standard_normal((T, Hkv, D)), off)


def test_broadcast_full_selection_is_dense():
    q, k, v, off = _bq_case([300, 0, 513, 129], 300, 4, 2, 8, seed=61)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 1000, broadcast_q=True)
    assert blocks.shape[2] == 2 and np.all(counts[1] == 0)  # q_len 300: two Q blocks
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.3, blocks, counts, broadcast_q=True)
    ref_out, ref_lse = jfa_oracle.forward(q, k, v, off, 0.3, broadcast_q=True)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], atol=1e-12)


@pytest.mark.parametrize("permille", [250, 600])
def test_broadcast_sparse_equals_torch_block_mask(permille):
    Lq, H = 300, 4
    q, k, v, off = _bq_case([700, 5, 0, 1000], Lq, H, 2, 8, seed=62)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, permille, broadcast_q=True)
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.25, blocks, counts, broadcast_q=True)
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        nqb, nkb = -(-Lq // QB), -(-n // KB)
        sel = torch.zeros(H, nqb, nkb, dtype=torch.bool)
        for h in range(H):
            for i in range(nqb):
                for j in blocks[b, h, i, :counts[b, h, i]]:
                    sel[h, i, int(j)] = True
        mask = sel.repeat_interleave(QB, dim=1)[:, :Lq].repeat_interleave(KB, dim=2)[:, :, :n]
        Q = torch.from_numpy(q).permute(1, 0, 2)
        K = torch.from_numpy(k[s0:s1]).permute(1, 0, 2)
        V = torch.from_numpy(v[s0:s1]).permute(1, 0, 2)
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=0.25,
                                                             enable_gqa=True)
        np.testing.assert_allclose(out[b], O.permute(1, 0, 2).numpy(), atol=1e-12)


def test_broadcast_selection_brute_force():
    Lq, H, D = 260, 2, 5
    q, k, v, off = _bq_case([300, 1, 0, 700], Lq, H, 1, D, seed=63)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 400, broadcast_q=True)
    for b in range(len(off) - 1):
        s0, n = int(off[b]), int(off[b + 1] - off[b])
        nk = -(-n // KB)
        for h in range(H):
            for i in range(-(-Lq // QB)):
                if nk == 0:
                    assert counts[b, h, i] == 0
                    continue
                kk = min(nk, max(1, -(-(400 * nk) // 1000)))
                rows = range(i * QB, min(Lq, (i + 1) * QB))
                qbar = [sum(q[r, h, d] for r in rows) / len(rows) for d in range(D)]
                sc = []
                for j in range(nk):
                    kr = range(s0 + j * KB, s0 + min(n, (j + 1) * KB))
                    kbar = [sum(k[r, 0, d] for r in kr) / len(kr) for d in range(D)]
                    sc.append(sum(a * c for a, c in zip(qbar, kbar)))
                best = sorted(sorted(range(nk), key=lambda j: (-sc[j], j))[:kk])
                assert list(blocks[b, h, i, :counts[b, h, i]]) == best


# ------------------------------------------- causal and sliding-window masks
# The TLX page keeps windowing in the sparse variant.  Reading: a Q block's
# candidates are the K blocks holding an admissible key of one of its rows,
# k counts from them, and the attention keeps a key only when it is both
# listed and admissible (a row left without one: O = 0, LSE = -inf).

LOCAL_MASKS = [(True, None), (False, (64, 0)), (False, (300, 200)), (True, (200, None)),
               (False, (0, 130))]


def _admissible(i, j, causal, window):
    wl, wr = (None, None) if window is None else window
    if causal and not (j <= i):
        return False
    if wl is not None and j < i - wl:
        return False
    if wr is not None and j > i + wr:
        return False
    return True


def _select_local_by_loops(q, k, off, permille, group, causal, window):
    """Candidates by testing every (row, key) pair of the Q block against
    every K block, then the pooled scores and a sort keyed on (-score, j)."""
    res = {}
    H, D = q.shape[1], q.shape[2]
    for b in range(len(off) - 1):
        s0, n = int(off[b]), int(off[b + 1] - off[b])
        nk = -(-n // KB)
        for h in range(H):
            kbar = []
            for j in range(nk):
                rows = range(s0 + j * KB, s0 + min(n, (j + 1) * KB))
                kbar.append([sum(k[r, h // group, d] for r in rows) / len(rows) for d in range(D)])
            for i in range(-(-n // QB)):
                qrows = range(i * QB, min(n, (i + 1) * QB))
                cand = [j for j in range(nk)
                        if any(_admissible(r, c, causal, window)
                               for r in qrows for c in range(j * KB, min(n, (j + 1) * KB)))]
                kk = min(len(cand), max(1, -(-(permille * len(cand)) // 1000)))
                qbar = [sum(q[s0 + r, h, d] for r in qrows) / len(qrows) for d in range(D)]
                sc = {j: sum(a * c for a, c in zip(qbar, kbar[j])) for j in cand}
                res[(b, h, i)] = sorted(sorted(cand, key=lambda j: (-sc[j], j))[:kk])
    return res


@pytest.mark.parametrize("causal,window", LOCAL_MASKS)
def test_local_full_selection_is_dense_local(causal, window):
    q, k, v, off = _case([300, 1, 700, 129], 4, 2, 8, seed=61)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 1000, causal=causal, window=window)
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.3, blocks, counts, causal=causal,
                                         window=window)
    ref_out, ref_lse = jfa_oracle.forward(q, k, v, off, 0.3, causal, window=window)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


@pytest.mark.parametrize("causal,window", LOCAL_MASKS[:3])
def test_local_selection_brute_force(causal, window):
    q, k, v, off = _case([300, 1, 700], 2, 1, 4, seed=62)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, 400, causal=causal, window=window)
    ref = _select_local_by_loops(q, k, off, 400, 2, causal, window)
    for (b, h, i), sel in ref.items():
        assert list(blocks[b, h, i, :counts[b, h, i]]) == sel, (b, h, i)


def _torch_local_block_masked(q, k, v, off, scale, blocks, counts, causal, window):
    """SDPA with the block mask AND the band (torch.tril / torch.triu on a
    ones matrix); rows whose mask is all False are set to O = 0, LSE = -inf."""
    out = np.zeros(q.shape)
    H = q.shape[1]
    lse = np.full((H, q.shape[0]), -np.inf)
    wl, wr = (None, None) if window is None else window
    if causal:
        wr = 0 if wr is None else min(wr, 0)
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        nqb, nkb = -(-n // QB), -(-n // KB)
        sel = torch.zeros(H, nqb, nkb, dtype=torch.bool)
        for h in range(H):
            for i in range(nqb):
                for j in blocks[b, h, i, :counts[b, h, i]]:
                    sel[h, i, int(j)] = True
        mask = sel.repeat_interleave(QB, dim=1)[:, :n].repeat_interleave(KB, dim=2)[:, :, :n]
        band = torch.ones(n, n, dtype=torch.bool)
        if wr is not None:
            band = torch.tril(band, diagonal=wr)
        if wl is not None:
            band = torch.triu(band, diagonal=-wl)
        mask = mask & band
        Q = torch.from_numpy(q[s0:s1]).permute(1, 0, 2)
        K = torch.from_numpy(k[s0:s1]).permute(1, 0, 2)
        V = torch.from_numpy(v[s0:s1]).permute(1, 0, 2)
        grp = Q.shape[0] // K.shape[0]
        O = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=scale, enable_gqa=grp != 1)
        S = (Q @ K.repeat_interleave(grp, dim=0).transpose(1, 2)) * scale
        L = torch.logsumexp(S.masked_fill(~mask, -math.inf), dim=-1)
        empty = ~mask.any(dim=-1)
        O = O.masked_fill(empty[..., None], 0.0)
        out[s0:s1] = O.permute(1, 0, 2).numpy()
        lse[:, s0:s1] = L.numpy()
    return out, lse


@pytest.mark.parametrize("causal,window", LOCAL_MASKS)
@pytest.mark.parametrize("permille", [250, 500])
def test_local_sparse_forward_equals_torch_masks(causal, window, permille):
    q, k, v, off = _case([700, 129, 1000, 5], 4, 2, 8, seed=63)
    blocks, counts, _ = jfa_oracle.block_select(q, k, off, permille, causal=causal, window=window)
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.25, blocks, counts, causal=causal,
                                         window=window)
    ref_out, ref_lse = _torch_local_block_masked(q, k, v, off, 0.25, blocks, counts, causal,
                                                 window)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_causal_row_without_listed_key():
    """Causal, one 300-key sequence, Q block 0 lists K block 1 only: rows
    0-127 see no admissible listed key (O = 0, LSE = -inf); row r in 128-255
    sees keys 128..r; Q block 1 lists K blocks 0 and 2."""
    q, k, v, off = _case([300], 1, 1, 4, seed=64)
    blocks = np.full((1, 1, 2, 3), -1, dtype=np.int64)
    counts = np.array([[[1, 2]]], dtype=np.int64)
    blocks[0, 0, 0, 0] = 1
    blocks[0, 0, 1, :2] = [0, 2]
    out, lse = jfa_oracle.forward_sparse(q, k, v, off, 0.5, blocks, counts, causal=True)
    assert np.all(out[:128] == 0.0) and np.all(np.isneginf(lse[0, :128]))
    for r in (128, 129, 200, 255, 256, 257, 299):
        keys = list(range(128, r + 1)) if r < 256 else list(range(0, 128)) + list(range(256, r + 1))
        e = [math.exp(0.5 * float(np.dot(q[r, 0], k[j, 0]))) for j in keys]
        o = sum(w * v[j, 0] for w, j in zip(e, keys)) / sum(e)
        np.testing.assert_allclose(out[r, 0], o, atol=1e-12)
        assert abs(lse[0, r] - math.log(sum(e))) < 1e-12


def _check_local(mod):
    causal, window = False, (300, 200)
    q, k, v, off = _case([300, 1, 700], 2, 1, 4, seed=62)
    blocks, counts, _ = mod.block_select(q, k, off, 400, causal=causal, window=window)
    ref = _select_local_by_loops(q, k, off, 400, 2, causal, window)
    for (b, h, i), sel in ref.items():
        assert list(blocks[b, h, i, :counts[b, h, i]]) == sel, (b, h, i)
    out, lse = mod.forward_sparse(q, k, v, off, 0.25, blocks, counts, causal=causal, window=window)
    ref_out, ref_lse = _torch_local_block_masked(q, k, v, off, 0.25, blocks, counts, causal,
                                                 window)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)


def test_unmutated_copy_passes_local():
    _check_local(_mutant_module("", ""))


@pytest.mark.parametrize("slip", [
    # the band ignored when choosing candidates
    ("hi = n - 1 if wr is None else min(n - 1, r1 + wr)", "hi = n - 1"),
    ("lo = 0 if wl is None else max(0, r0 - wl)", "lo = 0"),
    # k counted from all the sequence's K blocks
    ("kk = sparse_k_count(cand.size, permille)", "kk = min(cand.size, sparse_k_count(nk, permille))"),
    # the band ignored by the attention
    ("s = _scores(qrows, kb, scale, causal, r0, window)  # the band, if any",
     "s = _scores(qrows, kb, scale, causal, r0)"),
])
def test_planted_local_sparse_slips_are_caught(slip):
    with pytest.raises(AssertionError):
        _check_local(_mutant_module(*slip))
