"""Plain fp64 CPU oracle for jagged (packed, padding-free) softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: it exists so that tests, the smoke check and the timed
CPU baseline of the benchmark can check the CUDA library against an obviously
correct definition.  It shares no code, constants or helpers with the CUDA
path; both sides only read the same seeded inputs.

What is computed (sources, by page title and section):

* "Optimizing Jagged Flash Attention with TLX" (pytorch.org), Introduction:
  sequences are packed back to back and their boundaries live in an offsets
  tensor; attention runs over the packed tensors without padded tokens.
* Same page, section 1 ("The Challenge"): in broadcast-Q mode one dense Q is
  shared by every sequence and dQ is summed over the whole batch.
* "cuTile Kernels - FMHA Implementation" (build.nvidia.com), "Attention
  Basics": Attention(Q, K, V) = softmax(Q K^T * scale) V, with causal masking
  setting future scores to -inf before the softmax.
* Same page, "Flash Attention Algorithm": the tiled online softmax reaches
  exactly this result (up to rounding order), so the oracle is the plain
  definition written out, one (sequence, head) at a time, with no tiling.
* "Optimizing Jagged Flash Attention with TLX", "2-CTA collaborative MMA":
  the backward needs dQ, dK and dV (five products per K/V block).  The pages
  do not print the backward formulas; the oracle uses the gradient of the
  definition above, which is what those five products compute:
      dV = P^T dO,  dP = dO V^T,  Delta_i = sum_j P_ij dP_ij,
      dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q.

Readings where the pages are silent (each listed in the design notes):

* Layouts: self-attention q, k, v, out are [T, H, D] with T = offsets[B];
  lse is [H, T].  Broadcast-Q: q and dq are [Lq, H, D], k, v, dk, dv are
  [T, H, D], out and dout are [B, Lq, H, D], lse is [B, H, Lq].
* LSE is the natural-log log-sum-exp of the scaled scores of each query row.
* Causal (self-attention only) keeps key j for query i iff j <= i, both
  counted from the start of their sequence.
* A sequence of length 0 contributes no rows in self-attention; in broadcast
  mode it yields O = 0, LSE = -inf and no dQ contribution.
* GQA ("Optimizing Jagged Flash Attention with TLX", sections 3 and 4 name
  it as a supported variant without defining it): k and v carry H_kv heads
  with H_kv dividing the H query heads; query head h reads K/V head
  h // (H / H_kv), consecutive query heads sharing one K/V head, and dK / dV
  of a K/V head sum the contributions of its H / H_kv query heads.
* Sliding window (same sections, also undefined there): window = (wl, wr)
  keeps key j for query i iff i - wl <= j <= i + wr, positions counted from
  the start of the sequence; None (or a negative value) leaves that side
  unbounded.  Causal is the right bound wr = 0; windows apply to
  self-attention only, as causal masking does.

Parity pins (tests/test_oracle_pins.py): closed forms (length 1, constant V,
a hand-derived two-key example in tests/golden), row-stochasticity, LSE by a
direct sum, padded-dense equality against torch's float64 SDPA on CPU (a
library special case), float64 autograd of that library route, central finite
differences of the gradients, broadcast = stacked per-sequence attention, and
permutation invariants.  The query-row chunking (ROW_CHUNK) is pinned in
tests/test_oracle_chunks.py: blocks of 3 and 7 rows against the same torch
float64 routes, with planted slips (causal offset lost, dK / dV overwritten
instead of summed, block rows taken from the wrong place) caught.  GQA and
windows are pinned in tests/test_oracle_variants.py, the block-sparse
selection and forward (end of this file) in tests/test_oracle_sparse.py.
"""
from __future__ import annotations

import numpy as np

ROW_CHUNK = 1024  # query rows per dense score block, so 8192-long rows fit


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _seq_bounds(offsets):
    off = np.asarray(offsets, dtype=np.int64)
    if off.ndim != 1 or off.size < 1 or off[0] != 0 or np.any(np.diff(off) < 0):
        raise ValueError("offsets must be 1-D, start at 0 and be non-decreasing")
    return off


def _window(causal, window):
    """(wl, wr) with None for an unbounded side; causal bounds wr by 0."""
    wl, wr = (None, None) if window is None else window
    wl = None if wl is None or wl < 0 else int(wl)
    wr = None if wr is None or wr < 0 else int(wr)
    if causal:
        wr = 0 if wr is None else min(wr, 0)
    return wl, wr


def _scores(qc, kb, scale, causal, row0, window=None):
    """Scaled scores of query rows [row0, row0+len(qc)) against all keys.

    Causal masking follows "cuTile Kernels - FMHA Implementation",
    "Attention Basics": future keys (j > i) get -inf before the softmax.  A
    sliding window (wl, wr) also gives -inf to keys j < i - wl or j > i + wr.
    """
    s = scale * (qc @ kb.T)
    wl, wr = _window(causal, window)
    if wl is not None or wr is not None:
        i = np.arange(row0, row0 + qc.shape[0])[:, None]
        j = np.arange(kb.shape[0])[None, :]
        if wr is not None:
            s = np.where(j > i + wr, -np.inf, s)
        if wl is not None:
            s = np.where(j < i - wl, -np.inf, s)
    return s


def _lse_rows(s):
    """Natural log-sum-exp per row; -inf for a row with no admissible key."""
    m = np.max(s, axis=1)
    finite = np.isfinite(m)
    m0 = np.where(finite, m, 0.0)
    with np.errstate(divide="ignore"):
        lse = m0 + np.log(np.sum(np.exp(s - m0[:, None]), axis=1))
    return np.where(finite, lse, -np.inf)


def _probs(s, lse):
    out = np.zeros_like(s)
    ok = np.isfinite(lse)
    out[ok] = np.exp(s[ok] - lse[ok, None])
    return out


def _grad_scores(p, dp):
    """dS = P * (dP - Delta) with Delta_i = sum_j P_ij dP_ij: the gradient of
    sum(O * dO) with respect to the scaled scores, row by row."""
    delta = np.sum(p * dp, axis=1)
    return p * (dp - delta[:, None])


def _pairs(B, H, seqs, heads, group=1):
    """(sequence, query head) pairs to compute.  A sampled head brings in
    every query head of its K/V head's group, so that sampled dK / dV hold
    the whole sum."""
    bs = range(B) if seqs is None else seqs
    if heads is None:
        hs = range(H)
    else:
        hs = sorted({g * group + i for h in heads for g in [h // group] for i in range(group)})
    return [(b, h) for b in bs for h in hs]


def _heads(q, k, broadcast_q):
    """(H, H_kv, group): query heads, K/V heads, query heads per K/V head."""
    H, Hkv = q.shape[1], k.shape[1]
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("the K/V head count must divide the query head count")
    return H, Hkv, H // Hkv


def _check_mask_args(broadcast_q, causal, window):
    if broadcast_q and (causal or _window(False, window) != (None, None)):
        raise ValueError("causal and window masks are defined for self-attention only")


def forward(q, k, v, offsets, scale, causal=False, broadcast_q=False,
            seqs=None, heads=None, window=None):
    """Attention forward over packed sequences.

    Returns (out, lse) in the layouts given in the module docstring, with H
    query heads (k and v may carry fewer, see GQA above).  With `seqs` /
    `heads` only those (sequence, head) pairs are computed; the other
    entries are NaN (used to sample outputs of large workloads).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    off = _seq_bounds(offsets)
    B = off.size - 1
    T, Hkv, D = k.shape
    H, Hkv, group = _heads(q, k, broadcast_q)
    if v.shape != k.shape or off[-1] != T:
        raise ValueError("k, v must be [T, H_kv, D] with T = offsets[B]")
    _check_mask_args(broadcast_q, causal, window)
    if broadcast_q:
        Lq = q.shape[0]
        out = np.full((B, Lq, H, D), np.nan)
        lse = np.full((B, H, Lq), np.nan)
    else:
        if q.shape != (T, H, D):
            raise ValueError("self-attention q must be [T, H, D]")
        out = np.full((T, H, D), np.nan)
        lse = np.full((H, T), np.nan)
    for b, h in _pairs(B, H, seqs, heads, group):
        s0, s1 = int(off[b]), int(off[b + 1])
        kb, vb = k[s0:s1, h // group, :], v[s0:s1, h // group, :]
        qb = q[:, h, :] if broadcast_q else q[s0:s1, h, :]
        nq = qb.shape[0]
        ob = np.zeros((nq, D))
        lb = np.full(nq, -np.inf)
        if s1 > s0:
            for r0 in range(0, nq, ROW_CHUNK):
                r1 = min(nq, r0 + ROW_CHUNK)
                s = _scores(qb[r0:r1], kb, scale, causal, r0, window)
                l = _lse_rows(s)
                ob[r0:r1] = _probs(s, l) @ vb
                lb[r0:r1] = l
        if broadcast_q:
            out[b, :, h, :] = ob
            lse[b, h, :] = lb
        else:
            out[s0:s1, h, :] = ob
            lse[h, s0:s1] = lb
    return out, lse


def backward(q, k, v, offsets, dout, scale, causal=False, broadcast_q=False,
             seqs=None, heads=None, window=None):
    """Gradients (dq, dk, dv) of sum(out * dout) for the forward above.

    In broadcast-Q mode dq is the sum over all sequences of the per-sequence
    dQ_b, as the TLX JFA page (section 1) describes; sampling with `seqs`
    then sums only the sampled sequences.  With GQA, dk / dv of a K/V head
    sum over the query heads of its group.  Entries of unsampled pairs are
    NaN in dk / dv (and in dq for self-attention).
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    off = _seq_bounds(offsets)
    B = off.size - 1
    T, Hkv, D = k.shape
    H, Hkv, group = _heads(q, k, broadcast_q)
    _check_mask_args(broadcast_q, causal, window)
    pairs = _pairs(B, H, seqs, heads, group)
    dk = np.full((T, Hkv, D), np.nan)
    dv = np.full((T, Hkv, D), np.nan)
    for b, h in pairs:
        s0, s1 = int(off[b]), int(off[b + 1])
        dk[s0:s1, h // group, :] = 0.0
        dv[s0:s1, h // group, :] = 0.0
    if broadcast_q:
        dq = np.zeros_like(q)
        if heads is not None:
            dq[:] = np.nan
            for h in sorted({h for _, h in pairs}):
                dq[:, h, :] = 0.0
    else:
        dq = np.full((T, H, D), np.nan)
    for b, h in pairs:
        s0, s1 = int(off[b]), int(off[b + 1])
        kb, vb = k[s0:s1, h // group, :], v[s0:s1, h // group, :]
        if broadcast_q:
            qb, dob = q[:, h, :], dout[b, :, h, :]
        else:
            qb, dob = q[s0:s1, h, :], dout[s0:s1, h, :]
        nq = qb.shape[0]
        dqb = np.zeros((nq, D))
        dkb = np.zeros((s1 - s0, D))
        dvb = np.zeros((s1 - s0, D))
        if s1 > s0:
            for r0 in range(0, nq, ROW_CHUNK):
                r1 = min(nq, r0 + ROW_CHUNK)
                s = _scores(qb[r0:r1], kb, scale, causal, r0, window)
                p = _probs(s, _lse_rows(s))
                dp = dob[r0:r1] @ vb.T
                ds = _grad_scores(p, dp)
                dqb[r0:r1] = scale * (ds @ kb)
                dkb += scale * (ds.T @ qb[r0:r1])
                dvb += p.T @ dob[r0:r1]
        if broadcast_q:
            dq[:, h, :] += dqb
        else:
            dq[s0:s1, h, :] = dqb
        dk[s0:s1, h // group, :] += dkb
        dv[s0:s1, h // group, :] += dvb
    return dq, dk, dv


def delta_rowsum(out, dout, broadcast_q=False):
    """Delta = rowsum(dO * O), the backward pre-pass quantity, in fp64.

    For the exact O of the forward this equals sum_j P_ij dP_ij (used by
    `backward`); layout is that of lse ([H, T], or [B, H, Lq] in broadcast).
    """
    o, do = _as64(out), _as64(dout)
    d = np.sum(o * do, axis=-1)
    return np.moveaxis(d, -1, -2) if broadcast_q else d.T.copy()


# ------------------------------------------------------- block-sparse variant
#
# "Optimizing Jagged Flash Attention with TLX", section 3 ("Block-sparse
# attention"): a scoring step average-pools each Q block and each K block,
# keeps per Q block the top-k K/V blocks (k from a selection ratio), and the
# attention then runs over the selected blocks only.  Readings where the page
# is silent (listed in the design notes): K blocks are 128 keys, Q blocks 256
# query rows, both counted from the start of their sequence (the last one
# ragged); a block's pooled vector is the mean of its valid rows, per head
# (K/V head h // group for query head h); the block score is the dot product
# of the two pooled vectors; k = max(1, ceil(permille * n / 1000)) of the
# sequence's n K blocks, in integer arithmetic; ties go to the lower block
# index; the list is stored in ascending order.  In broadcast-Q mode the Q
# blocks are the 256-row blocks of the one dense Q (the same for every
# sequence); a sequence without keys gets an empty list (O = 0, LSE =
# -inf).  With a causal mask or a window (self-attention), the candidates
# are the K blocks that hold an admissible key of some row of the Q block,
# k counts from them, and the attention keeps a key only when it is both
# in a listed block and in the row's band (a row can then be left with no
# key: O = 0, LSE = -inf).

SPARSE_Q_BLOCK = 256
SPARSE_K_BLOCK = 128


def _cdiv(a, b):
    return -(-a // b)


def sparse_k_count(n_blocks, permille):
    """Selected K blocks out of n: max(1, ceil(permille * n / 1000)), at most n."""
    if n_blocks == 0:
        return 0
    return min(n_blocks, max(1, (permille * n_blocks + 999) // 1000))


def block_select(q, k, offsets, permille, broadcast_q=False, causal=False, window=None):
    """Top-k K blocks per (sequence, query head, Q block) by pooled scores.

    Returns (blocks, counts, scores): blocks int64 [B, H, nqb, kcap] holding
    the selected K block indices in ascending order in the first counts
    entries (-1 after them), counts int64 [B, H, nqb], and the fp64 block
    scores [B, H, nqb, kcap] (NaN where there is no block), with nqb =
    ceil(max_len / 256) (broadcast: ceil(q_len / 256)) and kcap =
    ceil(max_len / 128).
    """
    q, k = _as64(q), _as64(k)
    off = _seq_bounds(offsets)
    B = off.size - 1
    H, Hkv, group = _heads(q, k, broadcast_q)
    _check_mask_args(broadcast_q, causal, window)
    wl, wr = _window(causal, window)
    L = np.diff(off)
    max_len = int(L.max()) if B else 0
    nqb = _cdiv(q.shape[0] if broadcast_q else max_len, SPARSE_Q_BLOCK)
    kcap = _cdiv(max_len, SPARSE_K_BLOCK)
    blocks = np.full((B, H, nqb, kcap), -1, dtype=np.int64)
    counts = np.zeros((B, H, nqb), dtype=np.int64)
    scores = np.full((B, H, nqb, kcap), np.nan)
    for b in range(B):
        s0, n = int(off[b]), int(L[b])
        nk = _cdiv(n, SPARSE_K_BLOCK)
        nq = nqb if broadcast_q else _cdiv(n, SPARSE_Q_BLOCK)
        if nk == 0:
            continue  # no keys: empty lists
        for h in range(H):
            kbar = np.stack([k[s0 + j * SPARSE_K_BLOCK: s0 + min(n, (j + 1) * SPARSE_K_BLOCK),
                               h // group, :].mean(axis=0) for j in range(nk)])
            for i in range(nq):
                if broadcast_q:
                    qbar = q[i * SPARSE_Q_BLOCK: min(q.shape[0], (i + 1) * SPARSE_Q_BLOCK), h, :]
                else:
                    qbar = q[s0 + i * SPARSE_Q_BLOCK: s0 + min(n, (i + 1) * SPARSE_Q_BLOCK), h, :]
                sc = kbar @ qbar.mean(axis=0)
                scores[b, h, i, :nk] = sc
                # candidates: K blocks holding an admissible key of a row of the Q block
                r0, r1 = i * SPARSE_Q_BLOCK, min(n, (i + 1) * SPARSE_Q_BLOCK) - 1
                lo = 0 if wl is None else max(0, r0 - wl)
                hi = n - 1 if wr is None else min(n - 1, r1 + wr)
                cand = np.arange(lo // SPARSE_K_BLOCK, hi // SPARSE_K_BLOCK + 1)
                kk = sparse_k_count(cand.size, permille)
                order = cand[np.argsort(-sc[cand], kind="stable")]  # descending, ties: lower first
                blocks[b, h, i, :kk] = np.sort(order[:kk])
                counts[b, h, i] = kk
    return blocks, counts, scores


def forward_sparse(q, k, v, offsets, scale, blocks, counts, broadcast_q=False, causal=False,
                   window=None):
    """Attention in which query row i of a sequence sees only the keys of the
    K blocks listed for its Q block (i // 256): blocks[b, h, i // 256,
    :counts[b, h, i // 256]].  A row with no key gets O = 0, LSE = -inf.
    Layouts as forward (self-attention, or broadcast-Q: row i of the dense
    Q, out [B, q_len, H, D], lse [B, H, q_len])."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    off = _seq_bounds(offsets)
    B = off.size - 1
    T, Hkv, D = k.shape
    H, Hkv, group = _heads(q, k, broadcast_q)
    _check_mask_args(broadcast_q, causal, window)
    if broadcast_q:
        Lq = q.shape[0]
        out = np.zeros((B, Lq, H, D))
        lse = np.full((B, H, Lq), -np.inf)
    else:
        out = np.zeros((T, H, D))
        lse = np.full((H, T), -np.inf)
    for b in range(B):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        kblock = np.arange(n) // SPARSE_K_BLOCK
        nrows = q.shape[0] if broadcast_q else n
        for h in range(H):
            kb, vb = k[s0:s1, h // group, :], v[s0:s1, h // group, :]
            for i in range(_cdiv(nrows, SPARSE_Q_BLOCK)):
                r0, r1 = i * SPARSE_Q_BLOCK, min(nrows, (i + 1) * SPARSE_Q_BLOCK)
                keep = np.isin(kblock, blocks[b, h, i, :counts[b, h, i]])
                qrows = q[r0:r1, h, :] if broadcast_q else q[s0 + r0:s0 + r1, h, :]
                s = _scores(qrows, kb, scale, causal, r0, window)  # the band, if any
                s = np.where(keep[None, :], s, -np.inf)
                l = _lse_rows(s)
                if broadcast_q:
                    out[b, r0:r1, h, :] = _probs(s, l) @ vb
                    lse[b, h, r0:r1] = l
                else:
                    out[s0 + r0:s0 + r1, h, :] = _probs(s, l) @ vb
                    lse[h, s0 + r0:s0 + r1] = l
    return out, lse
