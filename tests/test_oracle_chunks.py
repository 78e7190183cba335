"""Pins for the oracle's query-row chunking.  CPU only.

The oracle splits the query rows of each (sequence, head) into blocks of
ROW_CHUNK rows so that long sequences fit in memory.  Three things happen
only when a sequence is longer than one block: blocks that start at a row
r0 > 0, the causal offset that the score block receives for them (query i of
the block is row r0 + i of the sequence: "cuTile Kernels - FMHA
Implementation", "Attention Basics", future keys masked), and dK / dV summed
over the blocks.  Here ROW_CHUNK is made small (3 and 7 rows) so that every
sequence spans several blocks, and the results are checked against the
padded torch float64 SDPA + autograd route and against stacked per-sequence
attention for broadcast-Q, both written without the oracle.  Planted slips in
exactly those three places must be caught.
"""
import importlib.util
import inspect
import sys

import numpy as np
import pytest
import torch

from oracle import jfa_oracle
from tests.test_oracle_pins import _bq_case, _self_case, _torch_padded_self

LENGTHS = [1, 17, 5, 33, 2, 64, 8]


def _check_self(mod, causal, chunk, monkeypatch):
    monkeypatch.setattr(mod, "ROW_CHUNK", chunk)
    H, D, scale = 2, 8, 0.3
    q, k, v, do, off = _self_case(LENGTHS, H, D, seed=31)
    out, lse = mod.forward(q, k, v, off, scale, causal)
    dq, dk, dv = mod.backward(q, k, v, off, do, scale, causal)
    O, dQ, dK, dV = _torch_padded_self(q, k, v, do, off, scale, causal)
    np.testing.assert_allclose(out, O, atol=1e-12)
    np.testing.assert_allclose(dq, dQ, atol=1e-11)
    np.testing.assert_allclose(dk, dK, atol=1e-11)
    np.testing.assert_allclose(dv, dV, atol=1e-11)
    # LSE by a direct log-sum-exp of the masked scores of each row
    for b in range(len(LENGTHS)):
        s0, s1 = off[b], off[b + 1]
        for h in range(H):
            s = scale * q[s0:s1, h] @ k[s0:s1, h].T
            if causal:
                s = np.where(np.triu(np.ones_like(s, dtype=bool), 1), -np.inf, s)
            ref = torch.logsumexp(torch.from_numpy(s), -1).numpy()
            np.testing.assert_allclose(lse[h, s0:s1], ref, atol=1e-12)


def _check_broadcast(mod, chunk, monkeypatch):
    monkeypatch.setattr(mod, "ROW_CHUNK", chunk)
    H, D, scale, Lq = 2, 8, 0.35, 20
    lengths = [3, 0, 9, 1, 4]
    q, k, v, do, off = _bq_case(lengths, Lq, H, D, seed=32)
    out, lse = mod.forward(q, k, v, off, scale, broadcast_q=True)
    dq, dk, dv = mod.backward(q, k, v, off, do, scale, broadcast_q=True)
    dq_sum = np.zeros_like(q)
    for b, n in enumerate(lengths):
        s0, s1 = off[b], off[b + 1]
        if n == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
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


@pytest.mark.parametrize("chunk", [3, 7])
@pytest.mark.parametrize("causal", [False, True])
def test_chunked_self_matches_padded_torch(monkeypatch, causal, chunk):
    assert max(LENGTHS) > 4 * chunk  # every long sequence spans several blocks
    _check_self(jfa_oracle, causal, chunk, monkeypatch)


@pytest.mark.parametrize("chunk", [3, 7])
def test_chunked_broadcast_matches_stacked_torch(monkeypatch, chunk):
    _check_broadcast(jfa_oracle, chunk, monkeypatch)


def test_chunking_does_not_change_results(monkeypatch):
    """Same inputs, ROW_CHUNK 7 against one block per sequence: identical up
    to rounding order."""
    H, D, scale = 2, 8, 0.3
    q, k, v, do, off = _self_case(LENGTHS, H, D, seed=33)
    full = [jfa_oracle.forward(q, k, v, off, scale, True)[0],
            *jfa_oracle.backward(q, k, v, off, do, scale, True)]
    monkeypatch.setattr(jfa_oracle, "ROW_CHUNK", 7)
    part = [jfa_oracle.forward(q, k, v, off, scale, True)[0],
            *jfa_oracle.backward(q, k, v, off, do, scale, True)]
    for a, b in zip(full, part):
        np.testing.assert_allclose(b, a, atol=1e-13)


# -------------------------------------------- planted mistakes are caught

def _mutant_module(replace_from, replace_to):
    """A copy of the oracle module with one textual slip planted."""
    src = inspect.getsource(jfa_oracle)
    if replace_from not in src:  # a stale slip must not pass as a caught one
        raise LookupError(replace_from)
    src = src.replace(replace_from, replace_to)
    spec = importlib.util.spec_from_loader("jfa_oracle_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src, "jfa_oracle_mutant", "exec"), mod.__dict__)
    sys.modules.pop("jfa_oracle_mutant", None)
    return mod


def test_planted_row0_slip_is_caught(monkeypatch):
    """Score blocks always told they start at row 0 (the causal offset lost)."""
    orig = jfa_oracle._scores

    def mutant(qc, kb, scale, causal, row0, window=None):
        return orig(qc, kb, scale, causal, 0, window)
    monkeypatch.setattr(jfa_oracle, "_scores", mutant)
    with pytest.raises(AssertionError):
        _check_self(jfa_oracle, True, 7, monkeypatch)


@pytest.mark.parametrize("slip", [("dkb += ", "dkb = "), ("dvb += ", "dvb = ")])
def test_planted_overwrite_of_block_sums_is_caught(monkeypatch, slip):
    """dK or dV of a sequence overwritten by each block instead of summed."""
    mod = _mutant_module(*slip)
    with pytest.raises(AssertionError):
        _check_self(mod, False, 7, monkeypatch)
    with pytest.raises(AssertionError):
        _check_broadcast(mod, 7, monkeypatch)


def test_planted_chunk_start_slip_is_caught(monkeypatch):
    """Every block's rows taken from the start of the sequence."""
    mod = _mutant_module("qb[r0:r1]", "qb[0:r1 - r0]")
    with pytest.raises(AssertionError):
        _check_self(mod, False, 7, monkeypatch)


def test_unmutated_copy_passes(monkeypatch):
    """The textual copy itself (no slip) passes, so the mutants above fail
    because of their slip and not because of the copying."""
    mod = _mutant_module("ROW_CHUNK = 1024", "ROW_CHUNK = 1024")
    _check_self(mod, True, 7, monkeypatch)
    _check_broadcast(mod, 7, monkeypatch)
