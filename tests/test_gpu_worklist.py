"""The device work lists, checked against a host re-derivation.

The schedulers ("Optimizing Jagged Flash Attention with TLX", section 2.2,
"Scheduling jagged tiles across SMs": only valid tiles become work, the
longest first) run on the GPU through jfa_worklist, which builds a list
exactly as its pass does and copies it out.  For every list: each expected
(sequence, head, tile) item appears exactly once and nothing else does, the
item count equals the count formula, and the cost of the items never
increases along the list (self-attention forward / dQ pass: key tiles of the
sequence; dK/dV pass: query tiles of the sequence; broadcast: all equal).
The causal forward takes each sequence's last query tile first.  The
broadcast dQ-pass list must cut the key-tile stream of every (head,
query-tile pair) into equal chunks that cover each key tile once.
"""
import collections
import math

import numpy as np
import pytest
import torch

import jfa_workloads as W

pytestmark = pytest.mark.gpu

FWD, KV, SELF_Q, BCAST_Q = 0, 1, 2, 3


def _cdiv(a, b):
    return -(-a // b)


def _run(lengths, H, which, causal=False, q_len=0):
    import jagged_flash_attention_gb300 as jfa
    L = np.asarray(lengths, dtype=np.int64)
    bq = q_len > 0
    dev = torch.device("cuda")
    off = torch.from_numpy(W.offsets_from_lengths(L)).to(dev)
    B, max_len = len(L), int(L.max())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cap = H * B * _cdiv(max_len, 128) + 4 * sms * max(1, _cdiv(q_len, 256)) + 16
    items = torch.full((cap, 4), -7, dtype=torch.int32, device=dev)
    count = torch.zeros(2, dtype=torch.int32, device=dev)
    jfa.jfa_worklist(off, B, H, max_len, q_len, bq, causal, which, items, cap, count)
    jfa.jfa_sync_and_check()
    n, nc = (int(v) for v in count.cpu())
    assert n >= 0, "device reported invalid offsets"
    return items[:n].cpu().numpy(), nc, sms


def _bucket(L, per):
    return min(_cdiv(int(L), per), 1023)


@pytest.mark.parametrize("case", ["jagged_self", "causal_self", "tiny_self", "many_short"])
def test_self_lists(case):
    if case == "many_short":  # several scheduler chunks, many equal buckets
        L, H, causal = np.random.default_rng(5).integers(1, 300, size=5000), 2, False
    else:
        w = W.WORKLOADS[case]
        L, H, causal = W.sample_lengths(w), w.H, w.causal
    for which, per_item in ((FWD, 256), (KV, 128), (SELF_Q, 256)):
        items, _, _ = _run(L, H, which, causal=causal)
        expect = collections.Counter(
            (b, h, t) for b in range(len(L)) for h in range(H)
            for t in range(_cdiv(int(L[b]), per_item)))
        got = collections.Counter(map(tuple, items[:, :3].tolist()))
        assert got == expect, (which, len(got), len(expect))
        assert len(items) == sum(H * _cdiv(int(l), per_item) for l in L)
        assert np.all(items[:, 3] == 0)
        cost = np.array([_bucket(L[b], 128) for b in items[:, 0]])
        assert np.all(np.diff(cost) <= 0), which
        if which == FWD and causal:
            # longest query tile of each (sequence, head) first
            last = {}
            for b, h, t in items[:, :3].tolist():
                if (b, h) in last:
                    assert t < last[(b, h)]
                last[(b, h)] = t


@pytest.mark.parametrize("case", ["broadcast_q", "skewed_broadcast_q", "with_empty"])
def test_broadcast_lists(case):
    if case == "with_empty":
        L, H, q_len = np.array([0, 5, 0, 0, 300, 1, 128, 129, 0, 4000]), 3, 300
    else:
        w = W.WORKLOADS[case]
        L, H, q_len = W.sample_lengths(w), w.H, w.q_len
    B = len(L)
    # forward: every sequence, even an empty one, owns its output rows
    items, _, _ = _run(L, H, FWD, q_len=q_len)
    expect = collections.Counter((b, h, t) for b in range(B) for h in range(H)
                                 for t in range(_cdiv(q_len, 256)))
    assert collections.Counter(map(tuple, items[:, :3].tolist())) == expect
    cost = np.array([_bucket(L[b], 128) for b in items[:, 0]])
    assert np.all(np.diff(cost) <= 0)
    # dK/dV pass: key blocks of non-empty sequences, all of equal cost
    items, _, _ = _run(L, H, KV, q_len=q_len)
    expect = collections.Counter((b, h, t) for b in range(B) for h in range(H)
                                 for t in range(_cdiv(int(L[b]), 128)))
    assert collections.Counter(map(tuple, items[:, :3].tolist())) == expect
    # heads outermost over the whole list (consecutive items share the dense Q)
    assert np.all(np.diff(items[:, 1]) >= 0)
    # dQ pass: equal chunks of the key-tile stream of every (head, pair)
    items, nc, sms = _run(L, H, BCAST_Q, q_len=q_len)
    pairs = _cdiv(q_len, 256)
    nt = [_cdiv(int(l), 128) for l in L]
    total = sum(nt)
    assert nc == min(max(1, _cdiv(2 * sms, H * pairs)), _cdiv(total, 4))
    assert len(items) == nc * H * pairs
    stream = [(b, j) for b in range(B) for j in range(nt[b])]
    covered = collections.defaultdict(list)
    for idx, (hp, b, j, n) in enumerate(items.tolist()):
        c, rem = divmod(idx, H * pairs)
        h, pair = divmod(rem, pairs)
        assert hp == h | (pair << 16)
        s0, s1 = c * total // nc, (c + 1) * total // nc
        assert n == s1 - s0 and n >= 1
        assert stream[s0] == (b, j)  # the chunk starts where the stream says
        covered[(h, pair)].extend(stream[s0:s1])
    for h in range(H):
        for pair in range(pairs):
            assert covered[(h, pair)] == stream
