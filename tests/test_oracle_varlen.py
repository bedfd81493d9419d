"""Pins for the oracle's varlen batches (CPU).

The varlen oracle applies the single-sequence definition to each packed
sequence.  These tests check it against a different route to the same
numbers: the plain single-sequence oracle run on the whole packed problem
after each token's relative indices have been turned into absolute KV rows
(and indices invalid for their own sequence into -1).  A wrong offset, a
missing per-sequence bound or a dkv row credited to the wrong sequence fails
here.
"""
import numpy as np
import torch

from oracle import dsa_oracle as O
from sparse_top_attention_gb300 import workloads as WL

LENGTHS = [40, 0, 70, 9]


def _with_out_of_sequence_indices(w):
    """Plant indices that are valid in the packed KV but not in their own
    sequence (>= that sequence's row count): they must be masked."""
    idx = w.topk_idxs.clone()
    cq, ck = w.cu_seqlens_q.tolist(), w.cu_seqlens_kv.tolist()
    for b in range(len(cq) - 1):
        n_rows = ck[b + 1] - ck[b]
        for t in range(cq[b], cq[b + 1], 7):
            idx[t, -1] = n_rows + 2      # beyond this sequence, inside the packed KV
            idx[t, -2] = n_rows          # the first row past the sequence
    w.topk_idxs = idx
    return w


def _absolute(w):
    """Relative indices -> absolute rows; invalid slots -> -1."""
    idx = w.topk_idxs.numpy().astype(np.int64)
    out = np.full_like(idx, -1)
    length = None if w.topk_length is None else w.topk_length.numpy()
    cq, ck = w.cu_seqlens_q.tolist(), w.cu_seqlens_kv.tolist()
    W = idx.shape[1]
    for b in range(len(cq) - 1):
        n_rows = ck[b + 1] - ck[b]
        for t in range(cq[b], cq[b + 1]):
            ln = W if length is None else min(max(int(length[t]), 0), W)
            for j in range(W):
                v = idx[t, j]
                if j < ln and 0 <= v < n_rows:
                    out[t, j] = ck[b] + v
    return torch.from_numpy(out.astype(np.int32))


def _both(w):
    fv = O.forward_varlen(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale,
                          w.cu_seqlens_q, w.cu_seqlens_kv)
    gv = O.backward_varlen(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale, w.dout,
                           w.cu_seqlens_q, w.cu_seqlens_kv)
    absidx = _absolute(w)
    # the absolute encoding is non-compact: the -1 entries carry the masking
    fp = O.forward(w.q, w.kv, absidx, None, w.sink, w.scale)
    gp = O.backward(w.q, w.kv, absidx, None, w.sink, w.scale, w.dout)
    return fv, gv, fp, gp


def test_varlen_equals_packed_absolute_rows():
    for compact in (False, True):
        w = _with_out_of_sequence_indices(WL.varlen(LENGTHS, H=4, topk=16, compact=compact, seed=5))
        fv, gv, fp, gp = _both(w)
        np.testing.assert_allclose(fv["out"], fp["out"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fv["lse"], fp["lse"], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(fv["count"], fp["count"])
        for k in ("dq", "dkv", "dsink"):
            np.testing.assert_allclose(gv[k], gp[k], rtol=1e-11, atol=1e-13)


def test_varlen_sequences_are_independent():
    w = WL.varlen(LENGTHS, H=4, topk=16, compact=False, seed=6)
    base_f = O.forward_varlen(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale,
                              w.cu_seqlens_q, w.cu_seqlens_kv)
    base_g = O.backward_varlen(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, w.dout,
                               w.cu_seqlens_q, w.cu_seqlens_kv)
    cq, ck = w.cu_seqlens_q.tolist(), w.cu_seqlens_kv.tolist()
    q2 = w.q.clone()
    q2[cq[2]:cq[3]] = -q2[cq[2]:cq[3]]            # change sequence 2 only
    f2 = O.forward_varlen(q2, w.kv, w.topk_idxs, None, w.sink, w.scale,
                          w.cu_seqlens_q, w.cu_seqlens_kv)
    g2 = O.backward_varlen(q2, w.kv, w.topk_idxs, None, w.sink, w.scale, w.dout,
                           w.cu_seqlens_q, w.cu_seqlens_kv)
    np.testing.assert_array_equal(f2["out"][:cq[2]], base_f["out"][:cq[2]])
    np.testing.assert_array_equal(g2["dkv"][:ck[2]], base_g["dkv"][:ck[2]])
    np.testing.assert_array_equal(g2["dkv"][ck[3]:], base_g["dkv"][ck[3]:])
    assert not np.allclose(g2["dkv"][ck[2]:ck[3]], base_g["dkv"][ck[2]:ck[3]])


def test_single_sequence_batch_is_the_plain_oracle():
    w = WL.varlen([57], H=4, topk=16, compact=False, seed=8)
    fv = O.forward_varlen(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale,
                          w.cu_seqlens_q, w.cu_seqlens_kv)
    fp = O.forward(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale)
    np.testing.assert_array_equal(fv["out"], fp["out"])
    np.testing.assert_array_equal(fv["lse"], fp["lse"])


def test_planted_varlen_mistakes_are_caught(monkeypatch):
    """Two plausible mistakes planted in the oracle (on the CPU) must each
    fail the packed-rows pin: relative indices read as absolute rows, and a
    sequence's dkv credited to the wrong rows."""
    import pytest
    orig_f, orig_b = O.forward_varlen, O.backward_varlen

    def absolute_rows(q, kv, idx, ln, sink, scale, cq, ck, d_v=512):
        return O.forward(q, kv, idx, ln, sink, scale, d_v)

    monkeypatch.setattr(O, "forward_varlen", absolute_rows)
    with pytest.raises(AssertionError):
        test_varlen_equals_packed_absolute_rows()
    monkeypatch.setattr(O, "forward_varlen", orig_f)

    def shifted_dkv(*a, **k):
        g = orig_b(*a, **k)
        g["dkv"] = np.roll(g["dkv"], 1, axis=0)
        return g

    monkeypatch.setattr(O, "backward_varlen", shifted_dkv)
    with pytest.raises(AssertionError):
        test_varlen_equals_packed_absolute_rows()
