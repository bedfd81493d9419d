"""fp64 CPU oracle for sparse MLA (DSA) attention with a per-head sink.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The library never calls
it, and it shares no code with the CUDA path.

This is the plain definition written out in float64.  Each token is handled
on its own and each step is one numpy expression: a library matmul, an
elementwise exp, a row sum.  There is no tiling, no online softmax and no
fusion.  Sources, cited by page title and section:

[P2] cuDNN frontend, "DSA backward SM90: fix three top-k and attention-sink
     boundary failures":
     Summary 1-3 (empty rows, padded columns, saturating sink), Why 1-3,
     "Not addressed" (delta = rowsum(O * dO); S*scale - lse <= 0 on live
     columns) and the Testing bullets (positive saturating sink gives
     dq = dkv = 0 and d_sink = -sum(dP_sum)).
[P3] flash-attention, "[CuTe, SM100] Support 1..128 Q heads in sparse MLA
     via in-kernel TMA padding": Agent Notes (one token, one top-k gather
     list; padded heads contribute nothing) and "Performance at DeepSeek-V4
     shapes" (shared KV; FLOP accounting).
[P4] cuDNN frontend, "DSA bwd SM100 fix dropped dKV gradients when topk width
     > total_S_kv": a column position >= S_kv is not invalid, and validity
     comes from the index value and the top-k bound.
[P1] NeMo Automodel PR 3467 (TileLang sparse-MLA backward fix): ValidMask is
     (idx >= 0) & (idx < S_kv).

Readings where the pages are silent:

* The LSE excludes the sink.  The backward folds the sink in through
  sigma(LSE - sink) [P2 Summary 3, Why 3].
* The sink is a natural-log logit per head and is not multiplied by ``scale``.
  A missing sink is sink = -inf.
* An empty row (no valid slot) has out = 0, LSE = -FLT_MAX (a finite
  stand-in for -inf), zero dq and no dkv contribution [P2 Summary 1].
* topk_length <= 0 gives an empty row; topk_length > W is clamped to W.
* A duplicate index is counted once per slot: each slot is its own softmax
  term and its own dkv contribution, which is what a gather computes.
* The backward's delta uses the output the caller hands in when ``out`` is
  given.  Otherwise it uses the oracle's own fp64 O.
* Varlen batches [P2 Why 1 reads topk_length per (batch, position)]: the
  sequences are packed along T and along the KV rows; each sequence is the
  single-sequence definition on its own slices, with its indices counted
  from its own first KV row.  The sink is shared by all sequences.
"""
from __future__ import annotations

import numpy as np

FLT_MAX = float(np.finfo(np.float32).max)
EMPTY_LSE = -FLT_MAX


def _np64(x):
    """Widen a torch tensor or array to a float64 numpy array (exact for bf16)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if x.dtype.is_floating_point:
            x = x.double()
        return x.numpy()
    return np.asarray(x)


def _np_int(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x).astype(np.int64)


def valid_slots(idx_row: np.ndarray, length, S_kv: int) -> np.ndarray:
    """Positions j of the valid slots of one token, in slot order.

    A slot j is valid iff 0 <= idx[j] < S_kv and, when a length is given,
    j < length [P1 ValidMask; P2 Why 2; P4].  The column position itself is
    never compared with S_kv [P4].
    """
    W = idx_row.shape[0]
    j = np.arange(W)
    ok = (idx_row >= 0) & (idx_row < S_kv)
    if length is not None:
        n = int(min(max(int(length), 0), W))
        ok &= j < n
    return j[ok]


def sigmoid(x):
    """Logistic function evaluated without overflow for any x, incl. +-inf."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def _sink64(sink, H):
    if sink is None:
        return np.full(H, -np.inf)
    return _np64(sink).astype(np.float64).reshape(H)


def token_forward(qt, kv, idx_row, length, sink, scale, d_v):
    """One token's forward with every head at once, all in fp64.

    Returns (sel, S, lse, g, P, O).  ``sel`` holds the KV rows of the valid
    slots.  S = scale * q . kv[sel] has shape [H, K].  ``lse`` is log sum_j
    exp(S_j) [H].  g = sigma(lse - sink) is the attention share; the sink
    takes 1 - g.  P_j = exp(S_j - lse) * g [H, K] and O = P . V [H, d_v].
    For an empty row, S and P are [H, 0], lse = EMPTY_LSE and O = 0.
    """
    H = qt.shape[0]
    S_kv = kv.shape[0]
    j = valid_slots(idx_row, length, S_kv)
    sel = idx_row[j]
    if sel.size == 0:
        return sel, np.zeros((H, 0)), np.full(H, EMPTY_LSE), np.zeros(H), \
            np.zeros((H, 0)), np.zeros((H, d_v))
    kvs = kv[sel]                                  # [K, D]
    S = scale * (qt @ kvs.T)                       # [H, K]
    m = S.max(axis=1)
    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
    g = sigmoid(lse - sink)
    P = np.exp(S - lse[:, None]) * g[:, None]
    O = P @ kvs[:, :d_v]
    return sel, S, lse, g, P, O


def forward(q, kv, topk_idxs, topk_length, sink, scale, d_v=512, tokens=None):
    """Sparse attention forward with a sink in the softmax denominator.

    For each token t and head h [P3 Agent Notes; P2 Summary 2-3]:
      s_j  = scale * q[t,h,:] . kv[idx_j, :]      (j over valid slots)
      lse  = log sum_j exp(s_j)                   (the sink is left out)
      out  = sum_j exp(s_j) / (sum_j exp(s_j) + exp(sink_h)) * kv[idx_j, :d_v]
    Returns a dict of fp64 arrays: out [T,H,d_v], lse [T,H] and the valid-slot
    count [T].  With ``tokens`` given, only those rows are filled; the other
    rows are NaN.
    """
    kv = _np64(kv)
    idx = _np_int(topk_idxs)
    length = _np_int(topk_length)
    T, H, _ = q.shape
    sk = _sink64(sink, H)
    toks = range(T) if tokens is None else tokens
    out = np.full((T, H, d_v), np.nan)
    lse = np.full((T, H), np.nan)
    count = np.full(T, -1, dtype=np.int64)
    for t in toks:
        sel, S, l, g, P, O = token_forward(_np64(q[t]), kv, idx[t],
                                           None if length is None else length[t], sk, scale, d_v)
        out[t] = O
        lse[t] = l
        count[t] = sel.size
    return {"out": out, "lse": lse, "count": count}


def token_backward(qt, kv, sel, P, lse, dout_t, O_use, sink, scale, d_v):
    """One token's backward, every head at once, in fp64.

    Returns (dq_t [H, D], contrib [K, D] to add into dkv[sel], dsink_t [H],
    delta [H]).  In an empty row the sink holds the whole denominator
    (p_sink = 1), dq is 0 and nothing goes to dkv [P2 Summary 1].
    """
    H, D = qt.shape
    delta = (dout_t * O_use).sum(axis=1)                 # rowsum(dO * O)
    if sel.size == 0:
        return np.zeros((H, D)), np.zeros((0, D)), -np.ones(H) * delta, delta
    p_sink = sigmoid(sink - lse)                         # = 1 - g
    kvs = kv[sel]
    dP = dout_t @ kvs[:, :d_v].T                         # [H, K]
    dS = P * (dP - delta[:, None])                       # [H, K]
    dq_t = scale * (dS @ kvs)                            # [H, D]
    contrib = scale * (dS.T @ qt)                        # [K, D]
    contrib[:, :d_v] += P.T @ dout_t
    return dq_t, contrib, -p_sink * delta, delta


def backward(q, kv, topk_idxs, topk_length, sink, scale, dout, d_v=512, out=None,
             tokens=None):
    """Gradients of the loss sum(dout * out) [P2 Not addressed; P2 Testing].

      delta  = sum_d dout[t,h,d] * O[t,h,d]   (O from ``out`` if given)
      dP_j   = dout[t,h,:] . kv[idx_j, :d_v]
      dS_j   = P_j * (dP_j - delta)
      dq     = scale * sum_j dS_j * kv[idx_j, :]
      dkv[r] = sum over (t,h,j) with idx_j = r of scale*dS_j*q[t,h,:] + P_j*[dout[t,h,:], 0]
      dsink  = -sum_t p_sink * delta,  p_sink = sigma(sink - lse) = 1 - g
    With ``tokens`` given, only those tokens contribute.  dq rows of other
    tokens are NaN, and dkv and dsink are the partial sums over ``tokens``.
    """
    kv = _np64(kv)
    idx = _np_int(topk_idxs)
    length = _np_int(topk_length)
    T, H, D = q.shape
    sk = _sink64(sink, H)
    toks = range(T) if tokens is None else tokens
    dq = np.full((T, H, D), np.nan)
    dkv = np.zeros(kv.shape)
    dsink = np.zeros(H)
    delta_all = np.full((T, H), np.nan)
    for t in toks:
        qt = _np64(q[t])
        sel, S, lse, g, P, O = token_forward(qt, kv, idx[t], None if length is None else length[t],
                                             sk, scale, d_v)
        Ouse = O if out is None else _np64(out[t])
        dq_t, contrib, dsink_t, delta = token_backward(qt, kv, sel, P, lse, _np64(dout[t]), Ouse, sk,
                                                       scale, d_v)
        delta_all[t] = delta
        dq[t] = dq_t
        if sel.size:
            np.add.at(dkv, sel, contrib)
        dsink += dsink_t
    return {"dq": dq, "dkv": dkv, "dsink": dsink, "delta": delta_all}


def _sequences(cu_seqlens_q, cu_seqlens_kv):
    cq, ck = _np_int(cu_seqlens_q), _np_int(cu_seqlens_kv)
    return [(int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])) for b in range(cq.size - 1)]


def forward_varlen(q, kv, topk_idxs, topk_length, sink, scale, cu_seqlens_q, cu_seqlens_kv,
                   d_v=512):
    """A varlen batch: sequence b is tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
    with KV rows cu_seqlens_kv[b] .. cu_seqlens_kv[b+1]-1, and its indices count
    from its own first row.  Each sequence is ``forward`` on its slices."""
    T, H, _ = q.shape
    out = np.full((T, H, d_v), np.nan)
    lse = np.full((T, H), np.nan)
    count = np.full(T, -1, dtype=np.int64)
    length = _np_int(topk_length)
    for t0, t1, r0, r1 in _sequences(cu_seqlens_q, cu_seqlens_kv):
        if t1 == t0:
            continue
        ref = forward(q[t0:t1], _np64(kv)[r0:r1], _np_int(topk_idxs)[t0:t1],
                      None if length is None else length[t0:t1], sink, scale, d_v)
        out[t0:t1], lse[t0:t1], count[t0:t1] = ref["out"], ref["lse"], ref["count"]
    return {"out": out, "lse": lse, "count": count}


def backward_varlen(q, kv, topk_idxs, topk_length, sink, scale, dout, cu_seqlens_q,
                    cu_seqlens_kv, d_v=512, out=None):
    """Gradients of a varlen batch: ``backward`` per sequence; dkv rows of a
    sequence receive only its own tokens' contributions, and dsink sums over
    all sequences."""
    T, H, D = q.shape
    kv64 = _np64(kv)
    dq = np.full((T, H, D), np.nan)
    dkv = np.zeros(kv64.shape)
    dsink = np.zeros(H)
    length = _np_int(topk_length)
    for t0, t1, r0, r1 in _sequences(cu_seqlens_q, cu_seqlens_kv):
        if t1 == t0:
            continue
        g = backward(q[t0:t1], kv64[r0:r1], _np_int(topk_idxs)[t0:t1],
                     None if length is None else length[t0:t1], sink, scale, dout[t0:t1], d_v,
                     out=None if out is None else out[t0:t1])
        dq[t0:t1] = g["dq"]
        dkv[r0:r1] += g["dkv"]
        dsink += g["dsink"]
    return {"dq": dq, "dkv": dkv, "dsink": dsink}


def tokens_referencing(topk_idxs, topk_length, S_kv, rows):
    """Tokens with at least one valid slot whose index is in ``rows``."""
    idx = _np_int(topk_idxs)
    length = _np_int(topk_length)
    T, W = idx.shape
    valid = (idx >= 0) & (idx < S_kv)
    if length is not None:
        n = np.clip(length, 0, W)
        valid &= np.arange(W)[None, :] < n[:, None]
    hit = valid & np.isin(idx, np.asarray(list(rows)))
    return np.nonzero(hit.any(axis=1))[0]


def valid_lists(topk_idxs, topk_length, S_kv):
    """Per token: the valid KV rows in slot order, and their count."""
    idx = _np_int(topk_idxs)
    length = _np_int(topk_length)
    T, W = idx.shape
    lists = []
    for t in range(T):
        j = valid_slots(idx[t], None if length is None else length[t], S_kv)
        lists.append(idx[t][j])
    return lists, np.array([len(x) for x in lists], dtype=np.int64)


def flops_forward(H, counts, d_qk=576, d_v=512):
    """Forward FLOPs with K = valid gathered slots: 2 * H * sum_t K_t * (d_qk + d_v)
    [P3 "Performance at DeepSeek-V4 shapes"]."""
    return 2.0 * H * float(np.sum(counts)) * (d_qk + d_v)
