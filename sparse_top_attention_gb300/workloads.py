"""Seeded synthetic inputs for sparse MLA (DSA) forward and backward.

This module only draws random numbers and lays out index tensors.  It holds
none of the attention arithmetic, so the CUDA path, the fp64 oracle, the tests
and the benchmark can all use it.

Workload shapes follow the DeepSeek-V4 measurement setup described on the
flash-attention page "[CuTe, SM100] Support 1..128 Q heads in sparse MLA via
in-kernel TMA padding" (section "Performance at DeepSeek-V4 shapes"): batch 1,
one KV tensor shared by every head, a sliding window of the 128 most recent
rows followed by a compressed causal top-k (512 for "flash", 1024 for "pro").
Rows are 576 wide (512 + 64) and the first 512 columns are V.

Encodings follow the cuDNN page "DSA backward SM90: fix three top-k and
attention-sink boundary failures" (Summary, items 1-2, and Why, item 2):
compact rows pack the valid entries to the left and carry ``topk_length``;
non-compact rows carry no length and mark unused slots with -1.

Every tensor is built on the host from a fixed seed.  ``make`` can then move
the result to a device, so that both sides of a parity test see identical
bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

D_QK = 576
D_V = 512
INT32_MIN = -(2 ** 31)
INT32_MAX = 2 ** 31 - 1
FLT_MAX = float(np.finfo(np.float32).max)

# Sink values that the edge-case workload cycles through per head.  Values of
# magnitude above 3.4e38 / log2(e) ~= 2.36e38 overflow once multiplied by
# log2(e) (cuDNN page, Summary item 3).
EDGE_SINKS = (None, 1e38, -1e38, 2.4e38, -2.4e38, FLT_MAX, -FLT_MAX)


@dataclass
class Workload:
    """One seeded problem instance (host tensors unless moved with ``to``)."""

    name: str
    q: torch.Tensor            # [T, H, 576] bf16
    kv: torch.Tensor           # [S_kv, 576] bf16
    topk_idxs: torch.Tensor    # [T, W] int32
    topk_length: Optional[torch.Tensor]  # [T] int32 or None
    sink: Optional[torch.Tensor]         # [H] fp32 or None
    dout: torch.Tensor         # [T, H, 512] bf16
    scale: float
    meta: dict = field(default_factory=dict)
    # A varlen batch: int32 [B + 1] token and KV-row offsets, else None.
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_kv: Optional[torch.Tensor] = None

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def S_kv(self) -> int:
        return int(self.kv.shape[0])

    @property
    def W(self) -> int:
        return int(self.topk_idxs.shape[1])

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        return Workload(self.name, mv(self.q), mv(self.kv), mv(self.topk_idxs),
                        mv(self.topk_length), mv(self.sink), mv(self.dout),
                        self.scale, dict(self.meta), mv(self.cu_seqlens_q),
                        mv(self.cu_seqlens_kv))


def _randn_bf16(gen: torch.Generator, shape, shift: float = 0.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    if shift:
        x += shift
    return x.to(torch.bfloat16)


def _window_and_compressed(T: int, topk: int, rng: np.random.Generator):
    """Per-token slot lists for the DeepSeek-V4 layout.

    Returns ``idx`` [T, 128 + topk] int32 in non-compact form: slots 0..127
    hold the window rows t-127..t (-1 where negative); the next ``topk`` slots
    hold ``T + c`` for min(topk, (t+1)//4) distinct compressed rows c with
    4c + 3 <= t, drawn uniformly without replacement, then -1 padding.
    """
    W = 128 + topk
    idx = np.full((T, W), -1, dtype=np.int64)
    t = np.arange(T)[:, None]
    win = t - 127 + np.arange(128)[None, :]
    idx[:, :128] = np.where(win >= 0, win, -1)
    n_avail = (np.arange(T) + 1) // 4           # number of c with 4c+3 <= t
    # Draw without replacement by ranking random keys; process in row chunks so
    # that the key matrix stays small.
    n_c_total = T // 4
    chunk = max(1, (1 << 24) // max(n_c_total, 1))
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        keys = rng.random((t1 - t0, n_c_total))
        cols = np.arange(n_c_total)[None, :]
        keys = np.where(cols < n_avail[t0:t1, None], keys, np.inf)
        k = min(topk, n_c_total)
        if k == 0:
            continue
        part = np.argpartition(keys, kth=k - 1, axis=1)[:, :k]
        pk = np.take_along_axis(keys, part, axis=1)
        order = np.argsort(pk, axis=1, kind="stable")
        part = np.take_along_axis(part, order, axis=1)
        pk = np.take_along_axis(pk, order, axis=1)
        sel = np.where(np.isfinite(pk), part + T, -1)
        idx[t0:t1, 128:128 + k] = sel
    return idx


def _compact(idx: np.ndarray, S_kv: int):
    """Pack the valid entries of each row to the left; return (idx, length)."""
    T, W = idx.shape
    valid = (idx >= 0) & (idx < S_kv)
    out = np.full_like(idx, -1)
    length = valid.sum(axis=1)
    for t in range(T):
        v = idx[t][valid[t]]
        out[t, :len(v)] = v
    return out, length


def dsv4(T: int, H: int, topk: int, compact: bool, seed: int, name: str,
         value_device: str = "cpu", d_qk: int = D_QK) -> Workload:
    """DeepSeek-V4-like layout: KV = T original rows + T/4 compressed rows.

    ``value_device`` chooses where q, kv, dout and sink are drawn (a seeded
    generator on that device); indices are always drawn on the host.  The two
    choices give different values from the same distributions.  ``d_qk`` is
    the row width: 576 (512 V + 64 rope) or 512 (V only, the width of the
    flash-attention page's performance table).
    """
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=value_device).manual_seed(seed)
    S_kv = T + T // 4
    idx = _window_and_compressed(T, topk, rng)
    length = None
    if compact:
        idx, length = _compact(idx, S_kv)
    q = _randn_bf16(gen, (T, H, d_qk))
    kv = _randn_bf16(gen, (S_kv, d_qk))
    dout = _randn_bf16(gen, (T, H, D_V))
    sink = torch.randn(H, generator=gen, dtype=torch.float32, device=gen.device)
    dev = gen.device
    return Workload(name, q, kv, torch.from_numpy(idx.astype(np.int32)).to(dev),
                    None if length is None else torch.from_numpy(length.astype(np.int32)).to(dev),
                    sink, dout, 1.0 / math.sqrt(d_qk),
                    {"T": T, "H": H, "S_kv": S_kv, "W": 128 + topk, "topk": topk,
                     "compact": compact, "seed": seed})


def varlen(lengths, H: int, topk: int, compact: bool, seed: int,
           value_device: str = "cpu", d_qk: int = D_QK) -> Workload:
    """A varlen batch of DeepSeek-V4-like sequences, packed.

    Sequence b has T_b = lengths[b] tokens and T_b + T_b // 4 KV rows, laid out
    as in ``dsv4`` with indices counted from its own first KV row.  All rows
    are padded to the same width 128 + topk.  A length of 0 gives an empty
    sequence (no tokens, no KV rows).  ``value_device`` chooses where q, kv,
    dout and sink are drawn, as in ``dsv4``.
    """
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=value_device).manual_seed(seed)
    W = 128 + topk
    idx_parts, len_parts, cu_q, cu_kv = [], [], [0], [0]
    for T_b in lengths:
        S_b = T_b + T_b // 4
        if T_b > 0:
            idx = _window_and_compressed(T_b, topk, rng)
            if compact:
                idx, ln = _compact(idx, S_b)
                len_parts.append(ln)
            idx_parts.append(idx)
        cu_q.append(cu_q[-1] + T_b)
        cu_kv.append(cu_kv[-1] + S_b)
    T, S_kv = cu_q[-1], cu_kv[-1]
    idx = np.concatenate(idx_parts, axis=0) if idx_parts else np.zeros((0, W), np.int64)
    q = _randn_bf16(gen, (T, H, d_qk))
    kv = _randn_bf16(gen, (S_kv, d_qk))
    dout = _randn_bf16(gen, (T, H, D_V))
    sink = torch.randn(H, generator=gen, dtype=torch.float32, device=gen.device)
    dev = gen.device
    length = (torch.from_numpy(np.concatenate(len_parts).astype(np.int32)).to(dev)
              if compact else None)
    return Workload(f"varlen{list(lengths)}", q, kv,
                    torch.from_numpy(idx.astype(np.int32)).to(dev), length, sink, dout,
                    1.0 / math.sqrt(d_qk),
                    {"lengths": list(lengths), "H": H, "topk": topk, "compact": compact,
                     "seed": seed},
                    torch.tensor(cu_q, dtype=torch.int32, device=dev),
                    torch.tensor(cu_kv, dtype=torch.int32, device=dev))


def random_rows(T: int, H: int, S_kv: int, W: int, max_valid: int, seed: int,
                compact: bool = False, d_qk: int = D_QK) -> Workload:
    """Token t takes n_t ~ U{0..min(max_valid, W, S_kv)} distinct rows of [0, S_kv)
    at random columns of W, the other columns -1 (or packed left with a
    topk_length when ``compact``).  For limit cases: T = 1, W = 1, the
    largest W, S_kv = 1, any H."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    idx = np.full((T, W), -1, dtype=np.int64)
    cap = min(max_valid, W, S_kv)
    for t in range(T):
        n = int(rng.integers(0, cap + 1))
        cols = rng.choice(W, size=n, replace=False)
        idx[t, cols] = rng.choice(S_kv, size=n, replace=False)
    length = None
    if compact:
        idx, length = _compact(idx, S_kv)
    q = _randn_bf16(gen, (T, H, d_qk))
    kv = _randn_bf16(gen, (S_kv, d_qk))
    dout = _randn_bf16(gen, (T, H, D_V))
    sink = torch.randn(H, generator=gen, dtype=torch.float32)
    return Workload(f"random_T{T}_H{H}_S{S_kv}_W{W}", q, kv, torch.from_numpy(idx.astype(np.int32)),
                    None if length is None else torch.from_numpy(length.astype(np.int32)),
                    sink, dout, 1.0 / math.sqrt(d_qk),
                    {"T": T, "H": H, "S_kv": S_kv, "W": W, "max_valid": max_valid, "seed": seed})


def tiny(seed: int = 1000) -> Workload:
    """T=64, S_kv=64, H=16, width 32, non-compact causal rows."""
    T, S_kv, H, W = 64, 64, 16, 32
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    idx = np.full((T, W), -1, dtype=np.int64)
    for t in range(T):
        n = min(W, t + 1)
        rows = rng.choice(t + 1, size=n, replace=False)
        cols = rng.choice(W, size=n, replace=False)
        idx[t, cols] = rows
    q = _randn_bf16(gen, (T, H, D_QK))
    kv = _randn_bf16(gen, (S_kv, D_QK))
    dout = _randn_bf16(gen, (T, H, D_V))
    sink = torch.randn(H, generator=gen, dtype=torch.float32)
    return Workload("tiny", q, kv, torch.from_numpy(idx.astype(np.int32)), None, sink,
                    dout, 1.0 / math.sqrt(D_QK),
                    {"T": T, "H": H, "S_kv": S_kv, "W": W, "compact": False, "seed": seed})


def edge(H: int, compact: bool, sub: int = 0, sink_override=None, T: int = 512,
         S_kv: int = 256, W: int = 1024, seed: Optional[int] = None) -> Workload:
    """Edge-case stress: width > S_kv, junk indices, empty rows, huge sinks.

    * n_t in {0..S_kv} distinct valid rows per token at random columns of W,
      so valid entries also sit at columns >= S_kv.
    * the other columns hold -1 (80 %), other negatives incl. INT32_MIN (10 %)
      and out-of-range values >= S_kv incl. INT32_MAX (10 %).
    * compact variant: same sets packed left, topk_length = n_t with ~10 % of
      tokens forced to 0, and valid-looking junk past topk_length.
    * kv ~ N(0,1) + 1; a quarter of (token, head) rows get q = -gamma with
      gamma in {4, 64} so that some LSE are far below -80.
    * sinks cycle through ``EDGE_SINKS`` (N(0,1) for the None entry); with
      H == 1, ``sub`` picks the value; ``sink_override`` forces every head.
    """
    if seed is None:
        seed = 1004 + 10 * sub + (1 if compact else 0) + 100 * H
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    idx = np.full((T, W), -1, dtype=np.int64)
    n = rng.integers(0, S_kv + 1, size=T)
    n[rng.random(T) < 0.05] = 0
    for t in range(T):
        rows = rng.choice(S_kv, size=n[t], replace=False)
        cols = rng.choice(W, size=n[t], replace=False)
        idx[t, cols] = rows
        free = np.ones(W, dtype=bool)
        free[cols] = False
        fc = np.nonzero(free)[0]
        u = rng.random(len(fc))
        neg = fc[(u >= 0.8) & (u < 0.9)]
        big = fc[u >= 0.9]
        idx[t, neg] = rng.integers(INT32_MIN, 0, size=len(neg))
        idx[t, big] = rng.integers(S_kv, INT32_MAX, size=len(big), endpoint=True)
        if len(neg):
            idx[t, neg[0]] = INT32_MIN
        if len(big):
            idx[t, big[0]] = INT32_MAX
    length = None
    if compact:
        packed = np.full_like(idx, -1)
        length = n.copy()
        length[rng.random(T) < 0.10] = 0
        for t in range(T):
            v = idx[t][(idx[t] >= 0) & (idx[t] < S_kv)]
            packed[t, :len(v)] = v
            # past the length: valid-looking rows that must still be ignored
            packed[t, len(v):] = rng.integers(0, S_kv, size=W - len(v))
        idx = packed
    q = _randn_bf16(gen, (T, H, D_QK))
    kv = _randn_bf16(gen, (S_kv, D_QK), shift=1.0)
    dout = _randn_bf16(gen, (T, H, D_V))
    neg_rows = rng.random((T, H)) < 0.25
    gam = np.where(rng.random((T, H)) < 0.5, 4.0, 64.0)
    qv = q.float()
    sel = torch.from_numpy(neg_rows)
    qv[sel] = -torch.from_numpy(gam)[sel].float()[:, None].expand(-1, D_QK)
    q = qv.to(torch.bfloat16)
    sink = torch.randn(H, generator=gen, dtype=torch.float32)
    for h in range(H):
        v = EDGE_SINKS[(h + sub) % len(EDGE_SINKS)] if H > 1 else EDGE_SINKS[sub % len(EDGE_SINKS)]
        if v is not None:
            sink[h] = v
    if sink_override is not None:
        sink[:] = sink_override
    return Workload(f"edge_h{H}_{'compact' if compact else 'noncompact'}_s{sub}", q, kv,
                    torch.from_numpy(idx.astype(np.int32)),
                    None if length is None else torch.from_numpy(length.astype(np.int32)),
                    sink, dout, 1.0 / math.sqrt(D_QK),
                    {"T": T, "H": H, "S_kv": S_kv, "W": W, "compact": compact, "seed": seed})


def make(name: str, **kw) -> Workload:
    """Build a named workload.

    ``tiny``     T=64,    H=16,  width 32, S_kv=64, non-compact
    ``flash``    T=4096,  H=128, window 128 + top-k 512, non-compact
    ``flash_h64``T=8192,  H=64,  window 128 + top-k 512, compact
    ``flash_t8k``T=8192,  H=128, window 128 + top-k 512, non-compact
    ``pro``      T=16384, H=128, window 128 + top-k 1024, non-compact
    ``edge``     T=512,   S_kv=256, width 1024 (see ``edge``)
    ``T``/``H`` keyword arguments shrink the DeepSeek-V4 layouts for fast tests.
    """
    if name == "tiny":
        return tiny(**kw)
    if name == "edge":
        return edge(**kw)
    table = {
        "flash": dict(T=4096, H=128, topk=512, compact=False, seed=1001),
        "flash_h64": dict(T=8192, H=64, topk=512, compact=True, seed=1002),
        "flash_t8k": dict(T=8192, H=128, topk=512, compact=False, seed=1005),
        "pro": dict(T=16384, H=128, topk=1024, compact=False, seed=1003),
    }
    if name not in table:
        raise KeyError(name)
    args = dict(table[name])
    args.update(kw)
    return dsv4(name=name, **args)


def valid_slot_count_formula(T: int, topk: int) -> np.ndarray:
    """Closed form of K_t for the DeepSeek-V4 layout: min(t+1,128)+min(topk,(t+1)//4)."""
    t = np.arange(T)
    return np.minimum(t + 1, 128) + np.minimum(topk, (t + 1) // 4)
