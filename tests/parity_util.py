"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances come from the acceptance bar for bf16 inputs with fp32 accumulation:
  - relative Frobenius error <= 1e-2 on out, dq, dkv and dsink;
  - |lse - ref| <= 1e-3 absolute;
  - no NaN or Inf anywhere;
  - exact zeros where the definition has structural zeros;
  - index handling bit-exact.
"""
import numpy as np
import torch

from oracle import dsa_oracle as O

REL_TOL = 1e-2
LSE_TOL = 1e-3


def np64(x):
    return x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x)


def rel_frob(a, ref):
    a, ref = np64(a), np64(ref)
    n = np.linalg.norm(ref)
    d = np.linalg.norm(a - ref)
    if n == 0:
        return 0.0 if d == 0 else float("inf")
    return float(d / n)


def assert_finite(**tensors):
    for k, v in tensors.items():
        if v is None:
            continue
        assert torch.isfinite(v.float()).all(), f"{k} has non-finite values"


def check_fwd(out, lse, ref, counts, rows=None):
    """Compare forward outputs on `rows` (all tokens if None)."""
    out_np, lse_np = np64(out), np64(lse)
    sel = np.arange(out_np.shape[0]) if rows is None else np.asarray(rows)
    assert_finite(out=out, lse=lse)
    empty = sel[counts[sel] == 0]
    live = sel[counts[sel] > 0]
    # empty rows: exact zeros and the bit-exact sentinel
    if len(empty):
        assert (out_np[empty] == 0).all()
        assert (lse.detach().cpu().numpy()[empty] == np.float32(O.EMPTY_LSE)).all()
    errs = {"out": rel_frob(out_np[sel], ref["out"][sel])}
    if len(live):
        errs["lse_abs"] = float(np.abs(lse_np[live] - ref["lse"][live]).max())
    else:
        errs["lse_abs"] = 0.0
    assert errs["out"] <= REL_TOL, errs
    assert errs["lse_abs"] <= LSE_TOL, errs
    return errs


def check_bwd(dq, dkv, dsink, g, counts, rows=None, check_dkv=True, check_dsink=True):
    assert_finite(dq=dq, dkv=dkv, dsink=dsink)
    dq_np = np64(dq)
    sel = np.arange(dq_np.shape[0]) if rows is None else np.asarray(rows)
    empty = sel[counts[sel] == 0]
    if len(empty):
        assert (dq_np[empty] == 0).all()
    errs = {"dq": rel_frob(dq_np[sel], g["dq"][sel])}
    if check_dkv:
        dkv_np = np64(dkv)
        zero_rows = np.nonzero((g["dkv"] == 0).all(axis=1))[0]
        assert (dkv_np[zero_rows] == 0).all(), "structural-zero dkv rows were written"
        errs["dkv"] = rel_frob(dkv_np, g["dkv"])
    if check_dsink and dsink is not None:
        errs["dsink"] = rel_frob(dsink, g["dsink"])
    for k, v in errs.items():
        assert v <= REL_TOL, errs
    return errs


def per_head_rel(a, ref):
    a, ref = np64(a), np64(ref)
    H = a.shape[1]
    return [rel_frob(a[:, h], ref[:, h]) for h in range(H)]


def check_per_head(a, ref, what):
    """Every head on its own within the bar (a head whose reference is all
    zero, e.g. under a positive saturating sink, must be exactly zero), so
    that one wrong sink-stress head cannot hide under the others' norm."""
    errs = per_head_rel(a, ref)
    bad = {h: e for h, e in enumerate(errs) if not e <= REL_TOL}
    assert not bad, f"{what}: heads over the bar {bad}"
    return errs


def check_per_head_dsink(dsink, ref):
    """d_sink head by head: exact zeros where the reference is zero (no sink
    share, or a sink that takes the whole denominator with out = 0), else a
    relative error within the bar."""
    a, r = np64(dsink), np64(ref)
    floor = 1e-3 * float(np.abs(r).max()) if r.size else 0.0
    for h in range(r.shape[0]):
        if r[h] == 0:
            assert a[h] == 0, (h, a[h])
        else:
            assert abs(a[h] - r[h]) <= REL_TOL * max(abs(r[h]), floor), (h, a[h], r[h])
