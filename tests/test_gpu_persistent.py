"""GPU parity for the persistent kernels' scheduling.

The forward launches one CTA per SM, k_bwd_dq and k_bwd_dkv two; each CTA
walks its items c, c + grid, ... ((token, head group) items, or tokens in
k_bwd_dkv) and keeps its barrier phases in running counts of items, blocks
and S steps.  These cases stress that
bookkeeping: long runs of empty tokens (every role must skip the same items),
fewer items than SMs, one item more than the grid, and items that differ
widely in block count next to each other.
"""
import numpy as np
import pytest
import torch

from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import check_bwd, check_fwd
from tests.test_gpu_parity import DEV, _lib, counts_of, oracle_exact, run  # noqa: F401

pytestmark = pytest.mark.gpu


def _empty_runs(w, keep_every, run_len):
    """Empty every token except those in short runs: tokens t with
    t % keep_every < run_len keep their rows, the others get none."""
    idx = w.topk_idxs.clone()
    t = torch.arange(idx.shape[0])
    empty = (t % keep_every) >= run_len
    if w.topk_length is None:
        idx[empty] = -1
        w.topk_idxs = idx
    else:
        ln = w.topk_length.clone()
        ln[empty] = 0
        w.topk_length = ln
    return w


def _check(w, deterministic=False):
    if deterministic:
        wd = w.to(DEV)
        out, lse = dsa.fwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, wd.scale)
        dq, dkv, dsink = dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse,
                                 wd.dout, wd.scale, deterministic=True)
        torch.cuda.synchronize()
        assert dsa.device_status() == 0
    else:
        out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)
    return counts


@pytest.mark.parametrize("H,compact", [(128, False), (40, True), (16, False)])
def test_long_runs_of_empty_tokens(H, compact):
    """About 85% of the tokens are empty, in runs of 17: with T = 1500 every
    CTA meets several empty items between non-empty ones."""
    w = WL.random_rows(1500, H, 900, 300, 300, seed=4100 + H, compact=compact)
    w = _empty_runs(w, keep_every=20, run_len=3)
    counts = _check(w)
    assert (counts == 0).sum() > 1200


def test_long_runs_of_empty_tokens_deterministic():
    w = _empty_runs(WL.random_rows(1200, 96, 700, 260, 260, seed=4200), keep_every=13, run_len=2)
    _check(w, deterministic=True)


def test_fewer_items_than_sms():
    """T = 20 at H = 128: 40 items, so most SMs get none and the grid is the
    item count."""
    _check(WL.random_rows(20, 128, 2000, 640, 640, seed=4300))


@pytest.mark.parametrize("per_sm", [1, 2])
def test_one_item_more_than_the_grid(per_sm):
    """T * G = per_sm * SMs + 1 items at H = 64 (one head group).  The forward
    launches one CTA per SM and the backward kernels two, so with per_sm = 1
    the forward's CTA 0 takes two items, and with per_sm = 2 the backward's
    CTA 0 takes two (items in k_bwd_dq, tokens in k_bwd_dkv)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _check(WL.random_rows(per_sm * sms + 1, 64, 1500, 520, 520, seed=4400 + per_sm))


def test_neighbouring_items_of_very_different_lengths():
    """Alternate one-block and sixteen-block tokens (W = 2048), so the CTAs'
    block and step counters advance by very different amounts per item."""
    T, H, S_kv, W = 400, 64, 4096, 2048
    w = WL.random_rows(T, H, S_kv, W, W, seed=4500)
    idx = w.topk_idxs.numpy().copy()
    rng = np.random.default_rng(4501)
    for t in range(T):
        n = 2048 if t % 2 == 0 else int(rng.integers(1, 100))
        idx[t] = -1
        cols = rng.choice(W, size=n, replace=False)
        idx[t, cols] = rng.choice(S_kv, size=n, replace=False)
    w.topk_idxs = torch.from_numpy(idx)
    _check(w)
