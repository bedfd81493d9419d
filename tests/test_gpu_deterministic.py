"""DSA_FLAG_DETERMINISTIC: dkv summed in 64-bit fixed point.

The pages name two dKV reductions: fp32 atomics (the SM90 design) and a
separate, ordered reduction (the SM100 design; cuDNN frontend "DSA bwd SM100
fix dropped dKV gradients when topk width > total_S_kv").  Here the ordered
variant is an order-independent one: integer adds of round(v * 2^32).  The
outputs must meet the same parity bar as the default mode and be the same
bits on every run.
"""
import pytest
import torch

from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import REL_TOL, check_bwd, check_fwd, rel_frob
from tests.test_gpu_parity import (DEV, SMALL, _lib, counts_of,  # noqa: F401
                                   oracle_exact)

pytestmark = pytest.mark.gpu


def fwd(wd):
    return dsa.fwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, wd.scale)


def bwd(wd, out, lse, deterministic):
    g = dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse, wd.dout, wd.scale,
                deterministic=deterministic)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    return g


@pytest.mark.parametrize("name,mk", SMALL, ids=[s[0] for s in SMALL])
def test_deterministic_parity_small(name, mk):
    w = mk()
    wd = w.to(DEV)
    out, lse = fwd(wd)
    dq, dkv, dsink = bwd(wd, out, lse, deterministic=True)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    eb = check_bwd(dq, dkv, dsink, g, counts)
    print(name, eb)


def test_deterministic_bits_repeat():
    """Five deterministic runs, interleaved with atomic-mode runs that perturb
    the scheduling and the L2 state, give the same dq, dkv and dsink bits.
    T = 2048 at H = 128: each window row is added to by 128 tokens and the
    compressed rows by many more, so the atomic order really varies."""
    w = WL.make("flash", T=2048, H=128)
    wd = w.to(DEV)
    out, lse = fwd(wd)
    first = [x.clone() for x in bwd(wd, out, lse, deterministic=True)]
    atomic = None
    for _ in range(4):
        atomic = bwd(wd, out, lse, deterministic=False)
        again = bwd(wd, out, lse, deterministic=True)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    # the two modes sum the same fp32 contributions; they agree far inside the bar
    assert rel_frob(first[1], atomic[1]) <= 1e-3
    assert torch.equal(first[0], atomic[0])  # dq never used atomics


def test_deterministic_workspace_is_larger():
    small = dsa.bwd_workspace_bytes(512, 128, 640, 640)
    det = dsa.bwd_workspace_bytes(512, 128, 640, 640, deterministic=True)
    assert det - small == 640 * 576 * 4 + 640 * 4 + 256  # int64 accumulator, per-row range check


DSA_ERR_RANGE = 7


def test_range_check_flags_a_row_that_may_wrap():
    """Huge contributions (dout scaled by 2^33) push the bound n_r * m_r of
    some rows past 2^31: the call completes without a fault and
    dsa_device_status reports DSA_ERR_RANGE, once.  The same inputs in fp32
    mode, and ordinary inputs in deterministic mode, report nothing."""
    w = WL.make("tiny")
    wd = w.to(DEV)
    out, lse = fwd(wd)
    big = (wd.dout.float() * 2.0 ** 33).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse, big, wd.scale,
            deterministic=True)
    assert dsa.device_status() == DSA_ERR_RANGE
    assert dsa.device_status() == 0  # read and cleared
    dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse, big, wd.scale,
            deterministic=False)
    assert dsa.device_status() == 0
    dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse, wd.dout, wd.scale,
            deterministic=True)
    assert dsa.device_status() == 0
