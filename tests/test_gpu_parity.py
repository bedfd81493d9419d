"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small workloads are compared element by element over every output.  They
span several 128-row blocks and ragged tails.  The full-size DeepSeek-V4
workloads run in the launch configuration the benchmark times, and the
comparisons there use:
  - sampled tokens (out, lse, dq);
  - sampled dkv rows, with the oracle run over every token that gathers them;
  - a run whose dout is zero outside a token sample, so the GPU's complete
    dkv and dsink must equal the oracle's sums over that sample.
"""
import math

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import (LSE_TOL, REL_TOL, check_bwd, check_fwd, np64, per_head_rel,
                               rel_frob)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_top_attention_gb300 import build as B
    B.build()
    dsa.library()


def run(w, dout=None, residual=False):
    wd = w.to(DEV)
    out, lse = dsa.fwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, wd.scale,
                       delta_residual=residual)
    d = wd.dout if dout is None else dout.to(DEV)
    dq, dkv, dsink = dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse, d,
                             wd.scale, delta_residual=residual)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    return out, lse, dq, dkv, dsink


def bf16_stored(x):
    """The oracle's own fp64 output, rounded to bf16 as the forward stores it."""
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def oracle_exact(w, dout=None, tokens=None):
    """Oracle forward and backward by the definition (delta from the fp64 O)."""
    ref = O.forward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale, tokens=tokens)
    g = O.backward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale,
                   w.dout if dout is None else dout, tokens=tokens)
    return ref, g


def oracle_all(w, dout=None, tokens=None):
    """Oracle forward, then the oracle backward whose delta is taken from the
    bf16-stored forward output.  That is the backward's contract (delta =
    rowsum(dout * out) of the out handed in), and it is how the cuDNN page
    "DSA backward SM90: fix three top-k and attention-sink boundary failures"
    ("Not addressed") checks its kernel: an fp64 recomputation that starts
    from the bf16 output the forward stored.  The bf16 out is derived from
    the oracle, never from the GPU."""
    ref = O.forward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale, tokens=tokens)
    g = O.backward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale,
                   w.dout if dout is None else dout, out=bf16_stored(ref["out"]), tokens=tokens)
    return ref, g


def counts_of(w):
    return O.valid_lists(w.topk_idxs, w.topk_length, w.S_kv)[1]


# ------------------------------------------------------------------ a1: bit-exact decode

SMALL = [
    ("tiny", lambda: WL.make("tiny")),
    ("flash_T512", lambda: WL.make("flash", T=512, H=128)),
    ("flash_h64_T512", lambda: WL.make("flash_h64", T=512, H=64)),
    ("edge_h24_nc", lambda: WL.edge(H=24, compact=False)),
    ("edge_h24_c", lambda: WL.edge(H=24, compact=True)),
    ("edge_h96_nc", lambda: WL.edge(H=96, compact=False)),
    ("edge_h96_c", lambda: WL.edge(H=96, compact=True)),
]


@pytest.mark.parametrize("name,mk", SMALL, ids=[s[0] for s in SMALL])
def test_compaction_bit_exact(name, mk):
    w = mk()
    lists, counts = O.valid_lists(w.topk_idxs, w.topk_length, w.S_kv)
    idx_out, cnt = dsa.topk_compact(w.topk_idxs.to(DEV),
                                    None if w.topk_length is None else w.topk_length.to(DEV), w.S_kv)
    cnt = cnt.cpu().numpy()
    idx_out = idx_out.cpu().numpy()
    np.testing.assert_array_equal(cnt, counts)
    for t in range(w.T):
        np.testing.assert_array_equal(idx_out[t, :counts[t]], lists[t])


# ------------------------------------------------------------------ small, every element

# In the edge workloads a quarter of the (token, head) rows have q = -gamma
# (gamma in {4, 64}) against kv with mean 1, so that some lse fall below -80.
# The gamma = 64 rows attend one-hot.  Their dS is set by the bf16 rounding
# of `out`, and through |q| = 64 they carry almost all of the dkv norm.
# Under the default contract (delta from the bf16 out, as on the cuDNN page
# "DSA backward SM90: fix three top-k and attention-sink boundary failures",
# section "Not addressed") no implementation can reproduce that rounding
# noise bit for bit.  So default-mode dkv on these workloads is held to
# 2e-2.  With DSA_FLAG_DELTA_RESIDUAL (that section's forward-side fix) the
# GPU must match the exact fp64 definition within the 1e-2 bar everywhere.
EDGE_CONTRACT_DKV_TOL = 2e-2


@pytest.mark.parametrize("name,mk", SMALL, ids=[s[0] for s in SMALL])
def test_fwd_bwd_parity_small(name, mk):
    """Default contract against the oracle whose delta uses the bf16-stored O."""
    w = mk()
    out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_all(w)
    counts = counts_of(w)
    ef = check_fwd(out, lse, ref, counts)
    edge = name.startswith("edge")
    eb = check_bwd(dq, dkv, dsink, g, counts,
                   dkv_tol=EDGE_CONTRACT_DKV_TOL if edge else REL_TOL)
    print(name, ef, eb)


@pytest.mark.parametrize("name,mk", SMALL, ids=[s[0] for s in SMALL])
def test_fwd_bwd_parity_exact_delta(name, mk):
    """DSA_FLAG_DELTA_RESIDUAL against the exact fp64 definition."""
    w = mk()
    out, lse, dq, dkv, dsink = run(w, residual=True)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    ef = check_fwd(out, lse, ref, counts)
    eb = check_bwd(dq, dkv, dsink, g, counts)
    print(name, ef, eb)


@pytest.mark.parametrize("sub", range(len(WL.EDGE_SINKS)))
@pytest.mark.parametrize("compact", [False, True])
def test_single_head_sink_cases(sub, compact):
    """H = 1 with each sink value, incl. +-1e38, +-2.4e38 and +-FLT_MAX."""
    w = WL.edge(H=1, compact=compact, sub=sub)
    out, lse, dq, dkv, dsink = run(w, residual=True)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)
    out2, lse2, dq2, dkv2, dsink2 = run(w)
    ref2, g2 = oracle_all(w)
    check_fwd(out2, lse2, ref2, counts)
    check_bwd(dq2, dkv2, dsink2, g2, counts, dkv_tol=EDGE_CONTRACT_DKV_TOL)
    sk = float(w.sink[0])
    if sk >= 1e38:  # the sink takes the whole denominator
        assert (np64(out) == 0).all() and (np64(dq) == 0).all() and (np64(dkv) == 0).all()


@pytest.mark.parametrize("sink", [math.inf, -math.inf])
def test_infinite_sinks(sink):
    w = WL.edge(H=24, compact=False, sink_override=sink)
    out, lse, dq, dkv, dsink = run(w, residual=True)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)
    if sink > 0:
        assert (np64(out) == 0).all() and (np64(dq) == 0).all() and (np64(dkv) == 0).all()
        # d_sink = -sum_t delta with delta from the (zero) output: exactly 0
        assert (np64(dsink) == 0).all()


def test_no_sink():
    w = WL.make("flash", T=300, H=64)
    w.sink = None
    out, lse, dq, dkv, dsink = run(w)
    assert dsink is None
    ref, g = oracle_all(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, None, g, counts, check_dsink=False)


def test_very_negative_lse_is_exercised():
    """Self-check that the edge workload really reaches lse < -80."""
    w = WL.edge(H=24, compact=False)
    _, lse, *_ = run(w)
    counts = counts_of(w)
    live = np64(lse)[counts > 0]
    assert live.min() < -80


def test_head_padding_is_invisible():
    """Heads 0..23 of H = 24 equal heads 0..23 of H = 32 whose extra heads
    have dout = 0 (the in-kernel padding analogue of the flash-attention
    page's bit-identity probe)."""
    w24 = WL.edge(H=24, compact=True, sink_override=0.5)
    w32 = WL.edge(H=32, compact=True, sink_override=0.5, seed=w24.meta["seed"])
    w32.topk_idxs, w32.topk_length, w32.kv = w24.topk_idxs, w24.topk_length, w24.kv
    w32.q = torch.cat([w24.q, w32.q[:, 24:]], dim=1).contiguous()
    dout32 = torch.cat([w24.dout, torch.zeros_like(w32.dout[:, 24:])], dim=1).contiguous()
    w32.dout = dout32
    a = run(w24)
    b = run(w32)
    assert torch.equal(a[0], b[0][:, :24])   # out
    assert torch.equal(a[1], b[1][:, :24])   # lse
    assert torch.equal(a[2], b[2][:, :24])   # dq
    # dkv: fp32 atomics land in any order, so the bf16 cast may differ by one ulp
    assert rel_frob(a[3], b[3]) <= 1e-3
    assert torch.allclose(a[4], b[4][:24], rtol=1e-5, atol=0)


def test_repeat_launch_stress():
    """Many launches of a workload with mixed empty and non-empty rows."""
    w = WL.edge(H=24, compact=True).to(DEV)
    out0, lse0 = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
    dq0, dkv0, ds0 = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out0, lse0, w.dout,
                             w.scale)
    for _ in range(100):
        out, lse = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
        dq, dkv, ds = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout,
                              w.scale)
        assert torch.equal(out, out0) and torch.equal(lse, lse0) and torch.equal(dq, dq0)
        assert rel_frob(dkv, dkv0) <= 1e-3   # atomic order: rare one-ulp bf16 flips
    assert dsa.device_status() == 0


# ------------------------------------------------------------------ full size, sampled

FULL = [
    ("flash", dict()),
    ("flash_h64", dict()),
    pytest.param("flash_t8k", dict(), marks=pytest.mark.slow),
    pytest.param("pro", dict(), marks=pytest.mark.slow),
]


def _sample_tokens(T, rng, n=10):
    base = [0, 1, 126, 127, 128, T // 2, T - 2, T - 1]
    return sorted(set(base + list(rng.integers(0, T, size=n))))


@pytest.mark.parametrize("name,kw", FULL)
def test_full_size_sampled(name, kw):
    w = WL.make(name, **kw)
    rng = np.random.default_rng(7)
    out, lse, dq, dkv, dsink = run(w)
    counts = counts_of(w)
    toks = _sample_tokens(w.T, rng)
    ref, g = oracle_all(w, tokens=toks)
    ef = check_fwd(out, lse, ref, counts, rows=toks)
    eb = check_bwd(dq, None, None, g, counts, rows=toks, check_dkv=False, check_dsink=False)
    # dkv rows: two window-only original rows and the two last compressed rows
    rows = [5, w.T // 3, w.S_kv - 1, w.S_kv - 2]
    rtoks = O.tokens_referencing(w.topk_idxs, w.topk_length, w.S_kv, rows)
    _, gr = oracle_all(w, tokens=rtoks)
    dkv_err = rel_frob(np64(dkv)[rows], gr["dkv"][rows])
    assert dkv_err <= REL_TOL, dkv_err
    print(name, ef, eb, {"dkv_rows": dkv_err, "ref_tokens": len(rtoks)})


@pytest.mark.parametrize("name", ["flash", "flash_h64"])
def test_full_size_masked_dout(name):
    """dout = 0 outside 12 tokens: the complete dkv and dsink of the full-size
    launch must equal the oracle's sums over those tokens."""
    w = WL.make(name)
    rng = np.random.default_rng(11)
    toks = _sample_tokens(w.T, rng, n=4)
    mask = torch.zeros(w.T, dtype=torch.bool)
    mask[toks] = True
    dout = torch.where(mask[:, None, None], w.dout, torch.zeros_like(w.dout))
    out, lse, dq, dkv, dsink = run(w, dout=dout)
    counts = counts_of(w)
    ref, g = oracle_all(w, dout=dout, tokens=toks)
    eb = check_bwd(dq, dkv, dsink, g, counts, rows=toks)
    others = np.setdiff1d(np.arange(w.T), toks)
    assert (np64(dq)[others] == 0).all()
    print(name, eb)
