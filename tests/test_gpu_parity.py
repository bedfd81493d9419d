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
from tests.parity_util import (LSE_TOL, REL_TOL, check_bwd, check_fwd, check_per_head,
                               check_per_head_dsink, np64, per_head_rel, rel_frob)

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
    """Oracle forward and backward by the definition (delta from the fp64 O).

    The backward forms the exact delta, sum_j P_j dP_j, itself (the accurate
    form in the cuDNN page "DSA backward SM90: fix three top-k and
    attention-sink boundary failures", section "Not addressed"), so every
    output of the default path is held to the exact definition."""
    ref = O.forward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale, tokens=tokens)
    g = O.backward(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale,
                   w.dout if dout is None else dout, tokens=tokens)
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
# The gamma = 64 rows attend one-hot: their dS is all rounding noise of the
# bf16 out unless the backward takes the exact delta, which it does.  Every
# output is held to the exact definition at the same bar.


@pytest.mark.parametrize("name,mk", SMALL, ids=[s[0] for s in SMALL])
def test_fwd_bwd_parity_small(name, mk):
    """Default path against the exact fp64 definition, every element."""
    w = mk()
    out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    ef = check_fwd(out, lse, ref, counts)
    eb = check_bwd(dq, dkv, dsink, g, counts)
    if name.startswith("edge"):
        check_per_head(out, ref["out"], "out")
        check_per_head(dq, g["dq"], "dq")
        check_per_head_dsink(dsink, g["dsink"])
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


EDGE_BWD = ([(H, c, None) for H in (24, 96) for c in (False, True)] +
            [(1, c, sub) for sub in range(len(WL.EDGE_SINKS)) for c in (False, True)])


@pytest.mark.parametrize("H,compact,sub", EDGE_BWD,
                         ids=[f"H{h}-{'c' if c else 'nc'}-{s}" for h, c, s in EDGE_BWD])
def test_bwd_only_parity(H, compact, sub):
    """dsa_bwd alone, fed the oracle's own forward outputs (its fp64 out
    rounded to bf16 as a forward stores it, and its lse in fp32), on every
    edge workload: this separates the backward kernels' error from the
    forward's.  All outputs against the exact definition, then head by head
    (a wrong sink-stress head cannot hide under the others' norm)."""
    w = WL.edge(H=H, compact=compact, sub=0 if sub is None else sub)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    wd = w.to(DEV)
    out = torch.from_numpy(bf16_stored(ref["out"])).to(torch.bfloat16).to(DEV)
    lse = torch.from_numpy(ref["lse"]).to(torch.float32).to(DEV)
    dq, dkv, dsink = dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse,
                             wd.dout, wd.scale)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    eb = check_bwd(dq, dkv, dsink, g, counts)
    ph = check_per_head(dq, g["dq"], "dq")
    check_per_head_dsink(dsink, g["dsink"])
    print(H, compact, sub, eb, "dq per head max", max(ph))


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
    check_fwd(out2, lse2, ref, counts)
    check_bwd(dq2, dkv2, dsink2, g, counts)
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
    ref, g = oracle_exact(w)
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
    ref, g = oracle_exact(w, tokens=toks)
    ef = check_fwd(out, lse, ref, counts, rows=toks)
    eb = check_bwd(dq, None, None, g, counts, rows=toks, check_dkv=False, check_dsink=False)
    # dkv rows: two window-only original rows and the two last compressed rows
    rows = [5, w.T // 3, w.S_kv - 1, w.S_kv - 2]
    rtoks = O.tokens_referencing(w.topk_idxs, w.topk_length, w.S_kv, rows)
    _, gr = oracle_exact(w, tokens=rtoks)
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
    ref, g = oracle_exact(w, dout=dout, tokens=toks)
    eb = check_bwd(dq, dkv, dsink, g, counts, rows=toks)
    others = np.setdiff1d(np.arange(w.T), toks)
    assert (np64(dq)[others] == 0).all()
    print(name, eb)
