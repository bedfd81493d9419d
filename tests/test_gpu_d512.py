"""GPU parity of the D_qk = D_v = 512 variant (rows with no rope part), the
width of the DeepSeek-V4 performance table on the flash-attention page
"[CuTe, SM100] Support 1..128 Q heads in sparse MLA via in-kernel TMA
padding" ("Performance at DeepSeek-V4 shapes")."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import REL_TOL, check_bwd, check_fwd, np64, rel_frob
from tests.test_gpu_parity import (_lib, _sample_tokens, counts_of, oracle_exact,  # noqa: F401
                                   run)
from tests.test_gpu_varlen import oracle_varlen, run_varlen

pytestmark = pytest.mark.gpu

SMALL = [
    ("flash_T512_h128", dict(T=512, H=128, topk=512, compact=False, seed=2001)),
    ("flash_T512_h64_compact", dict(T=512, H=64, topk=512, compact=True, seed=2002)),
    ("ragged_T300_h24", dict(T=300, H=24, topk=128, compact=True, seed=2003)),
    ("flash_T512_h16", dict(T=512, H=16, topk=512, compact=False, seed=2006)),
]


def d512(name, kw):
    return WL.dsv4(name=name, d_qk=512, **kw)


@pytest.mark.parametrize("name,kw", SMALL, ids=[c[0] for c in SMALL])
def test_d512_parity_small(name, kw):
    w = d512(name, kw)
    assert w.q.shape[2] == 512 and w.kv.shape[1] == 512
    out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)


def test_d512_deterministic_matches_atomic():
    w = d512(*SMALL[0]).to("cuda:0")
    out, lse = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
    a = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout, w.scale,
                deterministic=True)
    b = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout, w.scale,
                deterministic=True)
    c = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout, w.scale)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    assert torch.equal(a[1], b[1])
    assert rel_frob(a[1], c[1]) <= 1e-3


@pytest.mark.parametrize("H,topk,seed", [(64, 64, 2004), (8, 512, 2007)])
def test_d512_varlen(H, topk, seed):
    w = WL.varlen([200, 0, 333], H=H, topk=topk, compact=True, seed=seed, d_qk=512)
    out, lse, dq, dkv, dsink = run_varlen(w)
    ref, g = oracle_varlen(w)
    check_fwd(out, lse, ref, ref["count"])
    check_bwd(dq, dkv, dsink, g, ref["count"])


def test_d512_full_size_sampled():
    """The bench's D = 512 configuration (T = 8192, H = 128, flash layout) in
    its launch configuration, on sampled tokens and dkv rows."""
    w = WL.dsv4(T=8192, H=128, topk=512, compact=False, seed=2005, name="flash_t8k_d512",
                d_qk=512)
    rng = np.random.default_rng(9)
    out, lse, dq, dkv, dsink = run(w)
    counts = counts_of(w)
    toks = _sample_tokens(w.T, rng)
    ref, g = oracle_exact(w, tokens=toks)
    check_fwd(out, lse, ref, counts, rows=toks)
    check_bwd(dq, None, None, g, counts, rows=toks, check_dkv=False, check_dsink=False)
    rows = [5, w.T // 3, w.S_kv - 1, w.S_kv - 2]
    rtoks = O.tokens_referencing(w.topk_idxs, w.topk_length, w.S_kv, rows)
    _, gr = oracle_exact(w, tokens=rtoks)
    assert rel_frob(np64(dkv)[rows], gr["dkv"][rows]) <= REL_TOL
