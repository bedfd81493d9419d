"""dsa_bwd_no_alloc: the backward that allocates nothing, for callers that
cannot allocate device memory at call time (a plain C program holding only
its inputs and outputs; a serving loop under a fixed memory budget where a
cudaMalloc would synchronise the device).

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.  The tests call the entry point through
the C ABI:
  - twice in a row, for the fp32 and the int64 (DSA_FLAG_DETERMINISTIC)
    accumulators and both row widths.  Each time its outputs must match those
    of dsa_bwd (same kernels, workspace from torch): dq and d_sink exactly,
    dkv bitwise in deterministic mode, else up to the one-ulp bf16 flips that
    the order of fp32 atomics allows (the bound the other repeat-launch tests
    use);
  - on the largest flash-layout problem whose workspace fits the array,
    against the fp64 oracle.
A problem whose workspace exceeds the fixed 64 MiB array must be rejected
before anything launches, and a problem dsa_bwd rejects gets the same status.
"""
import ctypes

import pytest
import torch

from oracle import dsa_oracle as O
from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import check_bwd, rel_frob

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NO_ALLOC_BYTES = 64 << 20


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_top_attention_gb300 import build as B
    B.build()
    return dsa.library()


def _p(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _no_alloc(lib, w, prob, out, lse, stream, like):
    dq0, dkv0, ds0 = like
    dq = torch.full_like(dq0, float("nan"))
    dkv = torch.full_like(dkv0, float("nan"))
    ds = torch.full_like(ds0, float("nan"))
    rc = lib.dsa_bwd_no_alloc(ctypes.byref(prob), _p(w.q), _p(w.kv), _p(w.topk_idxs),
                              _p(w.topk_length), _p(w.sink), _p(out), _p(lse), _p(w.dout),
                              _p(dq), _p(dkv), _p(ds), stream)
    assert rc == 0, dsa.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    return dq, dkv, ds


@pytest.mark.parametrize("d_qk", [576, 512])
@pytest.mark.parametrize("deterministic", [False, True])
def test_no_alloc_backward_matches_workspace_backward(lib, deterministic, d_qk):
    """Both accumulator layouts (fp32, and int64 with DSA_FLAG_DETERMINISTIC)
    and both row widths, two calls in a row."""
    w = WL.make("flash", T=128, H=128, d_qk=d_qk).to(DEV)
    flags = dsa.FLAG_DETERMINISTIC if deterministic else 0
    prob = dsa.make_problem(w.T, w.H, w.S_kv, w.W, w.scale, flags, d_qk)
    assert 0 < lib.dsa_bwd_workspace_bytes(ctypes.byref(prob)) <= NO_ALLOC_BYTES
    out, lse = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
    ref = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout, w.scale,
                  deterministic=deterministic)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dq, dkv, ds = _no_alloc(lib, w, prob, out, lse, stream, ref)
        assert torch.equal(dq, ref[0])
        assert torch.equal(ds, ref[2])
        assert torch.isfinite(dkv.float()).all()
        if deterministic:  # integer adds: the same bits whatever the order
            assert torch.equal(dkv, ref[1])
        else:
            assert rel_frob(dkv, ref[1]) <= 1e-3


def test_no_alloc_near_the_limit_matches_the_oracle(lib):
    """The largest DeepSeek-V4 flash problem (H = 128, 640 slots per token)
    whose workspace still fits the array, against the fp64 oracle."""
    T = 16
    while True:
        nxt = dsa.make_problem(T + 16, 128, (T + 16) + (T + 16) // 4, 640, 1 / 24)
        if lib.dsa_bwd_workspace_bytes(ctypes.byref(nxt)) > NO_ALLOC_BYTES:
            break
        T += 16
    wh = WL.make("flash", T=T, H=128)
    w = wh.to(DEV)
    prob = dsa.make_problem(w.T, w.H, w.S_kv, w.W, w.scale)
    need = lib.dsa_bwd_workspace_bytes(ctypes.byref(prob))
    assert NO_ALLOC_BYTES // 2 < need <= NO_ALLOC_BYTES
    out, lse = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
    like = (torch.empty_like(w.q), torch.empty_like(w.kv), torch.empty_like(w.sink))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dq, dkv, ds = _no_alloc(lib, w, prob, out, lse, stream, like)
    g = O.backward(wh.q, wh.kv, wh.topk_idxs, wh.topk_length, wh.sink, wh.scale, wh.dout)
    counts = O.valid_lists(wh.topk_idxs, wh.topk_length, wh.S_kv)[1]
    check_bwd(dq, dkv, ds, g, counts)


def test_no_alloc_rejects_problems_beyond_the_array(lib):
    prob = dsa.make_problem(4096, 128, 5120, 640, 1 / 24)
    assert lib.dsa_bwd_workspace_bytes(ctypes.byref(prob)) > NO_ALLOC_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = lib.dsa_bwd_no_alloc(ctypes.byref(prob), fake, fake, fake, None, None, fake, fake, fake,
                              fake, fake, None, None)
    assert rc == 4  # DSA_ERR_WORKSPACE
    # what dsa_bwd rejects, rejected with the same status
    for kw, code in [(dict(H=129), 2), (dict(H=0), 1)]:
        T, H, S_kv, W = 16, kw["H"], 64, 32
        bad = dsa.make_problem(T, H, S_kv, W, 0.1)
        assert lib.dsa_bwd_no_alloc(ctypes.byref(bad), fake, fake, fake, None, None, fake, fake,
                                    fake, fake, fake, None, None) == code
