"""dsa_bwd_no_alloc: the backward that allocates nothing, for callers that
cannot allocate device memory at call time (a plain C program holding only
its inputs and outputs; a serving loop under a fixed memory budget where a
cudaMalloc would synchronise the device).

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.  The test calls the entry point through
the C ABI twice in a row.  Each time its outputs must match those of dsa_bwd
(same kernels, workspace from torch): dq and d_sink exactly, and dkv up to
the one-ulp bf16 flips that the order of fp32 atomics allows, the bound the
other repeat-launch tests use.  A problem whose workspace exceeds the fixed
64 MiB array must be rejected before anything launches.
"""
import ctypes

import pytest
import torch

from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import rel_frob

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


def test_no_alloc_backward_matches_workspace_backward(lib):
    w = WL.make("flash", T=128, H=128).to(DEV)
    prob = dsa.make_problem(w.T, w.H, w.S_kv, w.W, w.scale)
    assert 0 < lib.dsa_bwd_workspace_bytes(ctypes.byref(prob)) <= NO_ALLOC_BYTES
    out, lse = dsa.fwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale)
    dq0, dkv0, ds0 = dsa.bwd(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, out, lse, w.dout,
                             w.scale)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dq = torch.full_like(dq0, float("nan"))
        dkv = torch.full_like(dkv0, float("nan"))
        ds = torch.full_like(ds0, float("nan"))
        rc = lib.dsa_bwd_no_alloc(ctypes.byref(prob), _p(w.q), _p(w.kv), _p(w.topk_idxs),
                                  _p(w.topk_length), _p(w.sink), _p(out), _p(lse), _p(w.dout),
                                  _p(dq), _p(dkv), _p(ds), stream)
        assert rc == 0, dsa.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert dsa.device_status() == 0
        assert torch.equal(dq, dq0)
        assert torch.equal(ds, ds0)
        assert torch.isfinite(dkv.float()).all()
        assert rel_frob(dkv, dkv0) <= 1e-3


def test_no_alloc_rejects_problems_beyond_the_array(lib):
    prob = dsa.make_problem(4096, 128, 5120, 640, 1 / 24)
    assert lib.dsa_bwd_workspace_bytes(ctypes.byref(prob)) > NO_ALLOC_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = lib.dsa_bwd_no_alloc(ctypes.byref(prob), fake, fake, fake, None, None, fake, fake, fake,
                              fake, fake, None, None)
    assert rc == 4  # DSA_ERR_WORKSPACE
