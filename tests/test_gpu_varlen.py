"""GPU parity of the varlen entry points (dsa_fwd_varlen, dsa_bwd_varlen)
against the oracle's varlen batches, element by element."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import REL_TOL, check_bwd, check_fwd
from tests.test_gpu_parity import DEV, _lib  # noqa: F401
from tests.test_oracle_varlen import _with_out_of_sequence_indices

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, H, top-k, compact, seed
    ([200, 0, 333, 64], 64, 64, True, 11),
    ([200, 0, 333, 64], 64, 64, False, 12),
    ([700, 300], 128, 512, False, 13),     # 640 slots, several 128-row blocks
    ([1, 130, 2, 257], 24, 128, True, 14),  # ragged tails, padded head group
    ([600, 0, 250], 16, 512, False, 16),    # the 16-head forward, its KV ring wrapping
]


def run_varlen(w):
    wd = w.to(DEV)
    vl = (wd.cu_seqlens_q, wd.cu_seqlens_kv)
    out, lse = dsa.fwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, wd.scale, varlen=vl)
    dq, dkv, dsink = dsa.bwd(wd.q, wd.kv, wd.topk_idxs, wd.topk_length, wd.sink, out, lse,
                             wd.dout, wd.scale, varlen=vl)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    return out, lse, dq, dkv, dsink


def oracle_varlen(w):
    ref = O.forward_varlen(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale,
                           w.cu_seqlens_q, w.cu_seqlens_kv)
    g = O.backward_varlen(w.q, w.kv, w.topk_idxs, w.topk_length, w.sink, w.scale, w.dout,
                          w.cu_seqlens_q, w.cu_seqlens_kv)
    return ref, g


@pytest.mark.parametrize("lengths,H,topk,compact,seed", CASES)
def test_varlen_parity(lengths, H, topk, compact, seed):
    w = _with_out_of_sequence_indices(WL.varlen(lengths, H=H, topk=topk, compact=compact,
                                                seed=seed))
    out, lse, dq, dkv, dsink = run_varlen(w)
    ref, g = oracle_varlen(w)
    check_fwd(out, lse, ref, ref["count"])
    check_bwd(dq, dkv, dsink, g, ref["count"])


def test_varlen_sequence_without_kv_rows():
    """A sequence whose KV range is empty: every slot of its tokens is
    invalid, so its rows are empty (out 0, lse -FLT_MAX, dq 0)."""
    w = WL.varlen([90, 120], H=16, topk=64, compact=False, seed=15)
    ck = w.cu_seqlens_kv.tolist()
    # drop sequence 0's rows from its range; they stay in the packed tensor
    w.cu_seqlens_kv = torch.tensor([0, 0, ck[2]], dtype=torch.int32)
    out, lse, dq, dkv, dsink = run_varlen(w)
    ref, g = oracle_varlen(w)
    assert (ref["count"][:90] == 0).all()
    check_fwd(out, lse, ref, ref["count"])
    check_bwd(dq, dkv, dsink, g, ref["count"])
    np.testing.assert_array_equal(dq[:90].float().cpu().numpy(), 0.0)
