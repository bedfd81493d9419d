"""GPU parity at the limits of the sizes: no tokens, one token, the widest and
narrowest index rows, a single KV row, one head, a ragged head group
(H = 33), a head count that leaves a single real head in the last
64-head group of both the forward and the backward (H = 65), and last groups
that are partly filled (H = 48, 80, 112).  The widest rows
also run at 16 and 24 heads, where the forward uses its 16- and 32-head
instances, whose KV ring wraps many times within one item (16 blocks)."""
import numpy as np
import pytest
import torch

from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import check_bwd, check_fwd
from tests.test_gpu_parity import DEV, _lib, counts_of, oracle_exact, run  # noqa: F401

pytestmark = pytest.mark.gpu

CASES = [
    # T, H, S_kv, W, max_valid, compact
    ("one_token_widest_row", (1, 128, 4096, 2048, 1800, False)),
    ("widest_row_compact", (40, 64, 3000, 2048, 2048, True)),
    ("one_slot_per_token", (64, 16, 200, 1, 1, False)),
    ("one_kv_row", (48, 32, 1, 8, 1, False)),
    ("one_head", (256, 1, 700, 640, 600, False)),
    ("h33_ragged_head_group", (200, 33, 900, 300, 300, True)),
    ("h65_one_head_in_last_group", (200, 65, 900, 300, 300, False)),
    ("h128", (200, 128, 900, 300, 300, False)),
    ("h16_widest_rows", (64, 16, 3000, 2048, 2048, False)),
    ("h24_widest_rows_compact", (48, 24, 3000, 2048, 2048, True)),
    # partly filled last head groups: 48 of 64 heads; 16 and 48 real heads in
    # the second 64-head group (padded rows of k_bwd_dq's Q/dO tiles, and
    # k_bwd_dkv's 96- and 128-row head padding)
    ("h48_one_partial_group", (200, 48, 900, 300, 300, False)),
    ("h80_sixteen_heads_in_last_group", (160, 80, 900, 640, 600, True)),
    ("h112_forty_eight_heads_in_last_group", (160, 112, 900, 640, 600, False)),
]


@pytest.mark.parametrize("name,args", CASES, ids=[c[0] for c in CASES])
def test_limits_parity(name, args):
    T, H, S_kv, W, max_valid, compact = args
    w = WL.random_rows(T, H, S_kv, W, max_valid, seed=3000 + len(name), compact=compact)
    out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)


def test_no_tokens_is_a_no_op_that_clears_dkv():
    H, S_kv, W = 16, 50, 8
    q = torch.zeros(0, H, 576, dtype=torch.bfloat16, device=DEV)
    kv = torch.randn(S_kv, 576, device=DEV).to(torch.bfloat16)
    idx = torch.zeros(0, W, dtype=torch.int32, device=DEV)
    sink = torch.randn(H, device=DEV)
    out, lse = dsa.fwd(q, kv, idx, None, sink)
    assert out.shape == (0, H, 512) and lse.shape == (0, H)
    dout = torch.zeros(0, H, 512, dtype=torch.bfloat16, device=DEV)
    dkv = torch.full((S_kv, 576), 7.0, dtype=torch.bfloat16, device=DEV)
    dsink = torch.full((H,), 7.0, device=DEV)
    dsa.bwd(q, kv, idx, None, sink, out, lse, dout, dkv=dkv, dsink=dsink)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    assert (dkv == 0).all() and (dsink == 0).all()
