"""The Python binding's argument checks, on CPU.

The binding only marshals arguments: every tensor must be a contiguous CUDA
tensor of the documented dtype and shape, and anything else raises before the
library is called, so no call computes host tensors on the CPU instead.
"""
import math

import numpy as np
import pytest
import torch

from sparse_top_attention_gb300 import dsa

T, H, S_KV, W = 4, 16, 32, 8


def _host_inputs(d=576):
    q = torch.zeros(T, H, d, dtype=torch.bfloat16)
    kv = torch.zeros(S_KV, d, dtype=torch.bfloat16)
    idx = torch.zeros(T, W, dtype=torch.int32)
    sink = torch.zeros(H, dtype=torch.float32)
    return q, kv, idx, sink


@pytest.fixture
def no_library(monkeypatch):
    """Fails the test if the binding reaches for the CUDA library."""
    def _lib(*a, **k):
        raise AssertionError("the library was called")
    monkeypatch.setattr(dsa, "library", _lib)


def test_fwd_rejects_host_tensors(no_library):
    q, kv, idx, sink = _host_inputs()
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.fwd(q, kv, idx, None, sink)


def test_bwd_rejects_host_tensors(no_library):
    q, kv, idx, sink = _host_inputs()
    out = torch.zeros(T, H, 512, dtype=torch.bfloat16)
    lse = torch.zeros(T, H, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.bwd(q, kv, idx, None, sink, out, lse, out.clone())


def test_non_tensor_input_is_a_type_error(no_library):
    q, kv, idx, sink = _host_inputs()
    with pytest.raises(TypeError, match="torch.Tensor"):
        dsa.fwd(np.zeros((T, H, 576), np.float32), kv, idx, None, sink)


def test_default_scale_follows_the_row_width():
    for d in (576, 512):
        q, kv, idx, _ = _host_inputs(d)
        prob, dims = dsa._problem_from(q, kv, idx, None)
        assert dims == (T, H, S_KV, W) and prob.d_qk == d and prob.d_v == 512
        assert math.isclose(prob.scale, 1.0 / math.sqrt(d), rel_tol=1e-7)


def test_residual_buffer_must_have_room_for_both_halves():
    """With DSA_FLAG_DELTA_RESIDUAL the library writes 2*T*H*512 bf16 from
    out's first element on: out must be the first half of such a buffer."""
    both = torch.empty(2, T, H, 512, dtype=torch.bfloat16)
    dsa._need_residual_room(both[0], T, H)
    with pytest.raises(ValueError, match="first half"):
        dsa._need_residual_room(torch.empty(T, H, 512, dtype=torch.bfloat16), T, H)
    with pytest.raises(ValueError, match="first half"):
        dsa._need_residual_room(both[1], T, H)


def test_varlen_descriptor_checks_on_the_host():
    i32 = dict(dtype=torch.int32)
    with pytest.raises(ValueError, match="B \\+ 1"):
        dsa._varlen((torch.tensor([0], **i32), torch.tensor([0], **i32)), T, S_KV)
    with pytest.raises(ValueError, match="B \\+ 1"):
        dsa._varlen((torch.tensor([0, 2, 4], **i32), torch.tensor([0, 32], **i32)), T, S_KV)
    with pytest.raises(ValueError, match="int32 device tensor"):
        dsa._varlen((torch.tensor([0, 4], **i32), torch.tensor([0, 32], **i32)), T, S_KV)
