"""Python binding of the C ABI in ``include/dsa.h``: argument marshalling only.

Every step of the computation runs in the CUDA library.  This module does
three things only:
  - checks shapes, dtypes and devices;
  - allocates outputs and the workspace with torch when the caller passes
    none;
  - hands raw pointers and the current CUDA stream to the library.
If the library has not been built, every call raises.  There is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdsa.so")

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_ALIGNMENT",
    4: "DSA_ERR_WORKSPACE", 5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_TIMEOUT", 7: "DSA_ERR_RANGE",
}

# Every symbol that include/dsa.h declares.
EXPORTS = ("dsa_fwd", "dsa_bwd_workspace_bytes", "dsa_bwd", "dsa_bwd_preprocess", "dsa_bwd_main",
           "dsa_bwd_finalize", "dsa_bwd_no_alloc", "dsa_fwd_varlen", "dsa_bwd_varlen",
           "dsa_topk_compact", "dsa_device_status", "dsa_wait_selftest", "dsa_status_string",
           "dsa_version")
BWD_STAGES = ("dsa_bwd_preprocess", "dsa_bwd_main", "dsa_bwd_finalize")
FLAG_DELTA_RESIDUAL = 1
FLAG_DETERMINISTIC = 2


class Varlen(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("cu_seqlens_q", ctypes.c_void_p),
                ("cu_seqlens_kv", ctypes.c_void_p)]


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("S_kv", ctypes.c_int32),
                ("W", ctypes.c_int32), ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("scale", ctypes.c_float), ("flags", ctypes.c_uint32)]


class DsaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({_lib_status_string(code)})")
        self.code = code


_lib = None


def library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(p)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    prob = ctypes.POINTER(Problem)
    lib.dsa_fwd.argtypes = [prob, vp, vp, i32p, i32p, f32p, vp, f32p, vp]
    lib.dsa_fwd.restype = ctypes.c_int
    lib.dsa_bwd_workspace_bytes.argtypes = [prob]
    lib.dsa_bwd_workspace_bytes.restype = ctypes.c_size_t
    for name in ("dsa_bwd",) + BWD_STAGES:
        fn = getattr(lib, name)
        fn.argtypes = [prob, vp, vp, i32p, i32p, f32p, vp, f32p, vp, vp, vp, f32p, vp,
                       ctypes.c_size_t, vp]
        fn.restype = ctypes.c_int
    lib.dsa_bwd_no_alloc.argtypes = [prob, vp, vp, i32p, i32p, f32p, vp, f32p, vp, vp, vp, f32p,
                                     vp]
    lib.dsa_bwd_no_alloc.restype = ctypes.c_int
    vl = ctypes.POINTER(Varlen)
    lib.dsa_fwd_varlen.argtypes = [prob, vl, vp, vp, i32p, i32p, f32p, vp, f32p, vp]
    lib.dsa_fwd_varlen.restype = ctypes.c_int
    lib.dsa_bwd_varlen.argtypes = [prob, vl, vp, vp, i32p, i32p, f32p, vp, f32p, vp, vp, vp, f32p,
                                   vp, ctypes.c_size_t, vp]
    lib.dsa_bwd_varlen.restype = ctypes.c_int
    lib.dsa_topk_compact.argtypes = [prob, i32p, i32p, i32p, i32p, vp]
    lib.dsa_topk_compact.restype = ctypes.c_int
    lib.dsa_device_status.argtypes = [vp]
    lib.dsa_device_status.restype = ctypes.c_int
    lib.dsa_wait_selftest.argtypes = [ctypes.c_uint32, vp]
    lib.dsa_wait_selftest.restype = ctypes.c_int
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_version.argtypes = []
    lib.dsa_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _lib_status_string(code: int) -> str:
    try:
        return library().dsa_status_string(code).decode()
    except Exception:  # pragma: no cover - only used in error messages
        return "?"


def _ptr(x: Optional[torch.Tensor]):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, what: str):
    if code != 0:
        raise DsaError(code, what)


def make_problem(T, H, S_kv, W, scale, flags=0, d_qk=576) -> Problem:
    return Problem(int(T), int(H), int(S_kv), int(W), int(d_qk), 512, float(scale), int(flags))


def _need(x: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")


def _problem_from(q, kv, topk_idxs, scale, flags=0):
    """The problem of these tensors; q's last dimension is d_qk (576 or 512)."""
    T, H, d_qk = q.shape
    S_kv = kv.shape[0]
    W = topk_idxs.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d_qk)
    return make_problem(T, H, S_kv, W, scale, flags, d_qk), (T, H, S_kv, W)


def _need_residual_room(out, T, H):
    """With DSA_FLAG_DELTA_RESIDUAL the library reads/writes 2*T*H*512 bf16
    starting at out.data_ptr(): `out` must be the first half of such a buffer."""
    need = 2 * T * H * 512 * 2
    st = out.untyped_storage()
    have = st.nbytes() - (out.data_ptr() - st.data_ptr())
    if have < need:
        raise ValueError("delta_residual needs out to be the first half of a [2, T, H, 512] "
                         "bf16 buffer (e.g. the `out` returned by fwd(..., delta_residual=True))")


def _varlen(varlen, T, S_kv):
    """(cu_seqlens_q, cu_seqlens_kv) device int32 tensors -> a Varlen struct."""
    cu_q, cu_kv = varlen
    B = cu_q.numel() - 1
    if B < 1 or cu_kv.numel() != B + 1:
        raise ValueError("varlen needs cu_seqlens_q and cu_seqlens_kv of B + 1 >= 2 entries")
    for x, n in ((cu_q, "cu_seqlens_q"), (cu_kv, "cu_seqlens_kv")):
        if x.dtype != torch.int32 or not x.is_cuda or not x.is_contiguous():
            raise ValueError(f"{n}: contiguous int32 device tensor expected")
    return Varlen(B, cu_q.data_ptr(), cu_kv.data_ptr())


def fwd(q, kv, topk_idxs, topk_length=None, sink=None, scale=None, out=None, lse=None,
        stream=None, delta_residual=False, varlen=None):
    """Sparse MLA forward.  Returns (out bf16 [T,H,512], lse fp32 [T,H]).

    With ``delta_residual`` the output is the first half of a [2,T,H,512]
    buffer whose second half holds the rounding residual that the backward
    uses for an exact delta (DSA_FLAG_DELTA_RESIDUAL).  ``varlen`` =
    (cu_seqlens_q, cu_seqlens_kv) selects dsa_fwd_varlen: packed sequences
    whose indices count from their own first KV row."""
    prob, (T, H, S_kv, W) = _problem_from(q, kv, topk_idxs, scale,
                                          FLAG_DELTA_RESIDUAL if delta_residual else 0)
    D = prob.d_qk
    _need(q, "q", torch.bfloat16, (T, H, D))
    _need(kv, "kv", torch.bfloat16, (S_kv, D))
    _need(topk_idxs, "topk_idxs", torch.int32, (T, W))
    if topk_length is not None:
        _need(topk_length, "topk_length", torch.int32, (T,))
    if sink is not None:
        _need(sink, "sink", torch.float32, (H,))
    if out is None:
        if delta_residual:
            out = torch.empty(2, T, H, 512, dtype=torch.bfloat16, device=q.device)[0]
        else:
            out = torch.empty(T, H, 512, dtype=torch.bfloat16, device=q.device)
    if delta_residual:
        _need_residual_room(out, T, H)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, (T, H, 512))
    _need(lse, "lse", torch.float32, (T, H))
    if varlen is not None:
        vl = _varlen(varlen, T, S_kv)
        _check(library().dsa_fwd_varlen(ctypes.byref(prob), ctypes.byref(vl), _ptr(q), _ptr(kv),
                                        _ptr(topk_idxs), _ptr(topk_length), _ptr(sink), _ptr(out),
                                        _ptr(lse), _stream(stream)),
               "dsa_fwd_varlen")
        return out, lse
    _check(library().dsa_fwd(ctypes.byref(prob), _ptr(q), _ptr(kv), _ptr(topk_idxs),
                             _ptr(topk_length), _ptr(sink), _ptr(out), _ptr(lse), _stream(stream)),
           "dsa_fwd")
    return out, lse


def bwd_workspace_bytes(T, H, S_kv, W, scale=1.0 / 24.0, deterministic=False, d_qk=576) -> int:
    prob = make_problem(T, H, S_kv, W, scale, FLAG_DETERMINISTIC if deterministic else 0, d_qk)
    return int(library().dsa_bwd_workspace_bytes(ctypes.byref(prob)))


def bwd(q, kv, topk_idxs, topk_length, sink, out, lse, dout, scale=None, dq=None, dkv=None,
        dsink=None, workspace=None, stream=None, entry="dsa_bwd", delta_residual=False,
        deterministic=False, varlen=None):
    """Sparse MLA backward.  Returns (dq bf16, dkv bf16, dsink fp32 or None).

    ``entry`` selects ``dsa_bwd`` (all stages) or one of ``BWD_STAGES``.
    ``delta_residual`` must match the forward call that produced ``out``.
    ``deterministic`` (DSA_FLAG_DETERMINISTIC) makes dkv bitwise reproducible;
    a caller-provided workspace must then be sized with the same flag.
    ``varlen`` = (cu_seqlens_q, cu_seqlens_kv) selects dsa_bwd_varlen (all
    stages in one call)."""
    flags = (FLAG_DELTA_RESIDUAL if delta_residual else 0) | \
        (FLAG_DETERMINISTIC if deterministic else 0)
    prob, (T, H, S_kv, W) = _problem_from(q, kv, topk_idxs, scale, flags)
    D = prob.d_qk
    _need(q, "q", torch.bfloat16, (T, H, D))
    _need(kv, "kv", torch.bfloat16, (S_kv, D))
    _need(topk_idxs, "topk_idxs", torch.int32, (T, W))
    if topk_length is not None:
        _need(topk_length, "topk_length", torch.int32, (T,))
    if sink is not None:
        _need(sink, "sink", torch.float32, (H,))
    _need(out, "out", torch.bfloat16, (T, H, 512))
    _need(lse, "lse", torch.float32, (T, H))
    _need(dout, "dout", torch.bfloat16, (T, H, 512))
    if delta_residual:
        _need_residual_room(out, T, H)
    dev = q.device
    if dq is None:
        dq = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    if dkv is None:
        dkv = torch.empty(S_kv, D, dtype=torch.bfloat16, device=dev)
    if sink is not None and dsink is None:
        dsink = torch.empty(H, dtype=torch.float32, device=dev)
    nbytes = int(library().dsa_bwd_workspace_bytes(ctypes.byref(prob)))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if entry != "dsa_bwd" and entry not in BWD_STAGES:
        raise ValueError(entry)
    if varlen is not None:
        if entry != "dsa_bwd":
            raise ValueError("varlen runs all backward stages in one call")
        vl = _varlen(varlen, T, S_kv)
        _check(library().dsa_bwd_varlen(ctypes.byref(prob), ctypes.byref(vl), _ptr(q), _ptr(kv),
                                        _ptr(topk_idxs), _ptr(topk_length), _ptr(sink), _ptr(out),
                                        _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dkv), _ptr(dsink),
                                        _ptr(workspace),
                                        ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                        _stream(stream)),
               "dsa_bwd_varlen")
        return dq, dkv, dsink
    _check(getattr(library(), entry)(ctypes.byref(prob), _ptr(q), _ptr(kv), _ptr(topk_idxs),
                             _ptr(topk_length), _ptr(sink), _ptr(out), _ptr(lse), _ptr(dout),
                             _ptr(dq), _ptr(dkv), _ptr(dsink), _ptr(workspace),
                             ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                             _stream(stream)),
           entry)
    return dq, dkv, dsink


def topk_compact(topk_idxs, topk_length, S_kv, stream=None):
    """Valid KV rows per token in slot order, and their counts (device tensors)."""
    T, W = topk_idxs.shape
    _need(topk_idxs, "topk_idxs", torch.int32, (T, W))
    if topk_length is not None:
        _need(topk_length, "topk_length", torch.int32, (T,))
    prob = make_problem(T, 1, S_kv, W, 1.0)
    idx_out = torch.full((T, W), -1, dtype=torch.int32, device=topk_idxs.device)
    count = torch.empty(T, dtype=torch.int32, device=topk_idxs.device)
    _check(library().dsa_topk_compact(ctypes.byref(prob), _ptr(topk_idxs), _ptr(topk_length),
                                      _ptr(idx_out), _ptr(count), _stream(stream)),
           "dsa_topk_compact")
    return idx_out, count


def wait_selftest(limit_us: int, stream=None) -> None:
    """Queue the bounded-wait self-test (dsa_wait_selftest): a kernel whose
    barrier waits run out after ``limit_us`` microseconds.  The next
    ``device_status`` returns DSA_ERR_DEVICE_TIMEOUT."""
    _check(library().dsa_wait_selftest(int(limit_us), _stream(stream)), "dsa_wait_selftest")


def device_status(stream=None) -> int:
    """Synchronise the stream and return the library's device status code."""
    return int(library().dsa_device_status(_stream(stream)))
