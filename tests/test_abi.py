"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/dsa.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from sparse_top_attention_gb300 import build as B
from sparse_top_attention_gb300 import dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return dsa.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(dsa.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.dsa_version() == 100
    for code in range(8):
        assert len(lib.dsa_status_string(code)) > 0


def P(**kw):
    d = dict(T=4, H=16, S_kv=8, W=4, d_qk=576, d_v=512, scale=0.1, flags=0)
    d.update(kw)
    return dsa.Problem(**d)


def test_workspace_size_is_pure_host(lib):
    p = P(T=4096, H=128, S_kv=5120, W=640)
    n = lib.dsa_bwd_workspace_bytes(ctypes.byref(p))
    assert n >= 5120 * 576 * 4 + 4096 * 640 * 4 + 4 * 4096 * 128 * 4
    assert n % 256 == 0
    assert lib.dsa_bwd_workspace_bytes(ctypes.byref(P(H=0))) == 0
    # DSA_FLAG_DETERMINISTIC keeps dkv as int64 (4 more bytes per accumulator
    # element) plus one u32 per KV row and one word for its range check
    nd = lib.dsa_bwd_workspace_bytes(ctypes.byref(P(T=4096, H=128, S_kv=5120, W=640, flags=2)))
    assert nd - n == 5120 * 576 * 4 + 5120 * 4 + 256


@pytest.mark.parametrize("kw,code", [
    (dict(H=0), 1), (dict(H=129), 2), (dict(T=-1), 1), (dict(W=0), 1), (dict(S_kv=0), 1),
    (dict(d_qk=256), 2), (dict(d_v=576), 2), (dict(flags=4), 1), (dict(scale=float("nan")), 1),
    (dict(W=4096), 2), (dict(S_kv=3728271), 2),
])
def test_forward_rejects_before_launch(lib, kw, code):
    p = P(**kw)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    r = lib.dsa_fwd(ctypes.byref(p), fake, fake, fake, None, None, fake, fake, None)
    assert r == code


def test_null_and_misaligned_pointers_rejected(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    assert lib.dsa_fwd(ctypes.byref(p), None, a, a, None, None, a, a, None) == 1
    mis = ctypes.c_void_p((1 << 20) + 4)
    assert lib.dsa_fwd(ctypes.byref(p), mis, a, a, None, None, a, a, None) == 3
    # T = 0 is a no-op that launches nothing
    assert lib.dsa_fwd(ctypes.byref(P(T=0)), None, None, None, None, None, None, None, None) == 0


def test_backward_argument_checks(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    n = lib.dsa_bwd_workspace_bytes(ctypes.byref(p))
    # sink given but no dsink
    assert lib.dsa_bwd(ctypes.byref(p), a, a, a, None, a, a, a, a, a, a, None, a, n, None) == 1
    # workspace too small
    assert lib.dsa_bwd(ctypes.byref(p), a, a, a, None, None, a, a, a, a, a, None, a, n - 1, None) == 4
    # workspace misaligned
    w = ctypes.c_void_p((1 << 20) + 16)
    assert lib.dsa_bwd(ctypes.byref(p), a, a, a, None, None, a, a, a, a, a, None, w, n, None) == 3


@pytest.mark.parametrize("kw,code", [
    (dict(H=129), 2), (dict(d_qk=640), 2), (dict(S_kv=3728271), 2), (dict(H=0), 1),
    (dict(flags=8), 1),
])
def test_no_alloc_passes_the_check_status_through(lib, kw, code):
    """dsa_bwd_no_alloc validates a problem as dsa_bwd does and returns the
    same status (not a generic one), before it touches the device."""
    p = P(**kw)
    a = ctypes.c_void_p(1 << 20)
    n = ctypes.c_size_t(1 << 30)
    assert lib.dsa_bwd(ctypes.byref(p), a, a, a, None, None, a, a, a, a, a, None, a, n,
                       None) == code
    assert lib.dsa_bwd_no_alloc(ctypes.byref(p), a, a, a, None, None, a, a, a, a, a, None,
                                None) == code


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        dsa.library(str(tmp_path / "missing.so"))


def test_varlen_descriptor_checks(lib):
    """dsa_fwd_varlen / dsa_bwd_varlen reject a bad batch descriptor before
    any launch (the offsets themselves are never read on the host)."""
    p = P(T=4, H=16, S_kv=8, W=4)
    fake = ctypes.c_void_p(1 << 20)
    a4 = ctypes.c_void_p(1 << 21)
    assert lib.dsa_fwd_varlen(ctypes.byref(p), None, fake, fake, fake, None, None, fake, fake,
                              None) == 1
    for v, code in [(dsa.Varlen(0, a4.value, a4.value), 1), (dsa.Varlen(2, None, a4.value), 1),
                    (dsa.Varlen(2, a4.value, None), 1),
                    (dsa.Varlen(2, (1 << 21) + 2, a4.value), 3)]:
        assert lib.dsa_fwd_varlen(ctypes.byref(p), ctypes.byref(v), fake, fake, fake, None, None,
                                  fake, fake, None) == code
        assert lib.dsa_bwd_varlen(ctypes.byref(p), ctypes.byref(v), fake, fake, fake, None, None,
                                  fake, fake, fake, fake, fake, None, fake, ctypes.c_size_t(0),
                                  None) == code
