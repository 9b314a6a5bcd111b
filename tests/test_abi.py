"""The C ABI without a GPU: the library loads, exports every function the header
declares, rejects bad arguments on the host before any CUDA call, and sizes its
workspace."""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_flashattention_varlen_gb300 import _lib, build as pkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkbuild.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    assert "pattn_forward" in names and "pattn_workspace_size" in names
    assert set(names) == set(_lib.SIGNATURES), names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


ALIGNED = 1 << 20  # fake, aligned, never dereferenced: validation returns first


def fwd(lib, **kw):
    a = dict(out=ALIGNED, q=ALIGNED, kv=ALIGNED, bt=ALIGNED, sl=ALIGNED, cu=ALIGNED, B=2, tq=16,
             mq=8, mkv=650, hq=24, hkv=4, d=256, P=64, pages=22, scale=0.0625, causal=1)
    a.update(kw)
    return lib.pattn_forward(a["out"], a["q"], a["kv"], a["bt"], a["sl"], a["cu"], a["B"], a["tq"],
                             a["mq"], a["mkv"], a["hq"], a["hkv"], a["d"], a["P"], a["pages"],
                             a["scale"], a["causal"], None)


def test_host_validation(lib):
    INVALID, UNSUP = 1, 2
    assert fwd(lib, out=None) == INVALID
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, kv=ALIGNED + 8) == INVALID          # not 16-byte aligned
    assert fwd(lib, sl=ALIGNED + 2) == INVALID
    assert fwd(lib, hq=25) == INVALID                   # not a multiple of the kv heads
    assert fwd(lib, hkv=0) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, pages=0) == INVALID
    assert fwd(lib, causal=2) == INVALID
    assert fwd(lib, scale=float("nan")) == INVALID
    assert fwd(lib, scale=float("inf")) == INVALID
    assert fwd(lib, scale=-1.0) == UNSUP
    assert fwd(lib, d=64) == UNSUP
    assert fwd(lib, P=32) == UNSUP
    assert fwd(lib, hq=258, hkv=1) == UNSUP             # group above 128 rows
    assert fwd(lib, mkv=64 * 65536) == UNSUP            # KV tiles beyond the 16-bit item field
    assert fwd(lib, B=0) == 0 and fwd(lib, tq=0) == 0   # nothing to do


def append(lib, k=ALIGNED, v=ALIGNED, **kw):
    a = dict(out=ALIGNED, q=ALIGNED, kv=ALIGNED, bt=ALIGNED, sl=ALIGNED, cu=ALIGNED, B=2, tq=16,
             mq=8, mkv=650, hq=24, hkv=4, d=256, P=64, pages=22, scale=0.0625, causal=1)
    a.update(kw)
    return lib.pattn_forward_append(a["out"], a["q"], k, v, a["kv"], a["bt"], a["sl"], a["cu"], a["B"],
                                    a["tq"], a["mq"], a["mkv"], a["hq"], a["hkv"], a["d"], a["P"],
                                    a["pages"], a["scale"], a["causal"], None)


def test_append_host_validation(lib):
    INVALID = 1
    assert append(lib, k=None) == INVALID
    assert append(lib, v=None) == INVALID
    assert append(lib, k=ALIGNED + 4) == INVALID        # not 16-byte aligned
    assert append(lib, kv=None) == INVALID
    assert append(lib, hq=25) == INVALID
    assert append(lib, k=None, tq=0) == 0               # nothing to write or attend


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must not reach a GPU")
def test_valid_call_without_a_gpu_reports_cuda_error(lib):
    assert fwd(lib) == 3
    assert append(lib) == 3


def test_workspace_size(lib):
    ws = lib.pattn_workspace_size
    small = ws(2, 16, 8, 650, 24, 4, 256, 64)
    big = ws(64, 64, 1, 8192, 32, 8, 128, 64)
    assert small > 0 and big > 0
    assert ws(128, 128, 1, 8192, 32, 8, 128, 64) > big
    assert ws(2, 16, 8, 650, 24, 5, 256, 64) == 0
    assert ws(2, 16, 8, 650, 24, 4, 64, 64) == 0


def test_status_strings(lib):
    for code in range(7):
        assert lib.pattn_status_string(code)
    assert b"unknown" in lib.pattn_status_string(99)


def test_plan_items_host_validation(lib):
    INVALID, UNSUP = 1, 2
    counts = (ctypes.c_int32 * 4)()
    buf = (ctypes.c_int32 * 16)()

    def plan(**kw):
        a = dict(bt=ALIGNED, sl=ALIGNED, cu=ALIGNED, B=2, tq=16, mq=8, mkv=650, hq=24, hkv=4, d=256, P=64,
                 pages=22, causal=1, pre=ctypes.addressof(buf), dec=ctypes.addressof(buf), cap=4,
                 counts=ctypes.addressof(counts))
        a.update(kw)
        return lib.pattn_plan_items(a["bt"], a["sl"], a["cu"], a["B"], a["tq"], a["mq"], a["mkv"], a["hq"],
                                    a["hkv"], a["d"], a["P"], a["pages"], a["causal"], a["pre"], a["dec"],
                                    a["cap"], a["counts"], None)

    assert plan(sl=None) == INVALID
    assert plan(cu=ALIGNED + 2) == INVALID
    assert plan(hq=25) == INVALID
    assert plan(d=64) == UNSUP
    assert plan(P=32) == UNSUP
    assert plan(counts=None) == INVALID
    assert plan(cap=-1) == INVALID
    assert plan(pre=None) == INVALID
    # an empty batch needs no device: zero counts
    counts[0] = 7
    assert plan(B=0, tq=0) == 0 and list(counts) == [0, 0, 0, 0]
