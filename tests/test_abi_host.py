"""libmoe loads and exports every declared symbol; host-side checks (no GPU).

Only argument, shape, alignment and workspace checks run here: they return
before the library touches a device.
"""
import ctypes
import os
import re

import pytest

import mxfp4_mixture_experts_route_gb300 as moe
from libmoe_util import ensure_built

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    return ensure_built()


def test_exports_match_header(L):
    decl = set(re.findall(r"^\s*(?:int|const char\*)\s+(moe_\w+)\s*\(", open(HEADER).read(), re.M))
    assert decl == set(moe.EXPORTS)
    for name in decl:
        assert hasattr(L, name), name


def test_version_and_strerror(L):
    assert moe.abi_version() == 1
    for code in range(0, -10, -1):
        assert moe.strerror(code) and moe.strerror(code) != "unknown status"
    assert moe.strerror(-99) == "unknown status"


def test_workspace_bytes(L):
    s = moe.MoEShape.of(8, 4096, 256, 8, 512)
    n = moe.workspace_bytes(s)
    assert n % 256 == 0 and n > 8 * 8 * (4096 * 2 + 512 * 2 + 4096 * 4)


@pytest.mark.parametrize("kw,code", [
    (dict(S=0), moe.MOE_ERR_INVALID_ARG),
    (dict(d=200), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(I=96), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(k=9, E=8), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(k=17, E=64), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(E=513), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(S=1 << 18, k=8), moe.MOE_ERR_UNSUPPORTED_SHAPE),
])
def test_bad_shapes(L, kw, code):
    base = dict(S=8, d=256, E=8, k=2, I=128)
    base.update(kw)
    s = moe.MoEShape.of(**base)
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == code


def test_bad_flags_and_null_shape(L):
    s = moe.MoEShape.of(8, 256, 8, 2, 128)
    s.flags = 8
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_bytes(None, ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG


def _route_call(L, s, x=0x1000, wg=0x2000, bias=0x3000, off=None, ids=0x4000, w=0x5000, ws=0x10000,
                nbytes=None):
    if nbytes is None:
        nbytes = moe.workspace_bytes(s)
    return L.moe_route(ctypes.byref(s), x, wg, bias, off, ids, w, ws, nbytes, None)


def test_route_arg_checks(L):
    s = moe.MoEShape.of(8, 256, 8, 2, 128)
    assert _route_call(L, s, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _route_call(L, s, x=0x1008) == moe.MOE_ERR_ALIGNMENT
    assert _route_call(L, s, ws=0x10080) == moe.MOE_ERR_ALIGNMENT
    assert _route_call(L, s, nbytes=1024) == moe.MOE_ERR_WORKSPACE
    s2 = moe.MoEShape.of(8, 256, 8, 2, 128, logit_offset=True)
    assert _route_call(L, s2, off=None) == moe.MOE_ERR_INVALID_ARG


def test_experts_and_forward_arg_checks(L):
    s = moe.MoEShape.of(8, 256, 8, 2, 128, post_norm=True)
    n = moe.workspace_bytes(s)
    good = [0x1000 * (i + 1) for i in range(10)]
    # norm weight missing with MOE_POST_NORM
    args = good[:8] + [None, good[9]]
    assert L.moe_experts(ctypes.byref(s), *args, 0x100000, n, None) == moe.MOE_ERR_INVALID_ARG
    args = good[:3] + [good[3] + 4] + good[4:]
    assert L.moe_experts(ctypes.byref(s), *args, 0x100000, n, None) == moe.MOE_ERR_ALIGNMENT
    fwd = [0x1000 * (i + 1) for i in range(13)]
    fwd[10] = None
    assert L.moe_forward(ctypes.byref(s), *fwd, 0x100000, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_device_status(None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_init(0x100008, 4096, None) == moe.MOE_ERR_ALIGNMENT


def test_no_device_is_reported_not_crashed(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    s = moe.MoEShape.of(8, 256, 8, 2, 128)
    assert _route_call(L, s) == moe.MOE_ERR_NO_DEVICE
