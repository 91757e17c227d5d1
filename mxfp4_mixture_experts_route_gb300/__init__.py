"""Python binding of libmoe, the routed MXFP4 mixture-of-experts block on GB300.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  Tensors are PyTorch CUDA tensors (device memory and streams come from
PyTorch); the calls are the C entry points of include/moe.h under the same
names without the ``moe_`` prefix.  There is no CPU fallback: if libmoe.so is
missing, importing the binding's entry points raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_ALIGNMENT = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_CUDA = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_BAD_IDS = -7
MOE_ERR_BAD_SCALE = -8
MOE_ERR_NO_DEVICE = -9

MOE_POST_NORM = 1
MOE_LOGIT_OFFSET = 2

# every symbol include/moe.h declares
EXPORTS = ("moe_abi_version", "moe_strerror", "moe_workspace_bytes", "moe_workspace_init",
           "moe_route", "moe_experts", "moe_forward", "moe_forward_host", "moe_device_status",
           "moe_timing_enable", "moe_timing_collect", "moe_kernel_name", "moe_forward_noalloc",
           "moe_workspace_region", "moe_latent_workspace_bytes", "moe_latent_forward")

# workspace regions (moe_workspace_region)
MOE_WS_STATUS, MOE_WS_POS, MOE_WS_TILES, MOE_WS_XQ, MOE_WS_XS, MOE_WS_HQ, MOE_WS_HS, MOE_WS_Y, MOE_WS_LOGITS = range(9)


class MoEShape(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("norm_eps", ctypes.c_float)]

    @classmethod
    def of(cls, S, d, E, k, I, post_norm=False, logit_offset=False, norm_eps=1e-6):
        flags = (MOE_POST_NORM if post_norm else 0) | (MOE_LOGIT_OFFSET if logit_offset else 0)
        return cls(S, d, E, k, I, flags, norm_eps)


class LatentShape(ctypes.Structure):
    """moe_latent_shape: the latent-MoE layer around the routed block."""
    _fields_ = [("S", ctypes.c_int32), ("H", ctypes.c_int32), ("LAT", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("I", ctypes.c_int32),
                ("SI", ctypes.c_int32), ("flags", ctypes.c_uint32), ("norm_eps", ctypes.c_float)]

    @classmethod
    def of(cls, S, H, LAT, E, k, I, SI, logit_offset=False, norm_eps=1e-6):
        return cls(S, H, LAT, E, k, I, SI, MOE_LOGIT_OFFSET if logit_offset else 0, norm_eps)


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str, detail: int | None = None):
        self.code = code
        self.detail = detail
        msg = f"{where}: {strerror(code)} ({code})"
        if detail is not None:
            msg += f", detail {detail}"
        super().__init__(msg)


_lib = None

_P = ctypes.c_void_p
_SP = ctypes.POINTER(MoEShape)


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = load_library(LIB_PATH)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """A build of the library at `path` with the entry points' C types set."""
    L = ctypes.CDLL(path)
    L.moe_abi_version.restype = ctypes.c_int
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_strerror.argtypes = [ctypes.c_int]
    L.moe_workspace_bytes.argtypes = [_SP, ctypes.POINTER(ctypes.c_size_t)]
    L.moe_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
    L.moe_route.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.moe_experts.argtypes = [_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.moe_forward.argtypes = [_SP] + [_P] * 13 + [ctypes.c_size_t, _P]
    L.moe_forward_host.argtypes = [_SP] + [_P] * 13 + [ctypes.c_size_t, _P]
    L.moe_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
    L.moe_forward_noalloc.argtypes = [_SP] + [_P] * 14
    L.moe_workspace_region.argtypes = [_SP, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                                       ctypes.POINTER(ctypes.c_size_t)]
    _LSP = ctypes.POINTER(LatentShape)
    L.moe_latent_workspace_bytes.argtypes = [_LSP, ctypes.POINTER(ctypes.c_size_t)]
    L.moe_latent_forward.argtypes = [_LSP] + [_P] * 17 + [ctypes.c_size_t, _P]
    L.moe_timing_enable.argtypes = [ctypes.c_int]
    L.moe_timing_collect.argtypes = [_P, _P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    L.moe_kernel_name.argtypes = [ctypes.c_int]
    L.moe_kernel_name.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("moe_strerror", "moe_kernel_name"):
            getattr(L, name).restype = ctypes.c_int
    return L


def strerror(code: int) -> str:
    try:
        return lib().moe_strerror(code).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, where: str) -> None:
    if rc != MOE_OK:
        raise MoEError(rc, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def abi_version() -> int:
    return lib().moe_abi_version()


def workspace_bytes(shape: MoEShape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def workspace_region(shape: MoEShape, region: int) -> tuple[int, int]:
    """(byte offset, bytes) of one workspace region (MOE_WS_*)."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().moe_workspace_region(ctypes.byref(shape), region, ctypes.byref(off), ctypes.byref(n)),
           "moe_workspace_region")
    return off.value, n.value


def read_region(shape: MoEShape, ws, region: int, dtype=None):
    """A CPU copy of one workspace region (after the stream has finished): a
    uint8 tensor, viewed as `dtype` when given."""
    off, n = workspace_region(shape, region)
    t = ws[off:off + n].cpu()
    return t if dtype is None else t.view(dtype)


def new_workspace(shape: MoEShape, device="cuda", stream=None):
    """A device workspace (uint8 tensor, 256-byte aligned) prepared by moe_workspace_init."""
    import torch
    nbytes = workspace_bytes(shape)
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    ws = buf[off:off + nbytes]
    _check(lib().moe_workspace_init(ws.data_ptr(), nbytes, _stream(stream)), "moe_workspace_init")
    return ws


def route(shape, x, w_gate, bias, logit_off, ids, weights, ws, stream=None) -> None:
    _check(lib().moe_route(ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logit_off),
                           _ptr(ids), _ptr(weights), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")


def experts(shape, x, ids, weights, w13, w13s, w2, w2s, norm_w, out, ws, stream=None) -> None:
    _check(lib().moe_experts(ctypes.byref(shape), _ptr(x), _ptr(ids), _ptr(weights), _ptr(w13),
                             _ptr(w13s), _ptr(w2), _ptr(w2s), _ptr(norm_w), _ptr(out), _ptr(ws),
                             ws.numel(), _stream(stream)), "moe_experts")


def forward(shape, x, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids, weights, out, ws,
            stream=None) -> None:
    _check(lib().moe_forward(ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logit_off),
                             _ptr(w13), _ptr(w13s), _ptr(w2), _ptr(w2s), _ptr(norm_w), _ptr(ids),
                             _ptr(weights), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward")


def forward_host(shape, x_host, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w, ids_host,
                 weights_host, out_host, ws, stream=None) -> None:
    """x_host / ids_host / weights_host / out_host are (pinned) CPU tensors."""
    _check(lib().moe_forward_host(ctypes.byref(shape), _ptr(x_host), _ptr(w_gate), _ptr(bias),
                                  _ptr(logit_off), _ptr(w13), _ptr(w13s), _ptr(w2), _ptr(w2s),
                                  _ptr(norm_w), _ptr(ids_host), _ptr(weights_host), _ptr(out_host),
                                  _ptr(ws), ws.numel(), _stream(stream)), "moe_forward_host")


def latent_workspace_bytes(shape: LatentShape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_latent_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)), "moe_latent_workspace_bytes")
    return n.value


def latent_forward(shape, x, w_gate, bias, logit_off, w_ld, w13, w13s, w2, w2s, ln_w, w_up, w_sgu, w_sd,
                   ids, weights, out, ws, stream=None) -> None:
    _check(lib().moe_latent_forward(ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logit_off),
                                    _ptr(w_ld), _ptr(w13), _ptr(w13s), _ptr(w2), _ptr(w2s), _ptr(ln_w),
                                    _ptr(w_up), _ptr(w_sgu), _ptr(w_sd), _ptr(ids), _ptr(weights), _ptr(out),
                                    _ptr(ws), ws.numel(), _stream(stream)), "moe_latent_forward")


def device_status(ws, stream=None) -> tuple[int, int]:
    """(status, detail) latched on the device since the last call; clears it."""
    det = ctypes.c_int32(0)
    rc = lib().moe_device_status(_ptr(ws), ctypes.byref(det), _stream(stream))
    return rc, det.value


def check_device_status(ws, where="device", stream=None) -> None:
    rc, det = device_status(ws, stream)
    if rc != MOE_OK:
        raise MoEError(rc, where, det)


def timing_enable(max_launches: int) -> None:
    _check(lib().moe_timing_enable(max_launches), "moe_timing_enable")


def timing_collect(cap: int = 4096) -> list[tuple[str, float]]:
    """(kernel name, ms) of the launches recorded since enable / the last collect."""
    ids = (ctypes.c_int32 * cap)()
    ms = (ctypes.c_float * cap)()
    n = ctypes.c_int(0)
    _check(lib().moe_timing_collect(ids, ms, cap, ctypes.byref(n)), "moe_timing_collect")
    return [(lib().moe_kernel_name(ids[i]).decode(), ms[i]) for i in range(n.value)]


def kernel_names() -> list[str]:
    out, i = [], 0
    while (nm := lib().moe_kernel_name(i)) is not None:
        out.append(nm.decode())
        i += 1
    return out


class DeviceWeights:
    """Device copies of one block's weights and the step input, from host arrays
    (numpy or torch CPU): x / w_gate as bf16 bit patterns (uint16), the packed
    e2m1 and e8m0 tensors as uint8, bias / logit_off / norm_w as fp32."""

    def __init__(self, shape: MoEShape, x, w_gate, bias, logit_off, w13, w13s, w2, w2s, norm_w,
                 device="cuda"):
        import torch

        def up(a, dtype=None):
            if a is None:
                return None
            t = torch.as_tensor(a)
            if dtype is not None:
                t = t.view(dtype)
            return t.contiguous().to(device)

        self.shape = shape
        self.x = up(x, torch.bfloat16) if x is not None else None
        self.w_gate = up(w_gate, torch.bfloat16)
        self.bias = up(bias)
        self.logit_off = up(logit_off)
        self.w13, self.w13s, self.w2, self.w2s = up(w13), up(w13s), up(w2), up(w2s)
        self.norm_w = up(norm_w)
        S, k, d = shape.S, shape.k, shape.d
        self.ids = torch.empty((S, k), dtype=torch.int32, device=device)
        self.weights = torch.empty((S, k), dtype=torch.float32, device=device)
        self.out = torch.empty((S, d), dtype=torch.float32, device=device)
        self.ws = new_workspace(shape, device)

    def forward(self, x=None, stream=None):
        forward(self.shape, self.x if x is None else x, self.w_gate, self.bias, self.logit_off,
                self.w13, self.w13s, self.w2, self.w2s, self.norm_w, self.ids, self.weights,
                self.out, self.ws, stream)
        return self.ids, self.weights, self.out


class DeviceLatentWeights:
    """Device copies of one latent-MoE layer's weights and step input (host
    arrays: bf16 bit patterns as uint16, packed e2m1 / e8m0 as uint8, fp32)."""

    def __init__(self, shape: LatentShape, x, w_gate, bias, logit_off, w_ld, w13, w13s, w2, w2s, ln_w,
                 w_up, w_sgu, w_sd, device="cuda"):
        import torch

        def up(a, dtype=None):
            if a is None:
                return None
            t = torch.as_tensor(a)
            if dtype is not None:
                t = t.view(dtype)
            return t.contiguous().to(device)

        bf = torch.bfloat16
        self.shape = shape
        self.x = up(x, bf)
        self.w_gate, self.bias, self.logit_off = up(w_gate, bf), up(bias), up(logit_off)
        self.w_ld, self.w_up, self.ln_w = up(w_ld, bf), up(w_up, bf), up(ln_w)
        self.w13, self.w13s, self.w2, self.w2s = up(w13), up(w13s), up(w2), up(w2s)
        self.w_sgu, self.w_sd = up(w_sgu, bf), up(w_sd, bf)
        S, k, H = shape.S, shape.k, shape.H
        self.ids = torch.empty((S, k), dtype=torch.int32, device=device)
        self.weights = torch.empty((S, k), dtype=torch.float32, device=device)
        self.out = torch.empty((S, H), dtype=torch.float32, device=device)
        nbytes = latent_workspace_bytes(shape)
        buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-buf.data_ptr()) % 256
        self.ws = buf[off:off + nbytes]
        _check(lib().moe_workspace_init(self.ws.data_ptr(), nbytes, _stream(None)), "moe_workspace_init")

    def forward(self, x=None, stream=None):
        latent_forward(self.shape, self.x if x is None else x, self.w_gate, self.bias, self.logit_off, self.w_ld,
                       self.w13, self.w13s, self.w2, self.w2s, self.ln_w, self.w_up, self.w_sgu, self.w_sd,
                       self.ids, self.weights, self.out, self.ws, stream)
        return self.ids, self.weights, self.out
