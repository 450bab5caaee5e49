"""Python binding of libds4moe, the routed MoE FFN of a DeepSeek-V4-Flash layer
on GB300 (sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. PyTorch supplies device memory and streams. There is no CPU fallback:
if the compiled library cannot be loaded, importing the binding fails.

Entry points mirror the C ABI in include/ds4moe.h:
``Layer(desc, weights)`` = ds4moe_create, ``Layer.route`` = ds4moe_route,
``Layer.forward`` = ds4moe_forward, ``Layer.forward_rmsnorm`` =
ds4moe_forward_rmsnorm, ``Layer.forward_host`` = ds4moe_forward_host,
``rmsnorm`` = ds4moe_rmsnorm, ``route_noalloc`` =
ds4moe_route_noalloc, ``Dense`` = the ds4moe_dense_* calls.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import build as _build

ABI_VERSION = 1
F32, Q8_0, Q2S, Q4S = 0, 1, 2, 3
FMT = {"f32": F32, "q8_0": Q8_0, "q2s": Q2S, "q4s": Q4S}
ROUTE_LEARNED, ROUTE_HASH = 0, 1
STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_OOM", 4: "ERR_CUDA", 5: "ERR_DEVICE"}
DEVERR_TOKEN_ID, DEVERR_NONFINITE, DEVERR_TIMEOUT, DEVERR_INTERNAL = 1, 2, 4, 8

LIB_PATH = _build.LIB


class Ds4MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class _Desc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_uint32), ("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("route", ctypes.c_int32), ("vocab", ctypes.c_int32), ("router_fmt", ctypes.c_int32),
                ("routed_fmt", ctypes.c_int32), ("shared_fmt", ctypes.c_int32), ("route_scale", ctypes.c_float),
                ("max_tokens", ctypes.c_int32)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("router_w", "router_bias", "hash_table", "gate", "up", "down", "sh_gate", "sh_up", "sh_down")]


_lib = None


def lib():
    """Load libds4moe.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        if _build.stale():
            _build.build()
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libds4moe.so not found at {LIB_PATH}")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
        sigs = {
            "ds4moe_create": (i32, [ctypes.POINTER(_Desc), ctypes.POINTER(_Weights), ctypes.POINTER(vp)]),
            "ds4moe_destroy": (None, [vp]),
            "ds4moe_route": (i32, [vp, vp, vp, i32, vp, vp, vp]),
            "ds4moe_route_noalloc": (i32, [ctypes.POINTER(_Desc), ctypes.POINTER(_Weights), vp, vp, i32, vp, vp,
                                           vp, vp]),
            "ds4moe_forward": (i32, [vp, vp, i32, vp, vp, vp]),
            "ds4moe_forward_host": (i32, [vp, vp, i32, vp, vp, vp]),
            "ds4moe_forward_rmsnorm": (i32, [vp, vp, i32, vp, ctypes.c_float, vp, vp]),
            "ds4moe_rmsnorm": (i32, [vp, vp, i32, i32, ctypes.c_float, vp]),
            "ds4moe_get_device_error": (i32, [vp, vp, ctypes.POINTER(u32)]),
            "ds4moe_debug_scratch": (i32, [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_uint64)]),
            "ds4moe_device_bytes": (ctypes.c_uint64, [vp]),
            "ds4moe_profile_enable": (i32, [vp, i32]),
            "ds4moe_profile_collect": (i32, [vp]),
            "ds4moe_profile_read": (i32, [vp, ctypes.POINTER(ctypes.c_double), i32,
                                          ctypes.POINTER(ctypes.c_int64)]),
            "ds4moe_launch_count": (ctypes.c_uint64, [vp]),
            "ds4moe_debug_set_wait_limit": (i32, [vp, ctypes.c_int64]),
            "ds4moe_debug_fail_alloc": (i32, [i32]),
            "ds4moe_status_string": (ctypes.c_char_p, [i32]),
            "ds4moe_abi_version": (u32, []),
            "ds4moe_dense_create": (i32, [i32, i32, i32, vp, ctypes.POINTER(vp)]),
            "ds4moe_dense_forward": (i32, [vp, vp, i32, vp, vp]),
            "ds4moe_dense_get_device_error": (i32, [vp, vp, ctypes.POINTER(u32)]),
            "ds4moe_dense_destroy": (None, [vp]),
            "ds4moe_dense_device_bytes": (ctypes.c_uint64, [vp]),
            "ds4moe_dense_launch_count": (ctypes.c_uint64, [vp]),
            "ds4moe_dense_debug_config": (i32, [vp, i32, i32, i32, i32]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        if L.ds4moe_abi_version() != ABI_VERSION:
            raise ImportError("libds4moe ABI version mismatch")
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise Ds4MoeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


@dataclass
class LayerDesc:
    hidden: int
    n_experts: int
    top_k: int
    ffn: int
    n_shared: int
    route: int  # ROUTE_LEARNED | ROUTE_HASH
    vocab: int
    router_fmt: int
    routed_fmt: int
    shared_fmt: int
    route_scale: float = 1.0
    max_tokens: int = 1

    def c(self) -> _Desc:
        return _Desc(ABI_VERSION, self.hidden, self.n_experts, self.top_k, self.ffn, self.n_shared, self.route,
                     self.vocab, self.router_fmt, self.routed_fmt, self.shared_fmt, self.route_scale,
                     self.max_tokens)


class _CudaArray:
    """A device buffer described by __cuda_array_interface__ (for torch.as_tensor)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


class Layer:
    """One MoE layer handle (ds4moe_create). `weights` maps the names of
    ds4moe_weights (router_w, router_bias, hash_table, gate, up, down, sh_gate,
    sh_up, sh_down) to CUDA tensors in the canonical byte layouts."""

    def __init__(self, desc: LayerDesc, weights: dict):
        L = lib()
        self.desc = desc
        w = _Weights(*[_ptr(weights.get(n)) for n, _ in _Weights._fields_])
        h = ctypes.c_void_p()
        _check(L.ds4moe_create(ctypes.byref(desc.c()), ctypes.byref(w), ctypes.byref(h)), "ds4moe_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().ds4moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def device_bytes(self) -> int:
        return int(lib().ds4moe_device_bytes(self._h))

    STAGES = ("quantize", "route", "bucket", "gateup", "down", "combine")

    def profile(self, on: bool = True):
        """Record CUDA events around every stage of later forwards (ds4moe_profile_enable)."""
        _check(lib().ds4moe_profile_enable(self._h, 1 if on else 0), "ds4moe_profile_enable")

    def profile_collect(self):
        """Wait for the last forward's events and add its stage times (ds4moe_profile_collect)."""
        _check(lib().ds4moe_profile_collect(self._h), "ds4moe_profile_collect")

    def profile_read(self):
        """(per-stage total ms, number of collected calls) (ds4moe_profile_read)."""
        ms = (ctypes.c_double * len(self.STAGES))()
        calls = ctypes.c_int64()
        _check(lib().ds4moe_profile_read(self._h, ms, len(self.STAGES), ctypes.byref(calls)),
               "ds4moe_profile_read")
        return dict(zip(self.STAGES, list(ms))), int(calls.value)

    def launch_count(self) -> int:
        """Kernels launched by this handle since create (ds4moe_launch_count)."""
        return int(lib().ds4moe_launch_count(self._h))

    def forward(self, x, y, token_ids=None, stream=None, n_tok=None):
        """y += MoE(x) on the device (ds4moe_forward)."""
        n = x.shape[0] if n_tok is None else n_tok
        _check(lib().ds4moe_forward(self._h, _ptr(x), n, _ptr(token_ids), _ptr(y), _stream(stream)),
               "ds4moe_forward")

    def forward_rmsnorm(self, x, y, eps: float = 1e-6, token_ids=None, stream=None, n_tok=None):
        """y += MoE(RMSNorm(x)) on the device (ds4moe_forward_rmsnorm); y may be x."""
        n = x.shape[0] if n_tok is None else n_tok
        _check(lib().ds4moe_forward_rmsnorm(self._h, _ptr(x), n, _ptr(token_ids), eps, _ptr(y), _stream(stream)),
               "ds4moe_forward_rmsnorm")

    def forward_host(self, x, y, token_ids=None, stream=None):
        """y += MoE(x) on host tensors (ds4moe_forward_host; synchronises)."""
        _check(lib().ds4moe_forward_host(self._h, _ptr(x), x.shape[0], _ptr(token_ids), _ptr(y),
                                         _stream(stream)), "ds4moe_forward_host")

    def route(self, x=None, token_ids=None, ids_out=None, w_out=None, stream=None, n_tok=None):
        """Expert ids and weights (ds4moe_route). Returns (ids_out, w_out)."""
        import torch
        n = n_tok if n_tok is not None else (x.shape[0] if x is not None else token_ids.shape[0])
        dev = (x if x is not None else token_ids).device
        if ids_out is None:
            ids_out = torch.empty((n, self.desc.top_k), dtype=torch.int32, device=dev)
        if w_out is None:
            w_out = torch.empty((n, self.desc.top_k), dtype=torch.float32, device=dev)
        _check(lib().ds4moe_route(self._h, _ptr(x), _ptr(token_ids), n, _ptr(ids_out), _ptr(w_out),
                                  _stream(stream)), "ds4moe_route")
        return ids_out, w_out

    def set_wait_limit(self, cycles: int):
        """Bound of the decode expert kernels' hand-off waits, in SM cycles
        (0: the default); a test hook (ds4moe_debug_set_wait_limit)."""
        _check(lib().ds4moe_debug_set_wait_limit(self._h, int(cycles)), "ds4moe_debug_set_wait_limit")

    def device_error(self, stream=None) -> int:
        """Synchronise, read and clear the device error flags (0 = none)."""
        f = ctypes.c_uint32(0)
        st = lib().ds4moe_get_device_error(self._h, _stream(stream), ctypes.byref(f))
        if st not in (0, 5):
            raise Ds4MoeError(st, "ds4moe_get_device_error")
        return int(f.value)

    _SCRATCH = {"xq": (0, "|i1"), "dx": (1, "<f4"), "gs": (2, "<i2"), "ids": (3, "<i4"), "w": (4, "<f4"),
                "hq": (5, "|i1"), "dh": (6, "<f4"), "a": (7, "<f4")}

    def scratch(self, name: str):
        """Torch view (treat as read-only) of an intermediate buffer (ds4moe_debug_scratch), flat."""
        import torch
        which, typestr = self._SCRATCH[name]
        p, n = ctypes.c_void_p(), ctypes.c_uint64()
        _check(lib().ds4moe_debug_scratch(self._h, which, ctypes.byref(p), ctypes.byref(n)), "ds4moe_debug_scratch")
        itemsize = int(typestr[2:])
        return torch.as_tensor(_CudaArray(p.value, (n.value // itemsize,), typestr), device="cuda")


class Dense:
    """A dense Q8_0 matrix beside the MoE (ds4moe_dense_create): `w` is the
    canonical [n_out][n_in] Q8_0 matrix as a CUDA uint8 tensor."""

    def __init__(self, n_out: int, n_in: int, w, max_tokens: int = 1):
        L = lib()
        h = ctypes.c_void_p()
        _check(L.ds4moe_dense_create(n_out, n_in, max_tokens, _ptr(w), ctypes.byref(h)), "ds4moe_dense_create")
        self._h, self.n_out, self.n_in = h, n_out, n_in

    def close(self):
        if getattr(self, "_h", None):
            lib().ds4moe_dense_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, y=None, stream=None, n_tok=None):
        """y = W x (ds4moe_dense_forward); returns y."""
        import torch
        n = x.shape[0] if n_tok is None else n_tok
        if y is None:
            y = torch.empty((n, self.n_out), dtype=torch.float32, device=x.device)
        _check(lib().ds4moe_dense_forward(self._h, _ptr(x), n, _ptr(y), _stream(stream)), "ds4moe_dense_forward")
        return y

    def device_error(self, stream=None) -> int:
        f = ctypes.c_uint32(0)
        st = lib().ds4moe_dense_get_device_error(self._h, _stream(stream), ctypes.byref(f))
        if st not in (0, 5):
            raise Ds4MoeError(st, "ds4moe_dense_get_device_error")
        return int(f.value)

    def launch_count(self) -> int:
        return int(lib().ds4moe_dense_launch_count(self._h))

    def debug_config(self, ks=0, nst=0, ns=0, tc=0):
        """Override the kernel's K steps per stage, stages per warp, units per
        32 rows and block-dot step (tc 1: dp4a, 2: tensor cores; 0:
        automatic); a tuning and test hook (ds4moe_dense_debug_config)."""
        _check(lib().ds4moe_dense_debug_config(self._h, int(ks), int(nst), int(ns), int(tc)),
               "ds4moe_dense_debug_config")


def rmsnorm(x, out, eps: float = 1e-6, stream=None):
    """out = x / sqrt(mean(x^2) + eps) row-wise (ds4moe_rmsnorm); out may be x."""
    _check(lib().ds4moe_rmsnorm(_ptr(x), _ptr(out), x.shape[0], x.shape[1], eps, _stream(stream)),
           "ds4moe_rmsnorm")


NOALLOC_SCRATCH_BYTES = 512 * 1024


def route_noalloc(desc: LayerDesc, weights: dict, x=None, token_ids=None, ids_out=None, w_out=None,
                  err_flags=None, stream=None, n_tok=None):
    """Routing from the canonical router buffers in `weights` (router_w,
    router_bias or hash_table; CUDA tensors) with no handle and no device
    allocation by the library (ds4moe_route_noalloc). ids_out / w_out are
    allocated here by torch when not given. Returns (ids_out, w_out)."""
    import torch
    n = n_tok if n_tok is not None else (x.shape[0] if x is not None else token_ids.shape[0])
    dev = (x if x is not None else token_ids).device
    if ids_out is None:
        ids_out = torch.empty((n, desc.top_k), dtype=torch.int32, device=dev)
    if w_out is None:
        w_out = torch.empty((n, desc.top_k), dtype=torch.float32, device=dev)
    w = _Weights(*[_ptr(weights.get(name)) for name, _ in _Weights._fields_])
    _check(lib().ds4moe_route_noalloc(ctypes.byref(desc.c()), ctypes.byref(w), _ptr(x), _ptr(token_ids), n,
                                      _ptr(ids_out), _ptr(w_out), _ptr(err_flags), _stream(stream)),
           "ds4moe_route_noalloc")
    return ids_out, w_out


def fail_alloc(n: int):
    """Make the n-th device allocation the library makes from now on fail as
    if out of memory (0: off); a test hook (ds4moe_debug_fail_alloc)."""
    _check(lib().ds4moe_debug_fail_alloc(int(n)), "ds4moe_debug_fail_alloc")


def status_string(status: int) -> str:
    return lib().ds4moe_status_string(status).decode()
