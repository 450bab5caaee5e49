"""CPU oracle for the routed MoE FFN of a DeepSeek-V4-Flash layer.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg call it; the product library and its
Python binding never import it.

The arithmetic lives in ``ds4oracle.c`` (scalar C, one IEEE binary32 operation
per source operation, no contraction). This module compiles it and marshals
numpy arrays through ctypes; it adds no arithmetic of its own.

Pins (tests that tie the oracle to something other than itself) are in
``tests/test_oracle_pins.py``; every function here is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4oracle.c")
_LIB = os.path.join(_HERE, "libds4oracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

FMT = {"f32": 0, "q8_0": 1, "q2s": 2, "q4s": 3}
ROUTE = {"learned": 0, "hash": 1}


def build(force: bool = False, extra_flags=(), out: str | None = None) -> str:
    """Compile the oracle. `extra_flags`/`out` build a variant (used by the
    planted-mistake tests, which compile with -DORA_PLANT=n)."""
    out = out or _LIB
    if force or extra_flags or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, *extra_flags, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, out)
    return out


class OraLayer(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32),
        ("route", ctypes.c_int32), ("vocab", ctypes.c_int32),
        ("router_fmt", ctypes.c_int32), ("routed_fmt", ctypes.c_int32), ("shared_fmt", ctypes.c_int32),
        ("route_scale", ctypes.c_float),
        ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("hash_table", ctypes.c_void_p),
        ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
        ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p), ("sh_down", ctypes.c_void_p),
    ]


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        L = ctypes.CDLL(self.path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        sig = {
            "ora_half": (f32, [ctypes.c_uint16]),
            "ora_q8_dequant": (None, [vp, i64, vp]),
            "ora_q2s_dequant_f64": (None, [vp, i64, vp]),
            "ora_quantize": (None, [vp, ctypes.c_int, vp, vp, vp]),
            "ora_q8_dot": (i32, [vp, vp]),
            "ora_q2s_dot": (None, [vp, ctypes.c_int, vp, vp, vp, vp]),
            "ora_q4s_dequant_f64": (None, [vp, i64, vp]),
            "ora_q4s_dot": (None, [vp, ctypes.c_int, vp, vp, vp, vp]),
            "ora_row": (f32, [ctypes.c_int, vp, ctypes.c_int, vp, vp, vp, ctypes.c_int]),
            "ora_exp": (f32, [f32]),
            "ora_sigmoid": (f32, [f32]),
            "ora_silu": (f32, [f32]),
            "ora_route_token": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp]),
            "ora_route": (ctypes.c_int, [vp, vp, vp, ctypes.c_int, vp, vp, vp, vp]),
            "ora_expert": (None, [vp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp]),
            "ora_forward": (ctypes.c_int, [vp, vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_int]),
            "ora_rmsnorm": (None, [vp, vp, ctypes.c_int, ctypes.c_int, f32]),
            "ora_dense_q8": (None, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        self.L = L

    # -- formats -----------------------------------------------------------
    def half(self, bits: int) -> float:
        return float(self.L.ora_half(bits))

    def q8_dequant(self, blocks: np.ndarray) -> np.ndarray:
        nb = blocks.nbytes // 34
        out = np.empty(nb * 32, np.float32)
        self.L.ora_q8_dequant(_ptr(np.ascontiguousarray(blocks)), nb, _ptr(out))
        return out

    def q2s_dequant(self, sbs: np.ndarray) -> np.ndarray:
        n = sbs.nbytes // 84
        out = np.empty(n * 256, np.float64)
        self.L.ora_q2s_dequant_f64(_ptr(np.ascontiguousarray(sbs)), n, _ptr(out))
        return out

    def q4s_dequant(self, sbs: np.ndarray) -> np.ndarray:
        n = sbs.nbytes // 148
        out = np.empty(n * 256, np.float64)
        self.L.ora_q4s_dequant_f64(_ptr(np.ascontiguousarray(sbs)), n, _ptr(out))
        return out

    # -- CAS steps ----------------------------------------------------------
    def quantize(self, v: np.ndarray):
        v = np.ascontiguousarray(v, dtype=np.float32)
        n = v.size
        q = np.empty(n, np.int8)
        d = np.empty(n // 32, np.float32)
        gs = np.empty(n // 16, np.int16)
        self.L.ora_quantize(_ptr(v), n, _ptr(q), _ptr(d), _ptr(gs))
        return q, d, gs

    def q8_dot(self, blk: np.ndarray, xq: np.ndarray) -> int:
        return int(self.L.ora_q8_dot(_ptr(np.ascontiguousarray(blk)), _ptr(np.ascontiguousarray(xq))))

    def q2s_dot(self, sb: np.ndarray, j: int, xq32: np.ndarray, gs2: np.ndarray):
        A, B = ctypes.c_int32(), ctypes.c_int32()
        self.L.ora_q2s_dot(_ptr(np.ascontiguousarray(sb)), j, _ptr(np.ascontiguousarray(xq32)),
                           _ptr(np.ascontiguousarray(gs2, dtype=np.int16)), ctypes.byref(A), ctypes.byref(B))
        return A.value, B.value

    def q4s_dot(self, sb: np.ndarray, j: int, xq32: np.ndarray, gs2: np.ndarray):
        A, B = ctypes.c_int32(), ctypes.c_int32()
        self.L.ora_q4s_dot(_ptr(np.ascontiguousarray(sb)), j, _ptr(np.ascontiguousarray(xq32)),
                           _ptr(np.ascontiguousarray(gs2, dtype=np.int16)), ctypes.byref(A), ctypes.byref(B))
        return A.value, B.value

    def row(self, fmt: str, row: np.ndarray, K: int, xq, dx, gs, S: int = 1) -> np.float32:
        return np.float32(self.L.ora_row(FMT[fmt], _ptr(np.ascontiguousarray(row)), K, _ptr(xq), _ptr(dx),
                                         _ptr(gs), S))

    def exp(self, z: float) -> np.float32:
        return np.float32(self.L.ora_exp(float(z)))

    def sigmoid(self, z: float) -> np.float32:
        return np.float32(self.L.ora_sigmoid(float(z)))

    def silu(self, z: float) -> np.float32:
        return np.float32(self.L.ora_silu(float(z)))

    def rmsnorm(self, x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        T, H = x.shape
        out = np.empty_like(x)
        self.L.ora_rmsnorm(_ptr(x), _ptr(out), T, H, eps)
        return out

    def dense_q8(self, w: np.ndarray, N: int, K: int, x: np.ndarray, nthreads: int = 0) -> np.ndarray:
        """y[T][N] = W x for canonical Q8_0 rows w ([N][K]) and x [T][K] f32."""
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.nbytes == N * (K // 32) * 34
        y = np.empty((x.shape[0], N), np.float32)
        self.L.ora_dense_q8(_ptr(w), N, K, _ptr(x), x.shape[0], _ptr(y), nthreads or (os.cpu_count() or 1))
        return y

    # -- layer ---------------------------------------------------------------
    def layer(self, spec, w: dict) -> "BoundLayer":
        return BoundLayer(self, spec, w)


class BoundLayer:
    """An oracle view of one layer's weights (host arrays, canonical layouts)."""

    def __init__(self, ora: Oracle, spec, w: dict):
        self.ora, self.spec = ora, spec
        self._keep = {k: np.ascontiguousarray(v) for k, v in w.items()}
        g = self._keep.get
        self.c = OraLayer(
            spec.hidden, spec.n_experts, spec.top_k, spec.ffn, spec.n_shared,
            ROUTE[spec.route], spec.vocab,
            FMT[spec.router_fmt], FMT[spec.routed_fmt], FMT[spec.shared_fmt], spec.route_scale,
            _ptr(g("router_w")), _ptr(g("router_bias")), _ptr(g("hash_table")),
            _ptr(g("gate")), _ptr(g("up")), _ptr(g("down")),
            _ptr(g("sh_gate")), _ptr(g("sh_up")), _ptr(g("sh_down")),
        )

    def route(self, x: np.ndarray, tok=None):
        x = np.ascontiguousarray(x, dtype=np.float32)
        T = x.shape[0]
        s = self.spec
        ids = np.empty((T, s.top_k), np.int32)
        w = np.empty((T, s.top_k), np.float32)
        logits = np.zeros((T, s.n_experts), np.float32)
        keys = np.zeros((T, s.n_experts), np.float32)
        tk = None if tok is None else np.ascontiguousarray(tok, dtype=np.int32)
        bad = self.ora.L.ora_route(ctypes.byref(self.c), _ptr(x), _ptr(tk), T, _ptr(ids), _ptr(w),
                                   _ptr(logits), _ptr(keys))
        return ids, w, logits, keys, bad

    def expert(self, e: int, x: np.ndarray) -> dict:
        s = self.spec
        H, F = s.hidden, s.ffn
        out = dict(g=np.empty(F, np.float32), u=np.empty(F, np.float32), h=np.empty(F, np.float32),
                   hq=np.empty(F, np.int8), dh=np.empty(F // 32, np.float32), gsh=np.empty(F // 16, np.int16),
                   a=np.empty(H, np.float32))
        x = np.ascontiguousarray(x, dtype=np.float32)
        self.ora.L.ora_expert(ctypes.byref(self.c), e, _ptr(x), *(_ptr(out[k]) for k in
                                                                     ("g", "u", "h", "hq", "dh", "gsh", "a")))
        return out

    def forward(self, x: np.ndarray, y: np.ndarray | None = None, tok=None, nthreads: int = 0):
        """Returns (y + MoE(x), ids, w, n_bad_tokens)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        T, H = x.shape
        y = np.zeros_like(x) if y is None else np.array(y, dtype=np.float32, copy=True)
        ids = np.empty((T, self.spec.top_k), np.int32)
        w = np.empty((T, self.spec.top_k), np.float32)
        tk = None if tok is None else np.ascontiguousarray(tok, dtype=np.int32)
        bad = self.ora.L.ora_forward(ctypes.byref(self.c), _ptr(x), _ptr(tk), T, _ptr(y), _ptr(ids),
                                     _ptr(w), nthreads)
        if bad < 0:
            raise MemoryError("oracle forward: allocation failed")
        return y, ids, w, bad


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
