"""Seeded synthetic workloads for the routed MoE FFN of a DeepSeek-V4-Flash layer.

This package only generates inputs: weight bytes in the canonical formats,
router bias, hash table, activations and token ids. It holds none of the
layer's arithmetic, and it imports neither the CPU oracle nor the CUDA library;
both of them consume what it writes.

The layer shapes follow the DeepSeek V4 Flash architecture table on the
"DeepSeek V4 Flash -- DFlash Integration" page (Model Architecture): hidden
4096, 256 routed experts top-6 plus 1 shared, expert FFN 2048, hash routing on
the first 3 of 43 layers. The weight recipes are the workload descriptions of
the routed-MoE benchmark (2-bit superblocks for routed experts, Q8_0 for the
shared expert and router).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4synth.c")
_LIB = os.path.join(_HERE, "libds4synth.so")

# Tensor tags used to derive independent random streams.
T_ROUTER, T_BIAS, T_HASH, T_GATE, T_UP, T_DOWN, T_SH_GATE, T_SH_UP, T_SH_DOWN = range(1, 10)
T_X, T_TOK, T_PERM = 10, 11, 12
T_DENSE = 13

FMT_F32, FMT_Q8_0, FMT_Q2S, FMT_Q4S = "f32", "q8_0", "q2s", "q4s"


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u8p, i32p, f32p = (ctypes.c_void_p,) * 3
        L.ds4s_key.restype = ctypes.c_uint64
        L.ds4s_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        L.ds4s_q2s.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int]
        L.ds4s_q4s.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int]
        L.ds4s_q8.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int]
        L.ds4s_normal_f32.argtypes = [f32p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_float, ctypes.c_int]
        L.ds4s_uniform_f32.argtypes = [f32p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_float, ctypes.c_int]
        L.ds4s_token_ids.argtypes = [i32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64]
        L.ds4s_hash_table.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int]
        L.ds4s_permutation.argtypes = [i32p, ctypes.c_int32, ctypes.c_uint64]
        for f in ("ds4s_q2s", "ds4s_q4s", "ds4s_q8", "ds4s_normal_f32", "ds4s_uniform_f32", "ds4s_token_ids",
                  "ds4s_hash_table", "ds4s_permutation"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def key(seed: int, layer: int, tensor: int) -> int:
    return int(lib().ds4s_key(seed & (2**64 - 1), layer & 0xFFFFFFFF, tensor))


# ---------------------------------------------------------------------------
# Layer specifications (shapes + generation recipe)


@dataclass(frozen=True)
class LayerSpec:
    name: str
    hidden: int
    n_experts: int
    top_k: int
    ffn: int
    n_shared: int
    route: str  # "learned" | "hash"
    vocab: int
    router_fmt: str
    routed_fmt: str
    shared_fmt: str
    router_sigma: float
    bias: str  # "uniform" (U(-0.1, 0.1)) | "zipf" (Zipf(1.1) popularity) | "none"
    route_scale: float = 1.0
    q8_sigma: float = 0.02
    q2s_dsig: float = 0.01
    q4s_dsig: float = 0.002  # 4-bit codes are 5x wider: about the 2-bit format's weight spread


# Tiny layer: every weight Q8_0, fp32 router.
TINY = LayerSpec("tiny", 256, 16, 2, 128, 1, "learned", 0, FMT_F32, FMT_Q8_0, FMT_Q8_0,
                 router_sigma=0.05, bias="uniform")
# DeepSeek-V4-Flash-shaped layer with learned routing.
DS4 = LayerSpec("ds4", 4096, 256, 6, 2048, 1, "learned", 0, FMT_Q8_0, FMT_Q2S, FMT_Q8_0,
                router_sigma=0.0125, bias="uniform")
# Same layer, router bias giving a Zipf(s=1.1) expert popularity.
DS4_ZIPF = replace(DS4, name="ds4-zipf", bias="zipf")
# Same shapes, routed by a token-id hash table (first 3 layers of the model).
DS4_HASH = replace(DS4, name="ds4-hash", route="hash", vocab=129280, bias="none")
# A small layer with the DS4 formats, for fast tests that still span several tiles.
MICRO = LayerSpec("micro", 512, 8, 3, 256, 1, "learned", 0, FMT_Q8_0, FMT_Q2S, FMT_Q8_0,
                  router_sigma=0.02, bias="uniform")
MICRO_HASH = replace(MICRO, name="micro-hash", route="hash", vocab=1000, bias="none")
# The same shapes with 4-bit routed experts (the "q2 with the last 6 layers
# q4" variant of the DwarfStar model weights).
DS4_Q4 = replace(DS4, name="ds4-q4", routed_fmt=FMT_Q4S)
MICRO_Q4 = replace(MICRO, name="micro-q4", routed_fmt=FMT_Q4S)
MICRO_Q4_HASH = replace(MICRO_HASH, name="micro-q4-hash", routed_fmt=FMT_Q4S)
# DS4 router shapes with small experts, for router-only checks.
DS4_ROUTER_ONLY = replace(DS4, name="ds4-router", ffn=256, routed_fmt=FMT_Q8_0, n_shared=0)

N_STACK_LAYERS = 43
N_HASH_LAYERS = 3


N_Q4_LAYERS = 6


def stack_layer_spec(layer: int, q4_tail: bool = False) -> LayerSpec:
    """Layer l of the 43-layer stack: 0-2 hash routed, 3-42 learned; with
    q4_tail the last 6 layers' routed experts are 4-bit."""
    if q4_tail and layer >= N_STACK_LAYERS - N_Q4_LAYERS:
        return DS4_Q4
    return DS4_HASH if layer < N_HASH_LAYERS else DS4


def row_bytes(fmt: str, k: int) -> int:
    if fmt == FMT_F32:
        return 4 * k
    if fmt == FMT_Q8_0:
        assert k % 32 == 0
        return (k // 32) * 34
    if fmt == FMT_Q2S:
        assert k % 256 == 0
        return (k // 256) * 84
    if fmt == FMT_Q4S:
        assert k % 256 == 0
        return (k // 256) * 148
    raise ValueError(fmt)


def tensor_shapes(spec: LayerSpec) -> dict:
    """name -> (fmt, n_mat, rows, cols) for every weight tensor of the layer."""
    E, H, F = spec.n_experts, spec.hidden, spec.ffn
    d = {}
    if spec.route == "learned":
        d["router_w"] = (spec.router_fmt, 1, E, H)
    d["gate"] = (spec.routed_fmt, E, F, H)
    d["up"] = (spec.routed_fmt, E, F, H)
    d["down"] = (spec.routed_fmt, E, H, F)
    if spec.n_shared:
        d["sh_gate"] = (spec.shared_fmt, 1, F, H)
        d["sh_up"] = (spec.shared_fmt, 1, F, H)
        d["sh_down"] = (spec.shared_fmt, 1, H, F)
    return d


_TAGS = {"router_w": T_ROUTER, "gate": T_GATE, "up": T_UP, "down": T_DOWN,
         "sh_gate": T_SH_GATE, "sh_up": T_SH_UP, "sh_down": T_SH_DOWN}


def tensor_nbytes(spec: LayerSpec, name: str) -> int:
    fmt, n, r, c = tensor_shapes(spec)[name]
    return n * r * row_bytes(fmt, c)


def layer_nbytes(spec: LayerSpec) -> int:
    return sum(tensor_nbytes(spec, n) for n in tensor_shapes(spec))


def gen_tensor_into(spec: LayerSpec, seed: int, layer: int, name: str, ptr: int,
                    first_row: int = 0, n_rows: int | None = None, nthreads: int = 0) -> None:
    """Write rows [first_row, first_row+n_rows) of the flattened tensor `name`
    (all matrices stacked, i.e. n_mat*rows rows) into host memory at `ptr`."""
    fmt, n, r, c = tensor_shapes(spec)[name]
    total_rows = n * r
    if n_rows is None:
        n_rows = total_rows - first_row
    assert 0 <= first_row and first_row + n_rows <= total_rows
    k = key(seed, layer, _TAGS[name])
    L = lib()
    if fmt == FMT_Q2S:
        per = c // 256
        L.ds4s_q2s(ptr, first_row * per, n_rows * per, k, spec.q2s_dsig, nthreads)
    elif fmt == FMT_Q4S:
        per = c // 256
        L.ds4s_q4s(ptr, first_row * per, n_rows * per, k, spec.q4s_dsig, nthreads)
    elif fmt == FMT_Q8_0:
        per = c // 32
        sigma = spec.router_sigma if name == "router_w" else spec.q8_sigma
        L.ds4s_q8(ptr, first_row * per, n_rows * per, k, sigma, nthreads)
    elif fmt == FMT_F32:
        assert first_row == 0 and n_rows == total_rows
        sigma = spec.router_sigma if name == "router_w" else spec.q8_sigma
        L.ds4s_normal_f32(ptr, n_rows * c, k, sigma, 0.0, nthreads)
    else:
        raise ValueError(fmt)


def gen_tensor(spec: LayerSpec, seed: int, layer: int, name: str, nthreads: int = 0) -> np.ndarray:
    nb = tensor_nbytes(spec, name)
    out = np.empty(nb, dtype=np.uint8)
    gen_tensor_into(spec, seed, layer, name, out.ctypes.data, nthreads=nthreads)
    return out


def gen_bias(spec: LayerSpec, seed: int, layer: int) -> np.ndarray:
    """Selection bias b[E] (fp32).

    uniform: U(-0.1, 0.1).
    zipf:    a seeded permutation pi gives expert e the popularity rank pi(e)+1;
             p_r ~ r^-1.1, and b_e = 0.05 * ln(p_rank / p_1) = -0.055 * ln(rank).
    """
    E = spec.n_experts
    b = np.zeros(E, dtype=np.float32)
    if spec.bias == "uniform":
        lib().ds4s_uniform_f32(b.ctypes.data, E, key(seed, layer, T_BIAS), -0.1, 0.1, 1)
    elif spec.bias == "zipf":
        perm = np.empty(E, dtype=np.int32)
        lib().ds4s_permutation(perm.ctypes.data, E, key(seed, layer, T_PERM))
        b = (0.05 * (-1.1) * np.log(perm.astype(np.float64) + 1.0)).astype(np.float32)
    return b


def gen_hash_table(spec: LayerSpec, seed: int, layer: int, nthreads: int = 0) -> np.ndarray:
    t = np.empty((spec.vocab, spec.top_k), dtype=np.int32)
    lib().ds4s_hash_table(t.ctypes.data, spec.vocab, spec.n_experts, spec.top_k,
                          key(seed, layer, T_HASH), nthreads)
    return t


def gen_layer(spec: LayerSpec, seed: int, layer: int = 0, nthreads: int = 0) -> dict:
    """All weights of one layer as host arrays in the canonical byte layouts."""
    w = {n: gen_tensor(spec, seed, layer, n, nthreads) for n in tensor_shapes(spec)}
    if spec.route == "learned":
        w["router_bias"] = gen_bias(spec, seed, layer)
        if spec.router_fmt == FMT_F32:
            w["router_w"] = w["router_w"].view(np.float32).reshape(spec.n_experts, spec.hidden)
    else:
        w["hash_table"] = gen_hash_table(spec, seed, layer, nthreads)
    return w


def x_row_key(seed: int, token: int, attempt: int = 0) -> int:
    return key(seed, ((attempt & 0xFFF) << 20) | (token & 0xFFFFF), T_X)


def gen_x(spec: LayerSpec, seed: int, n_tok: int, attempts=None) -> np.ndarray:
    """x[T][H] ~ N(0,1) fp32; each token row has its own stream.
    attempts[t] selects a regenerated row for token t (default 0)."""
    x = np.empty((n_tok, spec.hidden), dtype=np.float32)
    for t in range(n_tok):
        a = 0 if attempts is None else int(attempts[t])
        lib().ds4s_normal_f32(x[t].ctypes.data, spec.hidden, x_row_key(seed, t, a), 1.0, 0.0, 1)
    return x


def gen_x_row(spec: LayerSpec, seed: int, token: int, attempt: int) -> np.ndarray:
    x = np.empty(spec.hidden, dtype=np.float32)
    lib().ds4s_normal_f32(x.ctypes.data, spec.hidden, x_row_key(seed, token, attempt), 1.0, 0.0, 1)
    return x


def gen_token_ids(spec: LayerSpec, seed: int, n_tok: int) -> np.ndarray:
    t = np.empty(n_tok, dtype=np.int32)
    vocab = spec.vocab if spec.vocab > 0 else 129280
    lib().ds4s_token_ids(t.ctypes.data, n_tok, vocab, key(seed, 0, T_TOK))
    return t


def gen_q8_matrix(seed: int, n_out: int, n_in: int, sigma: float = 0.02, nthreads: int = 0) -> np.ndarray:
    """A dense [n_out][n_in] Q8_0 matrix (canonical bytes), weights ~ N(0, sigma)
    quantised as the shared expert's are."""
    assert n_in % 32 == 0
    out = np.empty(n_out * (n_in // 32) * 34, dtype=np.uint8)
    lib().ds4s_q8(out.ctypes.data, 0, n_out * (n_in // 32), key(seed, 0, T_DENSE), sigma, nthreads)
    return out


def gen_dense_x(seed: int, n_tok: int, n_in: int) -> np.ndarray:
    """x[T][n_in] ~ N(0,1) fp32, one stream per token."""
    x = np.empty((n_tok, n_in), dtype=np.float32)
    for t in range(n_tok):
        lib().ds4s_normal_f32(x[t].ctypes.data, n_in, key(seed, t, T_DENSE + 1), 1.0, 0.0, 1)
    return x
