"""Float64 / integer brute-force references used to pin the oracle.

Everything here is written from the format and arithmetic definitions
directly, vectorised with numpy, and shares no code with ``oracle/``:
it unpacks bytes with numpy, decodes binary16 with numpy's own float16, and
does its sums in float64 or int64.
"""
import numpy as np


def unpack_q8(buf, rows, k):
    b = np.frombuffer(np.ascontiguousarray(buf).tobytes(), np.uint8).reshape(rows, k // 32, 34)
    d = b[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = b[:, :, 2:].copy().view(np.int8).astype(np.int64)
    return d, q  # d [rows][k/32], q [rows][k/32][32]


def dequant_q8(buf, rows, k):
    d, q = unpack_q8(buf, rows, k)
    return (d[:, :, None] * q).reshape(rows, k)


def unpack_q2s(buf, rows, k):
    b = np.frombuffer(np.ascontiguousarray(buf).tobytes(), np.uint8).reshape(rows, k // 256, 84)
    sm = b[:, :, 0:16].astype(np.int64)
    qs = b[:, :, 16:80].astype(np.int64)
    d = b[:, :, 80:82].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[:, :, 82:84].copy().view(np.float16)[..., 0].astype(np.float64)
    sc, mn = sm & 15, sm >> 4
    shifts = np.array([0, 2, 4, 6])
    q = ((qs[:, :, :, None] >> shifts) & 3).reshape(rows, k // 256, 256)
    return d, dmin, sc, mn, q


def dequant_q2s(buf, rows, k):
    d, dmin, sc, mn, q = unpack_q2s(buf, rows, k)
    scx = np.repeat(sc, 16, axis=2)
    mnx = np.repeat(mn, 16, axis=2)
    w = d[:, :, None] * scx * q - dmin[:, :, None] * mnx
    return w.reshape(rows, k)


def unpack_q4s(buf, rows, k):
    b = np.frombuffer(np.ascontiguousarray(buf).tobytes(), np.uint8).reshape(rows, k // 256, 148)
    sm = b[:, :, 0:16].astype(np.int64)
    qs = b[:, :, 16:144].astype(np.int64)
    d = b[:, :, 144:146].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[:, :, 146:148].copy().view(np.float16)[..., 0].astype(np.float64)
    sc, mn = sm & 15, sm >> 4
    q = ((qs[:, :, :, None] >> np.array([0, 4])) & 15).reshape(rows, k // 256, 256)
    return d, dmin, sc, mn, q


def dequant_q4s(buf, rows, k):
    d, dmin, sc, mn, q = unpack_q4s(buf, rows, k)
    scx = np.repeat(sc, 16, axis=2)
    mnx = np.repeat(mn, 16, axis=2)
    w = d[:, :, None] * scx * q - dmin[:, :, None] * mnx
    return w.reshape(rows, k)


def dequant(fmt, buf, rows, k):
    if fmt == "q8_0":
        return dequant_q8(buf, rows, k)
    if fmt == "q2s":
        return dequant_q2s(buf, rows, k)
    if fmt == "q4s":
        return dequant_q4s(buf, rows, k)
    return np.asarray(buf, np.float64).reshape(rows, k)


def round_half_away(v):
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def quantize_f64(v):
    """Per-32-block int8 quantisation done in float64: (q, dx, distance of
    v/dx to the nearest rounding boundary)."""
    v = np.asarray(v, np.float64).reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    dx = amax / 127.0
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(dx[:, None] > 0, v / dx[:, None], 0.0)
    q = np.clip(round_half_away(r), -127, 127)
    margin = np.abs(np.abs(r - np.trunc(r)) - 0.5)
    return q.astype(np.int64).reshape(-1), dx, margin.reshape(-1)


def ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(x).astype(np.float64)


def sigmoid64(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))


def silu64(z):
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def parse_golden(path):
    """Blocks of 'key values...' lines up to 'end'; '#' starts a comment."""
    blocks, cur = [], {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line == "end":
                blocks.append(cur)
                cur = {}
                continue
            head, *rest = line.split()
            cur.setdefault("_rows", []).append((head, rest))
    return blocks


def expand_hex(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out += [int(v, 16)] * int(n)
        else:
            out.append(int(t, 16))
    return out


def expand_num(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out += [float(v)] * int(n)
        else:
            out.append(float(t))
    return out
