"""Pins for the CPU oracle: each check ties one oracle function to something
other than itself -- a hand-worked value, a closed form, an exact float64 /
int64 brute force, an invariant, or a special case that reduces to a library
routine. Each check takes an ``oracle.Oracle`` so the planted-mistake test can
run the same checks against deliberately broken builds.
"""
import math
import os

import numpy as np

import synth
from tests import refmath as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- formats --

def check_binary16(ora):
    with open(os.path.join(GOLDEN, "binary16.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) != 2:
                continue
            bits, val = int(line[0], 16), float(line[1])
            got = ora.half(bits)
            assert got == val, (hex(bits), got, val)
            # and numpy's own binary16 agrees with the table
            assert float(np.array([bits], np.uint16).view(np.float16)[0]) == val


def _golden_q2s_blocks():
    out = []
    for blk in R.parse_golden(os.path.join(GOLDEN, "q2s_superblock.txt")):
        f = {}
        vals = []
        for head, rest in blk["_rows"]:
            if head in ("block",):
                continue
            if head in ("sm", "qs"):
                f[head] = R.expand_hex(rest)
            elif head in ("d", "dmin"):
                f[head] = int(rest[0], 16)
            else:
                vals.append((int(head), float(rest[0])))
        assert len(f["sm"]) == 16 and len(f["qs"]) == 64, f
        raw = bytes(f["sm"]) + bytes(f["qs"]) + f["d"].to_bytes(2, "little") + f["dmin"].to_bytes(2, "little")
        out.append((np.frombuffer(raw, np.uint8).copy(), vals))
    return out


def check_q2s_dequant_golden(ora):
    blocks = _golden_q2s_blocks()
    assert len(blocks) == 3
    for raw, vals in blocks:
        got = ora.q2s_dequant(raw)
        ref = R.dequant_q2s(raw, 1, 256)[0]
        for i, v in vals:
            assert got[i] == v, (i, got[i], v)
            assert ref[i] == v, (i, ref[i], v)
        # whole block: oracle and the independent numpy unpacking agree exactly
        assert np.array_equal(got, ref)


def check_q8_dequant_golden(ora):
    for blk in R.parse_golden(os.path.join(GOLDEN, "q8_0_block.txt")):
        d, q, vals = None, None, []
        for head, rest in blk["_rows"]:
            if head == "block":
                continue
            if head == "d":
                d = int(rest[0], 16)
            elif head == "q":
                q = [int(v) for v in rest]
            else:
                vals.append((int(head), float(rest[0])))
        raw = np.frombuffer(d.to_bytes(2, "little") + np.array(q, np.int8).tobytes(), np.uint8).copy()
        got = ora.q8_dequant(raw)
        ref = R.dequant_q8(raw, 1, 32)[0]
        for i, v in vals:
            assert got[i] == v and ref[i] == v, (i, got[i], ref[i], v)
        assert np.array_equal(got.astype(np.float64), ref)


# ------------------------------------------------------------ quantisation --

def check_quantize_golden(ora):
    for blk in R.parse_golden(os.path.join(GOLDEN, "quantize_block.txt")):
        rows = dict(blk["_rows"])
        x = np.array(R.expand_num(rows["x"]), np.float32)
        q, dx, gs = ora.quantize(x)
        assert dx[0] == float(rows["dx"][0])
        assert q.tolist() == [int(v) for v in R.expand_num(rows["q"])]
        assert gs.tolist() == [int(v) for v in rows["gs"]]


def check_quantize_vs_f64(ora, seed=5):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(32 * 512) * rng.choice([1e-3, 1.0, 50.0], 32 * 512)).astype(np.float32)
    q, dx, gs = ora.quantize(v)
    q64, dx64, margin = R.quantize_f64(v)
    # scale: the binary32 rounding of amax/127 (one correctly rounded division)
    assert np.all(np.abs(dx.astype(np.float64) - dx64) <= 0.5 * R.ulp32(dx))
    # codes: identical wherever v/dx is not within 1e-4 of a .5 boundary
    clear = margin > 1e-4
    assert clear.mean() > 0.99
    assert np.array_equal(q.astype(np.int64)[clear], q64[clear])
    assert np.all(np.abs(q.astype(np.int64) - q64) <= 1)
    # group sums are exact sums of the codes
    assert np.array_equal(gs.astype(np.int64), q.astype(np.int64).reshape(-1, 16).sum(1))


# --------------------------------------------------------------- block dots --

def check_block_dots_exact(ora, seed=7):
    """Integer block dots equal the int64 brute force on unpacked fields, and
    their float use reproduces the float64 dot of the dequantised values."""
    rng = np.random.default_rng(seed)
    for trial in range(40):
        sb = rng.integers(0, 256, 84, dtype=np.uint8)
        sb[80:82] = np.frombuffer(np.float16(rng.uniform(0.001, 0.02)).tobytes(), np.uint8)
        sb[82:84] = np.frombuffer(np.float16(rng.uniform(0.001, 0.02)).tobytes(), np.uint8)
        x = rng.standard_normal(256).astype(np.float32)
        xq, dx, gs = ora.quantize(x)
        d, dmin, sc, mn, q = R.unpack_q2s(sb, 1, 256)
        w64 = R.dequant_q2s(sb, 1, 256)[0]
        for j in range(8):
            A, B = ora.q2s_dot(sb, j, xq[32 * j:32 * j + 32], gs[2 * j:2 * j + 2])
            g0, g1 = 2 * j, 2 * j + 1
            qq = q[0, 0]
            a_ref = sum(int(sc[0, 0, g]) * int(np.dot(qq[16 * g:16 * g + 16], xq[16 * g:16 * g + 16].astype(np.int64)))
                        for g in (g0, g1))
            b_ref = sum(int(mn[0, 0, g]) * int(xq[16 * g:16 * g + 16].astype(np.int64).sum()) for g in (g0, g1))
            assert (A, B) == (a_ref, b_ref)
            # float64 identity: sum_i w_i * (dx*xq_i) == dx*(d*A - dmin*B)
            lhs = float(np.dot(w64[32 * j:32 * j + 32], xq[32 * j:32 * j + 32].astype(np.float64))) * float(dx[j])
            rhs = float(dx[j]) * (float(d[0, 0]) * A - float(dmin[0, 0]) * B)
            assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))
        blk = rng.integers(0, 256, 34, dtype=np.uint8)
        blk[0:2] = np.frombuffer(np.float16(rng.uniform(-0.01, 0.01)).tobytes(), np.uint8)
        I = ora.q8_dot(blk, xq[:32])
        assert I == int(np.dot(blk[2:].view(np.int8).astype(np.int64), xq[:32].astype(np.int64)))


def _sum_bound(terms):
    """Recursive-summation error bound (Higham, Accuracy and Stability of
    Numerical Algorithms, eq. 4.4) for n binary32 terms each carrying up to
    3 roundings of its own: (n + 3) * u * sum|t|."""
    t = np.abs(np.asarray(terms, np.float64))
    return (len(t) + 3) * 2.0 ** -24 * t.sum() * 1.0001


def check_row_sum_f64(ora, seed=11):
    """A whole row (CAS order) against the float64 dot of dequantised weights
    and dequantised activations, within the recursive-summation bound."""
    rng = np.random.default_rng(seed)
    for fmt, K in (("q2s", 4096), ("q2s", 2048), ("q8_0", 4096), ("q8_0", 2048)):
        if fmt == "q2s":
            row = np.empty(K // 256 * 84, np.uint8)
            synth.lib().ds4s_q2s(row.ctypes.data, int(rng.integers(1 << 30)), K // 256, 99, 0.01, 1)
        else:
            row = np.empty(K // 32 * 34, np.uint8)
            synth.lib().ds4s_q8(row.ctypes.data, int(rng.integers(1 << 30)), K // 32, 98, 0.02, 1)
        w = R.dequant(fmt, row, 1, K)[0]
        x = rng.standard_normal(K).astype(np.float32)
        xq, dx, gs = ora.quantize(x)
        xd = xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32)
        terms = (w * xd).reshape(-1, 32).sum(1)
        for S in (1, 8):
            got = float(ora.row(fmt, row, K, xq, dx, gs, S))
            ref = float(terms.sum())
            assert abs(got - ref) <= _sum_bound(terms) + 1e-30, (fmt, K, S, got, ref)


def _segment_row(name="cas_segments.txt"):
    """(row bytes, x, expected sums by S) of a hand-worked Q8_0 row."""
    blk = R.parse_golden(os.path.join(GOLDEN, name))[0]
    rows = dict(blk["_rows"])
    d = [int(v, 16) for v in rows["d"]]
    w = [int(v) for v in rows["w"]]
    nb = len(d)
    row = np.zeros(nb * 34, np.uint8)
    for b in range(nb):
        row[34 * b:34 * b + 2] = np.frombuffer(d[b].to_bytes(2, "little"), np.uint8)
        row[34 * b + 2] = np.uint8(w[b] & 0xFF)
    x = np.zeros(32 * nb, np.float32)
    x[::32] = 127.0
    return row, x, {k: float(rows[k][0]) for k in ("S1", "S4", "S8")}


def check_cas_segment_order(ora):
    """The segment structure of the row sum, on rows whose orders round
    differently (hand-worked in golden/cas_segments.txt, cas_segments16.txt)."""
    for name in ("cas_segments.txt", "cas_segments16.txt"):
        row, x, want = _segment_row(name)
        xq, dx, gs = ora.quantize(x)
        assert np.all(dx == 1.0)
        for S in (1, 4, 8):
            assert float(ora.row("q8_0", row, x.size, xq, dx, gs, S)) == want[f"S{S}"], (name, S)


def check_expert_rows_use_eight_segments(ora):
    """Routed and shared expert rows are summed in 8 segments: the hand-worked
    16-block row as gate row 0 of a routed expert and of the shared expert."""
    row, x, want = _segment_row("cas_segments16.txt")
    H, F, rb, rbd = 512, 64, 16 * 34, 2 * 34
    spec = synth.LayerSpec("seg", H, 2, 1, F, 1, "learned", 0, "f32", "q8_0", "q8_0",
                           router_sigma=0.0, bias="none")
    gate = np.zeros(2 * F * rb, np.uint8)
    gate[:rb] = row                                # routed expert 0, row 0
    sh_gate = np.zeros(F * rb, np.uint8)
    sh_gate[:rb] = row                             # shared expert, row 0
    w = {"router_w": np.zeros((2, H), np.float32), "router_bias": np.zeros(2, np.float32),
         "gate": gate, "up": np.zeros_like(gate), "down": np.zeros(2 * H * rbd, np.uint8),
         "sh_gate": sh_gate, "sh_up": np.zeros_like(sh_gate), "sh_down": np.zeros(H * rbd, np.uint8)}
    L = ora.layer(spec, w)
    assert float(L.expert(0, x)["g"][0]) == want["S8"]
    assert float(L.expert(2, x)["g"][0]) == want["S8"]


# ----------------------------------------------------------- exp / sigmoid --

def check_exp(ora):
    z = np.concatenate([np.linspace(-87, 88, 20001), np.linspace(-1, 1, 4001),
                        [0.0, -0.0, 1e-30, -1e-30, 0.5, -0.5, 10.0, -10.0]]).astype(np.float32)
    got = np.array([float(ora.exp(v)) for v in z])
    ref = np.exp(z.astype(np.float64))
    err_ulp = np.abs(got - ref) / R.ulp32(ref)
    assert err_ulp.max() <= 2.0, err_ulp.max()
    assert float(ora.exp(0.0)) == 1.0
    # clamping: beyond the range the value of the clamp point
    assert float(ora.exp(-200.0)) == float(ora.exp(-87.0))
    assert float(ora.exp(500.0)) == float(ora.exp(88.0))
    assert math.isfinite(float(ora.exp(88.0)))


def check_sigmoid_silu(ora):
    z = np.linspace(-30, 30, 6001).astype(np.float32)
    s = np.array([float(ora.sigmoid(v)) for v in z])
    assert np.all(np.abs(s - R.sigmoid64(z)) <= 4 * R.ulp32(R.sigmoid64(z)) + 1e-45)
    h = np.array([float(ora.silu(v)) for v in z])
    ref = R.silu64(z)
    assert np.all(np.abs(h - ref) <= 4 * R.ulp32(ref) + 1e-45)
    assert float(ora.sigmoid(0.0)) == 0.5 and float(ora.silu(0.0)) == 0.0


def check_rmsnorm(ora, seed=13):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((5, 4096)) * rng.uniform(0.1, 100, (5, 1))).astype(np.float32)
    out = ora.rmsnorm(x, 1e-6)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt((x64 ** 2).mean(1, keepdims=True) + 1e-6)
    assert np.all(np.abs(out - ref) <= 1e-6 * np.abs(ref).max(1, keepdims=True) + 8 * R.ulp32(ref))
    # special case: a constant row c normalises to c/sqrt(c^2+eps) ~ sign(c)
    c = np.full((1, 256), 3.0, np.float32)
    assert np.allclose(ora.rmsnorm(c, 0.0), 1.0, rtol=0, atol=2e-7)
    # eps matters when mean(x^2) is comparable: c = 1e-3, eps = 1e-6 -> 1/sqrt(2)
    c = np.full((1, 256), 1e-3, np.float32)
    assert np.allclose(ora.rmsnorm(c, 1e-6), 2 ** -0.5, rtol=1e-6, atol=0)


# ----------------------------------------------------------------- routing --

def _f32_router_layer(ora, logits, bias, k):
    E, H = len(logits), 256
    spec = synth.LayerSpec("hand", H, E, k, 128, 0, "learned", 0, "f32", "q8_0", "q8_0",
                           router_sigma=0.0, bias="none")
    rw = np.zeros((E, H), np.float32)
    rw[:, 0] = np.array(logits, np.float32)
    w = {"router_w": rw, "router_bias": np.array(bias, np.float32),
         "gate": np.zeros(1, np.uint8), "up": np.zeros(1, np.uint8), "down": np.zeros(1, np.uint8)}
    L = ora.layer(spec, w)
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    return L, x


def check_topk_golden(ora):
    blocks = R.parse_golden(os.path.join(GOLDEN, "topk_example.txt"))
    logits = None
    for blk in blocks:
        rows = dict(blk["_rows"])
        logits = [float(v) for v in rows.get("logits", [])] or logits
        bias = [float(v) for v in rows["bias"]]
        want = [int(v) for v in rows["ids"]]
        L, x = _f32_router_layer(ora, logits, bias, len(want))
        ids, w, lg, keys, bad = L.route(x)
        assert bad == 0
        assert ids[0].tolist() == want, (ids, want)
        assert np.array_equal(lg[0], np.array(logits, np.float32))
        s = R.sigmoid64(np.array(logits, np.float32))[want]
        assert np.allclose(w[0], s / s.sum(), rtol=4e-7, atol=0)


def _margin_ok(keys, k, margin=1e-5):
    ks = np.sort(keys.astype(np.float64))[::-1]
    return np.all(np.diff(ks[:k + 1]) < -margin)


def check_route_invariants(ora, spec=synth.MICRO, seed=21, T=64):
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    x = synth.gen_x(spec, seed, T)
    ids, wt, logits, keys, bad = L.route(x)
    assert bad == 0
    E, k, H = spec.n_experts, spec.top_k, spec.hidden
    W = R.dequant(spec.router_fmt, w["router_w"], E, H)
    for t in range(T):
        # k distinct ids in range, weights positive and summing to 1
        assert len(set(ids[t].tolist())) == k and ids[t].min() >= 0 and ids[t].max() < E
        assert np.all(wt[t] > 0) and abs(float(wt[t].astype(np.float64).sum()) - 1.0) <= k * 2.0 ** -23
        # logits: float64 brute force (dequantised router, dequantised x or raw x)
        if spec.router_fmt == "f32":
            ref = W @ x[t].astype(np.float64)
            bound = (H + 3) * 2.0 ** -24 * (np.abs(W) @ np.abs(x[t].astype(np.float64)))
        else:
            xq, dx, gs = ora.quantize(x[t])
            xd = xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32)
            terms = (W * xd).reshape(E, -1, 32).sum(2)
            ref = terms.sum(1)
            bound = (terms.shape[1] + 3) * 2.0 ** -24 * np.abs(terms).sum(1) * 1.0001
        assert np.all(np.abs(logits[t] - ref) <= bound + 1e-30)
        # keys = sigmoid(logit) + bias within a few ulp
        s64 = R.sigmoid64(logits[t])
        kref = s64 + w["router_bias"].astype(np.float64)
        assert np.all(np.abs(keys[t] - kref) <= 4 * R.ulp32(s64) + R.ulp32(kref))
        # selection: a stable descending arg-sort of the keys (library routine)
        order = np.argsort(-keys[t].astype(np.float64), kind="stable")
        assert ids[t].tolist() == order[:k].tolist()
        # renormalised weights against float64
        s = R.sigmoid64(logits[t])[ids[t]]
        assert np.allclose(wt[t], s / s.sum(), rtol=6e-7, atol=0)


def check_route_k_equals_E(ora, seed=23):
    spec = synth.LayerSpec("kE", 256, 8, 8, 128, 1, "learned", 0, "f32", "q8_0", "q8_0",
                           router_sigma=0.05, bias="uniform")
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    x = synth.gen_x(spec, seed, 8)
    ids, wt, lg, keys, bad = L.route(x)
    for t in range(8):
        assert ids[t].tolist() == np.argsort(-keys[t].astype(np.float64), kind="stable").tolist()
        s = R.sigmoid64(lg[t])
        assert np.allclose(wt[t], s[ids[t]] / s.sum(), rtol=6e-7)


def check_hash_route(ora, seed=25):
    spec = synth.MICRO_HASH
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    tok = synth.gen_token_ids(spec, seed, 50)
    tok[3] = spec.vocab - 1
    tok[4] = 0
    x = synth.gen_x(spec, seed, 50)
    ids, wt, _, _, bad = L.route(x, tok)
    assert bad == 0
    assert np.array_equal(ids, w["hash_table"][tok])
    assert np.all(wt == np.float32(1.0) / np.float32(spec.top_k))
    # table rows: k distinct experts each
    t = w["hash_table"]
    assert np.all(np.sort(t, 1)[:, 1:] != np.sort(t, 1)[:, :-1])
    # out-of-range ids are reported, not read
    tok2 = np.array([spec.vocab, -1, 5], np.int32)
    ids2, wt2, _, _, bad2 = L.route(x[:3], tok2)
    assert bad2 == 2 and np.all(ids2[:2] == -1) and np.all(wt2[:2] == 0)
    assert np.array_equal(ids2[2], t[5])


# ------------------------------------------------------------------ expert --

def check_expert_stages(ora, spec=synth.MICRO, seed=31, experts=(0, 3, None)):
    """Every stage of one expert against float64, given the previous stage's
    (checked) integer codes."""
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    H, F, E = spec.hidden, spec.ffn, spec.n_experts
    x = synth.gen_x(spec, seed, 1)[0]
    xq, dx, gs = ora.quantize(x)
    xd = xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32)
    for e in experts:
        e = E if e is None else e
        if e == E:
            fmt, Wg, Wu, Wd = spec.shared_fmt, w["sh_gate"], w["sh_up"], w["sh_down"]
        else:
            fmt = spec.routed_fmt
            n_gu, n_d = synth.tensor_nbytes(spec, "gate") // E, synth.tensor_nbytes(spec, "down") // E
            Wg, Wu = w["gate"][e * n_gu:(e + 1) * n_gu], w["up"][e * n_gu:(e + 1) * n_gu]
            Wd = w["down"][e * n_d:(e + 1) * n_d]
        G, U, D = R.dequant(fmt, Wg, F, H), R.dequant(fmt, Wu, F, H), R.dequant(fmt, Wd, H, F)
        o = L.expert(e, x)
        for M, v in ((G, o["g"]), (U, o["u"])):
            terms = (M * xd).reshape(F, -1, 32).sum(2)
            bound = (terms.shape[1] + 3) * 2.0 ** -24 * np.abs(terms).sum(1) * 1.0001
            assert np.all(np.abs(v - terms.sum(1)) <= bound), e
        href = R.silu64(o["g"]) * o["u"].astype(np.float64)
        assert np.all(np.abs(o["h"] - href) <= 6 * R.ulp32(href) + 1e-40)
        q64, dh64, margin = R.quantize_f64(o["h"])
        clear = margin > 1e-4
        assert np.array_equal(o["hq"].astype(np.int64)[clear], q64[clear])
        assert np.all(np.abs(o["dh"] - dh64) <= 0.5 * R.ulp32(o["dh"]))
        assert np.array_equal(o["gsh"].astype(np.int64), o["hq"].astype(np.int64).reshape(-1, 16).sum(1))
        hd = o["hq"].astype(np.float64) * np.repeat(o["dh"].astype(np.float64), 32)
        terms = (D * hd).reshape(H, -1, 32).sum(2)
        bound = (terms.shape[1] + 3) * 2.0 ** -24 * np.abs(terms).sum(1) * 1.0001
        assert np.all(np.abs(o["a"] - terms.sum(1)) <= bound), e


def check_shared_is_swiglu_mlp(ora, spec=synth.TINY, seed=33):
    """With the routed weights scaled to zero the layer is one SwiGLU MLP
    y = Wd (silu(Wg x) * (Wu x)); compare with that textbook MLP in float64 on
    the unquantised x, within the int8 quantisation error."""
    from dataclasses import replace
    w = synth.gen_layer(spec, seed, 0)
    sp0 = replace(spec, route_scale=0.0)
    L = ora.layer(sp0, w)
    x = synth.gen_x(spec, seed, 6)
    y, ids, wt, bad = L.forward(x)
    H, F = spec.hidden, spec.ffn
    G = R.dequant(spec.shared_fmt, w["sh_gate"], F, H)
    U = R.dequant(spec.shared_fmt, w["sh_up"], F, H)
    D = R.dequant(spec.shared_fmt, w["sh_down"], H, F)
    x64 = x.astype(np.float64)
    ref = (R.silu64(x64 @ G.T) * (x64 @ U.T)) @ D.T
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 2e-2, rel
    # and bit-exactly the oracle's own single-expert output
    for t in range(6):
        assert np.array_equal(y[t], L.expert(spec.n_experts, x[t])["a"])


def moe_f64(spec, w, x, tok=None):
    """The textbook routed MoE in float64 on unquantised activations:
    y = sum_j w_j * Wd_j (silu(Wg_j x) * (Wu_j x)) + shared MLP."""
    H, F, E, k = spec.hidden, spec.ffn, spec.n_experts, spec.top_k
    x64 = x.astype(np.float64)
    T = x.shape[0]
    y = np.zeros((T, H))
    n_gu, n_d = synth.tensor_nbytes(spec, "gate") // E, synth.tensor_nbytes(spec, "down") // E
    mats = {}

    def mlp(e, v):
        if e not in mats:
            if e == E:
                f, g, u, d = spec.shared_fmt, w["sh_gate"], w["sh_up"], w["sh_down"]
            else:
                f = spec.routed_fmt
                g, u = w["gate"][e * n_gu:(e + 1) * n_gu], w["up"][e * n_gu:(e + 1) * n_gu]
                d = w["down"][e * n_d:(e + 1) * n_d]
            mats[e] = (R.dequant(f, g, F, H), R.dequant(f, u, F, H), R.dequant(f, d, H, F))
        G, U, D = mats[e]
        return D @ (R.silu64(G @ v) * (U @ v))

    all_ids = []
    for t in range(T):
        if spec.route == "hash":
            ids = w["hash_table"][tok[t]]
            gw = np.full(k, 1.0 / k)
        else:
            Wr = R.dequant(spec.router_fmt, w["router_w"], E, H)
            s = R.sigmoid64(Wr @ x64[t])
            key = s + w["router_bias"].astype(np.float64)
            ids = np.argsort(-key, kind="stable")[:k]
            gw = s[ids] / s[ids].sum()
        all_ids.append(ids)
        for j in range(k):
            y[t] += gw[j] * spec.route_scale * mlp(int(ids[j]), x64[t])
        if spec.n_shared:
            y[t] += mlp(E, x64[t])
    return y, np.array(all_ids)


def check_layer_vs_textbook(ora, spec=synth.TINY, seed=35, T=8, tol=3e-2):
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    x = synth.gen_x(spec, seed, T)
    tok = synth.gen_token_ids(spec, seed, T) if spec.route == "hash" else None
    y, ids, wt, bad = L.forward(x, tok=tok)
    ref, ref_ids = moe_f64(spec, w, x, tok)
    same = np.all(ids == ref_ids, axis=1)
    assert same.mean() >= 0.75, (ids, ref_ids)
    rel = np.linalg.norm(y[same] - ref[same]) / np.linalg.norm(ref[same])
    assert rel < tol, rel


def check_combine_linearity(ora, spec=synth.MICRO, seed=37):
    """y is updated as y + acc with acc independent of y: forward(x, y0) equals
    the binary32 sum y0 + forward(x, 0) element by element."""
    w = synth.gen_layer(spec, seed, 0)
    L = ora.layer(spec, w)
    x = synth.gen_x(spec, seed, 3)
    y0 = np.random.default_rng(seed).standard_normal(x.shape).astype(np.float32) * 100
    y1, *_ = L.forward(x, y0)
    z, *_ = L.forward(x, None)
    assert np.array_equal(y1, (y0 + z).astype(np.float32))
    # threads do not change a bit
    z1, *_ = L.forward(x, None, nthreads=1)
    assert np.array_equal(z, z1)


# ------------------------------------------------------------ dense Q8_0 --

def _dense_golden():
    blk = R.parse_golden(os.path.join(GOLDEN, "dense_q8.txt"))[0]
    rows = dict(blk["_rows"])
    K, N = 64, 2
    x = np.zeros((2, K), np.float32)
    x[0, :3] = [float(v) for v in rows["x0"]]
    x[0, 32:35] = [float(v) for v in rows["x1"]]
    x[1] = -x[0]
    w = np.zeros((N, 2, 34), np.uint8)
    for r in range(N):
        for b, d in enumerate(rows[f"r{r}d"]):
            w[r, b, :2] = np.frombuffer(int(d, 16).to_bytes(2, "little"), np.uint8)
            q = [int(v) for v in rows[f"r{r}q{b}"]]
            w[r, b, 2:2 + len(q)] = np.array(q, np.int8).view(np.uint8)
    y = np.array([float(v) for v in rows["y"]], np.float32)
    return w.reshape(-1), N, K, x, y


def check_dense_golden(ora):
    """Hand-worked dense product (golden/dense_q8.txt), two tokens."""
    w, N, K, x, y = _dense_golden()
    got = ora.dense_q8(w, N, K, x, nthreads=1)
    assert got.tolist() == [y.tolist(), (-y).tolist()], got


def check_dense_segments(ora):
    """Dense rows are summed in min(8, blocks) segments like expert rows: the
    hand-worked 16-block row of golden/cas_segments16.txt gives its S = 8 sum."""
    row, x, want = _segment_row("cas_segments16.txt")
    y = ora.dense_q8(row, 1, x.size, x[None, :], nthreads=1)
    assert float(y[0, 0]) == want["S8"]


def check_dense_identity(ora, seed=17):
    """A closed form: W with one code 1 (scale 1) at column n of row n is the
    identity on the quantised activations, so y[t][n] = dx_t(n) * xq_t[n]
    (rows and columns, and tokens, kept apart)."""
    rng = np.random.default_rng(seed)
    K = N = 96
    w = np.zeros((N, K // 32, 34), np.uint8)
    for n in range(N):
        w[n, n // 32, :2] = np.frombuffer((0x3C00).to_bytes(2, "little"), np.uint8)
        w[n, n // 32, 2 + n % 32] = 1
    x = (rng.standard_normal((3, K)) * 5).astype(np.float32)
    y = ora.dense_q8(w.reshape(-1), N, K, x, nthreads=2)
    for t in range(3):
        q, dx, _ = ora.quantize(x[t])
        assert np.array_equal(y[t], (np.repeat(dx, 32) * q.astype(np.float32)).astype(np.float32))


def check_dense_vs_f64(ora, seed=19):
    """Random rows against the float64 sum of the float64 block terms, within
    the recursive-summation bound (nb + 3) * u * sum |p_b|."""
    rng = np.random.default_rng(seed)
    N, K, T = 40, 768, 2
    blocks = rng.integers(-127, 128, (N, K // 32, 32)).astype(np.int8)
    d = (rng.uniform(1e-3, 2e-2, (N, K // 32))).astype(np.float16)
    w = np.zeros((N, K // 32, 34), np.uint8)
    w[:, :, :2] = d.view(np.uint8).reshape(N, K // 32, 2)
    w[:, :, 2:] = blocks.view(np.uint8)
    x = rng.standard_normal((T, K)).astype(np.float32)
    y = ora.dense_q8(w.reshape(-1), N, K, x, nthreads=3)
    for t in range(T):
        q, dx, _ = ora.quantize(x[t])
        I = (blocks.astype(np.int64) * q.astype(np.int64).reshape(1, K // 32, 32)).sum(-1)
        terms = d.astype(np.float64) * dx.astype(np.float64)[None, :] * I
        ref = terms.sum(1)
        bound = (K // 32 + 3) * 2.0 ** -24 * np.abs(terms).sum(1) + 1e-30
        assert np.all(np.abs(y[t].astype(np.float64) - ref) <= bound)


# ------------------------------------------------------------ 4-bit (Q4S) --

def check_q4s_dequant_golden(ora):
    """The hand-worked 4-bit superblock (golden/q4s_superblock.txt), and the
    whole block against an independent numpy unpacking."""
    blk = R.parse_golden(os.path.join(GOLDEN, "q4s_superblock.txt"))[0]
    f, vals = {}, []
    for head, rest in blk["_rows"]:
        if head == "block":
            continue
        if head in ("sm", "qs"):
            f[head] = R.expand_hex(rest)
        elif head in ("d", "dmin"):
            f[head] = int(rest[0], 16)
        else:
            vals.append((int(head), float(rest[0])))
    assert len(f["sm"]) == 16 and len(f["qs"]) == 128
    raw = np.frombuffer(bytes(f["sm"]) + bytes(f["qs"]) + f["d"].to_bytes(2, "little") +
                        f["dmin"].to_bytes(2, "little"), np.uint8).copy()
    got = ora.q4s_dequant(raw)
    ref = R.dequant_q4s(raw, 1, 256)[0]
    for i, v in vals:
        assert got[i] == v and ref[i] == v, (i, got[i], ref[i], v)
    assert np.array_equal(got, ref)


def check_q4s_dots_exact(ora, seed=23):
    """4-bit block dots against int64 brute force on unpacked fields, and the
    float64 identity sum_i w_i * (dx*xq_i) = dx*(d*A - dmin*B)."""
    rng = np.random.default_rng(seed)
    for trial in range(30):
        sb = rng.integers(0, 256, 148, dtype=np.uint8)
        sb[144:146] = np.frombuffer(np.float16(rng.uniform(0.0005, 0.004)).tobytes(), np.uint8)
        sb[146:148] = np.frombuffer(np.float16(rng.uniform(0.0005, 0.004)).tobytes(), np.uint8)
        x = rng.standard_normal(256).astype(np.float32)
        xq, dx, gs = ora.quantize(x)
        d, dmin, sc, mn, q = R.unpack_q4s(sb, 1, 256)
        w64 = R.dequant_q4s(sb, 1, 256)[0]
        for j in range(8):
            A, B = ora.q4s_dot(sb, j, xq[32 * j:32 * j + 32], gs[2 * j:2 * j + 2])
            qq = q[0, 0]
            a_ref = sum(int(sc[0, 0, g]) * int(np.dot(qq[16 * g:16 * g + 16], xq[16 * g:16 * g + 16].astype(np.int64)))
                        for g in (2 * j, 2 * j + 1))
            b_ref = sum(int(mn[0, 0, g]) * int(xq[16 * g:16 * g + 16].astype(np.int64).sum())
                        for g in (2 * j, 2 * j + 1))
            assert (A, B) == (a_ref, b_ref)
            lhs = float(np.dot(w64[32 * j:32 * j + 32], xq[32 * j:32 * j + 32].astype(np.float64))) * float(dx[j])
            rhs = float(dx[j]) * (float(d[0, 0]) * A - float(dmin[0, 0]) * B)
            assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))


def check_q4s_row_f64(ora, seed=29):
    """4-bit rows in CAS order against the float64 dot of dequantised values,
    within the recursive-summation bound."""
    rng = np.random.default_rng(seed)
    for K in (4096, 512):
        row = np.empty(K // 256 * 148, np.uint8)
        synth.lib().ds4s_q4s(row.ctypes.data, int(rng.integers(1 << 30)), K // 256, 97, 0.002, 1)
        w = R.dequant_q4s(row, 1, K)[0]
        x = rng.standard_normal(K).astype(np.float32)
        xq, dx, gs = ora.quantize(x)
        xd = xq.astype(np.float64) * np.repeat(dx.astype(np.float64), 32)
        terms = (w * xd).reshape(-1, 32).sum(1)
        for S in (1, 8):
            got = float(ora.row("q4s", row, K, xq, dx, gs, S))
            assert abs(got - float(terms.sum())) <= _sum_bound(terms) + 1e-30, (K, S)


def check_q4s_layer(ora):
    """A 4-bit-expert layer: every stage against float64, and the whole layer
    against the textbook float64 MoE on unquantised activations."""
    check_expert_stages(ora, synth.MICRO_Q4, seed=53, experts=(0, 5, None))
    check_layer_vs_textbook(ora, synth.MICRO_Q4, seed=55, T=4, tol=3e-2)


ALL_CHECKS = [
    check_binary16, check_q2s_dequant_golden, check_q8_dequant_golden, check_quantize_golden,
    check_quantize_vs_f64, check_block_dots_exact, check_row_sum_f64, check_cas_segment_order,
    check_expert_rows_use_eight_segments, check_exp, check_sigmoid_silu,
    check_rmsnorm, check_topk_golden, check_route_invariants, check_route_k_equals_E, check_hash_route,
    check_expert_stages, check_shared_is_swiglu_mlp, check_layer_vs_textbook, check_combine_linearity,
    check_dense_golden, check_dense_segments, check_dense_identity, check_dense_vs_f64,
    check_q4s_dequant_golden, check_q4s_dots_exact, check_q4s_row_f64, check_q4s_layer,
]
