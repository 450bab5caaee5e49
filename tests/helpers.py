"""Shared test helpers: turn a synth.LayerSpec into library objects, upload
weights, and build margin-checked inputs with the oracle."""
import numpy as np

import synth

FMTS = {"f32": 0, "q8_0": 1, "q2s": 2, "q4s": 3}


def lib_desc(spec, max_tokens):
    import deepseek_v4_flash_gb300 as ds4
    return ds4.LayerDesc(spec.hidden, spec.n_experts, spec.top_k, spec.ffn, spec.n_shared,
                         ds4.ROUTE_HASH if spec.route == "hash" else ds4.ROUTE_LEARNED, spec.vocab,
                         FMTS[spec.router_fmt], FMTS[spec.routed_fmt], FMTS[spec.shared_fmt],
                         spec.route_scale, max_tokens)


def to_device(w: dict):
    import torch
    out = {}
    for k, v in w.items():
        out[k] = torch.from_numpy(np.ascontiguousarray(v)).cuda()
    return out


def make_layer(spec, w_host, max_tokens):
    import deepseek_v4_flash_gb300 as ds4
    dev = to_device(w_host)
    layer = ds4.Layer(lib_desc(spec, max_tokens), dev)
    del dev  # the library keeps its own copy
    return layer


def margin_ok_rows(keys, k, margin=1e-5):
    """Per row: every gap among the top k+1 keys exceeds `margin`."""
    ks = -np.sort(-keys.astype(np.float64), axis=1)[:, :k + 1]
    gaps = ks[:, :-1] - ks[:, 1:]
    return np.all(gaps > margin, axis=1)


def margin_inputs(ora_layer, spec, seed, T, margin=1e-5, max_attempts=64):
    """x[T][H] whose learned-routing keys have every top-(k+1) gap > margin;
    a failing token row is regenerated from its next stream."""
    attempts = np.zeros(T, dtype=np.int64)
    x = synth.gen_x(spec, seed, T)
    if spec.route != "learned":
        return x
    for _ in range(max_attempts):
        _, _, _, keys, _ = ora_layer.route(x)
        ok = margin_ok_rows(keys, spec.top_k, margin)
        if ok.all():
            return x
        for t in np.nonzero(~ok)[0]:
            attempts[t] += 1
            x[t] = synth.gen_x_row(spec, seed, int(t), int(attempts[t]))
    raise RuntimeError("could not satisfy the routing margin")


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def within_tolerance(got, ref):
    """The float tolerance of the routed-MoE spec: relative L2 <= 1e-4 and
    max |got - ref| <= 2e-3 * max |ref|."""
    ref64 = np.asarray(ref, np.float64)
    return rel_l2(got, ref) <= 1e-4 and float(np.abs(np.asarray(got, np.float64) - ref64).max()) <= \
        2e-3 * float(np.abs(ref64).max())
