"""The 43-layer stack of DeepSeek-V4-Flash-shaped MoE FFN layers (layers 0-2
hash routed, 3-42 learned top-6 + bias): a residual stream h of 4096 fp32 per
token passes through every layer as h <- h + MoE_l(RMSNorm(h)), as decode at
batch 1 and 8 and as a 4096-token prefill. Batch 1 runs twice: as
ds4moe_rmsnorm into a buffer then ds4moe_forward, and as
ds4moe_forward_rmsnorm on h in place (the RMSNorm folded into the router
kernel); batch 8 and the prefill take the folded form.

Each layer's weights are generated, uploaded, used by all three streams and
freed in turn, so the device holds one layer at a time. At every layer the
CUDA path's stream is compared with the oracle's bit for bit: in full for the
decode streams, on a sample of tokens for the prefill stream (the oracle
follows only those tokens; every layer treats each token on its own, so the
sample's rows are exact). No routing margin can be imposed on a stream that
evolves through 43 layers; both sides take every top-k decision in the same
binary32 arithmetic instead."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import make_layer

pytestmark = pytest.mark.gpu

EPS = 1e-6
PREFILL_T = 4096
SAMPLE = np.array([0, 1, 777, 2048, 4095])


def test_stack_43_layers_decode_b1_b8_and_prefill_4096():
    import torch
    import deepseek_v4_flash_gb300 as ds4
    ora = oracle.get()
    seed = 2026
    streams = {}
    for name, T, fused in (("b1", 1, False), ("b1-fused", 1, True), ("b8", 8, True), ("prefill", PREFILL_T, True)):
        x0 = synth.gen_x(synth.DS4, seed + T, T)
        tok = synth.gen_token_ids(synth.DS4_HASH, seed + T, T)
        rows = SAMPLE if name == "prefill" else np.arange(T)
        streams[name] = dict(
            T=T, rows=rows, fused=fused, h=torch.from_numpy(x0).cuda(), xn=torch.empty(T, synth.DS4.hidden, device="cuda"),
            tok=torch.from_numpy(tok).cuda(), tok_ref=np.ascontiguousarray(tok[rows]),
            h_ref=np.ascontiguousarray(x0[rows]))
    for l in range(synth.N_STACK_LAYERS):
        spec = synth.stack_layer_spec(l)
        w = synth.gen_layer(spec, seed, l)
        layer = make_layer(spec, w, PREFILL_T)
        ol = ora.layer(spec, w)
        for name, s in streams.items():
            hashed = spec.route == "hash"
            if s["fused"]:
                layer.forward_rmsnorm(s["h"], s["h"], EPS, s["tok"] if hashed else None)
            else:
                ds4.rmsnorm(s["h"], s["xn"], EPS)
                layer.forward(s["xn"], s["h"], s["tok"] if hashed else None)
            xr = ora.rmsnorm(s["h_ref"], EPS)
            s["h_ref"], _, _, bad = ol.forward(xr, s["h_ref"], s["tok_ref"] if hashed else None)
            assert bad == 0
        torch.cuda.synchronize()
        assert layer.device_error() == 0, f"layer {l}"
        for name, s in streams.items():
            got = s["h"].cpu().numpy()[s["rows"]]
            assert np.all(np.isfinite(got)), f"layer {l} {name}"
            assert np.array_equal(got.view(np.uint32), s["h_ref"].view(np.uint32)), \
                f"layer {l} ({spec.name}), stream {name}: {np.count_nonzero(got != s['h_ref'])} values differ"
        layer.close()
        del w, ol
