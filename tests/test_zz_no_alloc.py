"""ds4moe_route_noalloc (routing with no handle and no device allocation,
scratch in a fixed device array) against ds4moe_route on the same layer and
inputs: expert ids bit-exact, weights within the routed-MoE float tolerance
(and bit-exact, both sides following the same binary32 order), on two calls
in a row that share the fixed scratch.

Collected last on purpose: it must pass both alone in a fresh process and
after every other test has run in the same process."""
from dataclasses import replace

import numpy as np
import pytest

import synth
from tests.helpers import lib_desc, make_layer, to_device, within_tolerance

pytestmark = pytest.mark.gpu

# DS4 router shapes (H 4096, 256 experts, top-6, Q8_0 router) with small
# experts: only the router matters here.
DS4_ROUTER_SMALL = replace(synth.DS4_ROUTER_ONLY, name="ds4-router-small", ffn=64)


def _setup(spec, seed, max_tokens):
    w = synth.gen_layer(spec, seed, 0)
    layer = make_layer(spec, w, max_tokens)
    router = to_device({k: w[k] for k in ("router_w", "router_bias", "hash_table") if k in w})
    return layer, router


def _inputs(spec, seed, T):
    import torch
    x = torch.from_numpy(synth.gen_x(spec, seed, T)).cuda()
    tok = torch.from_numpy(synth.gen_token_ids(spec, seed, T)).cuda() if spec.route == "hash" else None
    return x, tok


def _same(a_ids, a_w, b_ids, b_w):
    ids_a, ids_b = a_ids.cpu().numpy(), b_ids.cpu().numpy()
    w_a, w_b = a_w.cpu().numpy(), b_w.cpu().numpy()
    assert np.array_equal(ids_a, ids_b), "expert ids differ"
    assert within_tolerance(w_a, w_b)
    assert np.array_equal(w_a.view(np.uint32), w_b.view(np.uint32)), "weights not bit-exact"


@pytest.mark.parametrize("spec,seed,sizes", [
    (DS4_ROUTER_SMALL, 41, (8, 64)),   # 64 tokens fill the 512 KiB scratch at 256 experts
    (synth.TINY, 43, (4, 37)),         # fp32 router, 16 experts
    (synth.MICRO_HASH, 45, (7, 300)),  # hash routing (no scratch)
])
def test_noalloc_matches_route_on_two_calls(spec, seed, sizes):
    import torch
    import deepseek_v4_flash_gb300 as ds4
    layer, router = _setup(spec, seed, max(sizes))
    desc = lib_desc(spec, max(sizes))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ins = [_inputs(spec, seed + 100 * i, T) for i, T in enumerate(sizes)]
    # two calls back to back on one stream; the second reuses the scratch
    outs = [ds4.route_noalloc(desc, router, x, tok, err_flags=err) for x, tok in ins]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (x, tok), (ids, w) in zip(ins, outs):
        ref_ids, ref_w = layer.route(x, tok)
        torch.cuda.synchronize()
        _same(ids, w, ref_ids, ref_w)
    assert layer.device_error() == 0


def test_noalloc_rejects_more_tokens_than_scratch():
    import torch
    import deepseek_v4_flash_gb300 as ds4
    spec = DS4_ROUTER_SMALL
    desc = lib_desc(spec, 65)
    w = {"router_w": torch.zeros(synth.tensor_nbytes(spec, "router_w"), dtype=torch.uint8, device="cuda"),
         "router_bias": torch.zeros(spec.n_experts, dtype=torch.float32, device="cuda")}
    x = torch.zeros(65, spec.hidden, device="cuda")
    with pytest.raises(ds4.Ds4MoeError) as e:
        ds4.route_noalloc(desc, w, x)
    assert e.value.status == 2  # DS4MOE_ERR_UNSUPPORTED: 65 * 32 * 256 > 512 KiB
    ids, wt = ds4.route_noalloc(desc, w, x, n_tok=64)  # the largest call that fits
    torch.cuda.synchronize()
    assert ids.shape == (64, spec.top_k) and bool((ids >= 0).all())
