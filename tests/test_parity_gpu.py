"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.

Bar: expert ids and every integer code bit-exact; floats within the routed-MoE
tolerance (relative L2 <= 1e-4 and max-abs <= 2e-3 * max|ref|) -- and, because
both sides follow the same binary32 operation order, bit-exact as well."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import make_layer, margin_inputs, within_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ora():
    return oracle.get()


_layers = {}


def _layer_pair(ora, spec, seed, max_tokens):
    key = (spec.name, seed, max_tokens)
    if key not in _layers:
        _layers.clear()
        import torch
        torch.cuda.empty_cache()
        w = synth.gen_layer(spec, seed, 0)
        _layers[key] = (w, ora.layer(spec, w), make_layer(spec, w, max_tokens))
    return _layers[key]


def run_case(ora, spec, seed, T, max_tokens=None, y_init=True):
    import torch
    w, ol, layer = _layer_pair(ora, spec, seed, max_tokens or T)
    x = margin_inputs(ol, spec, seed, T)
    tok = synth.gen_token_ids(spec, seed, T) if spec.route == "hash" else None
    y0 = (np.random.default_rng(seed + T).standard_normal(x.shape) * 10).astype(np.float32) if y_init \
        else np.zeros_like(x)
    ref, ids_ref, w_ref, bad = ol.forward(x, y0, tok)
    assert bad == 0
    xd, yd = torch.from_numpy(x).cuda(), torch.from_numpy(y0).cuda()
    td = torch.from_numpy(tok).cuda() if tok is not None else None
    layer.forward(xd, yd, td)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got = yd.cpu().numpy()
    k = spec.top_k
    # routing of every token through ds4moe_route, and the forward's own
    # routing (scratch of its last chunk of <= 64 tokens)
    ids, wts = layer.route(xd, td)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref), "expert ids differ"
    assert np.array_equal(wts.cpu().numpy().view(np.uint32), w_ref.view(np.uint32)), "gate weights differ"
    if T <= 64:
        fids = layer.scratch("ids")[:T * k].view(T, k).cpu().numpy()
        fw = layer.scratch("w")[:T * k].view(T, k).cpu().numpy()
        assert np.array_equal(fids, ids_ref) and np.array_equal(fw.view(np.uint32), w_ref.view(np.uint32))
    assert within_tolerance(got, ref)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
        f"not bit-exact: {np.count_nonzero(got != ref)} of {got.size} differ"
    return x, tok, got, layer


def test_tiny_layer_4_tokens(ora):
    run_case(ora, synth.TINY, 2026, 4)


@pytest.mark.parametrize("T", list(range(1, 17)) + [31, 32, 33, 63, 64, 65])
def test_micro_widths(ora, T):
    run_case(ora, synth.MICRO, 7, T, max_tokens=65)


@pytest.mark.parametrize("T", [1, 7, 64, 130])
def test_micro_hash(ora, T):
    run_case(ora, synth.MICRO_HASH, 9, T, max_tokens=130)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ds4_decode_1_token(ora, seed):
    run_case(ora, synth.DS4, seed, 1)


def test_ds4_batched_decode_32_zipf(ora):
    run_case(ora, synth.DS4_ZIPF, 11, 32)


# The decode dispatcher picks the tokens per unit, the blocks per SM and
# whether activations are staged in shared memory from the token count and
# the shared-memory footprint at the full DeepSeek-V4-Flash shape (the
# handle's max_tokens sizes the bucket table that shares that space), so
# every width class runs at that shape: one-token units (1-2 tokens), four-
# token units (3-4), eight-token units with staged (5-8) and unstaged
# (9-64) activations, a ragged last unit, and max_tokens both equal to the
# call and larger.
@pytest.mark.parametrize("T", [2, 3, 4, 5, 7, 9, 16, 33, 64])
def test_ds4_decode_widths(ora, T):
    run_case(ora, synth.DS4, 81, T)


@pytest.mark.parametrize("T", [2, 5, 9])
def test_ds4_decode_widths_larger_handle(ora, T):
    run_case(ora, synth.DS4, 83, T, max_tokens=64)


@pytest.mark.parametrize("T", [12, 48])
def test_ds4_zipf_decode_hot_experts(ora, T):
    """Zipf(1.1) popularity: hot experts hold more tokens than one unit, so
    they run several passes of eight tokens."""
    run_case(ora, synth.DS4_ZIPF, 85, T)


# ---- 4-bit routed experts (the "q2 with the last 6 layers q4" variant)

@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 9, 33, 64])
def test_micro_q4_widths(ora, T):
    run_case(ora, synth.MICRO_Q4, 91, T, max_tokens=65)


@pytest.mark.parametrize("T", [7, 130])
def test_micro_q4_hash(ora, T):
    run_case(ora, synth.MICRO_Q4_HASH, 93, T, max_tokens=130)


@pytest.mark.parametrize("T", [1, 8])
def test_ds4_q4_decode(ora, T):
    run_case(ora, synth.DS4_Q4, 95, T)


def test_ds4_batch_invariance(ora):
    """At the full shape, each of five tokens routed one by one gives the same
    bits as the five in one call (batched routing and expert units against
    single-token ones)."""
    import torch
    spec, T = synth.DS4, 5
    w, ol, layer = _layer_pair(ora, spec, 87, T)
    x = torch.from_numpy(margin_inputs(ol, spec, 87, T)).cuda()
    yb = torch.zeros(T, spec.hidden, device="cuda")
    layer.forward(x, yb)
    ids_b, w_b = layer.route(x)
    for t in range(T):
        y1 = torch.zeros(1, spec.hidden, device="cuda")
        layer.forward(x[t:t + 1].contiguous(), y1)
        ids1, w1 = layer.route(x[t:t + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(y1[0], yb[t])
        assert torch.equal(ids1[0], ids_b[t]) and torch.equal(w1[0], w_b[t])
    assert layer.device_error() == 0


def test_ds4_hash_prefill_512(ora):
    run_case(ora, synth.DS4_HASH, 13, 512)


def test_intermediate_codes_bit_exact(ora):
    """Activation codes, scales and group sums, and the SwiGLU codes of one
    expert slot, against the oracle's own quantiser and expert evaluation."""
    spec, T = synth.MICRO, 5
    x, tok, got, layer = run_case(ora, spec, 17, T, max_tokens=65)
    H, F, k = spec.hidden, spec.ffn, spec.top_k
    _, ol, _ = _layer_pair(ora, spec, 17, 65)
    xq = layer.scratch("xq")[:T * H].view(T, H).cpu().numpy()
    dx = layer.scratch("dx")[:T * H // 32].view(T, H // 32).cpu().numpy()
    gs = layer.scratch("gs")[:T * H // 16].view(T, H // 16).cpu().numpy()
    ids = layer.scratch("ids")[:T * k].view(T, k).cpu().numpy()
    hq = layer.scratch("hq").view(-1, F)
    dh = layer.scratch("dh").view(-1, F // 32)
    NS = k + spec.n_shared
    for t in range(T):
        q, d, g = ora.quantize(x[t])
        assert np.array_equal(xq[t], q) and np.array_equal(dx[t].view(np.uint32), d.view(np.uint32))
        assert np.array_equal(gs[t], g)
        for j, e in list(enumerate(ids[t])) + [(k, spec.n_experts)]:
            o = ol.expert(int(e), x[t])
            assert np.array_equal(hq[t * NS + j].cpu().numpy(), o["hq"])
            assert np.array_equal(dh[t * NS + j].cpu().numpy().view(np.uint32), o["dh"].view(np.uint32))


def test_route_entry_point(ora):
    import torch
    spec, T = synth.DS4, 8
    w, ol, layer = _layer_pair(ora, spec, 21, 8)
    x = margin_inputs(ol, spec, 21, T)
    ids_ref, w_ref, _, _, _ = ol.route(x)
    ids, wt = layer.route(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.array_equal(wt.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))


def test_linearity_and_determinism(ora):
    """forward(x, y0) == y0 + forward(x, 0) element by element (binary32), and
    two runs give the same bits."""
    import torch
    spec, T = synth.MICRO, 9
    w, ol, layer = _layer_pair(ora, spec, 23, 65)
    x = torch.from_numpy(margin_inputs(ol, spec, 23, T)).cuda()
    y0 = torch.randn(T, spec.hidden, device="cuda") * 50
    y1 = y0.clone()
    layer.forward(x, y1)
    z = torch.zeros_like(y0)
    layer.forward(x, z)
    z2 = torch.zeros_like(y0)
    layer.forward(x, z2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0 + z)
    assert torch.equal(z, z2)


def test_batch_invariance(ora):
    """A token's output does not depend on the other tokens of the call."""
    import torch
    spec, T = synth.MICRO, 12
    w, ol, layer = _layer_pair(ora, spec, 29, 65)
    x = torch.from_numpy(margin_inputs(ol, spec, 29, T)).cuda()
    yb = torch.zeros(T, spec.hidden, device="cuda")
    layer.forward(x, yb)
    for t in range(T):
        y1 = torch.zeros(1, spec.hidden, device="cuda")
        layer.forward(x[t:t + 1].contiguous(), y1)
        torch.cuda.synchronize()
        assert torch.equal(y1[0], yb[t])


def test_forward_host_matches_device(ora):
    import torch
    spec, T = synth.MICRO_HASH, 10
    w, ol, layer = _layer_pair(ora, spec, 31, 130)
    x = synth.gen_x(spec, 31, T)
    tok = synth.gen_token_ids(spec, 31, T)
    ref, *_ = ol.forward(x, None, tok)
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.zeros(T, spec.hidden).pin_memory()
    th = torch.from_numpy(tok).pin_memory()
    layer.forward_host(xh, yh, th)
    assert np.array_equal(yh.numpy().view(np.uint32), ref.view(np.uint32))


def test_bad_token_id_sets_flag_and_skips_token(ora):
    import torch
    spec, T = synth.MICRO_HASH, 6
    w, ol, layer = _layer_pair(ora, spec, 33, 130)
    x = synth.gen_x(spec, 33, T)
    tok = synth.gen_token_ids(spec, 33, T)
    tok[2] = spec.vocab + 5
    tok[4] = -3
    ref, ids_ref, _, bad = ol.forward(x, None, tok)
    assert bad == 2
    yd = torch.zeros(T, spec.hidden, device="cuda")
    layer.forward(torch.from_numpy(x).cuda(), yd, torch.from_numpy(tok).cuda())
    flags = layer.device_error()
    assert flags & 1
    got = yd.cpu().numpy()
    assert np.all(got[2] == 0) and np.all(got[4] == 0)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert layer.device_error() == 0  # cleared


def test_bad_token_id_single_token(ora):
    """One token (the single-token bucketing) whose id is out of range: the
    flag is raised and the token adds nothing, not even the shared expert."""
    import torch
    spec = synth.MICRO_HASH
    w, ol, layer = _layer_pair(ora, spec, 33, 130)
    x = synth.gen_x(spec, 34, 1)
    tok = np.array([spec.vocab + 5], dtype=np.int32)
    y0 = np.random.default_rng(34).standard_normal(x.shape).astype(np.float32)
    ref, _, _, bad = ol.forward(x, y0, tok)
    assert bad == 1 and np.array_equal(ref.view(np.uint32), y0.view(np.uint32))
    yd = torch.from_numpy(y0).cuda()
    layer.forward(torch.from_numpy(x).cuda(), yd, torch.from_numpy(tok).cuda())
    assert layer.device_error() & 1
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert layer.device_error() == 0


@pytest.mark.parametrize("T", [1, 5, 130])
def test_hash_rows_with_repeated_experts(ora, T):
    """Hash-table rows that name one expert twice or thrice: the expert's
    group holds several slots of the same token (single-token and batched
    decode bucketing, and the prefill path at 130 tokens), bit-exact against
    the oracle."""
    import torch
    spec, seed = synth.MICRO_HASH, 51
    w = synth.gen_layer(spec, seed, 0)
    tok = synth.gen_token_ids(spec, seed, T)
    rows = [[3, 3, 5], [6, 6, 6], [1, 2, 1], [7, 0, 7], [4, 4, 2]]
    for i, t in enumerate(tok):
        w["hash_table"][t] = rows[i % len(rows)]
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, max(65, T))
    x = synth.gen_x(spec, seed, T)
    y0 = np.random.default_rng(seed).standard_normal(x.shape).astype(np.float32)
    ref, ids_ref, _, bad = ol.forward(x, y0, tok)
    assert bad == 0
    yd = torch.from_numpy(y0).cuda()
    layer.forward(torch.from_numpy(x).cuda(), yd, torch.from_numpy(tok).cuda())
    assert layer.device_error() == 0
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    layer.close()


def test_nonfinite_input_sets_flag(ora):
    import torch
    spec = synth.MICRO
    w, ol, layer = _layer_pair(ora, spec, 35, 65)
    x = torch.randn(3, spec.hidden, device="cuda")
    x[1, 7] = float("inf")
    y = torch.zeros_like(x)
    layer.forward(x, y)
    assert layer.device_error() & 2


@pytest.mark.parametrize("H", [4096, 416, 256, 16384])
def test_rmsnorm_bit_exact(ora, H):
    """Widths with segments of 128, 13 (a tail of the unrolled chain) and 8
    words staged in shared memory, and a row too wide to stage."""
    import torch
    import deepseek_v4_flash_gb300 as ds4
    rng = np.random.default_rng(37 + H)
    x = (rng.standard_normal((33, H)) * rng.uniform(0.01, 100, (33, 1))).astype(np.float32)
    ref = ora.rmsnorm(x, 1e-6)
    xd = torch.from_numpy(x).cuda()
    out = torch.empty_like(xd)
    ds4.rmsnorm(xd, out, 1e-6)
    ds4.rmsnorm(xd, xd, 1e-6)  # in place
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert torch.equal(out, xd)


# ds4moe_forward_rmsnorm: the RMSNorm folded into the router kernel, on rows
# of very different scales, in place (y = x, the residual stream) and into a
# separate y, against the oracle's RMSNorm followed by its forward. Covers
# the decode path (one token per router cluster), the prefill path (clusters
# of eight tokens from 16 tokens on), the fp32 router (TINY) and hash routing.
@pytest.mark.parametrize("spec,seed,T,pf", [
    (synth.MICRO, 61, 1, False), (synth.MICRO, 61, 2, False), (synth.MICRO, 61, 9, False),
    (synth.MICRO, 61, 64, False), (synth.MICRO, 61, 130, False),
    (synth.MICRO_HASH, 63, 33, False), (synth.TINY, 65, 4, False),
    (synth.MICRO, 67, 3, True), (synth.MICRO, 67, 20, True), (synth.TINY, 69, 37, True),
    (synth.MICRO_HASH, 71, 17, True),
    (synth.DS4, 73, 1, False), (synth.DS4, 73, 8, False),
])
def test_forward_rmsnorm_bit_exact(ora, monkeypatch, spec, seed, T, pf):
    import torch
    if pf:
        monkeypatch.setenv("DS4MOE_PREFILL_MIN_TOKENS", "1")
    w = synth.gen_layer(spec, seed, 0)
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, T)
    rng = np.random.default_rng(seed + T)
    x = (synth.gen_x(spec, seed, T) * rng.uniform(0.01, 100, (T, 1))).astype(np.float32)
    tok = synth.gen_token_ids(spec, seed, T) if spec.route == "hash" else None
    y0 = (rng.standard_normal(x.shape) * 10).astype(np.float32)
    xr = ora.rmsnorm(x, 1e-6)
    ref_in_place, _, _, _ = ol.forward(xr, x.copy(), tok)
    ref_sep, _, _, _ = ol.forward(xr, y0.copy(), tok)
    td = torch.from_numpy(tok).cuda() if tok is not None else None
    hd = torch.from_numpy(x).cuda()
    xd, yd = hd.clone(), torch.from_numpy(y0).cuda()
    layer.forward_rmsnorm(xd, yd, 1e-6, td)
    layer.forward_rmsnorm(hd, hd, 1e-6, td)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got_sep, got_in_place = yd.cpu().numpy(), hd.cpu().numpy()
    assert np.array_equal(xd.cpu().numpy(), x), "x was written"
    assert np.array_equal(got_sep.view(np.uint32), ref_sep.view(np.uint32)), \
        f"separate y: {np.count_nonzero(got_sep != ref_sep)} values differ"
    assert np.array_equal(got_in_place.view(np.uint32), ref_in_place.view(np.uint32)), \
        f"in place: {np.count_nonzero(got_in_place != ref_in_place)} values differ"
    layer.close()


def test_forward_rmsnorm_rejects_overlap_and_misalignment(ora):
    import torch
    import deepseek_v4_flash_gb300 as ds4
    spec = synth.MICRO
    w, ol, layer = _layer_pair(ora, spec, 39, 65)
    buf = torch.zeros(8 * spec.hidden + 4, device="cuda")
    x = buf[:4 * spec.hidden].view(4, spec.hidden)
    with pytest.raises(ds4.Ds4MoeError):  # y overlaps x by part
        layer.forward_rmsnorm(x, buf[spec.hidden:5 * spec.hidden].view(4, spec.hidden))
    with pytest.raises(ds4.Ds4MoeError):  # x not 16-byte aligned
        layer.forward_rmsnorm(buf[1:1 + 4 * spec.hidden].view(4, spec.hidden), buf[4 * spec.hidden + 4:].view(4, spec.hidden))
    with pytest.raises(ds4.Ds4MoeError):
        layer.forward_rmsnorm(x, x, float("nan"))
    layer.forward_rmsnorm(x, x, 1e-6, n_tok=0)
    assert layer.device_error() == 0


def test_empty_and_too_many_tokens(ora):
    import torch
    import deepseek_v4_flash_gb300 as ds4
    spec = synth.MICRO
    w, ol, layer = _layer_pair(ora, spec, 39, 65)
    x = torch.zeros(66, spec.hidden, device="cuda")
    y = torch.zeros_like(x)
    layer.forward(x, y, n_tok=0)
    with pytest.raises(ds4.Ds4MoeError):
        layer.forward(x, y, n_tok=66)
    with pytest.raises(ds4.Ds4MoeError):
        layer.forward(x, x, n_tok=3)  # y must not alias x


# ---- the prefill path (tensor-core grouped GEMM), forced onto small calls
# by lowering the token threshold before the layer is created

@pytest.fixture
def prefill_always(monkeypatch):
    monkeypatch.setenv("DS4MOE_PREFILL_MIN_TOKENS", "1")


@pytest.mark.parametrize("spec,seed,T", [
    (synth.MICRO, 51, 1), (synth.MICRO, 51, 2), (synth.MICRO, 51, 7), (synth.MICRO, 51, 16),
    (synth.MICRO, 51, 33), (synth.MICRO, 51, 64),
    (synth.TINY, 53, 4),                 # Q8_0 routed experts, fp32 router
    (synth.MICRO_HASH, 55, 130),         # hash routing
    (synth.MICRO_Q4, 97, 1), (synth.MICRO_Q4, 97, 40),      # 4-bit routed experts
    (synth.MICRO_Q4_HASH, 99, 130),
])
def test_prefill_path_bit_exact(ora, prefill_always, spec, seed, T):
    run_case(ora, spec, seed, T, max_tokens=max(T, 64))


def test_prefill_multi_pass_experts(ora, prefill_always):
    """300 tokens over 8 experts (top-3): every expert sees more than one pass
    of 32 tokens, the shared expert ten."""
    run_case(ora, synth.MICRO, 57, 300, max_tokens=300)


def test_prefill_chunks(ora, monkeypatch):
    """A call larger than the prefill chunk runs chunk by chunk."""
    monkeypatch.setenv("DS4MOE_PREFILL_MIN_TOKENS", "65")
    run_case(ora, synth.MICRO_HASH, 59, 200, max_tokens=200)


def test_ds4_prefill_small(ora, prefill_always):
    run_case(ora, synth.DS4, 61, 5)


def test_ds4_zipf_prefill_256(ora):
    """Zipf(1.1) expert popularity over 256 tokens: hot experts take several
    passes on the prefill path."""
    run_case(ora, synth.DS4_ZIPF, 63, 256)


def test_ds4_q4_prefill_256(ora):
    """4-bit routed experts at the full layer shape on the prefill path."""
    run_case(ora, synth.DS4_Q4, 101, 256)


def test_decode_and_prefill_paths_agree(ora, monkeypatch):
    """The same tokens through the decode kernels and through the prefill
    kernels give the same bits."""
    import torch
    spec, T = synth.MICRO, 40
    w = synth.gen_layer(spec, 65, 0)
    ol = ora.layer(spec, w)
    x = torch.from_numpy(margin_inputs(ol, spec, 65, T)).cuda()
    monkeypatch.setenv("DS4MOE_PREFILL_MIN_TOKENS", "1")
    lp = make_layer(spec, w, T)
    monkeypatch.setenv("DS4MOE_PREFILL_MIN_TOKENS", "100000")
    ld = make_layer(spec, w, T)
    yp = torch.zeros(T, spec.hidden, device="cuda")
    yd = torch.zeros_like(yp)
    lp.forward(x, yp)
    ld.forward(x, yd)
    torch.cuda.synchronize()
    assert lp.device_error() == 0 and ld.device_error() == 0
    assert torch.equal(yp, yd)
    lp.close()
    ld.close()


def test_prefill_bad_token_ids(ora, prefill_always):
    """Hash token ids outside the table on the prefill path: the flag is set
    and those tokens add nothing, the others are exact."""
    import torch
    spec, T = synth.MICRO_HASH, 150
    w = synth.gen_layer(spec, 67, 0)
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, T)
    x = synth.gen_x(spec, 67, T)
    tok = synth.gen_token_ids(spec, 67, T)
    tok[3] = spec.vocab
    tok[77] = -1
    tok[149] = 1 << 30
    ref, _, _, bad = ol.forward(x, None, tok)
    assert bad == 3
    yd = torch.zeros(T, spec.hidden, device="cuda")
    layer.forward(torch.from_numpy(x).cuda(), yd, torch.from_numpy(tok).cuda())
    assert layer.device_error() & 1
    got = yd.cpu().numpy()
    assert np.all(got[[3, 77, 149]] == 0)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    layer.close()


def test_prefill_more_tokens_than_one_chunk(ora):
    """4100 tokens: one prefill chunk of 4096 and a second of 4."""
    import torch
    spec, T = synth.MICRO, 4100
    w = synth.gen_layer(spec, 69, 0)
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, T)
    x = synth.gen_x(spec, 69, T)
    ref, _, _, _ = ol.forward(x, None, None)
    yd = torch.zeros(T, spec.hidden, device="cuda")
    layer.forward(torch.from_numpy(x).cuda(), yd)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got = yd.cpu().numpy()
    assert within_tolerance(got, ref)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    layer.close()


def test_forward_host_replays(ora):
    """Decode-sized host calls replay one captured graph per token count:
    repeated calls with new inputs, several counts (the first call of each
    captures), pinned and pageable host tensors, learned and hash routing,
    each bit-exact against the oracle."""
    import torch
    for spec, seed, mt in ((synth.MICRO, 41, 65), (synth.MICRO_HASH, 43, 130)):
        w, ol, layer = _layer_pair(ora, spec, seed, mt)
        for i, T in enumerate((1, 3, 1, 64, 3, 1)):
            x = margin_inputs(ol, spec, seed + 7 * i, T)
            tok = synth.gen_token_ids(spec, seed + 7 * i, T) if spec.route == "hash" else None
            y0 = np.random.default_rng(seed + i).standard_normal(x.shape).astype(np.float32)
            ref, *_ = ol.forward(x, y0, tok)
            pin = i % 2 == 0
            xh, yh = torch.from_numpy(x), torch.from_numpy(y0.copy())
            th = torch.from_numpy(tok) if tok is not None else None
            if pin:
                xh, yh = xh.pin_memory(), yh.pin_memory()
                th = th.pin_memory() if th is not None else None
            layer.forward_host(xh, yh, th)
            assert np.array_equal(yh.numpy().view(np.uint32), ref.view(np.uint32)), (spec.name, T, pin)
        assert layer.device_error() == 0


def test_prefill_forward_host(ora, prefill_always):
    import torch
    spec, T = synth.MICRO, 70
    w = synth.gen_layer(spec, 71, 0)
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, T)
    x = synth.gen_x(spec, 71, T)
    y0 = (np.random.default_rng(71).standard_normal(x.shape) * 3).astype(np.float32)
    ref, _, _, _ = ol.forward(x, y0, None)
    yh = torch.from_numpy(y0.copy()).pin_memory()
    layer.forward_host(torch.from_numpy(x).pin_memory(), yh)
    assert np.array_equal(yh.numpy().view(np.uint32), ref.view(np.uint32))
    layer.close()


def test_prefill_nonfinite_input_sets_flag(ora, prefill_always):
    import torch
    spec = synth.MICRO
    w = synth.gen_layer(spec, 73, 0)
    layer = make_layer(spec, w, 80)
    x = torch.randn(80, spec.hidden, device="cuda")
    x[40, 3] = float("nan")
    y = torch.zeros_like(x)
    layer.forward(x, y)
    assert layer.device_error() & 2
    layer.close()


def test_oracle_exp_against_cuda_expf(ora):
    """The canonical exp (Cody-Waite reduction, degree-7 Taylor) against the
    GPU's own expf over a dense sweep (a check of the method, not a parity
    requirement: both sides of the parity tests use the canonical exp). The
    canonical exp is within 1 ulp of the correctly rounded value, the GPU's
    expf within its documented 2 ulp, so the two differ by at most 3."""
    import torch
    z = np.linspace(-87.0, 88.0, 20001).astype(np.float32)
    cuda = torch.exp(torch.from_numpy(z).cuda()).cpu().numpy()
    mine = np.array([float(ora.exp(float(v))) for v in z], dtype=np.float32)
    true = np.exp(z.astype(np.float64)).astype(np.float32)

    def ulps(a, b):
        return np.abs(a.view(np.int32).astype(np.int64) - b.view(np.int32).astype(np.int64))

    assert int(ulps(mine, true).max()) <= 1
    assert int(ulps(cuda, true).max()) <= 2
    assert int(ulps(mine, cuda).max()) <= 3
