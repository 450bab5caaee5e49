"""GPU parity of the dense Q8_0 product (output head, attention projections)
through the C ABI against the CPU oracle: bit-exact (both sides follow the
same binary32 order), and within the float tolerance of the MoE spec."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import within_tolerance

pytestmark = pytest.mark.gpu


def _run(n_out, n_in, T, seed, max_tokens=None, scale=1.0):
    import torch
    import deepseek_v4_flash_gb300 as ds4
    w = synth.gen_q8_matrix(seed, n_out, n_in)
    x = synth.gen_dense_x(seed, T, n_in) * np.float32(scale)
    ref = oracle.get().dense_q8(w, n_out, n_in, x)
    d = ds4.Dense(n_out, n_in, torch.from_numpy(w).cuda(), max_tokens=max_tokens or T)
    y = d.forward(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert d.device_error() == 0
    got = y.cpu().numpy()
    assert within_tolerance(got, ref)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
        f"not bit-exact: {np.count_nonzero(got != ref)} of {got.size} differ"
    d.close()


@pytest.mark.parametrize("n_out,n_in,T", [
    (32, 32, 1),        # one item, one block (one segment)
    (100, 512, 3),      # ragged rows (padding to 128), 16 blocks
    (64, 96, 2),        # 3 blocks: three one-block segments
    (96, 768, 9),       # 24 blocks (stages of 3), two passes of 8 tokens
    (4096, 4096, 5),    # an attention-projection shape
    (1000, 4096, 17),   # three passes, ragged last pass
    (40000, 512, 3),    # more 32-row items than 8-warp blocks have warps: 16 warps per block
    (39008, 256, 9),    # the same, two passes
])
def test_dense_shapes(n_out, n_in, T):
    _run(n_out, n_in, T, seed=n_out + n_in + T)


@pytest.mark.parametrize("n_out,n_in,T", [
    (4096, 4096, 3),    # split rows, passes of 4 tokens
    (4096, 4096, 2),    # split rows, passes of 2 tokens
    (3000, 1024, 1),    # split rows, ragged last item
    (300, 2048, 8),     # split rows, a full pass of 8
])
def test_dense_split_rows(n_out, n_in, T):
    """Rows split by segments over several warps (small matrices, one pass):
    the in-order sum of the stored segment sums gives the unsplit bits."""
    _run(n_out, n_in, T, seed=3 * n_out + n_in + T, max_tokens=8)


def test_dense_repeated_calls():
    """Calls of different widths on one handle: the arrival counters of split
    rows start over after every call."""
    import torch
    import deepseek_v4_flash_gb300 as ds4
    n_out, n_in = 2048, 4096
    w = synth.gen_q8_matrix(41, n_out, n_in)
    d = ds4.Dense(n_out, n_in, torch.from_numpy(w).cuda(), max_tokens=12)
    for i, T in enumerate([1, 8, 3, 12, 1, 5]):
        x = synth.gen_dense_x(100 + i, T, n_in)
        ref = oracle.get().dense_q8(w, n_out, n_in, x)
        got = d.forward(torch.from_numpy(x).cuda()).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {i} (T={T}) not bit-exact"
    assert d.device_error() == 0
    d.close()


def test_dense_launch_geometries_same_bits():
    """Every ring geometry, row split and block-dot step (dp4a, int8 tensor
    cores) gives the oracle's bits."""
    import torch
    import deepseek_v4_flash_gb300 as ds4
    n_out, n_in = 1024, 4096
    w = synth.gen_q8_matrix(43, n_out, n_in)
    d = ds4.Dense(n_out, n_in, torch.from_numpy(w).cuda(), max_tokens=8)
    for T in (1, 3, 8):
        x = synth.gen_dense_x(200 + T, T, n_in)
        ref = oracle.get().dense_q8(w, n_out, n_in, x).view(np.uint32)
        xd = torch.from_numpy(x).cuda()
        for tc in (1, 2):
            for ks, nst, ns in [(1, 6, 1), (2, 3, 2), (4, 2, 4), (8, 2, 8), (8, 3, 1), (4, 6, 8)]:
                d.debug_config(ks, nst, ns, tc)
                got = d.forward(xd).cpu().numpy().view(np.uint32)
                assert np.array_equal(got, ref), f"T={T} ks={ks} nst={nst} ns={ns} tc={tc}"
    with pytest.raises(ds4.Ds4MoeError):
        d.debug_config(3, 0, 0)   # 3 does not divide the 16 blocks of a segment
    with pytest.raises(ds4.Ds4MoeError):
        d.debug_config(0, 7, 0)
    with pytest.raises(ds4.Ds4MoeError):
        d.debug_config(0, 0, 3)
    with pytest.raises(ds4.Ds4MoeError):
        d.debug_config(0, 0, 0, 3)
    assert d.device_error() == 0
    d.close()


def test_dense_output_head_one_token():
    """The output head at full size: 129280 x 4096 (563 MB of Q8_0)."""
    _run(129280, 4096, 1, seed=777)


def test_dense_output_head_eight_tokens():
    """The output head at full size for a pass of 8 tokens (the tensor-core
    step, rows unsplit)."""
    _run(129280, 4096, 8, seed=778)


@pytest.mark.parametrize("T", [1, 8])
def test_dense_extreme_codes(T):
    """Every weight and activation code at +-127: the block dots reach
    +-32 * 127^2 = +-516,128, the largest the format allows, and must come out
    exact on both steps (fp16 codes, f32 accumulation on the tensor cores)."""
    import torch
    import deepseek_v4_flash_gb300 as ds4
    n_out, n_in = 256, 1024
    nb = n_in // 32
    blk = np.zeros((n_out, nb, 34), np.uint8)
    r = np.arange(n_out)[:, None]
    b = np.arange(nb)[None, :]
    d = (0.001 * (1 + (r * 7 + b * 3) % 50)).astype(np.float16)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(n_out, nb, 2)
    sign = np.where(((r + b) % 3 == 0)[..., None], -127, 127).astype(np.int8)
    blk[:, :, 2:] = np.broadcast_to(sign, (n_out, nb, 32)).view(np.uint8)
    w = blk.reshape(-1)
    # each 32-block of x is constant up to sign: codes +-127
    x = np.ones((T, n_in), np.float32)
    x *= np.where((np.arange(n_in)[None, :] // 32 + np.arange(T)[:, None]) % 2 == 0, 1.0, -3.5).astype(np.float32)
    ref = oracle.get().dense_q8(w, n_out, n_in, x)
    dn = ds4.Dense(n_out, n_in, torch.from_numpy(w).cuda(), max_tokens=T)
    y = dn.forward(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert dn.device_error() == 0
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
        f"not bit-exact: {np.count_nonzero(got != ref)} of {got.size} differ"
    dn.close()


def test_dense_wide_input():
    """n_in 16384: passes of 2 tokens (the codes of a pass fit 64 KB)."""
    _run(256, 16384, 3, seed=5)


def test_dense_zero_and_bad_calls():
    import torch
    import deepseek_v4_flash_gb300 as ds4
    w = torch.from_numpy(synth.gen_q8_matrix(1, 64, 256)).cuda()
    d = ds4.Dense(64, 256, w, max_tokens=4)
    x = torch.zeros(4, 256, device="cuda")
    y = d.forward(x)  # all-zero activations: zero scales, zero codes, y = 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(y) == 0
    d.forward(x, n_tok=0)
    with pytest.raises(ds4.Ds4MoeError):
        d.forward(x, n_tok=5)
    x[1, 3] = float("nan")
    d.forward(x)
    assert d.device_error() & 2
    d.close()
    with pytest.raises(ds4.Ds4MoeError):
        ds4.Dense(64, 100, w)  # n_in not a multiple of 32
