"""Failure detection in the forms that fault no GPU: a device allocation made
to fail on the host side, and bounded on-chip waits made to run out by a short
wait bound. Each failure must be reported (status or device flag), leave no
device memory behind, and leave the handle usable: the next call is bit-exact
against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import lib_desc, make_layer, margin_inputs, to_device

pytestmark = pytest.mark.gpu


def test_create_out_of_memory_at_every_allocation():
    """The n-th device allocation of ds4moe_create fails, for every n: create
    returns DS4MOE_ERR_OOM, hands back no handle and frees what it had
    allocated; once n exceeds the allocations a create makes, create succeeds."""
    import torch
    import deepseek_v4_flash_gb300 as ds4
    spec = synth.MICRO
    w = to_device(synth.gen_layer(spec, 91, 0))
    desc = lib_desc(spec, 100)  # decode and prefill scratch
    ds4.Layer(desc, w).close()  # the library's module (code, static data) is loaded once, here
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n = 1
    try:
        while True:
            ds4.fail_alloc(n)
            try:
                layer = ds4.Layer(desc, w)
            except ds4.Ds4MoeError as e:
                assert e.status == 3, f"allocation {n}: {e}"  # DS4MOE_ERR_OOM
                torch.cuda.synchronize()
                assert torch.cuda.mem_get_info()[0] == free0, f"allocation {n} left device memory behind"
                n += 1
                assert n < 64
                continue
            break
    finally:
        ds4.fail_alloc(0)
    assert n > 10  # weights, scratch and tickets each failed once
    layer.close()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


@pytest.mark.parametrize("spec,T", [(synth.MICRO, 1), (synth.MICRO, 8), (synth.DS4, 1)])
def test_wait_timeout_is_reported_and_handle_recovers(spec, T):
    """Hand-off waits bounded at one cycle give up at once: the device flag
    reports DS4MOE_DEVERR_TIMEOUT, and after it has been read the handle's
    next calls are bit-exact against the oracle again (the completion counters
    a block left unfinished are reset)."""
    import torch
    ora = oracle.get()
    seed = 93
    w = synth.gen_layer(spec, seed, 0)
    ol = ora.layer(spec, w)
    layer = make_layer(spec, w, 64)
    x = margin_inputs(ol, spec, seed, T)
    ref, *_ = ol.forward(x, None, None)
    xd = torch.from_numpy(x).cuda()
    layer.set_wait_limit(1)
    flags = 0
    for _ in range(4):
        layer.forward(xd, torch.zeros_like(xd))
        flags |= layer.device_error()
    assert flags & 4, "no wait ran out at a one-cycle bound"
    layer.set_wait_limit(0)  # the default bound again
    for _ in range(2):
        y = torch.zeros_like(xd)
        layer.forward(xd, y)
        assert layer.device_error() == 0
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    layer.close()
