"""Failure detection without a GPU fault: a pipeline wait that nothing completes gives up after
its limit, reports MOE_STATUS_WAIT_TIMEOUT through the device status word and lets its kernel
return; the context keeps working (a layer run afterwards matches the oracle)."""
import time

import pytest
import torch

import moe_inputs as mi
import block_fp8_mixture_topk_gb300 as moe
from moe_testutil import Layer, assert_output_close, routing_of
import oracle

pytestmark = pytest.mark.gpu
WAIT_TIMEOUT = 0x1


def timed(expire):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_selftest_bounded_wait(expire)
    torch.cuda.synchronize()
    return time.perf_counter() - t0


def test_completed_wait_returns_at_once_without_status():
    moe.moe_get_device_status(clear=True)
    assert timed(False) < 1.0
    assert moe.moe_get_device_status(clear=True) == 0


def test_expired_wait_reports_and_the_context_stays_usable():
    moe.moe_get_device_status(clear=True)
    dt = timed(True)
    assert 1.9 < dt < 60.0, dt                      # the 2 s limit of device time, then return
    assert moe.moe_get_device_status(clear=True) & WAIT_TIMEOUT
    assert moe.moe_get_device_status(clear=True) == 0  # cleared
    wl = mi.WORKLOADS["tiny"]
    layer = Layer(wl)
    hidden, logits = mi.hidden(wl), mi.router_logits(wl)
    rp, okw = routing_of(wl)
    out = layer.forward(hidden.cuda(), logits.cuda(), rp)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(clear=True) == 0
    w13q, w13s, w2q, w2s = layer.oracle_weights(range(wl.E))
    bits = hidden.contiguous().view(torch.int16).numpy().view("uint16")
    ref = oracle.moe_forward(bits, logits.numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize, **okw)["out"]
    assert_output_close(out, ref)
