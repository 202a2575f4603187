"""Failure detection on the GPU without a GPU fault: host-set fault
injection that must end every pass in a bounded wait with a status the host
reads (MOE_E_TIMEOUT or MOE_E_DEVICE), never a trap or a hang, with the
context usable and the next clean pass correct -- a dropped task type, a
corrupted count, and a task pushed twice caught by the debug claimed-twice
check.  (Survey of the pages: the early-exit and claim-twice races of
m.xxqk.cn/news/657744 section 3.3.)"""
import numpy as np
import pytest

import _harness as hz
import oracle
from persistent_megakernel_sm_gb300 import MOE_E_DEVICE, MOE_E_TIMEOUT, MOE_OK

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[1, 2], ids=["cta", "pair"])
def case(request):
    w, inp = hz.custom_case(300, 256, 16, 4, 384, 1, 0.6)
    dev = hz.upload(inp)
    ref, _ = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k, S=w.S)
    return w, inp, dev, ref, request.param


def _forward(layer, w, dev):
    import torch
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    layer.set_router_bias(dev["bias"])
    layer.forward(dev["x"], dev["router_w"], dev["w_gate"], dev["w_up"], dev["w_down"], out)
    return out


def _clean_pass_is_correct(layer, w, dev, ref):
    got, _ = hz.run_layer(layer, w, dev)
    assert layer.status() == MOE_OK
    hz.check_out(got, ref, "the pass after the fault")


@pytest.mark.parametrize("task_type", [2, 3, 4], ids=["gather", "gateup", "down"])
def test_dropped_task_type_times_out(case, task_type):
    w, inp, dev, ref, pair = case
    layer = hz.make_layer(w, pair=pair, timeout_ns=50_000_000, fault_drop_type=task_type)
    _forward(layer, w, dev)
    assert layer.status() == MOE_E_TIMEOUT
    layer.set_option("fault_drop_type", 0)
    _clean_pass_is_correct(layer, w, dev, ref)
    layer.close()


def test_corrupted_count_is_caught_by_the_plan(case):
    w, inp, dev, ref, pair = case
    layer = hz.make_layer(w, pair=pair, timeout_ns=50_000_000, fault_corrupt_count=3)
    _forward(layer, w, dev)
    assert layer.status() == MOE_E_DEVICE
    from persistent_megakernel_sm_gb300 import lib
    assert b"site 9" in lib.moe_last_error()
    layer.set_option("fault_corrupt_count", 0)
    _clean_pass_is_correct(layer, w, dev, ref)
    layer.close()


def test_debug_claims_pass_clean_runs_unchanged(case):
    # the check itself changes nothing: same bits as without it, status OK
    w, inp, dev, ref, pair = case
    base = hz.make_layer(w, pair=pair)
    a, _ = hz.run_layer(base, w, dev)
    base.close()
    layer = hz.make_layer(w, pair=pair, debug_claims=1)
    for _ in range(2):
        b, _ = hz.run_layer(layer, w, dev)
        assert layer.status() == MOE_OK
        assert np.array_equal(a, b)
    layer.close()


def test_task_pushed_twice_is_caught(case):
    w, inp, dev, ref, pair = case
    layer = hz.make_layer(w, pair=pair, timeout_ns=50_000_000, debug_claims=1, fault_repush=2)
    _forward(layer, w, dev)
    assert layer.status() == MOE_E_DEVICE
    from persistent_megakernel_sm_gb300 import lib
    assert b"site 50" in lib.moe_last_error()
    layer.set_option("fault_repush", -1)
    _clean_pass_is_correct(layer, w, dev, ref)
    layer.close()
