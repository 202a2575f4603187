"""moe_layer_calibrate: times candidate tile sizes, K splits and d bands on
the caller's inputs, keeps the fastest as options; the calibrated layer
still routes bit-exactly and matches the oracle within tolerance."""
import numpy as np
import pytest

import _harness as hz
import gen
import oracle

pytestmark = pytest.mark.gpu


def _calibrate(layer, w, dev, reps=2):
    import torch
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    layer.set_router_bias(dev["bias"])
    return layer.calibrate(dev["x"], dev["router_w"], dev["w_gate"], dev["w_up"], dev["w_down"],
                           out, reps=reps)


def test_calibrated_small_layer_parity():
    w, inp = hz.custom_case(300, 256, 16, 4, 384, 0, 0.6)
    dev = hz.upload(inp)
    layer = hz.make_layer(w)
    best = _calibrate(layer, w, dev)
    assert 0 < best < 1e6
    got, routing = hz.run_layer(layer, w, dev)
    assert layer.stat("tile_tokens") in (32, 64, 96, 128, 160, 192, 224, 256)
    assert layer.stat("split_k") in (1, 2, 4)
    assert layer.stat("bands") in (1, 2)
    hz.check_routing(w, inp, routing)
    ref, _ = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k, S=w.S)
    hz.check_out(got, ref)
    layer.close()


def test_calibrated_fine_workload_sampled():
    w = gen.WORKLOADS["fine"]
    inp = gen.make_inputs(w)
    dev = hz.upload(inp)
    layer = hz.make_layer(w)
    best = _calibrate(layer, w, dev, reps=3)
    assert 0 < best < 1e6
    got, routing = hz.run_layer(layer, w, dev)
    tokens = np.array([0, 3, 128, 300, 511], dtype=np.int32)
    ref = hz.oracle_rows_parallel(w, inp, tokens)
    hz.check_out(got[tokens], ref, "calibrated fine out")
    layer.close()
