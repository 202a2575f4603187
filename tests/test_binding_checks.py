"""The Python binding's argument checks, on CPU: the tensors every caller in
this repository builds (the test harness, the residual + RMSNorm and
calibration tests, bench.py) pass them, and tensors the kernels would read out
of bounds (wrong dtype, shape or layout, or on the host) are refused before
any C call.  The library is replaced by a recorder, so no GPU is needed."""
import numpy as np
import pytest
import torch

import _harness as hz
from persistent_megakernel_sm_gb300 import binding


class _OnDevice(torch.Tensor):
    """A host tensor that reports itself as a CUDA tensor (test stand-in)."""

    @property
    def is_cuda(self):
        return True


def _dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.as_subclass(_OnDevice)


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append(name)
            return 1 if name == "moe_layer_create" else 0
        return call


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(binding, "lib", r)
    layers = []
    r.layer = lambda w: layers.append(binding.MoELayer(w.d, w.f, w.E, w.k, w.S)) or layers[-1]
    yield r
    for layer in layers:  # the handles are the recorder's: close them while it is in place
        layer.close()


@pytest.fixture(scope="module")
def case():
    w, inp = hz.custom_case(40, 256, 8, 2, 384, 1, 0.3)  # d != f: a transpose shows
    dev = {key: _dev(inp[key]) for key in ("x", "router_w", "w_gate", "w_up", "w_down")}
    dev["bias"] = torch.from_numpy(inp["bias"]).as_subclass(_OnDevice)
    return w, dev


def _out(rows, d):
    return torch.empty((rows, d), dtype=torch.bfloat16).as_subclass(_OnDevice)


def test_every_caller_shape_passes(rec, case):
    w, dev = case
    layer = rec.layer(w)
    wts = (dev["router_w"], dev["w_gate"], dev["w_up"], dev["w_down"])
    layer.set_router_bias(dev["bias"])
    layer.forward(dev["x"][:w.T], *wts, _out(w.T, w.d), stream=0)
    layer.forward(dev["x"][:17], *wts, _out(17, w.d), stream=0)
    layer.forward(dev["x"][:0], *wts, _out(1, w.d), stream=0)  # T = 0 with a spare row
    gamma = _dev(np.zeros(w.d, dtype=np.uint16))
    layer.forward_residual_norm(dev["x"], *wts, _out(w.T, w.d), gamma, 1e-5, _out(w.T, w.d),
                                _out(w.T, w.d), stream=0)
    layer.calibrate(dev["x"], *wts, _out(w.T, w.d), reps=2, stream=0)
    layer.forward_noalloc(dev["x"], *wts, _out(w.T, w.d), stream=0)
    layer.forward_host(w.T, 4096, *wts, 8192, stream=0)
    assert rec.calls.count("moe_layer_forward") == 3
    for name in ("moe_layer_set_router_bias", "moe_layer_forward_residual_norm",
                 "moe_layer_calibrate", "moe_layer_forward_noalloc", "moe_layer_forward_host"):
        assert name in rec.calls, name


@pytest.mark.parametrize("what", ["dtype", "shape", "transposed", "layout", "host", "out_rows",
                                  "bias", "gamma"])
def test_bad_tensors_are_refused_before_the_call(rec, case, what):
    w, dev = case
    layer = rec.layer(w)
    x, wr, wg, wu, wd = (dev[key] for key in ("x", "router_w", "w_gate", "w_up", "w_down"))
    out = _out(w.T, w.d)
    if what == "dtype":
        x = x.float().as_subclass(_OnDevice)
    elif what == "shape":
        wg = wg[:, : w.f // 2]
    elif what == "transposed":
        wd = wd.transpose(1, 2).contiguous().as_subclass(_OnDevice)
    elif what == "layout":
        out = torch.empty((w.d, w.T), dtype=torch.bfloat16).t().as_subclass(_OnDevice)
    elif what == "host":
        wu = torch.empty(tuple(wu.shape), dtype=torch.bfloat16)
    elif what == "out_rows":
        out = _out(w.T - 1, w.d)
    before = list(rec.calls)
    with pytest.raises(binding.MoEError) as err:
        if what == "bias":
            layer.set_router_bias(torch.zeros(w.E, dtype=torch.float64).as_subclass(_OnDevice))
        elif what == "gamma":
            gamma = _dev(np.zeros(w.d + 8, dtype=np.uint16))
            layer.forward_residual_norm(x, wr, wg, wu, wd, out, gamma, 1e-5, _out(w.T, w.d),
                                        _out(w.T, w.d), stream=0)
        else:
            layer.forward(x, wr, wg, wu, wd, out, stream=0)
    assert err.value.code == binding.MOE_E_INVAL
    assert rec.calls == before, "the C library was called with a bad tensor"
