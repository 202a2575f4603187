"""moe_layer_forward_noalloc: the forward pass for callers that cannot
allocate device memory -- processes whose device memory belongs to another
allocator, runtimes that forbid allocation after start-up.  It runs on a
fixed scratch array inside the library instead of the workspace of
moe_layer_reserve.

Checked through the C ABI, two calls in a row per layer, against the regular
entry point (within the oracle's tolerance: the scratch may force another
down-projection tiling) and against the oracle itself, with the routing read
back through moe_layer_get_routing; then layers of different shapes one after
another on the one shared array; a device timeout read back through
moe_layer_status; and a layer too large for the scratch refused.  Named to be
collected last."""
import numpy as np
import pytest

import _harness as hz
import oracle
import persistent_megakernel_sm_gb300 as pkg

pytestmark = pytest.mark.gpu


def _noalloc_forward(layer, w, dev, out):
    lib = pkg.lib
    return lib.moe_layer_forward_noalloc(layer.h, w.T, dev["x"].data_ptr(),
                                         dev["router_w"].data_ptr(), dev["w_gate"].data_ptr(),
                                         dev["w_up"].data_ptr(), dev["w_down"].data_ptr(),
                                         out.data_ptr(), None)


def _routing(layer, w):
    import torch
    r = {
        "idx": torch.empty((w.T, w.k), dtype=torch.int32, device="cuda"),
        "w": torch.empty((w.T, w.k), dtype=torch.float32, device="cuda"),
        "counts": torch.empty(w.E, dtype=torch.int32, device="cuda"),
        "offsets": torch.empty(w.E + 1, dtype=torch.int32, device="cuda"),
        "perm": torch.empty(w.T * w.k, dtype=torch.int32, device="cuda"),
        "pos": torch.empty((w.T, w.k), dtype=torch.int32, device="cuda"),
    }
    layer.get_routing(**r)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in r.items()}


def _case(name):
    if name == "decode":
        return hz.named_case("decode")
    if name == "tiny_shared":
        return hz.custom_case(100, 384, 16, 4, 384, 1, 0.3)
    return hz.custom_case(48, 256, 8, 2, 256)


def _check_call(layer, w, inp, dev, ref_rows, ref_tokens, reserved, what, check_mem=False):
    """One no-allocation call: status, routing and outputs; with check_mem,
    that the call itself took no device memory."""
    import torch
    out = torch.zeros((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    rc = _noalloc_forward(layer, w, dev, out)
    assert rc == pkg.MOE_OK, pkg.lib.moe_last_error()
    torch.cuda.synchronize()
    if check_mem:
        assert torch.cuda.mem_get_info()[0] == free_before, "the call allocated device memory"
    assert layer.status() == pkg.MOE_OK, pkg.lib.moe_last_error()
    hz.check_routing_full(w, inp, _routing(layer, w))
    got = hz.from_dev_bf16(out)
    hz.check_out(got[ref_tokens], ref_rows, f"{what}: against the oracle")
    hz.check_out(got, reserved, f"{what}: against moe_layer_forward")
    return got


@pytest.mark.parametrize("name", ["tiny_shared", "decode"])
def test_noalloc_matches_oracle_and_reserved_workspace(name):
    w, inp = _case(name)
    dev = hz.upload(inp)
    # the regular entry point (workspace from moe_layer_reserve)
    ref_layer = hz.make_layer(w)
    reserved, _ = hz.run_layer(ref_layer, w, dev)
    ref_layer.close()
    tokens = np.arange(w.T)
    ref_rows = hz.oracle_rows_parallel(w, inp, tokens)
    # the no-allocation entry point: a handle without moe_layer_reserve
    layer = pkg.MoELayer(w.d, w.f, w.E, w.k, w.S)
    layer.set_router_bias(dev["bias"])
    for call in range(2):
        # the first call may load the module; later calls allocate nothing
        _check_call(layer, w, inp, dev, ref_rows, tokens, reserved, f"{name} call {call}",
                    check_mem=call == 1)
    layer.close()


def test_noalloc_layers_of_different_shapes_in_turn():
    # the scratch's layout follows T and the layer's sizes: small, decode,
    # small again on the one array, each result checked
    cases = {}
    for name in ("small", "decode"):
        w, inp = _case(name)
        dev = hz.upload(inp)
        ref_layer = hz.make_layer(w)
        reserved, _ = hz.run_layer(ref_layer, w, dev)
        ref_layer.close()
        tokens = np.arange(w.T) if w.T <= 64 else np.arange(0, w.T, 8)
        layer = pkg.MoELayer(w.d, w.f, w.E, w.k, w.S)
        layer.set_router_bias(dev["bias"])
        cases[name] = (w, inp, dev, layer, reserved, tokens,
                       hz.oracle_rows_parallel(w, inp, tokens))
    for name in ("small", "decode", "small"):
        w, inp, dev, layer, reserved, tokens, ref_rows = cases[name]
        _check_call(layer, w, inp, dev, ref_rows, tokens, reserved, f"{name} in turn")
    for c in cases.values():
        c[3].close()


def test_noalloc_device_status_is_readable():
    import torch
    # a dropped dependency notification with a short device wait budget: the
    # call's timeout is read back through moe_layer_status, then a clean call
    # on the same handle reports MOE_OK and is correct
    w, inp = _case("small")
    dev = hz.upload(inp)
    ref = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                       inp["w_down"], k=w.k, S=w.S)[0]
    layer = pkg.MoELayer(w.d, w.f, w.E, w.k, w.S)
    layer.set_option("timeout_ns", 50_000_000)
    layer.set_option("fault_drop_task", 0)
    out = torch.zeros((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_forward(layer, w, dev, out) == pkg.MOE_OK
    assert layer.status() == pkg.MOE_E_TIMEOUT
    layer.set_option("fault_drop_task", -1)
    assert _noalloc_forward(layer, w, dev, out) == pkg.MOE_OK
    assert layer.status() == pkg.MOE_OK
    hz.check_out(hz.from_dev_bf16(out), ref, "after the timeout")
    layer.close()


def test_noalloc_refuses_too_large_layers():
    import torch
    layer = pkg.MoELayer(7168, 2048, 256, 8, 1)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    rc = pkg.lib.moe_layer_forward_noalloc(layer.h, 8192, p, p, p, p, p, p, None)
    assert rc == pkg.MOE_E_INVAL
    assert b"scratch" in pkg.lib.moe_last_error()
    layer.close()
