"""moe_layer_forward_static: the forward pass for callers that cannot allocate
device memory (code running under CUDA-graph capture, processes whose device
memory belongs to another allocator, runtimes that forbid allocation after
start-up).  It uses a fixed scratch array inside the library instead of the
workspace of moe_layer_reserve.  Checked through the C ABI against the
regular entry point on two calls in a row, for a layer that fits and for one
that must be refused.  Named to be collected last."""
import ctypes

import numpy as np
import pytest

import _harness as hz
import persistent_megakernel_sm_gb300 as pkg

pytestmark = pytest.mark.gpu


def _static_forward(layer, w, dev, out):
    lib = pkg.lib
    rc = lib.moe_layer_forward_static(layer.h, w.T, dev["x"].data_ptr(), dev["router_w"].data_ptr(),
                                      dev["w_gate"].data_ptr(), dev["w_up"].data_ptr(),
                                      dev["w_down"].data_ptr(), out.data_ptr(), None)
    return rc


@pytest.mark.parametrize("case", ["tiny_shared", "decode"])
def test_static_scratch_matches_reserved_workspace(case):
    import torch
    if case == "decode":
        w, inp = hz.named_case("decode")
    else:
        w, inp = hz.custom_case(100, 384, 16, 4, 384, 1, 0.3)
    dev = hz.upload(inp)
    # the regular entry point (workspace from moe_layer_reserve)
    ref_layer = hz.make_layer(w)
    ref, _ = hz.run_layer(ref_layer, w, dev)
    # the no-allocation entry point: a handle without moe_layer_reserve
    layer = pkg.MoELayer(w.d, w.f, w.E, w.k, w.S)
    layer.set_router_bias(dev["bias"])
    for call in range(2):
        out = torch.zeros((w.T, w.d), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = _static_forward(layer, w, dev, out)
        assert rc == pkg.MOE_OK, pkg.lib.moe_last_error()
        torch.cuda.synchronize()
        if call == 1:  # the first call may load the module; later calls allocate nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        hz.check_out(hz.from_dev_bf16(out), ref, f"static call {call}")
    layer.close()
    ref_layer.close()


def test_static_scratch_refuses_too_large_layers():
    import torch
    layer = pkg.MoELayer(7168, 2048, 256, 8, 1)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    rc = pkg.lib.moe_layer_forward_static(layer.h, 8192, p, p, p, p, p, p, None)
    assert rc == pkg.MOE_E_INVAL
    assert b"scratch" in pkg.lib.moe_last_error()
    layer.close()
