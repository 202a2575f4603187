"""The residual add and RMSNorm fused into the combine
(moe_layer_forward_residual_norm) against the CPU oracle, and the same bits
in every execution mode.

out = bf16(residual + layer), norm_out = bf16(out * rsqrt(mean(out^2) + eps)
* gamma): the two steps that end the MoE megakernel in xxqk.cn/news/665650
section 1, read as the pre-norm block."""
import numpy as np
import pytest

import _harness as hz
import gen
import oracle

pytestmark = pytest.mark.gpu

EPS = 1e-5

CASES = {
    # T, d, E, k, f, S, router-bias std, options
    "small": (64, 256, 8, 2, 512, 0, 0.0, {}),
    "shared_expert": (100, 384, 16, 4, 256, 1, 0.5, {}),
    "fp32_partials": (96, 256, 8, 2, 512, 0, 0.3, {"split_k": 4}),
    "top16": (40, 128, 32, 16, 128, 1, 0.0, {}),
    "ragged_tiles": (300, 256, 16, 3, 384, 0, 0.6, {"tokens_per_tile": 64}),
}


def _extra(T, d, seed=5):
    rng = np.random.default_rng(seed)
    residual = oracle.f64_to_bf16(rng.standard_normal((T, d)) * 0.8)
    gamma = oracle.f64_to_bf16(1.0 + 0.25 * rng.standard_normal(d))
    return residual, gamma


def _run(w, inp, residual, gamma, mode=0, **opts):
    import torch
    dev = hz.upload(inp)
    layer = hz.make_layer(w, mode=mode, **opts)
    layer.set_router_bias(dev["bias"])
    out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    norm = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    layer.forward_residual_norm(dev["x"], dev["router_w"], dev["w_gate"], dev["w_up"],
                                dev["w_down"], hz.to_dev_bf16(residual), hz.to_dev_bf16(gamma),
                                EPS, out, norm)
    layer.check()
    torch.cuda.synchronize()
    got = hz.from_dev_bf16(out), hz.from_dev_bf16(norm)
    layer.close()
    return got


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", list(CASES))
def test_residual_norm_parity(name, pair):
    # GEMM tiles on one CTA and on CTA pairs (whose CTAs split each combine
    # tile's tokens: the norm waits for both halves)
    T, d, E, k, f, S, b, opts = CASES[name]
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    residual, gamma = _extra(T, d)
    out, norm = _run(w, inp, residual, gamma, pair=pair, **opts)
    _, acc = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k, S=w.S)
    ref_out, ref_norm, _ = oracle.residual_rmsnorm(acc, residual, gamma, EPS)
    hz.check_out(out, ref_out, "out = residual + layer")
    hz.check_out(norm, ref_norm, "RMSNorm(out) * gamma")


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", ["small", "shared_expert", "fp32_partials"])
def test_residual_norm_same_bits_in_every_mode(name, pair):
    T, d, E, k, f, S, b, opts = CASES[name]
    opts = dict(opts, pair=pair)
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    residual, gamma = _extra(T, d)
    base = _run(w, inp, residual, gamma, mode=0, **opts)
    for mode in (1, 2):
        got = _run(w, inp, residual, gamma, mode=mode, **opts)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1]), mode
    # the residual stream equals the plain forward's output plus the residual
    # only up to one rounding, but a zero residual gives the plain output bits
    zero = np.zeros_like(residual)
    out0, _ = _run(w, inp, zero, gamma, **opts)
    dev = hz.upload(inp)
    layer = hz.make_layer(w, **opts)
    plain, _ = hz.run_layer(layer, w, dev)
    layer.close()
    assert np.array_equal(out0, plain)


def test_residual_norm_fine_workload_sampled():
    w = gen.WORKLOADS["fine"]
    inp = gen.make_inputs(w)
    residual, gamma = _extra(w.T, w.d, seed=9)
    out, norm = _run(w, inp, residual, gamma)
    tokens = np.array([0, 1, 77, 255, 256, 400, 510, 511], dtype=np.int32)
    _, acc = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k, S=w.S, tokens=tokens)
    ref_out, ref_norm, _ = oracle.residual_rmsnorm(acc, residual[tokens], gamma, EPS)
    hz.check_out(out[tokens], ref_out, "fine out")
    hz.check_out(norm[tokens], ref_norm, "fine norm")
