"""CUDA path against the CPU oracle on small layers that span several tiles,
ragged tails and the layer's degenerate cases, through the C ABI -- with the
GEMM tiles on one CTA (pair=1) and on CTA pairs (pair=2) alike."""
import numpy as np
import pytest

import _harness as hz
import oracle

pytestmark = pytest.mark.gpu

# (T, d, E, k, f, S, bias std)
CASES = {
    "tiny": (64, 256, 8, 2, 512, 0, 0.0),
    "ragged_bias": (37, 256, 8, 2, 512, 0, 0.5),
    "one_token": (1, 256, 4, 1, 256, 0, 0.0),
    "shared_partial_dtile": (100, 384, 16, 4, 384, 1, 0.3),
    "k_equals_E": (48, 256, 6, 6, 256, 0, 0.0),
    "multi_mtile_skew": (300, 256, 4, 2, 256, 0, 2.0),
    "wide_E": (96, 256, 64, 8, 256, 0, 1.0),
    "top16": (40, 128, 32, 16, 128, 1, 0.0),
    # odd k above 1: the router stores each token's slots one word at a time
    "odd_k3": (70, 256, 12, 3, 256, 0, 0.4),
    "odd_k5_shared": (50, 256, 16, 5, 256, 1, 0.2),
}


def _full_check(w, inp, mode="persistent", **opts):
    dev = hz.upload(inp)
    layer = hz.make_layer(w, mode={"persistent": 0, "multikernel": 1, "static": 2}[mode], **opts)
    got, routing = hz.run_layer(layer, w, dev)
    hz.check_routing(w, inp, routing)
    ref, _ = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k, S=w.S)
    hz.check_out(got, ref)
    layer.close()
    return got


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", list(CASES))
def test_small_layer_parity(name, pair):
    T, d, E, k, f, S, b = CASES[name]
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    _full_check(w, inp, pair=pair)


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", ["tiny", "shared_partial_dtile", "multi_mtile_skew"])
def test_multikernel_ablation_bit_identical(name, pair):
    T, d, E, k, f, S, b = CASES[name]
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    a = _full_check(w, inp, "persistent", pair=pair)
    m = _full_check(w, inp, "multikernel", pair=pair)
    assert np.array_equal(a, m), "ablation and megakernel outputs differ"


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", ["tiny", "shared_partial_dtile", "multi_mtile_skew", "top16"])
def test_static_megakernel_bit_identical(name, pair):
    # one cooperative launch, round-robin tasks, grid barriers between stages
    T, d, E, k, f, S, b = CASES[name]
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    a = _full_check(w, inp, "persistent", pair=pair)
    s = _full_check(w, inp, "static", pair=pair)
    assert np.array_equal(a, s), "static megakernel and persistent megakernel outputs differ"
    s7 = _full_check(w, inp, "static", grid_ctas=7, pair=pair)
    assert np.array_equal(a, s7), "static megakernel depends on its grid size"


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("split_k", [1, 2, 4])
@pytest.mark.parametrize("tokens_per_tile", [32, 64, 256])
def test_tiling_options_same_result(split_k, tokens_per_tile, pair):
    w, inp = hz.custom_case(200, 256, 8, 2, 512, 0, 0.4)
    _full_check(w, inp, split_k=split_k, tokens_per_tile=tokens_per_tile, pair=pair)


def test_pair_width_is_automatic_and_reported():
    # pairs when the mean rows per expert reach 128, one CTA below
    for T, E, k, want in ((64, 8, 2, 1), (512, 8, 2, 2)):
        w, inp = hz.custom_case(T, 256, E, k, 256, 0, 0.0)
        dev = hz.upload(inp)
        layer = hz.make_layer(w)
        hz.run_layer(layer, w, dev)
        assert layer.stat("pair") == want
        assert layer.stat("grid") % want == 0
        layer.close()


def test_all_tokens_one_expert():
    w, inp = hz.custom_case(130, 256, 8, 1, 256, 0, 0.0)
    inp["bias"] = np.array([12.0] + [0.0] * 7, dtype=np.float32)
    _full_check(w, inp)


def test_identical_experts_give_one_ffn():
    w, inp = hz.custom_case(50, 256, 8, 2, 256, 0, 0.0, identical_experts=True)
    got = _full_check(w, inp)
    for t in (0, 17, 49):
        _, y = oracle.expert_ffn(inp["x"][t], inp["w_gate"][0], inp["w_up"][0], inp["w_down"][0])
        hz.check_out(got[t], oracle.f64_to_bf16(y), "identical experts")


@pytest.mark.parametrize("pair", [1, 2])
def test_grid_and_mover_overrides(pair):
    w, inp = hz.custom_case(160, 256, 16, 4, 256, 1, 0.5)
    _full_check(w, inp, grid_ctas=7, mover_ctas=3, pair=pair)
    _full_check(w, inp, grid_ctas=1, pair=pair)


def test_smaller_T_than_reserved_and_repeat():
    import torch
    w, inp = hz.custom_case(120, 256, 8, 2, 256, 0, 0.3)
    dev = hz.upload(inp)
    layer = hz.make_layer(w, T_max=512)
    ref, _ = oracle.layer(inp["x"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=w.k)
    for T in (120, 57, 120):
        got, routing = hz.run_layer(layer, w, dev, T=T)
        hz.check_out(got, ref[:T])
    # T = 0 is a no-op
    out = torch.zeros((1, w.d), dtype=torch.bfloat16, device="cuda")
    layer.forward(dev["x"][:0], dev["router_w"], dev["w_gate"], dev["w_up"], dev["w_down"], out)
    layer.check()
    layer.close()


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("name", ["tiny", "shared_partial_dtile", "multi_mtile_skew", "wide_E"])
def test_folded_gather_bit_identical(name, pair):
    # gate/up tiles gathering their token rows from x themselves, against the
    # gather tasks copying them into the permuted buffer: the same bits
    T, d, E, k, f, S, b = CASES[name]
    w, inp = hz.custom_case(T, d, E, k, f, S, b)
    folded = _full_check(w, inp, pair=pair, fold_gather=1)
    copied = _full_check(w, inp, pair=pair, fold_gather=0)
    assert np.array_equal(folded, copied), "folded and copied gathers differ"
    for mode in ("multikernel", "static"):
        other = _full_check(w, inp, mode, pair=pair, fold_gather=1)
        assert np.array_equal(folded, other), mode
