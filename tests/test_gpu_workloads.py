"""The five workloads at full size, in the launch configuration bench.py
times: routing compared with the oracle for every token (bit-exact expert
sets, counts, offsets, permutation, pos), outputs compared element by element
with the oracle -- every token of tiny, decode and fine; on skew and prefill at
least 512 tokens chosen so that every GEMM row group of the shared expert and
of the three largest experts, and every combine tile (whose rows span both d
bands), holds at least one compared token -- and the one-kernel-per-stage
ablation and the static persistent kernel reproducing the megakernel's bits.

Also the largest layer the boundary accepts: T = 32768 tokens, E = 256
experts, k = 16 (tiny d and f), where the plan's per-(router tile, expert)
count table no longer fits in shared memory and takes its global-memory path.
"""
import numpy as np
import pytest

import _harness as hz

pytestmark = pytest.mark.gpu

# tokens whose output rows are compared: None = all of them
SAMPLES = {"tiny": None, "decode": None, "fine": None, "skew": 512, "prefill": 512}


@pytest.fixture(scope="module", params=list(SAMPLES))
def workload(request):
    import torch
    name = request.param
    w, inp = hz.named_case(name)
    dev = hz.upload(inp)
    yield name, w, inp, dev
    del dev
    torch.cuda.empty_cache()


def test_workload_parity_and_ablation(workload):
    name, w, inp, dev = workload
    layer = hz.make_layer(w)
    got, routing = hz.run_layer(layer, w, dev)
    ref_route = hz.check_routing_full(w, inp, routing)
    if SAMPLES[name] is None:
        tokens = np.arange(w.T)
    else:
        tokens = hz.coverage_tokens(w.T, w.E, w.k, w.S, ref_route["idx"],
                                    bn=layer.stat("tile_tokens"),
                                    ct=layer.stat("combine_tokens"), n=SAMPLES[name], seed=123)
    ref = hz.oracle_rows_parallel(w, inp, tokens)
    hz.check_out(got[tokens], ref, f"{name} out ({len(tokens)} tokens)")
    # repeat: identical bits (deterministic summation order, no atomics in values)
    again, _ = hz.run_layer(layer, w, dev)
    assert np.array_equal(got, again), "megakernel is not deterministic"
    layer.set_option("mode", 1)
    abl, _ = hz.run_layer(layer, w, dev)
    assert np.array_equal(got, abl), "ablation differs from the megakernel"
    layer.set_option("mode", 2)
    sta, _ = hz.run_layer(layer, w, dev)
    assert np.array_equal(got, sta), "static megakernel differs from the persistent one"
    layer.close()


def test_largest_layer_global_plan_path():
    import torch
    # 256 router tiles x 256 experts: a 256 KB count table, above the
    # pipeline's shared memory, so the plan scans it in global memory
    w, inp = hz.custom_case(32768, 128, 256, 16, 128, bias_std=0.3)
    dev = hz.upload(inp)
    layer = hz.make_layer(w)
    got, routing = hz.run_layer(layer, w, dev)
    ref_route = hz.check_routing_full(w, inp, routing)
    tokens = hz.coverage_tokens(w.T, w.E, w.k, w.S, ref_route["idx"],
                                bn=layer.stat("tile_tokens"), ct=layer.stat("combine_tokens"),
                                n=2048, seed=7)
    ref = hz.oracle_rows_parallel(w, inp, tokens)
    hz.check_out(got[tokens], ref, f"T=32768 out ({len(tokens)} tokens)")
    layer.set_option("mode", 1)
    abl, _ = hz.run_layer(layer, w, dev)
    assert np.array_equal(got, abl), "ablation differs from the megakernel"
    layer.close()
    del dev
    torch.cuda.empty_cache()
