"""The seeded input generator: determinism, independence of streams and rows,
the requested distributions, and the committed per-workload metadata."""
import numpy as np
import pytest

import gen


def test_same_seed_same_bits_and_offsets_agree():
    a = gen.normal_bf16(gen.TID_W_GATE, (1 << 18,), 0.5)
    b = gen.normal_bf16(gen.TID_W_GATE, (1 << 18,), 0.5)
    assert np.array_equal(a, b)
    for first, n in [(0, 1), (1, 1), (12345, 1001), (77, 65536 + 3)]:
        c = gen.normal_bf16(gen.TID_W_GATE, (n,), 0.5, first=first)
        assert np.array_equal(c, a[first:first + n])


def test_streams_and_seeds_differ():
    a = gen.normal_bf16(gen.TID_W_GATE, (4096,), 1.0)
    b = gen.normal_bf16(gen.TID_W_UP, (4096,), 1.0)
    c = gen.normal_bf16(gen.TID_W_GATE, (4096,), 1.0, seed=1)
    assert (a != b).mean() > 0.9 and (a != c).mean() > 0.9


@pytest.mark.parametrize("std", [1.0, 0.0156, 0.3])
def test_normal_moments(std):
    v = gen.bf16_bits_to_f32(gen.normal_bf16(gen.TID_X, (1 << 20,), std)).astype(np.float64) / std
    assert abs(v.mean()) < 0.005
    assert abs(v.std() - 1.0) < 0.005
    assert abs((v ** 4).mean() - 3.0) < 0.05          # normal kurtosis
    assert abs((np.abs(v) < 1).mean() - 0.6827) < 0.003


def test_x_row_redraw_is_local():
    base = gen.x_rows(10, 64)
    r = np.zeros(10, dtype=np.int32)
    r[[2, 7]] = [1, 3]
    redrawn = gen.x_rows(10, 64, r)
    same = [i for i in range(10) if i not in (2, 7)]
    assert np.array_equal(base[same], redrawn[same])
    assert (base[2] != redrawn[2]).mean() > 0.9 and (base[7] != redrawn[7]).mean() > 0.9
    assert np.array_equal(redrawn, gen.x_rows(10, 64, r))


def test_zipf_targets():
    w = gen.WORKLOADS["skew"]
    c = gen.zipf_target_counts(w)
    assert abs(c.sum() - w.T * w.k) < 1e-6
    assert c.max() <= w.T + 1e-9 and c.min() > 0
    srt = np.sort(c)[::-1]
    free = srt < w.T - 1e-9
    # uncapped ranks keep the Zipf ratio (r / (r+1))^-1.2 between neighbours
    r = np.arange(1, w.E + 1)
    ratios = srt[1:][free[1:] & free[:-1]] / srt[:-1][free[1:] & free[:-1]]
    expect = ((r[1:] / r[:-1]) ** -1.2)[free[1:] & free[:-1]]
    assert np.allclose(ratios, expect)


@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_workload_metadata_present(name):
    w = gen.WORKLOADS[name]
    meta = gen.load_meta(name)
    assert meta is not None, "run tests/golden/make_inputs_meta.py"
    assert sum(meta["oracle_counts"]) == w.T * w.k
    if w.bias and w.bias[0] == "zipf":
        assert len(meta["bias"]) == w.E
    if meta.get("min_margin") is not None:
        assert meta["min_margin"] > 1e-3


def test_tiny_inputs_shapes():
    w = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(w)
    assert inp["x"].shape == (w.T, w.d) and inp["x"].dtype == np.uint16
    assert inp["router_w"].shape == (w.E, w.d)
    assert inp["w_gate"].shape == (w.E + w.S, w.f, w.d)
    assert inp["w_down"].shape == (w.E + w.S, w.d, w.f)
    assert inp["bias"] is None
    wr = gen.bf16_bits_to_f32(inp["router_w"]).astype(np.float64)
    assert abs(wr.std() * np.sqrt(w.d) - 1.0) < 0.05
