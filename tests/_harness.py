"""Shared helpers for the tests: seeded inputs (with the routing margin
enforced through the oracle), device upload, running the CUDA path through the
C ABI, and element-wise comparison against the oracle."""
from __future__ import annotations

import numpy as np

import gen
import oracle

MARGIN = 1e-3
RTOL = 1e-2
ATOL = 1e-2


def margin_safe_x(w: gen.Workload, wr, bias, seed=0):
    """x with every token's k-th / (k+1)-th logit gap above MARGIN (oracle)."""
    retry = np.zeros(w.T, dtype=np.int32)
    x = gen.x_rows(w.T, w.d, retry, seed)
    if w.k >= w.E:
        return x, retry
    gap = oracle.route(x, wr, bias, w.k)["gap"]
    for _ in range(64):
        bad = np.nonzero(gap <= MARGIN)[0]
        if bad.size == 0:
            return x, retry
        retry[bad] += 1
        x = gen.x_rows(w.T, w.d, retry, seed)
        gap[bad] = oracle.route(x[bad], wr, bias, w.k)["gap"]
    raise RuntimeError("routing margin not reached")


def custom_case(T, d, E, k, f, S=0, bias_std=0.0, seed=0, identical_experts=False):
    w = gen.Workload(f"T{T}d{d}E{E}k{k}f{f}S{S}", T, d, E, k, f, S,
                     ("normal", bias_std) if bias_std else ())
    wr = gen.router_w(w, seed)
    bias = gen.router_bias(w, seed) if bias_std else None
    x, retry = margin_safe_x(w, wr, bias, seed)
    wg, wu, wd = gen.expert_weights(w, seed)
    if identical_experts:
        wg[:] = wg[0]
        wu[:] = wu[0]
        wd[:] = wd[0]
    return w, {"x": x, "router_w": wr, "bias": bias, "w_gate": wg, "w_up": wu, "w_down": wd}


def named_case(name, with_experts=True):
    w = gen.WORKLOADS[name]
    return w, gen.make_inputs(w, with_experts=with_experts)


# ---- device side --------------------------------------------------------------

def to_dev_bf16(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def from_dev_bf16(t) -> np.ndarray:
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def upload(inp: dict) -> dict:
    import torch
    dev = {key: to_dev_bf16(inp[key]) for key in ("x", "router_w", "w_gate", "w_up", "w_down")}
    dev["bias"] = None if inp.get("bias") is None else torch.from_numpy(inp["bias"]).cuda()
    return dev


def make_layer(w: gen.Workload, T_max=None, **options):
    from persistent_megakernel_sm_gb300 import MoELayer
    layer = MoELayer(w.d, w.f, w.E, w.k, w.S)
    layer.reserve(T_max or w.T)
    for key, val in options.items():
        layer.set_option(key, val)
    return layer


def run_layer(layer, w: gen.Workload, dev: dict, T=None):
    """Forward through the C ABI; returns (out bits [T,d], routing dict)."""
    import torch
    T = w.T if T is None else T
    out = torch.empty((T, w.d), dtype=torch.bfloat16, device="cuda")
    layer.set_router_bias(dev["bias"])
    layer.forward(dev["x"][:T], dev["router_w"], dev["w_gate"], dev["w_up"], dev["w_down"], out)
    layer.check()
    r = {
        "idx": torch.empty((T, w.k), dtype=torch.int32, device="cuda"),
        "w": torch.empty((T, w.k), dtype=torch.float32, device="cuda"),
        "counts": torch.empty(w.E, dtype=torch.int32, device="cuda"),
        "offsets": torch.empty(w.E + 1, dtype=torch.int32, device="cuda"),
        "perm": torch.empty(T * w.k, dtype=torch.int32, device="cuda"),
        "pos": torch.empty((T, w.k), dtype=torch.int32, device="cuda"),
    }
    layer.get_routing(**r)
    torch.cuda.synchronize()
    return from_dev_bf16(out), {key: v.cpu().numpy() for key, v in r.items()}


# ---- comparisons ----------------------------------------------------------------

def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_routing(w: gen.Workload, inp: dict, got: dict, T=None):
    """Bit-exact expert sets, counts, offsets and permutation; weights to 1e-5."""
    T = w.T if T is None else T
    ref = oracle.route(inp["x"][:T], inp["router_w"], inp["bias"], w.k)
    counts, offsets, perm, pos = oracle.permute(ref["idx"], w.E)
    gi, ri = got["idx"], ref["idx"]
    assert np.array_equal(np.sort(gi, axis=1), np.sort(ri, axis=1)), "expert sets differ"
    assert np.array_equal(got["counts"], counts), "counts differ"
    assert np.array_equal(got["offsets"], offsets), "offsets differ"
    assert np.array_equal(got["perm"], perm), "permutation differs"
    # pos and w are per slot; the slot order inside a token may legitimately
    # differ, so match them by expert
    for t in range(T):
        gmap = {int(e): (int(p), float(v)) for e, p, v in zip(gi[t], got["pos"][t], got["w"][t])}
        for j in range(w.k):
            e = int(ri[t, j])
            gp, gv = gmap[e]
            assert gp == pos[t, j], f"pos differs at token {t} expert {e}"
            assert abs(gv - ref["w"][t, j]) <= 1e-5 + 1e-5 * abs(ref["w"][t, j]), \
                f"weight differs at token {t} expert {e}: {gv} vs {ref['w'][t, j]}"
    return ref


def check_out(got_bits: np.ndarray, ref_bits: np.ndarray, what="out"):
    g = bf16_to_f64(got_bits)
    r = bf16_to_f64(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements off, first at {tuple(i)}: "
                             f"got {g[tuple(i)]} ref {r[tuple(i)]}; max err {err.max():.3g}")
    return float(err.max())


# ---- the oracle on many tokens (ctypes releases the GIL, so threads run the
# single-threaded C oracle side by side) ----------------------------------------

def _threads():
    import os
    return max(1, min(32, os.cpu_count() or 1))


def oracle_route_parallel(x, wr, bias, k):
    from concurrent.futures import ThreadPoolExecutor
    T = x.shape[0]
    n = _threads()
    bounds = np.linspace(0, T, n + 1).astype(int)
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda ab: oracle.route(x[ab[0]:ab[1]], wr, bias, k)
                            if ab[1] > ab[0] else None, zip(bounds[:-1], bounds[1:])))
    parts = [q for q in parts if q is not None]
    return {key: np.concatenate([q[key] for q in parts]) for key in ("idx", "w", "gap")}


def oracle_rows_parallel(w, inp, tokens):
    from concurrent.futures import ThreadPoolExecutor
    tokens = np.asarray(tokens, dtype=np.int32)
    with ThreadPoolExecutor(_threads()) as ex:
        rows = list(ex.map(lambda t: oracle.layer(inp["x"], inp["router_w"], inp["bias"],
                                                  inp["w_gate"], inp["w_up"], inp["w_down"],
                                                  k=w.k, S=w.S, tokens=np.array([t]))[0][0],
                           tokens))
    return np.stack(rows)


def check_routing_full(w, inp, got, ref=None):
    """check_routing for large T, with the oracle's routing computed in parallel."""
    ref = ref or oracle_route_parallel(inp["x"], inp["router_w"], inp["bias"], w.k)
    counts, offsets, perm, pos = oracle.permute(ref["idx"], w.E)
    assert np.array_equal(np.sort(got["idx"], axis=1), np.sort(ref["idx"], axis=1)), \
        "expert sets differ"
    assert np.array_equal(got["counts"], counts), "counts differ"
    assert np.array_equal(got["offsets"], offsets), "offsets differ"
    assert np.array_equal(got["perm"], perm), "permutation differs"
    # match pos / w by expert: sort each token's slots by expert on both sides
    og = np.argsort(got["idx"], axis=1, kind="stable")
    orf = np.argsort(ref["idx"], axis=1, kind="stable")
    gp = np.take_along_axis(got["pos"], og, 1)
    rp = np.take_along_axis(pos, orf, 1)
    assert np.array_equal(gp, rp), "pos differs"
    gw = np.take_along_axis(got["w"].astype(np.float64), og, 1)
    rw = np.take_along_axis(ref["w"], orf, 1)
    assert np.all(np.abs(gw - rw) <= 1e-5 + 1e-5 * np.abs(rw)), "weights differ"
    assert np.all(ref["gap"] > MARGIN), "input violates the routing margin"
    return ref


# ---- which tokens a sampled full-size comparison checks ---------------------------

def expert_groups(rows: np.ndarray, bn: int):
    """The plan's row groups of one expert: its tokens (ascending) split into
    ceil(n / bn) balanced groups of a multiple of 16 rows."""
    n = len(rows)
    if n == 0:
        return []
    nmt = -(-n // bn)
    per = ((-(-n // nmt)) + 15) // 16 * 16
    return [rows[m * per:(m + 1) * per] for m in range(nmt) if m * per < n]


def coverage_tokens(T, E, k, S, idx, bn, ct, n, seed=0):
    """At least `n` distinct tokens such that every GEMM row group of the
    shared expert (bn consecutive tokens each) and of the three experts with
    the most tokens, and every combine tile (ct consecutive tokens, both d
    bands: a compared token's whole row is compared), holds one of them; the
    rest are drawn at random.  Sorted."""
    rng = np.random.default_rng(seed)
    pick = set()

    def one_of(cands):
        cands = np.asarray(cands)
        if cands.size and not pick.intersection(cands.tolist()):
            pick.add(int(rng.choice(cands)))

    for c0 in range(0, T, ct):
        one_of(np.arange(c0, min(T, c0 + ct)))
    if S:
        for g0 in range(0, T, bn):
            one_of(np.arange(g0, min(T, g0 + bn)))
    counts = np.bincount(np.asarray(idx).ravel(), minlength=E)
    for e in np.argsort(-counts, kind="stable")[:3]:
        rows = np.nonzero((np.asarray(idx) == e).any(axis=1))[0]
        for grp in expert_groups(rows, bn):
            one_of(grp)
    rest = np.setdiff1d(np.arange(T), np.fromiter(pick, dtype=np.int64))
    extra = max(0, min(n, T) - len(pick))
    if extra:
        pick.update(int(t) for t in rng.choice(rest, size=extra, replace=False))
    return np.array(sorted(pick), dtype=np.int64)
