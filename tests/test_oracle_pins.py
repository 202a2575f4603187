"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong rounding) fails at least
one of them: library routines (numpy matmul / sort / bincount), brute force on
tiny inputs, closed forms, and cases worked out by hand.
"""
import math

import numpy as np
import pytest

import oracle


# ---- an independent bf16 rounding (numpy frexp + rint, half to even) ---------

def np_round_bf16(v: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (as float64) of each double, ties to even (normals)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bits_of(vals: np.ndarray) -> np.ndarray:
    return (np.asarray(vals, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def as_bf16_bits(vals):
    """Exact bf16 bit patterns of values that are representable in bf16."""
    v = np.asarray(vals, dtype=np.float64)
    assert np.all(np_round_bf16(v) == v)
    return bits_of(v)


def rand_bf16(rng, shape, scale=1.0):
    return bits_of(np_round_bf16(rng.standard_normal(shape) * scale))


def f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def np_silu(z):
    return z / (1.0 + np.exp(-z))


def np_ffn(x, wg, wu, wd):
    """One expert on one token with numpy: Wd . bf16(silu(Wg x) * (Wu x))."""
    g = f64(wg) @ f64(x)
    u = f64(wu) @ f64(x)
    h = np_round_bf16(np_silu(g) * u)
    return h, f64(wd) @ h


# ---- bf16 -----------------------------------------------------------------------

def test_bf16_decode_matches_float32_reinterpretation():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_to_f64(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])


def test_bf16_round_trip_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    finite = np.isfinite(vals)
    back = oracle.f64_to_bf16(vals[finite])
    assert np.array_equal(back, bits[finite])


@pytest.mark.parametrize("value,expect", [
    (1.0 + 2.0 ** -8, 0x3F80),                 # half-way, even neighbour below
    (1.0 + 3 * 2.0 ** -8, 0x3F82),             # half-way, even neighbour above
    (-(1.0 + 2.0 ** -8), 0xBF80),
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above half-way
    (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),    # just below half-way
    (2.0 ** -133, 0x0001),                     # smallest subnormal
    (1.5 * 2.0 ** -133, 0x0002),               # subnormal tie -> even
    (0.5 * 2.0 ** -133, 0x0000),               # tie with zero -> even (zero)
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie above largest -> even = inf
    (-0.0, 0x8000),
    (3.0, 0x4040),
])
def test_bf16_rounding_cases(value, expect):
    assert int(oracle.f64_to_bf16(np.array([value]))[0]) == expect


def test_bf16_rounding_matches_frexp_rint():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))
    got = oracle.bf16_to_f64(oracle.f64_to_bf16(v))
    assert np.array_equal(got, np_round_bf16(v))


def test_silu_closed_form():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.e ** -1)) < 1e-15
    # silu(z) - silu(-z) = z
    for z in (0.3, 1.7, 5.0):
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14


# ---- router and top-k -----------------------------------------------------------

def test_router_logits_match_numpy_matmul():
    rng = np.random.default_rng(2)
    T, d, E = 7, 40, 5
    x = rand_bf16(rng, (T, d))
    wr = rand_bf16(rng, (E, d), 0.2)
    b = rng.standard_normal(E).astype(np.float32)
    L = oracle.router_logits(x, wr, b)
    ref = f64(x) @ f64(wr).T + b.astype(np.float64)
    assert np.allclose(L, ref, rtol=1e-13, atol=1e-13)
    L0 = oracle.router_logits(x, wr, None)
    assert np.allclose(L0, f64(x) @ f64(wr).T, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("E,k", [(8, 2), (16, 5), (6, 6), (1, 1), (32, 8)])
def test_topk_brute_force_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 50
    L = rng.standard_normal((T, E))
    L[3, :] = 0.25  # all tied: lower expert index first
    if E > 2:
        L[4, 1] = L[4, 2] = 3.0  # a tie at the top
    idx, w, p, gap = oracle.topk(L, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-L[t, e], e))
        assert list(idx[t]) == order[:k]
        kept = np.exp(L[t, order[:k]] - L[t].max())
        assert np.allclose(w[t], kept / kept.sum(), rtol=1e-13, atol=0)
        if k < E:
            assert gap[t] == pytest.approx(L[t, order[k - 1]] - L[t, order[k]], abs=1e-15)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    ex = np.exp(L - L.max(axis=1, keepdims=True))
    assert np.allclose(p, ex / ex.sum(axis=1, keepdims=True), rtol=1e-13)


def test_topk_with_k_equal_E_is_full_softmax():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((9, 7)) * 3
    idx, w, p, _ = oracle.topk(L, 7)
    full = np.zeros_like(L)
    for t in range(9):
        full[t, idx[t]] = w[t]
    ex = np.exp(L - L.max(axis=1, keepdims=True))
    assert np.allclose(full, ex / ex.sum(axis=1, keepdims=True), rtol=1e-13)


@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (256, 8), (32, 16)])
def test_renormalised_weights_need_no_softmax_denominator(E, k):
    # w_j = p_j / sum_kept p = exp(L_j - max) / sum_kept exp(L_s - max): the
    # softmax denominator over all E cancels (the kernel computes this form,
    # the oracle the softmax-then-renormalise one)
    rng = np.random.default_rng(E * 31 + k)
    L = rng.standard_normal((40, E)) * 2.5
    idx, w, _, _ = oracle.topk(L, k)
    for t in range(L.shape[0]):
        kept = L[t, idx[t]]
        e = np.exp(kept - kept.max())
        assert kept.max() == L[t].max()
        assert np.allclose(w[t], e / e.sum(), rtol=1e-12, atol=0)


def test_topk_hand_example_renormalisation():
    # logits 0, ln 2, ln 3: softmax is (1, 2, 3)/6; the top two are experts 2
    # and 1, renormalised to 3/5 and 2/5.
    x = as_bf16_bits([[1.0]])
    wr = as_bf16_bits([[0.0], [0.0], [0.0]])
    b = np.array([0.0, math.log(2.0), math.log(3.0)], dtype=np.float32)
    r = oracle.route(x, wr, b, 2)
    assert list(r["idx"][0]) == [2, 1]
    assert np.allclose(r["w"][0], [0.6, 0.4], atol=1e-6)
    assert np.allclose(r["p"][0], [1 / 6, 2 / 6, 3 / 6], atol=1e-6)


# ---- permutation ------------------------------------------------------------------

def test_permute_hand_example():
    idx = np.array([[2, 0], [0, 1], [2, 1]], dtype=np.int32)
    counts, offsets, perm, pos = oracle.permute(idx, 3)
    assert list(counts) == [2, 2, 2]
    assert list(offsets) == [0, 2, 4, 6]
    assert list(perm) == [0, 1, 1, 2, 0, 2]
    assert pos.tolist() == [[4, 0], [1, 2], [5, 3]]


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (64, 16, 5), (200, 64, 6), (5, 9, 9)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, pos = oracle.permute(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[E] == T * k and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(pos.ravel()), np.arange(T * k))       # bijection
    for t in range(T):
        for j in range(k):
            r = pos[t, j]
            assert perm[r] == t
            e = idx[t, j]
            assert offsets[e] <= r < offsets[e + 1]
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)  # tokens ascending, each once
        assert set(seg.tolist()) == {t for t in range(T) if e in idx[t]}


def test_permute_rejects_bad_indices():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 0]], dtype=np.int32), 4)
    with pytest.raises(ValueError):
        oracle.permute(np.array([[5]], dtype=np.int32), 4)


# ---- experts and the whole layer ------------------------------------------------------

def test_expert_ffn_matches_numpy():
    rng = np.random.default_rng(4)
    d, f = 24, 40
    x = rand_bf16(rng, (d,))
    wg = rand_bf16(rng, (f, d), d ** -0.5)
    wu = rand_bf16(rng, (f, d), d ** -0.5)
    wd = rand_bf16(rng, (d, f), f ** -0.5)
    h, y = oracle.expert_ffn(x, wg, wu, wd)
    h_ref, y_ref = np_ffn(x, wg, wu, wd)
    # h can differ only where silu(g)*u sits exactly on a bf16 half-way point
    assert np.array_equal(h, h_ref)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-13)


def test_layer_hand_computed():
    # T=1, d=2, f=1, E=2, k=1.  x = (1, 2); router = identity -> logits (1, 2),
    # expert 1 wins with weight 1.  g = 0.5*1 + 0.25*2 = 1, u = 1 + 2 = 3,
    # h = bf16(silu(1) * 3) = bf16(2.19317...) = 2.1875, y = (2.1875, -1.09375).
    x = as_bf16_bits([[1.0, 2.0]])
    wr = as_bf16_bits([[1.0, 0.0], [0.0, 1.0]])
    wg = as_bf16_bits([[[3.0, -1.0]], [[0.5, 0.25]]])
    wu = as_bf16_bits([[[1.0, 1.0]], [[1.0, 1.0]]])
    wd = as_bf16_bits([[[7.0], [7.0]], [[1.0], [-0.5]]])
    out, acc = oracle.layer(x, wr, None, wg, wu, wd, k=1)
    assert out[0].tolist() == [0x400C, 0xBF8C]
    assert acc[0].tolist() == [2.1875, -1.09375]


def _tiny_layer(rng, T, d, E, f, S=0, identical=False):
    x = rand_bf16(rng, (T, d))
    wr = rand_bf16(rng, (E, d), d ** -0.5)
    b = (rng.standard_normal(E) * 0.3).astype(np.float32)
    n = E + S
    if identical:
        wg = np.repeat(rand_bf16(rng, (1, f, d), d ** -0.5), n, axis=0)
        wu = np.repeat(rand_bf16(rng, (1, f, d), d ** -0.5), n, axis=0)
        wd = np.repeat(rand_bf16(rng, (1, d, f), f ** -0.5), n, axis=0)
    else:
        wg = rand_bf16(rng, (n, f, d), d ** -0.5)
        wu = rand_bf16(rng, (n, f, d), d ** -0.5)
        wd = rand_bf16(rng, (n, d, f), f ** -0.5)
    return x, wr, b, wg, wu, wd


@pytest.mark.parametrize("T,d,E,f", [(8, 32, 4, 32), (5, 16, 3, 24), (3, 8, 2, 12)])
def test_layer_k_equal_E_is_dense_mixture(T, d, E, f):
    rng = np.random.default_rng(T * d + E * f)
    x, wr, b, wg, wu, wd = _tiny_layer(rng, T, d, E, f)
    out, acc = oracle.layer(x, wr, b, wg, wu, wd, k=E)
    L = f64(x) @ f64(wr).T + b.astype(np.float64)
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    for t in range(T):
        ref = sum(p[t, e] * np_ffn(x[t], wg[e], wu[e], wd[e])[1] for e in range(E))
        assert np.allclose(acc[t], ref, rtol=1e-11, atol=1e-12)
        assert np.array_equal(f64(out[t]), np_round_bf16(acc[t]))


def test_layer_with_shared_expert_dense_check():
    rng = np.random.default_rng(11)
    T, d, E, f, k = 6, 16, 4, 20, 2
    x, wr, b, wg, wu, wd = _tiny_layer(rng, T, d, E, f, S=1)
    out, acc = oracle.layer(x, wr, b, wg, wu, wd, k=k, S=1)
    L = f64(x) @ f64(wr).T + b.astype(np.float64)
    for t in range(T):
        top = sorted(range(E), key=lambda e: (-L[t, e], e))[:k]
        wk = np.exp(L[t, top] - L[t, top].max())
        wk /= wk.sum()
        ref = sum(wk[j] * np_ffn(x[t], wg[e], wu[e], wd[e])[1] for j, e in enumerate(top))
        ref = ref + np_ffn(x[t], wg[E], wu[E], wd[E])[1]
        assert np.allclose(acc[t], ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_layer_identical_experts_is_one_ffn(k):
    rng = np.random.default_rng(20 + k)
    T, d, E, f = 7, 24, 5, 16
    x, wr, b, wg, wu, wd = _tiny_layer(rng, T, d, E, f, identical=True)
    out, acc = oracle.layer(x, wr, b, wg, wu, wd, k=k)
    for t in range(T):
        _, y = np_ffn(x[t], wg[0], wu[0], wd[0])
        assert np.allclose(acc[t], y, rtol=1e-12, atol=1e-13)


def test_layer_token_subset_equals_full():
    rng = np.random.default_rng(30)
    T, d, E, f, k = 12, 16, 6, 8, 2
    x, wr, b, wg, wu, wd = _tiny_layer(rng, T, d, E, f)
    full, _ = oracle.layer(x, wr, b, wg, wu, wd, k=k)
    sub = np.array([11, 0, 5], dtype=np.int32)
    part, _ = oracle.layer(x, wr, b, wg, wu, wd, k=k, tokens=sub)
    assert np.array_equal(part, full[sub])


def test_token_out_slot_order_and_weights():
    # token_out with explicit routing equals the weighted numpy sum
    rng = np.random.default_rng(31)
    d, f, E = 16, 12, 4
    _, _, _, wg, wu, wd = _tiny_layer(rng, 1, d, E, f)
    x = rand_bf16(rng, (d,))
    idx = np.array([3, 1], dtype=np.int32)
    w = np.array([0.7, 0.3])
    out, acc = oracle.token_out(x, idx, w, wg, wu, wd, E=E, S=0)
    ref = 0.7 * np_ffn(x, wg[3], wu[3], wd[3])[1] + 0.3 * np_ffn(x, wg[1], wu[1], wd[1])[1]
    assert np.allclose(acc, ref, rtol=1e-12, atol=1e-13)


# ---- residual add + RMSNorm after the combine ---------------------------------

def test_residual_rmsnorm_zero_residual_is_plain_output():
    # residual = 0: out is the combine value rounded once, i.e. the layer's output
    rng = np.random.default_rng(11)
    acc = rng.standard_normal((3, 64)) * 0.7
    zero = np.zeros((3, 64), dtype=np.uint16)
    gamma = as_bf16_bits(np.ones(64))
    out, _, _ = oracle.residual_rmsnorm(acc, zero, gamma, 1e-6)
    assert np.array_equal(f64(out), np_round_bf16(acc))


def test_residual_rmsnorm_hand_computed():
    # residual [1, 2, 3, 4] + acc [0.5, -0.5, 0.25, 0] -> out [1.5, 1.5, 3.25, 4]
    # mean square = (2.25 + 2.25 + 10.5625 + 16) / 4 = 7.765625
    res = as_bf16_bits([1.0, 2.0, 3.0, 4.0])[None, :]
    acc = np.array([[0.5, -0.5, 0.25, 0.0]])
    gamma = as_bf16_bits([1.0, 2.0, 0.5, -1.0])
    eps = 0.234375
    out, norm, norm64 = oracle.residual_rmsnorm(acc, res, gamma, eps)
    assert list(f64(out)[0]) == [1.5, 1.5, 3.25, 4.0]
    inv = 1.0 / math.sqrt(7.765625 + eps)  # = 1 / sqrt(8) exactly
    want = np.array([1.5 * inv, 1.5 * inv * 2.0, 3.25 * inv * 0.5, -4.0 * inv])
    assert np.allclose(norm64[0], want, rtol=0, atol=1e-15)
    assert np.array_equal(f64(norm)[0], np_round_bf16(want))


def test_residual_rmsnorm_unit_rms_and_scale_invariance():
    # eps = 0, gamma = 1: each row of out / rms has mean square 1, and scaling
    # the row by a power of two (exact in bf16) leaves the normalised row alone
    rng = np.random.default_rng(12)
    res = rand_bf16(rng, (4, 128))
    acc = np.zeros((4, 128))
    gamma = as_bf16_bits(np.ones(128))
    _, norm, norm64 = oracle.residual_rmsnorm(acc, res, gamma, 0.0)
    assert np.allclose(np.mean(norm64 ** 2, axis=1), 1.0, rtol=0, atol=1e-12)
    res8 = bits_of(f64(res) * 8.0)
    _, norm8, norm64_8 = oracle.residual_rmsnorm(acc, res8, gamma, 0.0)
    assert np.allclose(norm64_8, norm64, rtol=0, atol=1e-14)
    assert np.array_equal(norm8, norm)


def test_residual_rmsnorm_constant_row_gives_signed_gamma():
    # a row of equal values v normalises to sign(v) * gamma (eps = 0)
    res = as_bf16_bits(np.full((2, 32), 0.0))
    acc = np.vstack([np.full(32, 3.0), np.full(32, -0.125)])
    rng = np.random.default_rng(13)
    gamma = rand_bf16(rng, (32,))
    _, norm, _ = oracle.residual_rmsnorm(acc, res, gamma, 0.0)
    assert np.array_equal(f64(norm)[0], f64(gamma))
    assert np.array_equal(f64(norm)[1], -f64(gamma))


# ---- step 10: the spatial split of the CTAs (cost model) ----------------------

PHI32 = float(np.float32(1925e12) / np.float32(152))


def _work_by_enumeration(T, d, f, k, S, touched, ybytes):
    """Mover bytes, GEMM FLOPs and weight bytes of a layer, counted copy by
    copy, row by row and matrix by matrix (exact integers); ybytes is the size
    of one stored expert-output value the combine reads (2: bf16; 4 * ks: ks
    fp32 partial sums)."""
    moved = 0
    for _ in range(T * k):          # gather: a token row read, a permuted row written
        moved += d * 2 + d * 2
    for _ in range(T):              # combine: the token's expert outputs read, its row written
        for _ in range(k + S):
            moved += d * ybytes
        moved += d * 2
    flops = 0
    for _ in range(T * k + T * S):  # per row: gate and up (d x f MACs each), down (f x d)
        flops += 2 * (d * f) + 2 * (d * f) + 2 * (f * d)
    wbytes = 0
    for _ in range(touched + S):    # per touched expert: gate, up and down, bf16
        for _ in range(3):
            wbytes += f * d * 2
    return moved, flops, wbytes


def _random_layers(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        E = int(rng.integers(1, 65))
        yield dict(T=int(rng.integers(1, 48)), d=64 * int(rng.integers(1, 65)),
                   f=64 * int(rng.integers(1, 65)), k=int(rng.integers(1, min(E, 16) + 1)),
                   S=int(rng.integers(0, 2)), touched=int(rng.integers(1, E + 1)),
                   N=int(rng.integers(1, 300)), ybytes=int(rng.choice([2, 4, 8, 16])),
                   beta=float(10.0 ** rng.uniform(8, 12)),
                   phi=float(10.0 ** rng.uniform(10, 14)), bw=float(10.0 ** rng.uniform(11, 13)))


@pytest.mark.parametrize("seed", [0, 1])
def test_movers_minimise_the_slower_side(seed):
    # the split's real value is N a / (a + b) with a and b recounted here copy
    # by copy; the integer split is within one of the brute-force minimiser of
    # the slower side's time max(a / M, b / (N - M)) over M = 1 .. N - 1
    for c in _random_layers(150, seed):
        moved, flops, wbytes = _work_by_enumeration(c["T"], c["d"], c["f"], c["k"], c["S"],
                                                    c["touched"], c["ybytes"])
        beta, phi, bw = (float(np.float32(c[key])) for key in ("beta", "phi", "bw"))
        a = moved / beta
        b = max(flops / phi, c["N"] * wbytes / bw)
        m, x = oracle.movers(c["T"], c["d"], c["f"], c["k"], c["S"], c["touched"], c["N"],
                             c["ybytes"], c["beta"], c["phi"], c["bw"])
        assert abs(x - c["N"] * a / (a + b)) <= 1e-5 * c["N"], c
        N = c["N"]
        if N == 1:
            assert m == 1
            continue
        cost = [max(a / M, b / (N - M)) for M in range(1, N)]
        best = 1 + int(np.argmin(cost))
        assert 1 <= m <= max(N - 1, 1) and abs(m - best) <= 1, (c, m, best)


def test_movers_follow_a_three_to_one_ratio():
    # movers' work three times the GEMM side's: three quarters of the CTAs
    # move data (a swap of the two sides would give one quarter)
    T, d, f, k, S, touched, ybytes, N = 32, 512, 256, 4, 1, 6, 8, 16
    moved, flops, wbytes = _work_by_enumeration(T, d, f, k, S, touched, ybytes)
    bw = 6.79e12
    b = max(flops / PHI32, N * wbytes / float(np.float32(bw)))
    beta = moved / (3.0 * b)
    m, x = oracle.movers(T, d, f, k, S, touched, N, ybytes, beta, PHI32, bw)
    assert abs(x - 12.0) < 1e-4 and m == 12
    m, x = oracle.movers(T, d, f, k, S, touched, N, ybytes, moved / (b / 3.0), PHI32, bw)
    assert abs(x - 4.0) < 1e-4 and m == 4


def test_movers_round_to_the_nearest_split():
    # with a / b = 0.27 / 0.73 the real split of 10 CTAs is 2.7 movers, which
    # rounds to 3; with 0.23 / 0.77 it is 2.3, which rounds to 2
    T, d, f, k, S, touched, ybytes, N = 16, 256, 512, 2, 0, 3, 2, 10
    moved, flops, wbytes = _work_by_enumeration(T, d, f, k, S, touched, ybytes)
    bw = 6.79e12
    b = max(flops / PHI32, N * wbytes / float(np.float32(bw)))
    for frac, want in ((0.27, 3), (0.23, 2)):
        beta = moved / (frac / (1.0 - frac) * b)
        m, x = oracle.movers(T, d, f, k, S, touched, N, ybytes, beta, PHI32, bw)
        assert abs(x - 10 * frac) < 1e-4 and m == want


def test_movers_clamps():
    args = (64, 256, 256, 2, 0, 4)
    # data movement dwarfs the GEMMs: all CTAs but one move data
    assert oracle.movers(*args, 16, 4, 1e3, PHI32, 6.79e12)[0] == 15
    # the GEMMs dwarf data movement: one mover is kept
    assert oracle.movers(*args, 16, 4, 1e30, PHI32, 6.79e12)[0] == 1
    # one or two CTAs: a single mover (the other side shares it or the last CTA)
    for beta in (1e3, 1e30):
        assert oracle.movers(*args, 1, 4, beta, PHI32, 6.79e12)[0] == 1
        assert oracle.movers(*args, 2, 4, beta, PHI32, 6.79e12)[0] == 1


def test_movers_fall_as_more_experts_are_touched():
    # more touched experts means more weight bytes on the GEMM side
    prev = None
    for touched in range(1, 129, 8):
        m, _ = oracle.movers(512, 2048, 768, 8, 0, touched, 152, 4, 40e9, PHI32, 6.79e12)
        assert prev is None or m <= prev
        prev = m
    assert prev < oracle.movers(512, 2048, 768, 8, 0, 1, 152, 4, 40e9, PHI32, 6.79e12)[0]
