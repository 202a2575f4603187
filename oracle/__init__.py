"""CPU oracle of the MoE-layer forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
behind ``include/moe.h`` and its Python binding) never touches it and shares no
code with it.

This module is argument marshalling around ``moe_oracle.c`` (plain,
single-threaded C, fp64 accumulation); the arithmetic and the passages it
follows are documented there.  All bf16 tensors are passed as ``numpy.uint16``
bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoeoracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (no CUDA involved)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        u16 = ctypes.c_uint16
        lib.orc_bf16_to_f64.argtypes = [u16]
        lib.orc_bf16_to_f64.restype = dbl
        lib.orc_f64_to_bf16.argtypes = [dbl]
        lib.orc_f64_to_bf16.restype = u16
        lib.orc_bf16_to_f64_array.argtypes = [i64, vp, vp]
        lib.orc_f64_to_bf16_array.argtypes = [i64, vp, vp]
        lib.orc_silu.argtypes = [dbl]
        lib.orc_silu.restype = dbl
        lib.orc_router_logits.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        lib.orc_topk.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
        lib.orc_permute.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
        lib.orc_permute.restype = i32
        lib.orc_expert_ffn.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_token_out.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_layer_tokens.argtypes = [i32] * 6 + [vp] * 6 + [i32, vp, vp, vp]
        lib.orc_residual_rmsnorm.argtypes = [i32, i32, vp, vp, vp, dbl, vp, vp, vp]
        flt = ctypes.c_float
        lib.orc_movers.argtypes = [i32] * 7 + [flt, flt, flt, flt, ctypes.POINTER(flt)]
        lib.orc_movers.restype = i32
        for fn in (lib.orc_bf16_to_f64_array, lib.orc_f64_to_bf16_array, lib.orc_router_logits,
                   lib.orc_topk, lib.orc_expert_ffn, lib.orc_token_out, lib.orc_layer_tokens,
                   lib.orc_residual_rmsnorm):
            fn.restype = None
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---- bf16 -------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _L().orc_bf16_to_f64_array(bits.size, _p(bits), _p(out))
    return out


def f64_to_bf16(vals: np.ndarray) -> np.ndarray:
    vals = _c(vals, np.float64)
    out = np.empty(vals.shape, dtype=np.uint16)
    _L().orc_f64_to_bf16_array(vals.size, _p(vals), _p(out))
    return out


def silu(z: float) -> float:
    return _L().orc_silu(float(z))


# ---- routing -----------------------------------------------------------------

def router_logits(x: np.ndarray, router_w: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """L[t,e] = sum_i x[t,i] Wr[e,i] + b[e] in fp64, shape [T, E]."""
    x = _c(x, np.uint16)
    router_w = _c(router_w, np.uint16)
    bias = _c(bias, np.float32)
    T, d = x.shape
    E = router_w.shape[0]
    assert router_w.shape == (E, d)
    L = np.empty((T, E), dtype=np.float64)
    _L().orc_router_logits(T, d, E, _p(x), _p(router_w), _p(bias), _p(L))
    return L


def topk(L: np.ndarray, k: int):
    """Softmax over all E, top-k (p desc, expert asc), renormalise.

    Returns (idx int32 [T,k], w float64 [T,k], p float64 [T,E], gap float64 [T])."""
    L = _c(L, np.float64)
    T, E = L.shape
    assert 1 <= k <= E
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    p = np.empty((T, E), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    _L().orc_topk(T, E, k, _p(L), _p(idx), _p(w), _p(p), _p(gap))
    return idx, w, p, gap


def route(x, router_w, bias, k):
    L = router_logits(x, router_w, bias)
    idx, w, p, gap = topk(L, k)
    return {"logits": L, "idx": idx, "w": w, "p": p, "gap": gap}


def permute(idx: np.ndarray, E: int):
    """(counts [E], offsets [E+1], perm [T*k], pos [T,k]) of the canonical order."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    rc = _L().orc_permute(T, E, k, _p(idx), _p(counts), _p(offsets), _p(perm), _p(pos))
    if rc != 0:
        raise ValueError("invalid expert indices")
    return counts, offsets, perm, pos


# ---- experts and output --------------------------------------------------------

def expert_ffn(x_row, wg_e, wu_e, wd_e):
    """(h [f], y [d]) of one expert ([f,d], [f,d], [d,f] blocks) on one token."""
    x_row = _c(x_row, np.uint16)
    wg_e, wu_e, wd_e = (_c(a, np.uint16) for a in (wg_e, wu_e, wd_e))
    f, d = wg_e.shape
    assert x_row.shape == (d,) and wu_e.shape == (f, d) and wd_e.shape == (d, f)
    h = np.empty(f, dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    _L().orc_expert_ffn(d, f, _p(x_row), _p(wg_e), _p(wu_e), _p(wd_e), _p(h), _p(y))
    return h, y


def token_out(x_row, idx_row, w_row, w_gate, w_up, w_down, E: int, S: int):
    """(out bf16 bits [d], value before rounding float64 [d]) of one token."""
    x_row = _c(x_row, np.uint16)
    idx_row = _c(idx_row, np.int32)
    w_row = _c(w_row, np.float64)
    w_gate, w_up, w_down = (_c(a, np.uint16) for a in (w_gate, w_up, w_down))
    nt, f, d = w_gate.shape
    assert nt == E + S and w_down.shape == (nt, d, f)
    k = idx_row.shape[0]
    out = np.empty(d, dtype=np.uint16)
    acc = np.empty(d, dtype=np.float64)
    _L().orc_token_out(d, f, E, k, S, _p(x_row), _p(idx_row), _p(w_row), _p(w_gate), _p(w_up),
                       _p(w_down), _p(acc), _p(out))
    return out, acc


def layer(x, router_w, bias, w_gate, w_up, w_down, k: int, S: int = 0, tokens=None):
    """Output rows of the layer for the listed tokens (all tokens if None).

    Returns (out bf16 bits [n, d], value before rounding float64 [n, d])."""
    x = _c(x, np.uint16)
    router_w = _c(router_w, np.uint16)
    bias = _c(bias, np.float32)
    w_gate, w_up, w_down = (_c(a, np.uint16) for a in (w_gate, w_up, w_down))
    T, d = x.shape
    E = router_w.shape[0]
    nt, f, _ = w_gate.shape
    assert nt == E + S
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, d), dtype=np.uint16)
    acc = np.empty((n, d), dtype=np.float64)
    _L().orc_layer_tokens(T, d, f, E, k, S, _p(x), _p(router_w), _p(bias), _p(w_gate), _p(w_up),
                          _p(w_down), n, _p(tok), _p(out), _p(acc))
    return out, acc


def residual_rmsnorm(acc, residual, gamma, eps: float):
    """Residual add and RMSNorm after the combine (xxqk.cn/news/665650
    section 1 lists both as the megakernel's last steps).

    acc: the combine's rows before rounding, float64 [n, d] (``layer``'s second
    result); residual: bf16 bits [n, d]; gamma: bf16 bits [d].  Returns
    (out bf16 bits [n, d], norm_out bf16 bits [n, d], norm before rounding
    float64 [n, d]) with out = bf16(residual + acc) and
    norm_out = bf16(out / sqrt(mean(out^2) + eps) * gamma)."""
    acc = _c(acc, np.float64)
    residual = _c(residual, np.uint16)
    gamma = _c(gamma, np.uint16)
    n, d = acc.shape
    assert residual.shape == (n, d) and gamma.shape == (d,)
    out = np.empty((n, d), dtype=np.uint16)
    norm = np.empty((n, d), dtype=np.uint16)
    norm64 = np.empty((n, d), dtype=np.float64)
    _L().orc_residual_rmsnorm(n, d, _p(acc), _p(residual), _p(gamma), float(eps), _p(out),
                              _p(norm), _p(norm64))
    return out, norm, norm64


def movers(T: int, d: int, f: int, k: int, S: int, touched_routed: int, N: int,
           ybytes: float, beta: float, phi: float, bw: float):
    """The spatial split of the Weave abstract (CTAs for data movement against
    CTAs for the expert GEMMs, in the ratio of the two sides' work once
    routing is known), as ``moe_oracle.c: orc_movers`` defines it.

    touched_routed: routed experts with at least one token; N: CTAs; ybytes:
    bytes the combine reads per expert-output value (2 for bf16 outputs, 4 * ks
    for ks fp32 partial sums); beta (B/s per mover), phi (FLOP/s per GEMM
    worker), bw (B/s): the cost model's constants, each rounded to fp32 like
    the rest of the arithmetic.  Returns (M*, the value N*a/(a+b) before
    rounding)."""
    m_cont = ctypes.c_float(0.0)
    m = _L().orc_movers(int(T), int(d), int(f), int(k), int(S), int(touched_routed), int(N),
                        float(np.float32(ybytes)), float(np.float32(beta)),
                        float(np.float32(phi)), float(np.float32(bw)), ctypes.byref(m_cont))
    return int(m), float(m_cont.value)
