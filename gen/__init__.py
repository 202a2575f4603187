"""Seeded synthetic inputs for the MoE-layer forward pass.

This module draws the layer's inputs and nothing else: token activations ``x``,
the router weight, the expert weights and the router bias, as raw bfloat16 bit
patterns (``numpy.uint16``) or float32.  It holds none of the layer's
arithmetic, so both the CUDA path (through ``bench.py``) and the CPU oracle
(through ``tests/``) can take their inputs from here.

Workloads (the five layer shapes the method is measured on):

========  =====  =====  ===  ==  =====  =  ==================================
name      T      d      E    k   f      S  router bias
========  =====  =====  ===  ==  =====  =  ==================================
tiny      64     256    8    2   512    0  none
decode    256    4096   8    2   14336  0  none (near-uniform routing)
fine      512    2048   128  8   768    0  b_e ~ N(0, 0.5^2)
skew      4096   4096   64   6   1408   0  fitted so counts follow Zipf(1.2)
prefill   8192   7168   256  8   2048   1  b_e ~ N(0, 0.3^2)
========  =====  =====  ===  ==  =====  =  ==================================

(``decode_small``: decode with f = 2048, and ``prefill_small``: prefill's
expert shape with E = 32 and T = 1024, small cases for profiler captures.)

Distributions: x ~ N(0, 1); router_w ~ N(0, 1/d); w_gate, w_up ~ N(0, 1/d);
w_down ~ N(0, 1/f) ("N(0, 1/fan_in)" read as a variance).  Every workload uses
seed 0.  Layouts: x [T, d], router_w [E, d], w_gate / w_up [E+S, f, d],
w_down [E+S, d, f], all row-major; the shared expert (S = 1) is stored last.

Two per-workload facts are not drawn here but read from committed files in
``tests/golden/`` that a committed script computes with the CPU oracle:
the fitted router bias of ``skew`` and the per-token redraw counters
(``retry``) that keep the k-th and (k+1)-th router logits of every token more
than 1e-3 apart.  Token row t is drawn from its own stream, shifted by its
retry counter, so a redraw leaves every other row unchanged.
"""
from __future__ import annotations

import ctypes
import json
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_REPO = os.path.dirname(_HERE)
_GOLDEN = os.path.join(_REPO, "tests", "golden")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoegen.so")
_SRC = os.path.join(_HERE, "gen.c")

# stream ids of the generator (one per tensor)
TID_X = 1
TID_ROUTER_W = 2
TID_W_GATE = 3
TID_W_UP = 4
TID_W_DOWN = 5
TID_BIAS = 6
TID_EXPERT_PERM = 7

SEED = 0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    S: int = 0
    bias: tuple = field(default=())  # () | ("normal", std) | ("zipf", s)

    @property
    def n_experts_total(self) -> int:
        return self.E + self.S

    def weight_bytes(self) -> int:
        """bf16 bytes of every weight tensor (router + all experts)."""
        return 2 * (self.E * self.d + 3 * self.n_experts_total * self.f * self.d)

    def describe(self) -> str:
        return (f"T={self.T} d={self.d} E={self.E} k={self.k} f={self.f} S={self.S} "
                f"bias={self.bias or 'none'}")


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 8, 2, 512, 0, ()),
    "decode": Workload("decode", 256, 4096, 8, 2, 14336, 0, ()),
    "fine": Workload("fine", 512, 2048, 128, 8, 768, 0, ("normal", 0.5)),
    "skew": Workload("skew", 4096, 4096, 64, 6, 1408, 0, ("zipf", 1.2)),
    "prefill": Workload("prefill", 8192, 7168, 256, 8, 2048, 1, ("normal", 0.3)),
    # decode's shape with a narrower expert (f = 2048): 403 MB of weights, above
    # the L2 size, for profiling captures that must stay small
    "decode_small": Workload("decode_small", 256, 4096, 8, 2, 2048, 0, ()),
    # prefill's expert shape (d = 7168, f = 2048, top-8, one shared expert) with
    # 32 experts and 1024 tokens, so each expert still receives ~256 rows:
    # 2.9 GB of weights, for profiling captures that must stay small
    "prefill_small": Workload("prefill_small", 1024, 7168, 32, 8, 2048, 1, ("normal", 0.3)),
}


def build(force: bool = False) -> str:
    """Compile the generator (plain C, pthreads) into gen/_build."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, dbl = ctypes.c_uint64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.gen_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        lib.gen_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        lib.gen_uniform_f64.argtypes = [u64, u64, u64, u64, vp]
        lib.gen_x_rows.argtypes = [u64, u64, i32, i32, vp, vp, i32]
        for fn in (lib.gen_normal_bf16, lib.gen_normal_f32, lib.gen_uniform_f64, lib.gen_x_rows):
            fn.restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(tid: int, shape, std: float, seed: int = SEED, first: int = 0,
                out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _L().gen_normal_bf16(seed, tid, first, n, float(std), out.ctypes.data, _threads())
    return out


def normal_f32(tid: int, n: int, std: float, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _L().gen_normal_f32(seed, tid, 0, n, float(std), out.ctypes.data, _threads())
    return out


def uniforms(tid: int, n: int, seed: int = SEED, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().gen_uniform_f64(seed, tid, first, n, out.ctypes.data)
    return out


def x_rows(T: int, d: int, retry: np.ndarray | None = None, seed: int = SEED,
           out: np.ndarray | None = None) -> np.ndarray:
    if out is None:
        out = np.empty((T, d), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == T * d
    rp = None
    if retry is not None:
        retry = np.ascontiguousarray(retry, dtype=np.int32)
        assert retry.shape == (T,)
        rp = retry.ctypes.data
    _L().gen_x_rows(seed, TID_X, T, d, rp, out.ctypes.data, _threads())
    return out


def router_w(w: Workload, seed: int = SEED) -> np.ndarray:
    return normal_bf16(TID_ROUTER_W, (w.E, w.d), 1.0 / np.sqrt(w.d), seed)


def expert_weights(w: Workload, seed: int = SEED):
    """(w_gate [E+S,f,d], w_up [E+S,f,d], w_down [E+S,d,f]) as bf16 bits."""
    nt = w.n_experts_total
    wg = normal_bf16(TID_W_GATE, (nt, w.f, w.d), 1.0 / np.sqrt(w.d), seed)
    wu = normal_bf16(TID_W_UP, (nt, w.f, w.d), 1.0 / np.sqrt(w.d), seed)
    wd = normal_bf16(TID_W_DOWN, (nt, w.d, w.f), 1.0 / np.sqrt(w.f), seed)
    return wg, wu, wd


def zipf_target_counts(w: Workload) -> np.ndarray:
    """Target per-expert counts for the skewed workload.

    c_e proportional to rank^-s over E experts, total T*k, water-filled under
    the cap T (an expert can take each token at most once): capped experts are
    fixed at T and the excess is spread over the rest in proportion to their
    Zipf weight, repeated until nothing exceeds T.  Ranks map to experts by a
    seeded permutation.  Returned as float64 (not rounded)."""
    assert w.bias and w.bias[0] == "zipf"
    s = float(w.bias[1])
    total = float(w.T * w.k)
    weight = np.arange(1, w.E + 1, dtype=np.float64) ** (-s)
    capped = np.zeros(w.E, dtype=bool)
    c = np.zeros(w.E)
    for _ in range(w.E + 1):
        free = ~capped
        rem = total - w.T * capped.sum()
        c = np.where(capped, float(w.T), rem * weight / weight[free].sum())
        over = free & (c > w.T)
        if not over.any():
            break
        capped |= over
    order = np.argsort(uniforms(TID_EXPERT_PERM, w.E), kind="stable")
    out = np.empty(w.E)
    out[order] = c  # rank r -> expert order[r]
    return out


def _meta_path(name: str) -> str:
    return os.path.join(_GOLDEN, f"{name}_inputs.json")


def load_meta(name: str) -> dict | None:
    p = _meta_path(name)
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        return json.load(fh)


def router_bias(w: Workload, seed: int = SEED, meta: dict | None = None) -> np.ndarray | None:
    if not w.bias:
        return None
    if w.bias[0] == "normal":
        return normal_f32(TID_BIAS, w.E, float(w.bias[1]), seed)
    if w.bias[0] == "zipf":
        meta = meta if meta is not None else load_meta(w.name)
        if meta is None or "bias" not in meta:
            raise FileNotFoundError(
                f"fitted router bias for workload '{w.name}' missing: run "
                "tests/golden/make_inputs_meta.py")
        b = np.asarray(meta["bias"], dtype=np.float32)
        assert b.shape == (w.E,)
        return b
    raise ValueError(w.bias)


def retries(w: Workload, meta: dict | None = None) -> np.ndarray | None:
    """Per-token redraw counters from the committed metadata (None = all zero)."""
    meta = meta if meta is not None else load_meta(w.name)
    if meta is None or not meta.get("retry"):
        return None
    r = np.zeros(w.T, dtype=np.int32)
    for t, n in meta["retry"].items():
        r[int(t)] = int(n)
    return r


def make_inputs(w: Workload | str, seed: int = SEED, with_experts: bool = True,
                retry: np.ndarray | None = None, use_meta: bool = True) -> dict:
    """All inputs of one workload as numpy arrays (bf16 bits as uint16)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    meta = load_meta(w.name) if use_meta else None
    if retry is None and meta is not None:
        retry = retries(w, meta)
    out = {
        "x": x_rows(w.T, w.d, retry, seed),
        "router_w": router_w(w, seed),
        "bias": router_bias(w, seed, meta),
        "retry": retry,
    }
    if with_experts:
        out["w_gate"], out["w_up"], out["w_down"] = expert_weights(w, seed)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Reinterpret bf16 bit patterns as float32 (exact widening)."""
    return (a.astype(np.uint32) << 16).view(np.float32)
