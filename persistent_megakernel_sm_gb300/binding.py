"""ctypes binding of include/moe.h: argument marshalling only.

Each C entry point is exposed under its own name on ``lib`` (a ``ctypes.CDLL``
with argument and return types set from the header).  ``MoELayer`` wraps a
handle for callers holding torch tensors: it passes ``data_ptr()`` values and
the current CUDA stream, and turns non-zero status codes into ``MoEError``.
Every step of the layer runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmoe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe.h")

MOE_OK, MOE_E_INVAL, MOE_E_CUDA, MOE_E_TIMEOUT, MOE_E_DEVICE, MOE_E_NOMEM, MOE_E_STATE = range(7)
MOE_MODE_PERSISTENT, MOE_MODE_MULTIKERNEL, MOE_MODE_STATIC = 0, 1, 2

OPTIONS = {
    "mode": 1, "timeout_ns": 2, "mover_ctas": 3, "grid_ctas": 4, "split_k": 5,
    "tokens_per_tile": 6, "fault_drop_task": 7, "route_tokens": 8, "claim_ahead": 9,
    "trace": 10, "release": 11, "prefetch": 12, "bands": 13, "route_splits": 14, "l2_prefetch": 15,
    "pair": 16, "front_split": 17, "fault_drop_type": 18, "fault_corrupt_count": 19,
    "fault_repush": 20, "debug_claims": 21, "fold_gather": 22,
}
STATS = {"mover_ctas": 1, "tasks": 2, "grid": 3, "gemm_tasks": 4, "mover_tasks": 5, "stolen": 6,
         "ahead": 7, "trace_records": 8, "tile_tokens": 9, "split_k": 10, "bands": 11, "y_bytes": 12,
         "combine_tokens": 13, "pair": 14}
TASK_TYPES = {1: "route", 2: "gather", 3: "gateup", 4: "down", 5: "combine", 6: "plan"}

_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong

_SIGNATURES = {
    "moe_layer_create": ([_i32, _i32, _i32, _i32, _i32], _vp),
    "moe_layer_reserve": ([_vp, _i32, _vp], _i32),
    "moe_layer_set_router_bias": ([_vp, _vp], _i32),
    "moe_layer_forward": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "moe_layer_forward_host": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "moe_layer_forward_noalloc": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "moe_layer_forward_residual_norm": ([_vp, _i32] + [_vp] * 7 + [ctypes.c_float, _vp, _vp, _vp],
                                        _i32),
    "moe_layer_calibrate": ([_vp, _i32] + [_vp] * 6 + [_i32, _vp, _vp], _i32),
    "moe_layer_get_routing": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "moe_layer_status": ([_vp, _vp], _i32),
    "moe_layer_set_option": ([_vp, _i32, _i64], _i32),
    "moe_layer_get_stat": ([_vp, _i32], _i64),
    "moe_layer_workspace_bytes": ([_vp, _i32], _i64),
    "moe_layer_get_trace": ([_vp, _vp, _i32, _vp], _i32),
    "moe_layer_destroy": ([_vp], None),
    "moe_last_error": ([], ctypes.c_char_p),
}


class MoEError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"moe error {code}: {msg}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (raises OSError if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with persistent_megakernel_sm_gb300.build")
    dll = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(dll, name)
        fn.argtypes = args
        fn.restype = res
    _lib = dll
    return dll


class _LazyLib:
    def __getattr__(self, name):
        return getattr(load_library(), name)


lib = _LazyLib()


def header_symbols(header: str = HEADER) -> list[str]:
    """Names of the functions include/moe.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def _err(code: int):
    if code != MOE_OK:
        raise MoEError(code, (lib.moe_last_error() or b"").decode())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _check_tensor(name, t, dtype, shape, rows_at_least=False):
    """Refuse a tensor the kernels would read or write out of its bounds: wrong
    dtype or shape, not contiguous, or not on a CUDA device.  ``shape`` is the
    exact shape, except that with ``rows_at_least`` the first dimension may be
    larger (an output buffer with room for more rows)."""
    if t.dtype != dtype:
        raise MoEError(MOE_E_INVAL, f"{name}: dtype {t.dtype}, expected {dtype}")
    got = tuple(t.shape)
    ok = (len(got) == len(shape) and got[1:] == tuple(shape[1:]) and
          (got[0] >= shape[0] if rows_at_least else got[0] == shape[0]))
    if not ok:
        want = ("[>=%d, %s]" % (shape[0], ", ".join(map(str, shape[1:])))
                if rows_at_least else str(list(shape)))
        raise MoEError(MOE_E_INVAL, f"{name}: shape {list(got)}, expected {want}")
    if not t.is_contiguous():
        raise MoEError(MOE_E_INVAL, f"{name}: not contiguous")
    if not t.is_cuda:
        raise MoEError(MOE_E_INVAL, f"{name}: not a CUDA tensor")


class MoELayer:
    """One MoE layer handle (d, f, E, k, shared experts).

    The tensor-taking methods check each tensor's dtype (bf16; the bias fp32),
    shape, contiguity and device before the C call, so that a mismatched
    tensor raises ``MoEError`` instead of being read out of bounds."""

    def __init__(self, d: int, f: int, E: int, k: int, shared_experts: int = 0):
        h = lib.moe_layer_create(d, f, E, k, shared_experts)
        if not h:
            raise MoEError(MOE_E_INVAL, (lib.moe_last_error() or b"").decode())
        self.h = ctypes.c_void_p(h)
        self.d, self.f, self.E, self.k, self.S = d, f, E, k, shared_experts
        self._bias = None

    def reserve(self, T_max: int, stream=None):
        _err(lib.moe_layer_reserve(self.h, T_max, _stream_ptr(stream)))

    def _check_weights(self, router_w, w_gate, w_up, w_down):
        import torch
        bf, n = torch.bfloat16, self.E + self.S
        _check_tensor("router_w", router_w, bf, (self.E, self.d))
        _check_tensor("w_gate", w_gate, bf, (n, self.f, self.d))
        _check_tensor("w_up", w_up, bf, (n, self.f, self.d))
        _check_tensor("w_down", w_down, bf, (n, self.d, self.f))

    def _check_rows(self, T, **rows):
        import torch
        for name, t in rows.items():
            _check_tensor(name, t, torch.bfloat16, (T, self.d), rows_at_least=name != "x")

    def set_router_bias(self, bias):
        if bias is not None:
            import torch
            _check_tensor("bias", bias, torch.float32, (self.E,))
        self._bias = bias  # keep the tensor alive while the library holds its pointer
        _err(lib.moe_layer_set_router_bias(self.h, None if bias is None else bias.data_ptr()))

    def set_option(self, key, value: int):
        _err(lib.moe_layer_set_option(self.h, OPTIONS.get(key, key), int(value)))

    def forward(self, x, router_w, w_gate, w_up, w_down, out, stream=None):
        T = x.shape[0]
        self._check_weights(router_w, w_gate, w_up, w_down)
        self._check_rows(T, x=x, out=out)
        _err(lib.moe_layer_forward(self.h, T, x.data_ptr(), router_w.data_ptr(),
                                   w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
                                   out.data_ptr(), _stream_ptr(stream)))
        return out

    def forward_residual_norm(self, x, router_w, w_gate, w_up, w_down, residual, gamma, eps,
                              out, norm_out, stream=None):
        """moe_layer_forward_residual_norm: out = residual + layer(x), norm_out =
        RMSNorm(out) * gamma, fused into the combine."""
        import torch
        T = x.shape[0]
        self._check_weights(router_w, w_gate, w_up, w_down)
        self._check_rows(T, x=x, out=out, residual=residual, norm_out=norm_out)
        _check_tensor("gamma", gamma, torch.bfloat16, (self.d,))
        _err(lib.moe_layer_forward_residual_norm(
            self.h, T, x.data_ptr(), router_w.data_ptr(), w_gate.data_ptr(), w_up.data_ptr(),
            w_down.data_ptr(), residual.data_ptr(), gamma.data_ptr(), float(eps), out.data_ptr(),
            norm_out.data_ptr(), _stream_ptr(stream)))
        return out, norm_out

    def calibrate(self, x, router_w, w_gate, w_up, w_down, out, reps: int = 3, stream=None):
        """moe_layer_calibrate: time candidate tile sizes, K splits and d bands
        on these inputs and keep the fastest as options; returns the best mean
        time in microseconds."""
        T = x.shape[0]
        self._check_weights(router_w, w_gate, w_up, w_down)
        self._check_rows(T, x=x, out=out)
        best = ctypes.c_float(0.0)
        _err(lib.moe_layer_calibrate(self.h, T, x.data_ptr(), router_w.data_ptr(),
                                     w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
                                     out.data_ptr(), int(reps), ctypes.byref(best),
                                     _stream_ptr(stream)))
        return best.value

    def forward_noalloc(self, x, router_w, w_gate, w_up, w_down, out, stream=None):
        """moe_layer_forward_noalloc: the same pass on the library's fixed scratch,
        allocating nothing (for callers that cannot allocate device memory)."""
        T = x.shape[0]
        self._check_weights(router_w, w_gate, w_up, w_down)
        self._check_rows(T, x=x, out=out)
        _err(lib.moe_layer_forward_noalloc(self.h, T, x.data_ptr(), router_w.data_ptr(),
                                          w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
                                          out.data_ptr(), _stream_ptr(stream)))
        return out

    def forward_host(self, T, x_host_ptr, router_w, w_gate, w_up, w_down, out_host_ptr,
                     stream=None):
        """moe_layer_forward_host: x and out are host addresses of T x d bf16
        values each (pinned memory for asynchronous copies)."""
        self._check_weights(router_w, w_gate, w_up, w_down)
        _err(lib.moe_layer_forward_host(self.h, T, x_host_ptr, router_w.data_ptr(),
                                        w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
                                        out_host_ptr, _stream_ptr(stream)))

    def status(self, stream=None) -> int:
        return lib.moe_layer_status(self.h, _stream_ptr(stream))

    def check(self, stream=None):
        _err(self.status(stream))

    def get_routing(self, idx=None, w=None, counts=None, offsets=None, perm=None, pos=None,
                    stream=None):
        ptr = (lambda t: None if t is None else t.data_ptr())
        _err(lib.moe_layer_get_routing(self.h, ptr(idx), ptr(w), ptr(counts), ptr(offsets),
                                       ptr(perm), ptr(pos), _stream_ptr(stream)))

    def stat(self, key) -> int:
        return lib.moe_layer_get_stat(self.h, STATS.get(key, key))

    def trace(self, cap: int = 1 << 16, stream=None):
        """Task records of the last forward as a numpy array of dicts-of-arrays:
        cta, task id, type, t_claim, t_start, t_end (ns, %globaltimer)."""
        import numpy as np
        buf = np.zeros((cap, 4), dtype=np.uint64)
        n = lib.moe_layer_get_trace(self.h, buf.ctypes.data, cap, _stream_ptr(stream))
        if n < 0:
            raise MoEError(MOE_E_CUDA, (lib.moe_last_error() or b"").decode())
        buf = buf[:n]
        task = (buf[:, 0] & 0xffffffff).astype(np.int64)
        return {"cta": (buf[:, 0] >> 32).astype(np.int64), "task": task,
                "type": task >> 28, "t_claim": buf[:, 1].astype(np.int64),
                "t_start": buf[:, 2].astype(np.int64), "t_end": buf[:, 3].astype(np.int64)}

    def workspace_bytes(self, T_max: int) -> int:
        return lib.moe_layer_workspace_bytes(self.h, T_max)

    def close(self):
        if self.h:
            lib.moe_layer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
