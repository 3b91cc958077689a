"""fp64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The library's compute path never does: it has
no CPU fallback.

The arithmetic lives in ``gdr_oracle.c`` (plain C, fp64, one token at a time,
in the order of the per-token Loop on the Qwen3.5-9B NPU model card, section
"How it works"; and the plain row-wise steps on either side of the rule: q/k
L2 normalisation, beta from its logit, the gated RMSNorm of the outputs).
This module compiles it with gcc on first use and marshals numpy arrays to it;
it adds no arithmetic of its own.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (gcc, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    f = lib.oracle_gdr_sequential
    dp = ctypes.POINTER(ctypes.c_double)
    f.argtypes = [
        ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, ctypes.c_int,
    ]
    f.restype = ctypes.c_int
    lib.oracle_l2norm_rows.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_double, dp, dp]
    lib.oracle_l2norm_rows.restype = ctypes.c_int
    lib.oracle_sigmoid.argtypes = [ctypes.c_int64, dp, dp]
    lib.oracle_sigmoid.restype = ctypes.c_int
    lib.oracle_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_double, dp, dp, dp, dp]
    lib.oracle_gated_rmsnorm.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route calls to another build of the oracle source (used by
    the mutation tests, which compile deliberately broken copies)."""
    global _lib
    with _lock:
        saved, _lib = _lib, _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x), dtype=np.float64)


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def gdr_sequential(
    cu_seqlens,
    q,
    k,
    v,
    g,
    beta,
    state0,
    scale: float = 1.0,
    threads: Optional[int] = None,
) -> Tuple[np.ndarray, np.ndarray]:
    """Run the recurrence over packed sequences.

    Shapes: q, k [T, H_qk, d_k]; v [T, H_v, d_v]; g, beta [T, H_v];
    state0 [n, H_v, d_k, d_v]; cu_seqlens [n+1].  Returns (o [T, H_v, d_v],
    final state [n, H_v, d_k, d_v]), both float64.
    """
    cu = np.ascontiguousarray(np.asarray(cu_seqlens), dtype=np.int64)
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    state = _f64(state0).copy()
    n = cu.shape[0] - 1
    t = int(cu[-1]) if n > 0 else 0
    h_qk, d_k = q.shape[1], q.shape[2]
    h_v, d_v = v.shape[1], v.shape[2]
    assert k.shape == q.shape and g.shape == (v.shape[0], h_v) and beta.shape == g.shape
    assert state.shape == (n, h_v, d_k, d_v), (state.shape, (n, h_v, d_k, d_v))
    assert v.shape[0] >= t
    o = np.zeros((v.shape[0], h_v, d_v), dtype=np.float64)
    rc = _load().oracle_gdr_sequential(
        n, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), h_qk, h_v, d_k, d_v,
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(state), _ptr(o),
        int(threads if threads is not None else default_threads()),
    )
    if rc != 0:
        raise ValueError("oracle_gdr_sequential rejected its arguments")
    return o, state


def run_workload(w, threads: Optional[int] = None, scale: float = 1.0):
    """The oracle on a ``synth.Workload`` (its exact input values widened to fp64)."""
    return gdr_sequential(w.cu_seqlens, w.q, w.k, w.v, w.g, w.beta, w.state0, scale, threads)


# --- steps on either side of the rule (row-wise, fp64) ------------------------------

L2NORM_EPS = 1e-6   # reading: inside the square root (the pages give no eps for it)
RMSNORM_EPS = 1e-6  # the norm epsilon named in the Candle PR's bug log ("Bug 7")


def l2norm_rows(x, eps: float = L2NORM_EPS) -> np.ndarray:
    """x / sqrt(sum x^2 + eps) over the last axis."""
    a = _f64(x)
    d = a.shape[-1]
    y = np.empty_like(a)
    if _load().oracle_l2norm_rows(a.size // d, d, float(eps), _ptr(a), _ptr(y)) != 0:
        raise ValueError("oracle_l2norm_rows rejected its arguments")
    return y


def sigmoid(b) -> np.ndarray:
    a = _f64(b)
    y = np.empty_like(a)
    if _load().oracle_sigmoid(a.size, _ptr(a), _ptr(y)) != 0:
        raise ValueError("oracle_sigmoid rejected its arguments")
    return y


def gated_rmsnorm(o, z, w, eps: float = RMSNORM_EPS) -> np.ndarray:
    """w * o / sqrt(mean(o^2) + eps) * silu(z) over the last axis (w: one weight per channel)."""
    a, zz, ww = _f64(o), _f64(z), _f64(w)
    d = a.shape[-1]
    assert zz.shape == a.shape and ww.shape == (d,)
    y = np.empty_like(a)
    if _load().oracle_gated_rmsnorm(a.size // d, d, float(eps), _ptr(a), _ptr(zz), _ptr(ww), _ptr(y)) != 0:
        raise ValueError("oracle_gated_rmsnorm rejected its arguments")
    return y


def gdr_fused(cu_seqlens, q_raw, k_raw, v, g, beta_or_logits, state0, *, qk_l2norm: bool, beta_logits: bool,
              z=None, norm_weight=None, scale: float = 1.0, threads: Optional[int] = None):
    """The rule with its steps on either side, in order: q and k L2-normalised
    (when qk_l2norm), beta = sigmoid(logit) (when beta_logits), the recurrence,
    then (when z is given) the gated RMSNorm of every output row.  Returns
    (o or y, final state)."""
    q = l2norm_rows(q_raw) if qk_l2norm else _f64(q_raw)
    k = l2norm_rows(k_raw) if qk_l2norm else _f64(k_raw)
    beta = sigmoid(beta_or_logits) if beta_logits else _f64(beta_or_logits)
    o, s = gdr_sequential(cu_seqlens, q, k, v, g, beta, state0, scale, threads)
    if z is not None:
        o = gated_rmsnorm(o, z, norm_weight)
    return o, s
