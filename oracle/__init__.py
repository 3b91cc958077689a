"""fp64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The library's compute path never does: it has
no CPU fallback.

The arithmetic lives in ``gdr_oracle.c`` (plain C, fp64, one token at a time,
in the order of the per-token Loop on the Qwen3.5-9B NPU model card, section
"How it works").  This module compiles it with gcc on first use and marshals
numpy arrays to it; it adds no arithmetic of its own.
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
