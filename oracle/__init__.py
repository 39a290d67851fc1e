"""f64 CPU oracle for the Kimi Delta Attention (KDA) forward.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its Python binding) never does, and shares no code with
it.  Every routine works in float64 and follows the method's statement step
by step:

* ``gate``       -- g = -exp(A_log_h) * softplus(z + dt_bias_h)
  (kdafix-2026-10-02, "Fix 1 -- decay form").
* ``recurrent``  -- token-by-token state update S <- diag(alpha) S,
  u = v - S^T k, S <- S + beta k u^T, o = S^T (scale q)
  (kdafix-2026-10-02, "Fix 2 -- read scale": scale folded into q, read only).
* ``forward``    -- gate + recurrence from raw inputs, threaded over (b, h).
* ``chunked.chunked_wy`` -- an independent f64 chunked (WY) evaluation of the
  same function, used to check that the chunked and recurrent forms agree
  (kda-adjoint-2026-10-01, section 2: carry with decay_last = exp(G_last - G)).

The C routines live in ``kda_oracle.c`` and are built by :func:`build` with
gcc into ``oracle/_build/``.  Inputs may be numpy arrays or CPU torch tensors
of any float dtype; they are widened to float64 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i = ctypes.c_int
            lib.kda_oracle_softplus.argtypes = [ctypes.c_double]
            lib.kda_oracle_softplus.restype = ctypes.c_double
            lib.kda_oracle_gate.argtypes = [i, i, i, i, _D, _D, _D, _D]
            lib.kda_oracle_gate.restype = None
            lib.kda_oracle_recurrent_range.argtypes = [i, i, i, i, i, _D, _D, _D, _D, _D,
                                                       ctypes.c_double, _D, _D, _D, i, i]
            lib.kda_oracle_recurrent_range.restype = None
            lib.kda_oracle_forward_range.argtypes = [i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D,
                                                     ctypes.c_double, _D, _D, _D, i, i]
            lib.kda_oracle_forward_range.restype = None
            _lib = lib
    return _lib


def f64(x) -> np.ndarray:
    """Widen a numpy array or CPU torch tensor to a contiguous float64 array (exact)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def softplus(x: float) -> float:
    return _load().kda_oracle_softplus(float(x))


def gate(z, A_log, dt_bias) -> np.ndarray:
    """g = -exp(A_log[h]) * softplus(z + dt_bias[h, :]) for z of shape (B, H, T, K)."""
    z, A_log, dt_bias = f64(z), f64(A_log), f64(dt_bias)
    B, H, T, K = z.shape
    assert A_log.shape == (H,) and dt_bias.shape == (H, K)
    g = np.empty_like(z)
    _load().kda_oracle_gate(B, H, T, K, _p(z), _p(A_log), _p(dt_bias), _p(g))
    return g


def _dims(q, v):
    B, H, T, K = q.shape
    V = v.shape[-1]
    assert v.shape == (B, H, T, V)
    return B, H, T, K, V


def _split(n, parts):
    parts = max(1, min(parts, n))
    edges = [round(i * n / parts) for i in range(parts + 1)]
    return [(edges[i], edges[i + 1]) for i in range(parts) if edges[i + 1] > edges[i]]


def recurrent(q, k, v, g, beta, scale, h0=None, threads: int = 1):
    """Token-by-token recurrence given the log decay g. Returns (o, hT) in float64."""
    q, k, v, g, beta, h0 = (f64(a) for a in (q, k, v, g, beta, h0))
    B, H, T, K, V = _dims(q, v)
    assert k.shape == q.shape and g.shape == q.shape and beta.shape == (B, H, T)
    if h0 is not None:
        assert h0.shape == (B, H, K, V)
    o = np.zeros((B, H, T, V))
    hT = np.zeros((B, H, K, V))
    lib = _load()

    def run(r):
        lib.kda_oracle_recurrent_range(B, H, T, K, V, _p(q), _p(k), _p(v), _p(g), _p(beta),
                                       float(scale), _p(h0), _p(o), _p(hT), r[0], r[1])

    _run_ranges(run, B * H, threads)
    return o, hT


def forward(q, k, v, z, beta, A_log, dt_bias, scale, h0=None, threads: int = 1):
    """Gate + recurrence from raw inputs. Returns (o, hT) in float64."""
    q, k, v, z, beta, A_log, dt_bias, h0 = (f64(a) for a in (q, k, v, z, beta, A_log, dt_bias, h0))
    B, H, T, K, V = _dims(q, v)
    assert k.shape == q.shape and z.shape == q.shape and beta.shape == (B, H, T)
    assert A_log.shape == (H,) and dt_bias.shape == (H, K)
    if h0 is not None:
        assert h0.shape == (B, H, K, V)
    o = np.zeros((B, H, T, V))
    hT = np.zeros((B, H, K, V))
    lib = _load()

    def run(r):
        lib.kda_oracle_forward_range(B, H, T, K, V, _p(q), _p(k), _p(v), _p(z), _p(beta),
                                     _p(A_log), _p(dt_bias), float(scale), _p(h0), _p(o), _p(hT),
                                     r[0], r[1])

    _run_ranges(run, B * H, threads)
    return o, hT


def _run_ranges(fn, n, threads):
    # ctypes releases the GIL for the duration of each C call, so a thread pool
    # over disjoint (b, h) ranges runs the plain C loop on several cores.
    ranges = _split(n, threads)
    if len(ranges) == 1:
        fn(ranges[0])
        return
    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        list(ex.map(fn, ranges))
