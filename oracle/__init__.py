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
* ``backward``   -- the gradients of ``forward``'s outputs' adjoints with respect to
  every input, by reverse-mode differentiation of the same steps token by token
  (kda-adjoint-2026-10-01: the backward and its gradients dq, dk, dv, dg, dbeta and
  the state gradient).  Pinned by ``jvp`` below and by central differences.
* ``jvp``        -- forward-mode derivative (tangent propagation) of the same forward,
  written separately in numpy: the directional derivative of <d_o, o> + <dhT, hT>.
* ``chunked_backward.chunked_backward`` -- the backward organised as chunk-level adjoint
  equations (the form the GPU kernel takes), checked against ``backward`` in the tests.
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
            lib.kda_oracle_backward_range.argtypes = [i, i, i, i, i] + [_D] * 7 + [
                ctypes.c_double] + [_D] * 12 + [i, i, i]
            lib.kda_oracle_backward_range.restype = None
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


def backward(q, k, v, z, beta, A_log, dt_bias, scale, h0, d_o, dhT=None, threads: int = 1,
             mutant: int = 0) -> dict:
    """Gradients of L (with dL/do = d_o and dL/dhT = dhT) with respect to every input.

    Returns float64 arrays: dq, dk, dz, dg (B,H,T,K; dg is the gradient with respect to the log
    decay g), dv (B,H,T,V), dbeta (B,H,T), dA_log (H), ddt_bias (H,K) and dh0 (B,H,K,V) (the
    gradient with respect to the initial state, a zero state when h0 is None).  `mutant`
    plants a known mistake (tests only).
    """
    q, k, v, z, beta, A_log, dt_bias, h0, d_o, dhT = (
        f64(a) for a in (q, k, v, z, beta, A_log, dt_bias, h0, d_o, dhT))
    B, H, T, K, V = _dims(q, v)
    assert k.shape == q.shape and z.shape == q.shape and beta.shape == (B, H, T)
    assert A_log.shape == (H,) and dt_bias.shape == (H, K) and d_o.shape == v.shape
    for s_ in (h0, dhT):
        assert s_ is None or s_.shape == (B, H, K, V)
    out = {n: np.zeros(q.shape) for n in ("dq", "dk", "dz", "dg")}
    out["dv"] = np.zeros(v.shape)
    out["dbeta"] = np.zeros((B, H, T))
    out["dh0"] = np.zeros((B, H, K, V))
    dA_part = np.zeros((B, H))
    ddt_part = np.zeros((B, H, K))
    lib = _load()

    def run(r):
        lib.kda_oracle_backward_range(
            B, H, T, K, V, _p(q), _p(k), _p(v), _p(z), _p(beta), _p(A_log), _p(dt_bias),
            float(scale), _p(h0), _p(d_o), _p(dhT), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
            _p(out["dz"]), _p(out["dg"]), _p(out["dbeta"]), _p(dA_part), _p(ddt_part),
            _p(out["dh0"]),
            int(mutant), r[0], r[1])

    _run_ranges(run, B * H, threads)
    out["dA_log"] = dA_part.sum(axis=0)
    out["ddt_bias"] = ddt_part.sum(axis=0)
    return out


def jvp(q, k, v, z, beta, A_log, dt_bias, scale, h0, d_o, dhT, tangents: dict) -> float:
    """Directional derivative of <d_o, o> + <dhT, hT> along `tangents` (forward mode).

    `tangents` maps input names (q, k, v, z, beta, A_log, dt_bias, h0) to arrays of the
    inputs' shapes (missing = 0).  Every forward step is carried as a (value, tangent) pair
    with the product rule; this shares nothing with ``backward``.
    """
    q, k, v, z, beta, A_log, dt_bias, h0, d_o, dhT = (
        f64(a) for a in (q, k, v, z, beta, A_log, dt_bias, h0, d_o, dhT))
    B, H, T, K, V = _dims(q, v)
    tg = {n: (np.zeros_like(x) if tangents.get(n) is None else f64(tangents[n]))
          for n, x in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta),
                       ("A_log", A_log), ("dt_bias", dt_bias))}
    S = np.zeros((B, H, K, V)) if h0 is None else h0.copy()
    dS_ = np.zeros((B, H, K, V)) if tangents.get("h0") is None else f64(tangents["h0"]).copy()
    x = z + dt_bias[None, :, None, :]
    dx = tg["z"] + tg["dt_bias"][None, :, None, :]
    sp = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    sig = np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))), np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))
    m = np.exp(A_log)[None, :, None, None]
    dm = (np.exp(A_log) * tg["A_log"])[None, :, None, None]
    g = -m * sp
    dg = -dm * sp - m * sig * dx
    a = np.exp(g)
    da = a * dg
    total = 0.0
    for t in range(T):
        at, dat = a[:, :, t, :, None], da[:, :, t, :, None]
        kt, dkt = k[:, :, t], tg["k"][:, :, t]
        Sd = at * S
        dSd = dat * S + at * dS_
        u = v[:, :, t] - np.einsum("bhcj,bhc->bhj", Sd, kt)
        du = tg["v"][:, :, t] - np.einsum("bhcj,bhc->bhj", dSd, kt) - np.einsum("bhcj,bhc->bhj", Sd, dkt)
        bt, dbt = beta[:, :, t, None, None], tg["beta"][:, :, t, None, None]
        S = Sd + bt * kt[..., None] * u[:, :, None, :]
        dS_ = (dSd + dbt * kt[..., None] * u[:, :, None, :] + bt * dkt[..., None] * u[:, :, None, :]
               + bt * kt[..., None] * du[:, :, None, :])
        do_t = scale * (np.einsum("bhcj,bhc->bhj", dS_, q[:, :, t])
                        + np.einsum("bhcj,bhc->bhj", S, tg["q"][:, :, t]))
        total += float(np.sum(d_o[:, :, t] * do_t))
    if dhT is not None:
        total += float(np.sum(dhT * dS_))
    return total
