"""Thin Python binding over libkda's C ABI (``include/kda.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libkda.  Tensors are PyTorch CUDA tensors (PyTorch provides device
memory and streams); results are written into caller-provided or freshly
allocated tensors.  If the library has not been built this module raises --
there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

_lib = None

KDA_F32, KDA_BF16 = 0, 1
_DTYPES = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported size or chunk",
          -3: "pointer not 16-byte aligned", -4: "CUDA error", -5: "out of device memory",
          -6: "a kernel gave up on a bounded wait"}


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libkda (raises if it was not built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libkda is not built ({path} missing): run "
                               "gated_delta_rule_26_gb300.build.build() first")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        dp = ctypes.POINTER(Dims)
        lib.kda_gate.argtypes = [dp, i, vp, vp, vp, i, vp, vp]
        lib.kda_chunk_forward.argtypes = [dp, i, vp, vp, vp, vp, vp, vp, vp, f, vp, i, vp, vp, vp]
        lib.kda_chunk_forward_split.argtypes = lib.kda_chunk_forward.argtypes
        lib.kda_chunk_forward_fused.argtypes = lib.kda_chunk_forward.argtypes
        lib.kda_chunk_forward_split_noalloc.argtypes = lib.kda_chunk_forward.argtypes
        lib.kda_chunk_forward_scan.argtypes = lib.kda_chunk_forward.argtypes
        lib.kda_recurrent_step.argtypes = [dp, i, vp, vp, vp, vp, vp, vp, vp, f, vp, vp, vp]
        lib.kda_fused_recurrent.argtypes = [dp, i, vp, vp, vp, vp, vp, vp, vp, f, vp, vp, vp]
        lib.kda_chunk_backward.argtypes = [dp, i] + [vp] * 7 + [f] + [vp] * 12
        lib.kda_status_string.argtypes = [i]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_device_status.argtypes = [vp]
        lib.kda_device_status.restype = i
        lib.kda_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
        lib.kda_selftest_bounded_wait.restype = i
        lib.kda_launch_count.argtypes = []
        lib.kda_launch_count.restype = ctypes.c_ulonglong
        lib.kda_release_scratch.argtypes = []
        lib.kda_release_scratch.restype = i
        for fn in (lib.kda_gate, lib.kda_chunk_forward, lib.kda_recurrent_step,
                   lib.kda_fused_recurrent, lib.kda_chunk_backward):
            fn.restype = i
        _lib = lib
    return _lib


def device_status(stream=None) -> int:
    """Drain the stream and return (and clear) the library's bounded-wait timeout report:
    0 when no kernel gave up on a wait, -6 (KDA_ERR_TIMEOUT) otherwise."""
    return int(load().kda_device_status(_stream(stream)))


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch a kernel whose wait can never be satisfied; it ends after `limit_ns`."""
    _check("kda_selftest_bounded_wait", load().kda_selftest_bounded_wait(int(limit_ns),
                                                                          _stream(stream)))


def release_scratch() -> None:
    """Hand the blocks the library's scratch pool keeps for later calls back to the system."""
    _check("kda_release_scratch", load().kda_release_scratch())


def launch_count() -> int:
    """Kernels launched by libkda in this process so far."""
    return int(load().kda_launch_count())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkda takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise KdaError(fn, status)


def _f32(t):
    return None if t is None else t.to(torch.float32).contiguous()


def default_scale(K: int) -> float:
    """The read scale used when none is given: K ** -0.5."""
    return float(K) ** -0.5


def gate(z: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor, chunk: int = 0,
         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """g (chunk = 0) or the in-chunk cumulative log decay G, float32, shape of z (B, H, T, K)."""
    B, H, T, K = z.shape
    if out is None:
        out = torch.empty(B, H, T, K, device=z.device, dtype=torch.float32)
    d = Dims(B, H, T, K, K)
    st = load().kda_gate(ctypes.byref(d), _DTYPES[z.dtype], _ptr(z), _ptr(_f32(A_log)),
                         _ptr(_f32(dt_bias)), int(chunk), _ptr(out), _stream(stream))
    _check("kda_gate", st)
    return out


_CHUNK_FORMS = {"auto": "kda_chunk_forward", "split": "kda_chunk_forward_split",
                "fused": "kda_chunk_forward_fused",
                # the split form with the chunk-parallel state scan
                "scan": "kda_chunk_forward_scan",
                # the split form on the library's fixed scratch array (no allocation)
                "split_noalloc": "kda_chunk_forward_split_noalloc"}


def chunk_forward(q, k, v, z, beta, A_log, dt_bias, scale: Optional[float] = None,
                  h0: Optional[torch.Tensor] = None, chunk: int = 64,
                  out: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                  output_final_state: bool = True, stream=None, form: str = "auto"
                  ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KDA forward over (B, H, T) tokens; returns (o, hT) with o in q's dtype, hT float32.

    ``form`` selects the entry point: "auto" (kda_chunk_forward, which picks the faster
    form), "split" (kda_chunk_forward_split), "fused" (kda_chunk_forward_fused), "scan"
    (kda_chunk_forward_scan: the split form with the chunk-parallel state scan) or
    "split_noalloc" (kda_chunk_forward_split_noalloc: the split form without any device
    allocation, for B*H up to the limit its header comment states)."""
    fn = _CHUNK_FORMS[form]
    B, H, T, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = default_scale(K)
    if out is None:
        out = torch.empty(B, H, T, V, device=q.device, dtype=q.dtype)
    if hT is None and output_final_state:
        hT = torch.empty(B, H, K, V, device=q.device, dtype=torch.float32)
    d = Dims(B, H, T, K, V)
    A32, dt32 = _f32(A_log), _f32(dt_bias)
    st = getattr(load(), fn)(ctypes.byref(d), _DTYPES[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                             _ptr(z), _ptr(beta), _ptr(A32), _ptr(dt32), float(scale),
                             _ptr(h0), int(chunk), _ptr(out), _ptr(hT), _stream(stream))
    _check(fn, st)
    return out, hT


def recurrent_step(q, k, v, z, beta, A_log, dt_bias, state: torch.Tensor,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """One decode token per (b, h): updates ``state`` (B, H, K, V) float32 in place and returns o
    of shape (B, H, 1, V).  q, k, z are (B, H, 1, K), v (B, H, 1, V), beta (B, H, 1)."""
    B, H, _, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = default_scale(K)
    if out is None:
        out = torch.empty(B, H, 1, V, device=q.device, dtype=q.dtype)
    d = Dims(B, H, 1, K, V)
    st = load().kda_recurrent_step(ctypes.byref(d), _DTYPES[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(z), _ptr(beta), _ptr(_f32(A_log)), _ptr(_f32(dt_bias)),
                                   float(scale), _ptr(state), _ptr(out), _stream(stream))
    _check("kda_recurrent_step", st)
    return out


def fused_recurrent(q, k, v, z, beta, A_log, dt_bias, state: torch.Tensor,
                    scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """T tokens per (b, h) applied one by one with the state kept on chip; updates ``state``
    (B, H, K, V) float32 in place and returns o (B, H, T, V).  q, k, z are (B, H, T, K),
    v (B, H, T, V), beta (B, H, T)."""
    B, H, T, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = default_scale(K)
    if out is None:
        out = torch.empty(B, H, T, V, device=q.device, dtype=q.dtype)
    d = Dims(B, H, T, K, V)
    st = load().kda_fused_recurrent(ctypes.byref(d), _DTYPES[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(z), _ptr(beta), _ptr(_f32(A_log)), _ptr(_f32(dt_bias)),
                                    float(scale), _ptr(state), _ptr(out), _stream(stream))
    _check("kda_fused_recurrent", st)
    return out


def chunk_backward(q, k, v, z, beta, A_log, dt_bias, d_o, scale: Optional[float] = None,
                   h0: Optional[torch.Tensor] = None, dhT: Optional[torch.Tensor] = None,
                   want_dh0: bool = True, stream=None) -> dict:
    """Gradients of the chunked forward's inputs from d_o = dL/do and dhT = dL/dhT, to float32
    accuracy (kda_chunk_backward).

    Returns float32 tensors: dq, dk, dz (B, H, T, K), dv (B, H, T, V), dbeta (B, H, T),
    dA_log (H), ddt_bias (H, K) and dh0 (B, H, K, V) (None unless ``want_dh0``)."""
    B, H, T, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = default_scale(K)
    dev, f32 = q.device, torch.float32
    g = {"dq": torch.empty(B, H, T, K, device=dev, dtype=f32),
         "dk": torch.empty(B, H, T, K, device=dev, dtype=f32),
         "dv": torch.empty(B, H, T, V, device=dev, dtype=f32),
         "dz": torch.empty(B, H, T, K, device=dev, dtype=f32),
         "dbeta": torch.empty(B, H, T, device=dev, dtype=f32),
         "dA_log": torch.empty(H, device=dev, dtype=f32),
         "ddt_bias": torch.empty(H, K, device=dev, dtype=f32),
         "dh0": torch.empty(B, H, K, V, device=dev, dtype=f32) if want_dh0 else None}
    d = Dims(B, H, T, K, V)
    st = load().kda_chunk_backward(
        ctypes.byref(d), _DTYPES[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta),
        _ptr(_f32(A_log)), _ptr(_f32(dt_bias)), float(scale), _ptr(h0), _ptr(d_o), _ptr(dhT),
        _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dz"]), _ptr(g["dbeta"]),
        _ptr(g["dA_log"]), _ptr(g["ddt_bias"]), _ptr(g["dh0"]), _stream(stream))
    _check("kda_chunk_backward", st)
    return g
