"""Seeded synthetic inputs for the KDA forward and decode step.

This module holds only the input recipe (random draws, the L2 normalisation of
q and k, the sigmoid that maps a normal draw to beta); none of the method's
arithmetic.  The tests, the bench and the smoke check build inputs here and
hand the same tensors to both the CUDA library and the CPU oracle.

Recipe (Kimi-Linear-shaped synthetic inputs; all draws from a CPU
``torch.Generator`` in float32, then cast to the I/O dtype):

* q, k ~ N(0, 1), then L2-normalised over the key dimension K;
* v ~ N(0, 1);  z ~ N(0, 1);  beta = sigmoid(N(0, 1));
* dt_bias ~ N(0, dt_std^2) of shape (H, K) (0 when dt_std = 0);
* A_log per head ~ U[log 1, log 16] unless fixed explicitly;
* h0 ~ N(0, h0_std^2) in float32 (None when h0_std = 0);
* scale = K ** -0.5 (the default read scale).

Named workloads:

* ``small_fp32``   B1 H2 T32 K=V=8 chunk 16, fp32, dt_bias 0, h0 std 0.1,
  A_log fixed per run to one of {-3, 0, +2} (``A_log_value``) or a z sweep;
* ``multi_chunk_fp32``  B2 H8 T256 K=V=64 chunk 16, fp32, dt_bias std 0.1;
* ``prefill_bf16`` B8 H32 T4096 K=V=128 chunk 64, bf16 I/O, fp32 state, h0 = 0;
* ``long_bf16``    B1 H32 T65536 K=V=128 chunk 64, bf16 I/O, h0 std 0.1;
* ``decode_bf16``  B256 H32 K=V=128, one token per step, 64 steps, fp32 state
  std 0.1, bf16 q/k/v/z/beta.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

WORKLOADS = {
    "small_fp32": dict(B=1, H=2, T=32, K=8, V=8, chunk=16, dtype="f32", dt_std=0.0, h0_std=0.1),
    "multi_chunk_fp32": dict(B=2, H=8, T=256, K=64, V=64, chunk=16, dtype="f32", dt_std=0.1,
                             h0_std=0.0),
    "prefill_bf16": dict(B=8, H=32, T=4096, K=128, V=128, chunk=64, dtype="bf16", dt_std=0.1,
                         h0_std=0.0),
    "long_bf16": dict(B=1, H=32, T=65536, K=128, V=128, chunk=64, dtype="bf16", dt_std=0.1,
                      h0_std=0.1),
}
DECODE = dict(B=256, H=32, K=128, V=128, steps=64, dtype="bf16", dt_std=0.1, h0_std=0.1)
SEEDS = {"small_fp32": 1001, "multi_chunk_fp32": 1002, "prefill_bf16": 1003, "long_bf16": 1004,
         "decode_bf16": 1005}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class KdaInputs:
    B: int
    H: int
    T: int
    K: int
    V: int
    chunk: int
    dtype: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    z: torch.Tensor
    beta: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    h0: Optional[torch.Tensor]
    scale: float
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "KdaInputs":
        mv = lambda t: None if t is None else t.to(device, non_blocking=False).contiguous()
        return KdaInputs(self.B, self.H, self.T, self.K, self.V, self.chunk, self.dtype,
                         mv(self.q), mv(self.k), mv(self.v), mv(self.z), mv(self.beta),
                         mv(self.A_log), mv(self.dt_bias), mv(self.h0), self.scale, self.extra)


def _l2norm(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)


def make(B, H, T, K, V, *, chunk=16, dtype="f32", seed=0, dt_std=0.1, h0_std=0.0,
         A_log=None, A_log_value=None, z_sweep=None, scale=None) -> KdaInputs:
    """Draw one seeded input set.  ``A_log`` may be given as a sequence (one value per head);
    ``A_log_value`` fixes every head to one value; ``z_sweep=(lo, hi)`` replaces z by a linear
    sweep over (t, c) shared by all (b, h)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    f = torch.float32
    q = _l2norm(torch.randn(B, H, T, K, generator=gen, dtype=f))
    k = _l2norm(torch.randn(B, H, T, K, generator=gen, dtype=f))
    v = torch.randn(B, H, T, V, generator=gen, dtype=f)
    z = torch.randn(B, H, T, K, generator=gen, dtype=f)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=gen, dtype=f))
    if dt_std > 0:
        dt_bias = torch.randn(H, K, generator=gen, dtype=f) * dt_std
    else:
        dt_bias = torch.zeros(H, K, dtype=f)
    a_draw = torch.rand(H, generator=gen, dtype=f) * math.log(16.0)
    if A_log is not None:
        a = torch.tensor(list(A_log), dtype=f)
    elif A_log_value is not None:
        a = torch.full((H,), float(A_log_value), dtype=f)
    else:
        a = a_draw
    h0 = None
    if h0_std > 0:
        h0 = torch.randn(B, H, K, V, generator=gen, dtype=f) * h0_std
    if z_sweep is not None:
        lo, hi = z_sweep
        z = torch.linspace(lo, hi, T * K, dtype=f).reshape(1, 1, T, K).expand(B, H, T, K).clone()
    td = _TORCH_DTYPE[dtype]
    return KdaInputs(B, H, T, K, V, chunk, dtype, q.to(td), k.to(td), v.to(td), z.to(td),
                     beta.to(td), a, dt_bias, h0, float(K ** -0.5 if scale is None else scale))


@dataclass
class Adjoints:
    d_o: torch.Tensor               # (B, H, T, V) in the inputs' I/O dtype
    dhT: Optional[torch.Tensor]     # (B, H, K, V) float32


def adjoints(inp: KdaInputs, seed: int, with_dhT: bool = True, dhT_std: float = 1.0) -> Adjoints:
    """Seeded gradients of a loss with respect to o and hT (standard normal draws), the
    inputs of a backward pass: d_o in the I/O dtype, dhT in float32."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    f = torch.float32
    d_o = torch.randn(inp.B, inp.H, inp.T, inp.V, generator=gen, dtype=f)
    dhT = torch.randn(inp.B, inp.H, inp.K, inp.V, generator=gen, dtype=f) * dhT_std
    return Adjoints(d_o.to(_TORCH_DTYPE[inp.dtype]), dhT if with_dhT else None)


def workload(name: str, **overrides) -> KdaInputs:
    """The named workload with its fixed seed; keyword overrides replace recipe fields."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    seed = cfg.pop("seed", SEEDS[name])
    return make(seed=seed, **cfg)


@dataclass
class DecodeInputs:
    B: int
    H: int
    K: int
    V: int
    steps: int
    dtype: str
    q: torch.Tensor       # (steps, B, H, 1, K)
    k: torch.Tensor       # (steps, B, H, 1, K)
    v: torch.Tensor       # (steps, B, H, 1, V)
    z: torch.Tensor       # (steps, B, H, 1, K)
    beta: torch.Tensor    # (steps, B, H, 1)
    A_log: torch.Tensor   # (H,)
    dt_bias: torch.Tensor  # (H, K)
    state: torch.Tensor   # (B, H, K, V) float32
    scale: float


def decode(B=None, H=None, K=None, V=None, steps=None, seed=None, dtype=None) -> DecodeInputs:
    """Inputs for ``steps`` consecutive single-token decode steps (default: decode_bf16)."""
    cfg = dict(DECODE)
    for key, val in dict(B=B, H=H, K=K, V=V, steps=steps, dtype=dtype).items():
        if val is not None:
            cfg[key] = val
    B, H, K, V, S_, dt = cfg["B"], cfg["H"], cfg["K"], cfg["V"], cfg["steps"], cfg["dtype"]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(SEEDS["decode_bf16"] if seed is None else seed))
    f = torch.float32
    state = torch.randn(B, H, K, V, generator=gen, dtype=f) * cfg["h0_std"]
    q = _l2norm(torch.randn(S_, B, H, 1, K, generator=gen, dtype=f))
    k = _l2norm(torch.randn(S_, B, H, 1, K, generator=gen, dtype=f))
    v = torch.randn(S_, B, H, 1, V, generator=gen, dtype=f)
    z = torch.randn(S_, B, H, 1, K, generator=gen, dtype=f)
    beta = torch.sigmoid(torch.randn(S_, B, H, 1, generator=gen, dtype=f))
    dt_bias = torch.randn(H, K, generator=gen, dtype=f) * cfg["dt_std"]
    A_log = torch.rand(H, generator=gen, dtype=f) * math.log(16.0)
    td = _TORCH_DTYPE[dt]
    return DecodeInputs(B, H, K, V, S_, dt, q.to(td), k.to(td), v.to(td), z.to(td), beta.to(td),
                        A_log, dt_bias, state, float(K ** -0.5))
