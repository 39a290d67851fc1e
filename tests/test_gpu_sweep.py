"""Breadth sweeps on the GPU: many small seeded configurations (shapes, chunk sizes, dtypes,
gate strengths, initial states, empty and one-token sequences) through the C ABI, each
compared with the f64 oracle at the bars of the fixed-case parity tests:

* forward, fp32 I/O: max|x - y| / max|y| <= 1e-4 per tensor;
* forward, bf16 I/O: ||x - y||_2 / ||y||_2 <= 2e-2 and max|x - y| <= 5e-2;
* backward (fp32 accuracy for either I/O dtype): max|x - y| / max|y| <= 1e-4 per gradient,
  and for the batch sums dA_log and ddt_bias max|x - y| <= 1e-4 max sum|terms| (the bar of
  tests/test_gpu_backward.py, which states why).

The configurations come from one seeded generator, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_26_gb300 import inputs
from test_gpu_backward import reduced_scales

pytestmark = pytest.mark.gpu

FP32_BAR = 1e-4
BF16_REL, BF16_ABS = 2e-2, 5e-2


def _errors(got, ref, dtype):
    got = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    if ref.size == 0:
        return None
    if not np.all(np.isfinite(got)):
        return "non-finite"
    diff = np.abs(got - ref)
    if dtype == "f32":
        err = diff.max() / max(np.abs(ref).max(), 1e-30)
        return None if err <= FP32_BAR else f"max rel {err:.3e}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    return None if (rel <= BF16_REL and diff.max() <= BF16_ABS) else f"rel {rel:.3e} max {diff.max():.3e}"


def _case(rng):
    dims = [8 * int(x) for x in rng.integers(1, 17, size=2)]
    return dict(B=int(rng.integers(1, 3)), H=int(rng.integers(1, 4)),
                T=int(rng.choice([0, 1, int(rng.integers(2, 200))], p=[0.04, 0.06, 0.9])),
                K=dims[0], V=dims[1], chunk=int(rng.choice([16, 32, 64])),
                dtype=str(rng.choice(["f32", "bf16"])), seed=int(rng.integers(0, 1 << 30)),
                h0_std=float(rng.choice([0.0, 0.1, 0.5])), dt_std=float(rng.choice([0.0, 0.3])),
                A_log_value=float(rng.uniform(-3.0, 2.8)))


def test_forward_breadth_sweep(kda):
    rng = np.random.default_rng(2024)
    failures = []
    for n in range(160):
        c = _case(rng)
        # every fourth case takes the tensor-core shape (bf16, K = V = 128, chunk 64)
        if n % 4 == 0:
            c.update(K=128, V=128, chunk=64, dtype="bf16")
        inp = inputs.make(c["B"], c["H"], c["T"], c["K"], c["V"], chunk=c["chunk"],
                          dtype=c["dtype"], seed=c["seed"], dt_std=c["dt_std"],
                          h0_std=c["h0_std"], A_log_value=c["A_log_value"])
        d = inp.to("cuda")
        o, hT = kda.chunk_forward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp.scale,
                                  d.h0, c["chunk"])
        torch.cuda.synchronize()
        o_ref, h_ref = oracle.forward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log,
                                      inp.dt_bias, inp.scale, inp.h0, threads=4)
        for name, got, ref in (("o", o, o_ref), ("hT", hT, h_ref)):
            e = _errors(got, ref, c["dtype"])
            if e:
                failures.append((n, name, e, c))
    assert kda.device_status() == 0
    assert not failures, failures[:5]


def test_backward_breadth_sweep(kda):
    rng = np.random.default_rng(4048)
    failures = []
    for n in range(60):
        c = _case(rng)
        c["T"] = min(c["T"], 120)
        if n % 3 == 2:  # every third case takes the tensor-core form (K = V = 128)
            c.update(K=128, V=128)
        inp = inputs.make(c["B"], c["H"], c["T"], c["K"], c["V"], dtype=c["dtype"],
                          seed=c["seed"], dt_std=c["dt_std"], h0_std=c["h0_std"],
                          A_log_value=c["A_log_value"])
        adj = inputs.adjoints(inp, seed=c["seed"] + 1, with_dhT=bool(n % 3))
        d = inp.to("cuda")
        g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias,
                               adj.d_o.to("cuda"), inp.scale, h0=d.h0,
                               dhT=None if adj.dhT is None else adj.dhT.to("cuda"))
        torch.cuda.synchronize()
        ref = oracle.backward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log, inp.dt_bias,
                              inp.scale, inp.h0, adj.d_o, adj.dhT, threads=4)
        for name in ("dq", "dk", "dv", "dz", "dbeta", "dh0"):
            e = _errors(g[name], ref[name], "f32")
            if e:
                failures.append((n, name, e, c))
        for name, scale in reduced_scales(inp, ref).items():
            got = g[name].double().cpu().numpy()
            err = np.abs(got - ref[name]).max() / max(np.max(scale), 1e-30) if got.size else 0.0
            if not np.isfinite(err) or err > FP32_BAR:
                failures.append((n, name, f"{err:.3e} of sum|terms|", c))
    assert kda.device_status() == 0
    assert not failures, failures[:5]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_size_sweep(kda, dtype):
    """One input through every chunk size: each result within the bar of the oracle."""
    inp = inputs.make(2, 3, 211, 64, 64, dtype=dtype, seed=77, h0_std=0.2, dt_std=0.3)
    d = inp.to("cuda")
    o_ref, h_ref = oracle.forward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log, inp.dt_bias,
                                  inp.scale, inp.h0, threads=4)
    for chunk in (16, 32, 64):
        o, hT = kda.chunk_forward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp.scale,
                                  d.h0, chunk)
        torch.cuda.synchronize()
        for name, got, ref in (("o", o, o_ref), ("hT", hT, h_ref)):
            e = _errors(got, ref, dtype)
            assert e is None, (chunk, name, e)
