"""GPU parity of the backward (kda_chunk_backward, through the C ABI) against the f64 oracle's
reverse-mode gradients, on the same seeded inputs and output adjoints.

Bar: the backward computes to float32 accuracy whatever the I/O dtype (bf16 inputs are read
exactly; for K = V = 128 its state products are tensor-core products of bf16 hi/lo operand
halves, each within about 2^-15 of its exact value, the state and its adjoint float32), so
every per-token gradient and dh0 is held to the float32 bar, max|x - y| / max|y| <= 1e-4,
against the oracle evaluated on the identical (rounded) inputs.  dA_log[h] and
ddt_bias[h, c] are sums over the batch and the tokens (and, for dA_log, the channels) whose
terms can cancel by three orders of magnitude; the error of a float32 sum scales with the
sum of the magnitudes of its terms, so for these two the bar is max|x - y| <= 1e-4 max
sum|terms| per tensor (terms dg g and dz, from the oracle; max-normalised as for the other
tensors, so that an element whose terms all vanish is held to the tensor's scale).  Small cases run whole; the full-size
prefill workload runs whole on the GPU and is compared on one head (all 8 sequences, so that
the batch sums dA_log[h] and ddt_bias[h] are complete) that the oracle recomputes.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_26_gb300 import inputs

pytestmark = pytest.mark.gpu

BAR = 1e-4
NAMES = ("dq", "dk", "dv", "dz", "dbeta", "dA_log", "ddt_bias", "dh0")


def check(name, got, ref):
    got = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    if ref.size == 0:
        return
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= BAR, f"{name}: max rel {err:.3e} > {BAR}"


def reduced_scales(inp, ref):
    """sum |dg g| over (b, t, c) per head and sum |dz| over (b, t) per (head, channel)."""
    g = oracle.gate(inp.z, inp.A_log, inp.dt_bias)
    return {"dA_log": np.abs(ref["dg"] * g).sum(axis=(0, 2, 3)),
            "ddt_bias": np.abs(ref["dz"]).sum(axis=(0, 2))}


def check_reduced(name, got, ref, scale):
    got = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), name
    err = np.abs(got - ref).max() / max(np.max(scale), 1e-30) if ref.size else 0.0
    assert err <= BAR, f"{name}: error {err:.3e} of the largest sum of term magnitudes > {BAR}"


def check_all(g, ref, inp):
    scales = reduced_scales(inp, ref)
    for n in NAMES:
        if n in scales:
            check_reduced(n, g[n], ref[n], scales[n])
        else:
            check(n, g[n], ref[n])


def run_bwd(kda, inp, seed, with_dhT=True, threads=8):
    adj = inputs.adjoints(inp, seed=seed, with_dhT=with_dhT)
    d = inp.to("cuda")
    d_o = adj.d_o.to("cuda")
    dhT = adj.dhT.to("cuda") if with_dhT else None
    g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, d_o, inp.scale,
                           h0=d.h0, dhT=dhT)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log, inp.dt_bias,
                          inp.scale, inp.h0, adj.d_o, adj.dhT, threads=threads)
    return g, ref


@pytest.mark.parametrize("B,H,T,K,V,dtype,h0_std,A_log", [
    (1, 2, 32, 8, 8, "f32", 0.1, (-3.0, 2.0)),      # smallest config, two chunks
    (2, 8, 256, 64, 64, "f32", 0.0, None),          # 16 chunks
    (1, 3, 37, 32, 16, "f32", 0.3, None),           # ragged tail
    (1, 2, 1, 16, 8, "f32", 0.3, None),             # one token
    (1, 2, 16, 16, 8, "f32", 0.3, None),            # exactly one chunk
    (1, 2, 17, 16, 8, "f32", 0.3, None),            # one chunk and one token
    (1, 2, 70, 128, 64, "f32", 0.1, None),          # K > V
    (1, 2, 70, 64, 128, "f32", 0.1, None),          # K < V
    (1, 4, 300, 128, 128, "bf16", 0.1, None),       # the tensor-core form, bf16 I/O
    (2, 2, 77, 128, 128, "f32", 0.2, (-3.0, 2.0)),  # the tensor-core form, fp32 I/O, ragged
    (1, 2, 1, 128, 128, "f32", 0.3, None),          # the tensor-core form, one token
    (1, 2, 16, 128, 128, "bf16", 0.0, None),        # the tensor-core form, one chunk, no h0
])
def test_backward_matches_oracle(kda, B, H, T, K, V, dtype, h0_std, A_log):
    inp = inputs.make(B, H, T, K, V, dtype=dtype, seed=100 + T + K, h0_std=h0_std, A_log=A_log)
    g, ref = run_bwd(kda, inp, seed=200 + T)
    check_all(g, ref, inp)


def test_backward_without_final_state_gradient(kda):
    inp = inputs.make(1, 3, 90, 64, 32, dtype="f32", seed=31, h0_std=0.2)
    g, ref = run_bwd(kda, inp, seed=32, with_dhT=False)
    check_all(g, ref, inp)


def test_backward_strong_decay_and_z_sweep(kda):
    # A_log = ln 16 and z over [-6, 6]: per-token decay down to e^{-96}; every pairwise factor
    # is taken as one exponential of a non-positive difference, so nothing overflows
    inp = inputs.make(1, 2, 64, 32, 32, dtype="f32", seed=41, h0_std=0.1,
                      A_log_value=float(np.log(16.0)), z_sweep=(-6.0, 6.0))
    g, ref = run_bwd(kda, inp, seed=42)
    check_all(g, ref, inp)


def test_backward_tensor_core_form_without_dhT_and_strong_decay(kda):
    # K = V = 128 takes the tensor-core form; per-token decay down to e^{-96} and no dL/dhT
    inp = inputs.make(1, 2, 64, 128, 128, dtype="f32", seed=43, h0_std=0.1,
                      A_log_value=float(np.log(16.0)), z_sweep=(-6.0, 6.0))
    g, ref = run_bwd(kda, inp, seed=44, with_dhT=False)
    check_all(g, ref, inp)


@pytest.mark.parametrize("K,V", [(16, 8), (128, 128)])
def test_backward_empty_sequence(kda, K, V):
    inp = inputs.make(2, 3, 0, K, V, dtype="f32", seed=5, h0_std=0.1)
    adj = inputs.adjoints(inp, seed=6)
    d = inp.to("cuda")
    g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, adj.d_o.to("cuda"),
                           inp.scale, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"].cpu(), adj.dhT)
    assert torch.count_nonzero(g["dA_log"]).item() == 0
    assert torch.count_nonzero(g["ddt_bias"]).item() == 0
    assert g["dq"].shape == (2, 3, 0, K) and g["dv"].shape == (2, 3, 0, V)


def test_backward_is_deterministic(kda):
    inp = inputs.make(2, 4, 100, 128, 128, dtype="bf16", seed=51, h0_std=0.1)
    adj = inputs.adjoints(inp, seed=52)
    d = inp.to("cuda")
    args = (d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, adj.d_o.to("cuda"), inp.scale)
    a = kda.chunk_backward(*args, h0=d.h0, dhT=adj.dhT.to("cuda"))
    b = kda.chunk_backward(*args, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_backward_same_after_scratch_release(kda):
    # the scratch pool keeps its blocks between calls; releasing them changes nothing but memory
    inp = inputs.make(1, 2, 50, 128, 128, dtype="bf16", seed=61, h0_std=0.1)
    adj = inputs.adjoints(inp, seed=62)
    d = inp.to("cuda")
    args = (d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, adj.d_o.to("cuda"), inp.scale)
    a = kda.chunk_backward(*args, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    kda.release_scratch()
    b = kda.chunk_backward(*args, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_backward_segmented_schedule_sampled_heads(kda):
    """B*H = 160 sequences (just over the SM count) of a ragged length: the tensor-core form
    splits each walk into segments handed between CTAs; two heads of all five sequences are
    recomputed by the oracle."""
    inp = inputs.make(5, 32, 300, 128, 128, dtype="bf16", seed=71, h0_std=0.1)
    adj = inputs.adjoints(inp, seed=72)
    d = inp.to("cuda")
    g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, adj.d_o.to("cuda"),
                           inp.scale, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    for h in (3, 17):
        sl = lambda t: None if t is None else t[:, h:h + 1].contiguous()
        ref = oracle.backward(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.z), sl(inp.beta),
                              inp.A_log[h:h + 1], inp.dt_bias[h:h + 1], inp.scale, sl(inp.h0),
                              sl(adj.d_o), sl(adj.dhT), threads=8)
        for n in ("dq", "dk", "dv", "dz", "dbeta", "dh0"):
            check(n, g[n][:, h:h + 1], ref[n])
        gate = oracle.gate(sl(inp.z), inp.A_log[h:h + 1], inp.dt_bias[h:h + 1])
        check_reduced("dA_log", g["dA_log"][h:h + 1], ref["dA_log"],
                      np.abs(ref["dg"] * gate).sum(axis=(0, 2, 3)))
        check_reduced("ddt_bias", g["ddt_bias"][h:h + 1], ref["ddt_bias"],
                      np.abs(ref["dz"]).sum(axis=(0, 2)))


def test_backward_full_size_sampled_head(kda):
    """The prefill workload (B8 H32 T4096 K=V=128, bf16) whole on the GPU; head 5 of all eight
    sequences recomputed by the oracle (dA_log[5] and ddt_bias[5] sum exactly those)."""
    inp = inputs.workload("prefill_bf16")
    adj = inputs.adjoints(inp, seed=77)
    d = inp.to("cuda")
    g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, adj.d_o.to("cuda"),
                           inp.scale, h0=d.h0, dhT=adj.dhT.to("cuda"))
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    h = 5
    sl = lambda t: None if t is None else t[:, h:h + 1].contiguous()
    ref = oracle.backward(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.z), sl(inp.beta),
                          inp.A_log[h:h + 1], inp.dt_bias[h:h + 1], inp.scale, sl(inp.h0),
                          sl(adj.d_o), sl(adj.dhT), threads=8)
    for n in ("dq", "dk", "dv", "dz", "dbeta", "dh0"):
        check(n, g[n][:, h:h + 1], ref[n])
    gate = oracle.gate(sl(inp.z), inp.A_log[h:h + 1], inp.dt_bias[h:h + 1])
    check_reduced("dA_log", g["dA_log"][h:h + 1], ref["dA_log"],
                  np.abs(ref["dg"] * gate).sum(axis=(0, 2, 3)))
    check_reduced("ddt_bias", g["ddt_bias"][h:h + 1], ref["ddt_bias"],
                  np.abs(ref["dz"]).sum(axis=(0, 2)))
