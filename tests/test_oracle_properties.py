"""Property-based checks of the oracle over random shapes (hypothesis; skipped where it is not
installed).  Each property is one the method fixes for every input:

* the chunked WY evaluation equals the token recurrence, for any chunk size and length
  (kda-adjoint-2026-10-01, section 2: the chunk form is an exact rewriting);
* splitting a sequence and resuming from hT equals running it whole;
* the reverse-mode gradients contract with any direction to the forward-mode derivative.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import chunked  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


def _problem(B, H, T, K, V, seed, h0=True):
    rng = np.random.default_rng(seed)
    nrm = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = nrm(rng.normal(size=(B, H, T, K)))
    k = nrm(rng.normal(size=(B, H, T, K)))
    v = rng.normal(size=(B, H, T, V))
    z = rng.normal(size=(B, H, T, K)) * 1.5
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(B, H, T))))
    A = rng.uniform(-2.0, np.log(16.0), size=H)
    dt = 0.3 * rng.normal(size=(H, K))
    S0 = 0.3 * rng.normal(size=(B, H, K, V)) if h0 else None
    return q, k, v, z, beta, A, dt, S0


shapes = st.tuples(st.integers(1, 2), st.integers(1, 2), st.integers(1, 70),
                   st.integers(1, 9), st.integers(1, 9), st.integers(0, 10 ** 6))


@SETTINGS
@given(shapes, st.sampled_from([16, 32, 64]), st.booleans())
def test_chunked_form_equals_recurrence(shape, chunk, h0):
    B, H, T, K, V, seed = shape
    q, k, v, z, beta, A, dt, S0 = _problem(B, H, T, K, V, seed, h0)
    g = oracle.gate(z, A, dt)
    o_r, h_r = oracle.recurrent(q, k, v, g, beta, K ** -0.5, S0)
    o_c, h_c = chunked.chunked_wy(q, k, v, g, beta, K ** -0.5, S0, chunk)
    sc = max(1.0, np.abs(o_r).max(), np.abs(h_r).max())
    assert np.abs(o_c - o_r).max() <= 1e-10 * sc
    assert np.abs(h_c - h_r).max() <= 1e-10 * sc


@SETTINGS
@given(shapes, st.integers(0, 70))
def test_resume_equals_whole(shape, cut):
    B, H, T, K, V, seed = shape
    cut = min(cut, T)
    q, k, v, z, beta, A, dt, S0 = _problem(B, H, T, K, V, seed)
    o, h = oracle.forward(q, k, v, z, beta, A, dt, 0.7, S0)
    s1 = slice(0, cut)
    s2 = slice(cut, T)
    o1, h1 = oracle.forward(q[:, :, s1], k[:, :, s1], v[:, :, s1], z[:, :, s1], beta[:, :, s1],
                            A, dt, 0.7, S0)
    o2, h2 = oracle.forward(q[:, :, s2], k[:, :, s2], v[:, :, s2], z[:, :, s2], beta[:, :, s2],
                            A, dt, 0.7, h1)
    np.testing.assert_array_equal(np.concatenate([o1, o2], axis=2), o)
    np.testing.assert_array_equal(h2, h)


@SETTINGS
@given(shapes, st.booleans(), st.booleans())
def test_reverse_mode_contracts_to_forward_mode(shape, h0, with_dhT):
    B, H, T, K, V, seed = shape
    q, k, v, z, beta, A, dt, S0 = _problem(B, H, T, K, V, seed, h0)
    rng = np.random.default_rng(seed + 1)
    d_o = rng.normal(size=v.shape)
    dhT = rng.normal(size=(B, H, K, V)) if with_dhT else None
    grads = oracle.backward(q, k, v, z, beta, A, dt, K ** -0.5, S0, d_o, dhT)
    inputs = dict(q=q, k=k, v=v, z=z, beta=beta, A_log=A, dt_bias=dt)
    if h0:
        inputs["h0"] = S0
    tan = {n: rng.normal(size=np.shape(x)) for n, x in inputs.items()}
    j = oracle.jvp(q, k, v, z, beta, A, dt, K ** -0.5, S0, d_o, dhT, tan)
    names = {"q": "dq", "k": "dk", "v": "dv", "z": "dz", "beta": "dbeta", "A_log": "dA_log",
             "dt_bias": "ddt_bias", "h0": "dh0"}
    dot = sum(float(np.sum(grads[names[n]] * t)) for n, t in tan.items())
    scale = sum(float(np.sum(np.abs(grads[names[n]] * t))) for n, t in tan.items())
    assert abs(dot - j) <= 1e-12 * max(scale, 1e-30)
