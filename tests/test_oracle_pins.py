"""Pins for the f64 oracle, against facts fixed by the pages and by mathematics.

Each test ties the oracle to something other than itself: a high-precision
evaluation (mpmath), a library routine (numpy), a closed form derived by hand,
an invariant the method guarantees, a number the pages print, or an
independently organised evaluation (the chunked WY form).  The mutants at the
end plant known mistakes in the oracle (on the CPU) and check the pins catch them.
"""
import math
import os

import mpmath
import numpy as np
import pytest

import oracle
from oracle import chunked
from gated_delta_rule_26_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gate_np(z, A_log, dt):
    B, H, T, K = z.shape
    return oracle.gate(z, np.asarray(A_log, float), np.asarray(dt, float))


# ---------------------------------------------------------------- gate pins
def test_softplus_matches_high_precision():
    """softplus(x) = log(1 + e^x) to f64 round-off, including far tails (mpmath, 50 digits)."""
    mpmath.mp.dps = 50
    for x in [-745.0, -700.0, -40.0, -20.0, -6.0, -1.0, -1e-8, 0.0, 1e-8, 0.5, 1.0, 6.0, 20.0,
              40.0, 700.0]:
        ref = float(mpmath.log1p(mpmath.exp(mpmath.mpf(x))))
        got = oracle.softplus(x)
        assert got == pytest.approx(ref, rel=4e-16, abs=0.0), x


def test_gate_at_A0_is_minus_softplus():
    """At A_log = 0 the gate reduces to -softplus(z + dt_bias) (kdafix "Fix 1": forms agree at A = 0)."""
    z = np.linspace(-30, 30, 1201).reshape(1, 1, 1201, 1)
    g = _gate_np(z, [0.0], [[0.0]])
    ref = -np.logaddexp(0.0, z)  # numpy's own log(exp(0) + exp(z))
    np.testing.assert_allclose(g, ref, rtol=1e-15, atol=1e-300)


def test_gate_is_nonpositive_and_nan_free_over_sweep():
    """g <= 0 and alpha = exp(g) in [0, 1], finite, over z in [-6, 6] x A_log in {-3, 0, 2}
    and at extreme z (kdafix "Fix 1": NaN-impossible by construction)."""
    z = np.concatenate([np.linspace(-6, 6, 1201), [-1e4, -745.0, 745.0, 1e4]])
    for a in (-3.0, 0.0, 2.0, math.log(16.0), 20.0, -10.0):
        g = _gate_np(z.reshape(1, 1, -1, 1), [a], [[0.0]]).ravel()
        assert np.all(np.isfinite(g))
        assert np.all(g <= 0.0)
        alpha = np.exp(g)
        assert np.all((alpha >= 0.0) & (alpha <= 1.0))
        # strictly inside (0, 1] where no underflow can occur (|g| < 700)
        if a <= math.log(16.0):
            mid = np.abs(z) <= 6
            assert np.all(alpha[mid] > 0.0)


def test_gate_monotone_in_z_and_A():
    """softplus is increasing, exp(A) is increasing: g decreases in z and in A_log."""
    z = np.linspace(-6, 6, 601).reshape(1, 1, -1, 1)
    gs = [_gate_np(z, [a], [[0.0]]).ravel() for a in (-3.0, 0.0, 2.0)]
    for g in gs:
        assert np.all(np.diff(g) < 0)
    assert np.all(gs[0] > gs[1]) and np.all(gs[1] > gs[2])


def test_gate_dt_bias_enters_inside_softplus_per_channel():
    """dt_bias is added to z before softplus, per (head, key channel), broadcast over (b, t)."""
    rng = np.random.default_rng(0)
    B, H, T, K = 2, 3, 5, 4
    z = rng.normal(size=(B, H, T, K))
    A = rng.uniform(-1, 2, size=H)
    dt = rng.normal(size=(H, K))
    g = _gate_np(z, A, dt)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                for c in range(K):
                    ref = -math.exp(A[h]) * float(np.logaddexp(0.0, z[b, h, t, c] + dt[h, c]))
                    assert g[b, h, t, c] == pytest.approx(ref, rel=1e-14)


def test_gate_differs_from_prefix_form_and_order_flips_with_sign_of_A():
    """The FLA form -exp(A) softplus(z) and the superseded -softplus(exp(A) z) are different
    functions: equal only at A = 0; for A > 0 the FLA decay is stronger, for A < 0 weaker
    (kdafix "Fix 1": the order flips with the sign of A).  Proof sketch: h(l) =
    softplus(l z) - l softplus(z) is convex in l with h(1) = 0 and h'(1) < 0."""
    z = np.linspace(-6, 6, 241)
    for a in (-3.0, -0.5, 0.0, 0.5, 2.0):
        fla = _gate_np(z.reshape(1, 1, -1, 1), [a], [[0.0]]).ravel()
        pre = -np.logaddexp(0.0, math.exp(a) * z)
        if a == 0.0:
            np.testing.assert_array_equal(fla, -np.logaddexp(0.0, z))
            np.testing.assert_allclose(fla, pre, rtol=1e-15)
        elif a > 0:
            assert np.all(fla < pre)
        else:
            assert np.all(fla > pre)


# ---------------------------------------------------------------- scale pins
def _rand_problem(B=1, H=2, T=7, K=3, V=5, seed=0, h0=True):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(B, H, T, K))
    k = rng.normal(size=(B, H, T, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(B, H, T, V))
    z = rng.normal(size=(B, H, T, K))
    beta = 1 / (1 + np.exp(-rng.normal(size=(B, H, T))))
    A = rng.uniform(0, math.log(16), size=H)
    dt = rng.normal(size=(H, K)) * 0.1
    S0 = rng.normal(size=(B, H, K, V)) * 0.1 if h0 else None
    return q, k, v, z, beta, A, dt, S0


def test_scale_enters_only_the_read():
    """o(scale) = scale * o(1) and the final state does not depend on the scale at all
    (kdafix "Fix 2": the factor enters only o = q.S, never the state update)."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem()
    o1, h1 = oracle.forward(q, k, v, z, beta, A, dt, 1.0, S0)
    for s in (0.5, 3 ** -0.5, 2.0):
        os_, hs = oracle.forward(q, k, v, z, beta, A, dt, s, S0)
        np.testing.assert_array_equal(hs, h1)
        np.testing.assert_allclose(os_, s * o1, rtol=1e-13, atol=1e-15)
    o_half, _ = oracle.forward(q, k, v, z, beta, A, dt, 0.5, S0)
    np.testing.assert_array_equal(o_half, 0.5 * o1)  # power of two: exact


def test_missing_scale_signature_ratio_at_K8():
    """At K = 8, running without the read scale inflates every output by exactly 8**0.5 = 2.8284
    (kda-oracle-ci-2026-10-02: 'ratio 2.8284' on every line; value stored in tests/golden)."""
    with open(os.path.join(GOLDEN, "read_scale_ratio_K8.txt")) as fh:
        printed = float([ln for ln in fh if not ln.startswith("#")][0].split()[0])
    inp = inputs.workload("small_fp32", A_log_value=-3.0)
    o_fla, _ = oracle.forward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log, inp.dt_bias,
                              inp.scale, inp.h0)
    o_one, _ = oracle.forward(inp.q, inp.k, inp.v, inp.z, inp.beta, inp.A_log, inp.dt_bias,
                              1.0, inp.h0)
    ratio = o_one / o_fla
    assert round(float(np.median(ratio)), 4) == printed
    np.testing.assert_allclose(ratio, 8 ** 0.5, rtol=1e-12)


# ---------------------------------------------------------------- recurrence pins
def test_beta0_alpha1_is_identity_on_state():
    """beta = 0 with alpha = 1 (z -> -inf makes softplus exactly 0 in f64) leaves the state
    unchanged, and every read is scale * h0^T q."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(T=6)
    z = np.full_like(z, -1e4)
    beta = np.zeros_like(beta)
    o, hT = oracle.forward(q, k, v, z, beta, A, np.zeros_like(dt), 0.7, S0)
    np.testing.assert_array_equal(hT, S0)
    ref = 0.7 * np.einsum("bhkv,bhtk->bhtv", S0, q)
    np.testing.assert_allclose(o, ref, rtol=1e-14, atol=1e-15)


def test_beta0_is_pure_decay_closed_form():
    """With beta = 0 the state only decays: S_T = diag(prod_t alpha_t) S_0."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(T=9)
    beta = np.zeros_like(beta)
    o, hT = oracle.forward(q, k, v, z, beta, A, dt, 1.0, S0)
    g = oracle.gate(z, A, dt)
    decay = np.exp(g.sum(axis=2))  # (B, H, K)
    np.testing.assert_allclose(hT, decay[..., None] * S0, rtol=1e-13)
    # and the read at step t sees diag(prod_{s<=t} alpha_s) S_0
    cum = np.exp(np.cumsum(g, axis=2))
    ref = np.einsum("bhtk,bhkv,bhtk->bhtv", cum, S0, q)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-15)


def test_scalar_closed_form_three_steps():
    """K = V = 1, three tokens, written out by hand from the step definition:
    s_t = a_t (1 - b_t k_t^2) s_{t-1} + b_t k_t v_t, o_t = scale q_t s_t."""
    a = [0.9, 0.35, 0.6]
    b = [0.3, 0.8, 0.55]
    kk = [0.7, -1.2, 0.4]
    vv = [1.5, -0.25, 2.0]
    qq = [0.2, -0.9, 1.1]
    s0, sc = 0.8, 0.5
    g = np.log(np.array(a)).reshape(1, 1, 3, 1)
    s1 = a[0] * (1 - b[0] * kk[0] ** 2) * s0 + b[0] * kk[0] * vv[0]
    s2 = a[1] * (1 - b[1] * kk[1] ** 2) * s1 + b[1] * kk[1] * vv[1]
    s3 = a[2] * (1 - b[2] * kk[2] ** 2) * s2 + b[2] * kk[2] * vv[2]
    o, hT = oracle.recurrent(np.array(qq).reshape(1, 1, 3, 1), np.array(kk).reshape(1, 1, 3, 1),
                             np.array(vv).reshape(1, 1, 3, 1), g, np.array(b).reshape(1, 1, 3),
                             sc, np.array([[[[s0]]]]))
    np.testing.assert_allclose(o.ravel(), [sc * qq[0] * s1, sc * qq[1] * s2, sc * qq[2] * s3],
                               rtol=1e-14)
    assert hT.ravel()[0] == pytest.approx(s3, rel=1e-14)


def test_householder_form_with_rectangular_state():
    """The step equals the generalised-Householder form
    S_t = (I - b_t k_t k_t^T) diag(a_t) S_{t-1} + b_t k_t v_t^T   (K != V catches transposes)."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=2, H=2, T=11, K=3, V=5)
    o, hT = oracle.forward(q, k, v, z, beta, A, dt, 0.6, S0)
    g = oracle.gate(z, A, dt)
    for b_ in range(2):
        for h in range(2):
            S = S0[b_, h].copy()
            for t in range(11):
                kt = k[b_, h, t][:, None]
                P = np.eye(3) - beta[b_, h, t] * kt @ kt.T
                S = P @ (np.exp(g[b_, h, t])[:, None] * S) + beta[b_, h, t] * kt @ v[b_, h, t][None, :]
                np.testing.assert_allclose(o[b_, h, t], 0.6 * S.T @ q[b_, h, t], rtol=1e-12,
                                           atol=1e-14)
            np.testing.assert_allclose(hT[b_, h], S, rtol=1e-12, atol=1e-14)


def test_delta_rule_overwrites_value_at_a_key():
    """alpha = 1, beta = 1, unit key: after writing v at key k, reading with q = k returns v
    exactly, and writing a second value at the same key replaces the first (u = v - S^T k)."""
    K, V = 4, 3
    e = np.eye(K)
    k = np.stack([e[1], e[1], e[3], e[1]]).reshape(1, 1, 4, K)
    v = np.array([[1.0, 2.0, 3.0], [-4.0, 0.5, 7.0], [9.0, 8.0, 7.0], [0.25, 0.0, -1.0]])
    g = np.zeros((1, 1, 4, K))
    beta = np.ones((1, 1, 4))
    o, hT = oracle.recurrent(k, k, v.reshape(1, 1, 4, V), g, beta, 1.0)
    np.testing.assert_allclose(o[0, 0], v, rtol=0, atol=1e-15)
    ref = np.zeros((K, V))
    ref[1] = v[3]
    ref[3] = v[2]
    np.testing.assert_allclose(hT[0, 0], ref, atol=1e-15)


# ---------------------------------------------------------------- chunked form and carry
@pytest.mark.parametrize("T,chunk", [(16, 16), (32, 16), (256, 16), (37, 16), (64, 64), (100, 32)])
def test_chunked_wy_agrees_with_recurrence(T, chunk):
    """The chunked WY form and the token recurrence are the same function: one chunk, two
    chunks (the carry is live only from two chunks on), sixteen chunks, ragged tails."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=1, H=2, T=T, K=6, V=5, seed=T + chunk)
    g = oracle.gate(z, A, dt)
    o_r, h_r = oracle.recurrent(q, k, v, g, beta, 0.4, S0)
    o_c, h_c = chunked.chunked_wy(q, k, v, g, beta, 0.4, S0, chunk=chunk)
    scale_o = np.abs(o_r).max()
    assert np.abs(o_c - o_r).max() <= 1e-12 * scale_o
    assert np.abs(h_c - h_r).max() <= 1e-12 * np.abs(h_r).max()


def test_chunked_wy_small_workload_two_chunks():
    """The fixture shape the pages describe: B1 H2 T32 K=V=8, chunk 16, two chunks."""
    for a in (-3.0, 0.0, 2.0):
        inp = inputs.workload("small_fp32", A_log_value=a)
        g = oracle.gate(inp.z, inp.A_log, inp.dt_bias)
        o_r, h_r = oracle.recurrent(inp.q, inp.k, inp.v, g, inp.beta, inp.scale, inp.h0)
        o_c, h_c = chunked.chunked_wy(inp.q, inp.k, inp.v, g, inp.beta, inp.scale, inp.h0, 16)
        np.testing.assert_allclose(o_c, o_r, rtol=0, atol=1e-13)
        np.testing.assert_allclose(h_c, h_r, rtol=0, atol=1e-13)


def test_resume_from_final_state():
    """forward(T1) then forward(T2, h0 = hT1) equals forward(T1 + T2)."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=2, H=2, T=40, K=4, V=6, seed=3)
    o, h = oracle.forward(q, k, v, z, beta, A, dt, 0.5, S0)
    o1, h1 = oracle.forward(q[:, :, :17], k[:, :, :17], v[:, :, :17], z[:, :, :17],
                            beta[:, :, :17], A, dt, 0.5, S0)
    o2, h2 = oracle.forward(q[:, :, 17:], k[:, :, 17:], v[:, :, 17:], z[:, :, 17:],
                            beta[:, :, 17:], A, dt, 0.5, h1)
    np.testing.assert_array_equal(np.concatenate([o1, o2], axis=2), o)
    np.testing.assert_array_equal(h2, h)


def test_state_and_outputs_are_affine_in_the_initial_state():
    """The chunk-parallel scan composes per-segment maps S -> P S + Z: the final state (and
    every output) is affine in the initial state.  With a = f(0), f(S1) - a and f(S2) - a
    must add up to f(S1 + S2) - a and scale with the state, to rounding, for K != V."""
    q, k, v, z, beta, A, dt, S1 = _rand_problem(B=1, H=2, T=24, K=5, V=3, seed=11)
    A = np.array([-2.0, -1.0])  # a slow decay, so that the initial state still shows at the end
    rng = np.random.default_rng(12)
    S2 = rng.standard_normal(S1.shape) * 0.3
    f = lambda S: oracle.forward(q, k, v, z, beta, A, dt, 0.7, S)
    o0, h0 = f(np.zeros_like(S1))
    o1, h1 = f(S1)
    o2, h2 = f(S2)
    o12, h12 = f(S1 + 2.5 * S2)
    np.testing.assert_allclose(h12 - h0, (h1 - h0) + 2.5 * (h2 - h0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o12 - o0, (o1 - o0) + 2.5 * (o2 - o0), rtol=0, atol=1e-12)
    # and the map is not trivial: the initial state matters and the zero-state run does too
    assert np.abs(h1 - h0).max() > 1e-3 and np.abs(h0).max() > 1e-3


def test_threaded_oracle_matches_single_thread():
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=3, H=4, T=20, K=4, V=4, seed=5)
    a = oracle.forward(q, k, v, z, beta, A, dt, 0.5, S0, threads=1)
    b = oracle.forward(q, k, v, z, beta, A, dt, 0.5, S0, threads=5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- planted mistakes
def test_double_exp_carry_mutant_is_caught(monkeypatch):
    """Plant the kda-adjoint-2026-10-01 section 5b bug (exp of an already exponentiated G_last)
    into the chunked oracle: one chunk stays green, two chunks go red."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=1, H=2, T=32, K=8, V=8, seed=11)
    g = oracle.gate(z, A, dt)
    o_r, h_r = oracle.recurrent(q, k, v, g, beta, 0.5, S0)
    monkeypatch.setattr(chunked, "carry_decay", lambda G: np.exp(np.exp(G[-1])[None, :] - G))
    o1, _ = chunked.chunked_wy(q[:, :, :16], k[:, :, :16], v[:, :, :16], g[:, :, :16],
                               beta[:, :, :16], 0.5, S0, 16)
    o_r1, _ = oracle.recurrent(q[:, :, :16], k[:, :, :16], v[:, :, :16], g[:, :, :16],
                               beta[:, :, :16], 0.5, S0)
    np.testing.assert_allclose(o1, o_r1, atol=1e-12)  # one chunk cannot see the carry
    o_c, h_c = chunked.chunked_wy(q, k, v, g, beta, 0.5, S0, 16)
    assert np.abs(h_c - h_r).max() > 1e-2 * np.abs(h_r).max()
    assert np.abs(o_c[:, :, 16:] - o_r[:, :, 16:]).max() > 1e-2 * np.abs(o_r).max()


def test_wrong_sign_in_u_is_caught():
    """u = v + S^T k (sign flip) breaks the overwrite property pinned above."""
    K, V = 4, 3
    e = np.eye(K)
    k = np.stack([e[1], e[1]])
    v = np.array([[1.0, 2.0, 3.0], [-4.0, 0.5, 7.0]])
    S = np.zeros((K, V))
    for t in range(2):  # mutant recurrence, planted here on the CPU
        u = v[t] + S.T @ k[t]
        S = S + np.outer(k[t], u)
    assert not np.allclose(S.T @ k[1], v[1])


def test_prefix_gate_mutant_is_caught():
    """The superseded gate -softplus(exp(A) (z + dt_bias)) planted in place of the gate
    (here, on the CPU) breaks the monotonicity pin: for z < 0 it increases with A_log."""
    z = np.linspace(-6, -0.1, 200)
    mutant = lambda a: -np.logaddexp(0.0, math.exp(a) * z)
    g_lo, g_hi = mutant(-1.0), mutant(1.0)
    assert not np.all(g_lo > g_hi)  # the pin above requires g to decrease in A_log
    # and the oracle's own gate satisfies it on the same points
    ref_lo = _gate_np(z.reshape(1, 1, -1, 1), [-1.0], [[0.0]]).ravel()
    ref_hi = _gate_np(z.reshape(1, 1, -1, 1), [1.0], [[0.0]]).ravel()
    assert np.all(ref_lo > ref_hi)


def test_undecayed_read_mutant_is_caught():
    """u read from the state before its decay (u = v - S^T k, then S <- diag(alpha) S + b k u^T),
    planted here on the CPU, breaks the Householder-form pin whenever alpha != 1."""
    q, k, v, z, beta, A, dt, S0 = _rand_problem(B=1, H=1, T=6, K=3, V=5, seed=9)
    g = oracle.gate(z, A, dt)
    o_ref, h_ref = oracle.forward(q, k, v, z, beta, A, dt, 0.6, S0)
    S = S0[0, 0].copy()
    for t in range(6):
        kt = k[0, 0, t]
        u = v[0, 0, t] - S.T @ kt                      # mutant: undecayed state
        S = np.exp(g[0, 0, t])[:, None] * S + beta[0, 0, t] * np.outer(kt, u)
    assert np.abs(S - h_ref[0, 0]).max() > 1e-3 * np.abs(h_ref).max()
