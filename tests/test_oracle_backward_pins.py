"""Pins for the oracle's backward (the gradients of the KDA forward).

The reverse-mode gradients of ``oracle.backward`` are tied to things other than
themselves: the forward-mode derivative ``oracle.jvp`` (a separate tangent-propagation
code path), central finite differences of the forward oracle (the kda-adjoint-2026-10-01
page's own check: forward mode against central differences, agreeing to about 1e-9),
every coordinate against central differences on a tiny problem, hand-derived closed
forms when beta = 0 and the decay is off, and the exact linearity of the read in the
scale.  Planted mistakes in the backward (on the CPU) must break the pins.
"""
import numpy as np
import pytest

import oracle

NAMES = {"q": "dq", "k": "dk", "v": "dv", "z": "dz", "beta": "dbeta", "A_log": "dA_log",
         "dt_bias": "ddt_bias", "h0": "dh0"}


def _problem(B=2, H=3, T=37, K=5, V=4, seed=0, h0=True, dhT=True):
    rng = np.random.default_rng(seed)
    nrm = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    p = dict(q=nrm(rng.normal(size=(B, H, T, K))), k=nrm(rng.normal(size=(B, H, T, K))),
             v=rng.normal(size=(B, H, T, V)), z=rng.normal(size=(B, H, T, K)),
             beta=1.0 / (1.0 + np.exp(-rng.normal(size=(B, H, T)))),
             A_log=rng.uniform(-1.0, 1.0, size=H), dt_bias=0.3 * rng.normal(size=(H, K)),
             scale=K ** -0.5, h0=0.3 * rng.normal(size=(B, H, K, V)) if h0 else None)
    d_o = rng.normal(size=(B, H, T, V))
    dhT_ = rng.normal(size=(B, H, K, V)) if dhT else None
    return p, d_o, dhT_, rng


def _args(p):
    return (p["q"], p["k"], p["v"], p["z"], p["beta"], p["A_log"], p["dt_bias"], p["scale"], p["h0"])


def _directional(grads, tan):
    return sum(float(np.sum(grads[NAMES[n]] * t)) for n, t in tan.items())


def _tangents(p, rng, names=NAMES):
    return {n: rng.normal(size=np.shape(p[n])) for n in names
            if not (n == "h0" and p["h0"] is None)}


@pytest.mark.parametrize("shape", [(2, 3, 37, 5, 4), (1, 2, 16, 8, 8), (1, 1, 1, 3, 2),
                                   (1, 2, 50, 16, 12)])
@pytest.mark.parametrize("h0,dhT", [(True, True), (False, True), (True, False)])
def test_backward_equals_forward_mode_derivative(shape, h0, dhT):
    """<grad, direction> from the reverse pass equals the forward-mode derivative along that
    direction, to f64 round-off, for one token, exactly one 16-token block, and ragged
    multi-block lengths, with and without h0 and dhT."""
    B, H, T, K, V = shape
    p, d_o, dhT_, rng = _problem(B, H, T, K, V, seed=T + K, h0=h0, dhT=dhT)
    grads = oracle.backward(*_args(p), d_o, dhT_, threads=2)
    for _ in range(3):
        tan = _tangents(p, rng)
        j = oracle.jvp(*_args(p), d_o, dhT_, tan)
        assert _directional(grads, tan) == pytest.approx(j, rel=1e-12, abs=1e-12)


def test_forward_mode_agrees_with_central_differences():
    """The forward-mode derivative agrees with a central difference of the forward oracle
    (step 1e-6, truncation error ~1e-12 here) to within 1e-9 relative."""
    p, d_o, dhT_, rng = _problem()
    tan = _tangents(p, rng)
    j = oracle.jvp(*_args(p), d_o, dhT_, tan)

    def loss(eps):
        a = {n: (p[n] + eps * tan[n] if n in tan else p[n]) for n in p}
        o, hT = oracle.forward(a["q"], a["k"], a["v"], a["z"], a["beta"], a["A_log"],
                               a["dt_bias"], a["scale"], a["h0"])
        return float(np.sum(o * d_o) + np.sum(hT * dhT_))

    fd = (loss(1e-6) - loss(-1e-6)) / 2e-6
    assert abs(fd - j) <= 1e-9 * abs(j)


def test_every_coordinate_against_central_differences():
    """Brute force on a tiny problem: every coordinate of every gradient equals the central
    difference of the loss in that coordinate."""
    p, d_o, dhT_, _ = _problem(B=1, H=2, T=5, K=2, V=3, seed=3)
    grads = oracle.backward(*_args(p), d_o, dhT_)

    def loss(a):
        o, hT = oracle.forward(a["q"], a["k"], a["v"], a["z"], a["beta"], a["A_log"],
                               a["dt_bias"], a["scale"], a["h0"])
        return float(np.sum(o * d_o) + np.sum(hT * dhT_))

    eps = 1e-6
    for n, gname in NAMES.items():
        x = np.asarray(p[n], dtype=float)
        g = grads[gname]
        for idx in np.ndindex(x.shape):
            a = dict(p)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a[n] = xp
            lp = loss(a)
            a[n] = xm
            lm = loss(a)
            fd = (lp - lm) / (2 * eps)
            assert g[idx] == pytest.approx(fd, rel=1e-7, abs=1e-8), (n, idx)


def test_beta0_no_decay_closed_forms():
    """beta = 0 and z -> -inf (softplus underflows to 0, so g = 0 and alpha = 1): the state
    stays h0, o_t = scale h0^T q_t, and by hand
        dq_t = scale h0 d_o_t,  dh0 = dhT + scale sum_t q_t d_o_t^T,  dk = dv = dz = 0,
        dbeta_t = k_t^T (dhT + scale sum_{s >= t} q_s d_o_s^T) (v_t - h0^T k_t),
        dA_log = ddt_bias = 0."""
    p, d_o, dhT_, _ = _problem(B=1, H=2, T=21, K=4, V=3, seed=5)
    p["beta"] = np.zeros_like(p["beta"])
    p["z"] = np.full_like(p["z"], -1e4)
    g = oracle.backward(*_args(p), d_o, dhT_)
    sc, h0, q, k, v = p["scale"], p["h0"], p["q"], p["k"], p["v"]
    np.testing.assert_allclose(g["dq"], sc * np.einsum("bhcj,bhtj->bhtc", h0, d_o), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(g["dh0"], dhT_ + sc * np.einsum("bhtc,bhtj->bhcj", q, d_o), rtol=1e-13, atol=1e-14)
    for n in ("dk", "dv", "dz", "dA_log", "ddt_bias"):
        assert np.all(g[n] == 0.0), n
    T = q.shape[2]
    for t in range(T):
        dS = dhT_ + sc * np.einsum("bhsc,bhsj->bhcj", q[:, :, t:], d_o[:, :, t:])
        u = v[:, :, t] - np.einsum("bhcj,bhc->bhj", h0, k[:, :, t])
        ref = np.einsum("bhc,bhcj,bhj->bh", k[:, :, t], dS, u)
        np.testing.assert_allclose(g["dbeta"][:, :, t], ref, rtol=1e-12, atol=1e-13)


def test_gradients_scale_linearly_without_dhT():
    """With dhT = 0 every gradient reaches the loss only through o, which is linear in the
    scale: doubling the scale doubles every gradient (exactly: a power of two)."""
    p, d_o, _, _ = _problem(dhT=False)
    g1 = oracle.backward(*_args(p), d_o, None)
    p2 = dict(p, scale=2.0 * p["scale"])
    g2 = oracle.backward(*_args(p2), d_o, None)
    for n in NAMES.values():
        np.testing.assert_array_equal(g2[n], 2.0 * g1[n])


def test_threaded_backward_matches_single_thread():
    p, d_o, dhT_, _ = _problem(B=2, H=3, T=40)
    a = oracle.backward(*_args(p), d_o, dhT_, threads=1)
    b = oracle.backward(*_args(p), d_o, dhT_, threads=4)
    for n in NAMES.values():
        np.testing.assert_array_equal(a[n], b[n])


@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_planted_backward_mistakes_are_caught(mutant):
    """1: dk without the -Sd du term; 2: dalpha taken against the decayed state; 3: dS
    without diag(alpha).  Each breaks the forward-mode pin by far more than round-off."""
    p, d_o, dhT_, rng = _problem()
    tan = _tangents(p, rng)
    j = oracle.jvp(*_args(p), d_o, dhT_, tan)
    bad = oracle.backward(*_args(p), d_o, dhT_, mutant=mutant)
    assert abs(_directional(bad, tan) - j) > 1e-3 * abs(j)


def test_log_decay_gradient_against_central_differences():
    """dg, the gradient with respect to the log decay itself, coordinate by coordinate against
    central differences of the recurrence taken with g as its input (oracle.recurrent), on a
    tiny problem; and dz = dg (-e^{A_log}) sigmoid(z + dt_bias) on a larger one."""
    p, d_o, dhT_, _ = _problem(B=1, H=2, T=6, K=2, V=3, seed=13)
    grads = oracle.backward(*_args(p), d_o, dhT_)
    g = oracle.gate(p["z"], p["A_log"], p["dt_bias"])

    def loss(gg):
        o, hT = oracle.recurrent(p["q"], p["k"], p["v"], gg, p["beta"], p["scale"], p["h0"])
        return float(np.sum(o * d_o) + np.sum(hT * dhT_))

    eps = 1e-6
    for idx in np.ndindex(g.shape):
        gp, gm = g.copy(), g.copy()
        gp[idx] += eps
        gm[idx] -= eps
        fd = (loss(gp) - loss(gm)) / (2 * eps)
        assert grads["dg"][idx] == pytest.approx(fd, rel=1e-7, abs=1e-8), idx
    p, d_o, dhT_, _ = _problem(seed=14)
    grads = oracle.backward(*_args(p), d_o, dhT_)
    x = p["z"] + p["dt_bias"][None, :, None, :]
    sig = 1.0 / (1.0 + np.exp(-x))
    np.testing.assert_allclose(grads["dz"], grads["dg"] * (-np.exp(p["A_log"]))[None, :, None, None] * sig,
                               rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("T,chunk", [(16, 16), (37, 16), (50, 32), (64, 64), (100, 16)])
def test_chunked_backward_equals_reverse_mode(T, chunk):
    """The chunk-level adjoint equations (oracle.chunked_backward, the form the GPU kernel
    takes) equal the token reverse mode to f64 round-off, at several chunk sizes and ragged
    lengths; this pins the chunked backward's derivation independently of any GPU."""
    from oracle.chunked_backward import chunked_backward
    p, d_o, dhT_, _ = _problem(B=2, H=2, T=T, K=6, V=5, seed=T + chunk)
    ref = oracle.backward(*_args(p), d_o, dhT_)
    g = oracle.gate(p["z"], p["A_log"], p["dt_bias"])
    got = chunked_backward(p["q"], p["k"], p["v"], g, p["beta"], p["scale"], p["h0"], d_o,
                           dhT_, chunk)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        err = np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max()
        assert err <= 1e-10, (n, err)
