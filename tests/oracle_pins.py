"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- a closed form the recurrence implies, an invariant, a library
routine (numpy.correlate, scipy.special.expit, numpy.logaddexp,
numpy.linalg.norm), or brute force.

Every check takes ``fwd`` (a callable with ``oracle.forward``'s signature) so
that ``test_oracle_mutations.py`` can run the same checks against builds of the
oracle with a planted mistake and show that each mistake is caught.

The method is the "Gated DeltaNet layer" paragraph of the xwen CLAUDE.md page,
"Architecture cheat sheet (Qwen 3.6, ggml-org GGUF)" section.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import expit

D = 128
EPS = 1e-6


def rng_case(seed, Hk=1, Hv=2, T=8, N=1, s0_scale=0.02, conv0=True, lengths=None):
    """Small random inputs (numpy float32 values, fp64 state)."""
    r = np.random.default_rng(seed)
    C = D * (2 * Hk + Hv)
    if lengths is not None:
        N, T = len(lengths), sum(lengths)
    c = dict(
        Hk=Hk, Hv=Hv,
        x=r.standard_normal((T, C)).astype(np.float32),
        z=r.standard_normal((T, Hv * D)).astype(np.float32),
        a_raw=r.standard_normal((T, Hv)).astype(np.float32),
        b_raw=r.standard_normal((T, Hv)).astype(np.float32),
        conv_w=(0.25 * r.standard_normal((C, 4))).astype(np.float32),
        dt_bias=r.uniform(-2, 1, Hv).astype(np.float32),
        ssm_a=(-np.exp(r.uniform(0, math.log(16), Hv))).astype(np.float32),
        norm_w=(1 + 0.1 * r.standard_normal(D)).astype(np.float32),
        conv_state=(r.standard_normal((N, 3, C)) if conv0 else np.zeros((N, 3, C))).astype(np.float32),
        S=s0_scale * r.standard_normal((N, Hv, D, D)),
    )
    c["cu_seqlens"] = np.concatenate([[0], np.cumsum(lengths)]) if lengths is not None else [0, T]
    return c


def run(fwd, c, **kw):
    args = {k: c[k] for k in ("Hk", "Hv", "x", "z", "a_raw", "b_raw", "conv_w", "dt_bias",
                              "ssm_a", "norm_w", "conv_state", "S", "cu_seqlens")}
    args.update(kw)
    return fwd(**args)


def identity_taps(C):
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0          # tap 3 multiplies the current token (conv orientation reading)
    return w


def split_inter(inter):
    return inter[..., :D], inter[..., D:2 * D], inter[..., 2 * D:3 * D], inter[..., 3 * D], inter[..., 3 * D + 1]


def _silu_lib(u):
    return u * expit(u)


# --------------------------------------------------------------------------- gates
def check_gates(fwd):
    """beta = sigmoid(b_raw), g = ssm_a * softplus(a_raw + dt_bias) against
    scipy.special.expit / numpy.logaddexp, and the special values
    sigmoid(0) = 1/2, softplus(0) = ln 2, sigmoid(+-inf) = 1, 0."""
    c = rng_case(1, T=6)
    c["b_raw"][0, :] = 0.0
    c["b_raw"][1, 0] = np.inf
    c["b_raw"][1, 1] = -np.inf
    c["a_raw"][2, :] = -c["dt_bias"]
    r = run(fwd, c, want_inter=True)
    _, _, _, beta, g = split_inter(r.inter)
    assert np.all(beta[0] == 0.5)
    assert beta[1, 0] == 1.0 and beta[1, 1] == 0.0
    np.testing.assert_allclose(g[2], c["ssm_a"].astype(np.float64) * math.log(2.0), rtol=1e-15)
    ok = np.isfinite(c["b_raw"])
    np.testing.assert_allclose(beta[ok], expit(c["b_raw"].astype(np.float64))[ok], rtol=1e-15)
    ref_g = c["ssm_a"][None, :].astype(np.float64) * np.logaddexp(
        0.0, c["a_raw"].astype(np.float64) + c["dt_bias"][None, :].astype(np.float64))
    np.testing.assert_allclose(g, ref_g, rtol=1e-14)


# --------------------------------------------------------------------------- conv / silu / split / L2 / tiling
def check_conv_silu_split_l2_tiling(fwd):
    """Steps 1-5 against numpy.correlate (the conv as a per-channel 'valid'
    cross-correlation over [conv_state; x]), expit-SiLU, numpy.linalg.norm, and
    the tiled head map (v-head j reads q/k head j mod H_k)."""
    Hk, Hv, T = 2, 4, 7
    c = rng_case(2, Hk=Hk, Hv=Hv, T=T)
    r = run(fwd, c, want_inter=True)
    q_hat, k_hat, v, _, _ = split_inter(r.inter)
    x = c["x"].astype(np.float64)
    xx = np.concatenate([c["conv_state"][0].astype(np.float64), x], axis=0)
    W = c["conv_w"].astype(np.float64)
    C = x.shape[1]
    u = np.stack([np.correlate(xx[:, ch], W[ch], mode="valid") for ch in range(C)], axis=1)
    assert u.shape == (T, C)
    act = _silu_lib(u)
    for h in range(Hv):
        kh = h % Hk
        qa = act[:, kh * D:(kh + 1) * D]
        ka = act[:, Hk * D + kh * D:Hk * D + (kh + 1) * D]
        va = act[:, 2 * Hk * D + h * D:2 * Hk * D + (h + 1) * D]
        np.testing.assert_allclose(v[:, h], va, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(q_hat[:, h], qa / np.linalg.norm(qa, axis=1, keepdims=True),
                                   rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(k_hat[:, h], ka / np.linalg.norm(ka, axis=1, keepdims=True),
                                   rtol=1e-12, atol=1e-14)
    # tiling: heads j and j + Hk share q/k; j and j+1 do not (interleave would pair 0,1)
    assert np.array_equal(q_hat[:, 0], q_hat[:, 2]) and np.array_equal(k_hat[:, 1], k_hat[:, 3])
    assert not np.allclose(k_hat[:, 0], k_hat[:, 1])


def check_identity_taps(fwd):
    """Taps (0,0,0,1) make the conv the identity on the current token: v = silu(x)."""
    c = rng_case(3, T=5)
    c["conv_w"] = identity_taps(c["x"].shape[1])
    r = run(fwd, c, want_inter=True)
    _, _, v, _, _ = split_inter(r.inter)
    Hk = c["Hk"]
    for h in range(c["Hv"]):
        xv = c["x"][:, 2 * Hk * D + h * D:2 * Hk * D + (h + 1) * D].astype(np.float64)
        np.testing.assert_allclose(v[:, h], _silu_lib(xv), rtol=1e-14, atol=1e-300)


def check_l2_clamp(fwd):
    """Clamp form x / max(||x||, eps): a zero vector stays zero (no NaN) and a
    vector with norm below eps is scaled by 1/eps, not normalised."""
    c = rng_case(4, T=3, conv0=False)
    C = c["x"].shape[1]
    c["conv_w"] = identity_taps(C)
    c["x"][0, 0:D] = 0.0                    # q head 0, token 0: silu(0) = 0
    c["x"][1, 0:D] = 0.0
    c["x"][1, 5] = 1e-9                     # tiny: ||silu(x)|| ~ 5e-10 < eps
    r = run(fwd, c, want_inter=True)
    q_hat = r.inter[..., :D]
    assert np.all(q_hat[0, 0] == 0.0) and np.all(np.isfinite(r.out))
    expect = np.zeros(D)
    expect[5] = _silu_lib(np.float64(np.float32(1e-9))) / EPS
    np.testing.assert_allclose(q_hat[1, 0], expect, rtol=1e-13, atol=0)


# --------------------------------------------------------------------------- delta rule closed forms
def check_one_token_closed_form(fwd):
    """From S0 = 0, one token gives o = beta (k_hat . q_hat) v / sqrt(128)
    (before the gated norm) -- the decay cannot act on a zero state."""
    c = rng_case(5, Hk=2, Hv=4, T=1)
    c["S"][:] = 0.0
    r = run(fwd, c, want_inter=True)
    q, k, v, beta, _ = split_inter(r.inter)
    for h in range(4):
        expect = beta[0, h] * np.dot(k[0, h], q[0, h]) * v[0, h] / math.sqrt(D)
        np.testing.assert_allclose(r.prenorm[0, h * D:(h + 1) * D], expect, rtol=1e-12, atol=1e-15)
        # and the state is the rank-one write beta * v k^T
        np.testing.assert_allclose(r.S[0, h], beta[0, h] * np.outer(v[0, h], k[0, h]),
                                   rtol=1e-12, atol=1e-16)


def check_identity_state(fwd):
    """g = 0 (ssm_a = 0) and beta = 0 (b_raw = -inf) leave S bit-unchanged;
    then o = S0 q_hat / sqrt(128) for every token."""
    c = rng_case(6, T=5)
    c["ssm_a"][:] = 0.0
    c["b_raw"][:] = -np.inf
    r = run(fwd, c, want_inter=True)
    assert np.array_equal(r.S, c["S"])
    q = r.inter[..., :D]
    for h in range(c["Hv"]):
        np.testing.assert_allclose(r.prenorm[:, h * D:(h + 1) * D],
                                   q[:, h] @ c["S"][0, h].T / math.sqrt(D), rtol=1e-12, atol=1e-16)


def check_pure_decay(fwd):
    """beta = 0 alone: S_T = exp(sum_t g_t) S0 (closed form)."""
    c = rng_case(7, T=6, s0_scale=1.0)
    c["b_raw"][:] = -np.inf
    c["ssm_a"][:] = -0.3                    # keep the total decay representable
    r = run(fwd, c, want_inter=True)
    g = r.inter[..., 3 * D + 1]
    for h in range(c["Hv"]):
        np.testing.assert_allclose(r.S[0, h], np.exp(g[:, h].sum()) * c["S"][0, h], rtol=1e-12)


def check_recall_beta_one(fwd):
    """beta = 1 (b_raw = +inf): after each token S_t k_hat_t = v_t exactly, for
    any prior state and any g.  With the q channels equal to the k channels,
    q_hat = k_hat and so o_t = v_t / sqrt(128) at every token."""
    Hk, Hv = 1, 2
    c = rng_case(8, Hk=Hk, Hv=Hv, T=9, s0_scale=0.5)
    c["b_raw"][:] = np.inf
    c["x"][:, 0:D] = c["x"][:, D:2 * D]
    c["conv_w"][0:D] = c["conv_w"][D:2 * D]
    c["conv_state"][:, :, 0:D] = c["conv_state"][:, :, D:2 * D]
    r = run(fwd, c, want_inter=True)
    _, k, v, _, _ = split_inter(r.inter)
    for h in range(Hv):
        np.testing.assert_allclose(r.prenorm[:, h * D:(h + 1) * D], v[:, h] / math.sqrt(D),
                                   rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(r.S[0, h] @ k[-1, h], v[-1, h], rtol=1e-11, atol=1e-13)


def _silu_inv(y):
    """Preimage of y under silu on the branch x > -1.2785 (y > -0.2784)."""
    from scipy.optimize import brentq
    return brentq(lambda t: t * expit(t) - y, -1.2784645, 60.0, xtol=1e-15, rtol=1e-15)


def check_orthonormal_memory(fwd):
    """g = 0, beta = 1, S0 = 0 and orthonormal keys: after writing (k_i, v_i)
    for every i, S k_i = v_i for all of them.  Keys are the rotated pairs
    (e_2p +- e_2p+1)/sqrt(2), driven through identity taps and an inverted SiLU
    so the whole pipeline produces them."""
    Hk, Hv, m = 1, 1, 24
    c = rng_case(9, Hk=Hk, Hv=Hv, T=m, conv0=False)
    C = c["x"].shape[1]
    c["conv_w"] = identity_taps(C)
    c["ssm_a"][:] = 0.0
    c["b_raw"][:] = np.inf
    c["S"][:] = 0.0
    alpha = 0.2
    kpre = np.zeros((m, D))
    keys = np.zeros((m, D))
    pos, neg = _silu_inv(alpha), _silu_inv(-alpha)
    for t in range(m):
        p = t // 2
        kpre[t, 2 * p] = pos
        kpre[t, 2 * p + 1] = pos if t % 2 == 0 else neg
        keys[t, 2 * p] = 1.0
        keys[t, 2 * p + 1] = 1.0 if t % 2 == 0 else -1.0
    keys /= math.sqrt(2.0)
    c["x"][:, D:2 * D] = kpre.astype(np.float32)
    r = run(fwd, c, want_inter=True)
    k_hat, v = r.inter[:, 0, D:2 * D], r.inter[:, 0, 2 * D:3 * D]
    np.testing.assert_allclose(k_hat, keys, atol=1e-7)          # float32 preimages
    np.testing.assert_allclose(k_hat @ k_hat.T, np.eye(m), atol=2e-7)
    recalled = k_hat @ r.S[0, 0].T                               # row t = S k_t
    np.testing.assert_allclose(recalled, v, atol=5e-6 * np.abs(v).max())


def check_matrix_product_form(fwd):
    """Brute force in matrix form: S_t = e^{g_t} S_{t-1} (I - beta_t k k^T)
    + beta_t v k^T and o_t = S_t q_t / sqrt(128), composed with numpy matmuls
    from the oracle's own per-token q_hat, k_hat, v, beta, g."""
    c = rng_case(10, Hk=2, Hv=4, T=12, s0_scale=0.3)
    r = run(fwd, c, want_inter=True)
    q, k, v, beta, g = split_inter(r.inter)
    for h in range(4):
        S = c["S"][0, h].copy()
        for t in range(12):
            kk = k[t, h][:, None]
            S = np.exp(g[t, h]) * S @ (np.eye(D) - beta[t, h] * kk @ kk.T) + beta[t, h] * np.outer(v[t, h], k[t, h])
            np.testing.assert_allclose(r.prenorm[t, h * D:(h + 1) * D], S @ q[t, h] / math.sqrt(D),
                                       rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(r.S[0, h], S, rtol=1e-10, atol=1e-14)


# --------------------------------------------------------------------------- gated RMSNorm
def check_gated_rmsnorm(fwd):
    """With norm_w = 1 and z = 40 (silu(40) = 40 to 1e-16), the per-head RMS of
    y / 40 is sqrt(m / (m + eps)), m the head's mean o^2 -- normalisation over
    each head's 128 outputs with eps inside the root.  A head whose o is tiny
    (m << eps) comes out scaled by 1/sqrt(eps), not normalised."""
    c = rng_case(11, Hk=1, Hv=2, T=4)
    c["norm_w"][:] = 1.0
    c["z"][:] = 40.0
    # head 1: tiny values -> tiny o
    c["x"][:, 2 * D + D:2 * D + 2 * D] *= 1e-3
    c["conv_state"][:, :, 2 * D + D:] *= 1e-3
    c["S"][:, 1] *= 1e-3
    r = run(fwd, c)
    for h in range(2):
        o = r.prenorm[:, h * D:(h + 1) * D]
        y = r.out[:, h * D:(h + 1) * D] / 40.0
        m = np.mean(o * o, axis=1)
        np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(m / (m + EPS)), rtol=1e-12)
    assert np.mean(r.prenorm[:, D:] ** 2) < 1e-2 * EPS
    # with random weights / gates: y / (w silu(z)) is o scaled by one positive factor per row
    c2 = rng_case(12, Hk=1, Hv=2, T=3)
    r2 = run(fwd, c2)
    ratio = r2.out / (np.tile(c2["norm_w"], 2)[None, :] * _silu_lib(c2["z"].astype(np.float64)))
    for h in range(2):
        sl = slice(h * D, (h + 1) * D)
        f = ratio[:, sl] / r2.prenorm[:, sl]
        np.testing.assert_allclose(f, f[:, :1] * np.ones((1, D)), rtol=1e-9)


# --------------------------------------------------------------------------- conv state / resume / varlen
def check_conv_state_bookkeeping(fwd):
    """After a sequence the conv state is its last 3 raw rows (bit-exact);
    with fewer than 3 tokens the older rows come from the previous state."""
    for T in (1, 2, 3, 5):
        c = rng_case(13 + T, T=T)
        r = run(fwd, c)
        full = np.concatenate([c["conv_state"][0], c["x"]], axis=0)
        assert np.array_equal(r.conv_state[0], full[-3:])


def check_split_resume(fwd):
    """Running T1 tokens and then T2 from the returned states equals running
    T1 + T2 at once (bit-for-bit: same operations in the same order)."""
    c = rng_case(20, T=11)
    whole = run(fwd, c)
    a = {**c, "x": c["x"][:4], "z": c["z"][:4], "a_raw": c["a_raw"][:4], "b_raw": c["b_raw"][:4],
         "cu_seqlens": [0, 4]}
    ra = run(fwd, a)
    b = {**c, "x": c["x"][4:], "z": c["z"][4:], "a_raw": c["a_raw"][4:], "b_raw": c["b_raw"][4:],
         "cu_seqlens": [0, 7], "conv_state": ra.conv_state, "S": ra.S}
    rb = run(fwd, b)
    assert np.array_equal(np.concatenate([ra.out, rb.out]), whole.out)
    assert np.array_equal(rb.S, whole.S) and np.array_equal(rb.conv_state, whole.conv_state)


def check_varlen_independence(fwd):
    """Packed sequences (cu_seqlens) are independent: a packed run equals
    separate runs, including an empty sequence."""
    lengths = [3, 0, 5, 1]
    c = rng_case(21, lengths=lengths)
    packed = run(fwd, c)
    cu = c["cu_seqlens"]
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = {**c, "x": c["x"][t0:t1], "z": c["z"][t0:t1], "a_raw": c["a_raw"][t0:t1],
               "b_raw": c["b_raw"][t0:t1], "conv_state": c["conv_state"][s:s + 1],
               "S": c["S"][s:s + 1], "cu_seqlens": [0, L]}
        r = run(fwd, one)
        assert np.array_equal(r.out, packed.out[t0:t1])
        assert np.array_equal(r.S[0], packed.S[s])
        assert np.array_equal(r.conv_state[0], packed.conv_state[s])


ALL_CHECKS = [
    check_gates, check_conv_silu_split_l2_tiling, check_identity_taps, check_l2_clamp,
    check_one_token_closed_form, check_identity_state, check_pure_decay, check_recall_beta_one,
    check_orthonormal_memory, check_matrix_product_form, check_gated_rmsnorm,
    check_conv_state_bookkeeping, check_split_resume, check_varlen_independence,
]
