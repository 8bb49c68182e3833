"""Pins for the oracle's attention and the distortion decomposition theorem."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def test_attention_special_cases():
    rng = np.random.default_rng(0)
    d, L = 16, 40
    q = rng.standard_normal(d)
    V = rng.standard_normal((L, d))
    # all keys equal -> uniform weights -> mean of V
    K = np.tile(rng.standard_normal(d), (L, 1))
    assert np.allclose(oracle.attention(q, K, V), V.mean(0), atol=1e-14)
    # one dominant logit -> the value row of that token
    K = rng.standard_normal((L, d)) * 0.01
    K[13] = q * 1e3
    assert np.allclose(oracle.attention(q, K, V), V[13], atol=1e-12)
    # a single token
    assert np.allclose(oracle.attention(q, K[:1], V[:1]), V[0])
    # empty cache -> zeros
    assert np.all(oracle.attention(q, K[:0], V[:0]) == 0)


def test_attention_against_library_softmax_and_shift_invariance():
    rng = np.random.default_rng(1)
    d, L = 128, 333
    q = rng.standard_normal(d) * 3
    K = rng.standard_normal((L, d)) + 2.0
    V = rng.standard_normal((L, d))
    ref = softmax(K @ q / np.sqrt(d)) @ V
    o = oracle.attention(q, K, V)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-14)
    # adding a constant vector c to every key adds q.c to every logit: no change
    assert np.allclose(oracle.attention(q, K + rng.standard_normal(d), V), o, rtol=1e-10)


def test_decode_from_records_matches_reconstructed_attention():
    """Decode over packed records equals attention over the reconstructed rows,
    and the constant terms the GPU drops (q . mu_k, the code midpoints) do not
    change the output."""
    rng = np.random.default_rng(2)
    d, L, G = 128, 200, 4
    lam = 0.95 ** np.arange(d)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    mu_k = rng.standard_normal(d) * 2
    K = (rng.standard_normal((L, d)) * np.sqrt(lam)) @ Qm.T + mu_k
    V = (rng.standard_normal((L, d)) * np.sqrt(lam)) @ Qm.T
    bits, _ = oracle.allocate_bits(lam, 352)
    step = oracle.steps(lam, bits)
    kr, _, _ = oracle.encode(K, Qm.T, mu_k, step, bits)
    vr, _, _ = oracle.encode(V, Qm.T, np.zeros(d), step, bits)
    cal = dict(T_k_inv=Qm[None], mu_k=mu_k[None], step_k=step[None], bits_k=bits[None],
               U_v=Qm[None], mu_v=np.zeros((1, d)), step_v=step[None], bits_v=bits[None], W=11)
    q = rng.standard_normal((1, G, d))
    out = oracle.decode_attention(q, kr[None, None], vr[None, None], cal)
    Kh = oracle.reconstruct(kr, Qm, mu_k, step, bits)
    Vh = oracle.reconstruct(vr, Qm, np.zeros(d), step, bits)
    for g in range(G):
        assert np.allclose(out[0, g], oracle.attention(q[0, g], Kh, Vh), rtol=1e-12)
        # the folded score q'.u differs from q.k_hat/sqrt(d) by a per-query constant
        ck = (Kh - mu_k) @ Qm                   # coefficients of k_hat
        mid = np.where(bits > 0, (2.0 ** bits - 1) / 2, 0.0)
        u = np.where(bits > 0, ck / np.where(step > 0, step, 1) + mid, 0.0)
        qp = (Qm.T @ q[0, g]) * step / np.sqrt(d)
        diff = u @ qp - Kh @ q[0, g] / np.sqrt(d)
        assert np.ptp(diff) < 1e-9 * np.abs(Kh @ q[0, g]).max()
    # the budget can be all 8-bit channels: the output approaches exact attention
    bits8 = np.full(d, 8)
    step8 = oracle.steps(lam, bits8)
    kr8, _, _ = oracle.encode(K, Qm.T, mu_k, step8, bits8)
    vr8, _, _ = oracle.encode(V, Qm.T, np.zeros(d), step8, bits8)
    cal8 = dict(cal, step_k=step8[None], bits_k=bits8[None], step_v=step8[None],
                bits_v=bits8[None], W=32)
    o8 = oracle.decode_attention(q, kr8[None, None], vr8[None, None], cal8)
    for g in range(G):
        ex = oracle.attention(q[0, g], K, V)
        assert np.abs(o8[0, g] - ex).max() < 0.05 * np.abs(ex).max() + 4 * step8.max()


@pytest.mark.parametrize("which", ["k", "v", "kv"])
def test_distortion_decomposition_monte_carlo(which):
    """Theorem (additive error decomposition): under white noise of small
    variance injected in the transform domain, E|o - o_hat|^2 equals
    D_K + D_V with
        D_V = sum_i A_i^2 tr Cov(e_v,i)
        D_K = (1/d) sum_i A_i^2 |v_i - o|^2 q^T Cov(e_k,i) q,
    the first-order softmax perturbation, which reduces to the printed form
    sum_j q_j^2 sigma_j^2 when Cov is diagonal.  In the "kv" case the value
    noise is scaled so that both terms are equal: a dropped term or a nonzero
    cross term would then miss the prediction by half.

    10^5 trials; the bound is 3 Monte-Carlo standard errors plus 1e-4 of the
    prediction for the terms the first-order expansion leaves out.  Those
    start at sigma^4 (the sigma^3 term has odd Gaussian moments and vanishes):
    the same draws at ten times the noise move the relative deviation by
    3e-4, so at this noise level the neglected part is near 3e-6 of the
    prediction."""
    rng = np.random.default_rng({"k": 11, "v": 12, "kv": 13}[which])
    d, L, trials = 8, 16, 100000
    q = rng.standard_normal(d) * 2
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    Tm = rng.standard_normal((d, d)) + 3 * np.eye(d)       # a non-orthogonal transform
    Ti = np.linalg.inv(Tm)
    sig_k = 1e-3 * (1 + rng.random(d))                      # white per-coefficient std (keys)
    sig_v = 1e-3 * (1 + rng.random(d))                      # (values)
    o = oracle.attention(q, K, V)
    A = softmax(K @ q / np.sqrt(d))
    Cov = Ti @ np.diag(sig_k ** 2) @ Ti.T                   # key noise covariance in x
    DK = np.sum(A ** 2 * np.sum((V - o) ** 2, 1)) * (q @ Cov @ q) / d
    DV = np.sum(A ** 2) * np.sum(sig_v ** 2)                # orthogonal-free: tr of white noise
    if which == "kv":
        sig_v *= np.sqrt(DK / DV)
        DV = np.sum(A ** 2) * np.sum(sig_v ** 2)
        assert abs(DK - DV) < 1e-12 * DK
    pred = (DK if "k" in which else 0.0) + (DV if "v" in which else 0.0)
    errs = np.empty(trials)
    for t in range(trials):
        Kh = K + (rng.standard_normal((L, d)) * sig_k) @ Ti.T if "k" in which else K
        Vh = V + rng.standard_normal((L, d)) * sig_v if "v" in which else V
        errs[t] = np.sum((oracle.attention(q, Kh, Vh) - o) ** 2)
    se = errs.std() / np.sqrt(trials)
    assert abs(errs.mean() - pred) < 3 * se + 1e-4 * pred, (errs.mean(), pred, se)
