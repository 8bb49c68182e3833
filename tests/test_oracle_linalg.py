"""Pins for the oracle's statistics, Jacobi eigensolver and key transform.

Each check uses something other than the oracle itself: numpy's covariance
and LAPACK eigh as library cross-checks, brute-force loops, and the algebraic
identities the pages state (KLT decorrelation, generalized Parseval).
"""
import numpy as np
import pytest

import oracle


def _spd(d, seed, decay=0.9):
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return (Q * decay ** np.arange(d)) @ Q.T


def test_mean_and_moment_match_bruteforce_and_numpy():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((300, 7)) * np.arange(1, 8) + 3.0
    mu = oracle.mean(X)
    assert np.allclose(mu, [sum(X[i, j] for i in range(300)) / 300 for j in range(7)], rtol=1e-14)
    S = oracle.moment(X, mu)
    assert np.allclose(S, np.cov(X.T, bias=True), rtol=1e-12, atol=1e-12)
    # uncentered second moment by a plain double loop
    M = oracle.moment(X)
    brute = np.array([[sum(X[i, a] * X[i, b] for i in range(300)) / 300 for b in range(7)]
                      for a in range(7)])
    assert np.allclose(M, brute, rtol=1e-13)
    assert np.allclose(S, S.T) and np.linalg.eigvalsh(S).min() > 0


@pytest.mark.parametrize("d,seed", [(5, 0), (32, 1), (128, 2)])
def test_jacobi_against_lapack(d, seed):
    A = _spd(d, seed)
    w, V, sweeps = oracle.jacobi_eig(A)
    assert sweeps > 0
    ref = np.linalg.eigvalsh(A)[::-1]
    # LAPACK is backward stable: its eigenvalues are good to ~eps*|A| in absolute terms
    assert np.max(np.abs(w - ref)) < 1e-12 * ref[0]
    big = ref > 1e-3 * ref[0]
    assert np.max(np.abs(w - ref)[big] / ref[big]) < 1e-11
    assert np.linalg.norm(A @ V - V * w) <= 1e-12 * np.linalg.norm(A)
    assert np.linalg.norm(V.T @ V - np.eye(d)) <= 1e-13 * d
    assert np.all(np.diff(w) <= 0)
    # sign convention: the largest-magnitude entry of each eigenvector is positive
    idx = np.argmax(np.abs(V), axis=0)
    assert np.all(V[idx, np.arange(d)] > 0)


def test_jacobi_ties_and_nonconvergence():
    w, V, s = oracle.jacobi_eig(np.diag([1.0, 3.0, 3.0, 2.0]))
    assert list(w) == [3.0, 3.0, 2.0, 1.0]
    # equal eigenvalues keep the original index order
    assert np.allclose(V[:, 0], [0, 1, 0, 0]) and np.allclose(V[:, 1], [0, 0, 1, 0])
    # one sweep is not enough for a dense 64x64 matrix
    _, _, s = oracle.jacobi_eig(_spd(64, 3), max_sweeps=1)
    assert s == -1


def test_key_transform_decorrelates_and_whitens():
    d = 64
    Sk = _spd(d, 4, 0.93)
    Sq = _spd(d, 5, 0.95)
    kt = oracle.key_transform(Sk, Sq)
    assert kt["ok"]
    T, Ti, A = kt["T"], kt["T_inv"], kt["A"]
    # KLT decorrelation: off-diagonal coefficient covariance below 1e-6 of the trace
    C = T @ Sk @ T.T
    off = C - np.diag(np.diag(C))
    assert np.abs(off).max() < 1e-6 * np.trace(C)
    assert np.allclose(np.diag(C), kt["lam"], rtol=1e-10)
    # generalized Parseval: T^{-T} Sq T^{-1} = I, so E_q[(q . T^{-1} e)^2] = |e|^2
    P = Ti.T @ Sq @ Ti
    assert np.abs(P - np.eye(d)).max() < 1e-10
    assert np.allclose(Ti @ T, np.eye(d), atol=1e-10)
    assert np.allclose(A, np.linalg.inv(T).T, atol=1e-9)
    # lam = eigenvalues of Sq^{1/2} Sk Sq^{1/2} = eigenvalues of Sk Sq
    ref = np.sort(np.linalg.eigvals(Sk @ Sq).real)[::-1]
    assert np.allclose(kt["lam"], ref, rtol=1e-9)


def test_identity_query_metric_reduces_to_plain_klt():
    """With Sq = I the key transform is the orthogonal KLT U^T of Sk."""
    d = 16
    Sk = _spd(d, 6)
    kt = oracle.key_transform(Sk, np.eye(d))
    w, U, _ = oracle.jacobi_eig(Sk)
    assert np.allclose(kt["T"], U.T, atol=1e-12)
    assert np.allclose(kt["lam"], w, rtol=1e-12)
