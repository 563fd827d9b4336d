"""Pins for oracle.rotation against closed forms, an independent algorithm and invariants.

R = U · Hadamard · bit-reversal ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化",
section "OSCAR 的设计"); U from Q^T Q for keys and V^T S^T S V for values (same section).
"""
import numpy as np
import pytest
import torch

from oracle import rotation as rot
import synth


def test_bitrev_known_values_and_involution():
    assert list(rot.bitrev_permutation(8)) == [0, 4, 2, 6, 1, 5, 3, 7]
    assert list(rot.bitrev_permutation(4)) == [0, 2, 1, 3]
    p = rot.bitrev_permutation(128)
    assert np.array_equal(p[p], np.arange(128))
    assert p[1] == 64 and p[3] == 96 and p[127] == 127


def test_bitrev_matrix_action():
    x = np.arange(16.0) * 3 + 1
    P = rot.bitrev_matrix(16)
    assert np.array_equal(x @ P, x[rot.bitrev_permutation(16)])


def test_hadamard_closed_form_natural_order():
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]) / 2.0
    assert np.array_equal(rot.hadamard(4), H4)
    H = rot.hadamard(128)
    assert np.all(np.abs(np.abs(H) - 1 / np.sqrt(128)) == 0)
    assert np.max(np.abs(H @ H - np.eye(128))) < 1e-14       # symmetric and orthogonal
    # Sylvester recursion H_2n = [[H, H], [H, -H]] / sqrt(2)
    H64 = rot.hadamard(64)
    assert np.max(np.abs(H - np.block([[H64, H64], [H64, -H64]]) / np.sqrt(2))) < 1e-15


def _gram_schmidt(A):
    """Modified Gram-Schmidt with one re-orthogonalisation pass: Q with positive R diagonal."""
    A = np.array(A, dtype=np.float64)
    n = A.shape[1]
    Q = np.zeros_like(A)
    for j in range(n):
        v = A[:, j].copy()
        for _ in range(2):
            for i in range(j):
                v -= (Q[:, i] @ v) * Q[:, i]
        Q[:, j] = v / np.linalg.norm(v)
    return Q


def test_haar_matches_gram_schmidt():
    G = synth.gaussian_matrix(7, 128)
    U = rot.haar_orthogonal(G)
    assert np.max(np.abs(U @ U.T - np.eye(128))) < 1e-12
    assert np.max(np.abs(U - _gram_schmidt(G))) < 1e-10
    Rq = U.T @ G                                      # upper triangular, positive diagonal
    assert np.max(np.abs(np.tril(Rq, -1))) < 1e-10
    assert np.all(np.diag(Rq) > 0)


def test_compose_identity_closed_form():
    d = 16
    R = rot.compose(np.eye(d))
    perm = rot.bitrev_permutation(d)
    for i in range(d):
        for j in range(d):
            sign = -1.0 if bin(i & perm[j]).count("1") % 2 else 1.0
            assert R[i, j] == sign / 4.0


@pytest.mark.parametrize("seed", [1, 2])
def test_rotation_orthogonal_and_preserves_dot(seed):
    R = rot.rotation_from_gaussian(synth.gaussian_matrix(seed, 128))
    assert np.max(np.abs(R @ R.T - np.eye(128))) < 1e-12
    g = np.random.default_rng(seed)
    q, k = g.standard_normal(128) * 5, g.standard_normal(128) * 5
    assert abs((q @ R) @ (k @ R) - q @ k) <= 1e-12 * np.linalg.norm(q) * np.linalg.norm(k)


def test_eigenvectors_known_decomposition():
    d = 128
    V0 = rot.haar_orthogonal(synth.gaussian_matrix(11, d))
    lam = 1.0 / (np.arange(d) + 1.0) + 0.5                 # distinct, descending
    C = (V0 * lam) @ V0.T
    w, U = rot.canonical_eigenvectors(C)
    assert np.allclose(w, lam, rtol=0, atol=1e-12)
    # same columns up to sign, then the sign rule
    for j in range(d):
        col = V0[:, j] * (1 if V0[np.argmax(np.abs(V0[:, j])), j] > 0 else -1)
        assert np.max(np.abs(U[:, j] - col)) < 1e-9
        assert U[np.argmax(np.abs(U[:, j])), j] > 0
    res = np.max(np.abs(C @ U - U * w))
    assert res <= 1e-10 * np.max(np.abs(C))


def test_covariance_k_is_sum_of_outer_products():
    g = np.random.default_rng(3)
    Q = g.standard_normal((50, 2, 8))
    C = rot.covariance_k(Q)
    ref = sum(np.outer(Q[t, h], Q[t, h]) for t in range(50) for h in range(2))
    assert np.max(np.abs(C - ref)) < 1e-12


def test_covariance_v_against_library_causal_attention():
    g = np.random.default_rng(4)
    T, H, d = 40, 3, 16
    Q, K, V = g.standard_normal((T, H, d)), g.standard_normal((T, d)), g.standard_normal((T, d))
    C = rot.covariance_v(Q, K, V)
    ref = np.zeros((d, d))
    for h in range(H):
        q = torch.from_numpy(Q[:, h, :])[None, None]
        O = torch.nn.functional.scaled_dot_product_attention(
            q, torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None], is_causal=True)[0, 0].numpy()
        ref += O.T @ O
    assert np.max(np.abs(C - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_f32_copy_is_nearest():
    R = rot.rotation_from_gaussian(synth.gaussian_matrix(5, 32))
    R32 = rot.to_f32(R)
    up = np.nextafter(R32, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(R32, np.float32(-np.inf)).astype(np.float64)
    err = np.abs(R32.astype(np.float64) - R)
    assert np.all(err <= np.abs(up - R)) and np.all(err <= np.abs(dn - R))
