"""Oracle: the fixed per-(layer, head) rotation R = U · H · P (test infrastructure only).

[Article, "OSCAR 的设计"]: the final rotation is written R = U · Hadamard ·
bit-reversal; U aligns the directions attention uses, the Hadamard spreads
outlier energy, the bit-reversal balances the INT2 groups.  For keys U comes
from the query covariance Q^T Q (key error enters the logits through QK^T); for
values from the score-weighted value covariance V^T S^T S V.
[Abstract, "摘要"]: the covariances are estimated offline from a light
calibration pass and yield fixed orthogonal rotations.

Readings (the pages leave these open):
* Row-vector convention: a head vector x (1 x d) is rotated as x_rot = x · R.
* H is the Sylvester (natural-order) Walsh-Hadamard matrix normalised by
  1/sqrt(d): H[i][j] = (-1)^popcount(i & j) / sqrt(d).
* P is the bit-reversal permutation on log2(d) bits: (x · P)[i] = x[bitrev(i)].
* Haar U: the Q factor of the QR decomposition of a d x d standard-normal
  matrix, with each column multiplied by the sign of R_qr's diagonal entry so
  that the factorisation is unique (R_qr has a positive diagonal).
* Covariance U: eigenvectors of the symmetric covariance, columns ordered by
  descending eigenvalue, each column's sign chosen so that its entry of largest
  magnitude is positive (the lowest index wins a tie in magnitude).
* C_k = sum over the query heads h of a KV group of Q_h^T Q_h.
* C_v = sum over those heads of (S_h V)^T (S_h V) with S_h the causal
  row-softmax of Q_h K^T / sqrt(d) (the page's V^T S^T S V; the Chinese
  summary's garbled "VSS^T" is read the same way).
"""
from __future__ import annotations

import numpy as np


def bitrev(i: int, bits: int) -> int:
    """Reverse the low `bits` bits of i."""
    r = 0
    for _ in range(bits):
        r = (r << 1) | (i & 1)
        i >>= 1
    return r


def bitrev_permutation(d: int) -> np.ndarray:
    bits = d.bit_length() - 1
    assert 1 << bits == d, "d must be a power of two"
    return np.array([bitrev(i, bits) for i in range(d)], dtype=np.int64)


def bitrev_matrix(d: int) -> np.ndarray:
    """P with (x @ P)[i] == x[bitrev(i)]: column i holds a one in row bitrev(i)."""
    perm = bitrev_permutation(d)
    P = np.zeros((d, d))
    for i in range(d):
        P[perm[i], i] = 1.0
    return P


def hadamard(d: int) -> np.ndarray:
    """Normalised Sylvester Hadamard matrix, written entry by entry from its closed form."""
    H = np.empty((d, d))
    for i in range(d):
        for j in range(d):
            H[i, j] = -1.0 if bin(i & j).count("1") % 2 else 1.0
    return H / np.sqrt(d)


def haar_orthogonal(gauss: np.ndarray) -> np.ndarray:
    """Q of QR(gauss) with columns sign-fixed so R_qr has a positive diagonal."""
    Q, Rq = np.linalg.qr(np.asarray(gauss, np.float64))
    sgn = np.sign(np.diag(Rq))
    sgn[sgn == 0] = 1.0
    return Q * sgn[None, :]


def canonical_eigenvectors(C: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(eigenvalues descending, U with matching columns), sign rule as in the module docstring."""
    C = np.asarray(C, np.float64)
    w, V = np.linalg.eigh(C)
    order = np.argsort(-w, kind="stable")
    w, V = w[order], V[:, order].copy()
    for j in range(V.shape[1]):
        k = int(np.argmax(np.abs(V[:, j])))   # first index of the largest magnitude
        if V[k, j] < 0:
            V[:, j] = -V[:, j]
    return w, V


def compose(U: np.ndarray) -> np.ndarray:
    """R = U · H · P."""
    d = U.shape[0]
    return U @ hadamard(d) @ bitrev_matrix(d)


def rotation_from_gaussian(gauss: np.ndarray) -> np.ndarray:
    return compose(haar_orthogonal(gauss))


def rotation_from_covariance(C: np.ndarray) -> np.ndarray:
    return compose(canonical_eigenvectors(C)[1])


def to_f32(R64: np.ndarray) -> np.ndarray:
    """The device copy of R: each entry rounded to the nearest float32."""
    return np.asarray(R64, np.float64).astype(np.float32)


def covariance_k(Q: np.ndarray) -> np.ndarray:
    """C_k = sum_h Q_h^T Q_h for Q of shape [T][heads][d] (float64 values)."""
    Q = np.asarray(Q, np.float64)
    d = Q.shape[2]
    C = np.zeros((d, d))
    for h in range(Q.shape[1]):
        C += Q[:, h, :].T @ Q[:, h, :]
    return C


def causal_softmax_scores(Qh: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """S[t][u] = softmax over u <= t of scale * Qh[t] . K[u]; zero above the diagonal."""
    T = Qh.shape[0]
    S = np.zeros((T, T))
    for t in range(T):
        s = (K[: t + 1] @ Qh[t]) * scale
        p = np.exp(s - s.max())
        S[t, : t + 1] = p / p.sum()
    return S


def covariance_v(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float | None = None) -> np.ndarray:
    """C_v = sum_h (S_h V)^T (S_h V); Q [T][heads][d], K and V [T][d] (one KV head)."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    d = Q.shape[2]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    C = np.zeros((d, d))
    for h in range(Q.shape[1]):
        O = causal_softmax_scores(Q[:, h, :], K, scale) @ V
        C += O.T @ O
    return C
