"""OSCAR composite rotation, fp64 (oracle; test infrastructure only).

[ES] §2.2 A step 3 and [RU] composition paragraph: the final rotations are
products of three factors, R_K = U_Q * H_Had * P_br and R_V = U_S * H_Had * P_br.
[IT] "I tre fattori della rotazione": U aligns channels with the attention
importance directions, H_Had (Walsh-Hadamard) equalises channel importance,
P_br (bit reversal) reorders channels so every quantisation group gets a
balanced share of the importance hierarchy.

Readings (the pages leave these open):

* H_Had is the Sylvester-ordered Walsh-Hadamard matrix normalised to be
  orthogonal: H[i, j] = (-1)^popcount(i & j) / sqrt(d).
* P_br acts on a row vector by (x P)[j] = x[br(j)], br = reversal of the
  log2(d) index bits.  br is an involution, so P = P^T = P^-1 and the other
  convention gives the same matrix.
* Vectors are rows (the pages write C_Q = (1/N) sum q_n^T q_n for row vectors
  q_n), so a token x is rotated as x' = x R.
"""

import numpy as np


def popcount(a):
    """Number of set bits of each element of an integer array."""
    a = np.asarray(a, dtype=np.int64)
    count = np.zeros_like(a)
    while np.any(a):
        count += a & 1
        a = a >> 1
    return count


def hadamard(d=128):
    """Orthogonal Sylvester Walsh-Hadamard matrix of size d (a power of two).

    H[i, j] = (-1)^popcount(i & j) / sqrt(d)   ([IT] "I tre fattori", item 2;
    [ES] §2.2 A step 3, H_Had).
    """
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    parity = popcount(np.bitwise_and.outer(i, i)) % 2
    return np.where(parity == 0, 1.0, -1.0) / np.sqrt(d)


def bit_reverse(j, nbits=7):
    """Reverse the low ``nbits`` bits of index j ([ES] §2.2 A step 3, P_br)."""
    out = 0
    for b in range(nbits):
        if (j >> b) & 1:
            out |= 1 << (nbits - 1 - b)
    return out


def bit_reversal_matrix(d=128):
    """Permutation matrix P_br with (x @ P)[j] = x[br(j)]."""
    nbits = d.bit_length() - 1
    if 1 << nbits != d:
        raise ValueError("d must be a power of two")
    P = np.zeros((d, d))
    for j in range(d):
        P[bit_reverse(j, nbits), j] = 1.0
    return P


def composite_rotation(U, use_u=True, use_h=True, use_p=True):
    """R = U * H_Had * P_br in fp64 ([RU] composition paragraph; [ES] §2.2 A.3).

    ``U`` is the eigenbasis (columns are eigenvectors), given as data.  The
    three flags drop a factor (replace it by the identity) for the ablations
    the pages compare against: R = I is naive INT2, R = H P is Hadamard-only.
    """
    U = np.asarray(U, dtype=np.float64)
    d = U.shape[0]
    R = U.copy() if use_u else np.eye(d)
    if use_h:
        R = R @ hadamard(d)
    if use_p:
        R = R @ bit_reversal_matrix(d)
    return R


def rotate(X, R):
    """Rotate row vectors: X' = X R (fp64)."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64)


def unrotate(Xr, R):
    """Undo the rotation: X = X' R^T (R orthogonal)."""
    return np.asarray(Xr, dtype=np.float64) @ np.asarray(R, dtype=np.float64).T
