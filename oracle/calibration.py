"""Offline calibration: C_Q, C_S, eigenbases, clip thresholds (fp64).

Oracle; test infrastructure only.

[RU] "Техническая идея": for keys, C_Q = (1/N) sum_n q_n^T q_n and its
eigenvectors U_Q form the rotation basis; for values, the score-weighted
covariance C_S = (1/N) V^T S^T S V and its eigenvectors U_S.
[ES] §2.2 A steps 1-4: estimate C_Q and C_S on a small calibration set,
decompose them spectrally, compose R = U H P, estimate per-layer clipping
thresholds from the rotated calibration activations.
[ES] §2.1: logit distortion is governed by Q^T Q; output distortion is
weighted by the attention scores S, giving V^T S^T S V.

Readings:

* q_n are row vectors; N = number of calibration queries.
* S = softmax(Q K^T * sm_scale) row-wise over the calibration keys of one KV
  head (no causal mask), so S V is the attention output of the calibration
  queries; with several KV heads C_S averages (1/N) (S_h V_h)^T (S_h V_h)
  over the heads.  One (R_K, R_V, tau_K, tau_V) per layer, shared by its
  KV heads.
* Eigenvectors are sorted by descending eigenvalue (order and signs do not
  change R's validity, only which rotation is chosen).
* tau is the 99.9th percentile of |x R| over all calibration rows and
  channels of the layer (numpy's linear interpolation).
"""

import numpy as np

from . import rotation


def query_covariance(Q):
    """C_Q = (1/N) sum_n q_n^T q_n for rows q_n of Q [N, d]."""
    Q = np.asarray(Q, dtype=np.float64)
    return Q.T @ Q / Q.shape[0]


def score_weighted_value_covariance(Q, K_heads, V_heads, sm_scale):
    """C_S = (1/N) V^T S^T S V averaged over KV heads, S = softmax(Q K^T sm_scale)."""
    Q = np.asarray(Q, dtype=np.float64)
    N, d = Q.shape
    C = np.zeros((d, d))
    for K, V in zip(K_heads, V_heads):
        z = (Q @ np.asarray(K, dtype=np.float64).T) * sm_scale
        z = z - z.max(axis=1, keepdims=True)
        S = np.exp(z)
        S = S / S.sum(axis=1, keepdims=True)
        O = S @ np.asarray(V, dtype=np.float64)
        C += O.T @ O / N
    return C / len(K_heads)


def eigenbasis(C):
    """Eigenvectors of a symmetric C as columns, by descending eigenvalue."""
    w, U = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    order = np.argsort(w)[::-1]
    return U[:, order], w[order]


def clip_threshold(X_rot, percentile=99.9):
    """tau = the given percentile of |X_rot| over all entries."""
    return float(np.percentile(np.abs(np.asarray(X_rot, dtype=np.float64)), percentile))


def calibrate_layer(Q, K_heads, V_heads, sm_scale, percentile=99.9, flags=(True, True, True)):
    """U_K, U_V (fp64 [d, d]) and tau_K, tau_V for one layer."""
    U_K, _ = eigenbasis(query_covariance(Q))
    U_V, _ = eigenbasis(score_weighted_value_covariance(Q, K_heads, V_heads, sm_scale))
    R_K = rotation.composite_rotation(U_K, *flags)
    R_V = rotation.composite_rotation(U_V, *flags)
    tau_k = clip_threshold(np.concatenate([rotation.rotate(K, R_K) for K in K_heads]), percentile)
    tau_v = clip_threshold(np.concatenate([rotation.rotate(V, R_V) for V in V_heads]), percentile)
    return U_K, U_V, tau_k, tau_v
