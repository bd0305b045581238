"""Offline OSCAR calibration (host, numpy fp64): rotations and clip thresholds.

edge.aivizor.me "Together AI выпустила исходники OSCAR ...", paragraph
"Техническая идея": C_Q = (1/N) sum q_n^T q_n with eigenvectors U_Q for keys,
the score-weighted C_S = (1/N) V^T S^T S V with eigenvectors U_S for values.
gist.science "Resumen Técnico: OSCAR ...", §2.2 A: covariance estimation on a
small calibration set, spectral decomposition, R = U H_Had P_br, per-layer
clipping thresholds from the rotated calibration activations.

Readings: eigenvectors by descending eigenvalue; S = softmax(Q K^T sm_scale)
per KV head over that head's calibration keys, C_S averaged over heads; tau =
the 99.9th percentile (linear interpolation) of |x R| over all calibration
rows and channels of the layer.  The output feeds ``oscar_load_rotation``.
"""

import numpy as np


def fwht(X):
    """Orthonormal Walsh-Hadamard transform (Sylvester order) along the last axis, by butterflies."""
    Y = np.array(X, dtype=np.float64, copy=True)
    d = Y.shape[-1]
    h = 1
    while h < d:
        Y = Y.reshape(Y.shape[:-1] + (d // (2 * h), 2, h))
        a = Y[..., 0, :].copy()
        b = Y[..., 1, :].copy()
        Y[..., 0, :] = a + b
        Y[..., 1, :] = a - b
        Y = Y.reshape(Y.shape[:-3] + (d,))
        h *= 2
    return Y / np.sqrt(d)


def bit_reversal_indices(d):
    nb = d.bit_length() - 1
    return np.array([int(format(j, "0%db" % nb)[::-1], 2) for j in range(d)], dtype=np.int64)


def rotate(X, U, use_u=True, use_h=True, use_p=True):
    """x' = x U H P for rows x; (x P)[j] = x[br(j)]."""
    Y = np.asarray(X, dtype=np.float64)
    if use_u:
        Y = Y @ np.asarray(U, dtype=np.float64)
    if use_h:
        Y = fwht(Y)
    if use_p:
        Y = Y[..., bit_reversal_indices(Y.shape[-1])]
    return Y


def descending_eigenvectors(C):
    w, V = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    idx = np.argsort(-w, kind="stable")
    return V[:, idx], w[idx]


def calibrate_layer(Q, K_heads, V_heads, sm_scale=1.0 / np.sqrt(128.0), percentile=99.9,
                    flags=(True, True, True)):
    """(U_K, U_V, tau_k, tau_v) of one layer from calibration queries and per-head keys/values."""
    Q = np.asarray(Q, dtype=np.float64)
    n = Q.shape[0]
    C_Q = (Q.T @ Q) / n
    C_S = np.zeros_like(C_Q)
    for K, V in zip(K_heads, V_heads):
        logits = (Q @ np.asarray(K, dtype=np.float64).T) * sm_scale
        logits -= logits.max(axis=1, keepdims=True)
        S = np.exp(logits)
        S /= S.sum(axis=1, keepdims=True)
        O = S @ np.asarray(V, dtype=np.float64)
        C_S += (O.T @ O) / n
    C_S /= len(K_heads)
    U_K, _ = descending_eigenvectors(C_Q)
    U_V, _ = descending_eigenvectors(C_S)
    rk = np.concatenate([rotate(K, U_K, *flags) for K in K_heads])
    rv = np.concatenate([rotate(V, U_V, *flags) for V in V_heads])
    tau_k = float(np.percentile(np.abs(rk), percentile))
    tau_v = float(np.percentile(np.abs(rv), percentile))
    return U_K, U_V, tau_k, tau_v


def synthetic_layer_rotation(cfg, layer, n_kv_heads, n_cal=2048, n_keys=2048, flags=(True, True, True)):
    """Calibrate one layer on seeded synthetic calibration data (the pages' calibration
    set of real activations is not available; the generators stand in for it)."""
    from . import inputs
    Q = inputs.queries(cfg, layer, inputs.STREAM_Q_CAL, n_cal)
    Ks = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 0).astype(np.float64)
          for h in range(n_kv_heads)]
    Vs = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 1).astype(np.float64)
          for h in range(n_kv_heads)]
    return calibrate_layer(Q, Ks, Vs, flags=flags)
