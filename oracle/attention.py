"""Decode attention over the mixed cache, fp64 (oracle; test infrastructure only).

[IT] "Architettura del Sistema di Serving": the read kernel unpacks,
dequantises and undoes the rotation in one pass.  [ES] §2.2 B: the fused
kernel handles unpacking, de-quantisation, inverse rotation and the attention
computation for the INT2 history.  Because R is orthogonal, attention over
the dequantised, rotated-back history equals the plain definition
softmax(q K^T * scale) V over K_hat = x_hat'_K R_K^T and V_hat = x_hat'_V R_V^T;
the oracle computes exactly that definition.

Readings: sm_scale = 1/sqrt(128); query head h reads KV head h // g with
g = H_q / H_kv (consecutive query heads share a KV head); the output is fp32
(the hot path's output type) and is computed here in fp64.  A request with no
context (L = 0) has output 0.
"""

import numpy as np


def softmax_attention(q, K, V, sm_scale):
    """out[h] = sum_t softmax_t(q[h] . K[t] * sm_scale) V[t], fp64.

    The row maximum is subtracted before exponentiating; this changes no
    value of the softmax and keeps exp() finite.
    """
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    z = (q @ K.T) * sm_scale
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ V


def decode_gqa(q, K_heads, V_heads, sm_scale):
    """Decode output for one request.

    q: [H_q, d];  K_heads, V_heads: lists (one per KV head) of [L, d] arrays.
    Returns out [H_q, d] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    H_q = q.shape[0]
    H_kv = len(K_heads)
    g = H_q // H_kv
    out = np.zeros_like(q)
    for h in range(H_kv):
        out[h * g:(h + 1) * g] = softmax_attention(q[h * g:(h + 1) * g], K_heads[h], V_heads[h], sm_scale)
    return out
