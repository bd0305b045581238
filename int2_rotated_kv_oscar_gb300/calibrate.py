"""Offline OSCAR calibration of one layer: rotations and clip thresholds.

edge.aivizor.me "Together AI выпустила исходники OSCAR ...", paragraph
"Техническая идея": C_Q = (1/N) sum q_n^T q_n with eigenvectors U_Q for keys,
the score-weighted C_S = (1/N) V^T S^T S V with eigenvectors U_S for values.
gist.science "Resumen Técnico: OSCAR ...", §2.2 A: covariance estimation on a
small calibration set, spectral decomposition, R = U H_Had P_br, per-layer
clipping thresholds from the rotated calibration activations.

The covariances and the thresholds run on the GPU through the C ABI
(``oscar_calib_covariances``, ``oscar_calib_clip_threshold``); the spectral
decomposition runs on the host (numpy ``eigh``, fp64).  Readings:
eigenvectors by descending eigenvalue; S = softmax(Q K^T sm_scale) per KV
head over that head's calibration keys, C_S averaged over heads; tau = the
99.9th percentile (linear interpolation) of |x R| over all calibration rows
and channels of the layer.  The output feeds ``oscar_load_rotation``.
"""

import numpy as np
import torch

from . import abi


def descending_eigenvectors(C):
    """Eigenvectors of a symmetric C as columns, by descending eigenvalue, and the eigenvalues."""
    w, V = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    idx = np.argsort(-w, kind="stable")
    return V[:, idx], w[idx]


def rotation_flags(flags):
    use_u, use_h, use_p = flags
    return (abi.OSCAR_ROT_U if use_u else 0) | (abi.OSCAR_ROT_H if use_h else 0) | (abi.OSCAR_ROT_P if use_p else 0)


class CalibWorkspace:
    """A device workspace for the calibration calls (256-byte aligned)."""

    def __init__(self, n_queries, n_keys, n_kv_heads, n_clip_rows, device="cuda"):
        self.bytes = abi.oscar_calib_workspace_bytes(n_queries, n_keys, n_kv_heads, n_clip_rows)
        if self.bytes == 0:
            raise ValueError("calibration sizes out of range")
        self.tensor = torch.empty(self.bytes + 256, dtype=torch.uint8, device=device)
        self.ptr = self.tensor.data_ptr() + (-self.tensor.data_ptr()) % 256


def covariances(ctx, q, k, v, sm_scale, ws, stream=None):
    """C_Q, C_S (host float64 [128, 128]) from device float32 q [N, 128] and k, v [heads, M, 128]."""
    n_q, n_k, heads = q.shape[0], k.shape[1], k.shape[0]
    c = torch.empty((2, 128, 128), dtype=torch.float64, device=q.device)
    abi.oscar_calib_covariances(ctx, q, n_q, k, v, n_k, heads, sm_scale, c[0], c[1], ws.ptr, ws.bytes,
                                stream or torch.cuda.current_stream(q.device))
    c = c.cpu().numpy()
    return c[0], c[1]


def clip_threshold(ctx, x, U, flags, percentile, ws, stream=None):
    """The percentile of |x R| over every entry of device float32 x [rows, 128], R = U H P (by flags)."""
    return abi.oscar_calib_clip_threshold(ctx, x, x.shape[0], U, rotation_flags(flags), percentile, ws.ptr, ws.bytes,
                                          stream or torch.cuda.current_stream(x.device))


def calibrate_layer(ctx, Q, K_heads, V_heads, sm_scale=1.0 / np.sqrt(128.0), percentile=99.9,
                    flags=(True, True, True), device="cuda"):
    """(U_K, U_V, tau_k, tau_v) of one layer from calibration queries and per-head keys/values.

    U_K, U_V are float32 [128, 128] (what ``oscar_load_rotation`` takes); the
    thresholds are computed with exactly those matrices."""
    q = torch.as_tensor(np.asarray(Q, dtype=np.float32), device=device).contiguous()
    k = torch.as_tensor(np.stack([np.asarray(x, dtype=np.float32) for x in K_heads]), device=device).contiguous()
    v = torch.as_tensor(np.stack([np.asarray(x, dtype=np.float32) for x in V_heads]), device=device).contiguous()
    heads, n_k = k.shape[0], k.shape[1]
    ws = CalibWorkspace(q.shape[0], n_k, heads, heads * n_k, device=device)
    C_Q, C_S = covariances(ctx, q, k, v, sm_scale, ws)
    U_K = descending_eigenvectors(C_Q)[0].astype(np.float32)
    U_V = descending_eigenvectors(C_S)[0].astype(np.float32)
    tau_k = clip_threshold(ctx, k.view(heads * n_k, 128), U_K, flags, percentile, ws)
    tau_v = clip_threshold(ctx, v.view(heads * n_k, 128), U_V, flags, percentile, ws)
    return U_K, U_V, tau_k, tau_v


def synthetic_layer_rotation(ctx, cfg, layer, n_kv_heads, n_cal=2048, n_keys=2048, flags=(True, True, True),
                             device="cuda"):
    """Calibrate one layer on seeded synthetic calibration data (the pages' calibration
    set of real activations is not available; the generators stand in for it)."""
    from . import inputs
    Q = inputs.queries(cfg, layer, inputs.STREAM_Q_CAL, n_cal)
    Ks = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 0) for h in range(n_kv_heads)]
    Vs = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 1) for h in range(n_kv_heads)]
    return calibrate_layer(ctx, Q, Ks, Vs, flags=flags, device=device)
