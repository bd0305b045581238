"""GPU calibration (C_Q, C_S, clip thresholds) against the oracle's calibration.

[RU] "Техническая идея": C_Q = (1/N) sum q^T q, C_S = (1/N) V^T S^T S V;
[ES] §2.2 A steps 1-4: covariances, spectral decomposition on the host,
per-layer clip thresholds (here the 99.9th percentile of |x R|).  The GPU
sums fp32 products in fp64 across 32-row stages and runs the calibration
attention in fp32, so the covariances agree with the fp64 oracle to ~1e-6
of their largest entry; the thresholds are order statistics of |x R| with x R
in fp32 (error ~1e-7 of the largest |x R| against the oracle's fp64 rotation).
"""

import numpy as np
import pytest
import torch

from int2_rotated_kv_oscar_gb300 import abi, calibrate, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import calibration as ocal  # noqa: E402
from oracle import rotation as orot  # noqa: E402

SM = 1.0 / np.sqrt(128.0)
COV_TOL = 2e-6   # max |C_gpu - C_oracle| / max |C_oracle|
TAU_TOL = 5e-6   # relative


@pytest.fixture(scope="module")
def ctx():
    c = abi.oscar_create(abi.oscar_config(num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64,
                                          sink=64, recent=256, group=64, device=0))
    yield c
    abi.oscar_destroy(c)


def _data(cfg, n_q, n_k, heads, layer=0):
    Q = inputs.queries(cfg, layer, inputs.STREAM_Q_CAL, n_q).astype(np.float32)
    Ks = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_k, 0).astype(np.float32) for h in range(heads)]
    Vs = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_k, 1).astype(np.float32) for h in range(heads)]
    return Q, Ks, Vs


def _device(Q, Ks, Vs):
    q = torch.from_numpy(Q).cuda()
    k = torch.from_numpy(np.stack(Ks)).cuda()
    v = torch.from_numpy(np.stack(Vs)).cuda()
    return q, k, v


def _rel(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.mark.parametrize("n_q,n_k,heads", [(200, 150, 3), (33, 1, 1), (2048, 2048, 8)])
def test_covariances_match_the_oracle(ctx, n_q, n_k, heads):
    Q, Ks, Vs = _data(21, n_q, n_k, heads)
    q, k, v = _device(Q, Ks, Vs)
    ws = calibrate.CalibWorkspace(n_q, n_k, heads, heads * n_k)
    C_Q, C_S = calibrate.covariances(ctx, q, k, v, SM, ws)
    rq = _rel(C_Q, ocal.query_covariance(Q.astype(np.float64)))
    rs = _rel(C_S, ocal.score_weighted_value_covariance(Q.astype(np.float64), [x.astype(np.float64) for x in Ks],
                                                         [x.astype(np.float64) for x in Vs], SM))
    print("C_Q rel %.2e, C_S rel %.2e" % (rq, rs))
    assert rq <= COV_TOL and rs <= COV_TOL
    assert np.allclose(C_Q, C_Q.T, rtol=0, atol=1e-12 * np.abs(C_Q).max())


@pytest.mark.parametrize("flags", [(True, True, True), (False, False, False), (False, True, True), (True, False, False)])
@pytest.mark.parametrize("pct", [99.9, 50.0, 0.0, 100.0])
def test_clip_threshold_matches_the_oracle(ctx, flags, pct):
    rng = np.random.default_rng(5)
    n_rows = 777  # not a power of two: the sort pads with +inf
    X = (rng.standard_normal((n_rows, 128)) * np.where(rng.random(128) < 0.05, 20.0, 1.0)).astype(np.float32)
    U = np.linalg.qr(rng.standard_normal((128, 128)))[0].astype(np.float32)
    ws = calibrate.CalibWorkspace(1, 1, 1, n_rows)
    tau = calibrate.clip_threshold(ctx, torch.from_numpy(X).cuda(), U, flags, pct, ws)
    R = orot.composite_rotation(U.astype(np.float64), *flags)
    Y = orot.rotate(X.astype(np.float64), R)
    ref = ocal.clip_threshold(Y, pct)
    print("flags %s pct %.1f: tau %.8g ref %.8g" % (flags, pct, tau, ref))
    # x R in fp32: each entry is off by up to ~1e-7 of the row's magnitude, so
    # small order statistics get an absolute bound
    assert abs(tau - ref) <= TAU_TOL * abs(ref) + 1e-6 * np.abs(Y).max()


def test_calibrated_layer_matches_the_oracle(ctx):
    """The whole layer: C_Q, C_S on the GPU, eigh on the host, both thresholds on the GPU."""
    Q, Ks, Vs = _data(22, 2048, 1024, 8)
    U_K, U_V, tk, tv = calibrate.calibrate_layer(ctx, Q, Ks, Vs, SM)
    f64 = [x.astype(np.float64) for x in Ks], [x.astype(np.float64) for x in Vs]
    # thresholds of the GPU's own bases, by the oracle
    R_K = orot.composite_rotation(U_K.astype(np.float64))
    R_V = orot.composite_rotation(U_V.astype(np.float64))
    ref_k = ocal.clip_threshold(np.concatenate([orot.rotate(K, R_K) for K in f64[0]]), 99.9)
    ref_v = ocal.clip_threshold(np.concatenate([orot.rotate(V, R_V) for V in f64[1]]), 99.9)
    assert abs(tk - ref_k) <= TAU_TOL * ref_k and abs(tv - ref_v) <= TAU_TOL * ref_v
    # the bases are orthonormal eigenbases of the oracle's covariances (eigenvalues descending)
    C_Q = ocal.query_covariance(Q.astype(np.float64))
    C_S = ocal.score_weighted_value_covariance(Q.astype(np.float64), f64[0], f64[1], SM)
    for U, C in ((U_K, C_Q), (U_V, C_S)):
        U = U.astype(np.float64)
        assert np.abs(U.T @ U - np.eye(128)).max() < 1e-5
        lam = np.diag(U.T @ C @ U)
        assert np.all(np.diff(lam) <= 1e-5 * lam[0])
        off = U.T @ C @ U - np.diag(lam)
        assert np.abs(off).max() <= 1e-4 * lam[0]


def test_calibration_argument_errors(ctx):
    ws = calibrate.CalibWorkspace(16, 16, 1, 16)
    x = torch.zeros((16, 128), dtype=torch.float32, device="cuda")
    U = np.eye(128, dtype=np.float32)
    with pytest.raises(abi.OscarError) as e:
        abi.oscar_calib_clip_threshold(ctx, x, 16, U, abi.OSCAR_ROT_ALL, 100.5, ws.ptr, ws.bytes)
    assert e.value.status == 1  # OSCAR_ERR_INVALID_ARG
    with pytest.raises(abi.OscarError) as e:
        abi.oscar_calib_clip_threshold(ctx, x, 16, U, abi.OSCAR_ROT_ALL, 50.0, ws.ptr, 16)
    assert e.value.status == 6  # OSCAR_ERR_WORKSPACE
    c = torch.empty((2, 128, 128), dtype=torch.float64, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        abi.oscar_calib_covariances(ctx, x, 16, x, x, 16, 1, -1.0, c[0], c[1], ws.ptr, ws.bytes)
    assert e.value.status == 1  # OSCAR_ERR_INVALID_ARG
    # a zero input gives a zero threshold and zero covariances
    assert calibrate.clip_threshold(ctx, x, U, (True, True, True), 99.9, ws) == 0.0
    C_Q, C_S = calibrate.covariances(ctx, x, x.view(1, 16, 128), x.view(1, 16, 128), 0.1, ws)
    assert not C_Q.any() and not C_S.any()
