"""Pins of the oracle's rotation against what the pages and the mathematics fix.

Sources: ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit
per LLM" ("I tre fattori della rotazione"); edge.aivizor.me "Together AI
выпустила исходники OSCAR ..." (composition paragraph: R = U H P; deployment
paragraph: the lemma diag(H^T Lambda H) = tr(Lambda)/d); gist.science
"Resumen Técnico: OSCAR ..." §2.2 A.
"""

import os

import numpy as np
import pytest

from oracle import calibration, rotation


def _read_hadamards(path):
    mats, cur, d = {}, None, None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("d "):
            d = int(line.split()[1])
            cur = mats.setdefault(d, [])
            continue
        cur.append([float(x) for x in line.split()])
    return {k: np.array(v) for k, v in mats.items()}


def test_hadamard_matches_textbook_sylvester(golden_dir):
    for d, M in _read_hadamards(os.path.join(golden_dir, "hadamard_sylvester.txt")).items():
        assert np.array_equal(rotation.hadamard(d) * np.sqrt(d), M)


def test_hadamard_recursive_construction():
    # H_2d = [[H_d, H_d], [H_d, -H_d]] / sqrt(2): the Sylvester recursion.
    for d in (1, 2, 4, 8, 16, 32, 64):
        H = rotation.hadamard(d)
        H2 = np.block([[H, H], [H, -H]]) / np.sqrt(2)
        assert np.allclose(rotation.hadamard(2 * d), H2, atol=1e-15)


def test_hadamard_orthogonal_and_entries():
    H = rotation.hadamard(128)
    assert np.abs(H.T @ H - np.eye(128)).max() < 1e-13
    assert np.allclose(np.abs(H), 1 / np.sqrt(128))


def test_lemma_diag_equalised():
    # Lemma (deployment paragraph of the edge.aivizor.me page):
    # diag(H^T Lambda H) = tr(Lambda) / d for any diagonal Lambda.
    r = np.random.default_rng(1)
    H = rotation.hadamard(128)
    for _ in range(5):
        lam = np.diag(r.exponential(size=128) * 10)
        dg = np.diag(H.T @ lam @ H)
        assert np.abs(dg - np.trace(lam) / 128).max() < 1e-12


def test_bit_reversal_golden(golden_dir):
    for line in open(os.path.join(golden_dir, "bit_reversal.txt")):
        if line.startswith("#") or not line.strip():
            continue
        nbits, j, br = (int(x) for x in line.split())
        assert rotation.bit_reverse(j, nbits) == br


def test_bit_reversal_permutation_involution():
    br = [rotation.bit_reverse(j, 7) for j in range(128)]
    assert sorted(br) == list(range(128))
    assert all(rotation.bit_reverse(b, 7) == j for j, b in enumerate(br))
    P = rotation.bit_reversal_matrix(128)
    assert np.array_equal(P, P.T)
    assert np.array_equal(P @ P, np.eye(128))


def test_bit_reversal_acts_on_row_vectors():
    # (x P)[j] = x[br(j)]: a one-hot at channel 1 moves to channel 64.
    P = rotation.bit_reversal_matrix(128)
    x = np.zeros(128)
    x[1] = 1.0
    y = x @ P
    assert y[64] == 1.0 and y.sum() == 1.0
    x = np.arange(128.0)
    assert np.array_equal(x @ P, np.array([rotation.bit_reverse(j, 7) for j in range(128)], dtype=float))


def _random_orthogonal(seed, d=128):
    a = np.random.default_rng(seed).standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))


def test_composite_rotation_orthogonal():
    # I1: R = U H P is orthogonal (product of orthogonal factors).
    for s in range(3):
        R = rotation.composite_rotation(_random_orthogonal(s))
        assert np.abs(R.T @ R - np.eye(128)).max() < 1e-12


def test_composite_rotation_flags():
    U = _random_orthogonal(7)
    assert np.array_equal(rotation.composite_rotation(U, False, False, False), np.eye(128))
    assert np.allclose(rotation.composite_rotation(U, True, False, False), U)
    assert np.allclose(rotation.composite_rotation(U, False, True, True),
                       rotation.hadamard(128) @ rotation.bit_reversal_matrix(128))


def _decaying_queries(seed, n=4096, d=128):
    r = np.random.default_rng(seed)
    B = _random_orthogonal(seed + 100, d)
    sig = np.exp(-np.arange(d) / 32.0)
    return (r.standard_normal((n, d)) * sig) @ B.T


def test_rotated_query_covariance_has_equal_diagonal():
    # The lemma applied to the whole rotation: with U the eigenbasis of C_Q,
    # R^T C_Q R = P^T H^T Lambda H P has every diagonal entry tr(C_Q) / d.
    # Fails if U is transposed, if H is unnormalised or if x is rotated as R x.
    Q = _decaying_queries(3)
    C = calibration.query_covariance(Q)
    U, w = calibration.eigenbasis(C)
    R = rotation.composite_rotation(U)
    Xr = rotation.rotate(Q, R)
    Cr = Xr.T @ Xr / Xr.shape[0]
    assert np.abs(np.diag(Cr) - np.trace(C) / 128).max() < 1e-10 * np.trace(C)
    # and without the Hadamard factor the diagonal is the (unequal) spectrum
    Ru = rotation.composite_rotation(U, True, False, False)
    assert np.allclose(np.diag(Ru.T @ C @ Ru), w)
    assert np.diag(Ru.T @ C @ Ru).std() > 0.1 * np.trace(C) / 128


def test_planted_transposed_basis_breaks_the_lemma_pin():
    # A plausible mistake planted in the oracle's inputs (U^T instead of U)
    # must fail the equal-diagonal property above.
    Q = _decaying_queries(4)
    C = calibration.query_covariance(Q)
    U, _ = calibration.eigenbasis(C)
    R_bad = rotation.composite_rotation(U.T)
    dg = np.diag(R_bad.T @ C @ R_bad)
    assert np.abs(dg - np.trace(C) / 128).max() > 1e-3 * np.trace(C) / 128


def test_rotate_unrotate_roundtrip():
    R = rotation.composite_rotation(_random_orthogonal(9))
    X = np.random.default_rng(0).standard_normal((10, 128))
    assert np.abs(rotation.unrotate(rotation.rotate(X, R), R) - X).max() < 1e-12


@pytest.mark.parametrize("d", [3, 0, 100])
def test_hadamard_rejects_non_power_of_two(d):
    with pytest.raises(ValueError):
        rotation.hadamard(d)
