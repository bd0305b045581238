"""Pins of the oracle's cache segments, append/eviction model, attention and calibration.

Sources: ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit
per LLM" ("Architettura del Sistema di Serving e Layout di Memoria": 64 BF16
sink tokens, 256 BF16 recent tokens, INT2 history; the read kernel undoes the
rotation); edge.aivizor.me "Together AI выпустила исходники OSCAR ..."
("Техническая идея": C_Q and C_S and their eigenvectors); gist.science
"Resumen Técnico: OSCAR ..." §2.1, §2.2 A, §2.2 B.
"""

import os

import numpy as np
import pytest

from oracle import attention, cache, calibration, quant, rotation


def test_segments_golden(golden_dir):
    for line in open(os.path.join(golden_dir, "segments.txt")):
        if line.startswith("#") or not line.strip():
            continue
        L, a0, a1, h0, h1, r0, r1 = (int(x) for x in line.split())
        assert cache.segments(L) == ((a0, a1), (h0, h1), (r0, r1)), L


def test_segments_partition_the_context():
    for L in list(range(0, 700)) + [4096, 100000]:
        (a0, a1), (h0, h1), (r0, r1) = cache.segments(L)
        n = (a1 - a0) + max(0, h1 - h0) + max(0, r1 - r0)
        assert n == L
        assert r1 - r0 <= 256 and a1 - a0 <= 64


def _rand_orth(seed):
    a = np.random.default_rng(seed).standard_normal((128, 128))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))


def _bf16_like(x):
    # round fp64 values to bf16 precision (8 significant bits), as tokens are BF16
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("chunks", [[1] * 700, [300, 1, 399], [700], [64, 256, 1, 379]])
def test_incremental_append_equals_direct_definition(chunks):
    # The ring/eviction model must give, for every history position, exactly
    # quantize(rotate(token)) and keep sink/recent tokens exact.
    r = np.random.default_rng(11)
    Kt = _bf16_like(r.standard_normal((sum(chunks), 128)) * 3)
    Vt = _bf16_like(r.standard_normal((sum(chunks), 128)) * 3)
    R_K = rotation.composite_rotation(_rand_orth(1))
    R_V = rotation.composite_rotation(_rand_orth(2))
    c = cache.RequestCache(R_K, R_V, 6.0, 7.0)
    p = 0
    for n in chunks:
        c.append(Kt[p:p + n], Vt[p:p + n])
        p += n
    L = p
    want, _ = cache.expected_history(Kt, Vt, L, R_K, R_V, 6.0, 7.0)
    assert sorted(c.hist) == sorted(want)
    for pos, (kc, ks, vc, vs) in want.items():
        gc = c.hist[pos]
        assert np.array_equal(gc[0], kc) and np.array_equal(gc[1], ks)
        assert np.array_equal(gc[2], vc) and np.array_equal(gc[3], vs)
    K, V = c.dequantized()
    (s0, s1), (h0, h1), (r0, r1) = cache.segments(L)
    assert np.array_equal(K[s0:s1], Kt[s0:s1]) and np.array_equal(V[r0:r1], Vt[r0:r1])


def test_fresh_ring_append_skips_eviction():
    R = rotation.composite_rotation(_rand_orth(3))
    c = cache.RequestCache(R, R, 5.0, 5.0)
    c.length = 1000          # a shared prefix already held as sink/history
    k = np.ones((300, 128))
    c.append(k, k, fresh_ring=True)
    assert min(c.hist) == 1000 and max(c.hist) == 1043   # only new tokens < L - 256
    assert c.length == 1300


def test_dequantized_history_is_rotated_back():
    # A history token with tau = inf and values exactly on the levels
    # reconstructs exactly: x = (c - 1.5) s R^T.
    R = rotation.composite_rotation(_rand_orth(4))
    xr = np.tile(np.array([-1.5, -0.5, 0.5, 1.5]), 32)
    x = rotation.unrotate(xr[None], R)[0]
    c = cache.RequestCache(R, R, np.inf, np.inf)
    toks = np.zeros((321, 128))
    toks[64] = x
    c.append(toks, toks)
    K, _ = c.dequantized()
    assert np.abs(K[64] - x).max() < 1e-12


def test_attention_single_token_and_two_token_closed_form():
    # I5: one token -> its value; two tokens -> logistic weighting.
    r = np.random.default_rng(12)
    q = r.standard_normal((3, 8))
    K = r.standard_normal((2, 8))
    V = r.standard_normal((2, 8))
    out1 = attention.softmax_attention(q, K[:1], V[:1], 0.7)
    assert np.allclose(out1, np.repeat(V[:1], 3, axis=0))
    out2 = attention.softmax_attention(q, K, V, 0.7)
    for h in range(3):
        z1, z2 = 0.7 * q[h] @ K[0], 0.7 * q[h] @ K[1]
        w = 1.0 / (1.0 + np.exp(-(z1 - z2)))
        assert np.allclose(out2[h], w * V[0] + (1 - w) * V[1], atol=1e-14)


def test_attention_zero_query_is_mean_and_empty_is_zero():
    V = np.random.default_rng(13).standard_normal((9, 128))
    out = attention.softmax_attention(np.zeros((2, 128)), np.ones((9, 128)), V, 0.1)
    assert np.allclose(out, V.mean(0))
    assert np.array_equal(attention.softmax_attention(np.ones((1, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0), np.zeros((1, 4)))


def test_attention_brute_force_small():
    # I5 brute force: explicit loops over L <= 8 tokens.
    r = np.random.default_rng(14)
    for L in range(1, 9):
        q = r.standard_normal(128)
        K = r.standard_normal((L, 128))
        V = r.standard_normal((L, 128))
        z = [sum(q[i] * K[t, i] for i in range(128)) / np.sqrt(128) for t in range(L)]
        e = [np.exp(v) for v in z]
        want = sum(e[t] * V[t] for t in range(L)) / sum(e)
        got = attention.softmax_attention(q, K, V, 1 / np.sqrt(128))[0]
        assert np.abs(got - want).max() < 1e-12


def test_attention_rotation_invariance_on_bf16_data():
    # I4: attention(q R_K, K R_K, V R_V) R_V^T = attention(q, K, V).
    r = np.random.default_rng(15)
    R_K = rotation.composite_rotation(_rand_orth(5))
    R_V = rotation.composite_rotation(_rand_orth(6))
    q = _bf16_like(r.standard_normal((4, 128)))
    K = _bf16_like(r.standard_normal((300, 128)) * 4)
    V = _bf16_like(r.standard_normal((300, 128)) * 4)
    plain = attention.softmax_attention(q, K, V, 1 / np.sqrt(128))
    rot = attention.softmax_attention(q @ R_K, K @ R_K, V @ R_V, 1 / np.sqrt(128)) @ R_V.T
    assert np.abs(rot - plain).max() < 1e-12


def test_decode_gqa_head_mapping():
    # query head h reads KV head h // g
    r = np.random.default_rng(16)
    q = r.standard_normal((8, 16))
    Ks = [r.standard_normal((5, 16)) for _ in range(2)]
    Vs = [r.standard_normal((5, 16)) for _ in range(2)]
    out = attention.decode_gqa(q, Ks, Vs, 0.3)
    for h in range(8):
        assert np.allclose(out[h], attention.softmax_attention(q[h], Ks[h // 4], Vs[h // 4], 0.3)[0])


def test_calibration_closed_forms():
    # C_Q of a diagonal design; eigenbasis of a diagonal matrix; C_S with
    # uniform scores (Q = 0) equals mean(V)^T mean(V).
    Q = np.diag([3.0, 2.0, 1.0, 0.5])
    assert np.allclose(calibration.query_covariance(Q), np.diag([9.0, 4.0, 1.0, 0.25]) / 4)
    U, w = calibration.eigenbasis(np.diag([1.0, 5.0, 3.0, 2.0]))
    assert np.allclose(w, [5, 3, 2, 1]) and np.allclose(np.abs(U), np.eye(4)[:, [1, 2, 3, 0]])
    r = np.random.default_rng(17)
    V = r.standard_normal((6, 4))
    K = r.standard_normal((6, 4))
    C = calibration.score_weighted_value_covariance(np.zeros((5, 4)), [K], [V], 1.0)
    m = V.mean(0)
    assert np.allclose(C, np.outer(m, m))


def test_clip_threshold_percentile_golden():
    # 1..1000: the 99.9th percentile with linear interpolation is 999.001
    x = np.arange(1, 1001, dtype=float) * np.where(np.arange(1000) % 2, 1, -1)
    assert abs(calibration.clip_threshold(x) - 999.001) < 1e-9


def test_score_weighted_covariance_matches_output_second_moment():
    # C_S = (1/N) (S V)^T (S V): the second moment of the attention outputs,
    # checked by looping over the queries.
    r = np.random.default_rng(18)
    Q = r.standard_normal((7, 8))
    K = r.standard_normal((5, 8))
    V = r.standard_normal((5, 8))
    C = calibration.score_weighted_value_covariance(Q, [K], [V], 0.5)
    acc = np.zeros((8, 8))
    for n in range(7):
        o = attention.softmax_attention(Q[n], K, V, 0.5)[0]
        acc += np.outer(o, o)
    assert np.allclose(C, acc / 7)


def test_reconstruct_from_storage_matches_cache_model():
    # storing the model's state with the oracle's packer and reading it back
    # gives the same K_hat, V_hat as the model itself
    from oracle import layout
    r = np.random.default_rng(19)
    R_K = rotation.composite_rotation(_rand_orth(7))
    R_V = rotation.composite_rotation(_rand_orth(8))
    L = 777
    Kt = _bf16_like(r.standard_normal((L, 128)) * 2)
    Vt = _bf16_like(r.standard_normal((L, 128)) * 2)
    c = cache.RequestCache(R_K, R_V, 5.0, 6.0)
    c.append(Kt[:500], Vt[:500])
    c.append(Kt[500:], Vt[500:])
    (_, _), (h0, h1), _ = cache.segments(L)
    n_pages = (h1 + 63) // 64 - 1
    blocks = np.zeros((n_pages, 4608), dtype=np.uint8)
    for i in range(n_pages):
        lp = i + 1
        rows = [p for p in range(64 * lp, 64 * lp + 64) if h0 <= p < h1]
        kc = np.array([c.hist[p][0] for p in rows])
        ks = np.array([c.hist[p][1] for p in rows])
        vc = np.array([c.hist[p][2] for p in rows])
        vs = np.array([c.hist[p][3] for p in rows])
        blocks[i] = layout.pack_block(kc, ks, vc, vs)
    K, V = cache.reconstruct_from_storage(c.sink_k, c.sink_v, c.ring_k, c.ring_v, blocks, L, R_K, R_V)
    Km, Vm = c.dequantized()
    assert np.abs(K - Km).max() < 1e-12 and np.abs(V - Vm).max() < 1e-12


def test_calibrate_layer_composes_the_steps():
    # Queries with an exactly diagonal covariance diag(sigma^2) in a shuffled
    # channel order (+-1 columns of a 256-point Hadamard matrix, scaled):
    # U_K must be the signed permutation sorting sigma^2 in descending order.
    # Keys = unit rows: under R = U H P every |entry| is 1/sqrt(128), so that
    # is tau_K; with every factor off (R = I) tau_K = 1.  With zero scores
    # (sm_scale = 0) C_S = m^T m for the mean value row m, whose direction is
    # U_V's first column.
    import scipy.linalg
    d = 128
    r = np.random.default_rng(21)
    sig2 = r.permutation(np.linspace(1.0, 4.0, d))
    Q = scipy.linalg.hadamard(256)[:, :d] * np.sqrt(sig2)
    K = np.eye(d)[:64]
    V = r.standard_normal((64, d))
    U_K, U_V, tau_k, tau_v = calibration.calibrate_layer(Q, [K], [V], 0.0)
    perm = np.argsort(-sig2, kind="stable")
    assert np.allclose(np.abs(U_K), np.eye(d)[:, perm])
    assert abs(tau_k - 1.0 / np.sqrt(d)) < 1e-12
    m = V.mean(0)
    assert abs(abs(U_V[:, 0] @ m) - np.linalg.norm(m)) < 1e-9
    _, _, tau_k0, _ = calibration.calibrate_layer(Q, [K], [V], 0.0, flags=(False, False, False))
    assert abs(tau_k0 - 1.0) < 1e-12


def test_ring_rows_follow_the_documented_convention():
    # Recent position p >= 64 lives in ring row (p - 64) mod 256 (the storage
    # convention the C ABI documents for the 256 BF16 recent tokens of [IT]
    # "Architettura ..."): special cases, and after 400 appends the model's
    # window positions 144..399 occupy every row exactly once, each its own token.
    assert [cache.ring_slot(p) for p in (64, 65, 319, 320, 575, 576)] == [0, 1, 255, 0, 255, 0]
    r = np.random.default_rng(23)
    R = rotation.composite_rotation(_rand_orth(24))
    m = cache.RequestCache(R, R, 30.0, 30.0)
    toks = r.standard_normal((400, 128))
    for p in range(400):
        m.append(toks[p:p + 1], toks[p:p + 1])
    rows = sorted(cache.ring_slot(p) for p in range(144, 400))
    assert rows == list(range(256))
    for p in range(144, 400):
        assert np.array_equal(m.ring_k[cache.ring_slot(p)], toks[p])
