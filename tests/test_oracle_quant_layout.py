"""Pins of the oracle's quantiser and block layout.

Sources: ainsights.it "OSCAR: Come Together AI Comprime la KV Cache a 2-bit
per LLM" ("Il problema della quantizzazione a 2 bit": four levels, outliers
dominate the scale; "Architettura del Sistema di Serving": rotate, clip,
quantise, paged cache); gist.science "Resumen Técnico: OSCAR ..." §2.2 A.4
(clipping thresholds) and §2.2 B (paged INT2 history).
"""

import os

import numpy as np

from oracle import layout, quant


def _read_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "case":
            cur = {"name": f[1], "tau": float(f[3]), "scale": float(f[5]), "vals": [], "codes": []}
            cases.append(cur)
        else:
            cur["vals"].append(float(f[0]))
            cur["codes"].append(int(f[1]))
    return cases


def test_quant_golden_groups(golden_dir):
    for c in _read_cases(os.path.join(golden_dir, "quant_groups.txt")):
        x = np.zeros(64)
        x[:len(c["vals"])] = c["vals"]
        s = quant.group_scale(x, c["tau"])
        assert s == c["scale"], c["name"]
        codes = quant.group_codes(x, s)
        assert list(codes[:len(c["codes"])]) == c["codes"], c["name"]
        rest = 3 if s == 0 else 2
        assert np.all(codes[len(c["codes"]):] == rest)


def _nearest_level_codes(x, s):
    # Brute force: the nearest of the four levels (c - 1.5) s, ties to the
    # upper level.  A different formulation of the same quantiser.
    levels = (np.arange(4) - 1.5) * s
    out = np.zeros(x.shape, dtype=np.uint8)
    for i, v in enumerate(x):
        dist = np.abs(v - levels)
        best = 0
        for c in range(4):
            if dist[c] <= dist[best]:
                best = c
        out[i] = best
    return out


def test_threshold_codes_equal_nearest_level_brute_force():
    r = np.random.default_rng(5)
    for trial in range(40):
        x = r.standard_normal(64) * r.uniform(0.1, 10)
        tau = np.inf if trial % 2 else np.percentile(np.abs(x), 90)
        s = quant.group_scale(x, tau)
        # add exact ties at the thresholds and beyond the clip
        x[:3] = [-s, 0.0, s]
        x[3:5] = [4 * s, -4 * s]
        assert np.array_equal(quant.group_codes(x, s), _nearest_level_codes(x, s))


def test_identity_rotation_infinite_clip_is_textbook_absmax_int2():
    # I7: with R = I and tau = inf the method is plain symmetric absmax INT2:
    # scale = max|x| / 1.5 (in fp16), levels {-1.5, -0.5, 0.5, 1.5} * scale.
    r = np.random.default_rng(6)
    X = r.standard_normal((8, 128)) * 3
    codes, scales = quant.quantize_rows(X, np.inf)
    for t in range(8):
        for g in range(2):
            xg = X[t, 64 * g:64 * (g + 1)]
            s = float(np.float16(np.abs(xg).max() / 1.5))
            assert scales[t, g] == s
            assert np.array_equal(codes[t, 64 * g:64 * (g + 1)], _nearest_level_codes(xg, s))
    # the largest magnitude maps to an end level
    assert set(np.unique(codes)) <= {0, 1, 2, 3}


def test_clip_changes_only_the_scale():
    x = np.linspace(-5, 5, 64)
    s_clip = quant.group_scale(x, 2.0)
    assert s_clip == float(np.float16(2.0 / 1.5))
    c = quant.group_codes(x, s_clip)
    assert np.all(c[x >= s_clip] == 3) and np.all(c[x < -s_clip] == 0)


def test_dequantize_levels():
    codes = np.array([[0, 1, 2, 3] * 32])
    scales = np.array([[2.0, 0.5]])
    d = quant.dequantize_rows(codes, scales)
    assert np.array_equal(d[0, :4], [-3.0, -1.0, 1.0, 3.0])
    assert np.array_equal(d[0, 64:68], [-0.75, -0.25, 0.25, 0.75])


def test_fp16_round_to_nearest_even():
    # Known fp16 roundings: ties go to the even mantissa.
    assert quant.fp16_round(1 + 2.0**-11) == 1.0
    assert quant.fp16_round(1 + 3 * 2.0**-11) == 1 + 2.0**-9
    assert quant.fp16_round(65504.0) == 65504.0
    assert quant.fp16_round(2.0 / 3.0) == 1365 * 2.0**-11
    assert quant.fp16_round(2.0**-25) == 0.0          # tie between 0 and 2^-24 -> even (0)
    assert quant.fp16_round(3 * 2.0**-25) == 2 * 2.0**-24


def test_near_edge_and_midpoint_masks():
    s = 1.0
    x = np.zeros((1, 64))
    x[0, :6] = [1.0, 1.0 + 5e-7, -1.0 - 2e-6, 2e-7, 0.3, -0.5]
    m = quant.near_edge_mask(x, np.array([[s]]), group=64)
    assert list(m[0, :6]) == [True, True, False, True, False, False]
    # a/1.5 exactly on an fp16 midpoint (1 + 2^-11) is flagged; 1.2 is not
    x = np.zeros((2, 64))
    x[0, 0] = 1.5 * (1 + 2.0**-11)
    x[1, 0] = 1.5 * 1.2
    mm = quant.fp16_midpoint_mask(x, np.inf, group=64)
    assert mm[0, 0] and not mm[1, 0]


def test_layout_golden_positions(golden_dir):
    for line in open(os.path.join(golden_dir, "layout_positions.txt")):
        if line.startswith("#") or not line.strip():
            continue
        which, t, j, byte, bit = line.split()
        f = layout.k_code_position if which == "K" else layout.v_code_position
        assert f(int(t), int(j)) == (int(byte), int(bit)), line


def test_layout_is_a_bijection_on_the_code_area():
    for f in (layout.k_code_position, layout.v_code_position):
        seen = set()
        for t in range(64):
            for j in range(128):
                byte, bit = f(t, j)
                assert 0 <= byte < 2048 and bit in (0, 2, 4, 6)
                seen.add((byte, bit))
        assert len(seen) == 64 * 128


def test_tokens_own_whole_words_and_halves():
    # K: a token's codes fill whole 32-bit words; V: whole 16-bit halves.
    for t in range(64):
        kw = {layout.k_code_position(t, j)[0] // 4 for j in range(128)}
        assert len(kw) == 8
        vh = {layout.v_code_position(t, j)[0] // 2 for j in range(128)}
        assert len(vh) == 16
    kt = {}
    for t in range(64):
        for j in range(128):
            kt.setdefault(layout.k_code_position(t, j)[0] // 4, set()).add(t)
    assert all(len(v) == 1 for v in kt.values())


def test_pack_unpack_roundtrip():
    r = np.random.default_rng(8)
    kc = r.integers(0, 4, (64, 128)).astype(np.uint8)
    vc = r.integers(0, 4, (64, 128)).astype(np.uint8)
    ks = np.float16(r.uniform(0, 10, (64, 2))).astype(np.float64)
    vs = np.float16(r.uniform(0, 10, (64, 2))).astype(np.float64)
    blk = layout.pack_block(kc, ks, vc, vs)
    assert blk.size == 4608
    a, b, c, d = layout.unpack_block(blk)
    assert np.array_equal(a, kc) and np.array_equal(c, vc)
    assert np.array_equal(b, ks) and np.array_equal(d, vs)
    # scales at the documented byte offsets, little-endian fp16 [t][group]
    assert blk[2048:2050].view('<f2')[0] == np.float16(ks[0, 0])
    assert blk[4352 + 4 * 5 + 2:4352 + 4 * 5 + 4].view('<f2')[0] == np.float16(vs[5, 1])


def test_partial_block_leaves_rest_zero():
    kc = np.full((10, 128), 3, dtype=np.uint8)
    blk = layout.pack_block(kc, np.ones((10, 2)), kc, np.ones((10, 2)))
    a, _, c, _ = layout.unpack_block(blk)
    assert np.all(a[:10] == 3) and np.all(a[10:] == 0) and np.all(c[10:] == 0)


def test_vectorised_rows_equal_per_group_definition():
    r = np.random.default_rng(21)
    X = r.standard_normal((50, 128)) * r.uniform(0.1, 5, (50, 1))
    X[3, :64] = 0.0
    codes, scales = quant.quantize_rows(X, 2.5)
    for t in range(50):
        for g in range(2):
            xg = X[t, 64 * g:64 * (g + 1)]
            s = quant.group_scale(xg, 2.5)
            assert scales[t, g] == s
            assert np.array_equal(codes[t, 64 * g:64 * (g + 1)], quant.group_codes(xg, s))


def test_vectorised_unpack_equals_unpack_block():
    r = np.random.default_rng(22)
    blocks = r.integers(0, 256, (3, 4608)).astype(np.uint8)
    # keep the scale bytes finite fp16 values
    for i in range(3):
        blocks[i, 2048:2304] = np.float16(r.uniform(0, 4, 128)).view(np.uint8)
        blocks[i, 4352:4608] = np.float16(r.uniform(0, 4, 128)).view(np.uint8)
    kc, ks, vc, vs = layout.unpack_blocks(blocks)
    for i in range(3):
        a, b, c, d = layout.unpack_block(blocks[i])
        assert np.array_equal(kc[i], a) and np.array_equal(vc[i], c)
        assert np.array_equal(ks[i], b) and np.array_equal(vs[i], d)


def test_near_edge_band_is_relative_to_the_scale():
    # The exclusion band "within 1e-6 relative of a bin edge" is taken
    # relative to the group's scale s: at s = 1024 a value 5e-4 above the edge
    # s is inside it (band 1.024e-3); at s ~ 1e-3 a value 5e-7 above the edge 0
    # is outside it (band ~1e-9), though both would flip under an absolute band.
    big = np.zeros((1, 64))
    big[0, 0] = 1536.0                      # a = 1536, s = fp16(1024) = 1024
    big[0, 1] = 1024.0 + 5e-4
    small = np.zeros((1, 64))
    small[0, 0] = 1.5e-3                    # s = fp16(1e-3)
    small[0, 1] = 5e-7
    for X, col, want in ((big, 1, True), (small, 1, False)):
        X = np.concatenate([X, np.full((1, 64), 7.0)], axis=1)   # second group far from every edge
        _, scales = quant.quantize_rows(X, np.inf)
        mask = quant.near_edge_mask(X, scales)
        assert bool(mask[0, col]) == want
        assert not mask[0, 64:].any()
