"""INT2 group quantiser with clipping, fp64 (oracle; test infrastructure only).

[IT] "Il problema della quantizzazione a 2 bit": INT2 has only four
representable levels, and per-channel outliers dominate the scale factors.
[IT] "Architettura del Sistema di Serving": each history token is rotated,
clipped and quantised.  [ES] §2.2 A step 4: per-layer clipping thresholds
estimated from rotated calibration activations.

Readings (the pages give neither codebook, group size nor scale type; the
hot path's specification fixes group = 64 channels and one fp16 scale per
token per group, with no zero-point):

* clip:   a = min(max_j |x'_j|, tau) over the 64 rotated channels of a group;
* scale:  s = fp16(a / 1.5), fp16 round-to-nearest-even;
* code:   c = [x' >= -s] + [x' >= 0] + [x' >= s]  in {0, 1, 2, 3};
* level:  x_hat' = (c - 1.5) * s, i.e. the symmetric mid-rise levels
          {-1.5 s, -0.5 s, 0.5 s, 1.5 s}.  The thresholds -s, 0, s are the
          midpoints between neighbouring levels, so the code is the nearest
          level, ties going to the upper one.  Clipping changes only s.
* a group with s = 0 gets code 3 where x' >= 0 (all of it when a = 0) and
  dequantises to 0.
"""

import numpy as np

GROUP = 64
LEVEL_OFFSET = 1.5


def fp16_round(x):
    """Round fp64 values to the nearest fp16 value (ties to even), back in fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def group_scale(xg, tau):
    """Scale of one group: s = fp16(min(max|x'|, tau) / 1.5)."""
    a = min(float(np.max(np.abs(xg))), float(tau))
    return float(fp16_round(a / LEVEL_OFFSET))


def group_codes(xg, s):
    """Codes of one group for a given scale: [x >= -s] + [x >= 0] + [x >= s]."""
    xg = np.asarray(xg, dtype=np.float64)
    return ((xg >= -s).astype(np.uint8) + (xg >= 0).astype(np.uint8)
            + (xg >= s).astype(np.uint8))


def quantize_rows(Xr, tau, group=GROUP):
    """Quantise rotated rows Xr [n, d] group by group (vectorised over rows).

    Returns (codes uint8 [n, d], scales fp64 [n, d // group]); every scale is
    an fp16 value held in fp64.  Same arithmetic as group_scale/group_codes
    applied to each (row, group).
    """
    Xr = np.asarray(Xr, dtype=np.float64)
    n, d = Xr.shape
    ng = d // group
    Xg = Xr.reshape(n, ng, group)
    a = np.minimum(np.abs(Xg).max(axis=2), float(tau))
    scales = fp16_round(a / LEVEL_OFFSET)
    s = scales[:, :, None]
    codes = ((Xg >= -s).astype(np.uint8) + (Xg >= 0).astype(np.uint8) + (Xg >= s).astype(np.uint8))
    return codes.reshape(n, d), scales


def dequantize_rows(codes, scales, group=GROUP):
    """x_hat' = (c - 1.5) * s per group, fp64."""
    codes = np.asarray(codes, dtype=np.float64)
    scales = np.asarray(scales, dtype=np.float64)
    return (codes - LEVEL_OFFSET) * np.repeat(scales, group, axis=1)


def near_edge_mask(Xr, scales, rel=1e-6, group=GROUP):
    """Values lying within rel * s of a decision edge (-s, 0 or s).

    These are excluded from bit-exact code comparisons (their code depends on
    the last bit of the rotation arithmetic) and counted.
    """
    Xr = np.asarray(Xr, dtype=np.float64)
    s = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=1)
    band = rel * s
    return ((np.abs(Xr + s) <= band) | (np.abs(Xr) <= band)
            | (np.abs(Xr - s) <= band))


def fp16_midpoint_mask(Xr, tau, rel=1e-6, group=GROUP):
    """Groups whose a/1.5 lies within rel (relative) of an fp16 rounding midpoint.

    Their fp16 scale can round either way under a last-bit difference in a;
    they are excluded from scale and code comparisons and counted.
    """
    Xr = np.asarray(Xr, dtype=np.float64)
    n, d = Xr.shape
    ng = d // group
    a = np.minimum(np.abs(Xr).reshape(n, ng, group).max(axis=2), float(tau))
    v = a / LEVEL_OFFSET
    lo = fp16_round(v * (1 - rel))
    hi = fp16_round(v * (1 + rel))
    return lo != hi
