"""CPU: mistakes planted in the oracle must each fail at least one of its pins.

Each case patches one oracle function in memory (pytest's monkeypatch, undone
afterwards) with a plausible mistake -- a wrong tie rule, a dropped rounding
or clip, a wrong sign, index, bit count, operand order or transpose, an
off-by-one segment or ring row, a band taken in the wrong units -- and runs
the pins of test_oracle_rotation, test_oracle_quant_layout and
test_oracle_cache_attention; at least one must fail.  (U P H for U H P is not
a mistake: the Sylvester Hadamard matrix commutes with the bit-reversal
permutation, popcount(i & rev(j)) = popcount(rev(i) & j).)
"""

import inspect
import os

import numpy as np
import pytest

from oracle import attention, cache, calibration, layout, quant, rotation

import test_oracle_cache_attention as pins_cache
import test_oracle_quant_layout as pins_quant
import test_oracle_rotation as pins_rotation


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _pin_calls():
    """Every pin of the three modules as a zero-argument call (parametrized ones expanded)."""
    calls = []
    for mod in (pins_rotation, pins_quant, pins_cache):
        for name, fn in sorted(vars(mod).items()):
            if not name.startswith("test_") or not callable(fn):
                continue
            params = list(inspect.signature(fn).parameters)
            if not params:
                calls.append(fn)
                continue
            if params == ["golden_dir"]:  # the fixture of the golden-file pins
                calls.append(lambda f=fn: f(GOLDEN))
                continue
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            if len(params) == 1 and len(marks) == 1 and marks[0].args[0] == params[0]:
                calls.extend((lambda f=fn, v=v: f(v)) for v in marks[0].args[1])
    return calls


def _codes(X, s):
    return ((X >= -s).astype(np.uint8) + (X > 0).astype(np.uint8) + (X >= s).astype(np.uint8))


def _quantize(Xr, tau, group=quant.GROUP, codes=None, rounding=True, strided=False):
    Xr = np.asarray(Xr, dtype=np.float64)
    n, d = Xr.shape
    ng = d // group
    Xg = Xr.reshape(n, group, ng).transpose(0, 2, 1) if strided else Xr.reshape(n, ng, group)
    a = np.minimum(np.abs(Xg).max(axis=2), float(tau))
    sc = quant.fp16_round(a / 1.5) if rounding else a / 1.5
    s = sc[:, :, None]
    c = codes(Xg, s) if codes else ((Xg >= -s).astype(np.uint8) + (Xg >= 0).astype(np.uint8)
                                    + (Xg >= s).astype(np.uint8))
    c = c.transpose(0, 2, 1) if strided else c
    return c.reshape(n, d), sc


def _had(d=128, op=np.bitwise_and, norm=True):
    i = np.arange(d)
    parity = rotation.popcount(op.outer(i, i)) % 2
    return np.where(parity == 0, 1.0, -1.0) / (np.sqrt(d) if norm else 1.0)


def _rot_u_last(U, use_u=True, use_h=True, use_p=True):
    U = np.asarray(U, dtype=np.float64)
    d = U.shape[0]
    R = np.eye(d)
    if use_h:
        R = R @ rotation.hadamard(d)
    if use_p:
        R = R @ rotation.bit_reversal_matrix(d)
    return R @ U if use_u else R


def _segments(shift=0, hist_start=64):
    def seg(L):
        he = max(64, L - 256 + shift)
        return ((0, min(L, 64)), ((hist_start, he) if L > 64 else (64, 64)),
                ((max(64, L - 256 + shift), L) if L > 64 else (64, 64)))
    return seg


def _k_pos_swapped(t, j):
    T, u = divmod(t, 16)
    lane = 4 * (u % 8) + (j // 4) % 4
    word = 2 * (u // 8) + j // 64
    bit = 8 * (j % 4) + 2 * ((j // 32) % 2 + 2 * ((j // 16) % 2))
    return 512 * T + 16 * lane + 4 * word + bit // 8, bit % 8


def _v_pos_halves(t, j):
    T, u = divmod(t, 16)
    lane = 4 * (j % 8) + (u % 8) // 2
    word = 2 * (u // 8) + (j % 16) // 8
    bit = 16 * ((u + 1) % 2) + 2 * (j // 16)
    return 512 * T + 16 * lane + 4 * word + bit // 8, bit % 8


def _gqa_interleaved(q, K_heads, V_heads, sm):
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros_like(q)
    for hq in range(q.shape[0]):
        out[hq] = attention.softmax_attention(q[hq], K_heads[hq % len(K_heads)], V_heads[hq % len(K_heads)], sm)[0]
    return out


def _edge_absolute(Xr, scales, rel=1e-6, group=quant.GROUP):
    Xr = np.asarray(Xr, dtype=np.float64)
    s = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=1)
    return (np.abs(Xr + s) <= rel) | (np.abs(Xr) <= rel) | (np.abs(Xr - s) <= rel)


_softmax = attention.softmax_attention
_bitrev = rotation.bit_reverse
_quantize_rows = quant.quantize_rows
_cs = calibration.score_weighted_value_covariance
_had_ok = rotation.hadamard
_pack = layout.pack_block

MUTANTS = {
    "ties to the lower code": lambda mp: (mp.setattr(quant, "group_codes", lambda xg, s: _codes(np.asarray(xg, dtype=np.float64), s)),
                                          mp.setattr(quant, "quantize_rows", lambda X, tau, group=64: _quantize(X, tau, group, codes=_codes))),
    "scale not rounded to fp16": lambda mp: (mp.setattr(quant, "group_scale", lambda xg, tau: min(float(np.max(np.abs(xg))), float(tau)) / 1.5),
                                             mp.setattr(quant, "quantize_rows", lambda X, tau, group=64: _quantize(X, tau, group, rounding=False))),
    "no clip": lambda mp: (mp.setattr(quant, "group_scale", lambda xg, tau: float(quant.fp16_round(float(np.max(np.abs(xg))) / 1.5))),
                           mp.setattr(quant, "quantize_rows", lambda X, tau, group=64: _quantize_rows(X, np.inf, group))),
    "level offset 1 instead of 1.5": lambda mp: mp.setattr(quant, "dequantize_rows", lambda c, s, group=64: (np.asarray(c, dtype=np.float64) - 1.0) * np.repeat(np.asarray(s, dtype=np.float64), group, axis=1)),
    "groups strided across the row": lambda mp: mp.setattr(quant, "quantize_rows", lambda X, tau, group=64: _quantize(X, tau, group, strided=True)),
    "edge band absolute": lambda mp: mp.setattr(quant, "near_edge_mask", _edge_absolute),
    "Hadamard on i | j": lambda mp: mp.setattr(rotation, "hadamard", lambda d=128: _had(d, np.bitwise_or)),
    "Hadamard not normalised": lambda mp: mp.setattr(rotation, "hadamard", lambda d=128: _had(d, norm=False)),
    "bit reversal over 6 bits": lambda mp: mp.setattr(rotation, "bit_reverse", lambda j, nbits=7: _bitrev(j, nbits - 1)),
    "U applied last (H P U)": lambda mp: mp.setattr(rotation, "composite_rotation", _rot_u_last),
    "rotation transposed": lambda mp: mp.setattr(rotation, "rotate", lambda X, R: np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64).T),
    "inverse rotation not transposed": lambda mp: mp.setattr(rotation, "unrotate", lambda X, R: np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64)),
    "recent window of 255": lambda mp: mp.setattr(cache, "segments", _segments(shift=1)),
    "history from position 63": lambda mp: mp.setattr(cache, "segments", _segments(hist_start=63)),
    "ring row off by one": lambda mp: mp.setattr(cache, "ring_slot", lambda p: (p - 63) % 256),
    "softmax without sm_scale": lambda mp: mp.setattr(attention, "softmax_attention", lambda q, K, V, sm: _softmax(q, K, V, 1.0)),
    "GQA heads interleaved": lambda mp: mp.setattr(attention, "decode_gqa", _gqa_interleaved),
    "K code bit pairs swapped": lambda mp: mp.setattr(layout, "k_code_position", _k_pos_swapped),
    "V token halves swapped": lambda mp: mp.setattr(layout, "v_code_position", _v_pos_halves),
    "K and V scales swapped in the block": lambda mp: mp.setattr(layout, "pack_block", lambda kc, ks, vc, vs: _pack(kc, vs, vc, ks)),
    "C_S not averaged over queries": lambda mp: mp.setattr(calibration, "score_weighted_value_covariance", lambda Q, K, V, sm: _cs(Q, K, V, sm) * np.asarray(Q).shape[0]),
    "clip threshold of signed values": lambda mp: mp.setattr(calibration, "clip_threshold", lambda X, percentile=99.9: float(np.percentile(np.asarray(X, dtype=np.float64), percentile))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    MUTANTS[name](monkeypatch)
    for call in _pin_calls():
        try:
            call()
        except Exception:  # a failed check, or an error the mistake causes inside a pin
            return
    pytest.fail("no pin catches: " + name)


def test_the_pins_pass_on_the_unpatched_oracle():
    # the control: called this way, every pin passes, so each catch above is the planted mistake's
    calls = _pin_calls()
    assert len(calls) >= 45
    for call in calls:
        call()
