"""Mixed-precision KV cache semantics: segments and the append/eviction model.

Oracle; test infrastructure only.

[IT] "Architettura del Sistema di Serving e Layout di Memoria": the first 64
tokens stay BF16 (attention sinks), the last 256 tokens before the current
position stay BF16, everything else is INT2 after rotation and clipping.
[IT] "Guida Rapida": ``--oscar-sink-size 64 --oscar-recent-size 256``.
[ES] §2.2 B: sink and recent tokens in full BF16 precision, the intermediate
history INT2 after the fixed rotation and clipping, in a paged cache.

Readings:

* For a context of L tokens (positions 0..L-1, the new token included):
      sink    = [0, min(L, 64))
      recent  = [max(64, L - 256), L)
      history = [64, max(64, L - 256))
* Sink and recent tokens are stored unrotated (the pages apply the rotation
  only on the way into INT2).
* Storage: a sink page of 64 rows, a ring of 256 BF16 slots with position p
  (p >= 64) in slot (p - 64) mod 256, and INT2 pages of 64 positions; logical
  page i covers positions [64 i, 64 i + 64), so history starts at page 1.
* A token leaves the recent window (and is rotated, clipped, quantised into
  its history row) when the context grows past it by 256.
"""

import numpy as np

from . import quant, rotation

SINK = 64
RECENT = 256
PAGE = 64
HEAD_DIM = 128


def segments(L):
    """(sink, history, recent) position ranges of a context of length L."""
    sink = (0, min(L, SINK))
    hist_end = max(SINK, L - RECENT)
    history = (SINK, hist_end) if L > SINK else (SINK, SINK)
    recent = (max(SINK, L - RECENT), L) if L > SINK else (SINK, SINK)
    return sink, history, recent


def ring_slot(p):
    """Ring slot of a recent position p >= 64."""
    return (p - SINK) % RECENT


class RequestCache:
    """One request, one layer, one KV head: the oracle's model of the cache.

    Holds the sink rows, the ring slots (BF16 values kept in fp64) and the
    quantised history rows (codes, scales), keyed by position.
    """

    def __init__(self, R_K, R_V, tau_k, tau_v):
        self.R_K = np.asarray(R_K, dtype=np.float64)
        self.R_V = np.asarray(R_V, dtype=np.float64)
        self.tau_k = float(tau_k)
        self.tau_v = float(tau_v)
        self.length = 0
        self.sink_k = np.zeros((SINK, HEAD_DIM))
        self.sink_v = np.zeros((SINK, HEAD_DIM))
        self.ring_k = np.zeros((RECENT, HEAD_DIM))
        self.ring_v = np.zeros((RECENT, HEAD_DIM))
        self.hist = {}  # position -> (k_codes, k_scales, v_codes, v_scales)

    def _to_history(self, p, k, v):
        kc, ks = quant.quantize_rows(rotation.rotate(k[None], self.R_K), self.tau_k)
        vc, vs = quant.quantize_rows(rotation.rotate(v[None], self.R_V), self.tau_v)
        self.hist[p] = (kc[0], ks[0], vc[0], vs[0])

    def append(self, k_new, v_new, fresh_ring=False):
        """Append n tokens at positions [length, length + n).

        Phase 1 moves every ring token that falls out of the recent window
        into the history; phase 2 places each new token.  With fresh_ring the
        positions before ``length`` are taken to be sink/history already (a
        shared prefix) and nothing is evicted.
        """
        k_new = np.asarray(k_new, dtype=np.float64)
        v_new = np.asarray(v_new, dtype=np.float64)
        L0 = self.length
        L = L0 + k_new.shape[0]
        if not fresh_ring:
            for e in range(max(SINK, L0 - RECENT), max(SINK, L - RECENT)):
                if e >= L0:
                    break
                s = ring_slot(e)
                self._to_history(e, self.ring_k[s], self.ring_v[s])
        for i in range(k_new.shape[0]):
            p = L0 + i
            if p < SINK:
                self.sink_k[p] = k_new[i]
                self.sink_v[p] = v_new[i]
            elif p >= L - RECENT:
                s = ring_slot(p)
                self.ring_k[s] = k_new[i]
                self.ring_v[s] = v_new[i]
            else:
                self._to_history(p, k_new[i], v_new[i])
        self.length = L

    def dequantized(self):
        """K_hat, V_hat [L, 128]: exact BF16 rows for sink/recent, rotated-back
        dequantised rows x_hat' R^T for history."""
        L = self.length
        K = np.zeros((L, HEAD_DIM))
        V = np.zeros((L, HEAD_DIM))
        (s0, s1), (h0, h1), (r0, r1) = segments(L)
        K[s0:s1] = self.sink_k[s0:s1]
        V[s0:s1] = self.sink_v[s0:s1]
        for p in range(r0, r1):
            K[p] = self.ring_k[ring_slot(p)]
            V[p] = self.ring_v[ring_slot(p)]
        for p in range(h0, h1):
            kc, ks, vc, vs = self.hist[p]
            K[p] = rotation.unrotate(quant.dequantize_rows(kc[None], ks[None]), self.R_K)[0]
            V[p] = rotation.unrotate(quant.dequantize_rows(vc[None], vs[None]), self.R_V)[0]
        return K, V


def expected_history(tokens_k, tokens_v, L, R_K, R_V, tau_k, tau_v):
    """Direct definition of the history of a context of length L.

    Every position of [64, L - 256) holds quantize(rotate(token)).  Returns
    a dict position -> (k_codes, k_scales, v_codes, v_scales) plus the
    rotated fp64 rows (for the edge exclusion).
    """
    (_, _), (h0, h1), _ = segments(L)
    out = {}
    rot = {}
    if h1 > h0:
        Kr = rotation.rotate(np.asarray(tokens_k)[h0:h1], R_K)
        Vr = rotation.rotate(np.asarray(tokens_v)[h0:h1], R_V)
        kc, ks = quant.quantize_rows(Kr, tau_k)
        vc, vs = quant.quantize_rows(Vr, tau_v)
        for i, p in enumerate(range(h0, h1)):
            out[p] = (kc[i], ks[i], vc[i], vs[i])
            rot[p] = (Kr[i], Vr[i])
    return out, rot


def reconstruct_from_storage(sink_k, sink_v, ring_k, ring_v, blocks, L, R_K, R_V):
    """K_hat, V_hat [L, 128] (fp64) of one request and KV head from stored bytes.

    sink_k/v: [64, 128] BF16 values; ring_k/v: [256, 128] BF16 values (slot
    order); blocks: uint8 [n, 4608], the INT2 blocks of logical pages 1..n in
    order.  History rows are unpacked with the oracle's own layout map,
    dequantised and rotated back: x_hat = ((c - 1.5) s) R^T.
    """
    from . import layout
    K = np.zeros((L, HEAD_DIM))
    V = np.zeros((L, HEAD_DIM))
    (s0, s1), (h0, h1), (r0, r1) = segments(L)
    K[s0:s1] = np.asarray(sink_k, dtype=np.float64)[s0:s1]
    V[s0:s1] = np.asarray(sink_v, dtype=np.float64)[s0:s1]
    if r1 > r0:
        slots = [ring_slot(p) for p in range(r0, r1)]
        K[r0:r1] = np.asarray(ring_k, dtype=np.float64)[slots]
        V[r0:r1] = np.asarray(ring_v, dtype=np.float64)[slots]
    if h1 > h0:
        kc, ks, vc, vs = layout.unpack_blocks(blocks)
        n = h1 - h0          # history starts at row 0 of logical page 1
        kc = kc.reshape(-1, HEAD_DIM)[:n]
        vc = vc.reshape(-1, HEAD_DIM)[:n]
        ks = ks.reshape(-1, 2)[:n]
        vs = vs.reshape(-1, 2)[:n]
        K[h0:h1] = rotation.unrotate(quant.dequantize_rows(kc, ks), R_K)
        V[h0:h1] = rotation.unrotate(quant.dequantize_rows(vc, vs), R_V)
    return K, V
