"""Seeded synthetic inputs for the OSCAR hot path.

This module draws random data only: it holds none of the method's arithmetic
(no rotation, clipping, quantisation, packing or attention).  Both the CUDA
path's tests/benchmark and the CPU oracle consume what it produces.

Distributions (the pages' workloads are real-model KV activations with
per-channel outliers -- ainsights.it "Il problema della quantizzazione a 2 bit
nelle KV Cache"; gist.science §1 -- which synthetic data stands in for):

* K and V tokens: N(0, 1) fp32 per channel; 4 distinct seeded outlier channels
  per (layer, KV head), chosen separately for K and for V, scaled by 20; then
  rounded to BF16.  Calibration tokens use the same outlier channels with a
  different random stream.
* Queries: q = z diag(sigma) B^T with z ~ N(0, I), sigma_i = exp(-i / 32)
  (a decaying spectrum) and B a seeded random orthogonal matrix per layer.
* Page tables: a seeded permutation of the physical pages.

Seeds are ``numpy.random.default_rng([config, layer, head, stream])`` for the
small draws; bulk device draws use a ``torch.Generator`` seeded from the same
tuple.
"""

import numpy as np
import torch

HEAD_DIM = 128
N_OUTLIERS = 4
OUTLIER_FACTOR = 20.0

# random streams
STREAM_OUTLIER = 0
STREAM_KV_CAL = 1
STREAM_KV = 2
STREAM_Q_CAL = 3
STREAM_Q = 4
STREAM_PAGES = 5
STREAM_LENS = 6
STREAM_BASIS = 7
STREAM_APPEND = 8


def rng(*key):
    """numpy Generator for a tuple of non-negative ints."""
    return np.random.default_rng([int(k) for k in key])


def torch_seed(*key):
    """A 63-bit torch seed derived from a tuple of non-negative ints."""
    return int(rng(*key).integers(0, 2**63 - 1))


def outlier_channels(cfg, layer, head, which, d=HEAD_DIM):
    """The N_OUTLIERS distinct outlier channels of (layer, KV head); which = 0 for K, 1 for V."""
    return np.sort(rng(cfg, layer, head, STREAM_OUTLIER, which).choice(d, N_OUTLIERS, replace=False))


def to_bf16(x):
    """fp32 array -> torch.bfloat16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_to_f64(t):
    """torch.bfloat16 tensor -> float64 numpy array (exact)."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def kv_tokens(cfg, layer, head, stream, n, which, request=0, d=HEAD_DIM):
    """[n, d] fp32 outlier-channel Gaussian tokens for one KV head (numpy)."""
    x = rng(cfg, layer, head, stream, which, request).standard_normal((n, d)).astype(np.float32)
    x[:, outlier_channels(cfg, layer, head, which, d)] *= OUTLIER_FACTOR
    return x


def kv_tokens_bf16(cfg, layer, n_kv_heads, stream, n, request=0, d=HEAD_DIM):
    """(K, V) torch.bfloat16 [n, H_kv, d] on the CPU (numpy draws)."""
    k = np.stack([kv_tokens(cfg, layer, h, stream, n, 0, request, d) for h in range(n_kv_heads)], axis=1)
    v = np.stack([kv_tokens(cfg, layer, h, stream, n, 1, request, d) for h in range(n_kv_heads)], axis=1)
    return to_bf16(k), to_bf16(v)


def kv_tokens_device(cfg, layer, n_kv_heads, stream, n, device, request=0, d=HEAD_DIM):
    """(K, V) torch.bfloat16 [n, H_kv, d] drawn on ``device`` (bulk inputs)."""
    out = []
    for which in (0, 1):
        g = torch.Generator(device=device)
        g.manual_seed(torch_seed(cfg, layer, stream, which, request))
        x = torch.randn((n, n_kv_heads, d), generator=g, device=device, dtype=torch.float32)
        scale = torch.ones((n_kv_heads, d), dtype=torch.float32)
        for h in range(n_kv_heads):
            scale[h, outlier_channels(cfg, layer, h, which, d)] = OUTLIER_FACTOR
        x.mul_(scale.to(device))
        out.append(x.to(torch.bfloat16))
    return out[0], out[1]


def query_sigma(d=HEAD_DIM):
    """sigma_i = exp(-i / 32): the decaying query spectrum."""
    return np.exp(-np.arange(d) / 32.0)


def query_basis(cfg, layer, d=HEAD_DIM):
    """Seeded random orthogonal matrix (QR of a Gaussian, signs fixed by R's diagonal)."""
    a = rng(cfg, layer, 0, STREAM_BASIS).standard_normal((d, d))
    qm, r = np.linalg.qr(a)
    return qm * np.sign(np.diag(r))[None, :]


def queries(cfg, layer, stream, n, request=0, d=HEAD_DIM):
    """[n, d] fp64 queries z diag(sigma) B^T of one layer."""
    z = rng(cfg, layer, request, stream).standard_normal((n, d))
    return (z * query_sigma(d)[None, :]) @ query_basis(cfg, layer, d).T


def decode_queries_bf16(cfg, layer, batch, n_q_heads, step=0, d=HEAD_DIM):
    """torch.bfloat16 [batch, H_q, d] decode queries for one layer and step."""
    q = queries(cfg, layer, STREAM_Q, batch * n_q_heads, request=step, d=d)
    return to_bf16(q.reshape(batch, n_q_heads, d))


def shuffled_pages(cfg, num_pages, layer=0):
    """A seeded permutation of range(num_pages) (int32)."""
    return rng(cfg, layer, 0, STREAM_PAGES).permutation(num_pages).astype(np.int32)


def ragged_lengths(cfg, batch, lo, hi, n_shared=0, shared_lo=None):
    """Context lengths ~ U[lo, hi] (inclusive); the first n_shared ~ U[shared_lo, hi]."""
    g = rng(cfg, 0, 0, STREAM_LENS)
    lens = g.integers(lo, hi + 1, size=batch)
    if n_shared:
        lens[:n_shared] = g.integers(shared_lo, hi + 1, size=n_shared)
    return lens.astype(np.int64)
