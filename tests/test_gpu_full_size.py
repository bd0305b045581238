"""GPU parity at the full sizes of the decode and append workloads.

The oracle cannot redo these contexts whole in seconds, so each test checks
sampled outputs it can compute one by one -- whole requests of the decode
batch, whole pages of the INT2 history -- plus properties that hold at any
size (every output finite, no device error).  Inputs are drawn on the device
by the seeded generators; the oracle reads them back as its inputs.

* 100K-token context, 32 query / 8 KV heads, a decode loop of fused steps
  through the eviction path;
* 28 requests x 100K tokens, 32 query / 8 KV heads, shuffled page tables;
* bulk append of 131,072 tokens x 8 KV heads: sampled INT2 pages bit-exact;
* 64 ragged requests (8K..128K tokens), 64 query / 8 KV heads, the first 16
  sharing a 32K-token prefix through aliased page-table entries.
"""

import numpy as np
import pytest
import torch

from int2_rotated_kv_oscar_gb300 import abi, inputs
from int2_rotated_kv_oscar_gb300 import cache as kvcache

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import harness  # noqa: E402


def _device_tokens(cfg, Hkv, n, request):
    return inputs.kv_tokens_device(cfg, 0, Hkv, inputs.STREAM_KV, n, "cuda", request=request)


def _prefill(s, cfg, lens, b0=0, start=None, fresh=False, request_ids=None):
    """Append requests b0 .. b0 + len(lens) - 1 from position start[i] (default 0)
    to lens[i] in one call; returns the device token tensors per request."""
    B = len(lens)
    start = start or [0] * B
    ids = request_ids or list(range(b0, b0 + B))
    toks = [_device_tokens(cfg, s.Hkv, L, r) for L, r in zip(lens, ids)]
    k = torch.cat([t[0][p:] for t, p in zip(toks, start)])
    v = torch.cat([t[1][p:] for t, p in zip(toks, start)])
    cu = [0]
    for L, p in zip(lens, start):
        cu.append(cu[-1] + L - p)
    restore = harness.request_view(s, b0, b0 + B)
    try:
        s.append(0, k, v, list(start), cu, max(L - p for L, p in zip(lens, start)), fresh=fresh, batch=B)
    finally:
        restore()
    del k, v
    return toks


def _check_decode(s, out, q, lens, sample, tag):
    assert np.isfinite(out).all()
    errs = []
    for b in sample:
        ref = s.oracle_decode(0, b, lens[b], q[b])
        errs.append(np.abs(out[b] - ref).max())
    print("%s: max-abs vs oracle on requests %s: %s" % (tag, list(sample), ["%.2e" % e for e in errs]))
    assert max(errs) <= harness.DECODE_TOL


def _check_pages(s, b, tok, lpages, tag):
    rows = np.concatenate([np.arange(64 * i, 64 * i + 64) for i in lpages])
    idx = torch.from_numpy(rows).cuda()
    tk = inputs.bf16_to_f64(tok[0][idx])
    tv = inputs.bf16_to_f64(tok[1][idx])
    n_cmp, n_bad, n_edge, n_mid = harness.compare_sampled_pages(s, 0, b, lpages, tk, tv)
    print("%s: %d pages, compared %d codes, %d mismatches, %d near-edge excluded, %d midpoint groups"
          % (tag, len(lpages), n_cmp, n_bad, n_edge, n_mid))
    assert n_cmp > 0 and n_bad == 0


def test_100k_context_decode_loop_of_fused_steps():
    """One layer of the 36-layer 100K workload: prefill 100,000 tokens, then 16
    fused decode steps (append with eviction + decode), checked at the end."""
    cfg, Hq, Hkv, L0, steps = 2, 32, 8, 100_000, 16
    s = harness.Setup(Hq, Hkv, L0 + steps, 1, cfg=cfg)
    try:
        toks = _device_tokens(cfg, Hkv, L0 + steps, 0)
        restore = harness.request_view(s, 0, 1)
        try:
            s.append(0, toks[0][:L0], toks[1][:L0], [0], [0, L0], L0, batch=1)
        finally:
            restore()
        out = torch.empty((1, Hq, 128), dtype=torch.float32, device="cuda")
        for j in range(steps):
            p = L0 + j
            q = inputs.decode_queries_bf16(cfg, 0, 1, Hq, step=j)
            pos = torch.tensor([p], dtype=torch.int32, device="cuda")
            ap = kvcache.append_args(toks[0][p:p + 1], toks[1][p:p + 1], pos)
            dp = kvcache.decode_args(q.cuda(), out, pos + 1, L0 + steps)
            abi.oscar_decode_step(s.ctx, 0, s.cache.view(0), ap, dp, s.ws, s.ws_bytes, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert s.device_error() == 0
        L = L0 + steps
        _check_decode(s, out.cpu().numpy().astype(np.float64), q, [L], [0], "100K loop")
        # the pages the loop's evictions wrote, and a spread of prefill pages
        last = (L - 256) // 64 - 1
        _check_pages(s, 0, toks, [1, 2, 500, 1000, last - 1], "100K pages")
    finally:
        s.close()


def test_batch_28_requests_at_100k():
    """28 concurrent 100,000-token requests in one paged pool, one decode step."""
    cfg, Hq, Hkv, L, B = 3, 32, 8, 100_000, 28
    s = harness.Setup(Hq, Hkv, L, B, cfg=cfg)
    try:
        toks = None
        for b0 in range(0, B, 7):
            toks = _prefill(s, cfg, [L] * 7, b0=b0)
        assert s.device_error() == 0
        q = inputs.decode_queries_bf16(cfg, 0, B, Hq)
        out = s.decode(0, q, [L] * B)
        assert s.device_error() == 0
        _check_decode(s, out, q, [L] * B, [0, 13, 27], "28 x 100K")
        # pages of the last request appended (request 27)
        _check_pages(s, 27, toks[-1], [1, 777, 1557], "28 x 100K pages b=27")
    finally:
        s.close()


def test_bulk_append_131072_tokens_8_heads():
    """Prefill-append of 131,072 tokens x 8 KV heads: sampled INT2 pages bit-exact,
    sink and recent rows exact."""
    cfg, Hkv, L = 4, 8, 131_072
    s = harness.Setup(8, Hkv, L, 1, cfg=cfg)
    try:
        toks = _prefill(s, cfg, [L])[0]
        assert s.device_error() == 0
        n_hist_pages = (L - 256) // 64 - 1
        rng = np.random.default_rng(0)
        lpages = sorted(set([1, n_hist_pages] + rng.integers(1, n_hist_pages + 1, size=30).tolist()))
        _check_pages(s, 0, toks, lpages, "bulk append")
        c = s.cache
        sp, rs = int(c.sink_page[0]), int(c.ring_slot[0])
        assert torch.equal(c.k_sink[0][sp].transpose(0, 1), toks[0][:64])
        assert torch.equal(c.v_sink[0][sp].transpose(0, 1), toks[1][:64])
        ring_pos = torch.arange(L - 256, L, device="cuda")
        rows = (ring_pos - 64) % 256
        assert torch.equal(c.k_ring[0][rs][:, rows].transpose(0, 1), toks[0][L - 256:])
        assert torch.equal(c.v_ring[0][rs][:, rows].transpose(0, 1), toks[1][L - 256:])
    finally:
        s.close()


def test_ragged_64_requests_with_shared_prefix():
    """64 requests, lengths ~ U[8K, 128K], the first 16 sharing a 32K-token prefix
    (aliased history pages and sink page), GQA 8; one decode step each."""
    cfg, Hq, Hkv, B, n_shared, prefix = 5, 64, 8, 64, 16, 32 * 1024
    lens = inputs.ragged_lengths(cfg, B, 8 * 1024, 128 * 1024, n_shared=n_shared, shared_lo=prefix + 1024)
    lens = [int(x) for x in lens]
    s = harness.Setup(Hq, Hkv, max(lens), B, cfg=cfg, calibrate=False)
    try:
        pt = s.cache.page_table
        n_pre = prefix // 64
        for b in range(1, n_shared):
            pt[b, :n_pre] = pt[0, :n_pre]
            s.cache.sink_page[b] = s.cache.sink_page[0]
        # request 0 whole; requests 1..15 only their suffix, over a fresh ring
        toks0 = _prefill(s, cfg, [lens[0]], b0=0)[0]
        _prefill(s, cfg, lens[1:n_shared], b0=1, start=[prefix] * (n_shared - 1), fresh=True)
        for b0 in range(n_shared, B, 8):
            _prefill(s, cfg, lens[b0:b0 + 8], b0=b0)
        assert s.device_error() == 0
        q = inputs.decode_queries_bf16(cfg, 0, B, Hq)
        out = s.decode(0, q, lens)
        assert s.device_error() == 0
        _check_decode(s, out, q, lens, [0, 7, 15, 16, 40, 63], "ragged 64")
        # request 0's prefix pages are request 7's too
        _check_pages(s, 7, toks0, [1, n_pre // 2, n_pre - 1], "shared prefix via b=7")
    finally:
        s.close()
