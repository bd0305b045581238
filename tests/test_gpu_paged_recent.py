"""GPU: the paged BF16 recent window against the ring and the oracle.

With a recent page table the last 256 positions live in BF16 pages (row p % 64
of the page the table names for logical page p / 64) instead of a per-request
ring slot; the window, the evictions and every INT2 byte are the same as with
the ring, and so is every output (the tiles read the same values in the same
order).  Each request here owns five BF16 pages, logical page lp in page
lp % 5 (the window never touches more than five logical pages), so pages are
reused as the window moves, as a serving engine would recycle them.
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
from oracle import attention  # noqa: E402
from oracle import cache as ocache  # noqa: E402


def _pair(Hq, Hkv, Lmax, B, cfg):
    return (harness.Setup(Hq, Hkv, Lmax, B, cfg=cfg, calibrate=False),
            harness.Setup(Hq, Hkv, Lmax, B, cfg=cfg, calibrate=False, paged_recent=True))


def _same_storage(ring, paged, lens):
    """INT2 pages, sink pages and every window row equal in the two modes."""
    assert torch.equal(ring.cache.int2_pages[0].cpu(), paged.cache.int2_pages[0].cpu())
    assert torch.equal(ring.cache.k_sink[0].cpu(), paged.cache.k_sink[0].cpu())
    assert torch.equal(ring.cache.v_sink[0].cpu(), paged.cache.v_sink[0].cpu())
    for b, L in enumerate(lens):
        (_, _), _, (r0, r1) = ocache.segments(L)
        rows = [(p - 64) % 256 for p in range(r0, r1)]
        for x, y in zip(ring.readback(0, b, L), paged.readback(0, b, L)):
            assert np.array_equal(x[2][rows], y[2][rows]) and np.array_equal(x[3][rows], y[3][rows])


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2)])
def test_paged_steps_equal_the_ring(Hq, Hkv):
    """Fused decode steps across the sink boundary, the first eviction and steady state."""
    cfg, lens0, n_steps = 51, [60, 318, 700], 6
    B = len(lens0)
    toks = [inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, L + n_steps, b) for b, L in enumerate(lens0)]
    ring, paged = _pair(Hq, Hkv, max(lens0) + n_steps, B, cfg)
    try:
        cu = np.concatenate([[0], np.cumsum(lens0)]).tolist()
        for s in (ring, paged):
            s.append(0, torch.cat([t[0][:L] for t, L in zip(toks, lens0)]),
                     torch.cat([t[1][:L] for t, L in zip(toks, lens0)]), [0] * B, cu, max(lens0))
            assert s.device_error() == 0
        _same_storage(ring, paged, lens0)
        for step in range(n_steps):
            pos = [L + step for L in lens0]
            lens = [p + 1 for p in pos]
            k = torch.stack([t[0][p] for t, p in zip(toks, pos)]).cuda()
            v = torch.stack([t[1][p] for t, p in zip(toks, pos)]).cuda()
            q = inputs.decode_queries_bf16(cfg, 0, B, Hq, step=step).cuda()
            outs = []
            # the argument structs hold raw pointers: keep every tensor they name alive
            pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
            len_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
            for s in (ring, paged):
                out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
                ap = kvcache.append_args(k, v, pos_t)
                dp = kvcache.decode_args(q, out, len_t, max(lens))
                abi.oscar_decode_step(s.ctx, 0, s.cache.view(0), ap, dp, s.ws, s.ws_bytes,
                                      torch.cuda.current_stream())
                torch.cuda.synchronize()
                assert s.device_error() == 0
                outs.append(out.cpu().numpy().astype(np.float64))
            assert np.isfinite(outs[1]).all()
            assert np.array_equal(outs[0], outs[1]), "step %d" % step
            _same_storage(ring, paged, lens)
        errs = [np.abs(outs[1][b] - paged.oracle_decode(0, b, lens[b], q[b].cpu())).max() for b in range(B)]
        print("paged steps Hq %d Hkv %d: max-abs vs oracle %s" % (Hq, Hkv, ["%.2e" % e for e in errs]))
        assert max(errs) <= harness.DECODE_TOL
    finally:
        ring.close()
        paged.close()


@pytest.mark.parametrize("P,n", [(0, 1000), (0, 4096), (700, 40), (1000, 300), (300, 5)])
def test_paged_bulk_and_chunked_append(P, n):
    """A prefix (bulk) then a chunk: eviction of the old window from its pages, new rows
    into pages, codes bit-exact, decode equal to the ring and within the bound."""
    cfg, Hq, Hkv = 52, 32, 8
    L = P + n
    tk = inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, L, 0)
    ring, paged = _pair(Hq, Hkv, L, 1, cfg)
    try:
        for s in (ring, paged):
            if P:
                s.append(0, tk[0][:P], tk[1][:P], [0], [0, P], P)
            s.append(0, tk[0][P:], tk[1][P:], [P], [0, n], n)
            assert s.device_error() == 0
        _same_storage(ring, paged, [L])
        tok_k, tok_v = inputs.bf16_to_f64(tk[0]), inputs.bf16_to_f64(tk[1])
        n_cmp = n_bad = 0
        for h in range(Hkv):
            c, bad, _, _ = harness.compare_history_codes(paged, 0, 0, L, tok_k[:, h], tok_v[:, h], h)
            n_cmp += c
            n_bad += bad
        assert n_bad == 0
        q = inputs.decode_queries_bf16(cfg, 0, 1, Hq)
        got_r, got_p = ring.decode(0, q, [L]), paged.decode(0, q, [L])
        assert np.array_equal(got_r, got_p)
        err = np.abs(got_p[0] - paged.oracle_decode(0, 0, L, q[0])).max()
        print("paged append P=%d n=%d: %d codes, 0 mismatches; decode max-abs %.2e" % (P, n, n_cmp, err))
        assert err <= harness.DECODE_TOL
    finally:
        ring.close()
        paged.close()


@pytest.mark.parametrize("P,n", [(1000, 40), (2600, 32)])
def test_paged_extend_equals_the_ring(P, n):
    """Both extend paths read the window through the page table.  At P = 2600 the chunk kernel
    splits the history into three page ranges of seven BF16 tiles each, staged in shared memory,
    and the window's wrap point (L mod 256 = 72) falls inside tile 8, whose rows then come from
    two recent pages; at P = 1000 the tiles are read from global memory."""
    cfg, Hq, Hkv = 53, 32, 8
    L = P + n
    tk = inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, L, 0)
    q = inputs.decode_queries_bf16(cfg, 0, n, Hq).reshape(1, n, Hq, 128).cuda()
    ring, paged = _pair(Hq, Hkv, L, 1, cfg)
    try:
        outs = []
        for s in (ring, paged):
            s.append(0, tk[0][:P], tk[1][:P], [0], [0, P], P)
            s.append(0, tk[0][P:], tk[1][P:], [P], [0, n], n)
            wt, wp, nb = kvcache.extend_workspace(s.ctx, 1, n, L)
            out = torch.full((1, n, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            len1 = torch.tensor([L], dtype=torch.int32, device="cuda")
            pos1 = torch.tensor([P], dtype=torch.int32, device="cuda")
            abi.oscar_extend_chunk(s.ctx, 0, s.cache.view(0), q, out, len1, pos1, n, L, wp, nb,
                                   stream=torch.cuda.current_stream())
            view, tabs = s.cache.chunk_view(0, 0, n)
            out1 = torch.full((n, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            lenn = torch.full((n,), L, dtype=torch.int32, device="cuda")
            args = kvcache.decode_args(q[0], out1, lenn, L)
            lim = torch.arange(P + 1, L + 1, dtype=torch.int32, device="cuda")
            wdt, wd, wdb = kvcache.workspace(s.ctx, n, L + 1)  # the per-query path: n batch rows
            abi.oscar_extend_attention(s.ctx, 0, view, args, lim, wd, wdb, torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert s.device_error() == 0
            outs.append((out.cpu().numpy(), out1.cpu().numpy()))
            del wt, wdt, tabs
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
        R_K, R_V, _, _ = paged.rot[0]
        Ks, Vs = [], []
        for (sk, sv, rk, rv, blocks) in paged.readback(0, 0, L):
            K, V = ocache.reconstruct_from_storage(sk, sv, rk, rv, blocks, L, R_K, R_V)
            Ks.append(K)
            Vs.append(V)
        worst = 0.0
        for i in range(0, n, 3):
            ref = attention.decode_gqa(inputs.bf16_to_f64(q[0, i].cpu()), [K[:P + i + 1] for K in Ks],
                                       [V[:P + i + 1] for V in Vs], harness.SM_SCALE)
            worst = max(worst, float(np.abs(outs[1][0][0, i] - ref).max()), float(np.abs(outs[1][1][i] - ref).max()))
        assert worst <= harness.DECODE_TOL
    finally:
        ring.close()
        paged.close()


def test_shared_recent_pages():
    """Two requests alias one prefix's INT2 pages, sink page and BF16 recent pages
    (read-only prefix sharing) and both decode it within the bound."""
    cfg, Hq, Hkv, S = 54, 32, 8, 700
    tk = inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, S, 0)
    s = harness.Setup(Hq, Hkv, S, 2, cfg=cfg, calibrate=False, paged_recent=True)
    try:
        restore = harness.request_view(s, 0, 1)
        try:
            s.append(0, tk[0], tk[1], [0], [0, S], S, batch=1)
        finally:
            restore()
        c = s.cache
        c.page_table[1] = c.page_table[0]
        c.sink_page[1] = c.sink_page[0]
        c.recent_table[1] = c.recent_table[0]
        q = inputs.decode_queries_bf16(cfg, 0, 2, Hq)
        got = s.decode(0, q, [S, S])
        assert s.device_error() == 0
        for b in range(2):
            err = np.abs(got[b] - s.oracle_decode(0, b, S, q[b])).max()
            assert err <= harness.DECODE_TOL
    finally:
        s.close()


def test_bad_recent_page_sets_the_ring_bit():
    """A recent page id outside the pool is a device error bit; nothing faults."""
    cfg, Hq, Hkv, L = 55, 32, 8, 500
    tk = inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, L, 0)
    s = harness.Setup(Hq, Hkv, L, 1, cfg=cfg, calibrate=False, paged_recent=True)
    try:
        s.append(0, tk[0], tk[1], [0], [0, L], L)
        assert s.device_error() == 0
        s.cache.recent_table[0, (L - 1) // 64] = 10 ** 6
        q = inputs.decode_queries_bf16(cfg, 0, 1, Hq)
        s.decode(0, q, [L])
        err = s.device_error()
        assert err & abi.OSCAR_DEVERR_RING, err
    finally:
        s.close()
