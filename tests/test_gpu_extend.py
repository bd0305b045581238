"""GPU: extend (chunk) attention over the mixed cache against the oracle.

A request's prefix of P tokens and then a chunk of n tokens are appended
(two bulk appends); the chunk's n queries -- batch rows whose tables alias
the request's pages, sink page and ring slot -- attend, causally, to the
cache as it stands after the chunk's append: query i sees positions
p < P + i + 1, the sink and recent rows in BF16 and the older history in
INT2 (the split follows the cache length P + n).  The oracle reconstructs
the request's stored cache and runs plain softmax attention over each
query's positions.
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


@pytest.mark.parametrize("P,n,Hq,Hkv,cfg", [(10, 40, 8, 2, 31),      # sink only
                                             (100, 300, 32, 8, 32),   # history, wrapped ring, limits in both
                                             (1000, 8, 32, 8, 33),
                                             (5000, 64, 16, 2, 34)])  # GQA 8
def test_extend_attention_matches_the_oracle(P, n, Hq, Hkv, cfg):
    L = P + n
    s = harness.Setup(Hq, Hkv, L, n, cfg=cfg)
    try:
        toks = inputs.kv_tokens_device(cfg, 0, Hkv, inputs.STREAM_KV, L, "cuda", request=0)
        restore = harness.request_view(s, 0, 1)
        try:
            s.append(0, toks[0][:P], toks[1][:P], [0], [0, P], P, batch=1)
            s.append(0, toks[0][P:], toks[1][P:], [P], [0, n], n, batch=1)
        finally:
            restore()
        c = s.cache
        c.page_table[1:n] = c.page_table[0]
        c.sink_page[1:n] = c.sink_page[0]
        c.ring_slot[1:n] = c.ring_slot[0]
        q = inputs.decode_queries_bf16(cfg, 0, n, Hq)
        out = torch.full((n, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ctx_len = torch.full((n,), L, dtype=torch.int32, device="cuda")
        limit = torch.arange(P + 1, L + 1, dtype=torch.int32, device="cuda")
        args = kvcache.decode_args(q.cuda(), out, ctx_len, L)
        abi.oscar_extend_attention(s.ctx, 0, c.view(0), args, limit, s.ws, s.ws_bytes, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert s.device_error() == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        R_K, R_V, _, _ = s.rot[0]
        Ks, Vs = [], []
        for (sk, sv, rk, rv, blocks) in s.readback(0, 0, L):
            K, V = ocache.reconstruct_from_storage(sk, sv, rk, rv, blocks, L, R_K, R_V)
            Ks.append(K)
            Vs.append(V)
        rows = range(n) if n <= 64 else sorted(set(list(range(0, n, 7)) + [n - 1]))
        errs = []
        for i in rows:
            lim = P + i + 1
            ref = attention.decode_gqa(inputs.bf16_to_f64(q[i]), [K[:lim] for K in Ks], [V[:lim] for V in Vs],
                                       harness.SM_SCALE)
            errs.append(np.abs(got[i] - ref).max())
        print("extend P=%d n=%d: max-abs vs oracle %.2e over %d queries" % (P, n, max(errs), len(errs)))
        assert max(errs) <= harness.DECODE_TOL
    finally:
        s.close()


def test_extend_with_the_whole_cache_equals_decode():
    """limit = ctx_len: every query attends the whole cache, exactly as the decode does."""
    cfg, Hq, Hkv, L, B = 35, 32, 8, 3000, 3
    s = harness.Setup(Hq, Hkv, L, B, cfg=cfg)
    try:
        for b in range(B):
            toks = inputs.kv_tokens_device(cfg, 0, Hkv, inputs.STREAM_KV, L, "cuda", request=b)
            restore = harness.request_view(s, b, b + 1)
            try:
                s.append(0, toks[0], toks[1], [0], [0, L], L, batch=1)
            finally:
                restore()
        q = inputs.decode_queries_bf16(cfg, 0, B, Hq)
        dec = s.decode(0, q, [L] * B)
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ctx_len = torch.full((B,), L, dtype=torch.int32, device="cuda")
        args = kvcache.decode_args(q.cuda(), out, ctx_len, L)
        abi.oscar_extend_attention(s.ctx, 0, s.cache.view(0), args, ctx_len, s.ws, s.ws_bytes,
                                   torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert s.device_error() == 0
        assert np.array_equal(out.cpu().numpy().astype(np.float64), dec)
    finally:
        s.close()


def _extend_chunk(s, q, B, n, L, P):
    out = torch.full((B, n, s.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ctx_len = torch.full((B,), L, dtype=torch.int32, device="cuda")
    pos0 = torch.full((B,), P, dtype=torch.int32, device="cuda")
    nbytes = abi.oscar_extend_workspace_bytes(s.ctx, B, n, L)
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device="cuda")
    wptr = ws.data_ptr() + (-ws.data_ptr()) % 256
    abi.oscar_extend_chunk(s.ctx, 0, s.cache.view(0), q, out, ctx_len, pos0, n, L, wptr, nbytes,
                           stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("P,n,B,Hq,Hkv,cfg", [(10, 40, 1, 32, 8, 41),      # sink only
                                              (100, 300, 1, 32, 8, 42),    # 19 query groups, wrapped ring
                                              (1000, 8, 2, 16, 8, 43),     # GQA 2, half a group
                                              (5000, 33, 2, 32, 8, 44)])   # a group with one query
def test_extend_chunk_matches_the_oracle(P, n, B, Hq, Hkv, cfg):
    """The shared-unpack chunk kernel: one block per (request, KV head, 128 / g queries)."""
    L = P + n
    s = harness.Setup(Hq, Hkv, L, B, cfg=cfg)
    try:
        for b in range(B):
            tk = inputs.kv_tokens_device(cfg, 0, Hkv, inputs.STREAM_KV, L, "cuda", request=b)
            restore = harness.request_view(s, b, b + 1)
            try:
                s.append(0, tk[0][:P], tk[1][:P], [0], [0, P], P, batch=1)
                s.append(0, tk[0][P:], tk[1][P:], [P], [0, n], n, batch=1)
            finally:
                restore()
        q = inputs.decode_queries_bf16(cfg, 0, B * n, Hq).reshape(B, n, Hq, 128)
        out = _extend_chunk(s, q.cuda(), B, n, L, P)
        assert s.device_error() == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        R_K, R_V, _, _ = s.rot[0]
        worst = 0.0
        for b in range(B):
            Ks, Vs = [], []
            for (sk, sv, rk, rv, blocks) in s.readback(0, b, L):
                K, V = ocache.reconstruct_from_storage(sk, sv, rk, rv, blocks, L, R_K, R_V)
                Ks.append(K)
                Vs.append(V)
            rows = range(n) if n <= 64 else sorted(set(list(range(0, n, 7)) + [n - 1]))
            for i in rows:
                lim = P + i + 1
                ref = attention.decode_gqa(inputs.bf16_to_f64(q[b, i]), [K[:lim] for K in Ks],
                                           [V[:lim] for V in Vs], harness.SM_SCALE)
                worst = max(worst, float(np.abs(got[b, i] - ref).max()))
        print("extend chunk P=%d n=%d B=%d: max-abs vs oracle %.2e" % (P, n, B, worst))
        assert worst <= harness.DECODE_TOL
    finally:
        s.close()


def test_extend_chunk_refuses_gqa_above_4():
    s = harness.Setup(64, 8, 200, 1, cfg=45, calibrate=False)
    try:
        q = torch.zeros((1, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(abi.OscarError) as e:
            _extend_chunk(s, q, 1, 4, 200, 196)
        assert e.value.status == 2  # OSCAR_ERR_UNSUPPORTED
    finally:
        s.close()


@pytest.mark.parametrize("path,n", [("per_query", 16), ("per_query", 256), ("chunk", 16), ("chunk", 40),
                                    ("chunk", 64), ("chunk", 256)])
def test_extend_after_a_100k_prefix(path, n):
    """Both extend paths at the sizes the benchmark times: a chunk of n tokens after a
    100,000-token prefix (long page loops per block, many work items per (query, KV
    head), the records' merge at full width), checked on sampled queries.  The chunk
    kernel splits the history into 19, 9 and 7 page ranges for n = 16, 64 and 256 (two,
    three and three BF16 tiles staged per range); at n = 40 its second query group holds
    8 of 32 queries."""
    cfg, Hq, Hkv, P = 46, 32, 8, 100_000
    L = P + n
    s = harness.Setup(Hq, Hkv, L, 1, cfg=cfg)
    try:
        tk = inputs.kv_tokens_device(cfg, 0, Hkv, inputs.STREAM_KV, L, "cuda")
        s.append(0, tk[0][:P], tk[1][:P], [0], [0, P], P)
        s.append(0, tk[0][P:], tk[1][P:], [P], [0, n], n)
        del tk
        q = inputs.decode_queries_bf16(cfg, 0, n, Hq)
        if path == "per_query":
            out = torch.full((n, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            ctx_len = torch.full((n,), L, dtype=torch.int32, device="cuda")
            limit = torch.arange(P + 1, L + 1, dtype=torch.int32, device="cuda")
            ws_t, ws, ws_bytes = kvcache.workspace(s.ctx, n, L)
            view, _tables = s.cache.chunk_view(0, 0, n)
            abi.oscar_extend_attention(s.ctx, 0, view, kvcache.decode_args(q.cuda(), out, ctx_len, L), limit, ws,
                                       ws_bytes, torch.cuda.current_stream())
            torch.cuda.synchronize()
            got = out.cpu().numpy().astype(np.float64)
        else:
            got = _extend_chunk(s, q.reshape(1, n, Hq, 128).cuda(), 1, n, L, P)[0].cpu().numpy().astype(np.float64)
        assert s.device_error() == 0
        assert np.isfinite(got).all()
        R_K, R_V, _, _ = s.rot[0]
        Ks, Vs = [], []
        for (sk, sv, rk, rv, blocks) in s.readback(0, 0, L):
            K, V = ocache.reconstruct_from_storage(sk, sv, rk, rv, blocks, L, R_K, R_V)
            Ks.append(K)
            Vs.append(V)
        rows = sorted({0, n // 3, (2 * n) // 3, n - 1})
        errs = []
        for i in rows:
            lim = P + i + 1
            ref = attention.decode_gqa(inputs.bf16_to_f64(q[i]), [K[:lim] for K in Ks], [V[:lim] for V in Vs],
                                       harness.SM_SCALE)
            errs.append(float(np.abs(got[i] - ref).max()))
        print("extend %s after 100K, chunk %d: max-abs vs oracle %.2e over queries %s"
              % (path, n, max(errs), rows))
        assert max(errs) <= harness.DECODE_TOL
    finally:
        s.close()
