"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Append: packed codes bit-exact per (token, channel) except values within
1e-6 * s of a decision edge (excluded and counted) and groups whose a/1.5 sits
within 1e-6 of an fp16 rounding midpoint; fp16 scales exact otherwise; BF16
sink/recent rows exact.  Decode: max-abs <= 2e-3 against the oracle run on the
GPU's own stored cache (BF16-only contexts: max|diff| / max|ref| <= 1e-2 per
head as well).
"""

import numpy as np
import pytest
import torch

from int2_rotated_kv_oscar_gb300 import abi, inputs
from oracle import cache as ocache

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import harness  # noqa: E402


def _tokens(cfg, layer, Hkv, n, request=0):
    return inputs.kv_tokens_bf16(cfg, layer, Hkv, inputs.STREAM_KV, n, request)


def _check_codes(s, layer, b, L, k, v, tag):
    tk = inputs.bf16_to_f64(k)
    tv = inputs.bf16_to_f64(v)
    tot = [0, 0, 0, 0]
    for h in range(s.Hkv):
        r = harness.compare_history_codes(s, layer, b, L, tk[:, h], tv[:, h], h)
        tot = [a + c for a, c in zip(tot, r)]
    n_cmp, n_bad, n_edge, n_mid = tot
    print("%s: compared %d codes, %d mismatches, %d near-edge excluded, %d midpoint groups" % (tag, n_cmp, n_bad,
                                                                                                n_edge, n_mid))
    assert n_bad == 0
    return tot


def _check_bf16_rows(s, layer, b, L, k, v):
    (s0, s1), _, (r0, r1) = ocache.segments(L)
    tk = inputs.bf16_to_f64(k)
    tv = inputs.bf16_to_f64(v)
    for h, (sk, sv, rk, rv, _) in enumerate(s.readback(layer, b, L)):
        assert np.array_equal(sk[s0:s1], tk[s0:s1, h]) and np.array_equal(sv[s0:s1], tv[s0:s1, h])
        for p in range(r0, r1):
            slot = ocache.ring_slot(p)
            assert np.array_equal(rk[slot], tk[p, h]) and np.array_equal(rv[slot], tv[p, h])


def test_c1_single_layer_prefill_append_decode():
    """Single layer, 1 request, GQA 8/2, context 4096 = 64 sink + 3776 INT2 + 256 recent."""
    cfg, L = 1, 4096
    s = harness.Setup(8, 2, L, 1, cfg=cfg)
    try:
        k, v = _tokens(cfg, 0, 2, L)
        s.append(0, k[:L - 1], v[:L - 1], [0], [0, L - 1], L - 1)
        s.append(0, k[L - 1:], v[L - 1:], [L - 1])          # the decode step's own token
        assert s.device_error() == 0
        _check_bf16_rows(s, 0, 0, L, k, v)
        _check_codes(s, 0, 0, L, k, v, "c1")
        q = inputs.decode_queries_bf16(cfg, 0, 1, 8)
        out = s.decode(0, q, [L])
        assert s.device_error() == 0
        ref = s.oracle_decode(0, 0, L, q[0])
        err = np.abs(out[0] - ref).max()
        print("c1 decode max-abs %.3e, rel-linf %.3e" % (err, err / np.abs(ref).max()))
        assert err <= harness.DECODE_TOL
    finally:
        s.close()


@pytest.mark.parametrize("Hq,Hkv,tau_scale", [(6, 3, 1.0), (6, 3, 0.25), (32, 8, 0.25)])
def test_bulk_append_clipping_and_odd_head_counts(Hq, Hkv, tau_scale):
    """Bulk prefill append with thresholds far below the calibrated ones (most groups clip, so
    the codes come from the three comparisons rather than the floor of x / s + 2) and with 3 KV
    heads (the BF16 rows' 16-byte copies cover heads t / 16, t / 16 + 8, ...): codes bit-exact,
    BF16 rows exact, decode within the bound."""
    cfg, L = 3, 2500
    s = harness.Setup(Hq, Hkv, L, 1, cfg=cfg, tau_scale=tau_scale)
    try:
        k, v = _tokens(cfg, 0, Hkv, L)
        s.append(0, k, v, [0], [0, L], L)
        assert s.device_error() == 0
        _check_bf16_rows(s, 0, 0, L, k, v)
        _check_codes(s, 0, 0, L, k, v, "bulk Hkv=%d tau x %.2f" % (Hkv, tau_scale))
        q = inputs.decode_queries_bf16(cfg, 0, 1, Hq)
        out = s.decode(0, q, [L])
        assert s.device_error() == 0
        ref = s.oracle_decode(0, 0, L, q[0])
        err = np.abs(out[0] - ref).max()
        print("bulk Hkv=%d tau x %.2f: decode max-abs %.3e" % (Hkv, tau_scale, err))
        assert err <= harness.DECODE_TOL
    finally:
        s.close()


@pytest.mark.parametrize("L", [1, 63, 64, 65, 320, 321, 384, 1000, 4096])
def test_edge_lengths_incremental(L):
    """Contexts built token by token through the decode append (eviction at every step past 320)."""
    cfg = 2
    s = harness.Setup(8, 2, L, 1, cfg=cfg, calibrate=False)
    try:
        k, v = _tokens(cfg, 0, 2, L)
        pre = max(0, L - 70)
        if pre:
            s.append(0, k[:pre], v[:pre], [0], [0, pre], pre)
        for p in range(pre, L):
            s.append(0, k[p:p + 1], v[p:p + 1], [p])
        assert s.device_error() == 0
        _check_bf16_rows(s, 0, 0, L, k, v)
        _check_codes(s, 0, 0, L, k, v, "L=%d" % L)
        q = inputs.decode_queries_bf16(cfg, 0, 1, 8, step=L)
        out = s.decode(0, q, [L])
        ref = s.oracle_decode(0, 0, L, q[0])
        err = np.abs(out[0] - ref).max()
        assert err <= harness.DECODE_TOL, err
        if L <= 320:  # BF16-only context
            for hq in range(8):
                assert np.abs(out[0, hq] - ref[hq]).max() <= harness.BF16_REL_TOL * np.abs(ref[hq]).max()
    finally:
        s.close()


def test_batch_ragged_gqa8_shuffled_pages():
    """64 query / 8 KV heads (GQA 8), ragged lengths, shuffled page tables, multi-token appends."""
    cfg = 5
    lens = [70, 321, 700, 1500, 2900]
    B = len(lens)
    s = harness.Setup(64, 8, max(lens), B, cfg=cfg, calibrate=False)
    try:
        toks = [_tokens(cfg, 0, 8, L, request=b) for b, L in enumerate(lens)]
        k = torch.cat([t[0] for t in toks])
        v = torch.cat([t[1] for t in toks])
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        s.append(0, k, v, [0] * B, cu, max(lens))
        assert s.device_error() == 0
        for b, L in enumerate(lens):
            _check_bf16_rows(s, 0, b, L, *toks[b])
            _check_codes(s, 0, b, L, *toks[b], "gqa8 b=%d" % b)
        q = inputs.decode_queries_bf16(cfg, 0, B, 64)
        out = s.decode(0, q, lens)
        assert s.device_error() == 0
        for b, L in enumerate(lens):
            ref = s.oracle_decode(0, b, L, q[b])
            err = np.abs(out[b] - ref).max()
            assert err <= harness.DECODE_TOL, (b, err)
    finally:
        s.close()


def test_chunked_prefill_then_decode_steps():
    """A prompt appended in uneven chunks (phase-1 eviction from the ring), then decode steps."""
    cfg = 3
    L = 1800
    s = harness.Setup(32, 8, L + 8, 1, cfg=cfg, calibrate=False)
    try:
        k, v = _tokens(cfg, 0, 8, L + 8)
        p = 0
        for n in (100, 250, 1, 700, 749):
            s.append(0, k[p:p + n], v[p:p + n], [p], [0, n], n)
            p += n
        assert p == L
        q = inputs.decode_queries_bf16(cfg, 0, 1, 32)
        for step in range(8):
            s.append(0, k[p:p + 1], v[p:p + 1], [p])
            p += 1
            out = s.decode(0, q, [p])
            ref = s.oracle_decode(0, 0, p, q[0])
            assert np.abs(out[0] - ref).max() <= harness.DECODE_TOL
        assert s.device_error() == 0
        _check_codes(s, 0, 0, p, k[:p], v[:p], "chunked")
        _check_bf16_rows(s, 0, 0, p, k[:p], v[:p])
    finally:
        s.close()


def test_shared_prefix_aliased_pages():
    """Requests 1.. alias request 0's prefix pages and sink page; their own tokens are
    appended with OSCAR_APPEND_FRESH_RING (the prefix is already sink/history)."""
    cfg = 5
    prefix = 64 * 40
    lens = [prefix + 700, prefix + 300, prefix + 256]
    B = len(lens)
    s = harness.Setup(16, 2, max(lens), B, cfg=cfg, calibrate=False)
    try:
        n_pre = prefix // 64
        pt = s.cache.page_table
        for b in range(1, B):
            pt[b, :n_pre] = pt[0, :n_pre]
        s.cache.sink_page.zero_()            # one shared sink page
        k0, v0 = _tokens(cfg, 0, 2, lens[0], request=0)
        s.append(0, k0, v0, [0], [0, lens[0]], lens[0], batch=1)
        kk, vv, cu = [], [], [0]
        for b in range(1, B):
            kb, vb = _tokens(cfg, 0, 2, lens[b], request=b)
            kk.append(kb[prefix:])
            vv.append(vb[prefix:])
            cu.append(cu[-1] + lens[b] - prefix)
        # requests 1..B-1 only: a view whose row 0 is request 1
        view_pt = pt[1:].contiguous()
        s.cache.page_table = view_pt
        s.cache.sink_page = s.cache.sink_page[1:].contiguous()
        s.cache.ring_slot = s.cache.ring_slot[1:].contiguous()
        s.append(0, torch.cat(kk), torch.cat(vv), [prefix] * (B - 1), cu, max(lens) - prefix, fresh=True,
                 batch=B - 1)
        s.cache.page_table = pt
        s.cache.sink_page = torch.zeros(B, dtype=torch.int32, device="cuda")
        s.cache.ring_slot = torch.arange(B, dtype=torch.int32, device="cuda")
        assert s.device_error() == 0
        q = inputs.decode_queries_bf16(cfg, 0, B, 16)
        out = s.decode(0, q, lens)
        for b, L in enumerate(lens):
            ref = s.oracle_decode(0, b, L, q[b])
            assert np.abs(out[b] - ref).max() <= harness.DECODE_TOL, b
        # the shared part of request 1 equals request 0's tokens
        kb1, vb1 = _tokens(cfg, 0, 2, lens[1], request=1)
        kfull = torch.cat([k0[:prefix], kb1[prefix:]])
        vfull = torch.cat([v0[:prefix], vb1[prefix:]])
        _check_codes(s, 0, 1, lens[1], kfull, vfull, "prefix b=1")
    finally:
        s.close()


@pytest.mark.parametrize("flags", [0, abi.OSCAR_ROT_H | abi.OSCAR_ROT_P, abi.OSCAR_ROT_U, abi.OSCAR_ROT_U | abi.OSCAR_ROT_H])
def test_rotation_ablations(flags):
    """Naive INT2 (R = I), Hadamard-only (H P), U-only, U H: same kernels, R is data."""
    cfg, L = 4, 1200
    s = harness.Setup(8, 2, L, 1, cfg=cfg, flags=flags, calibrate=False)
    try:
        k, v = _tokens(cfg, 0, 2, L)
        s.append(0, k, v, [0], [0, L], L)
        _check_codes(s, 0, 0, L, k, v, "flags=%d" % flags)
        q = inputs.decode_queries_bf16(cfg, 0, 1, 8)
        out = s.decode(0, q, [L])
        ref = s.oracle_decode(0, 0, L, q[0])
        assert np.abs(out[0] - ref).max() <= harness.DECODE_TOL
    finally:
        s.close()


def test_empty_context_gives_zeros_and_sm_scale():
    s = harness.Setup(8, 2, 600, 2, cfg=6, calibrate=False)
    try:
        k, v = _tokens(6, 0, 2, 600)
        s.append(0, k, v, [0, 0], [0, 600, 600], 600)
        q = inputs.decode_queries_bf16(6, 0, 2, 8)
        out = s.decode(0, q, [600, 0])
        assert np.all(out[1] == 0.0)
        ref = s.oracle_decode(0, 0, 600, q[0])
        assert np.abs(out[0] - ref).max() <= harness.DECODE_TOL
    finally:
        s.close()


def test_bad_page_id_sets_device_error_and_gpu_stays_usable():
    s = harness.Setup(8, 2, 1000, 1, cfg=7, calibrate=False)
    try:
        k, v = _tokens(7, 0, 2, 1000)
        s.append(0, k, v, [0], [0, 1000], 1000)
        assert s.device_error() == 0
        saved = s.cache.page_table.clone()
        s.cache.page_table[0, 3] = 10 ** 6
        q = inputs.decode_queries_bf16(7, 0, 1, 8)
        s.decode(0, q, [1000])
        assert s.device_error() & abi.OSCAR_DEVERR_PAGE
        s.cache.page_table.copy_(saved)
        out = s.decode(0, q, [1000])
        assert s.device_error() == 0
        assert np.abs(out[0] - s.oracle_decode(0, 0, 1000, q[0])).max() <= harness.DECODE_TOL
    finally:
        s.close()


def test_host_argument_errors_launch_nothing():
    s = harness.Setup(8, 2, 500, 1, cfg=7, calibrate=False)
    try:
        v = s.cache.view(0)
        q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((1, 8, 128), dtype=torch.float32, device="cuda")
        lens = torch.tensor([10], dtype=torch.int32, device="cuda")
        from int2_rotated_kv_oscar_gb300 import cache as kvcache
        args = kvcache.decode_args(q, out, lens, 10)
        with pytest.raises(abi.OscarError) as e:
            abi.oscar_decode_attention(s.ctx, 0, v, args, s.ws, 16, None)
        assert e.value.status == 6
        with pytest.raises(abi.OscarError) as e:
            abi.oscar_decode_attention(s.ctx, 5, v, args, s.ws, s.ws_bytes, None)
        assert e.value.status == 1
        with pytest.raises(abi.OscarError):
            abi.oscar_load_rotation(s.ctx, 0, np.eye(128), np.eye(128), 1e6, 1.0)
        # k, v must be 16-byte aligned (the bulk append reads them by TMA)
        kv = torch.zeros((2 * 100 * 2 * 128 + 8,), dtype=torch.bfloat16, device="cuda")
        k_bad = kv[1:1 + 100 * 2 * 128].view(100, 2, 128)
        pos = torch.zeros(1, dtype=torch.int32, device="cuda")
        cu = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
        with pytest.raises(abi.OscarError) as e:
            abi.oscar_kv_append(s.ctx, 0, v, kvcache.append_args(k_bad, k_bad, pos, cu, 100), None)
        assert e.value.status == 1
        assert s.device_error() == 0
    finally:
        s.close()


@pytest.mark.parametrize("lens", [[1, 130, 2000], [100_000]])
def test_bf16_comparator_matches_plain_attention(lens):
    """The BF16 paged-cache decode (the comparator) against plain attention: short and
    partial pages, and a 100K context (long rings of staged tile halves per warp)."""
    from int2_rotated_kv_oscar_gb300 import cache as kvcache
    from oracle import attention
    cfg = 8
    B, Hq, Hkv = len(lens), 32, 8
    s = harness.Setup(Hq, Hkv, max(lens), B, cfg=cfg, calibrate=False)
    try:
        maxp = (max(lens) + 63) // 64
        bc = kvcache.BF16PagedCache(Hkv, B * maxp, B, maxp)
        bc.page_table.copy_(torch.from_numpy(inputs.shuffled_pages(cfg, B * maxp).reshape(B, maxp)))
        toks = []
        for b, L in enumerate(lens):
            k, v = _tokens(cfg, 0, Hkv, L, request=b)
            toks.append((k, v))
            for i in range((L + 63) // 64):
                ph = int(bc.page_table[b, i])
                n = min(64, L - 64 * i)
                bc.k_pages[ph, :, :n] = k[64 * i:64 * i + n].transpose(0, 1).cuda()
                bc.v_pages[ph, :, :n] = v[64 * i:64 * i + n].transpose(0, 1).cuda()
        q = inputs.decode_queries_bf16(cfg, 0, B, Hq)
        out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
        args = kvcache.decode_args(q.cuda(), out, torch.tensor(lens, dtype=torch.int32, device="cuda"), max(lens))
        abi.oscar_decode_attention_bf16(s.ctx, bc.view(), args, s.ws, s.ws_bytes, None)
        assert s.device_error() == 0
        o = out.cpu().numpy()
        for b, L in enumerate(lens):
            k, v = toks[b]
            tk, tv = inputs.bf16_to_f64(k), inputs.bf16_to_f64(v)
            ref = attention.decode_gqa(inputs.bf16_to_f64(q[b]), [tk[:, h] for h in range(Hkv)],
                                       [tv[:, h] for h in range(Hkv)], harness.SM_SCALE)
            assert np.abs(o[b] - ref).max() <= harness.DECODE_TOL
            for hq in range(Hq):
                assert np.abs(o[b, hq] - ref[hq]).max() <= harness.BF16_REL_TOL * np.abs(ref[hq]).max()
    finally:
        s.close()
