"""Shared setup for the GPU parity tests: seeded inputs, GPU cache, oracle checks.

The CUDA path is driven only through the C ABI (``int2_rotated_kv_oscar_gb300.abi``);
expected values come only from ``oracle``, on the same seeded inputs.
"""

import numpy as np
import torch

import oracle
from oracle import attention, cache as ocache, layout, quant, rotation
from int2_rotated_kv_oscar_gb300 import abi, inputs
from int2_rotated_kv_oscar_gb300 import cache as kvcache

SM_SCALE = 1.0 / np.sqrt(128.0)
DECODE_TOL = 2e-3          # max-abs vs the oracle on the GPU's own dequantised cache
BF16_REL_TOL = 1e-2        # BF16-only contexts: max|diff| / max|ref| per head
EDGE_REL = 1e-6            # codes within 1e-6 * s of a decision edge are excluded (counted)


def oracle_rotation(cfg, layer, Hkv, flags=(True, True, True), n_cal=2048, n_keys=2048):
    """Per-layer (U_K, U_V fp32, tau_k, tau_v fp32) from the oracle's calibration."""
    Q = inputs.queries(cfg, layer, inputs.STREAM_Q_CAL, n_cal)
    Ks = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 0) for h in range(Hkv)]
    Vs = [inputs.kv_tokens(cfg, layer, h, inputs.STREAM_KV_CAL, n_keys, 1) for h in range(Hkv)]
    U_K, U_V, tk, tv = oracle.calibration.calibrate_layer(Q, Ks, Vs, SM_SCALE, 99.9, flags)
    return U_K.astype(np.float32), U_V.astype(np.float32), np.float32(tk), np.float32(tv)


def rotations_for_oracle(U_K, U_V, flags):
    use = (bool(flags & abi.OSCAR_ROT_U), bool(flags & abi.OSCAR_ROT_H), bool(flags & abi.OSCAR_ROT_P))
    return (rotation.composite_rotation(U_K.astype(np.float64), *use),
            rotation.composite_rotation(U_V.astype(np.float64), *use))


class Setup:
    """One context + one mixed cache on cuda:0 for a batch of requests."""

    def __init__(self, Hq, Hkv, lengths_max, batch, num_layers=1, cfg=1, flags=abi.OSCAR_ROT_ALL, seed=0,
                 extra_pages=3, shuffle=True, calibrate=True, paged_recent=False, tau_scale=1.0):
        self.Hq, self.Hkv, self.batch, self.cfg = Hq, Hkv, batch, cfg
        self.flags = flags
        conf = abi.oscar_config(num_layers=num_layers, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                                page_size=64, sink=64, recent=256, group=64, device=0)
        self.ctx = abi.oscar_create(conf)
        self.rot = []
        for layer in range(num_layers):
            if calibrate:
                U_K, U_V, tk, tv = oracle_rotation(cfg, layer, Hkv, flags=(True, True, True))
            else:
                r = np.random.default_rng([cfg, layer, 99])
                U_K = np.linalg.qr(r.standard_normal((128, 128)))[0].astype(np.float32)
                U_V = np.linalg.qr(r.standard_normal((128, 128)))[0].astype(np.float32)
                tk, tv = np.float32(30.0), np.float32(30.0)
            # tau_scale < 1: thresholds below the calibrated ones, so that most groups clip
            tk, tv = np.float32(tk * tau_scale), np.float32(tv * tau_scale)
            abi.oscar_load_rotation(self.ctx, layer, U_K, U_V, tk, tv, flags)
            R_K, R_V = rotations_for_oracle(U_K, U_V, flags)
            self.rot.append((R_K, R_V, float(tk), float(tv)))
        self.max_pages = (lengths_max + 63) // 64 + 1
        num_pages = batch * self.max_pages + extra_pages
        # paged recent window: five BF16 pages per request, logical page lp in page lp % 5
        # (the window touches at most five logical pages), shuffled over the pool
        self.paged_recent = paged_recent
        self.cache = kvcache.MixedCache(num_layers, Hkv, num_pages, batch, batch, batch, self.max_pages,
                                        recent_pages=5 * batch + 2 if paged_recent else None)
        perm = inputs.shuffled_pages(cfg, num_pages, seed) if shuffle else np.arange(num_pages, dtype=np.int32)
        table = perm[:batch * self.max_pages].reshape(batch, self.max_pages)
        self.cache.page_table.copy_(torch.from_numpy(table))
        if paged_recent:
            rperm = inputs.shuffled_pages(cfg + 1000, 5 * batch + 2, seed)
            lp = np.arange(self.max_pages)
            rt = np.stack([rperm[5 * b + lp % 5] for b in range(batch)]).astype(np.int32)
            self.cache.recent_table.copy_(torch.from_numpy(rt))
        self.ws_tensor, self.ws, self.ws_bytes = kvcache.workspace(self.ctx, batch, lengths_max + 1)

    def close(self):
        abi.oscar_destroy(self.ctx)

    def append(self, layer, k, v, pos, cu=None, max_tok=None, fresh=False, batch=None):
        """k, v: CPU or CUDA bf16 [n, Hkv, 128]; pos: list of ints; cu: list of ints or None."""
        k = k.cuda()
        v = v.cuda()
        pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
        cu_t = None if cu is None else torch.tensor(cu, dtype=torch.int32, device="cuda")
        args = kvcache.append_args(k, v, pos_t, cu_t, max_tok, fresh)
        abi.oscar_kv_append(self.ctx, layer, self.cache.view(layer, batch), args, torch.cuda.current_stream())
        torch.cuda.synchronize()

    def decode(self, layer, q, lens, batch=None, max_ctx=None):
        B = q.shape[0]
        q = q.cuda()
        out = torch.full((B, self.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
        args = kvcache.decode_args(q, out, ctx_len, max(lens) if max_ctx is None else max_ctx)
        abi.oscar_decode_attention(self.ctx, layer, self.cache.view(layer, batch), args, self.ws, self.ws_bytes,
                                   torch.cuda.current_stream())
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)

    def device_error(self):
        return abi.oscar_check_device_error(self.ctx, torch.cuda.current_stream())

    def readback(self, layer, b, L):
        """Per KV head: (sink_k, sink_v, ring_k, ring_v, blocks of logical pages 1..n) as numpy."""
        c = self.cache
        sp = int(c.sink_page[b])
        rs = int(c.ring_slot[b])
        (_, _), (h0, h1), _ = ocache.segments(L)
        n_pages = (h1 + 63) // 64 - 1 if h1 > h0 else 0
        table = c.page_table[b, 1:1 + n_pages].cpu().numpy() if n_pages else np.zeros(0, dtype=np.int64)
        pages = c.int2_pages[layer][torch.from_numpy(table.astype(np.int64)).cuda()].cpu().numpy() if n_pages else None
        out = []
        sk = inputs.bf16_to_f64(c.k_sink[layer][sp])
        sv = inputs.bf16_to_f64(c.v_sink[layer][sp])
        if c.paged_recent:
            # gather the window's rows from the BF16 pages into ring order (row (p - 64) % 256)
            (_, _), _, (r0, r1) = ocache.segments(L)
            kp = inputs.bf16_to_f64(c.k_ring[layer])
            vp = inputs.bf16_to_f64(c.v_ring[layer])
            rt = c.recent_table[b].cpu().numpy()
            rk = np.zeros((self.Hkv, 256, 128))
            rv = np.zeros((self.Hkv, 256, 128))
            for p in range(r0, r1):
                rk[:, (p - 64) % 256] = kp[rt[p // 64], :, p % 64]
                rv[:, (p - 64) % 256] = vp[rt[p // 64], :, p % 64]
        else:
            rk = inputs.bf16_to_f64(c.k_ring[layer][rs])
            rv = inputs.bf16_to_f64(c.v_ring[layer][rs])
        for h in range(self.Hkv):
            blocks = pages[:, h, :] if n_pages else np.zeros((0, 4608), dtype=np.uint8)
            out.append((sk[h], sv[h], rk[h], rv[h], blocks))
        return out

    def oracle_decode(self, layer, b, L, q_bf16):
        """Oracle output [Hq, 128] on the GPU's own stored cache of request b."""
        R_K, R_V, _, _ = self.rot[layer]
        Ks, Vs = [], []
        for (sk, sv, rk, rv, blocks) in self.readback(layer, b, L):
            K, V = ocache.reconstruct_from_storage(sk, sv, rk, rv, blocks, L, R_K, R_V)
            Ks.append(K)
            Vs.append(V)
        return attention.decode_gqa(inputs.bf16_to_f64(q_bf16), Ks, Vs, SM_SCALE)


def compare_history_codes(setup, layer, b, L, tok_k, tok_v, h):
    """Bit-exact code comparison of request b / KV head h against the oracle's
    direct definition.  tok_k, tok_v: fp64 [L, 128] token values.  Returns
    (n_compared, n_mismatch, n_edge_excluded, n_midpoint_groups)."""
    R_K, R_V, tk, tv = setup.rot[layer]
    want, rot = ocache.expected_history(tok_k, tok_v, L, R_K, R_V, tk, tv)
    if not want:
        return 0, 0, 0, 0
    sk, sv, rk, rv, blocks = setup.readback(layer, b, L)[h]
    kc, ks, vc, vs = layout.unpack_blocks(blocks)
    kc = kc.reshape(-1, 128)
    vc = vc.reshape(-1, 128)
    ks = ks.reshape(-1, 2)
    vs = vs.reshape(-1, 2)
    positions = sorted(want)
    n = len(positions)
    assert positions[0] == 64 and positions[-1] == 64 + n - 1
    n_cmp = n_bad = n_edge = n_mid = 0
    for which, codes_g, scales_g, R, tau in ((0, kc, ks, R_K, tk), (1, vc, vs, R_V, tv)):
        X = np.array([rot[p][which] for p in positions])
        exp_codes = np.array([want[p][2 * which] for p in positions])
        exp_scales = np.array([want[p][2 * which + 1] for p in positions])
        mid = quant.fp16_midpoint_mask(X, tau)
        edge = quant.near_edge_mask(X, exp_scales)
        gmask = np.repeat(mid, 64, axis=1)
        ok_scale = (scales_g[:n] == exp_scales) | mid
        assert ok_scale.all(), "scale mismatch outside fp16 midpoint groups: %d" % (~ok_scale).sum()
        cmp = ~(edge | gmask)
        bad = (codes_g[:n] != exp_codes) & cmp
        n_cmp += int(cmp.sum())
        n_bad += int(bad.sum())
        n_edge += int((edge & ~gmask).sum())
        n_mid += int(mid.sum())
    return n_cmp, n_bad, n_edge, n_mid


def compare_sampled_pages(setup, layer, b, lpages, tok_k, tok_v):
    """Bit-exact code comparison of whole history pages against the oracle's
    direct definition, for large contexts where comparing every position would
    be slow.  lpages: logical page indices (>= 1, all 64 rows in the history);
    tok_k, tok_v: fp64 [len(lpages) * 64, H_kv, 128] token values of those pages
    in order.  Returns (n_compared, n_mismatch, n_edge_excluded, n_midpoint_groups)."""
    R_K, R_V, tk, tv = setup.rot[layer]
    c = setup.cache
    phys = c.page_table[b, torch.tensor(lpages, dtype=torch.int64, device="cuda")].long()
    pages = c.int2_pages[layer][phys].cpu().numpy()          # [n, H_kv, 4608]
    n_cmp = n_bad = n_edge = n_mid = 0
    for h in range(setup.Hkv):
        kc, ks, vc, vs = layout.unpack_blocks(pages[:, h, :])
        got = ((kc.reshape(-1, 128), ks.reshape(-1, 2)), (vc.reshape(-1, 128), vs.reshape(-1, 2)))
        for which, (tok, R, tau) in enumerate(((tok_k, R_K, tk), (tok_v, R_V, tv))):
            X = rotation.rotate(np.asarray(tok)[:, h], R)
            codes, scales = quant.quantize_rows(X, tau)
            mid = quant.fp16_midpoint_mask(X, tau)
            edge = quant.near_edge_mask(X, scales)
            gmask = np.repeat(mid, 64, axis=1)
            gc, gs = got[which]
            assert ((gs == scales) | mid).all(), "scale mismatch outside fp16 midpoint groups"
            cmp = ~(edge | gmask)
            n_cmp += int(cmp.sum())
            n_bad += int(((gc != codes) & cmp).sum())
            n_edge += int((edge & ~gmask).sum())
            n_mid += int(mid.sum())
    return n_cmp, n_bad, n_edge, n_mid


def request_view(setup, b0, b1):
    """Swap the cache's per-request tables for rows [b0, b1) (for appending a
    subset of the batch); returns a function that restores them."""
    c = setup.cache
    saved = (c.page_table, c.sink_page, c.ring_slot, c.recent_table)
    c.page_table = saved[0][b0:b1].contiguous()
    c.sink_page = saved[1][b0:b1].contiguous()
    c.ring_slot = saved[2][b0:b1].contiguous()
    if saved[3] is not None:
        c.recent_table = saved[3][b0:b1].contiguous()

    def restore():
        c.page_table, c.sink_page, c.ring_slot, c.recent_table = saved
    return restore
