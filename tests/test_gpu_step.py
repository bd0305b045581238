"""GPU: the fused decode step (oscar_decode_step) against its two parts.

oscar_decode_step appends one token per request and decodes in one launch;
its results must be bit-identical to oscar_kv_append followed by
oscar_decode_attention on the same inputs (the same arithmetic runs in both),
for every cache byte and every output value, while requests cross the sink
boundary (position 64), the first eviction (position 320) and steady-state
eviction.  The step's outputs are also checked against the oracle on the
GPU's own stored cache.
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


def _prefill(s, toks, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    s.append(0, torch.cat([t[0][:L] for t, L in zip(toks, lens)]), torch.cat([t[1][:L] for t, L in zip(toks, lens)]),
             [0] * len(lens), cu, max(lens))


def _cache_bytes(s):
    c = s.cache
    return [t[0].cpu().clone() for t in (c.int2_pages, c.k_sink, c.v_sink, c.k_ring, c.v_ring)]


@pytest.mark.parametrize("Hq,Hkv,flags", [(32, 8, abi.OSCAR_ROT_ALL), (16, 2, abi.OSCAR_ROT_ALL),
                                           (32, 8, abi.OSCAR_ROT_H | abi.OSCAR_ROT_P),  # butterfly, bit reversal
                                           (16, 2, abi.OSCAR_ROT_H), (32, 8, abi.OSCAR_ROT_P)])
def test_step_equals_append_then_decode(Hq, Hkv, flags):
    """Layers without U rotate the one-token writes, q and the output with the
    in-register butterfly and the bit-reversal index map instead of the dense
    product: the evicted rows' codes must still match the oracle bit for bit."""
    cfg = 11
    lens0 = [60, 318, 700]
    n_steps = 6
    B = len(lens0)
    toks = [inputs.kv_tokens_bf16(cfg, 0, Hkv, inputs.STREAM_KV, L + n_steps, b) for b, L in enumerate(lens0)]
    fused = harness.Setup(Hq, Hkv, max(lens0) + n_steps, B, cfg=cfg, calibrate=False, flags=flags)
    split = harness.Setup(Hq, Hkv, max(lens0) + n_steps, B, cfg=cfg, calibrate=False, flags=flags)
    try:
        for s in (fused, split):
            _prefill(s, toks, lens0)
            assert s.device_error() == 0
        for step in range(n_steps):
            pos = [L + step for L in lens0]
            lens = [p + 1 for p in pos]
            k = torch.stack([t[0][p] for t, p in zip(toks, pos)]).cuda()
            v = torch.stack([t[1][p] for t, p in zip(toks, pos)]).cuda()
            q = inputs.decode_queries_bf16(cfg, 0, B, Hq, step=step).cuda()
            pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
            len_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
            out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            ap = kvcache.append_args(k, v, pos_t)
            dp = kvcache.decode_args(q, out, len_t, max(lens))
            abi.oscar_decode_step(fused.ctx, 0, fused.cache.view(0), ap, dp, fused.ws, fused.ws_bytes,
                                  torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert fused.device_error() == 0
            split.append(0, k, v, pos)
            want = split.decode(0, q, lens)
            assert split.device_error() == 0
            got = out.cpu().numpy().astype(np.float64)
            assert np.isfinite(got).all()
            assert np.array_equal(got, want), "step %d: max diff %.3e" % (step, np.abs(got - want).max())
            for a, b in zip(_cache_bytes(fused), _cache_bytes(split)):
                assert torch.equal(a, b)
        errs = []
        for b in range(B):
            ref = fused.oracle_decode(0, b, lens[b], q[b].cpu())
            errs.append(np.abs(got[b] - ref).max())
        print("Hq %d Hkv %d flags %d: max-abs vs oracle after %d steps %s"
              % (Hq, Hkv, flags, n_steps, ["%.2e" % e for e in errs]))
        assert max(errs) <= harness.DECODE_TOL
        # the history rows (bulk prefill and the steps' evictions) against the oracle's definition
        n_cmp = n_bad = 0
        for b in range(B):
            tk = inputs.bf16_to_f64(toks[b][0][:lens[b]])
            tv = inputs.bf16_to_f64(toks[b][1][:lens[b]])
            for h in range(Hkv):
                c, bad, _, _ = harness.compare_history_codes(fused, 0, b, lens[b], tk[:, h], tv[:, h], h)
                n_cmp += c
                n_bad += bad
        print("flags %d: %d history codes compared, %d mismatches" % (flags, n_cmp, n_bad))
        assert n_bad == 0 and n_cmp > 0
    finally:
        fused.close()
        split.close()


def test_step_rejects_multi_token_appends():
    s = harness.Setup(32, 8, 100, 2, cfg=9, calibrate=False)
    try:
        k = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
        q = torch.zeros((2, 32, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((2, 32, 128), dtype=torch.float32, device="cuda")
        pos = torch.tensor([3, 3], dtype=torch.int32, device="cuda")
        cu = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
        dp = kvcache.decode_args(q, out, pos + 1, 4)
        # a cu_seqlens array, or fewer tokens than requests
        for ap in (kvcache.append_args(k, k, pos, cu, 1), kvcache.append_args(k[:1], k[:1], pos)):
            with pytest.raises(abi.OscarError) as e:
                abi.oscar_decode_step(s.ctx, 0, s.cache.view(0), ap, dp, s.ws, s.ws_bytes, None)
            assert e.value.status == 1  # OSCAR_ERR_INVALID_ARG
        assert s.device_error() == 0
    finally:
        s.close()
