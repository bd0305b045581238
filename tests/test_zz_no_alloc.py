"""The allocation-free decode entry point, checked against the workspace one.

oscar_decode_attention_noalloc serves callers that cannot allocate device
memory (a plugin whose host engine owns every device allocation, a serving
loop that must not call cudaMalloc once it runs): it takes its scratch from a
fixed array inside the library instead of a caller workspace.  Its results
must match oscar_decode_attention on the same inputs, call after call (the
array keeps the previous call's contents), and a call that needs more scratch
than the array holds must be refused before anything is launched.

This file is collected last so that a run stopping at its first failure has
run every other test before it.
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


def _noalloc_decode(s, q, lens):
    out = torch.full((q.shape[0], s.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    args = kvcache.decode_args(q.cuda(), out, ctx_len, max(lens))
    abi.oscar_decode_attention_noalloc(s.ctx, 0, s.cache.view(0), args, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    cfg = 9
    lens = [2500, 700]
    s = harness.Setup(32, 8, max(lens) + 1, len(lens), cfg=cfg, calibrate=False)
    try:
        toks = [inputs.kv_tokens_bf16(cfg, 0, 8, inputs.STREAM_KV, L, b) for b, L in enumerate(lens)]
        cu = [0, lens[0], lens[0] + lens[1]]
        s.append(0, torch.cat([t[0] for t in toks]), torch.cat([t[1] for t in toks]), [0, 0], cu, max(lens))
        assert s.device_error() == 0
        for call in range(2):
            # a different query on each call: the second call starts from the
            # scratch contents the first one left behind
            q = inputs.decode_queries_bf16(cfg, 0, len(lens), 32, step=call)
            want = s.decode(0, q, lens)
            got = _noalloc_decode(s, q, lens)
            assert s.device_error() == 0
            err = np.abs(got - want).max()
            print("call %d: max-abs difference to the workspace entry point %.3e" % (call, err))
            assert np.isfinite(got).all()
            assert err <= harness.DECODE_TOL
    finally:
        s.close()


def test_noalloc_decode_refuses_calls_larger_than_its_scratch():
    # 300 requests x 8 KV heads: the per-(request, KV head) q fragments alone
    # (8 KB each) need more workspace than the library's scratch holds
    B = 300
    s = harness.Setup(32, 8, 600, B, cfg=9, calibrate=False)
    try:
        need = abi.oscar_decode_workspace_bytes(s.ctx, B, 600)
        assert need > abi.NOALLOC_SCRATCH_BYTES
        q = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((B, 32, 128), dtype=torch.float32, device="cuda")
        lens = torch.full((B,), 10, dtype=torch.int32, device="cuda")
        args = kvcache.decode_args(q, out, lens, 600)
        with pytest.raises(abi.OscarError) as e:
            abi.oscar_decode_attention_noalloc(s.ctx, 0, s.cache.view(0), args, None)
        assert e.value.status == 6  # OSCAR_ERR_WORKSPACE
        assert s.device_error() == 0
    finally:
        s.close()


def test_noalloc_decode_at_the_edge_of_its_scratch():
    # the largest batch whose workspace fits the array (to within one more
    # request's share of its end): every block writes its record, so a plan
    # that overran the array would write past its end; the outputs must match
    # the workspace entry point and no device error may be raised
    cfg, max_ctx = 9, 2000
    conf = abi.oscar_config(num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64, sink=64,
                            recent=256, group=64, device=0)
    probe = abi.oscar_create(conf)
    try:
        B = 1
        while abi.oscar_decode_workspace_bytes(probe, B + 1, max_ctx) <= abi.NOALLOC_SCRATCH_BYTES:
            B += 1
        need = abi.oscar_decode_workspace_bytes(probe, B, max_ctx)
        step = abi.oscar_decode_workspace_bytes(probe, B + 1, max_ctx) - need
    finally:
        abi.oscar_destroy(probe)
    gap = abi.NOALLOC_SCRATCH_BYTES - need
    print("edge case: %d requests at max_ctx_len %d need %d of %d bytes (gap %d, one more request %d)"
          % (B, max_ctx, need, abi.NOALLOC_SCRATCH_BYTES, gap, step))
    assert 0 <= gap < step
    lens = [64 + (97 * b) % 1900 for b in range(B)]
    s = harness.Setup(32, 8, max_ctx, B, cfg=cfg, calibrate=False)
    try:
        k, v = inputs.kv_tokens_bf16(cfg, 0, 8, inputs.STREAM_KV, max(lens))
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        s.append(0, torch.cat([k[:L] for L in lens]), torch.cat([v[:L] for L in lens]), [0] * B, cu, max(lens))
        assert s.device_error() == 0
        ws_t, ws, ws_bytes = kvcache.workspace(s.ctx, B, max_ctx)
        for call in range(2):
            q = inputs.decode_queries_bf16(cfg, 0, B, 32, step=3 + call).cuda()
            ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
            want_t = torch.full((B, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
            abi.oscar_decode_attention(s.ctx, 0, s.cache.view(0), kvcache.decode_args(q, want_t, ctx_len, max_ctx),
                                       ws, ws_bytes, torch.cuda.current_stream())
            got_t = torch.full((B, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
            abi.oscar_decode_attention_noalloc(s.ctx, 0, s.cache.view(0),
                                               kvcache.decode_args(q, got_t, ctx_len, max_ctx),
                                               torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert s.device_error() == 0
            got, want = got_t.cpu().numpy(), want_t.cpu().numpy()
            assert np.isfinite(got).all()
            err = float(np.abs(got - want).max())
            print("edge case call %d: max-abs difference to the workspace entry point %.3e" % (call, err))
            assert err <= harness.DECODE_TOL
    finally:
        s.close()


@pytest.mark.parametrize("Hq", [32, 64])
def test_noalloc_capacity_at_long_contexts(Hq):
    # the largest batch of 100K- and 128K-token requests the scratch array serves (printed for the docs)
    conf = abi.oscar_config(num_layers=1, num_q_heads=Hq, num_kv_heads=8, head_dim=128, page_size=64, sink=64,
                            recent=256, group=64, device=0)
    ctx = abi.oscar_create(conf)
    try:
        caps = []
        for L in (100_000, 131_072):
            b = 1
            while abi.oscar_decode_workspace_bytes(ctx, b + 1, L) <= abi.NOALLOC_SCRATCH_BYTES:
                b += 1
            caps.append(b)
        print("no-alloc capacity at %d query / 8 KV heads: %d requests of 100K tokens, %d of 128K" % (Hq, *caps))
        assert caps[0] >= 1 and caps[1] >= 1
    finally:
        abi.oscar_destroy(ctx)
