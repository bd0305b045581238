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
    # 4 requests x 8 KV heads at an 8M-token maximum: 256 work items each, one
    # partial record apiece, more workspace than the library's scratch
    s = harness.Setup(32, 8, 600, 4, cfg=9, calibrate=False)
    try:
        need = abi.oscar_decode_workspace_bytes(s.ctx, 4, 8_000_000)
        assert need > abi.NOALLOC_SCRATCH_BYTES
        q = torch.zeros((4, 32, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.zeros((4, 32, 128), dtype=torch.float32, device="cuda")
        lens = torch.tensor([10, 10, 10, 10], dtype=torch.int32, device="cuda")
        args = kvcache.decode_args(q, out, lens, 8_000_000)
        with pytest.raises(abi.OscarError) as e:
            abi.oscar_decode_attention_noalloc(s.ctx, 0, s.cache.view(0), args, None)
        assert e.value.status == 6  # OSCAR_ERR_WORKSPACE
        assert s.device_error() == 0
    finally:
        s.close()
