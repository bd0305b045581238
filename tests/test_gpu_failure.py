"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every asynchronous wait of the kernels (a bulk or tensor copy landing, a
barrier between warp roles) is bounded, by a number of polls or by time on the
global timer, then sets OSCAR_DEVERR_TIMEOUT in the context's device error
word, skips the rest of its work and returns.  `oscar_selftest_bounded_wait`
runs both kinds on barriers that nothing completes and sets the bit only when
both gave up; the host reads it, and the same context then appends and decodes
as before, against the oracle.
"""

import time

import numpy as np
import pytest
import torch

from int2_rotated_kv_oscar_gb300 import abi, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import harness  # noqa: E402


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    cfg, L = 1, 700
    s = harness.Setup(8, 2, L, 1, cfg=cfg)
    try:
        assert s.device_error() == 0
        for polls in (1 << 10, 1 << 14):
            t0 = time.perf_counter()
            abi.oscar_selftest_bounded_wait(s.ctx, polls, torch.cuda.current_stream())
            bits = s.device_error()
            dt = time.perf_counter() - t0
            print("bounded waits of %d polls / %d us gave up after %.2f ms (host-timed)" % (polls, 4 * polls, 1e3 * dt))
            assert bits == abi.OSCAR_DEVERR_TIMEOUT
        assert s.device_error() == 0  # read and cleared
        with pytest.raises(abi.OscarError):
            abi.oscar_selftest_bounded_wait(s.ctx, 0, torch.cuda.current_stream())
        # the context is unharmed: a prefill append and a decode step, against the oracle
        k, v = inputs.kv_tokens_bf16(cfg, 0, 2, inputs.STREAM_KV, L)
        s.append(0, k, v, [0], [0, L], L)
        assert s.device_error() == 0
        q = inputs.decode_queries_bf16(cfg, 0, 1, 8)
        out = s.decode(0, q, [L])
        assert s.device_error() == 0
        ref = s.oracle_decode(0, 0, L, q[0])
        err = np.abs(out[0] - ref).max()
        print("decode after the timeouts: max-abs %.3e" % err)
        assert err <= harness.DECODE_TOL
    finally:
        s.close()
