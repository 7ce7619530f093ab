"""The allocation-free f16 entry point (attn_decode_f16_noalloc) against attn_decode_f16.

Some callers cannot allocate device memory -- a host that owns every byte of the GPU in a fixed
arena, or a foreign runtime that reaches this library only through its C ABI with nothing but
input and output buffers.  attn_decode_f16_noalloc serves them by keeping the split partials in
a static device array inside the library.  This file is collected last on purpose, so that a
run stopping at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL_F16, assert_close, dev, f16_kernel, forced_chunk
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def test_noalloc_matches_workspace_call_twice_in_a_row():
    gd = _gd()
    # split into many KV chunks, so the partials really live in the static scratch
    case = W.make_f16_case(901, 3, 16, 4, 128, [6000, 37, 4100], cache_cap=6000, scale=0.09)
    plan = gd.plan(3, 16, 4, 128, 6000)
    assert plan.merge == 1 and 0 < plan.ws_bytes <= gd.NOALLOC_SCRATCH_BYTES
    k, v, kv = dev(case.k), dev(case.v), dev(case.kv_len)
    for call in range(2):  # the second call must not see the first one's leftovers
        q = dev(case.q * (1.0 + call))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = gd.attn_decode_f16(q, k, v, kv, scale=case.scale)
        got = gd.attn_decode_f16_noalloc(q, k, v, kv, scale=case.scale, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), TOL_F16, f"call {call}")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    gd = _gd()
    T, H, Hk, D, cap = 4, 32, 8, 128, 1 << 20
    q = torch.zeros((T, H, D), dtype=torch.float32, device="cuda")
    kc = torch.zeros((1, 16, Hk, D), dtype=torch.float16, device="cuda")
    # the chunked split with 64-position chunks over 2^20 positions: ~1 GB of partials
    with f16_kernel("chunked"), forced_chunk(64):
        assert gd.workspace_bytes(T, H, Hk, D, cap) > gd.NOALLOC_SCRATCH_BYTES
        # refused on the size alone.  kv_len is passed as NULL, so that even if the size check
        # let the call through, attn_decode_f16 would stop at its own argument check and
        # nothing would launch over the deliberately tiny cache.
        st = gd.LIB.attn_decode_f16_noalloc(gd._ptr(q), gd._ptr(kc), gd._ptr(kc), gd._ptr(q),
                                            None, None, T, T, H, Hk, D, cap, cap, 0.1, None,
                                            gd._stream(None))
    assert st == gd.GQA_EWORKSPACE
    assert b"static scratch" in gd.LIB.gqa_last_error()
