"""The allocation-free f16 entry point (attn_decode_f16_noalloc).

Some callers cannot allocate device memory -- a host that owns every byte of the GPU in a fixed
arena, or a foreign runtime that reaches this library only through its C ABI with nothing but
input and output buffers.  attn_decode_f16_noalloc serves them by keeping the split partials
and the merge's arrival counters in a static device array inside the library.  Every call on a
device shares that array, so these tests chain calls of different kinds on it and check each
against the fp64 oracle and against attn_decode_f16 with a workspace of its own.  This file is
collected last on purpose, so that a run stopping at the first failure has already run every
other test.
"""

import pytest
import torch

from gpu_util import TOL_F16, _env, assert_close, dev, f16_kernel, forced_chunk, oracle_ref
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def _check_both(gd, case, seq_of=None, max_kv_len=None, what=""):
    """The no-alloc call against the oracle and against the workspace call; err must stay 0."""
    q, k, v, kv = dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gd.attn_decode_f16_noalloc(q, k, v, kv, scale=case.scale, seq_of=seq_of,
                                     max_kv_len=max_kv_len, err=err)
    ref = gd.attn_decode_f16(q, k, v, kv, scale=case.scale, seq_of=seq_of,
                             max_kv_len=max_kv_len)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    got = got.cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, f"{what}: against the oracle")
    assert_close(got, ref.cpu().numpy(), TOL_F16, f"{what}: against attn_decode_f16")


def test_noalloc_matches_oracle_twice_in_a_row():
    gd = _gd()
    # split into many KV chunks, so the partials really live in the static scratch
    case = W.make_f16_case(901, 3, 16, 4, 128, [6000, 37, 4100], cache_cap=6000, scale=0.09)
    plan = gd.plan(3, 16, 4, 128, 6000)
    assert plan.merge == 1 and 0 < plan.ws_bytes <= gd.NOALLOC_SCRATCH_BYTES
    for call in range(2):  # the second call must not see the first one's leftovers
        case.q = case.q * (1.0 + call)
        _check_both(gd, case, what=f"call {call}")


def test_noalloc_row_grouped_after_per_row():
    """Rows sharing a sequence (the tcgen05 row kernel, its merge counters at another index of
    the same static array) right after a per-row split call, then a per-row call again."""
    gd = _gd()
    per_row = W.make_f16_case(903, 3, 16, 4, 128, [6000, 37, 4100], cache_cap=6000, scale=0.09)
    L = [2500 + 31 * r for r in range(16)]
    grouped = W.make_f16_case(904, 16, 32, 8, 128, L, cache_cap=3000, seq_of=[0] * 16, n_seq=1,
                              name="grouped")
    plan = gd.plan(16, 32, 8, 128, 3000, n_seq=1)
    assert plan.row_group > 1 and plan.merge == 1
    assert plan.ws_bytes <= gd.NOALLOC_SCRATCH_BYTES
    _check_both(gd, per_row, what="per-row before")
    _check_both(gd, grouped, seq_of=dev(grouped.seq_of), what="grouped rows")
    _check_both(gd, grouped, seq_of=dev(grouped.seq_of), what="grouped rows again")
    _check_both(gd, per_row, what="per-row after")


def test_noalloc_recovers_after_a_merge_wait_runs_out():
    """A grouped call whose fused-merge waits all give up (GQA_MERGE_SPIN=0) flags the error and
    leaves the shared counters clean: the next call on the static array is exact."""
    gd = _gd()
    L = [1800 + 13 * r for r in range(16)]
    case = W.make_f16_case(905, 16, 32, 8, 128, L, cache_cap=2000, seq_of=[0] * 16, n_seq=1,
                           name="grouped")
    q, k, v, kv, so = dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len), dev(case.seq_of)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _env(GQA_MERGE_SPIN=0):
        gd.attn_decode_f16_noalloc(q, k, v, kv, scale=case.scale, seq_of=so, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & gd.ERR_TIMEOUT
    _check_both(gd, case, seq_of=so, what="after the timed-out call")


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
