"""Device-side failure handling: a bounded wait that runs out, on purpose, on a real GPU.

The row-grouped tcgen05 kernel merges a group's split partials inside the kernel, its chunk CTAs
waiting for one another on a counter in the caller's workspace.  That wait has an iteration
limit; the library lets a test lower it (GQA_MERGE_SPIN=0: every such wait gives up at once,
with nothing hung -- the CTAs only stop waiting).  The call must then report GQA_ERR_TIMEOUT,
leave the workspace's arrival counters at zero, and the next call on the same workspace must be
exact against the oracle.
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL_F16, _env, assert_close, dev, oracle_ref
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def _grouped_case(seed):
    # 16 causal-style rows of one sequence, lengths 1800 .. 1995: one row group per KV head,
    # split into chunks whose whole grid fits one CTA per SM (the fused-merge launch)
    L = [1800 + 13 * r for r in range(16)]
    return W.make_f16_case(seed, 16, 32, 8, 128, L, cache_cap=2000, seq_of=[0] * 16, n_seq=1,
                           name="grouped_rows_timeout")


def _counter_bytes(n_tok, grid_y):
    return (n_tok * grid_y * 4 + 255) // 256 * 256


def test_fused_merge_wait_runs_out_then_next_call_is_exact():
    gd = _gd()
    case = _grouped_case(961)
    T, H, Hk, D = case.n_tok, case.n_heads, case.n_kv_heads, case.head_dim
    L = int(case.kv_len.max())
    plan = gd.plan(T, H, Hk, D, L, n_seq=1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.row_group > 1 and plan.merge == 1
    assert plan.grid_x * plan.grid_y * plan.grid_z <= sms  # the fused merge, not merge_kernel
    ws = gd.alloc_workspace(T, H, Hk, D, L, n_seq=1)
    q, k, v, kv, so = dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len), dev(case.seq_of)
    cnt = _counter_bytes(T, plan.grid_y)

    for attempt in range(2):  # twice: a second timed-out call on the same workspace
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        with _env(GQA_MERGE_SPIN=0):
            gd.attn_decode_f16(q, k, v, kv, scale=case.scale, seq_of=so, max_kv_len=L, ws=ws,
                               err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & gd.ERR_TIMEOUT, f"attempt {attempt}: no timeout flagged"
        # every chunk CTA counted in twice and the last one reset the counters
        assert int(ws[:cnt].count_nonzero().item()) == 0, "arrival counters left non-zero"

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gd.attn_decode_f16(q, k, v, kv, scale=case.scale, seq_of=so, max_kv_len=L, ws=ws,
                             err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(ws[:cnt].count_nonzero().item()) == 0
    assert_close(got.cpu().numpy(), oracle_ref(case), TOL_F16, "after timeouts")


def test_merge_timeout_leaves_other_rows_alone():
    """The limit only touches the fused merge: a per-row split call under GQA_MERGE_SPIN=0 (its
    merge takes tickets and never waits) is exact and flags nothing."""
    gd = _gd()
    case = W.make_f16_case(962, 3, 16, 4, 128, [5000, 77, 2600], cache_cap=5000, scale=0.09)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _env(GQA_MERGE_SPIN=0):
        got = gd.attn_decode_f16(dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len),
                                 scale=case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got.cpu().numpy(), oracle_ref(case), TOL_F16, "per-row split")
    assert np.isfinite(got.cpu().numpy()).all()


def test_tq_rows_fused_merge_wait_runs_out_then_next_call_is_exact():
    """The TurboQuant row kernel's fused merge (16 causal rows of one sequence on a compressed
    cache) under GQA_MERGE_SPIN=0: the call flags GQA_ERR_TIMEOUT and leaves the arrival
    counters at zero, and the next call on the same workspace matches the oracle."""
    import oracle
    gd = _gd()
    L = [1800 + 13 * r for r in range(16)]
    c = W.make_tq_case(964, 16, 32, 8, 128, L, cache_cap=2000, seq_of=[0] * 16, n_seq=1)
    T, H, Hk, D, Lm = 16, 32, 8, 128, max(L)
    plan = gd.plan(T, H, Hk, D, Lm, -1, gd.KIND_TQ, n_seq=1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan.row_group > 1 and plan.merge == 1
    assert plan.grid_x * plan.grid_y * plan.grid_z <= sms  # the fused merge, not merge_kernel
    ws = gd.alloc_workspace(T, H, Hk, D, Lm, -1, gd.KIND_TQ, n_seq=1)
    cnt = _counter_bytes(T, plan.grid_y)
    i32 = lambda a: dev(np.ascontiguousarray(a).view(np.int32))  # noqa: E731
    args = (dev(c.q_rot), dev(c.q_jl), i32(c.k_polar), i32(c.k_jl), i32(c.k_norms),
            i32(c.v_polar), i32(c.v_norms), c.centroids, dev(c.signs), c.qjl_scale,
            dev(c.kv_len))

    def call(err):
        return gd.attn_decode_tq(*args, scale=c.scale, seq_of=dev(c.seq_of), max_kv_len=Lm,
                                 ws=ws, err=err)

    for attempt in range(2):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        with _env(GQA_MERGE_SPIN=0):
            call(err)
        torch.cuda.synchronize()
        assert int(err.item()) & gd.ERR_TIMEOUT, f"attempt {attempt}: no timeout flagged"
        assert int(ws[:cnt].count_nonzero().item()) == 0, "arrival counters left non-zero"
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = call(err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(ws[:cnt].count_nonzero().item()) == 0
    ref = oracle.decode_tq(c.q_rot, c.q_jl, c.k_polar, c.k_jl, c.k_norms, c.v_polar, c.v_norms,
                           c.centroids, c.signs, c.qjl_scale, c.scale, c.kv_len, c.seq_of)
    g = got.cpu().numpy().astype(np.float64)
    assert (np.abs(g - ref) / np.maximum(1.0, np.abs(ref))).max() <= 1e-4  # the TurboQuant bound
