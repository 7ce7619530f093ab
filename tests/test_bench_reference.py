"""bench.py's CPU legs on every cache kind: the reference arm's per-(row, KV head) oracle call
matches the whole-problem oracle, and the reference arm prints its JSON line."""

import contextlib
import io
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from gqa_decode_attention_03_gb300 import workloads as W  # noqa: E402


def _cases():
    return [
        W.make_f16_case(71, 2, 8, 2, 64, [40, 9], cache_cap=40, scale=0.125),
        W.make_q8_case(72, 2, 8, 2, 64, [30, 12], budget=16, cache_cap=30, scale=0.1),
        W.make_q8_case(73, 1, 4, 1, 64, [20], cache_cap=20, scale=0.1, scale_group=32),
        W.make_tq_case(74, 2, 8, 2, 64, [25, 7], cache_cap=28),
    ]


def _whole(case):
    if case.kind == "f16":
        return oracle.decode_f16(case.q, case.k, case.v, case.kv_len, case.scale,
                                 seq_of=case.seq_of)
    if case.kind == "q8":
        return oracle.decode_q8(case.q, case.kq, case.vq, case.ksc, case.vsc, case.kv_len,
                                case.scale, seq_of=case.seq_of, ids=case.ids, budget=case.budget)
    return oracle.decode_tq(case.q_rot, case.q_jl, case.k_polar, case.k_jl, case.k_norms,
                            case.v_polar, case.v_norms, case.centroids, case.signs,
                            case.qjl_scale, case.scale, case.kv_len, case.seq_of)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c.kind}-{c.name}")
def test_oracle_pair_matches_the_whole_problem(case):
    ref = _whole(case)
    G = case.n_heads // case.n_kv_heads
    for t in range(case.n_tok):
        for g in range(case.n_kv_heads):
            got = bench._oracle_pair(case, t, g)
            np.testing.assert_allclose(got[0], ref[t, g * G:(g + 1) * G], rtol=1e-12, atol=1e-14)
        assert bench._pair_bytes(case, t) > 0 or case.kv_len[t] == 0


@pytest.mark.parametrize("workload", ["tiny", "q8_sel"])
def test_reference_arm_prints_its_line(workload):
    class A:
        steps, warmup = 2, 3
    A.workload = workload
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(A)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"]


def test_cpu_baseline_uses_every_host_core():
    b = bench.cpu_baseline("tiny", budget_s=2.0)
    assert b["kind"] == "oracle" and b["value"] > 0
    assert b["cores"] == bench._cores() and b["host_cores"] == os.cpu_count()
    assert b["single_core"]["cores"] == 1 and b["single_core"]["value"] > 0
