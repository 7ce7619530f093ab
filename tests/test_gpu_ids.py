"""Selected-cell id lists that are not sorted, that repeat cells, or that are permuted.

The pages emit ids in ascending order (qsa2.metal, qsa_topk2), but the attention itself is a
function of the multiset of visited cells: the softmax and the weighted sum do not depend on
the order, and a cell listed twice counts twice (its exp(x) enters the sum twice and its V row
the output twice).  The oracle states exactly that; these tests hold the GPU path to it.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_Q8, assert_close, dev, forced_chunk, run_case
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _ref(case):
    return oracle.decode_q8(case.q, case.kq, case.vq, case.ksc, case.vsc, case.kv_len,
                            case.scale, seq_of=case.seq_of, ids=case.ids, budget=case.budget)


def _case(seed, D=256, G=12, Hk=2, L=(3000, 900, 5000), budget=640):
    return W.make_q8_case(seed, len(L), G * Hk, Hk, D, list(L), budget=budget, scale=1 / 16)


@pytest.mark.parametrize("chunk", [None, 128])
def test_unsorted_ids(chunk):
    case = _case(1301)
    rng = np.random.default_rng(1302)
    for t in range(case.n_tok):
        n = min(int(case.kv_len[t]), case.budget)
        case.ids[t, :n] = rng.permutation(case.ids[t, :n])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with forced_chunk(chunk):
        got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert_close(got, _ref(case), TOL_Q8, "unsorted ids")


@pytest.mark.parametrize("chunk", [None, 128])
def test_duplicated_ids_count_once_per_occurrence(chunk):
    case = _case(1303)
    rng = np.random.default_rng(1304)
    for t in range(case.n_tok):
        n = min(int(case.kv_len[t]), case.budget)
        dup = rng.choice(n, size=n // 3, replace=False)     # a third of the entries ...
        case.ids[t, dup] = case.ids[t, rng.integers(0, n, size=len(dup))]  # ... repeat others
    assert any(len(set(r[r >= 0].tolist())) < (r >= 0).sum() for r in case.ids)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with forced_chunk(chunk):
        got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert_close(got, _ref(case), TOL_Q8, "duplicated ids")


def test_permuting_ids_leaves_the_output_unchanged():
    """The same cells in another order: equal within the int8 tolerance (only the order of the
    fp32 sums changes), on the split path and on the single-chunk path."""
    case = _case(1305, L=(4000, 700, 2500))
    base = run_case(case).cpu().numpy()
    rng = np.random.default_rng(1306)
    for trial in range(3):
        perm = case.ids.copy()
        for t in range(case.n_tok):
            n = min(int(case.kv_len[t]), case.budget)
            perm[t, :n] = rng.permutation(perm[t, :n])
        got = run_case(case, ids=dev(perm)).cpu().numpy()
        assert_close(got, base, TOL_Q8, f"permutation {trial}")
    with forced_chunk(1 << 20):  # one chunk per row
        one = run_case(case).cpu().numpy()
    assert_close(one, base, TOL_Q8, "one chunk")
