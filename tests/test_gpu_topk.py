"""GPU parity of the block top-k selection (attn_select_topk) against the oracle: bit-exact ids,
and the selected int8 path fed by it."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_Q8, assert_close, dev, oracle_ref, run_case
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def _oracle_ids(scores, kv_len, budget):
    ids = np.full((len(kv_len), budget), -1, dtype=np.int64)
    for t, n in enumerate(kv_len):
        sel = oracle.select_topk_cells(scores[t], int(n), budget)
        ids[t, :len(sel)] = sel
    return ids


@pytest.mark.parametrize("levels", [None, 3, 17])
@pytest.mark.parametrize("budget", [1, 5, 64, 1024])
def test_topk_bit_exact(levels, budget):
    # lengths: multiples of 4 and not, shorter and longer than the budget, a row of blocks well
    # past the 1024 threads of a CTA, an empty row
    kv_len = np.array([8192, 8190, 4097, 3, budget, budget + 1, 0, 17000, 64, 65], np.int32)
    stride = 17000 // 4 + 1
    scores = W.make_block_scores(700 + budget, len(kv_len), stride, levels)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gd().attn_select_topk(dev(scores), dev(kv_len), budget, max_kv_len=17000,
                                 err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert np.array_equal(got, _oracle_ids(scores, kv_len, budget))


@pytest.mark.parametrize("dist", ["spread", "clustered", "clustered_ties"])
@pytest.mark.parametrize("budget", [7, 300, 4000])
def test_topk_few_candidates_after_any_step(dist, budget):
    """Score sets whose threshold bin holds only a few blocks after the first 8-bit step (scores
    spread over many binades), or only after the third (scores sharing their top 16 key bits),
    with equal scores among those blocks: the selection ranks them directly, bit-exact."""
    rng = np.random.default_rng(1200 + budget + len(dist))
    nb = 2049
    if dist == "spread":
        s = np.ldexp(rng.choice([-1.0, 1.0], nb) * (1.0 + rng.random(nb)), rng.integers(-60, 60, nb))
    elif dist == "clustered":
        s = 1.0 + rng.random(nb) * 2.0 ** -9
    else:
        s = 1.0 + rng.integers(0, 600, nb) * 2.0 ** -20
    scores = s.astype(np.float32).reshape(1, nb)
    kv_len = np.array([4 * nb - 3], np.int32)  # the last block holds one cell
    got = _gd().attn_select_topk(dev(scores), dev(kv_len), budget,
                                 max_kv_len=int(kv_len[0])).cpu().numpy()
    assert np.array_equal(got, _oracle_ids(scores, kv_len, budget))


def test_topk_signed_zero_and_infinities():
    s = np.array([[0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 0.0, -0.0]], np.float32)
    kv_len = np.array([30], np.int32)
    got = _gd().attn_select_topk(dev(s), dev(kv_len), 9, max_kv_len=30).cpu().numpy()
    assert np.array_equal(got, _oracle_ids(s, kv_len, 9))


def test_topk_feeds_the_selected_int8_path():
    """Block scores -> ids (GPU) -> int8 selected decode (GPU), against the oracle on the same
    chain: 48 heads over 4 KV heads, D=256, context 8192, budget 1024."""
    case = W.q8_selected()
    stride = 8192 // 4 + 1
    scores = W.make_block_scores(710, 1, stride)
    ids = _gd().attn_select_topk(dev(scores), dev(case.kv_len), 1024, max_kv_len=8192)
    case.ids = _oracle_ids(scores, case.kv_len, 1024).astype(np.int32)
    assert np.array_equal(ids.cpu().numpy(), case.ids)
    got = run_case(case, ids=ids).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, "topk -> q8_sel")


@pytest.mark.parametrize("max_kv", [49147, 184316, 184320, 200003, 260001])
def test_topk_staged_and_unstaged_rows(max_kv):
    """Rows whose block keys fit the shared-memory staging (max_kv_len / 4 + 1 <= 46080 blocks,
    past the 48 KB that needs no opt-in) and rows past it, which read the keys from global
    memory at every step of the threshold search."""
    kv_len = np.array([max_kv, max_kv - 3, 20000, 700, 0], np.int32)
    stride = max_kv // 4 + 1
    scores = W.make_block_scores(720 + max_kv % 97, len(kv_len), stride, 29)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gd().attn_select_topk(dev(scores), dev(kv_len), 2048, max_kv_len=max_kv,
                                 err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert np.array_equal(got, _oracle_ids(scores, kv_len, 2048))


def test_topk_nan_scores_rank_at_the_ends():
    """NaN scores rank through the same bit-pattern map: a positive NaN above +inf, a negative
    one below -inf."""
    s = np.array([[np.nan, 1.0, -np.nan, np.inf, 0.5, -np.inf, 2.0, 0.0]], np.float32)
    s[0, 2] = -np.float32(np.nan)
    kv_len = np.array([31, 31], np.int32)
    s = np.concatenate([s, s[:, ::-1].copy()])
    for budget in (1, 4, 5, 13, 30):
        got = _gd().attn_select_topk(dev(s), dev(kv_len), budget, max_kv_len=31).cpu().numpy()
        assert np.array_equal(got, _oracle_ids(s, kv_len, budget)), budget


def test_topk_kv_len_out_of_range_is_clamped_and_flagged():
    kv_len = np.array([-5, 900, 40], np.int32)
    scores = W.make_block_scores(731, 3, 200 // 4 + 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gd().attn_select_topk(dev(scores), dev(kv_len), 16, max_kv_len=200,
                                 err=err).cpu().numpy()
    assert int(err.item()) & _gd().ERR_KVLEN_RANGE
    assert np.array_equal(got, _oracle_ids(scores, np.array([0, 200, 40]), 16))
