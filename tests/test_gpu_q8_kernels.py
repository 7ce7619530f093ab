"""The two int8 decode kernels against the oracle: the tensor-core kernel (the default) and the
CUDA-core kernel (GQA_Q8_KERNEL=fma), over head dims, group sizes, scale groups of 64 and 32
dims (qsa2.metal's per-64 scales, FORWARD_MSL's per-32 blocks), dense and selected-cell
visits, split and unsplit rows, and the head splits the planner may choose (up to 16, 8 or 4
heads a CTA).  Every case also checks that both kernels agree with each other.
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import TOL_Q8, _env, assert_close, forced_chunk, oracle_ref, run_case
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(case, kernel, split, chunk):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _env(GQA_Q8_KERNEL="fma" if kernel == "fma" else None, GQA_HEAD_SPLIT=split), \
            forced_chunk(chunk):
        got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) == 0
    return got


@pytest.mark.parametrize("chunk", [None, 64])
@pytest.mark.parametrize("sg", [64, 32])
@pytest.mark.parametrize("D,G,split", [(64, 8, None), (128, 16, 1), (128, 16, None),
                                       (256, 12, 1), (256, 12, 2), (256, 12, 3), (256, 6, None),
                                       (128, 1, None), (64, 5, None)])
def test_q8_kernels_agree_with_the_oracle(D, G, split, sg, chunk):
    case = W.make_q8_case(1400 + D + G, 3, 2 * G, 2, D, [900, 1, 333], budget=500,
                          cache_cap=960, scale=1 / math.sqrt(D), scale_group=sg)
    ref = oracle_ref(case)
    mma = _run(case, "mma", split, chunk)
    assert_close(mma, ref, TOL_Q8, f"mma D{D} G{G} split{split} sg{sg} chunk{chunk}")
    fma = _run(case, "fma", None, chunk)
    assert_close(fma, ref, TOL_Q8, f"fma D{D} G{G} sg{sg} chunk{chunk}")
    assert_close(mma, fma, 2 * TOL_Q8, "mma vs fma")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_q8_dense_many_rows(D):
    # dense visits (no id list), 24 rows of mixed length: a grid that fills the GPU
    L = [int(x) for x in np.random.default_rng(D).integers(0, 1500, size=24)]
    case = W.make_q8_case(1450 + D, 24, 16, 2, D, L, cache_cap=1500, scale=1 / math.sqrt(D))
    ref = oracle_ref(case)
    for kernel in ("mma", "fma"):
        assert_close(_run(case, kernel, None, None), ref, TOL_Q8, f"{kernel} D{D}")


def test_q8_large_scores_stay_exact():
    # scores spread wide (scale 1): the lazy rescale and the weights' hi/lo split hold
    case = W.make_q8_case(1460, 2, 24, 2, 256, [2000, 700], budget=1024, cache_cap=2000,
                          scale=1.0)
    assert_close(_run(case, "mma", None, 128), oracle_ref(case), TOL_Q8, "peaked")
