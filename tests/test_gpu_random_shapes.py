"""Seeded random problems on every decode path against the oracle: head sizes, group sizes,
row counts, ragged and empty lengths, rows sharing sequences, cache capacities that are not
multiples of any tile, ids, scale groups and forced chunk lengths drawn from a fixed generator,
so the set is the same every run.  All parameters stay inside what the calls accept."""

import math

import numpy as np
import pytest

import oracle
from gpu_util import TOL_F16, TOL_Q8, assert_close, dev, f16_kernel, forced_chunk, oracle_ref, run_case
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_CASES = 48


def _draw(seed):
    r = np.random.default_rng(seed)
    T = int(r.integers(1, 7))
    n_seq = int(r.integers(1, T + 1))
    seq_of = r.integers(0, n_seq, T)
    seq_of[:n_seq] = np.arange(n_seq)  # every sequence used
    cap = int(r.integers(1, 700))
    L = r.integers(0, cap + 1, T)
    L[r.random(T) < 0.15] = 0
    chunk = [None, 64, 128, 192, 256, 512][int(r.integers(0, 6))]
    return r, T, n_seq, seq_of, cap, L, chunk


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_f16(i):
    r, T, n_seq, seq_of, cap, L, chunk = _draw(7000 + i)
    D = [64, 128, 256][int(r.integers(0, 3))]
    G = [1, 2, 3, 4, 6, 8, 12, 16][int(r.integers(0, 8))]
    Hk = int(r.integers(1, 4))
    case = W.make_f16_case(7100 + i, T, G * Hk, Hk, D, L, cache_cap=cap, seq_of=seq_of,
                           n_seq=n_seq, scale=1 / math.sqrt(D))
    ref = oracle_ref(case)
    for kernel in ("chunked", "rows_mma", "fma"):
        with f16_kernel(kernel), forced_chunk(chunk):
            got = run_case(case).cpu().numpy()
        assert_close(got, ref, TOL_F16, f"f16 #{i} D{D} G{G} Hk{Hk} T{T} {kernel} chunk{chunk}")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_q8(i):
    r, T, n_seq, seq_of, cap, L, chunk = _draw(8000 + i)
    D = [64, 128, 256][int(r.integers(0, 3))]
    G = [1, 2, 3, 4, 6, 12][int(r.integers(0, 6))]
    Hk = int(r.integers(1, 3))
    sg = [64, 32][int(r.integers(0, 2))]
    budget = int(r.integers(1, cap + 1)) if r.random() < 0.5 else None
    case = W.make_q8_case(8100 + i, T, G * Hk, Hk, D, L, budget=budget, cache_cap=cap,
                          seq_of=seq_of, n_seq=n_seq, scale=1 / math.sqrt(D), scale_group=sg)
    with forced_chunk(chunk):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8,
                 f"q8 #{i} D{D} G{G} Hk{Hk} T{T} sg{sg} budget{budget} chunk{chunk}")


@pytest.mark.parametrize("i", range(N_CASES))
@pytest.mark.parametrize("kernel", ["mma", "fma"])
def test_random_turboquant(i, kernel, monkeypatch):
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    if kernel != "mma":
        monkeypatch.setenv("GQA_TQ_KERNEL", kernel)
    r, T, n_seq, seq_of, cap, L, chunk = _draw(9000 + i)
    D = [32, 64, 128][int(r.integers(0, 3))]
    G = [1, 2, 3, 4, 5, 8, 12, 16][int(r.integers(0, 8))]
    Hk = int(r.integers(1, 3))
    c = W.make_tq_case(9100 + i, T, G * Hk, Hk, D, L, cache_cap=cap, seq_of=seq_of, n_seq=n_seq)
    i32 = lambda a: dev(np.ascontiguousarray(a).view(np.int32))  # noqa: E731
    with forced_chunk(None if chunk is None else max(chunk, 128)):
        got = gd.attn_decode_tq(dev(c.q_rot), dev(c.q_jl), i32(c.k_polar), i32(c.k_jl),
                                i32(c.k_norms), i32(c.v_polar), i32(c.v_norms), c.centroids,
                                dev(c.signs), c.qjl_scale, dev(c.kv_len), scale=c.scale,
                                seq_of=dev(c.seq_of)).cpu().numpy()
    ref = oracle.decode_tq(c.q_rot, c.q_jl, c.k_polar, c.k_jl, c.k_norms, c.v_polar, c.v_norms,
                           c.centroids, c.signs, c.qjl_scale, c.scale, c.kv_len, c.seq_of)
    assert_close(got, ref, 1e-4, f"tq #{i} D{D} G{G} Hk{Hk} T{T} {kernel} chunk{chunk}")
