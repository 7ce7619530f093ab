"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element."""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TOL_F16, TOL_Q8, assert_close, dev, f16_kernel, forced_chunk, forced_ctas,
                      oracle_ref, run_case, tol_of)
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


# ----------------------------------------------------------------------------- named workloads

@pytest.mark.parametrize("name", ["tiny", "gqa_d64_L1024", "gqa_d64_L4096"])
def test_small_named_workloads(name):
    case = W.NAMED[name]()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err).cpu().numpy()
    assert_close(got, oracle_ref(case), tol_of(case), name)
    assert int(err.item()) == 0


def test_long_context_all_rows():
    """16 sequences, lengths U[1024, 32768], H=32, Hk=8, D=128: every output element."""
    case = W.long_context()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err, max_kv_len=int(case.kv_len.max())).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, "long_ctx")
    assert int(err.item()) == 0


def test_q8_selected_workload():
    """int8 KV, 48 heads over 4 KV heads, D=256, 1024 sorted ids out of 8192."""
    case = W.q8_selected()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, "q8_sel")
    assert int(err.item()) == 0


def test_batched_sampled_rows():
    """64 x 8192 batch: the full GPU launch, checked on sampled rows the oracle computes."""
    case = W.batched()
    got = run_case(case).cpu().numpy()
    rows = [0, 1, 17, 42, 62, 63]
    assert_close(got[rows], oracle_ref(case, rows=rows), TOL_F16, "batched")
    assert np.isfinite(got).all()


def test_long_ctx_full_sampled_rows():
    """16 x 32768 (the fixed-length long-context sub-case): full launch, sampled rows."""
    case = W.long_context_full()
    got = run_case(case).cpu().numpy()
    rows = [0, 9, 15]
    assert_close(got[rows], oracle_ref(case, rows=rows), TOL_F16, "long_ctx_full")
    assert np.isfinite(got).all()


def test_prefill_chunk_rows():
    """16 causal rows at 8176.. of one sequence (row r sees 8177 + r positions)."""
    case = W.prefill_chunk()
    got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, "prefill_chunk")


# ----------------------------------------------------------------------------- shape sweep

SHAPES = [(D, G) for D in (64, 128, 256) for G in (1, 2, 3, 4, 6, 8, 12, 16)]


@pytest.mark.parametrize("kernel", ["chunked", "fma"])
@pytest.mark.parametrize("chunk", [None, 64, 128])
@pytest.mark.parametrize("D,G", SHAPES)
def test_f16_shapes_chunked(D, G, chunk, kernel):
    # rows: ragged lengths over several tiles, a one-position row, an empty row; 2 KV heads
    case = W.make_f16_case(100 + D + G, 4, 2 * G, 2, D, [300, 1, 0, 133], cache_cap=320,
                           scale=1 / math.sqrt(D))
    with forced_chunk(chunk), f16_kernel(kernel):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, f"f16 {kernel} D{D} G{G} chunk{chunk}")
    assert (got[2] == 0).all()


@pytest.mark.parametrize("ctas", [None, 1, 3, 16, 77])
@pytest.mark.parametrize("D,G", SHAPES)
def test_f16_shapes_stream_k(D, G, ctas):
    # the same rows under several stream-K grids: shares that cut segments anywhere, shares
    # smaller than a tile, shares spanning many segments, and an empty row in between
    case = W.make_f16_case(100 + D + G, 4, 2 * G, 2, D, [300, 1, 0, 133], cache_cap=320,
                           scale=1 / math.sqrt(D))
    with forced_ctas(ctas), f16_kernel("streamk"):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, f"f16 stream-K D{D} G{G} ctas{ctas}")
    assert (got[2] == 0).all()


@pytest.mark.parametrize("kernel", ["streamk", "chunked", "fma"])
def test_long_context_subset_both_kernels(kernel):
    """Both f16 kernels on the long-context shape (4 sequences), every output element."""
    case = W.long_context_4()
    with f16_kernel(kernel):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, f"long_ctx_4 {kernel}")


def test_peaked_attention_stays_exact():
    """Scores spread over ~60 in log2 units (large scale): the lazy rescale and the hi/lo split
    of p must keep the result at the oracle's value."""
    case = W.make_f16_case(409, 2, 8, 2, 128, [3000, 2000], cache_cap=3000, scale=2.0)
    with forced_chunk(512):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, "peaked")


@pytest.mark.parametrize("chunk", [None, 128])
@pytest.mark.parametrize("D,G", SHAPES)
def test_q8_shapes_with_ids(D, G, chunk):
    case = W.make_q8_case(200 + D + G, 3, 2 * G, 2, D, [700, 5, 260], budget=300, cache_cap=720,
                          scale=1 / math.sqrt(D))
    with forced_chunk(chunk):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, f"q8 D{D} G{G} chunk{chunk}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_q8_dense(D):
    case = W.make_q8_case(300 + D, 2, 8, 2, D, [333, 129], cache_cap=400, scale=0.05)
    got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, f"q8 dense D{D}")


@pytest.mark.parametrize("chunk", [None, 128])
@pytest.mark.parametrize("ids", [False, True])
@pytest.mark.parametrize("D,G", [(64, 4), (128, 4), (256, 12), (128, 3)])
def test_q8_scale_blocks_of_32(D, G, ids, chunk):
    # FORWARD_MSL's q8 cache: one f16 scale per 32-element block
    case = W.make_q8_case(330 + D + G, 3, 2 * G, 2, D, [700, 5, 260],
                          budget=300 if ids else None, cache_cap=720, scale=1 / math.sqrt(D),
                          scale_group=32)
    assert case.ksc.shape[-1] == D // 32
    with forced_chunk(chunk):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, f"q8/32 D{D} G{G} ids{ids} chunk{chunk}")


def test_q8_scale_blocks_of_32_differ_from_64():
    # the same codes read with their own 32-blocks and with the 64-dim reading differ: the
    # kernel really takes the group from the scale layout
    case = W.make_q8_case(341, 1, 8, 2, 128, [300], cache_cap=300, scale=0.1, scale_group=32)
    got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, "q8/32")
    wrong = W.make_q8_case(341, 1, 8, 2, 128, [300], cache_cap=300, scale=0.1)
    wrong.kq, wrong.vq, wrong.q = case.kq, case.vq, case.q
    wrong.ksc, wrong.vsc = case.ksc[..., ::2].copy(), case.vsc[..., ::2].copy()
    assert np.abs(run_case(wrong).cpu().numpy() - got).max() > 1e-3


# ----------------------------------------------------------------------------- properties

def test_gather_is_bit_exact():
    """q8_sel(cache, ids) == q8_sel(cache gathered by ids, ids = iota), bit for bit."""
    case = W.make_q8_case(401, 2, 24, 2, 256, [3000, 2500], budget=1024, cache_cap=3000,
                          scale=1 / 16)
    got = run_case(case, max_kv_len=3000).cpu().numpy()
    g = W.make_q8_case(402, 2, 24, 2, 256, [1024, 1024], cache_cap=1024, scale=1 / 16)
    for t in range(2):
        J = case.ids[t]
        g.kq[t], g.vq[t] = case.kq[t, J], case.vq[t, J]
        g.ksc[t], g.vsc[t] = case.ksc[t, J], case.vsc[t, J]
    g.q = case.q
    iota = dev(np.tile(np.arange(1024, dtype=np.int32), (2, 1)))
    g.budget = 1024
    got2 = run_case(g, ids=iota, max_kv_len=1024).cpu().numpy()
    assert np.array_equal(got, got2)


@pytest.mark.parametrize("kernel", ["streamk", "chunked"])
def test_split_matches_unsplit_and_is_deterministic(kernel):
    case = W.make_f16_case(403, 3, 16, 4, 128, [5000, 64, 3001], cache_cap=5000, scale=0.09)
    with f16_kernel(kernel):
        with forced_chunk(100000), forced_ctas(1):
            one = run_case(case).cpu().numpy()
        with forced_chunk(64), forced_ctas(200):
            many = run_case(case).cpu().numpy()
            again = run_case(case).cpu().numpy()
    assert np.array_equal(many, again)
    ref = oracle_ref(case)
    assert_close(one, ref, TOL_F16, "one share / chunk")
    assert_close(many, ref, TOL_F16, "many shares / chunks")


def test_rows_sharing_a_sequence():
    case = W.make_f16_case(404, 5, 8, 2, 64, [50, 700, 699, 1, 700], cache_cap=700,
                           seq_of=[1, 0, 0, 1, 1], n_seq=2, scale=0.125)
    got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, "shared sequences")


# ----------------------------------------------------------------------------- error paths

def test_out_of_range_ids_are_skipped_and_flagged():
    case = W.make_q8_case(405, 1, 8, 2, 128, [400], budget=64, cache_cap=500, scale=0.1)
    case.ids[0, 5] = 450    # >= kv_len
    case.ids[0, 9] = -3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) & _gd().ERR_ID_RANGE
    J = [int(x) for x in case.ids[0] if 0 <= x < 400]
    ref = oracle.decode_q8(case.q, case.kq, case.vq, case.ksc, case.vsc, case.kv_len, case.scale,
                           ids=np.array([J]), budget=len(J))
    assert_close(got, ref, TOL_Q8, "skipped ids")


def test_kv_len_past_capacity_is_clamped_and_flagged():
    case = W.make_f16_case(406, 2, 4, 1, 64, [100, 90], cache_cap=100, scale=0.125)
    kv = case.kv_len.copy()
    case.kv_len[0] = 1000    # claims more than the cache holds
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err, max_kv_len=100).cpu().numpy()
    assert int(err.item()) & _gd().ERR_KVLEN_RANGE
    case.kv_len = kv
    assert_close(got, oracle_ref(case), TOL_F16, "clamped")


def test_bad_sequence_index_gives_zeros_and_flag():
    case = W.make_f16_case(407, 2, 4, 1, 64, [10, 10], cache_cap=16, seq_of=[0, 0], n_seq=1)
    case.seq_of = np.array([0, 5], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) & _gd().ERR_SEQ_RANGE
    assert (got[1] == 0).all()
    case.q, case.kv_len, case.seq_of = case.q[:1], case.kv_len[:1], case.seq_of[:1]
    assert_close(got[:1], oracle_ref(case), TOL_F16, "row 0")


def test_workspace_too_small_is_refused():
    gd = _gd()
    case = W.make_f16_case(408, 1, 4, 1, 64, [5000], cache_cap=5000)
    with forced_chunk(128):
        with pytest.raises(gd.GqaError, match="EWORKSPACE"):
            gd.attn_decode_f16(dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len),
                               ws=torch.empty(16, dtype=torch.uint8, device="cuda"))


# ----------------------------------------------------------------------------- merge entry point

@pytest.mark.parametrize("D", [64, 128, 256])
def test_merge_entry_point(D):
    rng = np.random.default_rng(D)
    T, S, H = 3, 7, 5
    acc = rng.standard_normal((T, S, H, D))
    m = rng.standard_normal((T, S, H)) * 3
    l = rng.uniform(0.5, 20, (T, S, H))
    n_valid = np.array([7, 0, 3], dtype=np.int32)
    part = np.concatenate([acc, m[..., None], l[..., None]], axis=-1).astype(np.float32)
    got = _gd().attn_merge(dev(part), dev(n_valid)).cpu().numpy()
    ref = oracle.lse_merge(part[..., :D].astype(np.float64), part[..., D].astype(np.float64),
                           part[..., D + 1].astype(np.float64), n_valid)
    assert_close(got, ref, 1e-5, "merge")
    assert (got[1] == 0).all()


def test_workspace_reuse_leaves_counters_zero():
    """One zeroed workspace serves several split calls of different shapes; the arrival counters
    at its head are zero again after every call."""
    gd = _gd()
    cases = [W.make_f16_case(410 + i, T, 8, 2, 128, L, cache_cap=4000, scale=0.1)
             for i, (T, L) in enumerate([(3, [4000, 10, 2500]), (2, [300, 3999]),
                                         (4, [1, 2, 3, 4000])])]
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    with forced_chunk(128):
        for case in cases:
            got = gd.attn_decode_f16(dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len),
                                     scale=case.scale, max_kv_len=4000, ws=ws)
            torch.cuda.synchronize()
            assert_close(got.cpu().numpy(), oracle_ref(case), TOL_F16, "reused ws")
            assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0


# ----------------------------------------------------------------------------- row grouping

ROWS_KERNELS = {"umma": "chunked", "mma": "rows_mma"}  # grouped rows: tcgen05 or mma.sync
ROWS_PER_GROUP = {"umma": 64, "mma": 32}  # (row, head) pairs per group


@pytest.mark.parametrize("rows", ["umma", "mma"])
@pytest.mark.parametrize("chunk", [None, 64, 256])
@pytest.mark.parametrize("D,G", [(D, G) for D in (64, 128) for G in (1, 2, 4, 8)])
def test_rows_grouped_by_sequence(D, G, chunk, rows):
    """Rows sharing a sequence are served from one staged K/V tile per group: runs longer than a
    group (G=8 on the mma.sync kernel: 4 rows), causal and ragged lengths inside a group, an
    empty row, a row of one position, and sequences interleaved."""
    seq_of = [0] * 11 + [1, 1, 2] + [0] * 3 + [2]
    L = [400 + 7 * r for r in range(11)] + [1, 399, 0, 300, 5, 401, 250]
    case = W.make_f16_case(500 + D + G, len(seq_of), 2 * G, 2, D, L, cache_cap=480,
                           seq_of=seq_of, n_seq=3, scale=1 / math.sqrt(D))
    gd = _gd()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with forced_chunk(chunk), f16_kernel(ROWS_KERNELS[rows]):
        assert gd.plan(len(seq_of), 2 * G, 2, D, 480, n_seq=3).row_group == ROWS_PER_GROUP[rows] // G
        got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert_close(got, oracle_ref(case), TOL_F16, f"rows {rows} D{D} G{G} chunk{chunk}")
    assert (got[13] == 0).all()


def test_rows_grouped_matches_per_row_kernel():
    """The prefill chunk (16 causal rows over one cache) with row grouping on either row kernel
    and without it."""
    case = W.prefill_chunk()
    got = run_case(case).cpu().numpy()
    with f16_kernel("rows_mma"):
        got_mma = run_case(case).cpu().numpy()
    with _rows_off():
        per_row = run_case(case).cpu().numpy()
    ref = oracle_ref(case)
    assert_close(got, ref, TOL_F16, "grouped (tcgen05)")
    assert_close(got_mma, ref, TOL_F16, "grouped (mma.sync)")
    assert_close(per_row, ref, TOL_F16, "per row")


def _rows_off():
    from gpu_util import _env
    return _env(GQA_F16_ROWS="off")


@pytest.mark.parametrize("rows", ["umma", "mma"])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_rows_grouped_long_runs(G, rows):
    """Runs longer than a group (pairs per group / G rows: 64 or 32 for G = 1), split at
    multiples of the group size, with a second sequence starting mid-group."""
    seq_of = [0] * 150 + [1] * 5
    L = [100 + r for r in range(150)] + [60, 0, 61, 62, 1]
    case = W.make_f16_case(600 + G, len(seq_of), 2 * G, 2, 64, L, cache_cap=260, seq_of=seq_of,
                           n_seq=2, scale=0.125)
    with f16_kernel(ROWS_KERNELS[rows]):
        got = run_case(case).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_F16, f"long runs {rows} G{G}")


@pytest.mark.parametrize("rows", ["umma", "mma"])
@pytest.mark.parametrize("chunk", [None, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_one_sequence_rows_with_bad_entries(G, chunk, rows):
    """Rows of a single sequence (the chunked-prefill layout, where the tcgen05 row kernel takes
    fixed runs of rows as its groups): entries of seq_of out of range at a group's first and
    last row, mid-group and at the end give zero rows and the flag; an empty row, a row of one
    position and ragged lengths beside them stay exact."""
    T = 150
    L = [200 + (37 * t) % 101 for t in range(T)]
    L[5], L[64] = 0, 1
    case = W.make_f16_case(700 + G, T, 2 * G, 2, 64, L, cache_cap=320, seq_of=[0] * T, n_seq=1,
                           scale=0.125)
    bad = [0, 31, 32, 63, 100, 149]
    seq_bad = case.seq_of.copy()
    seq_bad[bad] = [1, -1, 3, 7, 1, 2]
    good = [t for t in range(T) if t not in bad]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = oracle_ref(case)
    case.seq_of = seq_bad
    with forced_chunk(chunk), f16_kernel(ROWS_KERNELS[rows]):
        assert _gd().plan(T, 2 * G, 2, 64, 320, n_seq=1).row_group == ROWS_PER_GROUP[rows] // G
        got = run_case(case, err=err).cpu().numpy()
    assert int(err.item()) & _gd().ERR_SEQ_RANGE
    assert (got[bad] == 0).all()
    assert_close(got[good], ref[good], TOL_F16, f"one sequence {rows} G{G} chunk{chunk}")


@pytest.mark.parametrize("pair_layout", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_merge_with_sigmoid_gate(D, pair_layout):
    """attn_merge_gated: the merge times sigmoid(gate), for a plain [T][H][D] gate and for the
    gate half of per-head [query | gate] pairs (stride 2 D)."""
    rng = np.random.default_rng(D + 7)
    T, S, H = 3, 6, 4
    acc = rng.standard_normal((T, S, H, D))
    m = rng.standard_normal((T, S, H)) * 2
    l = rng.uniform(0.5, 9, (T, S, H))
    n_valid = np.array([6, 2, 0], dtype=np.int32)
    part = np.concatenate([acc, m[..., None], l[..., None]], axis=-1).astype(np.float32)
    g = (rng.standard_normal((T, H, D)) * 3).astype(np.float32)
    if pair_layout:
        qfull = np.concatenate([rng.standard_normal((T, H, D)).astype(np.float32), g], axis=-1)
        gate_t = dev(qfull).view(-1)[D:]  # the gate half of each [query | gate] pair
        stride = 2 * D
    else:
        gate_t, stride = dev(g), D
    got = _gd().attn_merge(dev(part), dev(n_valid), gate=gate_t, gate_stride=stride)
    ref = oracle.gated_merge(part[..., :D].astype(np.float64), part[..., D].astype(np.float64),
                             part[..., D + 1].astype(np.float64), n_valid, g)
    assert_close(got.cpu().numpy(), ref, 1e-5, "gated merge")


@pytest.mark.parametrize("Hk,chunk,fused", [(2, None, None), (2, 256, False), (1, 256, True)])
def test_rows_grouped_many_groups_merge_paths(Hk, chunk, fused):
    """Forty sequences of three rows each.  The planner keeps the tcgen05 row kernel's grid within
    one CTA per SM; with 256-position chunks forced, 3 x 2 x 40 CTAs do not fit, so merge_kernel
    follows the row kernel, while 3 x 1 x 40 do, and the chunk CTAs of each group merge their own
    partials.  All against the oracle."""
    rng = np.random.default_rng(650 + Hk)
    seq_of = np.repeat(np.arange(40), 3)
    L = rng.integers(1, 700, seq_of.size)
    case = W.make_f16_case(651 + Hk, seq_of.size, 2 * Hk, Hk, 64, L, cache_cap=700,
                           seq_of=seq_of, n_seq=40, scale=0.125)
    gd = _gd()
    with forced_chunk(chunk):
        pl = gd.plan(case.n_tok, 2 * Hk, Hk, 64, 700, n_seq=40)
        got = run_case(case).cpu().numpy()
    ctas = pl.grid_x * pl.grid_y * pl.grid_z
    assert pl.row_group == 32
    if fused is None:
        assert ctas <= 152
    else:
        assert pl.merge == 1 and (ctas <= 152) == fused
    assert_close(got, oracle_ref(case), TOL_F16, f"many groups Hk{Hk} chunk{chunk}")
