"""GPU parity of attn_decode_tq (decode over a TurboQuant-compressed cache) against the fp64
oracle's decode_tq on the same seeded inputs, for the tensor-core kernel and the CUDA-core one:
one CTA per row, split rows merged by the last CTA, empty and ragged rows, rows sharing a
sequence, group sizes 1 to 16 and every head_dim, workspace reuse, out-of-range lengths flagged.

Tolerance: both sides decode the same packed words, f16 norms and fp32 centroids exactly; they
differ only by fp32 rounding of the dot products, the exp2 approximation and the order of the
sums.  |gpu - ref| <= 1e-4 * max(1, |ref|), the bound the int8 path uses."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, forced_chunk
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_TQ = 1e-4


@pytest.fixture(params=["mma", "fma"], autouse=True)
def tq_kernel(request, monkeypatch):
    """Every test runs on both kernels: tensor cores (the default) and CUDA cores."""
    if request.param == "mma":
        monkeypatch.delenv("GQA_TQ_KERNEL", raising=False)
    else:
        monkeypatch.setenv("GQA_TQ_KERNEL", request.param)
    return request.param


def _i32(a):
    return dev(np.ascontiguousarray(a).view(np.int32))


def run_tq(c, max_kv_len=None, ws=None, err=None, out=None, seq_of="case"):
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    so = dev(c.seq_of) if isinstance(seq_of, str) else seq_of
    return gd.attn_decode_tq(dev(c.q_rot), dev(c.q_jl), _i32(c.k_polar), _i32(c.k_jl),
                             _i32(c.k_norms), _i32(c.v_polar), _i32(c.v_norms), c.centroids,
                             dev(c.signs), c.qjl_scale, dev(c.kv_len), scale=c.scale, seq_of=so,
                             max_kv_len=max_kv_len, ws=ws, err=err, out=out)


def ref_tq(c, kv_len=None, rows=None):
    return oracle.decode_tq(c.q_rot, c.q_jl, c.k_polar, c.k_jl, c.k_norms, c.v_polar, c.v_norms,
                            c.centroids, c.signs, c.qjl_scale, c.scale,
                            c.kv_len if kv_len is None else kv_len, c.seq_of, rows=rows)


def check(got, ref, tol=TOL_TQ):
    got = got.detach().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= tol, f"max scaled error {err.max():.3e}"


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 4), (12, 4), (16, 4), (20, 4), (32, 4), (36, 4),
                                  (44, 4), (48, 4), (64, 4)])
def test_tq_group_sizes(D, H, Hk):
    """Group sizes 1 to 16: above 8 heads a group is served by several CTAs (9 heads: 3 x 3,
    11: 11 x 1, 12: 2 x 6, 16: 2 x 8)."""
    c = W.make_tq_case(2100 + D + H, 2, H, Hk, D, [300, 77])
    check(run_tq(c), ref_tq(c))


@pytest.mark.parametrize("chunk", [None, 128, 256, 384])
def test_tq_split_ragged_rows(chunk):
    # lengths straddling chunk and pass edges, an empty row, a one-position row; NaN norms past
    # every length
    L = [1000, 1, 0, 129, 511, 640]
    c = W.make_tq_case(2201, len(L), 16, 2, 128, L, cache_cap=1024)
    with forced_chunk(chunk):
        got = run_tq(c)
    ref = ref_tq(c)
    check(got, ref)
    assert torch.count_nonzero(got[2]) == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H", [8, 32, 48])
@pytest.mark.parametrize("chunk", [None, 128])
def test_tq_asymmetric_centroids(D, H, chunk):
    """Centroids that are not symmetric about zero (c3 - c2 - c1 + c0 != 0): the tensor-core
    kernel then needs the b0 b1 index plane as well; every other test draws the symmetric
    Lloyd-Max points, for which that plane drops out."""
    L = [700, 1, 0, 333]
    c = W.make_tq_case(2250 + D + H, len(L), H, 4, D, L, cache_cap=768)
    c.centroids = (np.array([-1.31, -0.17, 0.58, 1.73]) / np.sqrt(D)).astype(np.float32)
    assert c.centroids[3] - c.centroids[2] - c.centroids[1] + c.centroids[0] != 0
    with forced_chunk(chunk):
        got = run_tq(c)
    check(got, ref_tq(c))


@pytest.mark.parametrize("chunk", [None, 128])
def test_tq_shared_sequence_causal_rows(chunk):
    # chunked-prefill rows over one sequence: row r sees start + r + 1 positions
    L = [600 + r + 1 for r in range(6)]
    c = W.make_tq_case(2202, 6, 8, 2, 64, L, seq_of=[0] * 6, n_seq=1)
    with forced_chunk(chunk):
        check(run_tq(c), ref_tq(c))


def test_tq_named_prefill_chunk():
    c = W.tq_prefill_chunk()
    check(run_tq(c), ref_tq(c))


ROWS_CASES = [(D, G) for D in (64, 128) for G in (1, 2, 4, 8, 12, 16)]


@pytest.mark.parametrize("chunk", [None, 64, 256])
@pytest.mark.parametrize("D,G", ROWS_CASES)
def test_tq_rows_grouped_by_sequence(D, G, chunk, tq_kernel):
    """Rows sharing a sequence on the TurboQuant row kernel (the tensor-core path): runs longer
    than a group (64 / G rows), causal and ragged lengths, an empty row, a one-position row,
    sequences interleaved; against the oracle.  (The CUDA-core kernel serves each row alone.)"""
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    seq_of = [0] * 21 + [1, 1, 2] + [0] * 3 + [2]
    L = [300 + 7 * r for r in range(21)] + [1, 299, 0, 200, 5, 301, 150]
    c = W.make_tq_case(2300 + D + G, len(seq_of), 2 * G, 2, D, L, cache_cap=460,
                       seq_of=seq_of, n_seq=3)
    with forced_chunk(chunk):
        pl = gd.plan(len(seq_of), 2 * G, 2, D, 460, -1, gd.KIND_TQ, n_seq=3)
        if tq_kernel == "mma":
            hs = 1 if G <= 8 else 2
            assert pl.row_group == 64 // (G // hs) and pl.grid_y == 2 * hs
        else:
            assert pl.row_group == 1
        got = run_tq(c)
    check(got, ref_tq(c))
    assert torch.count_nonzero(got[23]) == 0


def test_tq_rows_match_one_cta_per_row(monkeypatch):
    """The prefill chunk grouped and one CTA per row (GQA_TQ_ROWS=off): both against the
    oracle."""
    c = W.tq_prefill_chunk()
    ref = ref_tq(c)
    grouped = run_tq(c).clone()
    monkeypatch.setenv("GQA_TQ_ROWS", "off")
    per_row = run_tq(c)
    check(grouped, ref)
    check(per_row, ref)


def test_tq_long_context_sampled_rows():
    # the full-size workload in the launch configuration the benchmark times; the oracle
    # recomputes three rows (the shortest, the longest, one between)
    c = W.tq_long_context()
    got = run_tq(c).cpu().numpy()
    order = np.argsort(c.kv_len)
    rows = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    check(got[rows], ref_tq(c, rows=rows))


def test_tq_workspace_reuse_and_two_calls():
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    c = W.make_tq_case(2203, 3, 32, 8, 128, [3000, 2000, 10], cache_cap=3000)
    ws = gd.alloc_workspace(3, 32, 8, 128, 3000, -1, gd.KIND_TQ, "cuda", 3)
    with forced_chunk(256):
        a = run_tq(c, ws=ws).clone()
        b = run_tq(c, ws=ws)
    assert torch.equal(a, b)
    check(a, ref_tq(c))
    cnt = -(-3 * 8 * 4 // 256) * 256
    assert torch.count_nonzero(ws[:cnt]) == 0   # arrival counters back at zero


def test_tq_length_out_of_range_is_flagged():
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    c = W.make_tq_case(2204, 2, 8, 2, 64, [200, 50], cache_cap=200)
    bad = c.kv_len.copy()
    bad[1] = 250   # beyond the cache: clamped to 200, bit flagged
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gd.attn_decode_tq(dev(c.q_rot), dev(c.q_jl), _i32(c.k_polar), _i32(c.k_jl),
                            _i32(c.k_norms), _i32(c.v_polar), _i32(c.v_norms), c.centroids,
                            dev(c.signs), c.qjl_scale, dev(bad), scale=c.scale,
                            seq_of=dev(c.seq_of), err=err)
    assert int(err.item()) & gd.ERR_KVLEN_RANGE
    check(got[0:1], ref_tq(c, rows=[0]))


@pytest.mark.parametrize("chunk", [None, 128])
def test_tq_head_dim_32_split_and_shared(chunk):
    # head_dim 32 (the CUDA-core kernel): split rows, rows sharing a sequence, an empty row, a
    # capacity that is not a multiple of 4
    L = [901, 0, 130, 899]
    c = W.make_tq_case(2206, 4, 8, 2, 32, L, cache_cap=902, seq_of=[0, 1, 1, 0], n_seq=2)
    with forced_chunk(chunk):
        check(run_tq(c), ref_tq(c))


@pytest.mark.parametrize("G", [12, 16])
def test_tq_head_split_many_rows(G):
    """Groups served by two CTAs of heads, with enough split rows that the arrival counters
    ([rows][KV heads x head split]) outgrow their first 256 bytes."""
    L = [700 - 23 * r for r in range(24)]
    c = W.make_tq_case(2209 + G, 24, 2 * G, 2, 64, L, cache_cap=700)
    with forced_chunk(128):
        check(run_tq(c), ref_tq(c))


@pytest.mark.parametrize("chunk", [None, 128])
def test_tq_twelve_heads_per_kv_head(chunk):
    """The int8 page's group shape (12 query heads per KV head, qsa2.metal qsa_attn2) over a
    TurboQuant cache: 48 heads over 4 KV heads, D = 128, split rows."""
    c = W.make_tq_case(2207, 2, 48, 4, 128, [2500, 700], cache_cap=2500)
    with forced_chunk(chunk):
        check(run_tq(c), ref_tq(c))


@pytest.mark.parametrize("chunk", [None, 256])
def test_tq_odd_capacity_and_stage_tails(chunk):
    """A cache capacity that is not a multiple of 4, lengths that end inside a 32-position
    stage and inside a 16-position block, at D = 128 and 64."""
    for D in (128, 64):
        L = [1003, 17, 33, 999, 1]
        c = W.make_tq_case(2208 + D, len(L), 8, 2, D, L, cache_cap=1003)
        with forced_chunk(chunk):
            check(run_tq(c), ref_tq(c))


def test_tq_rejects_large_group():
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    c = W.make_tq_case(2205, 1, 17, 1, 64, [64])
    with pytest.raises(gd.GqaError, match="GQA_EUNSUPPORTED"):
        run_tq(c)
