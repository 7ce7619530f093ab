"""CPU pins of the fp64 oracle (no GPU): closed forms, brute force, invariants, planted mistakes."""

import math

import numpy as np
import pytest

import oracle
import oracle.gqa_oracle as OG
import pins
from gqa_decode_attention_03_gb300 import workloads as W


def test_closed_forms():
    assert pins.check_closed_forms() == []


def test_brute_force_30_digits():
    assert pins.check_brute_force() == []


def test_invariants():
    assert pins.check_invariants() == []


def test_identical_keys_give_mean_of_v():
    c = W.make_f16_case(21, 1, 4, 1, 64, [33], scale=0.3)
    c.k[0, :33] = c.k[0, 0]  # every key equal -> uniform weights
    got = pins.oracle_case(c)
    mean = c.v[0, :33, 0].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(got[0], np.broadcast_to(mean, (4, 64)), rtol=1e-13, atol=1e-14)


def test_dominant_key_returns_its_row():
    c = W.make_f16_case(22, 1, 1, 1, 64, [40], scale=1.0)
    j = 17
    qn = c.q[0, 0].astype(np.float64)
    c.k[0, :40] = np.float16(0)
    c.k[0, j, 0] = (qn / np.linalg.norm(qn) * 8).astype(np.float16)  # x_j ~ 8 |q| ~ 64
    got = pins.oracle_case(c)[0, 0]
    xj = float(np.dot(qn, c.k[0, j, 0].astype(np.float64)))
    bound = 39 * math.exp(-xj) * np.abs(c.v[0, :40, 0].astype(np.float64)).max() * 2
    assert np.max(np.abs(got - c.v[0, j, 0].astype(np.float64))) <= bound


def test_permuting_positions_changes_nothing():
    c = W.make_f16_case(23, 1, 8, 2, 64, [45], scale=0.2)
    ref = pins.oracle_case(c)
    perm = np.random.default_rng(0).permutation(45)
    c.k[0, :45] = c.k[0, perm]
    c.v[0, :45] = c.v[0, perm]
    np.testing.assert_allclose(pins.oracle_case(c), ref, rtol=1e-12, atol=1e-13)


def test_empty_context_is_zero():
    c = W.make_f16_case(24, 2, 4, 2, 64, [0, 0], cache_cap=4)
    assert np.array_equal(pins.oracle_case(c), np.zeros((2, 4, 64)))
    acc, m, l, nv = oracle.split_partials_f16(c.q, c.k, c.v, c.kv_len, c.scale, 8)
    assert np.array_equal(oracle.lse_merge(acc, m, l, nv), np.zeros((2, 4, 64)))


def test_nan_past_length_is_never_read():
    # the generator fills positions >= kv_len with NaN; a finite answer shows none was read
    c = W.make_f16_case(25, 3, 4, 2, 64, [3, 9, 1], cache_cap=12, seq_of=[0, 0, 1])
    assert np.isnan(c.k[0, 9:]).all() and np.isfinite(pins.oracle_case(c)).all()


def test_selected_ids_equal_dense_over_gathered_cells():
    c = W.make_q8_case(26, 1, 12, 1, 128, [300], budget=40, scale=0.0625)
    ref = pins.oracle_case(c)
    J = c.ids[0, :40]
    g = W.make_q8_case(26, 1, 12, 1, 128, [40], scale=0.0625)
    g.kq[0, :40], g.vq[0, :40] = c.kq[0, J], c.vq[0, J]
    g.ksc[0, :40], g.vsc[0, :40] = c.ksc[0, J], c.vsc[0, J]
    g.q = c.q
    assert np.array_equal(pins.oracle_case(g), ref)


def test_selected_width_is_min_of_length_and_budget():
    c = W.make_q8_case(27, 2, 4, 1, 64, [5, 100], budget=8, scale=0.1)
    assert list(c.ids[0, :5]) == [0, 1, 2, 3, 4] and (c.ids[0, 5:] == -1).all()
    assert len(oracle.selected_positions(5, c.ids[0], 8)) == 5
    assert len(oracle.selected_positions(100, c.ids[1], 8)) == 8
    with pytest.raises(ValueError):
        oracle.selected_positions(3, np.array([0, 1, 5, 6]), 4)  # id 5 >= kv_len 3


def test_causal_rows_equal_truncated_decode():
    # flash_attention_tq.metal (cera 0.4.0): causal row r at position start+r sees [0, start+r]
    start, R = 20, 4
    c = W.make_f16_case(28, R, 4, 2, 64, [start + r + 1 for r in range(R)], cache_cap=start + R,
                        seq_of=[0] * R, n_seq=1)
    got = pins.oracle_case(c)
    for r in range(R):
        one = oracle.decode_f16(c.q[r:r + 1], c.k[:, :start + r + 1], c.v[:, :start + r + 1],
                                [start + r + 1], c.scale, seq_of=[0])
        assert np.array_equal(got[r], one[0])


def test_q8_dequant_cells_exact():
    vals = np.array([[-127, 1, 64, 0] * 16 + [5] * 64], dtype=np.int8)  # D = 128
    sc = np.array([[0.0125, 0.007]], dtype=np.float16)
    d = oracle.dequant_q8(vals, sc)
    s0, s1 = float(np.float16(0.0125)), float(np.float16(0.007))
    assert s0 == 0.0124969482421875  # 1638 / 1024 * 2**-7
    assert d[0, 0] == -127 * s0 and d[0, 2] == 64 * s0 and d[0, 64] == 5 * s1
    assert d[0, 63] == 0.0


def test_scale_folds_into_q():
    c = W.make_f16_case(29, 1, 4, 1, 64, [30], scale=0.25)
    ref = pins.oracle_case(c)
    c.q = c.q * 2  # exact in fp32
    c.scale = 0.125
    np.testing.assert_allclose(pins.oracle_case(c), ref, rtol=1e-14, atol=1e-15)


def test_merge_of_one_chunk_is_acc_over_l():
    rng = np.random.default_rng(3)
    acc = rng.standard_normal((1, 1, 2, 64))
    m = rng.standard_normal((1, 1, 2))
    l = rng.uniform(0.5, 4, (1, 1, 2))
    got = oracle.lse_merge(acc, m, l, [1])
    np.testing.assert_allclose(got[0], acc[0, 0] / l[0, 0][:, None], rtol=1e-15)


# ----------------------------------------------------------------------------- planted mistakes

def _mutants():
    """Plausible mistakes planted in the oracle; the battery must catch every one."""
    return {
        "kv head by modulo": ("_kv_head_of", lambda h, group: h % group),
        "scale dropped": ("_scores", lambda qg, K, scale: qg @ K.T),
        "scale squared": ("_scores", lambda qg, K, scale: scale * scale * (qg @ K.T)),
        "max sign flipped": ("_softmax_rows",
                             lambda x: (lambda e: e / e.sum(-1, keepdims=True))(
                                 np.exp(x.max(-1, keepdims=True) - x))),
        "not normalised": ("_softmax_rows", lambda x: np.exp(x - x.max(-1, keepdims=True))),
        "v rows reversed": ("_weighted_sum", lambda w, V: w @ V[::-1]),
        "k used for v": None,  # handled below via attend_positions
        "budget ignored": ("_width", lambda n, budget: max(int(n), 0)),
        "width off by one": ("_width",
                             lambda n, budget: max(int(n), 0) if budget is None
                             else max(0, min(max(int(n), 0), int(budget)) - 1)),
        "scale groups interleaved": ("_scale_index",
                                     lambda D, nsc: np.arange(D) % nsc),
        "scale groups reversed": ("_scale_index",
                                  lambda D, nsc: (nsc - 1) - np.arange(D) // (D // nsc)),
    }


@pytest.mark.parametrize("name", [k for k in _mutants()])
def test_planted_mistake_is_caught(name, monkeypatch):
    assert pins.battery() == []
    spec = _mutants()[name]
    if spec is None:
        orig = OG.attend_positions

        def wrong(qg, Khat, Vhat, scale):
            return orig(qg, Khat, Khat, scale)
        monkeypatch.setattr(OG, "attend_positions", wrong)
    else:
        monkeypatch.setattr(OG, spec[0], spec[1])
    assert pins.battery() != [], f"planted mistake '{name}' went unnoticed"


def test_planted_merge_mistakes_are_caught(monkeypatch):
    import numpy as _np

    def merge_without_weights(acc, m, l, n_valid):
        acc = _np.asarray(acc, _np.float64)
        T, S, H, D = acc.shape
        out = _np.zeros((T, H, D))
        for t in range(T):
            n = int(n_valid[t])
            if n:
                out[t] = acc[t, :n].sum(0) / _np.asarray(l)[t, :n].sum(0)[:, None]
        return out
    monkeypatch.setattr(oracle, "lse_merge", merge_without_weights)
    assert pins.check_closed_forms() != [] or pins.check_invariants() != []


# ----------------------------------------------------------------------------- block top-k

def _topk_brute(scores, n_kv, budget):
    """Plain Python: cells ranked by (score descending, cell ascending), first `budget` taken."""
    cells = sorted(range(n_kv), key=lambda c: (-float(scores[c // 4]), c))
    return sorted(cells[:budget]) if n_kv > budget else list(range(n_kv))


def topk_pin_failures():
    fails = []
    rng = np.random.default_rng(5)
    for trial in range(300):
        n_kv = int(rng.integers(1, 90))
        budget = int(rng.integers(1, 40))
        nb = n_kv // 4 + 1
        # few distinct non-zero values so that ties cross the threshold often
        scores = rng.choice(np.array([-3.5, -1.0, -0.25, 0.5, 2.0, 7.0], np.float32), size=nb)
        try:
            got = list(oracle.select_topk_cells(scores, n_kv, budget))
        except Exception as e:
            fails.append(f"raised {e!r}")
            break
        if got != _topk_brute(scores, n_kv, budget):
            fails.append(f"trial {trial}: n_kv {n_kv} budget {budget}")
            break
    return fails


def test_topk_matches_plain_ranking():
    assert topk_pin_failures() == []


def test_order_key_is_monotone():
    x = np.array([-np.inf, -3e38, -1.5, -1e-30, -0.0, 0.0, 1e-30, 2.0, 3e38, np.inf], np.float32)
    k = oracle.order_key(x)
    assert (np.diff(k.astype(np.int64)) > 0).all()


def test_topk_closed_cases():
    # page's short-row rule: n_kv <= budget selects every cell
    assert list(oracle.select_topk_cells(np.zeros(3, np.float32), 9, 9)) == list(range(9))
    # ties at the threshold go to the lower blocks, and to the first cells of a block:
    # blocks (cells) 0:(0-3)=1, 1:(4-7)=5, 2:(8-11)=5, 3:(12,13)=2; budget 6 -> cells 4..9
    s = np.array([1, 5, 5, 2], np.float32)
    assert list(oracle.select_topk_cells(s, 14, 6)) == [4, 5, 6, 7, 8, 9]
    # the partial last block holds n_kv % 4 cells: here 2 cells of the best block
    s = np.array([1, 1, 9], np.float32)
    assert list(oracle.select_topk_cells(s, 10, 3)) == [0, 8, 9]


@pytest.mark.parametrize("name", ["ties to higher cells", "full last block", "sign ignored"])
def test_planted_topk_mistakes_are_caught(name, monkeypatch):
    assert topk_pin_failures() == []
    if name == "ties to higher cells":
        def wrong(block_scores_row, n_kv, budget):
            n_kv = int(n_kv)
            if n_kv <= budget:
                return np.arange(n_kv)
            keys = OG.order_key(np.asarray(block_scores_row, np.float32)[np.arange(n_kv) // 4])
            order = np.argsort(-keys.astype(np.int64), kind="stable")[::-1]
            order = order[np.argsort(-keys[order].astype(np.int64), kind="stable")]
            return np.sort(order[:budget])
        monkeypatch.setattr(oracle, "select_topk_cells", wrong)
    elif name == "full last block":
        def wrong(block_scores_row, n_kv, budget):
            n = int(n_kv)
            return OG.select_topk_cells.__wrapped__(block_scores_row, (n // 4 + 1) * 4, budget)
        OG.select_topk_cells.__wrapped__ = OG.select_topk_cells
        monkeypatch.setattr(oracle, "select_topk_cells", wrong)
    else:
        monkeypatch.setattr(OG, "order_key",
                            lambda x: np.asarray(x, np.float32).view(np.uint32).astype(np.uint64))
    assert topk_pin_failures() != [], f"planted mistake '{name}' went unnoticed"


# ----------------------------------------------------------------------------- quantise on append

def test_quantize_roundtrip_within_half_a_step():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((5, 3, 128)) * rng.uniform(0.01, 100, (5, 3, 1))).astype(np.float32)
    q, s = oracle.quantize_q8(x)
    d = x.reshape(5, 3, 2, 64)
    amax = np.abs(d).max(-1)
    deq = q.reshape(5, 3, 2, 64).astype(np.float64) * (amax / 127.0)[..., None]
    # |x - q d| <= d / 2 (up to fp32 rounding of d), the largest element maps to +-127
    assert (np.abs(d - deq) <= (amax / 127.0)[..., None] * (0.5 + 1e-5)).all()
    big = np.abs(d).argmax(-1)
    assert (np.abs(np.take_along_axis(q.reshape(5, 3, 2, 64), big[..., None], -1)) == 127).all()
    assert np.array_equal(s, (amax / np.float32(127)).astype(np.float16))


def test_quantize_closed_cases():
    x = np.zeros((1, 64), np.float32)
    q, s = oracle.quantize_q8(x)
    assert (q == 0).all() and (s == 0).all()           # an all-zero group: scale 0, codes 0
    x = np.linspace(-1, 1, 64, dtype=np.float32)[None]  # amax 1: d = 1/127, q = rint(127 x)
    q, s = oracle.quantize_q8(x)
    assert np.array_equal(q[0], np.rint(x[0] / np.float32(1 / 127)).astype(np.int8))
    assert q[0, 0] == -127 and q[0, -1] == 127 and s[0, 0] == np.float16(1 / 127)
    # halves round to even: x = 2.5 d -> 2, 3.5 d -> 4 (d = 127 / 127 = 1 when amax = 127)
    x = np.zeros((1, 64), np.float32)
    x[0, :4] = [127.0, 2.5, 3.5, -2.5]
    q, _ = oracle.quantize_q8(x)
    assert list(q[0, :4]) == [127, 2, 4, -2]


def test_quantize_32_element_blocks():
    # FORWARD_MSL's kv_append_q8 block: 32 elements share d = amax / 127
    x = np.zeros((1, 64), np.float32)
    x[0, :32] = np.linspace(-2, 2, 32, dtype=np.float32)   # amax 2
    x[0, 32:] = np.linspace(-0.5, 0.25, 32, dtype=np.float32)  # amax 0.5
    q, s = oracle.quantize_q8(x, group=32)
    assert s.shape == (1, 2)
    assert s[0, 0] == np.float16(np.float32(2) / np.float32(127))
    assert s[0, 1] == np.float16(np.float32(0.5) / np.float32(127))
    assert q[0, 0] == -127 and q[0, 31] == 127 and q[0, 32] == -127
    assert q[0, 63] == np.rint(np.float32(0.25) / (np.float32(0.5) / np.float32(127)))
    # 32-groups of a row equal the 64-group code of each half quantised alone
    rng = np.random.default_rng(12)
    y = rng.standard_normal((3, 128)).astype(np.float32)
    q32, s32 = oracle.quantize_q8(y, group=32)
    for b in range(4):
        qb, sb = oracle.quantize_q8(np.tile(y[:, 32 * b:32 * (b + 1)], 2), group=64)
        assert np.array_equal(q32[:, 32 * b:32 * (b + 1)], qb[:, :32])
        assert np.array_equal(s32[:, b], sb[:, 0])
    with pytest.raises(ValueError):
        oracle.quantize_q8(y, group=16)


def test_dequant_reads_the_group_off_the_shapes():
    vals = np.arange(-64, 64, dtype=np.int8).reshape(1, 128)
    s64 = np.array([[0.5, 2.0]], np.float16)
    s32 = np.array([[0.5, 1.0, 2.0, 4.0]], np.float16)
    d64 = oracle.dequant_q8(vals, s64)
    d32 = oracle.dequant_q8(vals, s32)
    assert d64[0, 63] == -1 * 0.5 and d64[0, 64] == 0 * 2.0 and d64[0, 127] == 63 * 2.0
    assert d32[0, 31] == -33 * 0.5 and d32[0, 32] == -32 * 1.0 and d32[0, 95] == 31 * 2.0
    assert d32[0, 96] == 32 * 4.0
    with pytest.raises(ValueError):
        oracle.dequant_q8(vals, np.ones((1, 8), np.float16))


def test_gated_merge_closed_forms():
    rng = np.random.default_rng(4)
    acc = rng.standard_normal((1, 2, 1, 64))
    m = np.array([[[0.0], [np.log(3.0)]]])
    l = np.ones((1, 2, 1))
    base = oracle.lse_merge(acc, m, l, [2])
    # gate 0 halves the row; a large gate passes it, a very negative one closes it
    assert np.allclose(oracle.gated_merge(acc, m, l, [2], np.zeros((1, 1, 64))), base / 2)
    assert np.allclose(oracle.gated_merge(acc, m, l, [2], np.full((1, 1, 64), 40.0)), base)
    assert np.allclose(oracle.gated_merge(acc, m, l, [2], np.full((1, 1, 64), -40.0)), 0,
                       atol=1e-16)
    g = np.full((1, 1, 64), np.log(3.0))  # sigmoid(ln 3) = 3/4
    assert np.allclose(oracle.gated_merge(acc, m, l, [2], g), 0.75 * base, rtol=1e-14)


def test_output_gate_closed_forms():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 3, 64))
    g = rng.standard_normal((2, 3, 64)) * 4
    # sigmoid(g) + sigmoid(-g) = 1: the two gated rows add back to the row
    assert np.allclose(oracle.output_gate(x, g) + oracle.output_gate(x, -g), x, rtol=1e-14,
                       atol=1e-15)
    assert np.array_equal(oracle.output_gate(x, np.zeros_like(g)), x / 2)  # sigmoid(0) = 1/2
    assert np.allclose(oracle.output_gate(x, np.full_like(g, np.log(3.0))), 0.75 * x,
                       rtol=1e-14)  # sigmoid(ln 3) = 3/4
    assert np.allclose(oracle.output_gate(x, np.full_like(g, -np.log(3.0))), 0.25 * x,
                       rtol=1e-13)
    # element by element: one gate entry moves one output entry
    g2 = np.zeros_like(g)
    g2[1, 2, 7] = np.log(3.0)
    d = oracle.output_gate(x, g2) - x / 2
    assert np.count_nonzero(np.abs(d) > 1e-15) == 1 and abs(d[1, 2, 7] - 0.25 * x[1, 2, 7]) < 1e-14


# ----------------------------------------------------------------------------- TurboQuant

def _tq_oracle(c, rows=None):
    return oracle.decode_tq(c.q_rot, c.q_jl, c.k_polar, c.k_jl, c.k_norms, c.v_polar, c.v_norms,
                            c.centroids, c.signs, c.qjl_scale, c.scale, c.kv_len, c.seq_of, rows)


def _tq_dense_reference(c):
    """The same attention built another way: keys and values reconstructed element by element
    with Python integer bit operations, the query as the concatenation [q_rot | q_jl], the
    (pinned) dense oracle's attend_positions, then the inverse rotation as an explicit sum."""
    T, H, D = c.q_rot.shape
    G = H // c.n_kv_heads
    out = np.zeros((T, H, D))
    f16 = lambda bits: float(np.uint16(bits).view(np.float16))  # noqa: E731
    for t in range(T):
        s, L = int(c.seq_of[t]), int(c.kv_len[t])
        for h in range(H):
            g = h // G
            K2, V = [], []
            for j in range(L):
                kw = int(c.k_norms[s, g, j])
                norm, rn = f16(kw & 0xFFFF), f16(kw >> 16)
                vn = f16(int(c.v_norms[s, g, j]) & 0xFFFF)
                kp = [float(c.centroids[(int(c.k_polar[s, g, j, d // 16]) >> (2 * (d % 16))) & 3])
                      for d in range(D)]
                sb = [1.0 if (int(c.k_jl[s, g, j, d // 32]) >> (d % 32)) & 1 else -1.0
                      for d in range(D)]
                vp = [float(c.centroids[(int(c.v_polar[s, g, j, d // 16]) >> (2 * (d % 16))) & 3])
                      for d in range(D)]
                K2.append([norm * x for x in kp] + [norm * rn * c.qjl_scale * x for x in sb])
                V.append([vn * x for x in vp])
            q2 = np.concatenate([c.q_rot[t, h], c.q_jl[t, h]]).astype(np.float64)[None]
            acc = oracle.attend_positions(q2, np.array(K2), np.array(V), c.scale)[0] if L else \
                np.zeros(D)
            for i in range(D):
                hs = sum((acc[j] if bin(i & j).count("1") % 2 == 0 else -acc[j]) for j in range(D))
                out[t, h, i] = float(c.signs[i]) * hs / np.sqrt(D)
    return out


def test_tq_matches_dense_reconstruction():
    c = W.make_tq_case(31, 3, 4, 2, 32, [9, 0, 4], cache_cap=10)
    np.testing.assert_allclose(_tq_oracle(c), _tq_dense_reference(c), rtol=1e-12, atol=1e-13)


def test_tq_constant_values_rotate_to_one_spike():
    # every V index the same centroid and equal V norms: acc is constant, so H acc = D acc e_0
    c = W.make_tq_case(32, 1, 2, 1, 64, [12])
    c.v_polar[:] = np.uint32(0xAAAAAAAA)            # index 2 in every field
    c.v_norms[0, 0, :12] = W._half_bits(1.25)
    got = _tq_oracle(c)
    spike = float(c.signs[0]) * 64 * 1.25 * float(c.centroids[2]) / np.sqrt(64)
    assert np.allclose(got[0, :, 0], spike, rtol=1e-12) and np.allclose(got[0, :, 1:], 0, atol=1e-14)


def test_hadamard_is_self_inverse_up_to_d():
    for D in (32, 64, 128):
        H = oracle.hadamard(D)
        assert np.array_equal(H @ H, D * np.eye(D)) and (H[0] == 1).all()


@pytest.mark.parametrize("name", ["polar bit order", "signs as bits", "no sqrt(D)"])
def test_planted_tq_mistakes_are_caught(name, monkeypatch):
    c = W.make_tq_case(33, 2, 4, 2, 32, [6, 3], cache_cap=6)
    ref = _tq_dense_reference(c)
    if name == "polar bit order":
        monkeypatch.setattr(OG, "unpack_polar", lambda w, D: ((np.asarray(w, np.uint64)[..., :, None] >> (30 - 2 * np.arange(16, dtype=np.uint64))) & 3).reshape(np.asarray(w).shape[:-1] + (D,)))  # noqa: E501
    elif name == "signs as bits":
        orig = OG.unpack_signs
        monkeypatch.setattr(OG, "unpack_signs", lambda w, D: (orig(w, D) + 1) / 2)
    else:
        orig = OG.hadamard
        monkeypatch.setattr(OG, "hadamard", lambda D: orig(D) * np.sqrt(D))
    assert not np.allclose(_tq_oracle(c), ref, rtol=1e-9, atol=1e-12)
