"""Plain, slow fp64 statement of single-query grouped-query decode attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product path imports this.

What is computed, for query row ``t`` and query head ``h`` (all arithmetic in float64):

    g      = h // (n_heads // n_kv_heads)                 KV head of the group
    s      = seq_of[t]                                    which sequence's cache
    J      = 0 .. kv_len[t]-1                             dense decode, or
    J      = ids[t][0 : min(kv_len[t], budget)]           selected cells
    x_j    = scale * sum_d q[t,h,d] * K^[s,j,g,d]         for j in J
    w_j    = exp(x_j - max x) / sum_j' exp(x_j' - max x)
    out    = sum_j w_j * V^[s,j,g,:]                      (all zeros when J is empty)

K^ / V^ are the dequantised cache rows: an f16 value widened exactly, or an int8 value times
the f16 scale of its 64-dim group (both products are exact in float64).

Passages followed (page title, then the part of it):
  * attention_gqa.metal (cera 0.5.4 sources): one KV head serves all query heads of its group,
    head -> KV head by integer division by the group size; phase 1 scores scaled q.k, phase 2
    max / exp(x - max) / sum, phase 3 the probability-weighted sum of V rows.
  * flash_attention.metal (cera 0.2.0 sources): the same single-query decode as one online pass;
    a zero-length sequence writes zeros.
  * qsa2.metal (regolith), qsa_attn2 and qsa_attn3: int8 K/V rows times one f16 scale per 64
    dims; a row visits the first min(n_kv, budget) entries of its selected-cell id list; the
    split partials are the unnormalised accumulator with the chunk's max and sum.
  * qsa2.metal (regolith), qsa_merge2: the log-sum-exp merge of those partials.
  * flash_attention_tq.metal (cera 0.4.0 sources): a causal row at position p attends to [0, p].
  * qsa2.metal (regolith), qsa_topk2: the selected-cell id list, top `budget` cells by block score.
  * FORWARD_MSL (cherenkov docs), kv_append_q8: quantise-on-append, amax / 127 and rint.
  * flash_attention_tq.metal (cera 0.4.0 sources): decode over a TurboQuant cache (PolarQuant
    centroid dot plus QJL sign correction, rotated-space accumulation, inverse Hadamard).

Where the pages leave a step open, the reading taken is stated in the docstring of the function
that takes it.
"""

from __future__ import annotations

import numpy as np

SCALE_GROUP = 64  # dims sharing one f16 scale in qsa2.metal's int8 cache (qsa_attn2)
SCALE_GROUPS = (32, 64)  # also FORWARD_MSL's q8 planes: one scale per 32-element block


# ----------------------------------------------------------------------------- dequantisation

def dequant_f16(x) -> np.ndarray:
    """f16 cache values widened to float64 (exact)."""
    return np.asarray(x, dtype=np.float16).astype(np.float64)


def _scale_index(D: int, nsc: int) -> np.ndarray:
    """The scale of each dim: contiguous groups of D / nsc dims (32 or 64)."""
    if nsc <= 0 or D % nsc or D // nsc not in SCALE_GROUPS:
        raise ValueError(f"{nsc} scales for {D} dims: groups must hold 32 or 64 dims")
    return np.arange(D) // (D // nsc)


def dequant_q8(vals, scales) -> np.ndarray:
    """int8 values times the f16 scale of their group, in float64 (exact).

    ``vals[..., D]`` int8 and ``scales[..., D // group]`` f16.  The group is read off the shapes:
    64 dims as in qsa2.metal's qsa_attn2, where a K element is float(int8) *
    float(scale[row*4 + dim/64]); 32 dims as in FORWARD_MSL's q8 planes (one symmetric scale
    per 32-element block, read back by attn_part2_q8).
    """
    v = np.asarray(vals, dtype=np.int8).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    return v * s[..., _scale_index(v.shape[-1], s.shape[-1])]


# ----------------------------------------------------------------------------- the definition

def _kv_head_of(h: int, group: int) -> int:
    """Query head h reads KV head h // group (attention_gqa.metal, q_head_base = kv_head*group)."""
    return h // group


def _width(kv_len: int, budget) -> int:
    """Number of id-list entries a row visits: min(n_kv, budget) (qsa2.metal, qsa_attn2)."""
    n = max(int(kv_len), 0)
    return n if budget is None else min(n, int(budget))


def _scores(qg: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """x[h, j] = scale * q_h . K_j  (attention_gqa.metal phase 1)."""
    return scale * (qg @ K.T)


def _softmax_rows(x: np.ndarray) -> np.ndarray:
    """Safe softmax along the last axis: exp(x - max) / sum (attention_gqa.metal phase 2)."""
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _weighted_sum(w: np.ndarray, V: np.ndarray) -> np.ndarray:
    """out[h, :] = sum_j w[h, j] V_j (attention_gqa.metal phase 3)."""
    return w @ V


def attend_positions(qg, Khat, Vhat, scale) -> np.ndarray:
    """Attention of the query heads ``qg [G][D]`` over explicit rows ``Khat/Vhat [n][D]``.

    An empty row set gives zeros (flash_attention.metal, the seq_len == 0 guard).
    """
    qg = np.asarray(qg, dtype=np.float64)
    if len(Khat) == 0:
        return np.zeros((qg.shape[0], qg.shape[1]), dtype=np.float64)
    x = _scores(qg, np.asarray(Khat, np.float64), float(scale))
    return _weighted_sum(_softmax_rows(x), np.asarray(Vhat, np.float64))


def selected_positions(kv_len: int, ids_row=None, budget=None) -> np.ndarray:
    """Cache positions a row visits: dense 0..kv_len-1, or the first min(kv_len, budget) ids.

    Ids must lie in [0, kv_len): the selected list names cells of this row's context
    (qsa2.metal, qsa_topk2 emits only cells below n_kv).  An id outside it raises.
    """
    if ids_row is None:
        return np.arange(max(int(kv_len), 0), dtype=np.int64)
    if budget is None:
        raise ValueError("ids need a budget")
    J = np.asarray(ids_row, dtype=np.int64)[: _width(kv_len, budget)]
    if len(J) and (J.min() < 0 or J.max() >= kv_len):
        raise ValueError("an id lies outside [0, kv_len)")
    return J


def _decode(q, kv_rows, n_kv_heads, kv_len, scale, seq_of, ids, budget, rows):
    q = np.asarray(q)
    T, H, D = q.shape
    if H % n_kv_heads:
        raise ValueError("n_heads must be a multiple of n_kv_heads")
    G = H // n_kv_heads
    rows = range(T) if rows is None else list(rows)
    out = np.zeros((len(rows), H, D), dtype=np.float64)
    for i, t in enumerate(rows):
        s = t if seq_of is None else int(seq_of[t])
        J = selected_positions(int(kv_len[t]), None if ids is None else ids[t], budget)
        for g in range(n_kv_heads):
            heads = [h for h in range(H) if _kv_head_of(h, G) == g]
            Khat, Vhat = kv_rows(s, J, g)
            out[i, heads] = attend_positions(q[t, heads].astype(np.float64), Khat, Vhat, scale)
    return out


def decode_f16(q, k_cache, v_cache, kv_len, scale, seq_of=None, ids=None, budget=None, rows=None):
    """Decode attention over an f16 cache ``[n_seq][cap][n_kv_heads][D]``; returns float64.

    ``q [T][H][D]`` (fp32 values, widened exactly), ``kv_len[T]``, ``seq_of[T]`` (None: row t
    reads sequence t), optional ``ids [T][budget]``.  ``rows`` restricts the output to a subset
    of query rows (returned in that order).
    """
    def kv_rows(s, J, g):
        return dequant_f16(k_cache[s, J, g, :]), dequant_f16(v_cache[s, J, g, :])

    return _decode(q, kv_rows, k_cache.shape[2], kv_len, scale, seq_of, ids, budget, rows)


def decode_q8(q, k_vals, v_vals, k_scales, v_scales, kv_len, scale, seq_of=None, ids=None,
              budget=None, rows=None):
    """Decode attention over an int8 cache with one f16 scale per 64 dims; returns float64.

    Values ``[n_seq][cap][n_kv_heads][D]`` int8, scales ``[n_seq][cap][n_kv_heads][D/64]`` f16.
    """
    def kv_rows(s, J, g):
        return (dequant_q8(k_vals[s, J, g, :], k_scales[s, J, g, :]),
                dequant_q8(v_vals[s, J, g, :], v_scales[s, J, g, :]))

    return _decode(q, kv_rows, k_vals.shape[2], kv_len, scale, seq_of, ids, budget, rows)


# ----------------------------------------------------------------------------- split + merge

def _split(q, kv_rows, n_kv_heads, kv_len, scale, seq_of, ids, budget, chunk):
    """Chunked partials over the visited list: for chunk c (entries [c*chunk, (c+1)*chunk)),
    m = max_j x_j, p_j = exp(x_j - m), l = sum_j p_j, acc = sum_j p_j V^_j (unnormalised).

    Returns acc [T][S][H][D], m [T][S][H], l [T][S][H], n_valid [T]; chunks at or past
    n_valid[t] are left as acc = 0, m = -inf, l = 0 (qsa2.metal, qsa_attn2 writes nothing for
    them and qsa_merge2 reads only the first ceil(width / chunk)).
    """
    q = np.asarray(q)
    T, H, D = q.shape
    G = H // n_kv_heads
    J_all = [selected_positions(int(kv_len[t]), None if ids is None else ids[t], budget)
             for t in range(T)]
    n_valid = np.array([-(-len(J) // chunk) for J in J_all], dtype=np.int64)
    S = max(1, int(n_valid.max()) if T else 1)
    acc = np.zeros((T, S, H, D))
    m = np.full((T, S, H), -np.inf)
    l = np.zeros((T, S, H))
    for t in range(T):
        s = t if seq_of is None else int(seq_of[t])
        for g in range(n_kv_heads):
            heads = [h for h in range(H) if _kv_head_of(h, G) == g]
            for c in range(int(n_valid[t])):
                Jc = J_all[t][c * chunk:(c + 1) * chunk]
                Khat, Vhat = kv_rows(s, Jc, g)
                x = _scores(q[t, heads].astype(np.float64), Khat, float(scale))
                mc = x.max(axis=-1)
                p = np.exp(x - mc[:, None])
                m[t, c, heads] = mc
                l[t, c, heads] = p.sum(axis=-1)
                acc[t, c, heads] = _weighted_sum(p, Vhat)
    return acc, m, l, n_valid


def split_partials_f16(q, k_cache, v_cache, kv_len, scale, chunk, seq_of=None, ids=None,
                       budget=None):
    def kv_rows(s, J, g):
        return dequant_f16(k_cache[s, J, g, :]), dequant_f16(v_cache[s, J, g, :])

    return _split(q, kv_rows, k_cache.shape[2], kv_len, scale, seq_of, ids, budget, chunk)


def split_partials_q8(q, k_vals, v_vals, k_scales, v_scales, kv_len, scale, chunk, seq_of=None,
                      ids=None, budget=None):
    def kv_rows(s, J, g):
        return (dequant_q8(k_vals[s, J, g, :], k_scales[s, J, g, :]),
                dequant_q8(v_vals[s, J, g, :], v_scales[s, J, g, :]))

    return _split(q, kv_rows, k_vals.shape[2], kv_len, scale, seq_of, ids, budget, chunk)


def lse_merge(acc, m, l, n_valid) -> np.ndarray:
    """Log-sum-exp merge of split partials (qsa2.metal, qsa_merge2):

        M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out = sum_c acc_c e_c / L

    over the first ``n_valid[t]`` chunks of row t; a row with no valid chunk gives zeros.
    ``acc [T][S][H][D]``, ``m, l [T][S][H]`` (natural-log m).
    """
    acc = np.asarray(acc, np.float64)
    m = np.asarray(m, np.float64)
    l = np.asarray(l, np.float64)
    T, S, H, D = acc.shape
    out = np.zeros((T, H, D))
    for t in range(T):
        n = int(n_valid[t])
        if n == 0:
            continue
        M = m[t, :n].max(axis=0)                    # [H]
        e = np.exp(m[t, :n] - M[None, :])           # [n][H]
        L = (l[t, :n] * e).sum(axis=0)              # [H]
        out[t] = (acc[t, :n] * e[:, :, None]).sum(axis=0) / L[:, None]
    return out


# ----------------------------------------------------------------------------- block top-k

def order_key(x) -> np.ndarray:
    """Order-preserving map of fp32 values to uint32 (the `okey` that qsa2.metal's qsa_topk2
    applies but does not define; the plain reading): flip every bit of a negative value, set the
    sign bit of a non-negative one, so unsigned order follows float order (-0 < +0)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    neg = (u >> 31) == 1
    return np.where(neg, (~u) & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


def select_topk_cells(block_scores_row, n_kv: int, budget: int) -> np.ndarray:
    """Selected-cell ids of one row (qsa2.metal, qsa_topk2).

    Cells 0..n_kv-1 come in blocks of 4; cell c carries its block's score, block_scores_row[c//4]
    (the last block may be partial).  Rows with n_kv <= budget select every cell.  Otherwise the
    `budget` cells with the largest keys are selected, equal keys going to the lower cell index
    (qsa_topk2 takes whole blocks above the threshold key and, at the threshold, blocks in
    ascending order and the first cells of a block).  Returned ascending, as qsa_topk2 emits.
    """
    n_kv = max(int(n_kv), 0)
    if n_kv <= budget:
        return np.arange(n_kv, dtype=np.int64)
    cells = np.arange(n_kv)
    keys = order_key(np.asarray(block_scores_row, np.float32)[cells // 4])
    # stable sort on descending key keeps ascending cell order among equal keys
    order = np.argsort(-keys.astype(np.int64), kind="stable")
    return np.sort(order[:budget]).astype(np.int64)


# ----------------------------------------------------------------------------- quantise on append

def quantize_q8(x, group: int = SCALE_GROUP) -> tuple[np.ndarray, np.ndarray]:
    """int8 codes and f16 scales of fp32 rows ``x[..., D]``, one scale per ``group`` dims
    (FORWARD_MSL, kv_append_q8: 32-element blocks; 64 for the int8 cache read by qsa2.metal):

        d = amax|x_group| / 127,  q = rint(x / d) clamped to [-127, 127] (0 when d = 0),
        scale = f16(d)

    Every step is taken in fp32, as the kernel takes it, so that the integer codes follow from
    the same roundings (IEEE division, round half to even).
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    if group not in SCALE_GROUPS or D % group:
        raise ValueError("group must be 32 or 64 and divide head_dim")
    g = x.reshape(x.shape[:-1] + (D // group, group))
    amax = np.abs(g).max(axis=-1)                                   # fp32
    d = (amax / np.float32(127)).astype(np.float32)                 # fp32 division
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d[..., None] > 0, np.rint(g / d[..., None]), np.float32(0))
    q = np.clip(q, -127, 127).astype(np.int8).reshape(x.shape)
    return q, d.astype(np.float16)


def output_gate(out, gate) -> np.ndarray:
    """The sigmoid output gate both model pages apply to an attention row after the merge
    (qsa2.metal, qsa_merge2; FORWARD_MSL, attn_combine): out * 1 / (1 + exp(-gate)), element by
    element; gate [T][H][D] is the second half of each head's [query | gate] pair there."""
    g = np.asarray(gate, np.float64)
    return np.asarray(out, np.float64) * (1.0 / (1.0 + np.exp(-g)))


def gated_merge(acc, m, l, n_valid, gate) -> np.ndarray:
    """The merge followed by the sigmoid output gate (qsa2.metal, qsa_merge2; FORWARD_MSL,
    attn_combine): output_gate(lse_merge(...), gate)."""
    return output_gate(lse_merge(acc, m, l, n_valid), gate)


# ----------------------------------------------------------------------------- TurboQuant KV

def unpack_polar(words, D: int) -> np.ndarray:
    """2-bit centroid indices, 16 per uint32, index k of a word in bits 2k..2k+1
    (flash_attention_tq.metal, the PolarQuant fields)."""
    w = np.asarray(words, dtype=np.uint64)[..., :, None]
    return ((w >> (2 * np.arange(16, dtype=np.uint64))) & 3).reshape(w.shape[:-2] + (D,))


def unpack_signs(words, D: int) -> np.ndarray:
    """QJL sign bits, 32 per uint32, bit k of a word for dim 32 w + k, as +-1."""
    w = np.asarray(words, dtype=np.uint64)[..., :, None]
    b = ((w >> np.arange(32, dtype=np.uint64)) & 1).reshape(w.shape[:-2] + (D,))
    return 2.0 * b.astype(np.float64) - 1.0


def half_pair(words):
    """(low f16, high f16) of uint32 words, widened to float64."""
    w = np.asarray(words, dtype=np.uint32)
    lo = (w & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (w >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    return lo, hi


def hadamard(D: int) -> np.ndarray:
    """Walsh-Hadamard matrix in Sylvester order, H[i, j] = (-1)^popcount(i & j) (unnormalised;
    the butterfly of flash_attention_tq.metal's epilogue computes H x)."""
    i = np.arange(D)
    bits = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(bits % 2 == 0, 1.0, -1.0)


def decode_tq(q_rot, q_jl, k_polar, k_jl, k_norms, v_polar, v_norms, centroids, signs,
              qjl_scale, scale, kv_len, seq_of=None, rows=None) -> np.ndarray:
    """Decode attention over a TurboQuant-compressed cache (flash_attention_tq.metal); float64.

    Layouts (head-major, as the page's compressed regions are: each KV head's positions
    contiguous): k_polar, v_polar [n_seq][Hk][cap][D/16] uint32; k_jl [n_seq][Hk][cap][D/32]
    uint32; k_norms [n_seq][Hk][cap] uint32 = (f16 norm, f16 residual norm) in the (low, high)
    halves; v_norms [n_seq][Hk][cap] uint32, f16 norm in
    the low half.  q_rot, q_jl [T][H][D] fp32 (the query already rotated and JL-projected).
    For row t, head h (KV head g = h // G) and visited position j:

        polar_j = sum_d q_rot[d] c[kidx_j(d)]
        signed_j = sum_d q_jl[d] s_j(d)                 (s = +-1 from the sign bits)
        x_j = (norm_j polar_j + norm_j rn_j qjl_scale signed_j) scale
        acc[d] = sum_j softmax(x)_j vnorm_j c[vidx_j(d)]            (rotated space)
        out = signs * (H acc) / sqrt(D)                  (the inverse randomized Hadamard)

    The page's precomputed per-head sum of q_jl is the sum over d of q_jl[d]: with it, twice the
    sum over set bits minus that sum is signed_j.  An empty row gives zeros.
    """
    q_rot = np.asarray(q_rot, np.float64)
    q_jl = np.asarray(q_jl, np.float64)
    T, H, D = q_rot.shape
    Hk = k_polar.shape[1]
    G = H // Hk
    c = np.asarray(centroids, np.float64)
    Hd = hadamard(D)
    sg = np.asarray(signs, np.float64)
    rows = range(T) if rows is None else list(rows)
    out = np.zeros((len(rows), H, D))
    for i, t in enumerate(rows):
        s = t if seq_of is None else int(seq_of[t])
        L = max(int(kv_len[t]), 0)
        if L == 0:
            continue
        for h in range(H):
            g = _kv_head_of(h, G)
            kidx = unpack_polar(k_polar[s, g, :L], D)
            ks = unpack_signs(k_jl[s, g, :L], D)
            norm, rn = half_pair(k_norms[s, g, :L])
            vidx = unpack_polar(v_polar[s, g, :L], D)
            vnorm, _ = half_pair(v_norms[s, g, :L])
            polar = c[kidx] @ q_rot[t, h]
            signed = ks @ q_jl[t, h]
            x = (norm * polar + norm * rn * qjl_scale * signed) * scale
            w = _softmax_rows(x[None, :])[0]
            acc = w @ (vnorm[:, None] * c[vidx])
            out[i, h] = sg * (Hd @ acc) / np.sqrt(D)
    return out
