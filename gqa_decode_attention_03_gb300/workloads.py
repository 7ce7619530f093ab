"""Seeded synthetic inputs for decode attention.

This module only draws random numbers and lays them out; it holds none of the attention
arithmetic.  Tests, ``bench.py`` and ``smoke()`` build their inputs here and hand the same host
arrays to both the CUDA library and the CPU oracle.

Recipe (numpy ``PCG64``; one child stream per tensor and per sequence from
``SeedSequence(seed).spawn``, so the values do not depend on the thread count):

* q: fp32 N(0, 1).
* f16 K/V: fp32 N(0, 1) rounded to f16 (round to nearest even).
* int8 K/V: uniform integers in [-127, 127]; scales: f16 of uniform [0.005, 0.02], one per
  64 dims of each (cell, KV head) row.
* Cache positions at or past a sequence's length are filled with NaN (f16) or NaN scales
  (int8), so any read of them that reaches the output shows up as NaN.
* Selected ids: ``budget`` distinct positions drawn without replacement from [0, kv_len),
  sorted ascending; rows with kv_len <= budget get 0..kv_len-1 then -1 padding.
* long-context lengths: uniform integers in [1024, 32768].
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F16_NAN = np.float16(np.nan)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _gen(ss) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(ss))


def _fill_normal_f16(dst: np.ndarray, seq_streams, kv_len_per_seq) -> None:
    """dst [n_seq][cap][Hk][D] f16: N(0,1) at positions < kv_len of each sequence, NaN past it."""
    n_seq = dst.shape[0]

    def one(s):
        L = int(kv_len_per_seq[s])
        dst[s, L:] = F16_NAN
        if L == 0:
            return
        g = _gen(seq_streams[s])
        # generate in slabs of positions through one reused fp32 buffer (no page-fault churn)
        row = dst.shape[2] * dst.shape[3]
        step = max(1, (1 << 22) // max(1, row))
        buf = np.empty(step * row, dtype=np.float32)
        for p0 in range(0, L, step):
            p1 = min(L, p0 + step)
            n = (p1 - p0) * row
            g.standard_normal(out=buf[:n], dtype=np.float32)
            dst[s, p0:p1] = buf[:n].reshape(dst[s, p0:p1].shape)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(n_seq)))


def _fill_q8(vals: np.ndarray, scales: np.ndarray, seq_streams, kv_len_per_seq) -> None:
    n_seq = vals.shape[0]

    def one(s):
        L = int(kv_len_per_seq[s])
        vals[s, L:] = 0
        scales[s, L:] = F16_NAN
        if L == 0:
            return
        g = _gen(seq_streams[s])
        vals[s, :L] = g.integers(-127, 128, size=vals[s, :L].shape, dtype=np.int16).astype(np.int8)
        scales[s, :L] = g.uniform(0.005, 0.02, size=scales[s, :L].shape).astype(np.float16)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(n_seq)))


@dataclass
class Case:
    """One decode-attention problem, all arrays on the host."""
    name: str
    q: np.ndarray                      # [T][H][D] float32
    kv_len: np.ndarray                 # [T] int32
    seq_of: np.ndarray                 # [T] int32
    scale: float
    n_kv_heads: int
    cache_cap: int
    kind: str                          # "f16" or "q8"
    k: np.ndarray | None = None        # f16 [n_seq][cap][Hk][D]
    v: np.ndarray | None = None
    kq: np.ndarray | None = None       # int8 [n_seq][cap][Hk][D]
    vq: np.ndarray | None = None
    ksc: np.ndarray | None = None      # f16 [n_seq][cap][Hk][D/64]
    vsc: np.ndarray | None = None
    ids: np.ndarray | None = None      # [T][budget] int32
    budget: int | None = None
    seed: int = 0
    meta: dict = field(default_factory=dict)
    scale_group: int = 64              # int8: dims per f16 scale (64, or 32)

    @property
    def n_tok(self):
        return self.q.shape[0]

    @property
    def n_heads(self):
        return self.q.shape[1]

    @property
    def head_dim(self):
        return self.q.shape[2]

    @property
    def n_seq(self):
        return (self.k if self.kind == "f16" else self.kq).shape[0]

    def visited(self, t: int) -> int:
        """Positions row t visits (dense: kv_len; selected: min(kv_len, budget))."""
        L = max(int(self.kv_len[t]), 0)
        return L if self.ids is None else min(L, int(self.budget))

    def kv_bytes(self) -> int:
        """K/V (and scale) bytes the rows must read once per KV head: the algorithmic KV read."""
        D, Hk = self.head_dim, self.n_kv_heads
        per_pos = 2 * D * 2 if self.kind == "f16" else 2 * (D + 2 * (D // self.scale_group))
        if self.ids is None and len(set(self.seq_of.tolist())) < self.n_tok:
            # rows sharing a sequence (causal prefill rows) need each position once
            tot = 0
            for s in set(self.seq_of.tolist()):
                tot += max(self.visited(t) for t in range(self.n_tok) if self.seq_of[t] == s)
            return tot * Hk * per_pos
        return sum(self.visited(t) for t in range(self.n_tok)) * Hk * per_pos

    def algorithmic_bytes(self) -> int:
        """KV bytes + ids + q (fp32) + out (fp32) (+ block scores read by the selection when the
        ids are chosen in the step): the bytes a perfect pipeline moves per step."""
        extra = 2 * self.q.size * 4
        if self.ids is not None:
            extra += sum(self.visited(t) for t in range(self.n_tok)) * 4
        if "block_scores" in self.meta:
            extra += self.meta["block_scores"].nbytes
        return self.kv_bytes() + extra

    def flops(self) -> int:
        """4*D flops per (query head, visited position): 2*D for q.k, 2*D for p.v."""
        return sum(self.visited(t) for t in range(self.n_tok)) * self.n_heads * 4 * self.head_dim


def make_f16_case(seed, n_tok, n_heads, n_kv_heads, head_dim, kv_len, cache_cap=None,
                  seq_of=None, n_seq=None, scale=None, name="f16") -> Case:
    """Random f16-cache problem.  ``kv_len`` per row; ``seq_of`` defaults to row t -> sequence t."""
    kv_len = np.asarray(kv_len, dtype=np.int32).reshape(n_tok)
    seq_of = (np.arange(n_tok, dtype=np.int32) if seq_of is None
              else np.asarray(seq_of, dtype=np.int32).reshape(n_tok))
    n_seq = int(seq_of.max()) + 1 if n_seq is None else n_seq
    cap = int(max(1, kv_len.max())) if cache_cap is None else int(cache_cap)
    per_seq = np.zeros(n_seq, dtype=np.int64)
    for t in range(n_tok):
        per_seq[seq_of[t]] = max(per_seq[seq_of[t]], min(int(kv_len[t]), cap))
    ss = np.random.SeedSequence(seed).spawn(2 + 2 * n_seq)
    q = _gen(ss[0]).standard_normal((n_tok, n_heads, head_dim), dtype=np.float32)
    k = np.empty((n_seq, cap, n_kv_heads, head_dim), dtype=np.float16)
    v = np.empty_like(k)
    _fill_normal_f16(k, ss[2:2 + n_seq], per_seq)
    _fill_normal_f16(v, ss[2 + n_seq:], per_seq)
    scale = 1.0 / math.sqrt(head_dim) if scale is None else float(scale)
    return Case(name, q, kv_len, seq_of, scale, n_kv_heads, cap, "f16", k=k, v=v, seed=seed)


def make_q8_case(seed, n_tok, n_heads, n_kv_heads, head_dim, kv_len, budget=None,
                 cache_cap=None, seq_of=None, n_seq=None, scale=None, name="q8",
                 scale_group=64) -> Case:
    """Random int8-cache problem with one f16 scale per ``scale_group`` dims (64, or 32 as in
    FORWARD_MSL's q8 planes) and (if ``budget``) sorted ids."""
    if head_dim % 64 or scale_group not in (32, 64):
        raise ValueError("int8 caches need head_dim % 64 == 0 and groups of 32 or 64 dims")
    kv_len = np.asarray(kv_len, dtype=np.int32).reshape(n_tok)
    seq_of = (np.arange(n_tok, dtype=np.int32) if seq_of is None
              else np.asarray(seq_of, dtype=np.int32).reshape(n_tok))
    n_seq = int(seq_of.max()) + 1 if n_seq is None else n_seq
    cap = int(max(1, kv_len.max())) if cache_cap is None else int(cache_cap)
    per_seq = np.zeros(n_seq, dtype=np.int64)
    for t in range(n_tok):
        per_seq[seq_of[t]] = max(per_seq[seq_of[t]], min(int(kv_len[t]), cap))
    ss = np.random.SeedSequence(seed).spawn(3 + 2 * n_seq)
    q = _gen(ss[0]).standard_normal((n_tok, n_heads, head_dim), dtype=np.float32)
    shape = (n_seq, cap, n_kv_heads, head_dim)
    kq = np.empty(shape, dtype=np.int8)
    vq = np.empty(shape, dtype=np.int8)
    ksc = np.empty(shape[:3] + (head_dim // scale_group,), dtype=np.float16)
    vsc = np.empty_like(ksc)
    _fill_q8(kq, ksc, ss[3:3 + n_seq], per_seq)
    _fill_q8(vq, vsc, ss[3 + n_seq:], per_seq)
    ids = None
    if budget is not None:
        g = _gen(ss[1])
        ids = np.full((n_tok, budget), -1, dtype=np.int32)
        for t in range(n_tok):
            L = int(kv_len[t])
            if L <= budget:
                ids[t, :max(L, 0)] = np.arange(max(L, 0), dtype=np.int32)
            else:
                ids[t] = np.sort(g.choice(L, size=budget, replace=False)).astype(np.int32)
    scale = 1.0 / math.sqrt(head_dim) if scale is None else float(scale)
    return Case(name, q, kv_len, seq_of, scale, n_kv_heads, cap, "q8", kq=kq, vq=vq, ksc=ksc,
                vsc=vsc, ids=ids, budget=budget, seed=seed, scale_group=scale_group)


LLOYD_MAX_2BIT = (-1.5104, -0.4528, 0.4528, 1.5104)  # 2-bit Gaussian quantiser points


@dataclass
class TqCase:
    """A decode problem over a TurboQuant-compressed cache (host arrays)."""
    name: str
    q_rot: np.ndarray      # [T][H][D] fp32
    q_jl: np.ndarray       # [T][H][D] fp32
    k_polar: np.ndarray    # [n_seq][Hk][cap][D/16] uint32 (head-major, as on the page)
    k_jl: np.ndarray       # [n_seq][Hk][cap][D/32] uint32
    k_norms: np.ndarray    # [n_seq][Hk][cap] uint32: f16 norm | f16 residual norm << 16
    v_polar: np.ndarray    # [n_seq][Hk][cap][D/16] uint32
    v_norms: np.ndarray    # [n_seq][Hk][cap] uint32: f16 norm
    centroids: np.ndarray  # [4] fp32
    signs: np.ndarray      # [D] fp32, +-1
    qjl_scale: float
    scale: float
    kv_len: np.ndarray
    seq_of: np.ndarray
    seed: int = 0
    kind: str = "tq"
    ids = None
    budget = None
    meta: dict = field(default_factory=dict)

    @property
    def n_kv_heads(self):
        return self.k_polar.shape[1]

    @property
    def n_tok(self):
        return self.q_rot.shape[0]

    @property
    def n_heads(self):
        return self.q_rot.shape[1]

    @property
    def head_dim(self):
        return self.q_rot.shape[2]

    @property
    def n_seq(self):
        return self.k_polar.shape[0]

    @property
    def cache_cap(self):
        return self.k_polar.shape[2]

    def visited(self, t: int) -> int:
        return max(int(self.kv_len[t]), 0)

    def pos_bytes(self) -> int:
        """Packed bytes of one (position, KV head): K polar + sign words + norm pair, V polar +
        norm."""
        D = self.head_dim
        return 4 * (D // 16 + D // 32 + 1) + 4 * (D // 16 + 1)

    def kv_bytes(self) -> int:
        """Packed cache bytes the rows must read once per KV head (rows sharing a sequence
        need each position once)."""
        tot = 0
        for s in set(self.seq_of.tolist()):
            tot += max([self.visited(t) for t in range(self.n_tok) if self.seq_of[t] == s] + [0])
        return tot * self.n_kv_heads * self.pos_bytes()

    def algorithmic_bytes(self) -> int:
        """Packed cache + q_rot + q_jl + out (fp32) + signs."""
        return self.kv_bytes() + 3 * self.q_rot.size * 4 + self.head_dim * 4

    def flops(self) -> int:
        """6*D flops per (query head, visited position): q_rot.c, q_jl.s and p.v, 2*D each."""
        return sum(self.visited(t) for t in range(self.n_tok)) * self.n_heads * 6 * self.head_dim


def _half_bits(x) -> np.ndarray:
    return np.asarray(x, np.float16).view(np.uint16).astype(np.uint32)


def make_tq_case(seed, n_tok, n_heads, n_kv_heads, head_dim, kv_len, cache_cap=None,
                 seq_of=None, n_seq=None, scale=None, name="tq") -> TqCase:
    """Random TurboQuant problem: q_rot, q_jl N(0, 1); uniform random 2-bit indices and sign
    bits; K norms U[0.5, 2], residual norms U[0, 0.5], V norms U[0.5, 2] (f16); centroids the
    2-bit Gaussian Lloyd-Max points over sqrt(D); random +-1 signs; qjl_scale sqrt(pi/2) / D
    (the factor flash_attention_tq.metal's header gives).  Past a sequence's length the packed
    words are zero and the norm words hold f16 NaN.  Each sequence draws from its own stream."""
    D = head_dim
    if D % 32:
        raise ValueError("head_dim must be a multiple of 32")
    kv_len = np.asarray(kv_len, dtype=np.int32).reshape(n_tok)
    seq_of = (np.arange(n_tok, dtype=np.int32) if seq_of is None
              else np.asarray(seq_of, dtype=np.int32).reshape(n_tok))
    n_seq = int(seq_of.max()) + 1 if n_seq is None else n_seq
    cap = int(max(1, kv_len.max())) if cache_cap is None else int(cache_cap)
    g = _gen(np.random.SeedSequence(seed).spawn(1)[0])
    q_rot = g.standard_normal((n_tok, n_heads, D), dtype=np.float32)
    q_jl = g.standard_normal((n_tok, n_heads, D), dtype=np.float32)
    shp = (n_seq, n_kv_heads, cap)
    k_polar = np.zeros(shp + (D // 16,), np.uint32)
    k_jl = np.zeros(shp + (D // 32,), np.uint32)
    v_polar = np.zeros(shp + (D // 16,), np.uint32)
    k_norms = np.empty(shp, np.uint32)
    v_norms = np.empty(shp, np.uint32)
    seq_len = [max([int(kv_len[t]) for t in range(n_tok) if seq_of[t] == s] + [0])
               for s in range(n_seq)]
    streams = np.random.SeedSequence(seed).spawn(2 + n_seq)[2:]
    nan = int(_half_bits(np.float16(np.nan)))

    def halves(gs, n, lo, hi):  # f16 bit patterns of U[lo, hi) draws
        x = gs.random((n_kv_heads, n), dtype=np.float32) * np.float32(hi - lo) + np.float32(lo)
        return x.astype(np.float16).view(np.uint16).astype(np.uint32)

    def one(s):  # sequence s: random words and norms below its length, NaN norms past it
        L = seq_len[s]
        k_norms[s, :, L:] = nan | (nan << 16)
        v_norms[s, :, L:] = nan
        if L == 0:
            return
        gs = _gen(streams[s])
        for arr in (k_polar, k_jl, v_polar):
            arr[s, :, :L] = gs.integers(0, 0xFFFFFFFF, size=arr[s, :, :L].shape,
                                        dtype=np.uint32, endpoint=True)
        k_norms[s, :, :L] = halves(gs, L, 0.5, 2.0) | (halves(gs, L, 0.0, 0.5) << 16)
        v_norms[s, :, :L] = halves(gs, L, 0.5, 2.0)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(n_seq)))
    signs = np.where(g.integers(0, 2, D) == 1, 1.0, -1.0).astype(np.float32)
    cents = (np.array(LLOYD_MAX_2BIT) / math.sqrt(D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    return TqCase(name, q_rot, q_jl, k_polar, k_jl, k_norms, v_polar, v_norms, cents, signs,
                  float(math.sqrt(math.pi / 2) / D), scale, kv_len, seq_of, seed)


def make_block_scores(seed, n_tok, stride, levels=None) -> np.ndarray:
    """Block scores [n_tok][stride] fp32 for the top-k selection: N(0, 1), or (``levels``) drawn
    from that many distinct values so that equal scores cross the selection threshold."""
    g = _gen(np.random.SeedSequence(seed).spawn(1)[0])
    if levels is None:
        return g.standard_normal((n_tok, stride), dtype=np.float32)
    vals = np.linspace(-2.0, 2.0, levels, dtype=np.float32)
    return vals[g.integers(0, levels, size=(n_tok, stride))]


# ----------------------------------------------------------------------------- named workloads

def tiny() -> Case:
    """1 query token, 4 heads over 1 KV head, D=64, 256 positions, scale 1/8."""
    return make_f16_case(1001, 1, 4, 1, 64, [256], scale=1 / 8, name="tiny_h4_hk1_d64_L256")


def gqa_d64(seq_len: int) -> Case:
    """1 query token, 32 heads over 8 KV heads, D=64, seq_len 1024 or 4096, scale 1/8."""
    return make_f16_case(1002, 1, 32, 8, 64, [seq_len], scale=1 / 8,
                         name=f"gqa_h32_hk8_d64_L{seq_len}")


def long_context_lengths(seed=1003, n=16, lo=1024, hi=32768) -> np.ndarray:
    return _gen(np.random.SeedSequence(seed).spawn(1)[0]).integers(lo, hi + 1, size=n).astype(np.int32)


def long_context() -> Case:
    """16 sequences, lengths uniform in [1024, 32768], 32 heads / 8 KV heads, D=128, cap 32768."""
    L = long_context_lengths()
    return make_f16_case(1003, 16, 32, 8, 128, L, cache_cap=32768, scale=1 / math.sqrt(128),
                         name="long_ctx_b16_U1024-32768_h32_hk8_d128")


def long_context_full() -> Case:
    """The long-context shape with every sequence at the full 32768 positions (16 x 32768,
    32 heads / 8 KV heads, D=128): the fixed-length sub-case of the long-context workload."""
    return make_f16_case(1011, 16, 32, 8, 128, [32768] * 16, cache_cap=32768,
                         scale=1 / math.sqrt(128), name="long_ctx_full_b16_L32768_h32_hk8_d128")


def long_context_4() -> Case:
    """The long-context shape with 4 sequences (a smaller case for profiler captures)."""
    L = long_context_lengths(seed=1007, n=4)
    return make_f16_case(1007, 4, 32, 8, 128, L, cache_cap=32768, scale=1 / math.sqrt(128),
                         name="long_ctx_b4_U1024-32768_h32_hk8_d128")


def q8_selected() -> Case:
    """int8 KV, 4 KV heads x 12 = 48 heads, D=256, context 8192, 1024 sorted ids, scale 1/16."""
    return make_q8_case(1004, 1, 48, 4, 256, [8192], budget=1024, scale=1 / 16,
                        name="q8_sel_h48_hk4_d256_ctx8192_b1024")


def q8_topk_selected() -> Case:
    """q8_selected with its ids chosen on the GPU from block scores: the 2049 block scores of the
    8192-cell context (N(0, 1), seed 1008) go through the top-1024 selection first."""
    c = q8_selected()
    c.name = "q8_topk_sel_h48_hk4_d256_ctx8192_b1024"
    c.meta["block_scores"] = make_block_scores(1008, c.n_tok, 8192 // 4 + 1)
    return c


def batched() -> Case:
    """64 sequences of 8192 positions, 32 heads / 8 KV heads, D=128."""
    return make_f16_case(1005, 64, 32, 8, 128, [8192] * 64, scale=1 / math.sqrt(128),
                         name="batched_b64_L8192_h32_hk8_d128")


def prefill_chunk(start_pos=8176, n_rows=16) -> Case:
    """16 causal rows at positions start_pos..start_pos+15 of one sequence (row r sees
    start_pos + r + 1 positions), 32 heads / 8 KV heads, D=128, cap start_pos + n_rows."""
    L = [start_pos + r + 1 for r in range(n_rows)]
    return make_f16_case(1006, n_rows, 32, 8, 128, L, cache_cap=start_pos + n_rows,
                         seq_of=[0] * n_rows, n_seq=1, scale=1 / math.sqrt(128),
                         name=f"prefill_chunk_r{n_rows}_pos{start_pos}_h32_hk8_d128")


def tq_long_context() -> TqCase:
    """The long-context shape over a TurboQuant-compressed cache: 16 sequences, lengths uniform
    in [1024, 32768], 32 heads / 8 KV heads, D=128, cap 32768."""
    return make_tq_case(1009, 16, 32, 8, 128, long_context_lengths(), cache_cap=32768,
                        name="tq_long_ctx_b16_h32_hk8_d128_cap32768")


def tq_prefill_chunk(start_pos=8176, n_rows=16) -> TqCase:
    """Chunked prefill over a TurboQuant cache: 16 causal rows of one sequence (row r sees
    start_pos + r + 1 positions), 32 heads / 8 KV heads, D=128."""
    L = [start_pos + r + 1 for r in range(n_rows)]
    return make_tq_case(1010, n_rows, 32, 8, 128, L, cache_cap=start_pos + n_rows,
                        seq_of=[0] * n_rows, n_seq=1,
                        name=f"tq_prefill_chunk_r{n_rows}_pos{start_pos}_h32_hk8_d128")


NAMED = {
    "tiny": tiny,
    "gqa_d64_L1024": lambda: gqa_d64(1024),
    "gqa_d64_L4096": lambda: gqa_d64(4096),
    "long_ctx": long_context,
    "long_ctx_4": long_context_4,
    "long_ctx_full": long_context_full,
    "q8_sel": q8_selected,
    "q8_topk_sel": q8_topk_selected,
    "batched": batched,
    "prefill_chunk": prefill_chunk,
    "tq_long_ctx": tq_long_context,
    "tq_prefill_chunk": tq_prefill_chunk,
}
