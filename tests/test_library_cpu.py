"""CPU checks of the C-ABI library: it loads, exports what the header declares, and its host
logic (planner, argument checks) behaves, all without launching anything."""

import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "gqa_decode.h"


@pytest.fixture(scope="module")
def gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))
                  - {"if", "defined"})


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("attn_decode_f16", "attn_decode_q8_sel", "attn_merge", "attn_decode_plan",
              "attn_decode_workspace_bytes", "gqa_status_string", "gqa_last_error",
              "gqa_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(gd):
    lib = ctypes.CDLL(str(gd._LIB_PATH))
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
    assert set(declared_functions()) <= set(gd.EXPORTS) | set(declared_functions())
    assert gd.LIB.gqa_abi_version() == 9
    assert set(gd.EXPORTS) == set(declared_functions())


def test_status_strings(gd):
    assert gd.LIB.gqa_status_string(0) == b"GQA_OK"
    assert gd.LIB.gqa_status_string(2) == b"GQA_EWORKSPACE"
    assert gd.LIB.gqa_status_string(99) == b"GQA_UNKNOWN"


def test_plan_long_context_stream_k(gd, monkeypatch):
    # opt-in stream-K: 16 rows x 8 KV heads up to 32768 positions, f16, D=128, on 152 SMs:
    # two CTAs per SM, each an equal share of the (row, KV head, position) stream
    monkeypatch.setenv("GQA_F16_SPLIT", "streamk")
    p = gd.plan(16, 32, 8, 128, 32768, -1, gd.KIND_F16, num_sms=152)
    assert p.streamk == 1 and p.merge == 1 and p.tile == 64
    assert (p.grid_x, p.grid_y, p.grid_z) == (304, 1, 1) and p.n_split == 304
    counters = -(-16 * 8 * 4 // 256) * 256
    records = (304 + 16 * 8) * 4 * 130 * 4   # (CTAs + segments) x G=4 x (D+2) floats
    assert p.ws_bytes == counters + records
    q = gd.plan(1, 4, 1, 64, 100, -1, gd.KIND_F16, num_sms=152)
    assert q.streamk == 1 and q.grid_x == 1


def test_plan_long_context_chunked(gd, monkeypatch):
    # the default: chunks of min(8192, one wave of 2 CTAs per SM at max length) positions, and
    # at most 4096 for rows longer than 8192
    p = gd.plan(16, 32, 8, 128, 32768, -1, gd.KIND_F16, num_sms=152)
    assert p.streamk == 0 and p.tile == 64 and p.chunk == 4096
    assert p.n_split == 8 and p.merge == 1
    assert (p.grid_x, p.grid_y, p.grid_z) == (8, 8, 16)
    # rows of at most 8192 keep chunks of up to 8192 (64 x 8192: one chunk a row)
    b = gd.plan(64, 32, 8, 128, 8192, -1, gd.KIND_F16, num_sms=152)
    assert b.chunk == 8192 and b.n_split == 1 and b.merge == 0
    part = 16 * 8 * 32 * 130 * 4
    counters = -(-16 * 8 * 4 // 256) * 256          # per-(row, KV head) arrival counters
    assert p.ws_bytes == counters + -(-part // 256) * 256 + 16 * 4
    # a grid that fits the GPU merges each row inside a cluster of its chunk CTAs: 8 chunks
    # a row (1 row x 8 KV heads x 4096 positions, D=64: 64 CTAs)
    q = gd.plan(1, 32, 8, 64, 4096, -1, gd.KIND_F16, num_sms=152)
    assert q.chunk == 512 and q.n_split == 8
    # ... down to one 128-position stage a chunk (1024 positions)
    q = gd.plan(1, 32, 8, 64, 1024, -1, gd.KIND_F16, num_sms=152)
    assert q.chunk == 128 and q.n_split == 8
    r = gd.plan(1, 4, 1, 64, 100, -1, gd.KIND_F16, num_sms=152)
    assert r.n_split == 1 and r.merge == 0 and r.ws_bytes == 0 and r.chunk == 128
    # without the cluster merge: chunks of at least two 128-position stages
    monkeypatch.setenv("GQA_F16_CLUSTER", "0")
    q = gd.plan(1, 32, 8, 64, 4096, -1, gd.KIND_F16, num_sms=152)
    assert q.chunk == 256 and q.n_split == 16
    # a grid past the SM count keeps the rule: 8 rows x 8 KV heads x 5 chunks of 896
    off = gd.plan(8, 32, 8, 64, 4096, -1, gd.KIND_F16, num_sms=152)
    monkeypatch.delenv("GQA_F16_CLUSTER")
    on = gd.plan(8, 32, 8, 64, 4096, -1, gd.KIND_F16, num_sms=152)
    assert (on.chunk, on.n_split) == (off.chunk, off.n_split) == (896, 5)


def test_plan_selected_width_caps_chunks(gd):
    # int8 + 1024 ids over a context of 8192: the visited list is 1024 long (chunked mode);
    # the grid (8 chunks x 4 KV heads) is far below 152 SMs, so the tensor-core kernel's 12
    # query heads of a KV head spread over 3 CTAs of 4 heads each (96 CTAs)
    p = gd.plan(1, 48, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152)
    assert p.streamk == 0 and p.tile == 64 and p.n_split == -(-1024 // p.chunk)
    assert p.grid_y == 4 * 3 and p.chunk == 128


def test_plan_q8_head_split(gd, monkeypatch):
    # a grid that fills the GPU keeps the default of up to 8 heads a CTA (12 -> 2 x 6)
    p = gd.plan(64, 48, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152)
    assert p.grid_y == 4 * 2 and p.grid_z == 64
    # a small grid splits further while it still fits on the SMs, never below 4 heads a CTA:
    # 16 heads -> 4 CTAs of 4 (8 chunks x 4 KV heads x 4 = 128 CTAs)
    q = gd.plan(1, 64, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152)
    assert q.grid_y == 4 * 4 and q.n_split == 8
    # ... but not past the SM count: on 64 SMs, 8 x 4 x 2 = 64 CTAs
    assert gd.plan(1, 64, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=64).grid_y == 4 * 2
    # 4 heads a KV head: nothing to split
    assert gd.plan(1, 16, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152).grid_y == 4
    # a forced split wins; the CUDA-core kernel keeps its 4 heads a CTA
    monkeypatch.setenv("GQA_HEAD_SPLIT", "1")
    assert gd.plan(1, 48, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152).grid_y == 4
    monkeypatch.delenv("GQA_HEAD_SPLIT")
    monkeypatch.setenv("GQA_Q8_KERNEL", "fma")
    assert gd.plan(64, 48, 4, 256, 8192, 1024, gd.KIND_Q8, num_sms=152).grid_y == 4 * 3


def test_plan_groups_rows_sharing_a_sequence(gd, monkeypatch):
    # 16 causal rows over one sequence (n_seq 1), G=4: one group of up to 16 rows (64 (row,
    # head) pairs, each twice in the tcgen05 MMA's 128 rows); chunks of 64-position tiles sized
    # for 1 group x 8 KV heads on one CTA per SM: 8 * 8192 / 152 -> 432 -> 448 positions
    p = gd.plan(16, 32, 8, 128, 8192, -1, gd.KIND_F16, num_sms=152, n_seq=1)
    assert p.row_group == 16 and p.chunk == 448 and p.n_split == 19 and p.tile == 64
    assert (p.grid_x, p.grid_y, p.grid_z) == (19, 8, 1)   # one group slot
    # 64 rows of 32 sequences (pairs): 32 slots
    q = gd.plan(64, 32, 8, 128, 8192, -1, gd.KIND_F16, num_sms=152, n_seq=32)
    assert q.row_group == 16 and q.grid_z == 32
    # D=64 keeps the 64-position tile on the tcgen05 row kernel
    assert gd.plan(16, 32, 8, 64, 8192, -1, gd.KIND_F16, num_sms=152, n_seq=1).tile == 64
    # the mma.sync row kernel: two groups of 8 rows (2 sets of 16 pairs) on two CTAs per SM:
    # 16 * 8192 / 304 -> 432 -> 448 positions
    monkeypatch.setenv("GQA_F16_ROWS", "mma")
    m = gd.plan(16, 32, 8, 128, 8192, -1, gd.KIND_F16, num_sms=152, n_seq=1)
    assert m.row_group == 8 and m.chunk == 448 and m.n_split == 19
    assert (m.grid_x, m.grid_y, m.grid_z) == (19, 8, 2)   # two group slots
    assert gd.plan(64, 32, 8, 128, 8192, -1, gd.KIND_F16, num_sms=152, n_seq=32).row_group == 8
    monkeypatch.delenv("GQA_F16_ROWS")
    # every row its own sequence, D=256, int8, or group size 3: no grouping
    assert gd.plan(16, 32, 8, 128, 8192, num_sms=152).row_group == 1
    assert gd.plan(16, 32, 8, 256, 8192, num_sms=152, n_seq=1).row_group == 1
    assert gd.plan(16, 48, 4, 128, 8192, 64, gd.KIND_Q8, num_sms=152, n_seq=1).row_group == 1
    assert gd.plan(16, 24, 8, 128, 8192, num_sms=152, n_seq=1).row_group == 1


def test_plan_small_rows_are_not_split(gd):
    # 256 positions of f16 D=64 are 64 KB of K/V: below the 128 KB split threshold
    p = gd.plan(1, 4, 1, 64, 256, -1, gd.KIND_F16, num_sms=152)
    assert p.n_split == 1 and p.merge == 0
    q = gd.plan(1, 4, 1, 64, 513, -1, gd.KIND_F16, num_sms=152)   # 131 328 bytes: split
    assert q.n_split > 1


def test_plan_rejects_bad_shapes(gd):
    with pytest.raises(gd.GqaError, match="EINVAL"):
        gd.plan(1, 32, 8, 96, 10, num_sms=152)             # head_dim
    with pytest.raises(gd.GqaError, match="EINVAL"):
        gd.plan(1, 30, 8, 64, 10, num_sms=152)             # heads not a multiple
    with pytest.raises(gd.GqaError, match="EUNSUPPORTED"):
        gd.plan(1, 34, 2, 64, 10, num_sms=152)             # group 17
    with pytest.raises(gd.GqaError, match="EINVAL"):
        gd.plan(1, 4, 1, 64, 10, 0, gd.KIND_Q8, num_sms=152)  # budget 0
    with pytest.raises(gd.GqaError, match="EINVAL"):
        gd.plan(1, 4, 1, 64, -1, num_sms=152)              # negative length


def test_decode_rejects_bad_arguments_before_any_launch(gd):
    L = gd.LIB
    P = ctypes.c_void_p
    good = P(1 << 20)
    # NULL q
    st = L.attn_decode_f16(None, good, good, good, good, None, 1, 1, 4, 1, 64, 16, 16, 0.1, None,
                           0, None, None)
    assert st == gd.GQA_EINVAL and b"NULL" in L.gqa_last_error()
    # misaligned cache
    st = L.attn_decode_f16(good, P((1 << 20) + 2), good, good, good, None, 1, 1, 4, 1, 64, 16,
                           16, 0.1, None, 0, None, None)
    assert st == gd.GQA_EINVAL and b"aligned" in L.gqa_last_error()
    # non-finite scale
    st = L.attn_decode_f16(good, good, good, good, good, None, 1, 1, 4, 1, 64, 16, 16,
                           float("inf"), None, 0, None, None)
    assert st == gd.GQA_EINVAL
    # seq_of NULL with fewer sequences than rows
    st = L.attn_decode_f16(good, good, good, good, good, None, 2, 1, 4, 1, 64, 16, 16, 0.1, None,
                           0, None, None)
    assert st == gd.GQA_EINVAL
    # ids without a budget
    st = L.attn_decode_q8_sel(good, good, good, good, good, good, 0, good, good, None, 1, 1, 4, 1,
                              64, 16, 16, 0.1, None, 0, None, None)
    assert st == gd.GQA_EINVAL
    # n_tok == 0 is a no-op
    st = L.attn_decode_f16(None, None, None, None, None, None, 0, 1, 4, 1, 64, 16, 16, 0.1, None,
                           0, None, None)
    assert st == gd.GQA_OK
    # merge: bad head_dim
    assert L.attn_merge(good, good, 2, 1, 4, 100, good, None) == gd.GQA_EINVAL


def test_plan_turboquant(gd):
    # TurboQuant cache, D=128: 88 bytes per (position, KV head); 8 KV heads over 32768
    # positions split into chunks of whole 128-position passes, merged by the last CTA
    p = gd.plan(1, 32, 8, 128, 32768, -1, gd.KIND_TQ, num_sms=152)
    assert p.tile == 128 and p.streamk == 0 and p.row_group == 1
    assert p.grid_y == 8 and p.grid_z == 1 and p.chunk % 128 == 0
    assert p.n_split == -(-32768 // p.chunk) and p.merge == 1
    # compute-sized chunks for 8 CTAs per SM: one row of 8 KV heads -> 8 x 32768 / 1216 -> 256
    assert p.chunk == 256 and p.n_split == 128
    # ... and at most 1792 positions
    r = gd.plan(16, 32, 8, 128, 32768, -1, gd.KIND_TQ, num_sms=152)
    assert r.chunk == 1792 and (r.grid_x, r.grid_y, r.grid_z) == (19, 8, 16)
    # a row of at most 32 KB (372 positions of 88 bytes) is not split
    q = gd.plan(1, 32, 8, 128, 372, -1, gd.KIND_TQ, num_sms=152)
    assert q.n_split == 1 and q.merge == 0 and q.ws_bytes == 0
    q = gd.plan(1, 32, 8, 128, 373, -1, gd.KIND_TQ, num_sms=152)
    assert q.n_split == 2 and q.chunk == 256


def test_plan_groups_turboquant_rows(gd, monkeypatch):
    # 16 causal rows over one TurboQuant sequence, G=4: one group of 16 rows (64 pairs), chunks
    # of 32-position stages for 8 KV heads on one CTA per SM: 8 * 8192 / 152 -> 432 -> 448
    monkeypatch.delenv("GQA_TQ_KERNEL", raising=False)
    monkeypatch.delenv("GQA_TQ_ROWS", raising=False)
    p = gd.plan(16, 32, 8, 128, 8192, -1, gd.KIND_TQ, num_sms=152, n_seq=1)
    assert p.row_group == 16 and p.tile == 32 and p.chunk == 448 and p.n_split == 19
    assert (p.grid_x, p.grid_y, p.grid_z) == (19, 8, 1)
    # 12 heads per KV head: two CTAs of 6 heads, 10 rows a group
    q = gd.plan(16, 48, 4, 128, 8192, -1, gd.KIND_TQ, num_sms=152, n_seq=1)
    assert q.row_group == 10 and q.grid_y == 8
    # head_dim 32, the CUDA-core kernel, or grouping switched off: one CTA per row
    assert gd.plan(16, 32, 8, 32, 8192, -1, gd.KIND_TQ, num_sms=152, n_seq=1).row_group == 1
    monkeypatch.setenv("GQA_TQ_ROWS", "off")
    assert gd.plan(16, 32, 8, 128, 8192, -1, gd.KIND_TQ, num_sms=152, n_seq=1).row_group == 1


def test_turboquant_argument_checks(gd):
    # rejected on the host before any device call
    cents = (ctypes.c_float * 4)(0.0, 0.0, 0.0, 0.0)
    def call(head_dim=128, n_heads=32, n_kv_heads=8, ptr=16):
        P = ctypes.c_void_p(ptr)
        return gd.LIB.attn_decode_tq(P, P, P, P, P, P, P, cents, P, 1.0, 1.0, P, P, None, 1, 1,
                                     n_heads, n_kv_heads, head_dim, 64, 64, None, 0, None, None)
    assert call(head_dim=256) == gd.GQA_EINVAL
    assert call(n_heads=30) == gd.GQA_EINVAL
    assert call(n_heads=136, n_kv_heads=8) == gd.GQA_EUNSUPPORTED  # group of 17
    assert call(ptr=0) == gd.GQA_EINVAL
    assert call(ptr=8) == gd.GQA_EINVAL                           # caches 16-byte aligned
