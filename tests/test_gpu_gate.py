"""GPU parity of the gated decode calls (attn_decode_f16_gated, attn_decode_q8_sel_gated,
attn_decode_tq_gated) against the oracle's decode composed with its sigmoid output gate.

The gate multiplies every output element after the merge (qsa2.metal qsa_merge2, FORWARD_MSL
attn_combine).  Each kernel that writes output rows applies it: the single-chunk epilogues, the
last-CTA merge, the stream-K merge, both row kernels, the in-kernel merge of the tcgen05 row
kernel, merge_kernel after grouped rows, and the TurboQuant finish (after the inverse
rotation).  Every path is run with a plain [T][H][D] gate (stride D) and with the pages'
per-head [query | gate] pairs (stride 2 D).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TOL_F16, TOL_Q8, _env, assert_close, dev, f16_kernel, forced_chunk,
                      oracle_ref)
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def _gate(seed, T, H, D, layout):
    """(device gate tensor, stride, host gate [T][H][D]): N(0, 2) values; in the pair layout the
    gate is the second half of each head's [query | gate] vector of 2 D floats."""
    g = np.random.default_rng(seed).standard_normal((T, H, D)).astype(np.float32) * 2
    if layout == "plain":
        return dev(g), D, g
    pair = np.random.default_rng(seed + 1).standard_normal((T, H, 2 * D)).astype(np.float32)
    pair[:, :, D:] = g
    flat = dev(pair.reshape(-1))
    return flat[D:], 2 * D, g


def _f16(case, gate, gs, so=None, err=None):
    return _gd().attn_decode_f16(dev(case.q), dev(case.k), dev(case.v), dev(case.kv_len),
                                 scale=case.scale, seq_of=so, err=err, gate=gate,
                                 gate_stride=gs)


LAYOUTS = ["plain", "pair"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("path", ["unsplit", "split", "streamk", "fma"])
def test_f16_per_row_gated(path, layout):
    case = W.make_f16_case(1201, 3, 16, 4, 128, [3000, 37, 1700], cache_cap=3000, scale=0.09)
    gate, gs, g = _gate(1202, 3, 16, 128, layout)
    env = {"unsplit": (f16_kernel("chunked"), forced_chunk(3072)),
           "split": (f16_kernel("chunked"), forced_chunk(256)),
           "streamk": (f16_kernel("streamk"), forced_chunk(None)),
           "fma": (f16_kernel("fma"), forced_chunk(256))}[path]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with env[0], env[1]:
        got = _f16(case, gate, gs, err=err).cpu().numpy()
    assert int(err.item()) == 0
    assert_close(got, oracle.output_gate(oracle_ref(case), g), TOL_F16, f"f16 {path} {layout}")


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("path", ["umma_fused", "umma_merge_kernel", "mma_merge_kernel",
                                  "umma_unsplit"])
def test_f16_grouped_rows_gated(path, layout):
    L = [1500 + 11 * r for r in range(16)] + [0, 40]
    case = W.make_f16_case(1203, 18, 32, 8, 128, L, cache_cap=1700, seq_of=[0] * 16 + [1, 1],
                           n_seq=2, scale=1 / math.sqrt(128))
    gate, gs, g = _gate(1204, 18, 32, 128, layout)
    kern, chunk = {"umma_fused": ("chunked", None), "umma_merge_kernel": ("chunked", 64),
                   "mma_merge_kernel": ("rows_mma", 128), "umma_unsplit": ("chunked", 1728)}[path]
    gd = _gd()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with f16_kernel(kern), forced_chunk(chunk):
        plan = gd.plan(18, 32, 8, 128, 1700, n_seq=2)
        assert plan.row_group > 1
        ctas = plan.grid_x * plan.grid_y * plan.grid_z
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        if path == "umma_fused":
            assert plan.merge and ctas <= sms
        elif path == "umma_merge_kernel":
            assert plan.merge and ctas > sms
        elif path == "umma_unsplit":
            assert not plan.merge
        got = _f16(case, gate, gs, so=dev(case.seq_of), err=err).cpu().numpy()
    assert int(err.item()) == 0
    ref = oracle.output_gate(oracle_ref(case), g)
    assert_close(got, ref, TOL_F16, f"grouped {path} {layout}")
    assert (got[16] == 0).all()  # an empty row stays zero


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("chunk", [None, 128])
def test_q8_selected_gated(chunk, layout):
    case = W.make_q8_case(1205, 2, 24, 2, 256, [2000, 300], budget=512, scale=1 / 16)
    gate, gs, g = _gate(1206, 2, 24, 256, layout)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with forced_chunk(chunk):
        got = _gd().attn_decode_q8_sel(dev(case.q), dev(case.kq), dev(case.vq), dev(case.ksc),
                                       dev(case.vsc), dev(case.kv_len), ids=dev(case.ids),
                                       scale=case.scale, err=err, gate=gate,
                                       gate_stride=gs).cpu().numpy()
    assert int(err.item()) == 0
    assert_close(got, oracle.output_gate(oracle_ref(case), g), TOL_Q8, f"q8 {chunk} {layout}")


def _i32(a):
    return dev(np.ascontiguousarray(a).view(np.int32))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("kernel", ["mma", "fma"])
@pytest.mark.parametrize("chunk", [None, 128])
def test_tq_gated(kernel, chunk, layout):
    c = W.make_tq_case(1207, 3, 16, 4, 128, [2500, 0, 700], cache_cap=2500)
    gate, gs, g = _gate(1208, 3, 16, 128, layout)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _env(GQA_TQ_KERNEL="fma" if kernel == "fma" else None), forced_chunk(chunk):
        got = _gd().attn_decode_tq(dev(c.q_rot), dev(c.q_jl), _i32(c.k_polar), _i32(c.k_jl),
                                   _i32(c.k_norms), _i32(c.v_polar), _i32(c.v_norms), c.centroids,
                                   dev(c.signs), c.qjl_scale, dev(c.kv_len), scale=c.scale,
                                   err=err, gate=gate, gate_stride=gs).cpu().numpy()
    assert int(err.item()) == 0
    ref = oracle.decode_tq(c.q_rot, c.q_jl, c.k_polar, c.k_jl, c.k_norms, c.v_polar, c.v_norms,
                           c.centroids, c.signs, c.qjl_scale, c.scale, c.kv_len, c.seq_of)
    assert_close(got, oracle.output_gate(ref, g), 1e-4, f"tq {kernel} {chunk} {layout}")
    assert (got[1] == 0).all()


def test_gate_arguments_are_checked():
    gd = _gd()
    case = W.make_f16_case(1209, 1, 4, 1, 64, [10])
    q, k, kv = dev(case.q), dev(case.k), dev(case.kv_len)
    out = torch.empty_like(q)
    g = torch.zeros(4 * 64, dtype=torch.float32, device="cuda")
    st = gd.LIB.attn_decode_f16_gated(gd._ptr(q), gd._ptr(k), gd._ptr(k), gd._ptr(out),
                                      gd._ptr(kv), None, 1, 1, 4, 1, 64, 10, 10, 0.1, gd._ptr(g),
                                      32, None, 0, None, gd._stream(None))
    assert st == gd.GQA_EINVAL  # stride below head_dim
    st = gd.LIB.attn_decode_f16_gated(gd._ptr(q), gd._ptr(k), gd._ptr(k), gd._ptr(out),
                                      gd._ptr(kv), None, 1, 1, 4, 1, 64, 10, 10, 0.1, None, 64,
                                      None, 0, None, gd._stream(None))
    assert st == gd.GQA_EINVAL  # no gate
