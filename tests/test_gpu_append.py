"""GPU parity of quantise-on-append (kv_append_q8): bit-exact int8 codes and f16 scales against
the oracle, and the int8 decode path over a cache written by it."""

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


@pytest.mark.parametrize("group", [64, 32])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_codes_bit_exact(D, group):
    rng = np.random.default_rng(D)
    n_seq, cap, Hk, n_new, seq, t0 = 3, 40, 2, 17, 1, 9
    # magnitudes over many decades, exact halves of a step, an all-zero group
    x = (rng.standard_normal((2, n_new, Hk, D)) * 10.0 ** rng.uniform(-3, 3, (2, n_new, Hk, 1)))
    x = x.astype(np.float32)
    x[0, 3, 1, :group] = 0.0
    x[1, 5, 0, :4] = [127.0, 2.5, 3.5, -2.5]
    x[1, 5, 0, 4:group] = 0.0
    kq = torch.full((n_seq, cap, Hk, D), 99, dtype=torch.int8, device="cuda")
    vq = kq.clone()
    ksc = torch.full((n_seq, cap, Hk, D // group), 7.0, dtype=torch.float16, device="cuda")
    vsc = ksc.clone()
    _gd().kv_append_q8(dev(x[0]), dev(x[1]), kq, vq, ksc, vsc, seq, t0)
    for side, (q, s) in enumerate(((kq, ksc), (vq, vsc))):
        rq, rs = oracle.quantize_q8(x[side], group)
        q, s = q.cpu().numpy(), s.cpu().numpy()
        assert np.array_equal(q[seq, t0:t0 + n_new], rq)
        assert np.array_equal(s[seq, t0:t0 + n_new].view(np.uint16), rs.view(np.uint16))
        # nothing else touched
        mask = np.ones((n_seq, cap), bool)
        mask[seq, t0:t0 + n_new] = False
        assert (q[mask] == 99).all() and (s[mask] == 7.0).all()


@pytest.mark.parametrize("group", [64, 32])
def test_append_then_decode(group):
    """fp32 K/V -> kv_append_q8 -> attn_decode_q8_sel (selected ids) against the oracle on the
    oracle-quantised cache: 12 heads over 2 KV heads, D=256, 700 positions, budget 300; scale
    groups of 64 dims and FORWARD_MSL's 32-element blocks."""
    rng = np.random.default_rng(77)
    Hk, D, L, budget = 2, 256, 700, 300
    case = W.make_q8_case(720, 1, 24, Hk, D, [L], budget=budget, cache_cap=L, scale=1 / 16,
                          scale_group=group)
    k32 = rng.standard_normal((L, Hk, D)).astype(np.float32)
    v32 = rng.standard_normal((L, Hk, D)).astype(np.float32)
    kq, ksc = oracle.quantize_q8(k32, group)
    vq, vsc = oracle.quantize_q8(v32, group)
    case.kq[0], case.vq[0], case.ksc[0], case.vsc[0] = kq, vq, ksc, vsc
    gd = _gd()
    kq_d = torch.zeros((1, L, Hk, D), dtype=torch.int8, device="cuda")
    vq_d = torch.zeros_like(kq_d)
    ksc_d = torch.zeros((1, L, Hk, D // group), dtype=torch.float16, device="cuda")
    vsc_d = torch.zeros_like(ksc_d)
    for t0 in range(0, L, 256):  # appended in pieces, as a decode loop would
        n = min(256, L - t0)
        gd.kv_append_q8(dev(k32[t0:t0 + n]), dev(v32[t0:t0 + n]), kq_d, vq_d, ksc_d, vsc_d, 0, t0)
    got = gd.attn_decode_q8_sel(dev(case.q), kq_d, vq_d, ksc_d, vsc_d, dev(case.kv_len),
                                ids=dev(case.ids), scale=case.scale).cpu().numpy()
    assert_close(got, oracle_ref(case), TOL_Q8, "append -> q8_sel")
