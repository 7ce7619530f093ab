"""The decode calls inside CUDA graphs, as a serving loop replays them: captured once with a
caller-owned workspace, replayed several times, each replay bit-identical to the eager call
(the split merge's arrival counters return to zero every call, so replays need no reset)."""

import numpy as np
import pytest
import torch

from gpu_util import dev, forced_chunk
from gqa_decode_attention_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gd():
    from gqa_decode_attention_03_gb300 import gqa_decode
    return gqa_decode


def _graph_equals_eager(fn, out):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # eager, on the capture stream (warms attributes and caches)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    return ref


@pytest.mark.parametrize("rows_share", [False, True])
def test_f16_split_in_a_graph(rows_share):
    gd = _gd()
    if rows_share:  # causal rows of one sequence: row-grouped kernel + merge kernel
        L = [3000 + r for r in range(8)]
        c = W.make_f16_case(901, 8, 16, 4, 128, L, cache_cap=3008, seq_of=[0] * 8, n_seq=1,
                            scale=0.088)
    else:
        c = W.make_f16_case(902, 4, 16, 4, 128, [5000, 17, 4096, 2500], cache_cap=5000,
                            scale=0.088)
    q, k, v, kv, so = dev(c.q), dev(c.k), dev(c.v), dev(c.kv_len), dev(c.seq_of)
    out = torch.empty_like(q)
    with forced_chunk(512):
        ws = gd.alloc_workspace(c.n_tok, c.n_heads, c.n_kv_heads, 128, c.cache_cap,
                                n_seq=c.n_seq, device="cuda")

        def call():
            gd.attn_decode_f16(q, k, v, kv, scale=c.scale, seq_of=so, out=out, ws=ws)

        assert gd.plan(c.n_tok, c.n_heads, c.n_kv_heads, 128, c.cache_cap,
                       n_seq=c.n_seq).merge == 1
        _graph_equals_eager(call, out)


def test_q8_selected_in_a_graph():
    gd = _gd()
    c = W.make_q8_case(903, 2, 24, 2, 256, [3000, 900], budget=512, cache_cap=3000, scale=1 / 16)
    q, kq, vq, ksc, vsc = dev(c.q), dev(c.kq), dev(c.vq), dev(c.ksc), dev(c.vsc)
    kv, ids = dev(c.kv_len), dev(c.ids)
    out = torch.empty_like(q)
    ws = gd.alloc_workspace(2, 24, 2, 256, 3000, 512, gd.KIND_Q8, "cuda")

    def call():
        gd.attn_decode_q8_sel(q, kq, vq, ksc, vsc, kv, ids=ids, scale=c.scale, out=out, ws=ws)

    _graph_equals_eager(call, out)


def test_turboquant_in_a_graph():
    gd = _gd()
    c = W.make_tq_case(904, 3, 32, 8, 128, [4000, 50, 2048], cache_cap=4000)
    i32 = lambda a: dev(np.ascontiguousarray(a).view(np.int32))  # noqa: E731
    args = (dev(c.q_rot), dev(c.q_jl), i32(c.k_polar), i32(c.k_jl), i32(c.k_norms),
            i32(c.v_polar), i32(c.v_norms), c.centroids, dev(c.signs), c.qjl_scale, dev(c.kv_len))
    out = torch.empty_like(args[0])
    ws = gd.alloc_workspace(3, 32, 8, 128, 4000, -1, gd.KIND_TQ, "cuda", 3)

    def call():
        gd.attn_decode_tq(*args, scale=c.scale, out=out, ws=ws)

    _graph_equals_eager(call, out)
