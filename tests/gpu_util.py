"""Helpers shared by the GPU parity tests: move a workloads.Case to the device, run the CUDA
path through the C ABI, and compare against the oracle with the stated tolerance."""

import os
from contextlib import contextmanager

import numpy as np
import torch

import pins

TOL_F16 = 2e-3   # f16 KV: |gpu - ref| <= tol * max(1, |ref|)
TOL_Q8 = 1e-4    # int8 KV (dequantised identically on both sides)


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


@contextmanager
def forced_chunk(n):
    """Runs the block with the planner's chunk length forced (None: planner's own choice)."""
    old = os.environ.get("GQA_FORCE_CHUNK")
    if n is not None:
        os.environ["GQA_FORCE_CHUNK"] = str(n)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("GQA_FORCE_CHUNK", None)
        else:
            os.environ["GQA_FORCE_CHUNK"] = old


@contextmanager
def _env(**kw):
    old = {k: os.environ.get(k) for k in kw}
    for k, v in kw.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = str(v)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@contextmanager
def f16_kernel(name):
    """Runs the block with the f16 path on one kernel: "chunked" (tensor cores, chunked grid:
    the default; grouped rows on the tcgen05 kernel), "rows_mma" (the same with grouped rows on
    the mma.sync kernel), "streamk" (tensor cores, stream-K split) or "fma" (CUDA cores,
    chunked)."""
    env = {"streamk": dict(GQA_F16_KERNEL=None, GQA_F16_SPLIT="streamk", GQA_F16_ROWS=None),
           "chunked": dict(GQA_F16_KERNEL=None, GQA_F16_SPLIT=None, GQA_F16_ROWS=None),
           "rows_mma": dict(GQA_F16_KERNEL=None, GQA_F16_SPLIT=None, GQA_F16_ROWS="mma"),
           "fma": dict(GQA_F16_KERNEL="fma", GQA_F16_SPLIT=None, GQA_F16_ROWS=None)}[name]
    with _env(**env):
        yield


@contextmanager
def forced_ctas(n):
    """Runs the block with the stream-K grid forced to n CTAs (None: the planner's choice)."""
    with _env(GQA_FORCE_CTAS=n):
        yield


def run_case(case, err=None, max_kv_len=None, ids=None, seq_of="case"):
    from gqa_decode_attention_03_gb300 import gqa_decode as gd
    q = dev(case.q)
    kv = dev(case.kv_len)
    so = dev(case.seq_of) if isinstance(seq_of, str) else seq_of
    if case.kind == "f16":
        return gd.attn_decode_f16(q, dev(case.k), dev(case.v), kv, scale=case.scale, seq_of=so,
                                  max_kv_len=max_kv_len, err=err)
    ids_t = dev(case.ids) if (ids is None and case.ids is not None) else ids
    return gd.attn_decode_q8_sel(q, dev(case.kq), dev(case.vq), dev(case.ksc), dev(case.vsc), kv,
                                 ids=ids_t, budget=case.budget if ids_t is not None else None,
                                 scale=case.scale, seq_of=so, max_kv_len=max_kv_len, err=err)


def tol_of(case):
    return TOL_F16 if case.kind == "f16" else TOL_Q8


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bound = tol * np.maximum(1.0, np.abs(ref))
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (f"{what}: max |err| {err.max():.3e} at {worst}, "
                                  f"ref {ref[worst]:.6f} got {got[worst]:.6f}, tol {tol}")
    return float(err.max())


def oracle_ref(case, rows=None):
    return pins.oracle_case(case, rows=rows)
