"""Checks that pin the fp64 oracle to something other than itself.

Each check returns a list of failure strings (empty = pass), so that the planted-mistake test
can run the whole battery against a deliberately broken oracle and require it to fail.

* closed forms: tests/golden/closed_forms.json (values at 40 digits from the derivations);
* brute force: a direct 30-digit ``decimal`` evaluation of the definition on tiny random
  problems (its own loops, its own dequantisation, its own exp);
* invariants fixed by the mathematics: one position returns V[0]; identical keys return the
  mean of V; permuting cache positions changes nothing; split-then-merge equals unsplit.
"""

from __future__ import annotations

import json
from decimal import Decimal, getcontext
from pathlib import Path

import numpy as np

import oracle
from gqa_decode_attention_03_gb300 import workloads as W

GOLDEN = Path(__file__).with_name("golden") / "closed_forms.json"


def load_golden():
    return json.loads(GOLDEN.read_text())


def golden_arrays(case):
    """Dense numpy inputs of one closed-form case."""
    q = np.asarray(case["q"], dtype=np.float32)
    kv_len = np.asarray(case["kv_len"], dtype=np.int32)
    exp = np.asarray([[[float(x) for x in row] for row in head] for head in case["expected"]])
    arr = dict(q=q, kv_len=kv_len, scale=float(case["scale"]), expected=exp)
    if case["kind"] == "f16":
        arr["k"] = np.asarray(case["k"], dtype=np.float16)
        arr["v"] = np.asarray(case["v"], dtype=np.float16)
    else:
        arr["kq"] = np.asarray(case["kq"], dtype=np.int8)
        arr["vq"] = np.asarray(case["vq"], dtype=np.int8)
        arr["ksc"] = np.asarray(case["ksc"], dtype=np.float16)
        arr["vsc"] = np.asarray(case["vsc"], dtype=np.float16)
    if "ids" in case:
        arr["ids"] = np.asarray(case["ids"], dtype=np.int32)
        arr["budget"] = int(case["budget"])
    return arr


def oracle_on(arr):
    ids, budget = arr.get("ids"), arr.get("budget")
    if "k" in arr:
        return oracle.decode_f16(arr["q"], arr["k"], arr["v"], arr["kv_len"], arr["scale"],
                                 ids=ids, budget=budget)
    return oracle.decode_q8(arr["q"], arr["kq"], arr["vq"], arr["ksc"], arr["vsc"],
                            arr["kv_len"], arr["scale"], ids=ids, budget=budget)


def _close(a, b, tol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return a.shape == b.shape and bool(np.all(np.abs(a - b) <= tol * np.maximum(1.0, np.abs(b))))


def check_closed_forms(tol=1e-13):
    fails = []
    doc = load_golden()
    for case in doc["cases"]:
        arr = golden_arrays(case)
        try:
            got = oracle_on(arr)
        except Exception as e:  # a broken oracle may raise
            fails.append(f"{case['name']}: raised {e!r}")
            continue
        if not _close(got, arr["expected"], tol):
            fails.append(f"{case['name']}: mismatch")
    mc = doc["merge"]
    acc = np.asarray([[[[float(x) for x in mc["acc"][c]]] for c in range(2)]])  # [1][2][1][D]
    m = np.asarray([[[float(mc["m"][0])], [float(mc["m"][1])]]])
    l = np.asarray([[[float(mc["l"][0])], [float(mc["l"][1])]]])
    try:
        got = oracle.lse_merge(acc, m, l, np.array([2]))
        if not _close(got[0, 0], [float(x) for x in mc["expected"]], tol):
            fails.append("merge_two_chunks: mismatch")
    except Exception as e:
        fails.append(f"merge_two_chunks: raised {e!r}")
    return fails


# ----------------------------------------------------------------------------- brute force

def _brute_row(qh, krows, vrows, scale):
    """30-digit evaluation of one (row, head): explicit loops, decimal exp."""
    getcontext().prec = 30
    if not krows:
        return [Decimal(0)] * len(qh)
    sc = Decimal(scale)
    x = [sc * sum(a * b for a, b in zip(qh, k)) for k in krows]
    mx = max(x)
    e = [(xi - mx).exp() for xi in x]
    z = sum(e)
    return [sum(e[j] * vrows[j][d] for j in range(len(e))) / z for d in range(len(qh))]


def brute_force(case):
    """Whole-problem brute force for a workloads.Case (f16 or q8)."""
    T, H, D = case.q.shape
    G = H // case.n_kv_heads
    out = np.zeros((T, H, D))
    for t in range(T):
        s = int(case.seq_of[t])
        L = max(int(case.kv_len[t]), 0)
        if case.ids is None:
            cells = list(range(L))
        else:
            cells = [int(c) for c in case.ids[t][:min(L, case.budget)]]
        for h in range(H):
            g = h // G
            qh = [Decimal(float(x)) for x in case.q[t, h]]
            if case.kind == "f16":
                kr = [[Decimal(float(x)) for x in case.k[s, j, g]] for j in cells]
                vr = [[Decimal(float(x)) for x in case.v[s, j, g]] for j in cells]
            else:
                def deq(vals, scl, grp=case.scale_group):
                    return [Decimal(int(vals[d])) * Decimal(float(scl[d // grp])) for d in range(D)]
                kr = [deq(case.kq[s, j, g], case.ksc[s, j, g]) for j in cells]
                vr = [deq(case.vq[s, j, g], case.vsc[s, j, g]) for j in cells]
            out[t, h] = [float(x) for x in _brute_row(qh, kr, vr, case.scale)]
    return out


def tiny_cases():
    """Tiny random problems: GQA groups of 2, ragged and empty rows, shared sequences, ids."""
    f = W.make_f16_case(7, 4, 4, 2, 8, [5, 0, 1, 3], cache_cap=6, seq_of=[0, 1, 2, 0],
                        scale=0.35, name="brute_f16")
    q = W.make_q8_case(8, 2, 4, 2, 128, [6, 3], budget=4, cache_cap=7, scale=0.0625,
                       name="brute_q8")
    q32 = W.make_q8_case(9, 2, 4, 2, 64, [5, 4], cache_cap=5, scale=0.125, scale_group=32,
                         name="brute_q8_g32")
    return [f, q, q32]


def oracle_case(case, rows=None):
    if case.kind == "f16":
        return oracle.decode_f16(case.q, case.k, case.v, case.kv_len, case.scale,
                                 seq_of=case.seq_of, ids=case.ids, budget=case.budget, rows=rows)
    return oracle.decode_q8(case.q, case.kq, case.vq, case.ksc, case.vsc, case.kv_len,
                            case.scale, seq_of=case.seq_of, ids=case.ids, budget=case.budget,
                            rows=rows)


def check_brute_force(tol=1e-12):
    fails = []
    for case in tiny_cases():
        try:
            got = oracle_case(case)
        except Exception as e:
            fails.append(f"{case.name}: raised {e!r}")
            continue
        if not _close(got, brute_force(case), tol):
            fails.append(f"{case.name}: oracle != 30-digit brute force")
    return fails


# ----------------------------------------------------------------------------- invariants

def check_invariants():
    fails = []
    try:
        # one position: softmax of one score is exactly 1, so out is V[0] bit for bit
        c = W.make_f16_case(11, 1, 4, 2, 64, [1], scale=0.125)
        got = oracle_case(c)
        for h in range(4):
            if not np.array_equal(got[0, h], c.v[0, 0, h // 2].astype(np.float64)):
                fails.append("one position != V[0]")
                break
        # split then merge == unsplit, several chunk lengths, dense and selected
        c = W.make_f16_case(12, 3, 6, 2, 64, [37, 1, 20], cache_cap=40, scale=0.2)
        ref = oracle_case(c)
        for chunk in (1, 4, 16, 64):
            acc, m, l, nv = oracle.split_partials_f16(c.q, c.k, c.v, c.kv_len, c.scale, chunk)
            if not _close(oracle.lse_merge(acc, m, l, nv), ref, 1e-12):
                fails.append(f"split({chunk}) + merge != unsplit")
        c = W.make_q8_case(13, 2, 4, 1, 64, [50, 9], budget=12, cache_cap=50, scale=0.1)
        ref = oracle_case(c)
        acc, m, l, nv = oracle.split_partials_q8(c.q, c.kq, c.vq, c.ksc, c.vsc, c.kv_len,
                                                 c.scale, 5, ids=c.ids, budget=c.budget)
        if not _close(oracle.lse_merge(acc, m, l, nv), ref, 1e-12):
            fails.append("q8 split + merge != unsplit")
    except Exception as e:
        fails.append(f"invariants raised {e!r}")
    return fails


def battery():
    return check_closed_forms() + check_brute_force() + check_invariants()
