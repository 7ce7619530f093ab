"""Writes closed_forms.json: small decode-attention problems whose answer has a closed form.

Run from the repository root:  python tests/golden/make_closed_forms.py

The expected values are evaluated from the closed forms below with Python's ``decimal`` module
at 40 significant digits.  This script calls neither the CUDA library nor the oracle; the tests
use the fixture to pin the oracle (and, on a GPU, the kernels too).  Every input value is
exactly representable in its storage type (f16 cache values, fp32 q, int8 + f16 scales).

Definitions: single-query decode attention as in attention_gqa.metal (cera 0.5.4: scaled q.k,
safe softmax, weighted sum of V rows, head h -> KV head h // group); the int8 dequantisation of
qsa2.metal (qsa_attn2: int8 value times the f16 scale of its 64-dim group); the selected width
min(n_kv, budget) of qsa_attn2; the zero output for an empty context of flash_attention.metal
(cera 0.2.0); the log-sum-exp merge of qsa2.metal's qsa_merge2.
"""

import json
from decimal import Decimal, getcontext
from pathlib import Path

getcontext().prec = 40
D = 64


def dexp(x):
    return Decimal(x).exp()


def sigmoid(x):
    return Decimal(1) / (Decimal(1) + dexp(-Decimal(x)))


def zeros(*shape):
    if len(shape) == 1:
        return [0.0] * shape[0]
    return [zeros(*shape[1:]) for _ in range(shape[0])]


def case_sigmoid_pair():
    # one head, one KV head; two keys along dim 0; x0 = 0.5*2 = 1, x1 = 0.5*(-1) = -0.5
    q = zeros(1, 1, D); q[0][0][0] = 1.0
    K = zeros(1, 2, 1, D); K[0][0][0][0] = 2.0; K[0][1][0][0] = -1.0
    V = zeros(1, 2, 1, D); V[0][0][0][1] = 3.0; V[0][1][0][1] = -5.0; V[0][1][0][2] = 0.5
    w0 = sigmoid(Decimal("1.5"))
    out = [Decimal(0)] * D
    out[1] = w0 * 3 + (1 - w0) * (-5)
    out[2] = (1 - w0) * Decimal("0.5")
    return dict(name="sigmoid_pair", kind="f16", q=q, k=K, v=V, kv_len=[2], scale=0.5,
                expected=[[[str(x) for x in out]]],
                derivation="w0 = sigmoid(x0 - x1) = sigmoid(1.5); out = w0 V0 + (1 - w0) V1")


def case_geometric():
    # K_j = j e0, q = e0, scale 1/4 -> weights proportional to r^j, r = e^(1/4)
    L = 7
    q = zeros(1, 1, D); q[0][0][0] = 1.0
    K = zeros(1, L, 1, D); V = zeros(1, L, 1, D)
    for j in range(L):
        K[0][j][0][0] = float(j)
        V[0][j][0][0] = float(j)
        V[0][j][0][3] = float(j % 2)
    r = dexp(Decimal("0.25"))
    Z = sum(r ** j for j in range(L))
    out = [Decimal(0)] * D
    out[0] = sum(j * r ** j for j in range(L)) / Z
    out[3] = sum(r ** j for j in range(L) if j % 2) / Z
    return dict(name="geometric", kind="f16", q=q, k=K, v=V, kv_len=[L], scale=0.25,
                expected=[[[str(x) for x in out]]],
                derivation="w_j = r^j / sum r^j with r = e^(1/4); out0 = sum j w_j; "
                           "out3 = sum over odd j of w_j")


def case_uniform_keys():
    # identical keys -> uniform weights -> the mean of the V rows
    L = 5
    q = zeros(1, 2, D)
    for d in range(D):
        q[0][0][d] = 0.25 * ((d % 7) - 3)
        q[0][1][d] = -0.5 * ((d % 3) - 1)
    K = zeros(1, L, 1, D); V = zeros(1, L, 1, D)
    for j in range(L):
        for d in range(D):
            K[0][j][0][d] = 0.125 * ((d % 5) - 2)
            V[0][j][0][d] = (j + 1) * (d + 1) / 8.0
    mean = [Decimal(L + 1) / 2 * Decimal(d + 1) / 8 for d in range(D)]
    return dict(name="uniform_keys", kind="f16", q=q, k=K, v=V, kv_len=[L], scale=0.125,
                expected=[[[str(x) for x in mean], [str(x) for x in mean]]],
                derivation="all x_j equal -> w_j = 1/L -> out_d = (L+1)/2 * (d+1)/8")


def case_gqa_map():
    # 4 heads over 2 KV heads: KV head 0 has V rows = 1, KV head 1 has V rows = -2 (constant
    # rows make every softmax give the constant), so heads 0,1 -> 1 and heads 2,3 -> -2
    L = 3
    q = zeros(1, 4, D)
    for h in range(4):
        for d in range(D):
            q[0][h][d] = 0.5 if (d + h) % 4 == 0 else -0.25
    K = zeros(1, L, 2, D); V = zeros(1, L, 2, D)
    for j in range(L):
        for g in range(2):
            for d in range(D):
                K[0][j][g][d] = 0.25 * (((j + 2 * g + d) % 5) - 2)
                V[0][j][g][d] = 1.0 if g == 0 else -2.0
    exp = [[str(Decimal(1))] * D] * 2 + [[str(Decimal(-2))] * D] * 2
    return dict(name="gqa_map", kind="f16", q=q, k=K, v=V, kv_len=[L], scale=0.125,
                expected=[exp], derivation="constant V rows per KV head; head h reads KV head h//2")


def case_empty():
    q = zeros(1, 2, D); q[0][0][0] = 1.0
    K = zeros(1, 1, 1, D); V = zeros(1, 1, 1, D); V[0][0][0][0] = 9.0
    return dict(name="empty_context", kind="f16", q=q, k=K, v=V, kv_len=[0], scale=1.0,
                expected=[[["0"] * D, ["0"] * D]], derivation="kv_len = 0 writes zeros")


def case_q8_tanh():
    # int8: K_0[0] = 64 * 2^-6 = 1, K_1[0] = -64 * 2^-6 = -1; q = e0, scale 1/16
    # V rows: +-127 * 2^-7 in dims 0..63 (group 0) -> out = 0.9921875 * tanh(1/16)
    q = zeros(1, 1, D); q[0][0][0] = 1.0
    kq = zeros(1, 2, 1, D); ksc = zeros(1, 2, 1, 1)
    vq = zeros(1, 2, 1, D); vsc = zeros(1, 2, 1, 1)
    kq[0][0][0][0] = 64; kq[0][1][0][0] = -64
    ksc[0][0][0][0] = 2.0 ** -6; ksc[0][1][0][0] = 2.0 ** -6
    for d in range(D):
        vq[0][0][0][d] = 127; vq[0][1][0][d] = -127
    vsc[0][0][0][0] = 2.0 ** -7; vsc[0][1][0][0] = 2.0 ** -7
    w0 = sigmoid(Decimal(2) / 16)
    val = Decimal("0.9921875") * (2 * w0 - 1)
    return dict(name="q8_tanh", kind="q8", q=q, kq=kq, vq=vq, ksc=ksc, vsc=vsc, kv_len=[2],
                scale=0.0625, expected=[[[str(val)] * D]],
                derivation="w0 = sigmoid(1/16 - (-1/16)); out = 0.9921875 (2 w0 - 1)")


def case_q8_selected():
    # 6 cells, ids = [1, 4, 5] with budget 2 -> only cells 1 and 4 are visited
    # K_1 . q = 2, K_4 . q = 0 (via int8 32 * 2^-4 = 2); V_1 = 1, V_4 = -1 (127 * scale 1/127 is
    # not exact in f16, so use 64 * 2^-6 = 1); cells 0, 2, 3, 5 carry large values that would
    # change the answer if visited
    q = zeros(1, 1, D); q[0][0][0] = 1.0
    kq = zeros(1, 6, 1, D); ksc = zeros(1, 6, 1, 1)
    vq = zeros(1, 6, 1, D); vsc = zeros(1, 6, 1, 1)
    for j in range(6):
        ksc[0][j][0][0] = 2.0 ** -4
        vsc[0][j][0][0] = 2.0 ** -6
        for d in range(D):
            vq[0][j][0][d] = 100
        kq[0][j][0][0] = 127
    kq[0][1][0][0] = 32; kq[0][4][0][0] = 0
    for d in range(D):
        vq[0][1][0][d] = 64; vq[0][4][0][d] = -64
    w1 = sigmoid(Decimal(2) * Decimal("0.5"))
    val = w1 - (1 - w1)
    return dict(name="q8_selected", kind="q8", q=q, kq=kq, vq=vq, ksc=ksc, vsc=vsc, kv_len=[6],
                ids=[[1, 4, 5]], budget=2, scale=0.5, expected=[[[str(val)] * D]],
                derivation="width = min(6, 2) = 2 -> cells 1, 4; x = (1, 0); "
                           "out = sigmoid(1) - (1 - sigmoid(1))")


def merge_case():
    # two chunks: m = (0, ln 3), l = (1, 1), acc rows a and b -> (a + 3 b) / 4 ... written out
    a = [Decimal(d) / 4 for d in range(D)]
    b = [Decimal(-d) / 8 + 1 for d in range(D)]
    out = [(x + 3 * y) / 4 for x, y in zip(a, b)]
    return dict(name="merge_two_chunks", m=[0.0, str(Decimal(3).ln())], l=[1.0, 1.0],
                acc=[[str(x) for x in a], [str(x) for x in b]], expected=[str(x) for x in out],
                derivation="e = (exp(0 - ln3), 1) = (1/3, 1); L = 4/3; out = (a/3 + b) / (4/3)")


def main():
    cases = [case_sigmoid_pair(), case_geometric(), case_uniform_keys(), case_gqa_map(),
             case_empty(), case_q8_tanh(), case_q8_selected()]
    doc = {
        "about": "closed-form decode-attention cases; expected values at 40 digits from the "
                 "derivation strings (decimal module), written by make_closed_forms.py",
        "cite": {
            "f16": "attention_gqa.metal (cera 0.5.4): scaled q.k, safe softmax, weighted V sum, "
                   "head h -> KV head h // group; flash_attention.metal (cera 0.2.0): empty "
                   "context writes zeros",
            "q8": "qsa2.metal (regolith), qsa_attn2: int8 value times f16 scale per 64 dims; "
                  "visits the first min(n_kv, budget) ids",
            "merge": "qsa2.metal (regolith), qsa_merge2: log-sum-exp merge of chunk partials",
        },
        "cases": cases,
        "merge": merge_case(),
    }
    path = Path(__file__).with_name("closed_forms.json")
    path.write_text(json.dumps(doc, indent=0))
    print("wrote", path)


if __name__ == "__main__":
    main()
