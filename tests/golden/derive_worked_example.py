"""Derive the expected values of ``worked_example_forward.json`` from its
inputs, in exact arithmetic, independently of the oracle.

The layer forward (Engram.forward on the page of
vllm.models.deepseek_v4_1.common.engram; the gate of
_engram_gate_finish_kernel on the page of vllm.models.deepseek_v41.amd.engram):

* rows: one row per hash column, global row = row_offset[c] + id, a zero row
  for an id outside [0, rows[c]); A[t] = the rows concatenated (k = c*E + j);
* kv = A . wkv^T (wkv is [N, K]); copy h's key = kv[h*D:(h+1)*D], the value
  is the last D columns;
* hr = 1/sqrt(sum hidden^2 / D + eps), kr = 1/sqrt(sum key^2 / D + eps),
  dot = sum(hidden*q*k*key) * hr * kr / sqrt(D), gi = +-sqrt(max(|dot|,
  clamp)) (negative only when dot < 0), gate = sigmoid(gi), 0 when masked;
* out = hidden + gate*value rounded once to bf16 (8 significant bits,
  nearest, ties to even); a masked token keeps hidden's values, -0.0
  included.

Sums are exact rationals (``fractions``); roots, exponentials and the
sigmoid are 50-digit decimals (``decimal``).  Nothing here imports the
oracle or the CUDA package.

    python tests/golden/derive_worked_example.py           # print the expected block
    python tests/golden/derive_worked_example.py --write   # rewrite it in the fixture
"""
from __future__ import annotations

import json
import math
import os
import sys
from decimal import Decimal, localcontext
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))
FIXTURE = os.path.join(HERE, "worked_example_forward.json")
DIGITS = 50


def _dec(x) -> Decimal:
    """A rational as a decimal of DIGITS significant digits."""
    x = Fraction(x)
    with localcontext() as ctx:
        ctx.prec = DIGITS
        return Decimal(x.numerator) / Decimal(x.denominator)


def _sigmoid(x: Decimal) -> Decimal:
    with localcontext() as ctx:
        ctx.prec = DIGITS
        return Decimal(1) / (Decimal(1) + (-x).exp())


def _round_bf16(y: Decimal) -> float:
    """Nearest bf16 value (8 significant bits, ties to even) of a decimal
    that is not near a tie; raises if it lies within 1e-12 ulp of one."""
    if y == 0:
        return 0.0
    with localcontext() as ctx:
        ctx.prec = DIGITS
        a = abs(y)
        e = int(math.floor(math.log2(float(a))))
        # correct a floating misjudgement of the binade at a power of two
        while Decimal(2) ** e > a:
            e -= 1
        while Decimal(2) ** (e + 1) <= a:
            e += 1
        ulp = Decimal(2) ** (e - 7)
        q = a / ulp
        fl = int(q)
        frac = q - fl
        if abs(frac - Decimal("0.5")) < Decimal("1e-12"):
            raise ValueError(f"{y} is too close to a bf16 tie to round from 50 digits")
        r = fl + (1 if frac > Decimal("0.5") else 0)
        v = float(Decimal(r) * ulp)
    return -v if y < 0 else v


def _fmt(x: Decimal) -> str:
    """Exact integers as such, everything else to 25 significant digits."""
    if x == x.to_integral_value():
        return str(int(x))
    with localcontext() as ctx:
        ctx.prec = 25
        return str(+x)


def derive(ex: dict) -> dict:
    c = ex["config"]
    T, D, H, E = c["T"], c["dim"], c["hc_mult"], c["head_dim"]
    C = (c["max_ngram_size"] - 1) * c["n_heads"]
    # eps and clamp as the decimal numbers the fixture writes (1e-6 exactly)
    eps, clamp = Fraction(str(c["eps"])), _dec(Fraction(str(c["clamp"])))
    table = [[Fraction(v) for v in r] for r in ex["table"]]
    wkv = [[Fraction(v) for v in r] for r in ex["wkv"]]
    q = [[Fraction(v) for v in r] for r in ex["q_weight"]]
    k = [[Fraction(v) for v in r] for r in ex["k_weight"]]
    n_bad = 0
    rows_out, kv_out, dots, gates, outs = [], [], [], [], []
    for t in range(T):
        A = []
        for col in range(C):
            i = ex["hash_ids"][t][col]
            if 0 <= i < ex["rows"][col]:
                A += table[ex["row_offset"][col] + i]
            else:
                n_bad += 1
                A += [Fraction(0)] * E
        kv = [sum(a * w for a, w in zip(A, wrow)) for wrow in wkv]
        rows_out.append([float(a) for a in A])
        kv_out.append([float(v) for v in kv])
        value = kv[H * D:(H + 1) * D]
        active = ex["token_mask"][t] != 0
        dot_t, gate_t, out_t = [], [], []
        for h in range(H):
            x = [Fraction(v) for v in ex["hidden"][t][h]]
            key = kv[h * D:(h + 1) * D]
            s_hh = sum(v * v for v in x)
            s_kk = sum(v * v for v in key)
            s_hk = sum(x[d] * q[h][d] * k[h][d] * key[d] for d in range(D))
            with localcontext() as ctx:
                ctx.prec = DIGITS
                den = (_dec(s_hh / D + eps).sqrt() * _dec(s_kk / D + eps).sqrt()
                       * _dec(D).sqrt())
                dot = _dec(s_hk) / den
                gi = max(abs(dot), clamp).sqrt()
                if dot < 0:
                    gi = -gi
                g = _sigmoid(gi) if active else Decimal(0)
            dot_t.append(_fmt(dot))
            gate_t.append(_fmt(g))
            if active:
                out_t.append([_round_bf16(_dec(x[d]) + g * _dec(value[d])) for d in range(D)])
            else:
                out_t.append(list(ex["hidden"][t][h]))  # hidden's values, -0.0 included
        dots.append(dot_t)
        gates.append(gate_t)
        outs.append(out_t)
    return {"n_bad": n_bad, "rows": rows_out, "kv": kv_out, "dot": dots, "gate": gates,
            "out": outs}


def load() -> dict:
    with open(FIXTURE) as f:
        return json.load(f)


def main(argv) -> int:
    ex = load()
    exp = derive(ex)
    if "--write" in argv:
        ex["expected"] = exp
        with open(FIXTURE, "w") as f:
            json.dump(ex, f, indent=2)
            f.write("\n")
    else:
        print(json.dumps(exp, indent=1))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
