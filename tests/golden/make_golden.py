"""Write the golden fixtures of tests/golden/.

Imports only ``oracle/`` and the seeded input generators; never the CUDA path.
Run from the repository root:  python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import math
import os
import sys
from fractions import Fraction
from decimal import Decimal, getcontext

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from oracle import linear_logprob as O  # noqa: E402
from invariant_selected_token_gb300 import workloads  # noqa: E402


def rn_fp32(q: Fraction) -> float:
    """Round a nonzero rational to the nearest fp32 (ties to even), normal range."""
    neg = q < 0
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    scale = Fraction(2) ** (23 - e)
    m = q * scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = float(Fraction(fl) / scale)
    return -v if neg else v


def closed_forms():
    out = {"neg_log_V": {str(V): -math.log(V) for V in (2, 1024, 151936)},
           "softplus": {}}
    for d in (-3.0, -0.5, 0.0, 0.75, 4.0, 20.0):
        out["softplus"][repr(d)] = -math.log1p(math.exp(d))
    out["_source"] = ("softmax over V equal logits gives probability 1/V; two-class softmax "
                      "gives log p0 = -log(1 + exp(l1 - l0)); values by Python math")
    return out


def tile_tree():
    out = {"_source": "recursive bisection of the 128-wide tiles, lower half takes the extra tile"}
    for V in (151936, 1024):
        nt = O.n_vocab_tiles(V)
        out[str(V)] = {"n_tiles": nt}
        for d in (1, 2, 3):
            out[str(V)][str(1 << d)] = [b - a for a, b in O.tile_tree_nodes(nt, d)]
    return out


def contract_constants():
    getcontext().prec = 80
    ln2 = Fraction(Decimal(2).ln())
    log2e = Fraction(1 / Decimal(2).ln())
    sqrt2 = Fraction(Decimal(2).sqrt())
    hi = Fraction(rn_fp32(ln2))
    lo = rn_fp32(ln2 - hi)
    c = {"log2e": rn_fp32(log2e), "ln2_hi": float(hi), "ln2_lo": lo,
         "shifter": 12582912.0, "sqrt2": rn_fp32(sqrt2)}
    for k in range(8):
        c["inv_fact%d" % k] = rn_fp32(Fraction(1, math.factorial(k)))
    for k in range(5):
        c["two_over_%d" % (2 * k + 3)] = rn_fp32(Fraction(2, 2 * k + 3))
    return {k: float(v).hex() for k, v in c.items()}


def tiny_oracle():
    w = workloads.tiny()
    lp, lse = O.selected_logprob(w.hidden, w.W, w.targets, rows=range(8))
    return {"_source": "oracle/linear_logprob.py on workloads.tiny(seed=0), rows 0..7",
            "targets": w.targets[:8].tolist(), "logprob": lp.tolist(), "lse": lse.tolist()}


def main():
    files = {"closed_forms.json": closed_forms(), "tile_tree.json": tile_tree(),
             "contract_constants.json": contract_constants(), "tiny_oracle.json": tiny_oracle()}
    for name, obj in files.items():
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(obj, f, indent=1, sort_keys=True)
            f.write("\n")
        print("wrote", name)


if __name__ == "__main__":
    main()
