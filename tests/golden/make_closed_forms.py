#!/usr/bin/env python3
"""Writes closed_forms.txt: closed-form attention outputs in 40-digit decimal arithmetic.

Run from anywhere: ``python tests/golden/make_closed_forms.py`` rewrites the file beside this
script; ``--check`` compares instead of writing (exit status 1 on a difference). It imports
nothing from the oracle or the package: the outputs are the softmax of the chosen score
matrix written out with Python's decimal module, so they pin the oracle from outside.
"""

from __future__ import annotations

import os
import sys
from decimal import Decimal, getcontext

getcontext().prec = 40

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "closed_forms.txt")

HEADER = """\
# Closed-form fixtures for exact attention forward, head dim d = 64.
#
# Definition: "Flash attention in PyTorch, then in Triton", section "Attention's table of
# scores" — the scores are q.k^T divided by the square root of the head's 64 channels, the
# causal mask puts minus infinity above the diagonal (each token sees the tokens up to its
# own), a softmax turns each row into probabilities, and those weigh the values.
#
# With k_j set to unit vectors, the scaled score matrix S is chosen directly:
# q_i[e] = 8 * S[i][e] gives S[i][j] = q_i . k_j / sqrt(64). The expected outputs are the
# softmax closed forms o_i = sum_j exp(S_ij) v_j / sum_j exp(S_ij) over the visible keys,
# evaluated in 40-digit decimal arithmetic and printed to 17 significant digits. They do
# not come from the oracle or from any GPU code.
#
# Line formats:
#   case <name> N=<n>
#   in <q|k|v> <row> <dim> <value>        (every entry not listed is 0)
#   out <causal 0|1> <row> <dim> <value>  (every output entry not listed is exactly 0)
"""

# (comment, name, S as decimal strings, value entries (row, dim, value string))
CASES = [
    ("""\
# Asymmetric 2x2 scores S = [[1, 2], [0, 1]] pin the 1/sqrt(d) scale, the orientation of
# q.k^T (its transpose would give row 0 the weights of [1, 0]) and the causal diagonal
# (causal row 0 sees key 0 only, so it returns v_0 exactly).
""", "asym2", [["1", "2"], ["0", "1"]], [(0, 0, "1"), (0, 1, "2"), (1, 0, "-3"), (1, 3, "0.5")]),
    ("""\
# Three keys, S = [[0.5, 3, -1], [-1, 1.5, 2], [2, -0.25, 0.75]], values on dim 5 only
# (1, -2, 4). Causal rows see 1, 2 and 3 keys; non-causal rows see all three.
""", "three3", [["0.5", "3", "-1"], ["-1", "1.5", "2"], ["2", "-0.25", "0.75"]],
     [(0, 5, "1"), (1, 5, "-2"), (2, 5, "4")]),
]

D = 64


def fmt_in(x: Decimal) -> str:
    return format(x.normalize(), "f") if x != x.to_integral_value() else str(int(x))


def closed_form(S, v, causal):
    """o[i][e] for every row and dim, softmax over the visible keys, in decimal."""
    n = len(S)
    out = []
    for i in range(n):
        vis = range(i + 1) if causal else range(n)
        w = [S[i][j].exp() for j in vis]
        tot = sum(w, Decimal(0))
        out.append([sum((w[t] * v[j][e] for t, j in enumerate(vis)), Decimal(0)) / tot for e in range(D)])
    return out


def render() -> str:
    parts = [HEADER]
    for comment, name, s_txt, v_entries in CASES:
        n = len(s_txt)
        S = [[Decimal(x) for x in row] for row in s_txt]
        v = [[Decimal(0)] * D for _ in range(n)]
        for row, dim, val in v_entries:
            v[row][dim] = Decimal(val)
        lines = ["", comment.rstrip("\n"), f"case {name} N={n}"]
        for i in range(n):
            for e in range(n):
                if S[i][e] != 0:
                    lines.append(f"in q {i} {e} {fmt_in(8 * S[i][e])}")
        for j in range(n):
            lines.append(f"in k {j} {j} 1")
        for row, dim, val in v_entries:
            lines.append(f"in v {row} {dim} {val}")
        outs = {c: closed_form(S, v, c) for c in (0, 1)}
        for i in range(n):
            for c in (0, 1):
                for e in range(D):
                    x = outs[c][i][e]
                    if x != 0:
                        lines.append(f"out {c} {i} {e} {format(x, '.17g')}")
        parts.append("\n".join(lines) + "\n")
    return "".join(parts)


def main(argv):
    text = render()
    if "--check" in argv:
        with open(OUT) as f:
            same = f.read() == text
        print("closed_forms.txt matches" if same else "closed_forms.txt differs from the generator")
        return 0 if same else 1
    with open(OUT, "w") as f:
        f.write(text)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
