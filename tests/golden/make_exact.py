"""Write tests/golden/exact_d4_t3.json from the exact rational oracle.

The fixture is a hand-chosen tiny problem (head_dim 4, three tokens, a
non-symmetric initial state so that a transposed [key][value] layout gives a
different answer, one token with beta = 1 and a unit key so the delta rule's
overwrite is exact).  Expected values come only from ``oracle.exact``.

Run from the repository root:  python tests/golden/make_exact.py
"""
from __future__ import annotations

import json
import os
import sys
from fractions import Fraction as F

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle.exact import exact_forward  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_d4_t3.json")


def problem():
    alpha = [F(1, 2), F(3, 4), F(1, 1)]
    beta = [F(1, 1), F(1, 3), F(2, 5)]
    # token 0: unit key (beta = 1 -> S_1 k_0 = v_0 exactly)
    k = [[F(0), F(3, 5), F(0), F(4, 5)],
         [F(1, 2), F(-1, 2), F(1, 2), F(1, 2)],
         [F(1), F(0), F(0), F(0)]]
    q = [[F(1), F(0), F(0), F(0)],
         [F(0), F(1, 2), F(-1), F(1, 4)],
         [F(2, 3), F(1, 3), F(0), F(-1, 3)]]
    v = [[F(1), F(-2), F(1, 2), F(0)],
         [F(0), F(1), F(1), F(-1)],
         [F(3), F(0), F(-1, 4), F(1, 8)]]
    S0 = [[F(0), F(1), F(0), F(0)],       # S0[0][1] = 1: value 0, key 1
          [F(0), F(0), F(0), F(2)],       # S0[1][3] = 2
          [F(-1), F(0), F(0), F(0)],      # S0[2][0] = -1
          [F(0), F(0), F(1, 2), F(0)]]    # S0[3][2] = 1/2
    return alpha, beta, q, k, v, S0


def main():
    alpha, beta, q, k, v, S0 = problem()
    scaled_out, S = exact_forward(alpha, beta, q, k, v, S0)
    s = lambda x: f"{x.numerator}/{x.denominator}"
    doc = {
        "what": "gated delta rule, head_dim 4, 3 tokens, one (sequence, head); exact rationals",
        "source": ("definition S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T, "
                   "o_t = S_t q_t / sqrt(d); 'Gated Delta Net on AMD: why ROCm stumbles on "
                   "hybrid-attention LLMs', section 'What Gated Delta Net is, in plain language'; "
                   "'marcsun13/ggml-gated-delta-net' model card, section 'Ops' (state [value][key], "
                   "1/sqrt(head_dim) scale, log-domain gate)"),
        "generator": "tests/golden/make_exact.py (oracle.exact only)",
        "gate": "g_t = log(alpha_t)",
        "alpha": [s(x) for x in alpha], "beta": [s(x) for x in beta],
        "q": [[s(x) for x in r] for r in q], "k": [[s(x) for x in r] for r in k],
        "v": [[s(x) for x in r] for r in v], "state_in": [[s(x) for x in r] for r in S0],
        "out_times_sqrt_d": [[s(x) for x in r] for r in scaled_out],
        "state_out": [[s(x) for x in r] for r in S],
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
