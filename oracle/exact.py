"""Exact rational evaluation of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Used to write and re-check the small fixtures under ``tests/golden/``.  It
evaluates the definition in its matrix-product form,
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
    o_t * sqrt(d) = S_t q_t,
with ``fractions.Fraction`` entries, so the result has no rounding at all.
The gate enters as alpha_t = exp(g_t) given directly as a rational number
(the float64 oracles receive g_t = log(alpha_t)).  The output is returned
pre-multiplied by sqrt(d) so that it stays rational.

This is a different formulation from the step-by-step form in
``gdn_oracle.c`` and ``recurrent_np`` (explicit (I - beta k k^T) products
instead of decay / read / overwrite), in exact arithmetic.
Sources: "Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention
LLMs", section "What Gated Delta Net is, in plain language";
"marcsun13/ggml-gated-delta-net" model card, section "Ops" (state
[value][key], 1/sqrt(head_dim) output scale, log-domain gate).
"""
from __future__ import annotations

from fractions import Fraction


def _matmul(A, B):
    n, m, p = len(A), len(B), len(B[0])
    return [[sum((A[i][l] * B[l][j] for l in range(m)), Fraction(0)) for j in range(p)]
            for i in range(n)]


def exact_forward(alpha, beta, q, k, v, S0):
    """alpha, beta: length-T lists of Fractions; q, k, v: T lists of length-d
    Fraction vectors; S0: d x d Fractions, S0[i][j] with i = value, j = key.
    Returns (scaled_out, S_T): scaled_out[t][i] = sqrt(d) * o_t[i]."""
    d = len(S0)
    S = [row[:] for row in S0]
    scaled_out = []
    for t in range(len(alpha)):
        kt, vt, qt = k[t], v[t], q[t]
        # M = I - beta k k^T
        M = [[(Fraction(1) if i == j else Fraction(0)) - beta[t] * kt[i] * kt[j]
              for j in range(d)] for i in range(d)]
        SM = _matmul(S, M)
        S = [[alpha[t] * SM[i][j] + beta[t] * vt[i] * kt[j] for j in range(d)]
             for i in range(d)]
        scaled_out.append([sum((S[i][j] * qt[j] for j in range(d)), Fraction(0))
                           for i in range(d)])
    return scaled_out, S
