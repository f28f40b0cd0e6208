"""The chunked path's operand precision, emulated on the CPU.

The chunked kernels feed tensor-core products with 16-bit operands and
accumulate in fp32.  Raw bf16 inputs (q, k, v) enter exactly; every derived
operand (the state S, the chunk transform Z = [T; P T], R and the scaled
corrections U~) is carried as a bf16 hi + lo pair, and each product of two
derived operands keeps three terms (hi*hi + hi*lo + lo*hi).  This module
restates that arithmetic in numpy, independently of the CUDA sources, and
holds it against the float64 oracle (the token-by-token recurrence) with the
parity metric (max-abs error / RMS).  T = (I + A)^-1 is solved here in
float64 and rounded to fp32; the kernels' blocked solve reaches about fp32
accuracy, so the split terms are what this compares.

What it pins:
  * the scheme meets the bf16 parity bound (3e-3) with a tenfold margin in
    every gate regime below;
  * no term can go: dropping any one split term breaks the bound in at least
    one regime, and so does carrying Z as a single fp16 term;
  * for decode attention (bound 1e-4), the probabilities need their hi + lo
    pair in the P V product: one bf16 term misses the bound.

Chunk algebra (chunk of C = 64 tokens from state S0, G the in-chunk running
sum of max(g, -30), gamma = exp(G)): A[r,i] = beta_r exp(G_r - G_i) k_r.k_i
(i < r), T = (I + A)^-1, P[r,i] = exp(G_r - G_i) q_r.k_i (i <= r),
R = beta (V - gamma K S0^T), U = T R, O = (gamma Q S0^T + P U)/sqrt(d),
S = gamma_C S0 + (exp(G_C - G) U)^T K: the unrolled gated delta rule of
"Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention LLMs",
section "What Gated Delta Net is, in plain language", in chunked form.
"""
import itertools

import numpy as np
import pytest

import oracle
from linear_attention_sequence_gated_gb300 import workloads as W

C = 64
BOUND = 3e-3


def bf16(x):
    """x (fp32) rounded to the nearest bf16, ties to even, as fp32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def split(x, kind="bf16"):
    rnd = bf16 if kind == "bf16" else f16
    hi = rnd(x)
    return hi, rnd(np.asarray(x, np.float32) - hi)


def mm(a, b):
    """Exact products of 16-bit values, the sum rounded to fp32 (TMEM)."""
    return (a.astype(np.float64) @ b.astype(np.float64)).astype(np.float32)


def split_product(A, B, terms, kind="bf16"):
    """A @ B from split operands, keeping the listed terms ('hh', 'hl', 'lh')."""
    parts = {"h": split(A, kind)[0], "l": split(A, kind)[1]}
    bparts = {"h": split(B, kind)[0], "l": split(B, kind)[1]}
    out = np.zeros((A.shape[0], B.shape[1]), np.float64)
    for t in terms:
        out += parts[t[0]].astype(np.float64) @ bparts[t[1]].astype(np.float64)
    return out.astype(np.float32)


KERNEL = {"PT": ("hh", "hl", "lh"), "X": ("h", "l"), "ZR": ("hh", "hl", "lh"), "dS": ("h", "l"),
          "zkind": "bf16"}
VARIANTS = {
    "Z R without Z lo * R hi": dict(KERNEL, ZR=("hh", "hl")),
    "Z R without Z hi * R lo": dict(KERNEL, ZR=("hh", "lh")),
    "state increment without U~ lo": dict(KERNEL, dS=("h",)),
    "P T without P lo * T": dict(KERNEL, PT=("hh", "hl")),
    "[K;Q] S^T without S lo": dict(KERNEL, X=("h",)),
}


def chunked(inp, cfg):
    """Output and final state of the chunked form with the operand precision
    `cfg` (which split terms each product keeps)."""
    q, k, v, g, beta, S0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "state"))
    B, T, H, d = v.shape
    out = np.zeros((B, T, H, d), np.float32)
    s_out = np.zeros((B, H, d, d), np.float32)
    tril_strict = np.tril(np.ones((C, C), bool), -1)
    tril = np.tril(np.ones((C, C), bool), 0)
    for b, h in itertools.product(range(B), range(H)):
        S = np.zeros((d, d), np.float32) if S0 is None else S0[b, h].astype(np.float32)
        for t0 in range(0, T, C):
            n = min(C, T - t0)
            K, Q, V = (np.zeros((C, d), np.float32) for _ in range(3))
            K[:n], Q[:n], V[:n] = k[b, t0:t0 + n, h], q[b, t0:t0 + n, h], v[b, t0:t0 + n, h]
            gg, bb = np.zeros(C, np.float32), np.zeros(C, np.float32)
            gg[:n], bb[:n] = g[b, t0:t0 + n, h], beta[b, t0:t0 + n, h]
            G = np.cumsum(np.maximum(gg, -30.0)).astype(np.float32)
            gam = np.exp(G).astype(np.float32)
            diff = np.where(tril, G[:, None] - G[None, :], 0.0)
            dec = np.where(tril, np.exp(diff), 0.0).astype(np.float32)
            A = np.where(tril_strict, mm(K, K.T) * dec * bb[:, None], 0.0).astype(np.float32)
            P = np.where(tril, mm(Q, K.T) * dec, 0.0).astype(np.float32)
            Tm = np.linalg.inv(np.eye(C) + A.astype(np.float64)).astype(np.float32)
            Z = np.concatenate([Tm, split_product(P, Tm, cfg["PT"])], 0)
            Sp = dict(zip("hl", split(S)))
            XK = sum(mm(K, Sp[t].T) for t in cfg["X"])
            XQ = sum(mm(Q, Sp[t].T) for t in cfg["X"])
            R = (bb[:, None] * (V - gam[:, None] * XK)).astype(np.float32)
            ZR = split_product(Z, R, cfg["ZR"], cfg["zkind"])
            U, PU = ZR[:C], ZR[C:]
            out[b, t0:t0 + n, h] = ((gam[:, None] * XQ + PU) / np.sqrt(d))[:n]
            end = G[n - 1]
            Ut = (np.exp(end - G)[:, None] * U).astype(np.float32)
            Ut[n:] = 0.0
            Up = dict(zip("hl", split(Ut)))
            dS = sum(mm(Up[t].T, K) for t in cfg["dS"])
            S = (np.float32(np.exp(end)) * S + dS).astype(np.float32)
        s_out[b, h] = S
    return out, s_out


# (head_dim, heads, tokens, gate shift, initial-state std, seed): the benchmark
# gates (shift 2, fast forgetting) and slower ones, where errors in the state
# live longer
REGIMES = [
    (128, 1, 1024, 2.0, 0.0, 11),
    (128, 1, 1024, 0.0, 0.02, 13),
    (64, 2, 1024, -4.0, 0.02, 16),
    (256, 1, 512, -4.0, 0.02, 17),
]


# Z as a single fp16 term (with R as an fp16 hi + lo pair) halves the Z
# products and the Z bytes; it is checked on the benchmark gates over a
# longer run, where its error is clearest
FP16_Z = dict(KERNEL, ZR=("hh", "hl"), zkind="f16")
FP16_Z_REGIME = [(128, 2, 2048, 2.0, 0.02, 12)]


def regime_errors(cfg, regimes=REGIMES):
    errs = []
    for d, H, T, shift, std, seed in regimes:
        w = W.Workload(f"prec_{d}_{shift}", 1, T, H, d, "bf16", shift, std, seed=seed)
        inp = W.to_numpy_f32(W.make_inputs(w, "cpu"))
        ref_o, ref_s = oracle.recurrent_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                          inp["state"])
        o, s = chunked(inp, cfg)
        errs.append(max(oracle.parity_error(o, ref_o), oracle.parity_error(s, ref_s)))
    return errs


def test_kernel_scheme_meets_the_bound_with_margin():
    errs = regime_errors(KERNEL)
    assert max(errs) <= BOUND / 10, errs


@pytest.mark.parametrize("name", list(VARIANTS))
def test_every_split_term_is_needed(name):
    errs = regime_errors(VARIANTS[name])
    assert max(errs) > BOUND, (name, errs)


def test_single_fp16_z_term_breaks_the_bound():
    errs = regime_errors(FP16_Z, FP16_Z_REGIME)
    assert max(errs) > BOUND, errs


# ---------------------------------------------------------------- decode attention
#
# The attention kernel's path for 16-bit inputs forms the scores from exact
# products (fp32 accumulation), keeps the online softmax in log2 units over
# steps of 16 keys, and feeds the probabilities to the P V product as a
# 16-bit hi + lo pair.  The op's bound is max-abs / RMS <= 1e-4 against the
# float64 oracle (softmax attention as written).

ATTN_BOUND = 1e-4
LOG2E = 1.4426950408889634


def attention_mma(q, k, v, scale, p_terms):
    """Decode attention with the probabilities entering P V as `p_terms`
    ('hl': bf16 hi + lo, 'h': one bf16 term); q (B, H, n_q, d), k and v
    (B, Hkv, n_kv, d) as fp32 values of bf16 data."""
    B, H, n_q, d = q.shape
    Hkv, n_kv = k.shape[1], k.shape[2]
    rep = H // Hkv
    out = np.zeros((B, n_q, H, v.shape[3]))
    sl = np.float32(scale * LOG2E)
    for b, h, i in itertools.product(range(B), range(H), range(n_q)):
        kv = h // rep
        s = (mm(k[b, kv], q[b, h, i][:, None])[:, 0] * sl).astype(np.float32)
        m, l = -np.inf, np.float32(0.0)
        o = np.zeros(v.shape[3], np.float32)
        for j0 in range(0, n_kv, 16):
            sc = s[j0:j0 + 16]
            m_new = max(m, float(sc.max()))
            cf = np.float32(np.exp2(m - m_new))
            p = np.exp2(sc - np.float32(m_new)).astype(np.float32)
            l = np.float32(l * cf + p.sum(dtype=np.float32))
            ph, plo = split(p)
            pe = ph + plo if p_terms == "hl" else ph
            o = (o * cf + mm(pe[None, :], v[b, kv, j0:j0 + 16])[0]).astype(np.float32)
            m = m_new
        out[b, i, h] = o / l
    return out


@pytest.mark.parametrize("scale", [None, 1.0])
def test_attention_probabilities_need_hi_and_lo(scale):
    """The hi + lo pair meets the attention bound tenfold; one bf16 term for
    the probabilities does not meet it (scale None: 1/sqrt(d); 1.0: a peaked
    softmax)."""
    from oracle.attn import attention
    w = W.AttnWorkload("prec_attn", 2, 8, 2, 1, 1000, 128, "bf16", seed=21)
    inp = {n: x.float().numpy() for n, x in W.make_attn_inputs(w, "cpu").items() if x is not None}
    s = float(np.float32(1.0 / np.sqrt(w.d) if scale is None else scale))
    ref = attention(inp["q"], inp["k"], inp["v"], None, s)
    hl = oracle.parity_error(attention_mma(inp["q"], inp["k"], inp["v"], s, "hl"), ref)
    one = oracle.parity_error(attention_mma(inp["q"], inp["k"], inp["v"], s, "h"), ref)
    assert hl <= ATTN_BOUND / 10, hl
    assert one > ATTN_BOUND, one
