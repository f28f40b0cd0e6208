"""Pins for the float64 oracle (CPU only).

The oracle is pinned to facts that do not come from the oracle itself:
exact rational results of the definition's matrix-product form, closed forms
of special cases (beta = 0, g = 0, g -> -inf, a single step from zero, a
one-hot [value][key] state), invariants (overwrite property of the delta
rule, row equivariance, linearity, carrying the state across calls) and a
brute-force chunked evaluation.  The last test plants plausible mistakes in
a copy of the recurrence and checks that at least one pin catches each.

Definition: S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t / sqrt(d), state [value][key] ("marcsun13/ggml-gated-delta-net"
model card, section "Ops"; "Gated Delta Net on AMD: why ROCm stumbles on
hybrid-attention LLMs", section "What Gated Delta Net is, in plain language").
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.exact import exact_forward

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "exact_d4_t3.json")


def rand_problem(seed, B=2, T=7, H=3, d=8, state=True, unit=True, gate_shift=0.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, d))
    k = r.standard_normal((B, T, H, d))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, H, d))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, H))))
    g = -np.log1p(np.exp(r.standard_normal((B, T, H)) + gate_shift))
    S0 = r.standard_normal((B, H, d, d)) * 0.3 if state else None
    # float32-representable inputs so the C oracle (float32 in) sees the same values
    f = lambda a: None if a is None else a.astype(np.float32).astype(np.float64)
    return f(q), f(k), f(v), f(g), f(beta), f(S0)


def c_impl(q, k, v, g, beta, S0):
    return oracle.recurrent_c(q, k, v, g, beta, S0)


# the C oracle takes float32 inputs; the golden fixture's rationals (and its
# gates log(alpha)) are not all float32-representable, so that pin allows the
# input rounding there.  Every other pin feeds float32-exact values.
c_impl.input_tol = 1e-6


def np_impl(q, k, v, g, beta, S0):
    return oracle.recurrent_np(q, k, v, g, beta, S0)


IMPLS = {"c": c_impl, "numpy": np_impl}


def rel(a, b):
    scale = max(1e-300, float(np.max(np.abs(b))))
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) / scale


# --------------------------------------------------------------------------
# pins, each written as a predicate over an implementation so the mutation
# test below can run the same checks against deliberately broken copies
# --------------------------------------------------------------------------

def pin_golden_exact(impl):
    doc = json.load(open(GOLDEN))
    fr = lambda s: Fraction(s)
    alpha = np.array([float(fr(x)) for x in doc["alpha"]])
    beta = np.array([float(fr(x)) for x in doc["beta"]])
    mat = lambda key: np.array([[float(fr(x)) for x in row] for row in doc[key]])
    q, k, v, S0 = mat("q"), mat("k"), mat("v"), mat("state_in")
    T, d = q.shape
    g = np.log(alpha)
    out, S = impl(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                  beta[None, :, None], S0[None, None])
    exp_out = mat("out_times_sqrt_d") / math.sqrt(d)
    exp_S = mat("state_out")
    tol = getattr(impl, "input_tol", 1e-12)
    return rel(out[0, :, 0], exp_out) < tol and rel(S[0, 0], exp_S) < tol


def pin_identity(impl):
    """beta = 0 and g = 0: the state passes through unchanged and every
    output is the matrix-vector product S0 q / sqrt(d)."""
    q, k, v, g, beta, S0 = rand_problem(1)
    g[:] = 0.0
    beta[:] = 0.0
    out, S = impl(q, k, v, g, beta, S0)
    d = q.shape[-1]
    want = np.einsum("bhij,bthj->bthi", S0, q) / math.sqrt(d)
    return np.array_equal(S, S0) and rel(out, want) < 1e-13


def pin_overwrite(impl):
    """beta = 1 and a unit key: after the step the state maps k_t to v_t
    exactly, whatever the previous state and the gate."""
    q, k, v, g, beta, S0 = rand_problem(2, T=5)
    beta[:] = 1.0
    # keys with four entries of +-1/2: unit norm exactly in binary floating point
    r = np.random.default_rng(20)
    k[:] = 0.0
    for idx in np.ndindex(k.shape[:3]):
        pos = r.choice(k.shape[-1], 4, replace=False)
        k[idx + (pos,)] = r.choice([-0.5, 0.5], 4)
    out, S = impl(q, k, v, g, beta, S0)
    kT, vT = k[:, -1], v[:, -1]                        # (B, H, d)
    got = np.einsum("bhij,bhj->bhi", S, kT)
    return rel(got, vT) < 1e-12


def pin_forgetting(impl):
    """g = -inf at token t0 erases everything before it: the outputs from t0
    on and the final state equal a fresh run started at t0 from zeros."""
    q, k, v, g, beta, S0 = rand_problem(3, T=9)
    t0 = 4
    g[:, t0] = -np.inf
    out, S = impl(q, k, v, g, beta, S0)
    sl = lambda a: a[:, t0:].copy()
    g2 = sl(g)
    g2[:, 0] = 0.0
    out2, S2 = impl(sl(q), sl(k), sl(v), g2, sl(beta), None)
    return rel(out[:, t0:], out2) < 1e-12 and rel(S, S2) < 1e-12


def pin_pure_decay(impl):
    """beta = 0: S_T = exp(sum g) S0 and o_t = exp(G_t) S0 q_t / sqrt(d)."""
    q, k, v, g, beta, S0 = rand_problem(4, T=6)
    beta[:] = 0.0
    out, S = impl(q, k, v, g, beta, S0)
    G = np.cumsum(g, axis=1)                            # (B, T, H)
    d = q.shape[-1]
    want_S = np.exp(G[:, -1])[:, :, None, None] * S0
    want_o = np.exp(G)[..., None] * np.einsum("bhij,bthj->bthi", S0, q) / math.sqrt(d)
    return rel(S, want_S) < 1e-12 and rel(out, want_o) < 1e-12


def pin_single_step(impl):
    """One token from a zero state: S_1 = beta v k^T, o_1 = beta (k.q) v / sqrt(d)."""
    q, k, v, g, beta, _ = rand_problem(5, T=1)
    out, S = impl(q, k, v, g, beta, None)
    d = q.shape[-1]
    b = beta[:, 0]
    want_S = b[..., None, None] * np.einsum("bhi,bhj->bhij", v[:, 0], k[:, 0])
    kq = np.sum(k[:, 0] * q[:, 0], axis=-1)
    want_o = (b * kq)[..., None] * v[:, 0] / math.sqrt(d)
    return rel(S, want_S) < 1e-13 and rel(out[:, 0], want_o) < 1e-13


def pin_layout(impl):
    """state[i][j] = 1 (value i, key j), beta = 0, g = 0, q = e_j: the single
    nonzero output is out[i] = 1/sqrt(d).  A [key][value] reading puts it at
    out[j] instead."""
    d = 8
    i, j = 2, 5
    S0 = np.zeros((1, 1, d, d))
    S0[0, 0, i, j] = 1.0
    q = np.zeros((1, 1, 1, d))
    q[..., j] = 1.0
    k = np.zeros_like(q)
    v = np.zeros_like(q)
    z = np.zeros((1, 1, 1))
    out, S = impl(q, k, v, z, z, S0)
    want = np.zeros(d)
    want[i] = 1.0 / math.sqrt(d)
    return np.allclose(out[0, 0, 0], want, rtol=0, atol=1e-15) and np.array_equal(S, S0)


def pin_row_equivariance(impl):
    """Value rows are independent: permuting the value index of v, of the
    initial state's rows and of the outputs commutes with the op."""
    q, k, v, g, beta, S0 = rand_problem(6)
    perm = np.random.default_rng(7).permutation(q.shape[-1])
    out, S = impl(q, k, v, g, beta, S0)
    out_p, S_p = impl(q, k, v[..., perm], g, beta, S0[:, :, perm, :])
    return rel(out_p, out[..., perm]) < 1e-12 and rel(S_p, S[:, :, perm, :]) < 1e-12


def pin_linearity(impl):
    """The op is jointly linear in (v, S0)."""
    q, k, v1, g, beta, S1 = rand_problem(8)
    _, _, v2, _, _, S2 = rand_problem(9)
    # multiples of 2^-12: the combination below is exact in float32 as well
    v1, v2, S1, S2 = (np.round(x * 4096.0) / 4096.0 for x in (v1, v2, S1, S2))
    a, b = 0.75, -1.25
    o1, T1 = impl(q, k, v1, g, beta, S1)
    o2, T2 = impl(q, k, v2, g, beta, S2)
    o3, T3 = impl(q, k, a * v1 + b * v2, g, beta, a * S1 + b * S2)
    return rel(o3, a * o1 + b * o2) < 1e-12 and rel(T3, a * T1 + b * T2) < 1e-12


def pin_state_carry(impl):
    """One call over [0, T) equals [0, T1) then [T1, T) with the final state
    fed back as the initial state, for every split point."""
    q, k, v, g, beta, S0 = rand_problem(10, T=6)
    out, S = impl(q, k, v, g, beta, S0)
    # the C oracle takes its initial state in float32, so the carried state is
    # rounded once there; the numpy twin carries it in float64
    tol = getattr(impl, "input_tol", 1e-12)
    for t1 in range(1, q.shape[1]):
        a = lambda x: x[:, :t1]
        z = lambda x: x[:, t1:]
        oa, Sa = impl(a(q), a(k), a(v), a(g), a(beta), S0)
        ob, Sb = impl(z(q), z(k), z(v), z(g), z(beta), Sa)
        if rel(np.concatenate([oa, ob], axis=1), out) > tol or rel(Sb, S) > tol:
            return False
    return True


def pin_definition_form(impl):
    """Brute force with explicit d x d matrices in the printed form
    S_t = alpha S (I - beta k k^T) + beta v k^T on tiny inputs."""
    q, k, v, g, beta, S0 = rand_problem(11, B=1, T=5, H=2, d=4)
    out, S = impl(q, k, v, g, beta, S0)
    d = q.shape[-1]
    for h in range(q.shape[2]):
        M = S0[0, h].copy()
        for t in range(q.shape[1]):
            kt, vt, qt = k[0, t, h], v[0, t, h], q[0, t, h]
            M = math.exp(g[0, t, h]) * M @ (np.eye(d) - beta[0, t, h] * np.outer(kt, kt)) \
                + beta[0, t, h] * np.outer(vt, kt)
            if rel(out[0, t, h], M @ qt / math.sqrt(d)) > 1e-12:
                return False
        if rel(S[0, h], M) > 1e-12:
            return False
    return True


def _key_head_problem(seed, H, Hk, T):
    """q, k with Hk heads, v / g / beta / state with H heads."""
    q, k, v, g, beta, S0 = rand_problem(seed, B=2, T=T, H=H)
    return q[:, :, :Hk].copy(), k[:, :, :Hk].copy(), v, g, beta, S0


def pin_key_heads_single_step(impl):
    """Fewer key heads than value heads, one token from zeros: value head h
    reads key head h % Hk (the tiled mapping of the model card's contract
    notes), so S_1[h] = beta_h v_h k_{h%Hk}^T and o_1[h] = beta_h
    (k_{h%Hk} . q_{h%Hk}) v_h / sqrt(d), written out head by head."""
    for H, Hk in ((4, 2), (6, 3), (4, 1)):
        q, k, v, g, beta, _ = _key_head_problem(30 + H + Hk, H, Hk, 1)
        out, S = impl(q, k, v, g, beta, None)
        d = q.shape[-1]
        for h in range(H):
            j = h % Hk
            b = beta[:, 0, h]
            want_S = b[:, None, None] * np.einsum("bi,bj->bij", v[:, 0, h], k[:, 0, j])
            want_o = (b * np.sum(k[:, 0, j] * q[:, 0, j], axis=-1))[:, None] * v[:, 0, h] / math.sqrt(d)
            if rel(S[:, h], want_S) > 1e-13 or rel(out[:, 0, h], want_o) > 1e-13:
                return False
    return True


def pin_key_heads_tiled_expansion(impl):
    """Fewer key heads equals passing q, k expanded by tiling the head axis
    (heads 0..Hk-1 repeated H/Hk times), over several tokens and a state."""
    H, Hk = 6, 2
    q, k, v, g, beta, S0 = _key_head_problem(40, H, Hk, 5)
    out, S = impl(q, k, v, g, beta, S0)
    qe, ke = np.tile(q, (1, 1, H // Hk, 1)), np.tile(k, (1, 1, H // Hk, 1))
    out_e, S_e = impl(qe, ke, v, g, beta, S0)
    return rel(out, out_e) < 1e-13 and rel(S, S_e) < 1e-13


PINS = [pin_golden_exact, pin_identity, pin_overwrite, pin_forgetting, pin_pure_decay,
        pin_single_step, pin_layout, pin_row_equivariance, pin_linearity, pin_state_carry,
        pin_definition_form, pin_key_heads_single_step, pin_key_heads_tiled_expansion]


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(impl, pin):
    assert pin(IMPLS[impl])


def test_golden_fixture_is_current():
    """The stored fixture equals a fresh exact evaluation of its own inputs."""
    doc = json.load(open(GOLDEN))
    fr = lambda rows: [[Fraction(x) for x in r] for r in rows]
    scaled, S = exact_forward([Fraction(x) for x in doc["alpha"]],
                              [Fraction(x) for x in doc["beta"]],
                              fr(doc["q"]), fr(doc["k"]), fr(doc["v"]), fr(doc["state_in"]))
    assert scaled == fr(doc["out_times_sqrt_d"])
    assert S == fr(doc["state_out"])


def test_c_matches_numpy_twin():
    q, k, v, g, beta, S0 = rand_problem(12, B=3, T=11, H=2, d=16)
    o1, S1 = oracle.recurrent_c(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrent_np(q, k, v, g, beta, S0)
    assert rel(o1, o2) < 1e-13 and rel(S1, S2) < 1e-13


def test_c_matches_numpy_twin_key_heads():
    q, k, v, g, beta, S0 = _key_head_problem(17, 6, 3, 9)
    o1, S1 = oracle.recurrent_c(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrent_np(q, k, v, g, beta, S0)
    assert rel(o1, o2) < 1e-13 and rel(S1, S2) < 1e-13


def test_c_zero_initial_state_pointer():
    q, k, v, g, beta, _ = rand_problem(13)
    o1, S1 = oracle.recurrent_c(q, k, v, g, beta, None)
    o2, S2 = oracle.recurrent_c(q, k, v, g, beta, np.zeros((2, 3, 8, 8)))
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_c_threads_do_not_change_result():
    q, k, v, g, beta, S0 = rand_problem(14, B=4, T=9, H=4, d=16)
    o1, S1 = oracle.recurrent_c(q, k, v, g, beta, S0, n_threads=1)
    o2, S2 = oracle.recurrent_c(q, k, v, g, beta, S0, n_threads=4)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


@pytest.mark.parametrize("chunk", [1, 2, 4, 8, 16, 64])
def test_chunked_algebra_matches_recurrence(chunk):
    """The WY/UT chunk algebra the prefill path uses reproduces the
    recurrence in float64 for every length from 1 to 130 (ragged tails,
    several chunks)."""
    base = rand_problem(15, B=1, T=130, H=2, d=8)
    for T in list(range(1, 20)) + [31, 63, 64, 65, 100, 127, 128, 129, 130]:
        q, k, v, g, beta = (x[:, :T] for x in base[:5])
        S0 = base[5]
        o_r, S_r = oracle.recurrent_np(q, k, v, g, beta, S0)
        o_c, S_c = oracle.chunked_np(q, k, v, g, beta, S0, chunk=chunk)
        assert rel(o_c, o_r) < 1e-12, (T, chunk)
        assert rel(S_c, S_r) < 1e-12, (T, chunk)


def test_chunked_algebra_fast_and_slow_gates():
    for shift in (-3.0, 2.0, 6.0):
        q, k, v, g, beta, S0 = rand_problem(16, B=1, T=150, H=1, d=16, gate_shift=shift)
        o_r, S_r = oracle.recurrent_c(q, k, v, g, beta, S0)
        o_c, S_c = oracle.chunked_np(q, k, v, g, beta, S0, chunk=64)
        assert rel(o_c, o_r) < 1e-11 and rel(S_c, S_r) < 1e-11


# --------------------------------------------------------------------------
# planted mistakes: each broken copy of the recurrence must fail some pin
# --------------------------------------------------------------------------

def _mutant(kind):
    def impl(q, k, v, g, beta, state=None):
        q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
        B, T, H, d = v.shape
        Hk = q.shape[2]
        out = np.zeros((B, T, H, d))
        s_out = np.zeros((B, H, d, d))
        for b in range(B):
            for h in range(H):
                hk = h // (H // Hk) if kind == "grouped_heads" else h % Hk
                S = np.zeros((d, d)) if state is None else np.array(state[b, h], dtype=np.float64)
                for t in range(T):
                    a = np.exp(-g[b, t, h]) if kind == "gate_sign" else np.exp(g[b, t, h])
                    kt, vt, qt, bt = k[b, t, hk], v[b, t, h], q[b, t, hk], beta[b, t, h]
                    if kind == "no_decay":
                        a = 1.0
                    S_old = S
                    if kind != "decay_after":
                        S = a * S
                    Sread = S.T if kind == "transposed" else S
                    r = Sread @ kt
                    if kind == "delta_sign":
                        S = S - bt * np.outer(vt - r, kt)
                    elif kind == "beta_on_v_only":
                        S = S + np.outer(bt * vt - r, kt)
                    elif kind == "outer_swapped":
                        S = S + bt * np.outer(kt, vt - r)
                    elif kind == "no_read":
                        S = S + bt * np.outer(vt, kt)
                    else:
                        S = S + bt * np.outer(vt - r, kt)
                    if kind == "decay_after":
                        S = a * S
                    Semit = S_old if kind == "emit_old_state" else S
                    if kind == "transposed":
                        Semit = Semit.T
                    qq = kt if kind == "emit_with_key" else qt
                    scale = 1.0 if kind == "no_scale" else 1.0 / np.sqrt(d)
                    out[b, t, h] = Semit @ qq * scale
                s_out[b, h] = S
        return out, s_out
    return impl


MUTANTS = ["gate_sign", "no_decay", "decay_after", "transposed", "delta_sign",
           "beta_on_v_only", "outer_swapped", "no_read", "emit_old_state", "emit_with_key",
           "no_scale", "grouped_heads"]


def test_unmutated_copy_passes_every_pin():
    impl = _mutant("none")
    assert all(p(impl) for p in PINS)


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistake_is_caught(kind):
    impl = _mutant(kind)
    with np.errstate(all="ignore"):
        failed = [p.__name__ for p in PINS if not p(impl)]
    assert failed, f"mutant {kind} passed every pin"


# --------------------------------------------------------------------------
# the op's optional fused preprocessing: q and k divided by their Euclidean
# norm per (sequence, token, key head) before the recurrence (a zero vector
# stays zero).  Pinned by facts of the normalisation itself, against the
# plain recurrence that the pins above hold: exactly-unit inputs pass
# through unchanged, a power-of-two rescaling of any q or k changes nothing,
# parallel q and k give the closed-form single step, and zero vectors write
# nothing and read nothing.
# --------------------------------------------------------------------------

def half_unit(shape, seed, zero_every=0):
    """Vectors with four entries of +-1/2 (unit norm exactly in binary
    floating point); with zero_every > 0 every such token is all zeros."""
    r = np.random.default_rng(seed)
    x = np.zeros(shape)
    for idx in np.ndindex(shape[:-1]):
        if zero_every and idx[1] % zero_every == zero_every - 1:
            continue
        pos = r.choice(shape[-1], 4, replace=False)
        x[idx + (pos,)] = r.choice([-0.5, 0.5], 4)
    return x


def pin_norm_unit_inputs_unchanged(impl):
    """Already-unit q and k (and zero vectors) are left as they are: the
    normalised op equals the plain recurrence bit for bit."""
    q, k, v, g, beta, S0 = rand_problem(40, T=9, d=8)
    q, k = half_unit(q.shape, 41, zero_every=4), half_unit(k.shape, 42, zero_every=3)
    o1, S1 = impl(q, k, v, g, beta, S0)
    o2, S2 = oracle.recurrent_np(q, k, v, g, beta, S0)
    return rel(o1, o2) < 1e-14 and rel(S1, S2) < 1e-14 and np.isfinite(o1).all()


def pin_norm_scale_invariance(impl):
    """q and k rescaled by powers of two, a different one per token and head
    (exact in float32), give the same result as the unscaled inputs."""
    q, k, v, g, beta, S0 = rand_problem(43, T=9, d=8, unit=False)
    r = np.random.default_rng(44)
    cq = 2.0 ** r.integers(-6, 7, size=q.shape[:3] + (1,))
    ck = 2.0 ** r.integers(-6, 7, size=k.shape[:3] + (1,))
    o1, S1 = impl(q, k, v, g, beta, S0)
    o2, S2 = impl(q * cq, k * ck, v, g, beta, S0)
    return rel(o1, o2) < 1e-14 and rel(S1, S2) < 1e-14


def pin_norm_parallel_single_step(impl):
    """From a zero state, one token with q = a u and k = c u (the same
    direction u, any positive a, c): S = beta v u^T / |u| and o = beta v /
    sqrt(d) exactly, since the unit key and query meet at 1."""
    _, _, v, g, beta, _ = rand_problem(45, T=1, d=8)
    r = np.random.default_rng(46)
    u = r.standard_normal(v.shape).astype(np.float32).astype(np.float64)
    a = 2.0 ** r.integers(-3, 4, size=v.shape[:3] + (1,))
    c = 2.0 ** r.integers(-3, 4, size=v.shape[:3] + (1,))
    out, S = impl(u * a, u * c, v, g, beta, None)
    d = v.shape[-1]
    want_o = beta[..., None] * v / math.sqrt(d)
    un = u / np.linalg.norm(u, axis=-1, keepdims=True)
    want_S = beta[:, 0, :, None, None] * v[:, 0, :, :, None] * un[:, 0, :, None, :]
    return rel(out, want_o) < 1e-13 and rel(S, want_S) < 1e-13


NORM_PINS = [pin_norm_unit_inputs_unchanged, pin_norm_scale_invariance,
             pin_norm_parallel_single_step]


def c_norm(q, k, v, g, beta, S0):
    return oracle.recurrent_c(q, k, v, g, beta, S0, l2norm_qk=True)


def np_norm(q, k, v, g, beta, S0):
    return oracle.recurrent_np(q, k, v, g, beta, S0, l2norm_qk=True)


NORM_IMPLS = {"c": c_norm, "numpy": np_norm}


@pytest.mark.parametrize("impl", list(NORM_IMPLS))
@pytest.mark.parametrize("pin", NORM_PINS, ids=lambda p: p.__name__)
def test_oracle_norm_pin(impl, pin):
    assert pin(NORM_IMPLS[impl])


def test_norm_c_matches_numpy_twin_key_heads():
    q, k, v, g, beta, S0 = _key_head_problem(47, 6, 3, 9)
    q, k = q * 4.0, k * 0.25                     # exact in float32
    o1, S1 = oracle.recurrent_c(q, k, v, g, beta, S0, l2norm_qk=True)
    o2, S2 = oracle.recurrent_np(q, k, v, g, beta, S0, l2norm_qk=True)
    assert rel(o1, o2) < 1e-13 and rel(S1, S2) < 1e-13


def _norm_mutant(kind):
    def nrm(x, axis=-1, power=0.5):
        n = np.sum(x * x, axis=axis, keepdims=True) ** power
        if kind == "zero_to_nan":
            return x / n
        return np.divide(x, n, out=np.zeros_like(x), where=n > 0)

    def impl(q, k, v, g, beta, S0):
        q, k = np.asarray(q, dtype=np.float64), np.asarray(k, dtype=np.float64)
        if kind in ("none", "zero_to_nan"):
            q, k = nrm(q), nrm(k)
        elif kind == "q_only":
            q = nrm(q)
        elif kind == "k_only":
            k = nrm(k)
        elif kind == "squared_norm":
            q, k = nrm(q, power=1.0), nrm(k, power=1.0)
        elif kind == "over_heads":
            q, k = nrm(q, axis=2), nrm(k, axis=2)
        elif kind == "k_norm_for_both":
            n = np.sqrt(np.sum(k * k, axis=-1, keepdims=True))
            q, k = q / n, k / n
        return oracle.recurrent_np(q, k, v, g, beta, S0)
    return impl


NORM_MUTANTS = ["skip", "q_only", "k_only", "squared_norm", "over_heads", "zero_to_nan",
                "k_norm_for_both"]


def test_unmutated_norm_copy_passes_every_norm_pin():
    impl = _norm_mutant("none")
    assert all(p(impl) for p in NORM_PINS)


@pytest.mark.parametrize("kind", NORM_MUTANTS)
def test_planted_norm_mistake_is_caught(kind):
    impl = _norm_mutant(kind)
    with np.errstate(all="ignore"):
        failed = [p.__name__ for p in NORM_PINS if not p(impl)]
    assert failed, f"mutant {kind} passed every normalisation pin"
