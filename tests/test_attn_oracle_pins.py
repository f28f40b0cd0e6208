"""Pins for the float64 decode-attention oracle (CPU only).

The oracle (oracle/attn.py) is pinned to facts that do not come from it:
closed forms of softmax attention (one key, two keys as a logistic weight,
equal scores, a single unmasked key), invariances (a constant added to a row
of the mask, scale folded into q), the grouped query-head -> kv-head mapping
written out head by head, and a 50-digit brute force with mpmath on tiny
inputs.  The last tests plant plausible mistakes in a copy of the oracle and
check that at least one pin catches each.

Definition ("marcsun13/ggml-gated-delta-net" model card, section
"flash_attn"): out[b, i, h] = softmax_j(scale q[b,h,i] . k[b,hk,j] +
mask[b,0,i,j]) v[b,hk,:], hk = h // (n_heads / n_heads_kv), result shaped
(n_seqs, n_q, n_heads, head_dim).
"""
import math

import numpy as np
import pytest

from oracle.attn import attention


def problem(seed, B=2, H=4, Hkv=2, n_q=3, n_kv=5, d=8, mask=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, n_q, d))
    k = r.standard_normal((B, Hkv, n_kv, d))
    v = r.standard_normal((B, Hkv, n_kv, d))
    m = r.standard_normal((B, 1, n_q, n_kv)) if mask else None
    return q, k, v, m


def rel(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) / max(1e-300, float(np.max(np.abs(b))))


def pin_single_key(impl):
    """One key: the softmax weight is 1, every output row is that key's v."""
    q, k, v, m = problem(1, n_kv=1)
    out = impl(q, k, v, m, 0.7)
    rep = q.shape[1] // k.shape[1]
    for h in range(q.shape[1]):
        for i in range(q.shape[2]):
            if rel(out[:, i, h], v[:, h // rep, 0]) > 1e-15:
                return False
    return True


def pin_two_keys_logistic(impl):
    """Two keys: weight of key 0 is the logistic 1 / (1 + exp(s1 - s0))."""
    q, k, v, m = problem(2, B=1, H=2, Hkv=1, n_q=2, n_kv=2)
    scale = 0.4
    out = impl(q, k, v, m, scale)
    for h in range(2):
        for i in range(2):
            s = [scale * sum(q[0, h, i, e] * k[0, 0, j, e] for e in range(q.shape[-1])) + m[0, 0, i, j]
                 for j in range(2)]
            w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
            want = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 0, 1]
            if rel(out[0, i, h], want) > 1e-14:
                return False
    return True


def pin_equal_scores_mean(impl):
    """scale 0 and no mask: all scores equal, the output is the mean of v."""
    q, k, v, _ = problem(3)
    out = impl(q, k, v, None, 0.0)
    want = v.mean(axis=2)                                   # (B, Hkv, d)
    rep = q.shape[1] // k.shape[1]
    return all(rel(out[:, i, h], want[:, h // rep]) < 1e-14
               for h in range(q.shape[1]) for i in range(q.shape[2]))


def pin_single_unmasked_key(impl):
    """-inf on every key but j*: the output is v[j*]."""
    q, k, v, _ = problem(4, n_kv=6)
    B, _, n_q, n_kv = q.shape[0], 0, q.shape[2], k.shape[2]
    m = np.full((B, 1, n_q, n_kv), -np.inf)
    js = [(b * 3 + i) % n_kv for b in range(B) for i in range(n_q)]
    for b in range(B):
        for i in range(n_q):
            m[b, 0, i, js[b * n_q + i]] = 0.0
    out = impl(q, k, v, m, 1.3)
    rep = q.shape[1] // k.shape[1]
    for b in range(B):
        for i in range(n_q):
            for h in range(q.shape[1]):
                if rel(out[b, i, h], v[b, h // rep, js[b * n_q + i]]) > 1e-15:
                    return False
    return True


def pin_row_shift_invariance(impl):
    """Adding a constant to one query row of the mask leaves the output unchanged."""
    q, k, v, m = problem(5)
    out = impl(q, k, v, m, 0.5)
    m2 = m + np.arange(m.shape[2])[None, None, :, None] * 3.25 - 7.0
    return rel(impl(q, k, v, m2, 0.5), out) < 1e-13


def pin_scale_into_q(impl):
    """scale s with q equals scale 1 with s q."""
    q, k, v, m = problem(6)
    return rel(impl(q, k, v, m, 0.375), impl(0.375 * q, k, v, m, 1.0)) < 1e-13


def pin_large_scores(impl):
    """Scores near 1000 (exp overflows in float64 without the row maximum
    taken out) still give the softmax: two keys 2 apart weigh 1 : e^-2."""
    q, k, v, _ = problem(7, B=1, H=1, Hkv=1, n_q=1, n_kv=2)
    m = np.array([[[[1000.0, 998.0]]]])
    out = impl(q * 0.0, k, v, m, 1.0)
    w0 = 1.0 / (1.0 + math.exp(-2.0))
    return rel(out[0, 0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1]) < 1e-14


def pin_empty_and_fully_masked(impl):
    """n_kv == 0 and an all -inf mask row give zero rows (the reading taken
    where the page is silent); other rows are unaffected."""
    q, k, v, m = problem(8)
    out0 = impl(q, k[:, :, :0], v[:, :, :0], m[..., :0], 1.0)
    if out0.shape != (q.shape[0], q.shape[2], q.shape[1], v.shape[-1]) or np.any(out0 != 0):
        return False
    m2 = m.copy()
    m2[0, 0, 1, :] = -np.inf
    out = impl(q, k, v, m2, 1.0)
    ref = impl(q, k, v, m, 1.0)
    return np.all(out[0, 1] == 0) and rel(out[1], ref[1]) < 1e-15 and rel(out[0, 0], ref[0, 0]) < 1e-15


def pin_mpmath_brute_force(impl):
    """50-digit evaluation of the definition with explicit loops (mpmath)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    q, k, v, m = problem(9, B=1, H=4, Hkv=2, n_q=2, n_kv=4, d=4)
    scale = 0.6
    out = impl(q, k, v, m, scale)
    rep = 2
    for h in range(4):
        for i in range(2):
            hk = h // rep
            s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[0, h, i, e]) * mpmath.mpf(k[0, hk, j, e])
                                                  for e in range(4)) + mpmath.mpf(m[0, 0, i, j])
                 for j in range(4)]
            w = [mpmath.e ** x for x in s]
            tot = mpmath.fsum(w)
            for c in range(4):
                want = mpmath.fsum(w[j] * mpmath.mpf(v[0, hk, j, c]) for j in range(4)) / tot
                if abs(float(want) - out[0, i, h, c]) > 1e-14 * max(1.0, abs(float(want))):
                    return False
    return True


PINS = [pin_single_key, pin_two_keys_logistic, pin_equal_scores_mean, pin_single_unmasked_key,
        pin_row_shift_invariance, pin_scale_into_q, pin_large_scores, pin_empty_and_fully_masked,
        pin_mpmath_brute_force]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_attention_oracle_pin(pin):
    assert pin(attention)


# --------------------------------------------------------------------------
# planted mistakes
# --------------------------------------------------------------------------

def _mutant(kind):
    def impl(q, k, v, mask=None, scale=None):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, n_q, dk = q.shape
        Hkv, n_kv, dv = k.shape[1], k.shape[2], v.shape[3]
        rep = H // Hkv
        scale = 1.0 / np.sqrt(dk) if scale is None else scale
        out = np.zeros((B, n_q, H, dv))
        for b in range(B):
            for h in range(H):
                hk = h % Hkv if kind == "tiled_heads" else h // rep
                hv = h % Hkv if kind == "v_head_tiled" else hk
                for i in range(n_q):
                    if n_kv == 0:
                        continue
                    sc = 1.0 if kind == "no_scale" else scale
                    s = sc * (k[b, hk] @ q[b, h, i])
                    if mask is not None and kind != "mask_ignored":
                        s = s + (mask[b, 0, 0] if kind == "mask_row0" else mask[b, 0, i])
                    top = 0.0 if kind == "no_max" else np.max(s)
                    if top == -np.inf:
                        continue
                    e = np.exp(s - top)
                    wts = e if kind == "unnormalised" else e / np.sum(e)
                    out[b, i, h] = wts @ v[b, hv]
        return out
    return impl


MUTANTS = ["tiled_heads", "v_head_tiled", "no_scale", "mask_ignored", "mask_row0", "no_max",
           "unnormalised"]


def test_unmutated_copy_passes_every_pin():
    assert all(p(_mutant("none")) for p in PINS)


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistake_is_caught(kind):
    impl = _mutant(kind)
    with np.errstate(all="ignore"):
        failed = [p.__name__ for p in PINS if not p(impl)]
    assert failed, f"mutant {kind} passed every pin"
