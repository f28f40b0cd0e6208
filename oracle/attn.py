"""Oracle for decode attention (the flash_attn op) -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` may import this module; the product path never does, and this
module imports nothing from the product.

What it computes, in float64, straight from the definition of softmax
attention ("marcsun13/ggml-gated-delta-net" model card, section
"flash_attn": its shape table, the note that grouped-query attention is
native with k and v carrying n_heads_kv heads, the additive mask of shape
(n_seqs, 1, n_q, n_kv) and the (n_seqs, n_q, n_heads, head_dim) result):

    for every sequence b, query head h, query i:
        hk      = h // (n_heads / n_heads_kv)          (grouped heads, as repeat_kv)
        s_j     = scale * (q[b, h, i] . k[b, hk, j]) + mask[b, 0, i, j]
        p_j     = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
        out[b, i, h] = sum_j p_j v[b, hk, j]

Readings where the page is silent: a row whose scores are all -inf (every key
masked), and n_kv == 0, give a zero output row; the result is float64 (the
kernel's own accumulation precision is its choice).
"""
from __future__ import annotations

import numpy as np


def attention(q, k, v, mask=None, scale=None):
    """q: (B, H, n_q, dk); k: (B, Hkv, n_kv, dk); v: (B, Hkv, n_kv, dv);
    mask: (B, 1, n_q, n_kv) additive or None; scale: float or None for
    1/sqrt(dk).  Returns out (B, n_q, H, dv) float64."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, n_q, dk = q.shape
    Hkv, n_kv, dv = k.shape[1], k.shape[2], v.shape[3]
    assert k.shape == (B, Hkv, n_kv, dk) and v.shape == (B, Hkv, n_kv, dv)
    assert H % Hkv == 0
    rep = H // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    m = None if mask is None else np.asarray(mask, dtype=np.float64)
    if m is not None:
        assert m.shape == (B, 1, n_q, n_kv)
    out = np.zeros((B, n_q, H, dv))
    for b in range(B):
        for h in range(H):
            hk = h // rep
            for i in range(n_q):
                if n_kv == 0:
                    continue
                s = scale * (k[b, hk] @ q[b, h, i])
                if m is not None:
                    s = s + m[b, 0, i]
                top = np.max(s)
                if top == -np.inf:
                    continue
                e = np.exp(s - top)
                out[b, i, h] = (e / np.sum(e)) @ v[b, hk]
    return out
