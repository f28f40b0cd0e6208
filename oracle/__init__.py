"""Oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches the product path:
the two share no code, headers, tables or helpers.

Contents
--------
``recurrent_c``      the float64 token-by-token recurrence in plain C
                     (``gdn_oracle.c``), OpenMP over (sequence, head) pairs.
``recurrent_np``     the same recurrence in numpy, float64, for tiny cases and
                     as an independent twin of the C code.
``l2_normalize``     x / |x| per vector in float64 (zero stays zero): the
                     op's optional fused q / k preprocessing, which both
                     recurrences above apply when asked (``l2norm_qk``).
``chunked_np``       a float64 chunked (WY / UT-transform) evaluation of the
                     same recurrence, used only to check the chunk algebra
                     that the CUDA prefill path relies on against the
                     recurrence itself on tiny inputs.

Definition followed (see ``gdn_oracle.c`` for the step-by-step form):
S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t / sqrt(d), state indexed [value][key].
Sources: "Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention LLMs",
section "What Gated Delta Net is, in plain language" (delta rule overwrites,
the gate scales what is kept); "marcsun13/ggml-gated-delta-net" model card,
section "Ops" and its shape table (signature, shapes, [value][key] state,
zeros as the fresh state, identity key-head mapping, 1/sqrt(head_dim) on the
output, log-domain gate exponentiated by the op).  With fewer key heads than
value heads (q, k carrying n_k heads), value head h reads key head h % n_k:
the tiled convention the same model card's contract notes give for upstream.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into a shared library beside it (gcc, -O2, OpenMP,
    no fast-math, no machine-specific flags) and return its path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = lib.gdn_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 7
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def recurrent_c(q, k, v, g, beta, state=None, n_threads: int = 0, l2norm_qk: bool = False):
    """float64 recurrence in C.  q, k: (B, T, Hk, d); v: (B, T, H, d); g, beta:
    (B, T, H); state: (B, H, d, d) [value][key] or None for zeros; value head
    h reads key head h % Hk (Hk == H: identity).  Inputs are taken as float32
    (exact for bf16 data).  l2norm_qk: q and k are first divided by their
    Euclidean norm per (sequence, token, key head), in float64 (a zero vector
    stays zero).  Returns (out (B,T,H,d), state_out (B,H,d,d)), both
    float64."""
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    B, T, H, d = v.shape
    Hk = q.shape[2]
    assert k.shape == q.shape and q.shape == (B, T, Hk, d) and 1 <= Hk <= max(H, 1)
    assert g.shape == (B, T, H) and beta.shape == (B, T, H)
    st = None if state is None else _f32(state)
    if st is not None:
        assert st.shape == (B, H, d, d)
    out = np.empty((B, T, H, d), dtype=np.float64)
    s_out = np.empty((B, H, d, d), dtype=np.float64)
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = _load().gdn_oracle_forward(p(q), p(k), p(v), p(g), p(beta), p(st), p(out), p(s_out),
                                    B, T, H, Hk, d, int(n_threads), int(bool(l2norm_qk)))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_forward failed ({rc})")
    return out, s_out


def l2_normalize(x):
    """x / |x| over the last axis in float64; an all-zero vector stays zero."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.divide(x, n, out=np.zeros_like(x), where=n > 0)


def recurrent_np(q, k, v, g, beta, state=None, l2norm_qk: bool = False):
    """The same float64 recurrence in numpy, token by token:
    decay, read r = S k, overwrite S += beta (v - r) k^T, emit S q / sqrt(d).
    q, k may carry fewer heads (Hk) than v: value head h reads key head h % Hk.
    l2norm_qk: q and k are first replaced by l2_normalize(q), l2_normalize(k)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    if l2norm_qk:
        q, k = l2_normalize(q), l2_normalize(k)
    B, T, H, d = v.shape
    Hk = q.shape[2]
    out = np.zeros((B, T, H, d))
    s_out = np.zeros((B, H, d, d))
    for b in range(B):
        for h in range(H):
            hk = h % Hk
            S = np.zeros((d, d)) if state is None else np.array(state[b, h], dtype=np.float64)
            for t in range(T):
                S = np.exp(g[b, t, h]) * S
                r = S @ k[b, t, hk]
                S = S + beta[b, t, h] * np.outer(v[b, t, h] - r, k[b, t, hk])
                out[b, t, h] = S @ q[b, t, hk] / np.sqrt(d)
            s_out[b, h] = S
    return out, s_out


def chunked_np(q, k, v, g, beta, state=None, chunk: int = 64):
    """float64 chunked evaluation of the same recurrence (test-only).

    Within a chunk of n tokens starting from state S0, write G_r for the
    inclusive running sum of g inside the chunk and u_r = beta_r (v_r -
    exp(g_r) S_{r-1} k_r) for the correction each token writes.  Unrolling
    S_r = exp(g_r) S_{r-1} + u_r k_r^T gives
        S_r = exp(G_r) S0 + sum_{i<=r} exp(G_r - G_i) u_i k_i^T,
    and substituting back into the definition of u_r gives a unit
    lower-triangular system for the rows u_r:
        (I + A) U = diag(beta) V - diag(beta exp(G)) K S0^T,
        A[r, i] = beta_r exp(G_r - G_i) (k_r . k_i)   for i < r.
    With T = (I + A)^-1 (the UT transform of the chunk):
        U   = T (diag(beta) V - diag(beta exp(G)) K S0^T)
        O   = (diag(exp(G)) Q S0^T + P U) / sqrt(d),
              P[r, i] = exp(G_r - G_i) (q_r . k_i)  for i <= r
        S_n = exp(G_{n-1}) S0 + (diag(exp(G_{n-1} - G)) U)^T K.
    The last chunk may be shorter than ``chunk``.
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, d = q.shape
    out = np.zeros((B, T, H, d))
    s_out = np.zeros((B, H, d, d))
    for b in range(B):
        for h in range(H):
            S = np.zeros((d, d)) if state is None else np.array(state[b, h], dtype=np.float64)
            for s in range(0, T, chunk):
                e = min(T, s + chunk)
                n = e - s
                Q, K, V = q[b, s:e, h], k[b, s:e, h], v[b, s:e, h]
                bt = beta[b, s:e, h]
                G = np.cumsum(g[b, s:e, h])
                D = G[:, None] - G[None, :]                      # G_r - G_i
                lower = np.tril(np.ones((n, n), dtype=bool), -1)  # i < r
                A = np.where(lower, bt[:, None] * np.exp(np.where(lower, D, 0.0)) * (K @ K.T), 0.0)
                Tm = np.linalg.inv(np.eye(n) + A)
                R = bt[:, None] * V - (bt * np.exp(G))[:, None] * (K @ S.T)
                U = Tm @ R
                incl = np.tril(np.ones((n, n), dtype=bool), 0)   # i <= r
                P = np.where(incl, np.exp(np.where(incl, D, 0.0)) * (Q @ K.T), 0.0)
                out[b, s:e, h] = (np.exp(G)[:, None] * (Q @ S.T) + P @ U) / np.sqrt(d)
                S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * U).T @ K
            s_out[b, h] = S
    return out, s_out


def parity_error(x, ref, abs_floor: float = 1e-6) -> float:
    """max |x - ref| / RMS(ref) over the whole tensor (the parity metric).
    When RMS(ref) is 0 the absolute max error divided by ``abs_floor`` is
    returned, so a bound of 1 then means |err| <= abs_floor."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return err / rms if rms > 0 else err / abs_floor
