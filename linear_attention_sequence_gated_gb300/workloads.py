"""Seeded synthetic inputs for the gated delta rule.

This module only draws random inputs; it holds none of the recurrence's
arithmetic, so the CUDA path and the float64 oracle can both be fed from it.

The workloads follow the shapes the "marcsun13/ggml-gated-delta-net" model
card measures on (section "Measured": 32 value heads, head_dim 128, one
token per step, 24 layers) plus batched decode and long prefill of the same
head geometry.  Distributions:
  q, k   ~ N(0, 1), then L2-normalised per (sequence, token, head) in fp32
  v      ~ N(0, 1)
  beta   = sigmoid(N(0, 1))
  g      = -softplus(N(0, 1) + gate_shift)   (log-domain gate, always <= 0)
  state  ~ N(0, state_std) fp32, [value][key]; state_std 0 means zeros
q, k, v are cast to the workload dtype (bf16 or fp32) after normalisation;
g, beta and the state stay fp32.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                # n_seqs
    T: int                # n_tokens
    H: int                # n_heads (value heads)
    d: int                # head_dim
    dtype: str            # "f32" or "bf16" for q, k, v
    gate_shift: float     # g = -softplus(N(0,1) + gate_shift)
    state_std: float      # 0 -> zero initial state
    layers: int = 1       # independent layers (distinct states) per step
    seed: int = 0
    Hk: int = 0           # heads of q and k (0: one per value head); divides H

    @property
    def n_k(self) -> int:
        return self.Hk or self.H

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny_b1_t64_h4_d32_f32", 1, 64, 4, 32, "f32", 0.0, 0.0, seed=0)
DECODE_24L = Workload("decode_b1_h32_d128_bf16_24layers", 1, 1, 32, 128, "bf16", 0.0, 0.02,
                      layers=24, seed=1)
DECODE_B64 = Workload("decode_b64_h32_d128_bf16", 64, 1, 32, 128, "bf16", 0.0, 0.02, seed=2)
PREFILL_4K = Workload("prefill_b1_t4096_h32_d128_bf16", 1, 4096, 32, 128, "bf16", 2.0, 0.0, seed=3)
PREFILL_16K = Workload("prefill_b8_t16384_h32_d128_bf16", 8, 16384, 32, 128, "bf16", 2.0, 0.02,
                       seed=4)
PREFILL_16K_D64 = PREFILL_16K.replace(name="prefill_b8_t16384_h64_d64_bf16", H=64, d=64, seed=5)
PREFILL_16K_D256 = PREFILL_16K.replace(name="prefill_b8_t16384_h16_d256_bf16", H=16, d=256, seed=6)
# a short run of tokens per sequence (multi-token / speculative decode)
MULTITOKEN_B64_T4 = Workload("multitoken_b64_t4_h32_d128_bf16", 64, 4, 32, 128, "bf16", 0.0, 0.02,
                             seed=7)
# fewer key heads than value heads (16 q/k heads shared by 32 value heads)
DECODE_B64_HK16 = Workload("decode_b64_h32_hk16_d128_bf16", 64, 1, 32, 128, "bf16", 0.0, 0.02,
                           seed=8, Hk=16)

ALL = [TINY, DECODE_24L, DECODE_B64, PREFILL_4K, PREFILL_16K, PREFILL_16K_D64, PREFILL_16K_D256,
       MULTITOKEN_B64_T4, DECODE_B64_HK16]
BY_NAME = {w.name: w for w in ALL}


def _gen(seed: int, device):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def make_inputs(w: Workload, device="cpu", layer: int = 0, B: int | None = None,
                T: int | None = None, seed: int | None = None):
    """Draw one layer's inputs for workload ``w`` on ``device``.

    Returns a dict with q, k (B, T, Hk, d) and v (B, T, H, d) in the workload
    dtype, g, beta (B, T, H) fp32 and state (B, H, d, d) fp32 or None.  ``B``/``T`` override
    the workload's sizes (same distributions), ``layer`` selects one of the
    workload's independent layers."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    s = (w.seed if seed is None else seed) * 1000 + layer
    gen = _gen(s, device)
    H, d = w.H, w.d
    shape = (B, T, H, d)
    qk_shape = (B, T, w.n_k, d)
    q = torch.randn(qk_shape, generator=gen, device=device, dtype=torch.float32)
    k = torch.randn(qk_shape, generator=gen, device=device, dtype=torch.float32)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen, device=device))
    g = -torch.nn.functional.softplus(
        torch.randn((B, T, H), generator=gen, device=device) + w.gate_shift)
    state = None
    if w.state_std > 0:
        state = torch.randn((B, H, d, d), generator=gen, device=device) * w.state_std
    dt = w.torch_dtype
    return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
            "g": g.contiguous(), "beta": beta.contiguous(), "state": state}


def to_numpy_f32(inputs):
    """fp32 numpy copies (exact for bf16) of a ``make_inputs`` dict."""
    out = {}
    for key, val in inputs.items():
        out[key] = None if val is None else val.detach().float().cpu().numpy()
    return out


# ------------------------------------------------------------------ decode attention

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Decode attention: q (B, H, n_q, d); k (B, Hkv, n_kv, d); v (B, Hkv,
    n_kv, dv), dv = d unless given; optional
    additive mask (B, 1, n_q, n_kv).  q, k, v ~ N(0, 1); the mask, when
    present, is 0 on visible keys and -inf on the last ``masked_tail`` keys
    of each query row shifted by the query index (a causal tail, as when the
    queries are the newest tokens of the cache), plus N(0, mask_std)."""
    name: str
    B: int
    H: int
    Hkv: int
    n_q: int
    n_kv: int
    d: int
    dtype: str            # "f32", "bf16" or "f16" for q, k, v and the mask
    mask: bool = False
    masked_tail: int = 0
    mask_std: float = 0.0
    seed: int = 0
    dv_: int = 0          # head_dim of v when it differs from q / k's (0: same as d)

    @property
    def dv(self) -> int:
        return self.dv_ or self.d

    @property
    def torch_dtype(self):
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    def replace(self, **kw) -> "AttnWorkload":
        return dataclasses.replace(self, **kw)


# the shape timed on the model card (section "Measured": 16 query heads over 4
# kv heads, head_dim 256, one query) at its two cache lengths
ATTN_KV512 = AttnWorkload("attn_b1_h16_kv4_q1_n512_d256_bf16", 1, 16, 4, 1, 512, 256, "bf16",
                          seed=20)
ATTN_KV141 = ATTN_KV512.replace(name="attn_b1_h16_kv4_q1_n141_d256_bf16", n_kv=141, seed=21)
# batched decode over a long cache: the cache streams from HBM
ATTN_B64_KV4K = AttnWorkload("attn_b64_h32_kv8_q1_n4096_d128_bf16", 64, 32, 8, 1, 4096, 128,
                             "bf16", seed=22)

ATTN_ALL = [ATTN_KV512, ATTN_KV141, ATTN_B64_KV4K]
ATTN_BY_NAME = {w.name: w for w in ATTN_ALL}


def make_attn_inputs(w: AttnWorkload, device="cpu", seed: int | None = None):
    """q, k, v (and mask or None) for ``w`` on ``device``, in the workload dtype."""
    gen = _gen((w.seed if seed is None else seed) * 1000 + 7, device)
    f = dict(generator=gen, device=device, dtype=torch.float32)
    q = torch.randn((w.B, w.H, w.n_q, w.d), **f)
    k = torch.randn((w.B, w.Hkv, w.n_kv, w.d), **f)
    v = torch.randn((w.B, w.Hkv, w.n_kv, w.dv), **f)
    mask = None
    if w.mask:
        mask = torch.randn((w.B, 1, w.n_q, w.n_kv), **f) * w.mask_std
        if w.masked_tail > 0:
            j = torch.arange(w.n_kv, device=device)[None, :]
            i = torch.arange(w.n_q, device=device)[:, None]
            hidden = j >= (w.n_kv - w.masked_tail + i)
            mask = mask.masked_fill(hidden[None, None], float("-inf"))
    dt = w.torch_dtype
    return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
            "mask": None if mask is None else mask.to(dt).contiguous()}
