"""GB300 (sm_103a) gated delta rule: Python binding of libgdn.so.

This module only marshals arguments: it checks torch tensors, takes their
device pointers and the current CUDA stream, and calls the C ABI declared in
``include/gdn.h``.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If ``libgdn.so`` has not been
built (``python -m linear_attention_sequence_gated_gb300._build``) every
call raises.

    out, final_state = forward(q, k, v, g, beta, state)

q, k, v: (n_seqs, n_tokens, n_heads, head_dim) bf16 or fp32 CUDA tensors,
g, beta: (n_seqs, n_tokens, n_heads) fp32, state: (n_seqs, n_heads, head_dim,
head_dim) fp32 [value][key] or None (zeros).  out is fp32 and already carries
1/sqrt(head_dim).  ("marcsun13/ggml-gated-delta-net" model card, section
"Ops" and its shape table.)  q and k may carry fewer heads n_k (dividing
n_heads): value head i then reads key head i % n_k, the tiled mapping of the
model card's contract notes.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

OK = 0
ERR_ARG, ERR_HEADDIM, ERR_ALIGN, ERR_ALIAS, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_NOMEM, \
    ERR_DTYPE, ERR_SHAPE, ERR_SCRATCH = -1, -2, -3, -4, -5, -6, -7, -8, -9, -10, -11
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2
PATHS = {"auto": 0, "recurrent": 1, "chunked": 2}
OPT_L2NORM_QK = 0x100
OPT_OUT_BF16 = 0x200

# Every symbol include/gdn.h declares.
EXPORTS = ["gdn_forward", "gdn_forward_bf16", "gdn_forward_ex", "gdn_workspace_bytes",
           "gdn_select_path", "gdn_supports", "gdn_get_device_status", "gdn_status_string",
           "gdn_version", "gdn_flash_attn", "gdn_flash_attn_supports", "gdn_forward_noalloc",
           "gdn_selftest_wait_timeout"]

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str = "gdn"):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


def lib():
    """The loaded libgdn.so (ctypes), raising if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libgdn.so not found at {LIB_PATH}; build it with "
                "`python -m linear_attention_sequence_gated_gb300._build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        fwd = [vp, vp, vp, fp, fp, fp, fp, fp, i, i, i, i]
        L.gdn_forward.argtypes = fwd + [vp]
        L.gdn_forward_bf16.argtypes = fwd + [vp]
        L.gdn_forward_ex.argtypes = fwd[:11] + [i, i, i, i, vp, sz, vp]
        for f in (L.gdn_forward, L.gdn_forward_bf16, L.gdn_forward_ex):
            f.restype = i
        L.gdn_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.gdn_workspace_bytes.restype = sz
        L.gdn_select_path.argtypes = [i, i, i, i, i]
        L.gdn_select_path.restype = i
        L.gdn_supports.argtypes = [i]
        L.gdn_supports.restype = i
        L.gdn_get_device_status.argtypes = [vp]
        L.gdn_get_device_status.restype = i
        L.gdn_status_string.argtypes = [i]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_version.restype = i
        L.gdn_flash_attn.argtypes = [vp, vp, vp, vp, fp] + [i] * 7 + [ctypes.c_float, i, vp]
        L.gdn_flash_attn.restype = i
        L.gdn_flash_attn_supports.argtypes = [i, i, i]
        L.gdn_flash_attn_supports.restype = i
        L.gdn_forward_noalloc.argtypes = fwd[:11] + [i, i, i, i, vp]
        L.gdn_forward_noalloc.restype = i
        L.gdn_selftest_wait_timeout.argtypes = [vp]
        L.gdn_selftest_wait_timeout.restype = i
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def supports(head_dim: int) -> int:
    """Bit mask: 1 = recurrent path, 2 = chunked path, 0 = unsupported."""
    return int(lib().gdn_supports(int(head_dim)))


def select_path(n_seqs: int, n_tokens: int, n_heads: int, head_dim: int,
                dtype: str = "bf16") -> str:
    """The path AUTO takes for these sizes: "recurrent" or "chunked"."""
    dt = DTYPE_BF16 if dtype in ("bf16", "bfloat16") else DTYPE_F32
    r = int(lib().gdn_select_path(int(n_seqs), int(n_tokens), int(n_heads), int(head_dim), dt))
    if r < 0:
        raise GdnError(r, "gdn_select_path")
    return {v: k for k, v in PATHS.items()}[r]


def workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, dtype="bf16", path="auto") -> int:
    dt = DTYPE_BF16 if dtype in ("bf16", "bfloat16") else DTYPE_F32
    return int(lib().gdn_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, dt, PATHS[path]))


def device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status word."""
    return int(lib().gdn_get_device_status(_stream_handle(stream)))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def forward(q, k, v, g, beta, state=None, *, out=None, state_out=None, path: str = "auto",
            workspace=None, stream=None, l2norm_qk: bool = False, out_dtype=None):
    """Run the gated delta rule over every token of every sequence.

    Returns (out, final_state).  ``state_out`` may be ``state`` itself for
    an in-place update.  ``workspace`` is an optional uint8 CUDA tensor of at
    least ``workspace_bytes(...)`` bytes; without it the library allocates
    stream-ordered scratch when the chosen path needs any.  ``l2norm_qk``
    divides q and k by their norm per (sequence, token, head) inside the op
    (the library's GDN_OPT_L2NORM_QK).  ``out_dtype`` torch.bfloat16 writes
    the output as bf16, each value the fp32 one rounded to nearest even
    (GDN_OPT_OUT_BF16); a given ``out`` must have that dtype.  The default is
    fp32, or the dtype of a given ``out``."""
    import torch
    L = lib()
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError(f"q/k/v must be bf16 or fp32, got {q.dtype}")
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be (n_seqs, n_tokens, heads, head_dim)")
    B, T, H, d = v.shape
    Hk = q.shape[2]
    if tuple(q.shape) != (B, T, Hk, d) or Hk < 1 or H % Hk != 0:
        raise ValueError(f"q: expected (n_seqs, n_tokens, n_k, head_dim) with n_k dividing "
                         f"{H}, got {tuple(q.shape)}")
    for name, t, shape, dtype in (("k", k, (B, T, Hk, d), q.dtype), ("v", v, (B, T, H, d), q.dtype),
                                  ("g", g, (B, T, H), torch.float32),
                                  ("beta", beta, (B, T, H), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name}: expected {shape} {dtype}, got {tuple(t.shape)} {t.dtype}")
    tensors = [q, k, v, g, beta]
    if state is not None:
        if tuple(state.shape) != (B, H, d, d) or state.dtype != torch.float32:
            raise ValueError("state must be (n_seqs, n_heads, head_dim, head_dim) fp32")
        tensors.append(state)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"out_dtype must be float32 or bfloat16, got {out_dtype}")
    if out is None:
        out = torch.empty((B, T, H, d), dtype=out_dtype, device=q.device)
    if state_out is None:
        state_out = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device)
    tensors += [out, state_out]
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
        if t.device != q.device:
            raise ValueError("all tensors must be on one CUDA device")
    if tuple(out.shape) != (B, T, H, d) or out.dtype != out_dtype:
        raise ValueError(f"out must be (n_seqs, n_tokens, n_heads, head_dim) {out_dtype}")
    if tuple(state_out.shape) != (B, H, d, d) or state_out.dtype != torch.float32:
        raise ValueError("state_out must be (n_seqs, n_heads, head_dim, head_dim) fp32")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    with torch.cuda.device(q.device):
        rc = L.gdn_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                              _ptr(out), _ptr(state_out), B, T, H, Hk, d, dt,
                              PATHS[path] | (OPT_L2NORM_QK if l2norm_qk else 0)
                              | (OPT_OUT_BF16 if out_dtype == torch.bfloat16 else 0),
                              ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != OK:
        raise GdnError(rc, "gdn_forward_ex")
    return out, state_out


def flash_attn_supports(n_q: int, head_dim_k: int, head_dim_v: int) -> bool:
    """Whether ``flash_attn`` serves this shape (fewer than 20 queries; key and
    value head dims each 64, 128 or 256, equal or not)."""
    return bool(lib().gdn_flash_attn_supports(int(n_q), int(head_dim_k), int(head_dim_v)))


def flash_attn(q, k, v, mask=None, scale=None, *, out=None, stream=None):
    """Decode attention: out[b, i, h] = softmax_j(scale q[b,h,i] . k[b,hk,j] +
    mask[b,0,i,j]) v[b,hk,j], hk = h // (n_heads / n_heads_kv).

    q: (n_seqs, n_heads, n_q, dk); k: (n_seqs, n_heads_kv, n_kv, dk); v:
    (n_seqs, n_heads_kv, n_kv, dv), all of one dtype (fp32, bf16 or fp16);
    mask: (n_seqs, 1, n_q, n_kv) of the same dtype, additive, or None; scale
    defaults to 1/sqrt(dk).  Returns out (n_seqs, n_q, n_heads, dv) fp32.  ("marcsun13/ggml-gated-delta-net" model
    card, section "flash_attn".)"""
    import math
    import torch
    L = lib()
    dts = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}
    if q.dtype not in dts:
        raise TypeError(f"q/k/v must be fp32, bf16 or fp16, got {q.dtype}")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, H, n_q, dk = q.shape
    Hkv, n_kv = k.shape[1], k.shape[2]
    dv = v.shape[3]
    if tuple(k.shape) != (B, Hkv, n_kv, dk) or tuple(v.shape) != (B, Hkv, n_kv, dv):
        raise ValueError(f"k, v: expected (n_seqs, n_heads_kv, n_kv, dk / dv), got {tuple(k.shape)}, "
                         f"{tuple(v.shape)}")
    tensors = [q, k, v]
    if mask is not None:
        if tuple(mask.shape) != (B, 1, n_q, n_kv):
            raise ValueError(f"mask: expected {(B, 1, n_q, n_kv)}, got {tuple(mask.shape)}")
        tensors.append(mask)
    for t in tensors:
        if t.dtype != q.dtype:
            raise TypeError("q, k, v and mask must share one dtype")
    if out is None:
        out = torch.empty((B, n_q, H, dv), dtype=torch.float32, device=q.device)
    tensors.append(out)
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
        if t.device != q.device:
            raise ValueError("all tensors must be on one CUDA device")
    if tuple(out.shape) != (B, n_q, H, dv) or out.dtype != torch.float32:
        raise ValueError("out must be (n_seqs, n_q, n_heads, dv) fp32")
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    with torch.cuda.device(q.device):
        rc = L.gdn_flash_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), B, H, Hkv, n_q,
                              n_kv, dk, dv, float(scale), dts[q.dtype], _stream_handle(stream))
    if rc != OK:
        raise GdnError(rc, "gdn_flash_attn")
    return out
