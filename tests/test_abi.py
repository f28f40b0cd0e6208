"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/gdn.h declares, answers the capability / workspace / path
queries, and rejects bad arguments on the host before touching CUDA.

Every call here that passes (made-up) device addresses is one the library
must reject during host validation; no call in this file can reach a launch.
"""
import math
import ctypes
import os
import re

import pytest

import linear_attention_sequence_gated_gb300 as gdn
from linear_attention_sequence_gated_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return gdn.lib()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gdn_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert "gdn_forward" in names and "gdn_forward_bf16" in names
    for n in names:
        assert hasattr(L, n), f"libgdn.so does not export {n}"
    assert set(names) == set(gdn.EXPORTS)


def test_library_is_built_for_sm_103a():
    # the compile flags pin the single target architecture
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.NVCC_FLAGS)


def test_supports(L):
    assert gdn.supports(32) == 1
    assert gdn.supports(96) == 1                            # recurrent only
    for d in (64, 128, 256):
        assert gdn.supports(d) == 3
    for d in (0, -1, 16, 48, 100, 160, 192, 512):
        assert gdn.supports(d) == 0


def test_status_strings(L):
    for code in range(-11, 1):
        s = gdn.status_string(code)
        assert s and s != "unknown status"
    assert gdn.status_string(-99) == "unknown status"
    assert L.gdn_version() >= 100


def test_workspace_and_path_queries(L):
    assert L.gdn_workspace_bytes(1, 1, 32, 128, 1, 1) == 0          # recurrent needs none
    assert L.gdn_workspace_bytes(-1, 1, 32, 128, 1, 0) == 0         # invalid sizes -> 0
    assert L.gdn_workspace_bytes(1, 0, 32, 128, 1, 0) == 0          # no tokens -> 0
    assert gdn.select_path(1, 1, 32, 128) == "recurrent"
    assert gdn.select_path(1, 5, 32, 32) == "recurrent"
    assert gdn.select_path(1, 4096, 32, 32) == "recurrent"            # no chunked d = 32
    assert gdn.select_path(1, 4096, 32, 96) == "recurrent"            # no chunked d = 96
    # measured switch points: (pairs, head_dim) -> first chunked length
    for pairs, d, t_switch in ((32, 64, 56), (128, 64, 32), (256, 64, 40), (2048, 64, 56),
                               (16, 128, 56), (32, 128, 48), (48, 128, 40), (64, 128, 32),
                               (72, 128, 32), (96, 128, 24), (128, 128, 24), (2048, 128, 24),
                               (8, 256, 40), (12, 256, 40), (16, 256, 32), (24, 256, 16),
                               (32, 256, 16), (256, 256, 16)):
        H = math.gcd(pairs, 32)                                       # B x H == pairs
        B = pairs // H
        assert gdn.select_path(B, t_switch - 1, H, d) == "recurrent"
        assert gdn.select_path(B, t_switch, H, d) == "chunked"
        assert gdn.select_path(B, 4096, H, d, "f32") == "recurrent"    # chunked is bf16 only
    assert L.gdn_select_path(1, 10, 1, 48, 1) == gdn.ERR_HEADDIM
    assert L.gdn_select_path(1, -1, 1, 128, 1) == gdn.ERR_ARG
    assert L.gdn_select_path(-1, 10, 1, 128, 1) == gdn.ERR_ARG
    assert L.gdn_select_path(1, 10, 1, 128, 5) == gdn.ERR_ARG
    # head_dim 64 / 128 with many (sequence, head) pairs: the fused chunked kernel keeps
    # everything on chip; head_dim 128 with fewer than 80 pairs keeps transform tiles
    assert L.gdn_workspace_bytes(8, 16384, 32, 128, 1, 2) == 0
    assert L.gdn_workspace_bytes(1, 4096, 32, 128, 1, 2) == 32 * 64 * 32768
    assert L.gdn_workspace_bytes(2, 4096, 40, 128, 1, 2) == 0            # 80 pairs: fused
    assert L.gdn_workspace_bytes(8, 16384, 64, 64, 1, 2) == 0
    # head_dim 256: one 32 KB chunk-transform tile per (sequence, head, chunk)
    assert L.gdn_workspace_bytes(8, 16384, 16, 256, 1, 2) == 8 * 16 * 256 * 32768
    assert L.gdn_workspace_bytes(2, 65, 3, 256, 1, 2) == 2 * 3 * 2 * 32768
    assert L.gdn_workspace_bytes(1, 4096, 16, 256, 1, 1) == 0      # recurrent path: none
    assert L.gdn_workspace_bytes(1, 4096, 16, 256, 0, 2) == 0      # chunked is bf16 only


# fake, well-aligned device addresses; every call below must fail validation
BASE = 1 << 40
MB = 1 << 20


def call(L, q=BASE, k=BASE + 64 * MB, v=BASE + 128 * MB, g=BASE + 192 * MB,
         beta=BASE + 256 * MB, s_in=BASE + 320 * MB, out=BASE + 512 * MB,
         s_out=BASE + 768 * MB, B=1, T=4, H=2, Hk=0, d=64, dtype=1, path=0, ws=None,
         ws_bytes=0):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.gdn_forward_ex(p(q), p(k), p(v), p(g), p(beta), p(s_in), p(out), p(s_out),
                            B, T, H, Hk, d, dtype, path, p(ws), ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), gdn.ERR_ARG), (dict(T=-1), gdn.ERR_ARG), (dict(H=-2), gdn.ERR_ARG),
    (dict(d=0), gdn.ERR_ARG), (dict(dtype=7), gdn.ERR_ARG), (dict(path=9), gdn.ERR_ARG),
    (dict(d=48), gdn.ERR_HEADDIM), (dict(d=96, path=2), gdn.ERR_HEADDIM),
    (dict(d=160), gdn.ERR_HEADDIM), (dict(d=512), gdn.ERR_HEADDIM),
    (dict(q=None), gdn.ERR_ARG), (dict(k=None), gdn.ERR_ARG), (dict(v=None), gdn.ERR_ARG),
    (dict(g=None), gdn.ERR_ARG), (dict(beta=None), gdn.ERR_ARG), (dict(out=None), gdn.ERR_ARG),
    (dict(s_out=None), gdn.ERR_ARG),
    (dict(q=BASE + 8), gdn.ERR_ALIGN), (dict(v=BASE + 128 * MB + 4), gdn.ERR_ALIGN),
    (dict(out=BASE + 512 * MB + 2), gdn.ERR_ALIGN), (dict(s_in=BASE + 320 * MB + 8), gdn.ERR_ALIGN),
    (dict(s_out=BASE + 768 * MB + 4), gdn.ERR_ALIGN), (dict(g=BASE + 192 * MB + 2), gdn.ERR_ALIGN),
    (dict(out=BASE), gdn.ERR_ALIAS),                         # out on top of q
    (dict(out=BASE + 256 * MB), gdn.ERR_ALIAS),              # out on top of beta
    (dict(out=BASE + 768 * MB), gdn.ERR_ALIAS),              # out == state_out
    (dict(s_out=BASE + 64 * MB), gdn.ERR_ALIAS),             # state_out on k
    (dict(s_out=BASE + 320 * MB + 16), gdn.ERR_ALIAS),       # partial overlap with state_in
    (dict(s_out=BASE + 192 * MB), gdn.ERR_ALIAS),            # state_out on g
    (dict(B=1 << 20, T=1 << 20, H=1 << 20, d=256), gdn.ERR_ARG),   # size overflow
    (dict(B=70000, H=70000, T=1), gdn.ERR_ARG),              # more (b, h) pairs than a grid row
    (dict(Hk=-1), gdn.ERR_ARG), (dict(Hk=3), gdn.ERR_ARG),   # key heads: negative, > n_heads
    (dict(H=6, Hk=4), gdn.ERR_ARG),                          # key heads must divide n_heads
    (dict(H=4, Hk=2, out=BASE + 512), gdn.ERR_ALIAS),       # out inside q's (B,T,Hk,d) span
])
def test_host_validation_rejects(L, kw, code):
    assert call(L, **kw) == code


def test_recurrent_path_rejects_unsupported_headdim(L):
    assert call(L, d=48, path=1) == gdn.ERR_HEADDIM


def test_chunked_path_rejects_fp32_and_headdim_32(L):
    assert call(L, dtype=0, path=2) == gdn.ERR_DTYPE
    assert call(L, d=32, path=2) == gdn.ERR_HEADDIM


def test_empty_batch_is_a_no_op(L):
    # n_seqs == 0 or n_heads == 0: nothing to do, no pointer needed, no CUDA call
    assert call(L, B=0, q=None, k=None, v=None, g=None, beta=None, out=None, s_out=None) == gdn.OK
    assert call(L, H=0, q=None, k=None, v=None, g=None, beta=None, out=None, s_out=None) == gdn.OK


def test_typed_entry_points_validate(L):
    p = ctypes.c_void_p
    assert L.gdn_forward(p(BASE), p(BASE), p(BASE), p(BASE + 8), p(BASE), None, p(BASE),
                         p(BASE), 1, 1, 1, 48, None) == gdn.ERR_HEADDIM
    assert L.gdn_forward_bf16(p(BASE), p(BASE), p(BASE), p(BASE), p(BASE), None, None,
                              p(BASE + 4096), 1, 1, 1, 64, None) == gdn.ERR_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(RuntimeError, match="libgdn.so not found"):
        gdn.lib()



# ------------------------------------------------------------ decode attention

def test_flash_attn_supports(L):
    for d in (64, 128, 256):
        for n_q in (1, 5, 19):
            assert gdn.flash_attn_supports(n_q, d, d)
        assert not gdn.flash_attn_supports(20, d, d)      # the vector variant only
        assert not gdn.flash_attn_supports(0, d, d)
    for dk in (64, 128, 256):                             # key and value widths apart
        for dv in (64, 128, 256):
            assert gdn.flash_attn_supports(1, dk, dv)
    for d in (32, 48, 96, 512):
        assert not gdn.flash_attn_supports(1, d, d)
        assert not gdn.flash_attn_supports(1, d, 128)
        assert not gdn.flash_attn_supports(1, 128, d)


def attn_call(L, q=BASE, k=BASE + 64 * MB, v=BASE + 128 * MB, mask=BASE + 192 * MB,
              out=BASE + 256 * MB, B=1, H=16, Hkv=4, n_q=1, n_kv=512, dk=256, dv=256, scale=0.0625,
              dtype=1):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.gdn_flash_attn(p(q), p(k), p(v), p(mask), p(out), B, H, Hkv, n_q, n_kv, dk, dv,
                            ctypes.c_float(scale), dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), gdn.ERR_ARG), (dict(n_kv=-1), gdn.ERR_ARG), (dict(n_q=-1), gdn.ERR_ARG),
    (dict(dtype=3), gdn.ERR_ARG), (dict(dk=48, dv=48), gdn.ERR_HEADDIM),
    (dict(dk=128, dv=96), gdn.ERR_HEADDIM), (dict(n_q=20), gdn.ERR_SHAPE),
    (dict(Hkv=3), gdn.ERR_ARG), (dict(Hkv=0), gdn.ERR_ARG), (dict(Hkv=32), gdn.ERR_ARG),
    (dict(scale=float("inf")), gdn.ERR_ARG), (dict(scale=float("nan")), gdn.ERR_ARG),
    (dict(q=None), gdn.ERR_ARG), (dict(out=None), gdn.ERR_ARG), (dict(k=None), gdn.ERR_ARG),
    (dict(v=None), gdn.ERR_ARG),
    (dict(q=BASE + 8), gdn.ERR_ALIGN), (dict(k=BASE + 64 * MB + 4), gdn.ERR_ALIGN),
    (dict(out=BASE + 256 * MB + 8), gdn.ERR_ALIGN), (dict(mask=BASE + 192 * MB + 1), gdn.ERR_ALIGN),
    (dict(out=BASE), gdn.ERR_ALIAS), (dict(out=BASE + 128 * MB + 4096), gdn.ERR_ALIAS),
    (dict(out=BASE + 192 * MB), gdn.ERR_ALIAS),
    (dict(B=1 << 20, H=1 << 20, Hkv=1 << 20, n_kv=1 << 20), gdn.ERR_ARG),
])
def test_flash_attn_host_validation_rejects(L, kw, code):
    assert attn_call(L, **kw) == code


def test_flash_attn_empty_is_a_no_op(L):
    # no queries at all: nothing to do and no pointer needed
    assert attn_call(L, B=0, q=None, k=None, v=None, mask=None, out=None) == gdn.OK
    assert attn_call(L, n_q=0, q=None, k=None, v=None, mask=None, out=None) == gdn.OK
    assert attn_call(L, H=0, Hkv=0, q=None, k=None, v=None, mask=None, out=None) == gdn.OK


def test_option_bits(L):
    # GDN_OPT_L2NORM_QK and GDN_OPT_OUT_BF16 are accepted in the path
    # argument (alone or together); unknown bits are not
    for opt in (gdn.OPT_L2NORM_QK, gdn.OPT_OUT_BF16, gdn.OPT_L2NORM_QK | gdn.OPT_OUT_BF16):
        assert L.gdn_workspace_bytes(1, 4096, 32, 128, 1, 2 | opt) == 32 * 64 * 32768
        # a valid option still goes through host validation (here: misaligned q)
        assert call(L, q=BASE + 8, path=opt) == gdn.ERR_ALIGN
    assert L.gdn_workspace_bytes(1, 4096, 32, 128, 1, 2 | 0x400) == 0
    assert call(L, path=0x400) == gdn.ERR_ARG
    assert call(L, path=0x101 | 0x800) == gdn.ERR_ARG
    assert call(L, path=-1) == gdn.ERR_ARG


def test_bf16_output_extent_is_two_bytes_per_element(L):
    """With GDN_OPT_OUT_BF16 the output occupies 2-byte elements: an out
    buffer ending 1904 bytes before state_out overlaps it as fp32 (8192
    bytes) but not as bf16 (4096 bytes).  The bf16 call then stops at its
    too-small workspace instead, still on the host."""
    s_out = BASE + 768 * MB
    kw = dict(out=s_out - 6000, d=256, path=2, ws=BASE + 900 * MB, ws_bytes=16)
    assert call(L, **kw) == gdn.ERR_ALIAS
    assert call(L, **{**kw, "path": 2 | gdn.OPT_OUT_BF16}) == gdn.ERR_WORKSPACE


def test_gdn_entry_points_reject_f16(L):
    assert call(L, dtype=2) == gdn.ERR_ARG
