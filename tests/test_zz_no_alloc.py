"""The allocation-free entry point, gdn_forward_noalloc, against gdn_forward_ex.

gdn_forward_noalloc serves callers that cannot allocate device memory while
they run (a framework that has reserved the device for its own arena, a
decode loop that must not stall on an allocation).  The chunked calls that
need scratch -- head_dim 256, and head_dim 128 with few (sequence, head)
pairs -- then use a fixed 64 MiB array inside the library instead of caller
or stream-ordered memory.  These tests call it
through the C ABI twice in a row, with different inputs (the array keeps the
previous call's contents), and compare each result with the existing entry
point's on the same inputs.  Both run the same deterministic kernels on the
same inputs, only with the scratch at another address, so the results must be
identical bit for bit (a scratch-addressing fault that moved them by less than
the parity bound would still be caught); the bf16 parity bound of the other
tests is checked as well.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import linear_attention_sequence_gated_gb300 as gdn
from linear_attention_sequence_gated_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 3e-3          # max |x - ref| / RMS(ref), the bound of the bf16 parity tests


@pytest.fixture(scope="module")
def L():
    from linear_attention_sequence_gated_gb300 import _build
    _build.build()
    return gdn.lib()


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def rel_err(x, ref):
    x, ref = x.double(), ref.double()
    return ((x - ref).abs().max() / ref.pow(2).mean().sqrt()).item()


def noalloc(L, inp, out, st_out, path=gdn.PATHS["chunked"]):
    B, T, H, d = inp["v"].shape
    Hk = inp["q"].shape[2]
    stream = torch.cuda.current_stream().cuda_stream
    return L.gdn_forward_noalloc(ptr(inp["q"]), ptr(inp["k"]), ptr(inp["v"]), ptr(inp["g"]),
                                 ptr(inp["beta"]), ptr(inp["state"]), ptr(out), ptr(st_out),
                                 B, T, H, Hk, d, gdn.DTYPE_BF16, path, ctypes.c_void_p(stream))


def test_two_calls_in_a_row_match_the_existing_entry_point(L):
    # head_dim 256 on the chunked path: 2 x 4 heads x 16 chunks = 128 scratch tiles (4 MiB)
    for seed in (71, 72):
        w = W.Workload(f"noalloc_{seed}", 2, 1000, 4, 256, "bf16", 0.0, 0.02, seed=seed)
        inp = W.make_inputs(w, "cuda")
        assert L.gdn_workspace_bytes(w.B, w.T, w.H, w.d, gdn.DTYPE_BF16, 2) > 0
        ref_out, ref_st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      inp["state"], path="chunked")
        out = torch.full_like(ref_out, float("nan"))
        st = torch.full_like(ref_st, float("nan"))
        assert noalloc(L, inp, out, st) == gdn.OK
        torch.cuda.synchronize()
        assert gdn.device_status() == gdn.OK
        assert rel_err(out, ref_out) <= TOL
        assert rel_err(st, ref_st) <= TOL
        assert torch.equal(out, ref_out) and torch.equal(st, ref_st)


def test_head_dim_128_with_and_without_scratch_and_auto(L):
    # 8 (sequence, head) pairs: the two-kernel path, which takes scratch;
    # 96 pairs: the one-kernel path, which needs none and goes straight through
    for H, seed in ((4, 73), (48, 74)):
        w = W.Workload(f"noalloc_d128_h{H}", 2, 300, H, 128, "bf16", 0.0, 0.02, seed=seed)
        need = L.gdn_workspace_bytes(w.B, w.T, w.H, w.d, gdn.DTYPE_BF16, gdn.PATHS["auto"])
        assert (need > 0) == (w.B * w.H < 80)
        inp = W.make_inputs(w, "cuda")
        ref_out, ref_st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      inp["state"])
        out, st = torch.empty_like(ref_out), torch.empty_like(ref_st)
        assert noalloc(L, inp, out, st, path=gdn.PATHS["auto"]) == gdn.OK
        torch.cuda.synchronize()
        assert gdn.device_status() == gdn.OK
        assert rel_err(out, ref_out) <= TOL and rel_err(st, ref_st) <= TOL
        assert torch.equal(out, ref_out) and torch.equal(st, ref_st)


SCRATCH = 64 << 20


def test_a_call_that_needs_exactly_the_whole_scratch(L):
    # 1 sequence x 4096 tokens x 32 heads at head_dim 128 takes the two-kernel
    # path: 32 pairs x 64 chunks x 32 KiB = 64 MiB, the whole array
    w = W.Workload("noalloc_full", 1, 4096, 32, 128, "bf16", 2.0, 0.02, seed=75)
    assert L.gdn_workspace_bytes(w.B, w.T, w.H, w.d, gdn.DTYPE_BF16, gdn.PATHS["auto"]) == SCRATCH
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["state"])
    out = torch.full_like(ref_out, float("nan"))
    st = torch.full_like(ref_st, float("nan"))
    assert noalloc(L, inp, out, st, path=gdn.PATHS["auto"]) == gdn.OK
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    assert torch.equal(out, ref_out) and torch.equal(st, ref_st)


def test_one_chunk_beyond_the_scratch_is_rejected_before_any_work(L):
    # one more token opens a 65th chunk: 64 MiB + 32 x 32 KiB
    w = W.Workload("noalloc_over", 1, 4097, 32, 128, "bf16", 2.0, 0.02, seed=76)
    assert L.gdn_workspace_bytes(w.B, w.T, w.H, w.d, gdn.DTYPE_BF16, gdn.PATHS["auto"]) == \
        SCRATCH + 32 * 32768
    inp = W.make_inputs(w, "cuda")
    out = torch.full((w.B, w.T, w.H, w.d), 7.0, device="cuda")
    st = torch.full((w.B, w.H, w.d, w.d), 7.0, device="cuda")
    torch.cuda.synchronize()
    assert noalloc(L, inp, out, st, path=gdn.PATHS["auto"]) == gdn.ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((st == 7.0).all())     # nothing was written


def test_rejects_calls_beyond_the_fixed_scratch(L):
    # 8 sequences x 16 heads x 256 chunks of head_dim 256 would need 1 GiB; the
    # check happens on the host before any pointer is used
    fake = ctypes.c_void_p(1 << 40)
    rc = L.gdn_forward_noalloc(fake, fake, fake, fake, fake, None, fake, fake,
                               8, 16384, 16, 16, 256, gdn.DTYPE_BF16, gdn.PATHS["chunked"], None)
    assert rc == gdn.ERR_SCRATCH
    assert "64 MiB" in gdn.status_string(rc)


def test_options_pass_through(L):
    """Option bits in the path argument reach the kernels through this entry
    point as through gdn_forward_ex: q/k normalisation and a bf16 output on
    the scratch-using head_dim-256 path, bit for bit."""
    w = W.Workload("noalloc_opts", 2, 300, 4, 256, "bf16", 0.0, 0.02, seed=77)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["state"], path="chunked", l2norm_qk=True,
                                  out_dtype=torch.bfloat16)
    out = torch.full_like(ref_out, float("nan"))
    st = torch.full_like(ref_st, float("nan"))
    path = gdn.PATHS["chunked"] | gdn.OPT_L2NORM_QK | gdn.OPT_OUT_BF16
    assert noalloc(L, inp, out, st, path=path) == gdn.OK
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    assert out.dtype == torch.bfloat16
    assert torch.equal(out, ref_out) and torch.equal(st, ref_st)
