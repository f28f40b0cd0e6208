"""GPU parity: the CUDA library (called through its C ABI via the binding)
against the float64 oracle on the same seeded inputs.

Metric: max |gpu - oracle| / RMS(oracle) over the whole compared tensor,
separately for out and final_state.  Bounds: 1e-4 for fp32 q/k/v and 3e-3 for
bf16 q/k/v.  The recurrent path computes in fp32 throughout, so it is also
held to 1e-4 for bf16 inputs (their upcast is exact).

Workloads follow the shapes measured on the "marcsun13/ggml-gated-delta-net"
model card (section "Measured": 32 value heads x head_dim 128, one token per
step, 24 layers) plus batched decode and long prefill; see
linear_attention_sequence_gated_gb300/workloads.py for the distributions.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_attention_sequence_gated_gb300 as gdn
from linear_attention_sequence_gated_gb300 import workloads as W
import oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 3e-3}
TOL_RECURRENT = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_attention_sequence_gated_gb300 import _build
    _build.build()
    oracle.build()


def run_gpu(inp, path="auto", state_out=None):
    out, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                          path=path, state_out=state_out)
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    return out, st


def run_oracle(inp):
    n = W.to_numpy_f32(inp)
    return oracle.recurrent_c(n["q"], n["k"], n["v"], n["g"], n["beta"], n["state"])


def errs(out, st, ref_out, ref_st):
    return (oracle.parity_error(out.double().cpu().numpy(), ref_out),
            oracle.parity_error(st.double().cpu().numpy(), ref_st))


def check(inp, dtype, path="auto", tol=None):
    out, st = run_gpu(inp, path)
    ref_out, ref_st = run_oracle(inp)
    e_out, e_st = errs(out, st, ref_out, ref_st)
    tol = TOL[dtype] if tol is None else tol
    assert e_out <= tol and e_st <= tol, (e_out, e_st, tol)
    return e_out, e_st


def paths_for(d, T, dtype="bf16"):
    caps = gdn.supports(d)
    ps = []
    if caps & 1:
        ps.append("recurrent")
    if caps & 2 and dtype == "bf16":
        ps.append("chunked")
    return ps


# ---------------------------------------------------------------- workloads

def test_tiny_workload_all_paths():
    w = W.TINY
    inp = W.make_inputs(w, "cuda")
    for path in ["auto"] + paths_for(w.d, w.T, w.dtype):
        tol = TOL_RECURRENT if path == "recurrent" else TOL[w.dtype]
        check(inp, w.dtype, path, tol)


def test_decode_24_layers():
    w = W.DECODE_24L
    for layer in range(w.layers):
        inp = W.make_inputs(w, "cuda", layer=layer)
        check(inp, w.dtype, "auto", TOL_RECURRENT)


def test_batched_decode_b64():
    w = W.DECODE_B64
    inp = W.make_inputs(w, "cuda")
    check(inp, w.dtype, "auto", TOL_RECURRENT)


@pytest.mark.parametrize("path", ["auto", "recurrent", "chunked"])
def test_prefill_4k_full(path):
    w = W.PREFILL_4K
    if path == "chunked" and not gdn.supports(w.d) & 2:
        pytest.skip("chunked path not built")
    inp = W.make_inputs(w, "cuda")
    check(inp, w.dtype, path, TOL_RECURRENT if path == "recurrent" else None)


N_SMS = 152


def ctas_per_pair(w, path):
    """CTAs one (sequence, head) pair takes on the chunked path: the state walk
    of the two-kernel path (which needs a workspace) runs head_dim / 64
    value-row blocks per pair, the one-kernel path one CTA per pair.  (When
    the walk's last pairs run as a second launch of 32-row blocks, those
    pairs are the last range of pairs, which sampled_pairs also samples.)"""
    if path == "auto":
        path = gdn.select_path(w.B, w.T, w.H, w.d, w.dtype)
    if path == "chunked" and gdn.workspace_bytes(w.B, w.T, w.H, w.d, "bf16", "chunked"):
        return w.d // 64
    return 1


def sampled_pairs(w, n, per_cta=1):
    """n random (sequence, head) pairs plus the first and the last, plus one
    pair from every wave of 152 CTAs (pairs are laid out b * H + h in launch
    order, `per_cta` CTAs each), so that a fault tied to the second or a
    later CTA on an SM cannot hide between samples."""
    r = np.random.default_rng(1234)
    pairs = {(0, 0), (w.B - 1, w.H - 1)}
    n_pairs = w.B * w.H
    per_wave = max(1, N_SMS // per_cta)
    for first in range(0, n_pairs, per_wave):
        i = int(r.integers(first, min(n_pairs, first + per_wave)))
        pairs.add(divmod(i, w.H))
    while len(pairs) < n + 2:
        pairs.add((int(r.integers(w.B)), int(r.integers(w.H))))
    return sorted(pairs)


_SAMPLE_REF = {}


def sampled_reference(w, inp, pairs):
    """The oracle on the sampled pairs, as one batch of independent problems
    (one OpenMP thread per pair); cached per workload and sample."""
    key = (w.name, tuple(pairs))
    if key not in _SAMPLE_REF:
        bs = [b for b, _ in pairs]
        hs = [h for _, h in pairs]
        Hk = inp["q"].shape[2]
        hks = [h % Hk for h in hs]
        # gather the sampled pairs on the device, then copy only them
        f32 = lambda t: t.float().cpu().numpy()
        pick = lambda x, heads: np.ascontiguousarray(
            f32(torch.stack([x[b, :, hh] for b, hh in zip(bs, heads)]))[:, :, None])
        n = {key_: inp[key_] for key_ in ("q", "k", "v", "g", "beta")}
        st = None if inp["state"] is None else np.ascontiguousarray(
            f32(torch.stack([inp["state"][b, h] for b, h in pairs]))[:, None])
        _SAMPLE_REF[key] = oracle.recurrent_c(pick(n["q"], hks), pick(n["k"], hks),
                                              pick(n["v"], hs), pick(n["g"], hs),
                                              pick(n["beta"], hs), st)
    return _SAMPLE_REF[key]


@pytest.mark.parametrize("wname", [W.PREFILL_16K.name, W.PREFILL_16K_D64.name,
                                   W.PREFILL_16K_D256.name])
@pytest.mark.parametrize("path", ["auto", "recurrent", "chunked"])
def test_long_prefill_full_size_sampled(wname, path):
    """Full-size launch (the configuration the benchmark times); the oracle
    recomputes every output and the final state of a sample of (sequence,
    head) pairs, which are independent problems: at least one pair from
    every wave of CTAs."""
    w = W.BY_NAME[wname]
    if path == "chunked" and not gdn.supports(w.d) & 2:
        pytest.skip("chunked path not built")
    inp = W.make_inputs(w, "cuda")
    out, st = run_gpu(inp, path)
    tol = TOL_RECURRENT if path == "recurrent" else TOL[w.dtype]
    pairs = sampled_pairs(w, 6, ctas_per_pair(w, path))
    ref_out, ref_st = sampled_reference(w, inp, pairs)
    got_out = np.stack([out[b, :, h].double().cpu().numpy() for b, h in pairs])
    got_st = np.stack([st[b, h].double().cpu().numpy() for b, h in pairs])
    e_out = oracle.parity_error(got_out.ravel(), ref_out.ravel())
    e_st = oracle.parity_error(got_st.ravel(), ref_st.ravel())
    assert e_out <= tol and e_st <= tol, (e_out, e_st, len(pairs))


# ------------------------------------------------------ shapes and dtypes

@pytest.mark.parametrize("d", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 7, 63, 64, 65, 200])
def test_head_dims_dtypes_lengths(d, dtype, T):
    w = W.Workload("matrix", 2, T, 3, d, dtype, 0.0, 0.02, seed=77)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    for path in ["auto"] + paths_for(d, T, dtype):
        out, st = run_gpu(inp, path)
        e_out, e_st = errs(out, st, ref_out, ref_st)
        tol = TOL_RECURRENT if path == "recurrent" else TOL[dtype]
        assert e_out <= tol and e_st <= tol, (path, e_out, e_st)


# At head_dim 128 the chunked path has two kernels: one CTA per (sequence,
# head) pair when there are at least 80 pairs, a chunk-transform pass plus a
# state walk on value-row blocks below that.  The small cases above (6 pairs)
# take the second; these take the first, with ragged tails and fewer key heads.
ONE_KERNEL_D128_PAIRS = 80


@pytest.mark.parametrize("T", [1, 7, 63, 64, 65, 200, 1000])
def test_head_dim_128_one_kernel_chunked_path(T):
    w = W.Workload("d128_many_pairs", 2, T, 48, 128, "bf16", 0.0, 0.02, seed=78)
    assert w.B * w.H >= ONE_KERNEL_D128_PAIRS
    assert gdn.workspace_bytes(w.B, w.T, w.H, w.d, "bf16", "chunked") == 0
    check(W.make_inputs(w, "cuda"), "bf16", "chunked")


def test_head_dim_128_one_kernel_chunked_path_key_heads_and_carry():
    """Fewer key heads (48 value heads over 12) on the one-kernel path, and
    one call against two calls split off a chunk boundary."""
    w = W.Workload("d128_many_pairs_gqa", 2, 200, 48, 128, "bf16", 0.0, 0.02, seed=79)
    inp = W.make_inputs(w, "cuda")
    inp["q"] = inp["q"][:, :, :12].contiguous()
    inp["k"] = inp["k"][:, :, :12].contiguous()
    ref_out, ref_st = run_oracle(inp)
    out, st = run_gpu(inp, "chunked")
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)
    t1 = 100
    a = {key: (val[:, :t1].contiguous() if key != "state" else val) for key, val in inp.items()}
    b = {key: (val[:, t1:].contiguous() if key != "state" else None) for key, val in inp.items()}
    oa, sa = run_gpu(a, "chunked")
    b["state"] = sa
    ob, sb = run_gpu(b, "chunked")
    e_out, e_st = errs(torch.cat([oa, ob], dim=1), sb, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


@pytest.mark.parametrize("shift", [-2.0, 2.0, 6.0])
def test_gate_regimes(shift):
    """Slow (alpha ~ 0.88), fast (~0.12) and near-total (~0.002) decay."""
    w = W.Workload("gates", 1, 300, 4, 128, "bf16", shift, 0.02, seed=31)
    inp = W.make_inputs(w, "cuda")
    for path in paths_for(w.d, w.T):
        check(inp, "bf16", path, TOL_RECURRENT if path == "recurrent" else None)


# ------------------------------------------------------------- edge cases

def test_extreme_gates_and_betas():
    """g = 0 (no decay), g = -inf (total reset), g = -1e4, beta = 0 and 1."""
    w = W.Workload("edge", 1, 130, 2, 64, "f32", 0.0, 0.05, seed=5)
    inp = W.make_inputs(w, "cuda")
    g, beta = inp["g"], inp["beta"]
    g[:, 0:10] = 0.0
    g[:, 17] = -float("inf")
    g[:, 70] = -1e4
    beta[:, 20:30] = 0.0
    beta[:, 40:45] = 1.0
    for path in paths_for(w.d, w.T, "f32"):
        check(inp, "f32", path, TOL["f32"])


# The chunked kernels, one case per kernel: head_dim 64 and head_dim 128 with
# at least 80 (sequence, head) pairs run the one-kernel path; head_dim 128
# with fewer pairs and head_dim 256 run the chunk-transform pass plus the
# state walk on value-row blocks.
# Every chunked kernel and state-walk width on a 152-SM GB300: the two-kernel
# walk takes 32-row value blocks while (pairs x head_dim / 32) <= 152, else
# 64-row blocks; head_dim 128 runs the two-kernel path below 80 pairs.
CHUNKED_KERNELS = [("d64", 2, 4, 64), ("d128_one_kernel", 2, 48, 128),
                   ("d128_two_kernel_bv32", 2, 4, 128), ("d128_two_kernel_bv64", 2, 24, 128),
                   ("d256_bv32", 2, 4, 256), ("d256_bv64", 2, 12, 256)]


def plant_extremes(inp):
    """Method edge cases over 200 tokens (chunks 0-63, 64-127, 128-191 and a
    ragged 192-199): a whole chunk of g = 0 (no decay), g = -inf (a total
    reset) at a chunk's first token, mid-chunk, on a chunk's last token and
    on the very last token, g = -1e4, a run of beta = 1 and of beta = 0, a
    whole chunk of beta = 0 (that chunk only decays the state), and k = 0
    rows (the token writes nothing)."""
    g, beta, k = inp["g"], inp["beta"], inp["k"]
    g[:, 0:64] = 0.0
    g[:, 64] = -float("inf")
    g[:, 100] = -float("inf")
    g[:, 127] = -float("inf")
    g[:, 150] = -1e4
    g[:, 199] = -float("inf")
    beta[:, 20:30] = 1.0
    beta[:, 30:36] = 0.0
    beta[:, 128:192] = 0.0
    k[:, 40:44] = 0
    k[:, 160] = 0
    return inp


@pytest.mark.parametrize("name,B,H,d", CHUNKED_KERNELS)
def test_extreme_gates_and_betas_chunked(name, B, H, d):
    """The chunked tensor-core kernels held to the method's edge cases: the
    clamp of g before the in-chunk running sum, decays that flush to zero,
    no NaN from (-inf) - (-inf), beta = 0 / 1 rows and a beta = 0 chunk in
    the UT transform, k = 0 rows."""
    w = W.Workload(f"edge_{name}", B, 200, H, d, "bf16", 0.0, 0.05, seed=6)
    inp = plant_extremes(W.make_inputs(w, "cuda"))
    out, st = run_gpu(inp, "chunked")
    assert torch.isfinite(out).all() and torch.isfinite(st).all()
    ref_out, ref_st = run_oracle(inp)
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)
    # the same inputs on the recurrent path, at its own bound
    check(inp, "bf16", "recurrent", TOL_RECURRENT)


@pytest.mark.parametrize("name,B,H,d", CHUNKED_KERNELS)
def test_reset_on_last_token_leaves_only_that_token_chunked(name, B, H, d):
    """g = -inf and beta = 1 on the last token with unit k: the final state is
    exactly v k^T of that token, whatever came before (forgetting pin)."""
    w = W.Workload(f"reset_{name}", B, 130, H, d, "bf16", 0.0, 0.05, seed=8)
    inp = W.make_inputs(w, "cuda")
    inp["g"][:, -1] = -float("inf")
    inp["beta"][:, -1] = 1.0
    out, st = run_gpu(inp, "chunked")
    k = inp["k"][:, -1].float()
    v = inp["v"][:, -1].float()
    Hk = k.shape[1]
    kk = k[:, torch.arange(H, device="cuda") % Hk]
    expect = v[:, :, :, None] * kk[:, :, None, :]
    err = ((st - expect).abs().max() / expect.pow(2).mean().sqrt()).item()
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("name,B,H,d", CHUNKED_KERNELS)
def test_in_place_state_update_chunked(name, B, H, d):
    """state_out == state_in on every chunked kernel: the value-row blocks of
    the two-kernel walk each read their own rows before writing them."""
    w = W.Workload(f"inplace_{name}", B, 150, H, d, "bf16", 0.0, 0.02, seed=16)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    st = inp["state"].clone()
    out, st2 = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st,
                           state_out=st, path="chunked")
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    assert st2.data_ptr() == st.data_ptr()
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


@pytest.mark.parametrize("B,H,d", [(1, 38, 128), (1, 39, 128), (1, 19, 256), (1, 20, 256)])
def test_state_walk_width_boundary(B, H, d):
    """The state walk takes 32-row value blocks while (pairs x head_dim / 32)
    fits one wave of 152 SMs, else 64-row blocks: 38 pairs at head_dim 128
    and 19 at 256 are the last 32-row cases, 39 and 20 the first 64-row
    ones.  Each against the oracle, in place, over a ragged tail."""
    w = W.Workload(f"walkw_h{H}_d{d}", B, 150, H, d, "bf16", 0.0, 0.02, seed=17)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    st = inp["state"].clone()
    out, _ = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st,
                         state_out=st, path="chunked")
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


@pytest.mark.parametrize("B,H,d", [(1, 40, 256), (2, 23, 256), (1, 77, 128)])
def test_state_walk_mixed_value_blocks(B, H, d):
    """When 64-row value blocks leave a partial last wave whose pairs fit one
    wave at 32 rows, the pairs of the full waves take 64-row blocks and the
    rest a second launch of 32-row blocks (on 152 SMs: 40 pairs at head_dim
    256 -> 38 + 2, 46 -> 38 + 8, 77 at 128 -> 76 + 1).  Every pair, both
    launches, against the oracle, in place, over a ragged tail."""
    w = W.Workload(f"walkmix_b{B}_h{H}_d{d}", B, 150, H, d, "bf16", 0.0, 0.02, seed=23)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    st = inp["state"].clone()
    out, _ = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st,
                         state_out=st, path="chunked")
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    o, s_ = out.double().cpu().numpy(), st.double().cpu().numpy()
    for b in range(B):                    # each pair on its own: a wrong block is not diluted
        for h in range(H):
            e_out = oracle.parity_error(o[b, :, h], ref_out[b, :, h])
            e_st = oracle.parity_error(s_[b, h], ref_st[b, h])
            assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (b, h, e_out, e_st)


def test_state_walk_mixed_value_blocks_with_options():
    """The two launches of a mixed value-block walk (on 152 SMs: 38 pairs at
    64 rows, 2 at 32) with 8 key heads for 40 value heads, q / k normalised
    inside the op and a bf16 output: every pair against the normalising
    oracle, its output rounded to bf16 (a rounding of at most 2^-8 of each
    element on top of the bf16-input bound)."""
    w = W.Workload("walkmix_opts", 1, 150, 40, 256, "bf16", 0.0, 0.02, seed=29, Hk=8)
    inp = raw_qk(W.make_inputs(w, "cuda"), seed=30)
    out, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                          path="chunked", l2norm_qk=True, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    assert out.dtype == torch.bfloat16
    n = W.to_numpy_f32(inp)
    ref_out, ref_st = oracle.recurrent_c(n["q"], n["k"], n["v"], n["g"], n["beta"], n["state"],
                                         l2norm_qk=True)
    o, s_ = out.double().cpu().numpy(), st.double().cpu().numpy()
    for h in range(w.H):
        ro = ref_out[0, :, h]
        tol_o = TOL["bf16"] + 2.0 ** -8 * np.abs(ro).max() / max(np.sqrt((ro ** 2).mean()), 1e-30)
        e_out = oracle.parity_error(o[0, :, h], ro)
        e_st = oracle.parity_error(s_[0, h], ref_st[0, h])
        assert e_out <= tol_o and e_st <= TOL["bf16"], (h, e_out, e_st)


def test_concurrent_calls_on_two_streams():
    """Two head_dim-256 chunked calls (each needs a workspace, taken
    stream-ordered from the library's pool) in flight at once on two
    streams, with different inputs: each equals the same call made alone."""
    ws = [W.Workload(f"conc_{i}", 2, 300, 4, 256, "bf16", 0.0, 0.02, seed=40 + i) for i in range(2)]
    inps = [W.make_inputs(w, "cuda") for w in ws]
    alone = []
    for inp in inps:
        o, s_ = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                            path="chunked")
        alone.append((o, s_))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    together = [None, None]
    for rep in range(3):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                together[i] = gdn.forward(inps[i]["q"], inps[i]["k"], inps[i]["v"], inps[i]["g"],
                                          inps[i]["beta"], inps[i]["state"], path="chunked",
                                          stream=streams[i])
        torch.cuda.synchronize()
        assert gdn.device_status() == gdn.OK
        for i in range(2):
            assert torch.equal(together[i][0], alone[i][0]) and torch.equal(together[i][1], alone[i][1])


def _named_call(fn, inp, out, st_out):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    B, T, H, d = inp["v"].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["g"]), p(inp["beta"]),
              p(inp["state"]), p(out), p(st_out), B, T, H, d, stream)


@pytest.mark.parametrize("T,with_state", [(1, True), (5, False), (200, True)])
@pytest.mark.parametrize("d", [64, 128])
def test_named_entry_point_fp32(T, with_state, d):
    """gdn_forward, the signature as named (fp32 q/k/v, AUTO path), called
    through ctypes on device tensors, against the oracle."""
    w = W.Workload("named_f32", 2, T, 4, d, "f32", 0.0, 0.02 if with_state else 0.0, seed=21)
    inp = W.make_inputs(w, "cuda")
    out = torch.full((2, T, 4, d), float("nan"), device="cuda")
    st = torch.full((2, 4, d, d), float("nan"), device="cuda")
    assert _named_call(gdn.lib().gdn_forward, inp, out, st) == gdn.OK
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    ref_out, ref_st = run_oracle(inp)
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["f32"] and e_st <= TOL["f32"], (e_out, e_st)


@pytest.mark.parametrize("B,T,H,d", [(2, 1, 4, 128), (2, 7, 4, 64), (2, 300, 4, 128),
                                     (2, 300, 48, 128), (1, 200, 3, 256), (2, 150, 4, 64)])
def test_named_entry_point_bf16(B, T, H, d):
    """gdn_forward_bf16 (AUTO path: recurrent at short runs, every chunked
    kernel at long ones) through ctypes, against the oracle."""
    w = W.Workload("named_bf16", B, T, H, d, "bf16", 0.0, 0.02, seed=22)
    inp = W.make_inputs(w, "cuda")
    out = torch.full((B, T, H, d), float("nan"), device="cuda")
    st = torch.full((B, H, d, d), float("nan"), device="cuda")
    assert _named_call(gdn.lib().gdn_forward_bf16, inp, out, st) == gdn.OK
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    ref_out, ref_st = run_oracle(inp)
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


def test_null_state_means_zeros():
    w = W.Workload("z", 2, 9, 3, 64, "bf16", 0.0, 0.0, seed=9)
    inp = W.make_inputs(w, "cuda")
    assert inp["state"] is None
    check(inp, "bf16", "recurrent", TOL_RECURRENT)
    zeros = dict(inp, state=torch.zeros(2, 3, 64, 64, device="cuda"))
    o1, s1 = run_gpu(inp)
    o2, s2 = run_gpu(zeros)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_in_place_state_update():
    w = W.Workload("inplace", 2, 5, 4, 128, "bf16", 0.0, 0.02, seed=10)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    st = inp["state"].clone()
    out, st2 = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st, state_out=st)
    torch.cuda.synchronize()
    assert st2.data_ptr() == st.data_ptr()
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= TOL_RECURRENT and e_st <= TOL_RECURRENT


def test_zero_tokens_copies_state():
    w = W.Workload("t0", 2, 1, 2, 64, "f32", 0.0, 0.02, seed=11)
    inp = W.make_inputs(w, "cuda")
    e = lambda x: x[:, :0].contiguous()
    out, st = gdn.forward(e(inp["q"]), e(inp["k"]), e(inp["v"]), e(inp["g"]), e(inp["beta"]),
                          inp["state"])
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(st, inp["state"])
    out, st = gdn.forward(e(inp["q"]), e(inp["k"]), e(inp["v"]), e(inp["g"]), e(inp["beta"]), None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st) == 0


def test_state_carry_across_calls():
    """[0, T) in one call == [0, T1) then [T1, T) with the state fed back,
    including splits that are not chunk-aligned."""
    w = W.Workload("carry", 2, 300, 4, 128, "bf16", 0.0, 0.02, seed=12)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    for t1 in (1, 64, 100, 257):
        a = {key: (val[:, :t1].contiguous() if key != "state" else val) for key, val in inp.items()}
        b = {key: (val[:, t1:].contiguous() if key != "state" else None) for key, val in inp.items()}
        oa, sa = run_gpu(a)
        b["state"] = sa
        ob, sb = run_gpu(b)
        e_out, e_st = errs(torch.cat([oa, ob], dim=1), sb, ref_out, ref_st)
        assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (t1, e_out, e_st)


def test_no_writes_outside_outputs():
    """Outputs sit inside NaN-filled guard regions that must stay untouched."""
    w = W.Workload("guard", 2, 70, 3, 64, "bf16", 0.0, 0.02, seed=13)
    inp = W.make_inputs(w, "cuda")
    B, T, H, d = 2, 70, 3, 64
    pad = 4096
    for path in paths_for(d, T):
        ob = torch.full((B * T * H * d + 2 * pad,), float("nan"), device="cuda")
        sb = torch.full((B * H * d * d + 2 * pad,), float("nan"), device="cuda")
        out = ob[pad:pad + B * T * H * d].view(B, T, H, d)
        st = sb[pad:pad + B * H * d * d].view(B, H, d, d)
        gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                    out=out, state_out=st, path=path)
        torch.cuda.synchronize()
        for buf in (ob, sb):
            assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[-pad:]).all(), path
        assert torch.isfinite(out).all() and torch.isfinite(st).all()


def test_chunked_path_rejects_fp32_inputs():
    w = W.Workload("f32chunk", 1, 64, 2, 64, "f32", 0.0, 0.02, seed=15)
    inp = W.make_inputs(w, "cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                    path="chunked")
    assert ei.value.status == gdn.ERR_DTYPE


def test_rejects_bad_arguments_without_launching():
    """out overlapping state_in is rejected on the host; nothing is written."""
    w = W.Workload("bad", 1, 4, 2, 64, "bf16", 0.0, 0.02, seed=14)
    inp = W.make_inputs(w, "cuda")
    before = inp["state"].clone()
    bad_out = inp["state"].view(-1)[: 1 * 4 * 2 * 64].view(1, 4, 2, 64)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                    out=bad_out)
    torch.cuda.synchronize()
    assert ei.value.status == gdn.ERR_ALIAS
    assert torch.equal(inp["state"], before)


# ---------------------------------------------------------------- key heads

@pytest.mark.parametrize("path", ["recurrent", "chunked"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Hk", [1, 2, 4])
def test_fewer_key_heads(path, d, Hk):
    """q and k with Hk < H heads: value head i reads key head i % Hk (the
    tiled mapping).  Lengths span several chunks and a ragged tail."""
    H, T = 8, 150
    w = W.Workload(f"gqa_d{d}_hk{Hk}", 2, T, H, d, "bf16", 0.0, 0.02, seed=40 + Hk)
    inp = W.make_inputs(w, "cuda")
    inp["q"] = inp["q"][:, :, :Hk].contiguous()
    inp["k"] = inp["k"][:, :, :Hk].contiguous()
    check(inp, "bf16", path, TOL_RECURRENT if path == "recurrent" else None)


def test_fewer_key_heads_fp32_decode():
    H, Hk = 32, 16
    w = W.Workload("gqa_decode_f32", 4, 3, H, 128, "f32", 0.0, 0.02, seed=44)
    inp = W.make_inputs(w, "cuda")
    inp["q"] = inp["q"][:, :, :Hk].contiguous()
    inp["k"] = inp["k"][:, :, :Hk].contiguous()
    check(inp, "f32", "auto", TOL["f32"])


def test_fewer_key_heads_rejects_non_divisor():
    w = W.Workload("gqa_bad", 1, 4, 6, 64, "bf16", 0.0, 0.02, seed=45)
    inp = W.make_inputs(w, "cuda")
    with pytest.raises(ValueError):
        gdn.forward(inp["q"][:, :, :4].contiguous(), inp["k"][:, :, :4].contiguous(), inp["v"],
                    inp["g"], inp["beta"], inp["state"])


@pytest.mark.parametrize("wname", [W.MULTITOKEN_B64_T4.name, W.DECODE_B64_HK16.name])
def test_short_run_and_key_head_workloads_full_size(wname):
    """The benchmark's multi-token (4 tokens, 64 sequences) and fewer-key-heads
    decode workloads at full size, every output and the whole final state."""
    w = W.BY_NAME[wname]
    inp = W.make_inputs(w, "cuda")
    check(inp, w.dtype, "auto", TOL_RECURRENT)


@pytest.mark.parametrize("T", [2, 3, 7, 8, 9, 15, 16, 17, 23, 33, 63])
@pytest.mark.parametrize("d", [32, 64, 96, 128, 256])
def test_multi_token_runs_recurrent(T, d):
    """Short runs (2..63 tokens): windows of staged tokens with ragged last
    windows, for every head_dim, against the oracle."""
    w = W.Workload(f"short_d{d}_t{T}", 3, T, 4, d, "bf16", 0.0, 0.02, seed=60 + T)
    inp = W.make_inputs(w, "cuda")
    check(inp, "bf16", "recurrent", TOL_RECURRENT)


# ---------------------------------------------------------------- failure path

def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    """A wait that gives up (a barrier nothing completes, bounded to ~0.1 ms)
    reports GDN_ERR_TIMEOUT through the device status word, which the query
    clears; the next call runs normally."""
    L = gdn.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert gdn.device_status() == gdn.OK
    assert L.gdn_selftest_wait_timeout(ctypes.c_void_p(stream)) == gdn.OK
    assert gdn.device_status() == gdn.ERR_TIMEOUT
    assert gdn.device_status() == gdn.OK                 # read and cleared
    w = W.Workload("after_timeout", 1, 100, 2, 128, "bf16", 0.0, 0.02, seed=90)
    check(W.make_inputs(w, "cuda"), "bf16", "chunked")


# ------------------------------------------------- fused q / k normalisation

def raw_qk(inp, seed, Hk=None):
    """Unnormalised q, k in place of the workload's: N(0, 1) times a
    per-token, per-head power of two in [1/8, 8], and a few all-zero
    vectors (which must stay zero)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    out = dict(inp)
    for name in ("q", "k"):
        x = inp[name]
        B, T, Hx, d = x.shape
        raw = torch.randn((B, T, Hx, d), generator=gen, device="cuda")
        e = torch.randint(-3, 4, (B, T, Hx, 1), generator=gen, device="cuda").float()
        raw = raw * torch.pow(2.0, e)
        raw[:, T // 3::7, 0] = 0.0
        out[name] = raw.to(x.dtype).contiguous()
    return out


def check_l2norm(inp, dtype, path, tol):
    out, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                          path=path, l2norm_qk=True)
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    n = W.to_numpy_f32(inp)
    ref_out, ref_st = oracle.recurrent_c(n["q"], n["k"], n["v"], n["g"], n["beta"], n["state"],
                                         l2norm_qk=True)
    e_out, e_st = errs(out, st, ref_out, ref_st)
    assert e_out <= tol and e_st <= tol, (path, e_out, e_st)


@pytest.mark.parametrize("d", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("T", [1, 5, 70, 200])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fused_qk_l2norm(d, T, dtype):
    """q and k normalised inside the op (GDN_OPT_L2NORM_QK) on every path:
    the recurrent kernels fold the norms into their butterfly, the chunked
    kernels into per-token scalars of the chunk algebra."""
    w = W.Workload(f"l2n_d{d}_t{T}", 2, T, 4, d, dtype, 0.0, 0.02, seed=80 + T)
    inp = raw_qk(W.make_inputs(w, "cuda"), seed=81 + d)
    for path in ["auto"] + paths_for(d, T, dtype):
        tol = TOL_RECURRENT if path == "recurrent" else TOL[dtype]
        check_l2norm(inp, dtype, path, tol)


@pytest.mark.parametrize("H,Hk", [(48, 48), (48, 12), (8, 2)])
def test_fused_qk_l2norm_chunked_kernels_and_key_heads(H, Hk):
    """The one-kernel head_dim-128 path (96 pairs), fewer key heads, and the
    two-kernel path, with in-op normalisation and a ragged tail."""
    w = W.Workload(f"l2n_h{H}_hk{Hk}", 2, 150, H, 128, "bf16", 2.0, 0.02, seed=82)
    inp = W.make_inputs(w, "cuda")
    inp["q"] = inp["q"][:, :, :Hk].contiguous()
    inp["k"] = inp["k"][:, :, :Hk].contiguous()
    inp = raw_qk(inp, seed=83)
    for path in ("chunked", "recurrent"):
        check_l2norm(inp, "bf16", path, TOL_RECURRENT if path == "recurrent" else TOL["bf16"])


def test_fused_qk_l2norm_of_unit_inputs_changes_nothing_measurable():
    """On already-normalised inputs (the workloads') the option leaves the
    result within fp32 rounding of the plain call."""
    w = W.Workload("l2n_unit", 2, 130, 4, 128, "bf16", 0.0, 0.02, seed=84)
    inp = W.make_inputs(w, "cuda")
    for path in ("recurrent", "chunked"):
        o1, s1 = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                             path=path)
        o2, s2 = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                             path=path, l2norm_qk=True)
        torch.cuda.synchronize()
        rel = lambda a, b: ((a - b).abs().max() / b.pow(2).mean().sqrt()).item()
        # bf16 q / k normalised in fp32 have norms within ~2^-8 of 1
        assert rel(o2, o1) < 2e-2 and rel(s2, s1) < 2e-2, path


# ------------------------------------------------------------- bf16 output

def check_bf16_out(inp, path, l2norm=False):
    """GDN_OPT_OUT_BF16: the output is the fp32 output of the same call
    rounded to nearest even, element by element (torch converts float32 to
    bfloat16 the same way), and the state is the same bit for bit."""
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"])
    o32, s32 = gdn.forward(*args, path=path, l2norm_qk=l2norm)
    o16, s16 = gdn.forward(*args, path=path, l2norm_qk=l2norm, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    assert o16.dtype == torch.bfloat16 and o16.shape == o32.shape
    assert torch.equal(o16, o32.to(torch.bfloat16)), path
    assert torch.equal(s16, s32), path


@pytest.mark.parametrize("d", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("T", [1, 5, 70])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bf16_output_is_the_fp32_output_rounded(d, T, dtype):
    """Every path and head_dim: one-token and windowed recurrent kernels,
    and the chunked kernels over a ragged tail."""
    w = W.Workload(f"o16_d{d}_t{T}", 2, T, 4, d, dtype, 0.0, 0.02, seed=90 + T)
    inp = W.make_inputs(w, "cuda")
    for path in paths_for(d, T, dtype):
        check_bf16_out(inp, path)


@pytest.mark.parametrize("name,B,H,d", CHUNKED_KERNELS)
def test_bf16_output_on_every_chunked_kernel(name, B, H, d):
    """Each chunked kernel and state-walk width: the one-kernel path stages a
    bf16 O tile for its TMA store, the state walk stores 4 rounded values at
    a time; with and without q / k normalisation."""
    w = W.Workload(f"o16_{name}", B, 200, H, d, "bf16", 0.0, 0.05, seed=92)
    inp = W.make_inputs(w, "cuda")
    check_bf16_out(inp, "chunked")
    check_bf16_out(raw_qk(inp, seed=93), "chunked", l2norm=True)


def test_bf16_output_writes_nothing_outside_it():
    """A caller-provided bf16 output inside NaN guard regions (70 tokens: the
    last chunk is ragged), on both paths."""
    w = W.Workload("o16_guard", 2, 70, 3, 64, "bf16", 0.0, 0.02, seed=94)
    inp = W.make_inputs(w, "cuda")
    B, T, H, d = 2, 70, 3, 64
    pad = 4096
    for path in paths_for(d, T):
        ob = torch.full((B * T * H * d + 2 * pad,), float("nan"), dtype=torch.bfloat16,
                        device="cuda")
        out = ob[pad:pad + B * T * H * d].view(B, T, H, d)
        o, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                            out=out, path=path)
        torch.cuda.synchronize()
        assert o.data_ptr() == out.data_ptr()
        assert torch.isnan(ob[:pad]).all() and torch.isnan(ob[-pad:]).all(), path
        ref, _ = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                             path=path)
        torch.cuda.synchronize()
        assert torch.equal(out, ref.to(torch.bfloat16)), path


# ------------------------------------------------ random configuration sweep

def test_random_configurations_against_the_oracle():
    """A seeded sweep over the configuration space the other tests cover one
    axis at a time: sequences, tokens (chunk boundaries and ragged tails),
    heads and key heads, head_dim, dtype, gate regime, path, q/k
    normalisation and bf16 output together.  Each result is held to its
    path's bound against the oracle; a bf16 output additionally to its one
    rounding (2^-8 of each element's magnitude: bf16 keeps an 8-bit
    significand)."""
    rng = np.random.default_rng(2024)
    for case in range(40):
        d = int(rng.choice([32, 64, 96, 128, 256]))
        dtype = str(rng.choice(["bf16", "f32"]))
        B = int(rng.integers(1, 4))
        H = int(rng.choice([1, 2, 4, 6, 8]))
        Hk = int(rng.choice([x for x in range(1, H + 1) if H % x == 0]))
        T = int(rng.choice([1, 2, 7, 63, 64, 65, 130, 200]))
        g_shift = float(rng.choice([0.0, 2.0]))
        l2norm = bool(rng.integers(0, 2))
        out16 = bool(rng.integers(0, 2))
        paths = ["auto"] + paths_for(d, T, dtype)
        path = paths[int(rng.integers(0, len(paths)))]
        w = W.Workload(f"rand_{case}", B, T, H, d, dtype, g_shift, 0.02, seed=300 + case)
        inp = W.make_inputs(w, "cuda")
        inp["q"] = inp["q"][:, :, :Hk].contiguous()
        inp["k"] = inp["k"][:, :, :Hk].contiguous()
        if l2norm:
            inp = raw_qk(inp, seed=400 + case)
        out, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"],
                              path=path, l2norm_qk=l2norm,
                              out_dtype=torch.bfloat16 if out16 else torch.float32)
        torch.cuda.synchronize()
        assert gdn.device_status() == gdn.OK
        n = W.to_numpy_f32(inp)
        ref_out, ref_st = oracle.recurrent_c(n["q"], n["k"], n["v"], n["g"], n["beta"],
                                             n["state"], l2norm_qk=l2norm)
        e_out, e_st = errs(out.float(), st, ref_out, ref_st)
        chunked = path == "chunked" or (path == "auto" and
                                        gdn.select_path(B, T, H, d, dtype) == "chunked")
        tol = TOL["bf16"] if chunked else (TOL_RECURRENT if dtype == "bf16" else TOL[dtype])
        tol_out = tol
        if out16 and ref_out.size:
            tol_out += 2.0 ** -8 * float(np.abs(ref_out).max() / np.sqrt((ref_out ** 2).mean()))
        what = (case, B, T, H, Hk, d, dtype, path, l2norm, out16)
        assert e_out <= tol_out and e_st <= tol, (what, e_out, e_st)


# ------------------------------------------------ back-to-back state reuse

@pytest.mark.parametrize("T", [1, 5])
def test_default_reads_state_after_the_previous_kernel(T):
    """A call that reads the state the previous call on the stream is still
    writing (in place, back to back, launched with programmatic stream
    serialization) sees the finished state: ten chained steps equal one
    ten-token run."""
    w = W.Workload("chain", 2, 10 * T, 4, 128, "bf16", 0.0, 0.02, seed=23)
    inp = W.make_inputs(w, "cuda")
    ref_out, ref_st = run_oracle(inp)
    st = inp["state"].clone()
    outs = []
    for i in range(10):
        sl = slice(i * T, (i + 1) * T)
        o, _ = gdn.forward(inp["q"][:, sl].contiguous(), inp["k"][:, sl].contiguous(),
                           inp["v"][:, sl].contiguous(), inp["g"][:, sl].contiguous(),
                           inp["beta"][:, sl].contiguous(), st, state_out=st, path="recurrent")
        outs.append(o)
    torch.cuda.synchronize()
    e_out, e_st = errs(torch.cat(outs, dim=1), st, ref_out, ref_st)
    assert e_out <= TOL_RECURRENT and e_st <= TOL_RECURRENT, (e_out, e_st)


# ------------------------------------------------------------- maximum sizes

def _check_sample(w, inp, out, st, pairs, tol):
    ref_out, ref_st = sampled_reference(w, inp, pairs)
    got_out = np.stack([out[b, :, h].double().cpu().numpy() for b, h in pairs])
    got_st = np.stack([st[b, h].double().cpu().numpy() for b, h in pairs])
    e_out = oracle.parity_error(got_out.ravel(), ref_out.ravel())
    e_st = oracle.parity_error(got_st.ravel(), ref_st.ravel())
    assert e_out <= tol and e_st <= tol, (e_out, e_st)


def test_decode_with_65536_sequence_head_pairs():
    """One decode launch over 2048 sequences x 32 heads (a 65,536-row grid,
    4 GiB of fp32 state updated in place); the oracle recomputes a sample of
    pairs with at least one from every wave of blocks."""
    w = W.Workload("decode_b2048_h32_d128", 2048, 1, 32, 128, "bf16", 0.0, 0.02, seed=91)
    inp = W.make_inputs(w, "cuda")
    st0 = inp["state"]
    pairs = sampled_pairs(w, 24, per_cta=1)
    ref = sampled_reference(w, inp, pairs)            # before the in-place update
    out, st = gdn.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st0,
                          state_out=st0)
    torch.cuda.synchronize()
    assert gdn.device_status() == gdn.OK
    got_out = np.stack([out[b, :, h].double().cpu().numpy() for b, h in pairs])
    got_st = np.stack([st[b, h].double().cpu().numpy() for b, h in pairs])
    assert oracle.parity_error(got_out.ravel(), ref[0].ravel()) <= TOL_RECURRENT
    assert oracle.parity_error(got_st.ravel(), ref[1].ravel()) <= TOL_RECURRENT


@pytest.mark.parametrize("T,H,d", [(131072, 2, 64), (65536, 2, 128)])
def test_long_sequences_chunked(T, H, d):
    """Long runs on the chunked path: 2048 chunks of 64 tokens on the
    one-kernel path (head_dim 64) and 1024 chunks on the two-kernel path
    (head_dim 128, two (sequence, head) pairs, a 64 MiB transform workspace),
    every output and the final state against the oracle."""
    w = W.Workload(f"long_t{T}_d{d}", 1, T, H, d, "bf16", 0.0, 0.02, seed=92)
    inp = W.make_inputs(w, "cuda")
    out, st = run_gpu(inp, "chunked")
    _check_sample(w, inp, out, st, [(0, h) for h in range(H)], TOL["bf16"])


def test_long_run_recurrent_window():
    """65,536 tokens through the windowed recurrent kernel (8192 windows)."""
    w = W.Workload("long_rec", 1, 65536, 4, 64, "bf16", 0.0, 0.02, seed=93)
    inp = W.make_inputs(w, "cuda")
    out, st = run_gpu(inp, "recurrent")
    _check_sample(w, inp, out, st, [(0, h) for h in range(4)], TOL_RECURRENT)
