"""GPU parity for decode attention (the flash_attn op) against the float64
oracle (oracle/attn.py), through the C ABI via the binding.

Metric: max |gpu - oracle| / RMS(oracle) over the whole output.  The kernel
accumulates in fp32 from exactly upcast inputs; scores carry a relative
error of a few fp32 ulps times sqrt(head_dim), which moves the softmax
weights by well under 1e-5 of themselves at these score magnitudes, so the
bound is 1e-4 (fully masked rows and an empty cache must give exact zeros).
"""
import numpy as np
import pytest
import torch

import linear_attention_sequence_gated_gb300 as gdn
from linear_attention_sequence_gated_gb300 import workloads as W
from oracle.attn import attention
import oracle

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_attention_sequence_gated_gb300 import _build
    _build.build()


def np64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def run_and_check(w, scale=None, tol=TOL):
    inp = W.make_attn_inputs(w, "cuda")
    out = gdn.flash_attn(inp["q"], inp["k"], inp["v"], inp["mask"], scale)
    torch.cuda.synchronize()
    s = 1.0 / np.sqrt(w.d) if scale is None else scale      # w.d: the q / k width
    # the oracle takes the kernel's scale as the float32 value it receives
    s = float(np.float32(s))
    ref = attention(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), np64(inp["mask"]), s)
    got = out.double().cpu().numpy()
    assert got.shape == ref.shape
    err = oracle.parity_error(got, ref)
    assert err <= tol, (w, err)
    return got, ref


@pytest.mark.parametrize("wname", list(W.ATTN_BY_NAME))
def test_benchmark_workloads_full_size(wname):
    run_and_check(W.ATTN_BY_NAME[wname])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("dk,dv", [(64, 128), (64, 256), (128, 64), (128, 256), (256, 64),
                                   (256, 128)])
@pytest.mark.parametrize("n_kv", [1, 33, 257, 1000])
def test_unequal_key_and_value_widths(dtype, dk, dv, n_kv):
    """head_dim_k != head_dim_v (the model card's capability query takes the
    two widths apart): every pair of 64 / 128 / 256, grouped heads, a mask."""
    w = W.AttnWorkload(f"kv_{dtype}_{dk}_{dv}_{n_kv}", 2, 8, 2, 3, n_kv, dk, dtype, mask=True,
                       mask_std=1.0, seed=n_kv + dk + 3 * dv, dv_=dv)
    got, _ = run_and_check(w)
    assert got.shape == (2, 3, 8, dv)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("n_kv", [1, 31, 32, 33, 141, 257, 1000])
def test_matrix(dtype, d, n_kv):
    w = W.AttnWorkload(f"m_{dtype}_{d}_{n_kv}", 2, 8, 2, 3, n_kv, d, dtype, mask=True,
                       mask_std=1.0, seed=n_kv + d)
    run_and_check(w)


@pytest.mark.parametrize("H,Hkv,n_q", [(8, 8, 1), (16, 4, 1), (32, 1, 19), (12, 3, 7), (4, 2, 19)])
def test_head_groups_and_query_counts(H, Hkv, n_q):
    """Rows of a kv head = (n_heads / n_heads_kv) * n_q, several 16-row blocks
    when large (32 query heads over one kv head with 19 queries: 608 rows)."""
    w = W.AttnWorkload(f"g_{H}_{Hkv}_{n_q}", 2, H, Hkv, n_q, 300, 128, "bf16", mask=True,
                       mask_std=0.5, seed=H * 100 + n_q)
    run_and_check(w)


def test_long_cache_many_tiles_per_cta():
    w = W.AttnWorkload("long", 2, 8, 2, 2, 20000, 128, "bf16", seed=5)
    run_and_check(w)


def test_causal_tail_and_fully_masked_rows():
    """A causal tail on the newest keys; with a tail longer than the cache
    the first queries see no key at all and must come back as zero rows."""
    w = W.AttnWorkload("causal", 2, 8, 4, 5, 200, 64, "bf16", mask=True, masked_tail=4, seed=6)
    run_and_check(w)
    w2 = w.replace(name="all_masked", n_kv=40, masked_tail=42, seed=7)
    got, ref = run_and_check(w2)
    # query 0 sees keys j < 40 - 42 + 0: none
    assert np.all(got[:, 0] == 0.0) and np.all(ref[:, 0] == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_scale_argument_and_large_scores(dtype):
    """Peaked and uniform softmax on both kernel paths (packed FMAs for fp32,
    tensor-core MMAs with hi + lo probabilities for 16-bit inputs)."""
    w = W.AttnWorkload(f"scale_{dtype}", 1, 4, 4, 2, 100, 256, dtype, seed=8)
    run_and_check(w, scale=1.0)        # scores of magnitude ~ 16: a peaked softmax
    run_and_check(w, scale=0.0)        # uniform weights: the mean of v


def test_empty_cache_gives_zeros():
    w = W.AttnWorkload("empty", 2, 4, 2, 3, 0, 128, "bf16", seed=9)
    inp = W.make_attn_inputs(w, "cuda")
    out = torch.full((2, 3, 4, 128), 7.0, device="cuda")
    gdn.flash_attn(inp["q"], inp["k"], inp["v"], None, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_rejects_unsupported_shapes():
    w = W.AttnWorkload("wide", 1, 4, 4, 20, 64, 128, "bf16", seed=10)
    inp = W.make_attn_inputs(w, "cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.flash_attn(inp["q"], inp["k"], inp["v"])
    assert e.value.status == gdn.ERR_SHAPE
