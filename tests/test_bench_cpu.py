"""The roofline arithmetic of bench.py, pinned to the figures the design
states (CPU only).  These are the algorithmic bytes and flops that the
reported `achieved` numbers divide by the measured time."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from linear_attention_sequence_gated_gb300 import workloads as W  # noqa: E402


def test_decode_bytes():
    # 8 d^2 (fp32 state in and out) + 3 d * 2 (bf16 q, k, v) + 4 d (fp32 out) + 8 (g, beta)
    assert bench.decode_bytes_per_head(128, 2) == 131072 + 768 + 512 + 8 == 132360
    # one 32-head layer: 4.24 MB per launch; 64 sequences: 271.1 MB
    assert bench.run_bytes(1, 1, 32, 32, 128, 2) == 32 * 132360 == 4235520
    assert bench.run_bytes(64, 1, 32, 32, 128, 2) == 64 * 32 * 132360 == 271073280
    # 16 key heads for 32 value heads: q and k are read once per key head
    assert bench.run_bytes(64, 1, 32, 16, 128, 2) == 271073280 - 64 * 16 * 2 * 128 * 2
    # a 4-token run: the state once, per-token inputs four times
    assert bench.run_bytes(64, 4, 32, 32, 128, 2) == 64 * 32 * (131072 + 4 * 1288)


def test_prefill_bytes_and_flops():
    assert bench.prefill_bytes_per_token_head(128, 2) == 1288
    # issued MMA tiles per (token, head) at C = 64: 10 C d + 6 d^2
    assert bench.chunked_flops_per_token_head(128) == 81920 + 98304 == 180224
    assert bench.chunked_flops_per_token_head(64) == 65536
    assert bench.chunked_flops_per_token_head(256) == 557056
    # the 4096-token prefill: 23.6 GFLOP per call
    w = W.PREFILL_4K
    assert w.B * w.T * w.H * bench.chunked_flops_per_token_head(w.d) == 23622320128


def test_attention_bytes():
    # 64 sequences x 8 kv heads x 4096 keys x 128 (bf16 k and v), 32 query heads, one query,
    # fp32 output: 1.075 GB per call
    w = W.ATTN_B64_KV4K
    kv = 2 * 64 * 8 * 4096 * 128 * 2
    q = 64 * 32 * 1 * 128 * 2
    out = 64 * 1 * 32 * 128 * 4
    mask = 64 * 1 * 4096 * 2 if w.mask else 0
    assert bench.attn_bytes(w, 2) == kv + q + out + mask == 1075314688


def test_launch_counts():
    assert bench.launches_per_call("recurrent", 0) == 1
    assert bench.launches_per_call("chunked", 0) == 1          # one-kernel chunked path
    assert bench.launches_per_call("chunked", 1 << 20) == 2    # transform pass + state walk
    # the state walk's value-block split on 152 SMs: one launch of 32-row
    # blocks (32 pairs x 128), one of 64-row blocks filling whole waves (76
    # pairs x 128), or full waves of 64-row blocks then the rest at 32 rows
    # (8 x 16 pairs x 256: 114 + 14; 77 x 128: 76 + 1)
    assert bench.launches_per_call("chunked", 1, 32, 128, 152) == 2
    assert bench.launches_per_call("chunked", 1, 76, 128, 152) == 2
    assert bench.launches_per_call("chunked", 1, 128, 256, 152) == 3
    assert bench.launches_per_call("chunked", 1, 77, 128, 152) == 3
    assert bench.launches_per_call("chunked", 1, 40, 256, 152) == 3
    assert bench.launches_per_call("chunked", 1, 60, 256, 152) == 2    # rest of 22 > one 32-row wave


def test_one_thread_oracle_call_keeps_the_default_thread_count():
    """The bench times the oracle on one thread once; the CPU baselines
    measured after it must still see every OpenMP thread."""
    import numpy as np
    import oracle
    oracle.build()
    before = oracle.max_threads()
    rng = np.random.default_rng(0)
    x = {n: rng.standard_normal(s).astype(np.float32)
         for n, s in (("q", (1, 2, 2, 8)), ("k", (1, 2, 2, 8)), ("v", (1, 2, 2, 8)),
                      ("g", (1, 2, 2)), ("beta", (1, 2, 2)))}
    oracle.recurrent_c(x["q"], x["k"], x["v"], -np.abs(x["g"]), x["beta"], None, n_threads=1)
    assert oracle.max_threads() == before
