"""Host-side pins of bench.py's accounting: the decode roofline's algorithmic bytes,
the prefill FLOPs, the traffic table's consistency and the phase names."""

import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from decoder_only_forward_gb300 import synthetic  # noqa: E402


def test_mixtral_decode_bytes_by_hand():
    # One decode step at position 1026 (1027 readable K/V rows, f32 cache), counted by hand:
    #   per layer: Wq|Wk|Wv (4096 + 2*1024) x 4096, Wo 4096 x 4096, two experts' gate/up
    #   2 x 2 x 14336 x 4096 and down 2 x 4096 x 14336, router 8 x 4096 (all bf16),
    #   two f32 norm vectors of 4096, and K/V 2 x 8 x 128 x 1027 f32 values;
    #   then the head 32000 x 4096 bf16, one embedding row and the f32 output norm.
    per_layer = (2 * ((4096 + 2048) * 4096 + 4096 * 4096 + 2 * 2 * 14336 * 4096 + 2 * 4096 * 14336 + 8 * 4096)
                 + 2 * 4 * 4096 + 2 * 8 * 128 * 1027 * 4)
    total = 32 * per_layer + 2 * 32000 * 4096 + 2 * 4096 + 4 * 4096
    assert total == 25_767_469_056
    assert bench.decode_bytes(synthetic.workload("mixtral-8x7b"), 1026, 4) == total


def test_sliding_window_caps_the_kv_read():
    w = synthetic.workload("mistral-7b")
    a = bench.decode_bytes(w, 4095, 4)     # the window is full at position 4095
    b = bench.decode_bytes(w, 9000, 4)
    assert a == b
    c = bench.decode_bytes(w, 100, 4)
    assert a - c == w["n_layers"] * 2 * w["n_kv_heads"] * w["head_dim"] * (4096 - 101) * 4


def test_prefill_flops_by_hand_on_the_toy():
    w = synthetic.workload("toy")
    h, f, hd, nq, nkv, V, L = w["hidden"], w["ffn"], w["head_dim"], w["n_heads"], w["n_kv_heads"], w["vocab"], \
        w["n_layers"]
    P = 10
    lin = (nq + 2 * nkv) * hd * h + h * nq * hd + 3 * f * h
    attn = 4 * hd * nq * P * (P + 1) // 2
    assert bench.prefill_flops(w, P) == L * (2 * P * lin + attn) + 2 * V * h


def test_traffic_table_is_near_the_algorithmic_bytes():
    # A stored DRAM measurement of the decode step (keyed to the current source) lies
    # within 2% of the algorithmic bytes of the captured position.
    t = bench.measured_traffic("mixtral-8x7b", "step")
    if t is None:
        pytest.skip("no traffic figure for the current decode source")
    alg = bench.decode_bytes(synthetic.workload("mixtral-8x7b"), 1026, 4)
    assert alg <= t <= 1.02 * alg
    assert bench.measured_traffic("mixtral-8x7b", "no-such-kernel") is None


@pytest.mark.parametrize("fused", [False, True])
def test_phase_summary_names_and_sums(fused):
    w = dict(synthetic.workload("toy"), n_layers=3)
    ppl = 5
    n = w["n_layers"] * ppl + 1
    rng = np.random.default_rng(0)
    rows = []
    for _ in range(4):
        d = rng.integers(1000, 5000, n)
        rows.append(np.concatenate([[0], np.cumsum(d)]).astype(np.int64))
    out = bench.phase_summary(w, rows, False, fused)
    names = ["qkv", "attn", "oproj"] + (["ffn", "ffn_sum"] if fused else ["gateup", "down"])
    assert [k for k in out if k not in ("lmhead", "total")] == names
    assert abs(sum(out[k] for k in names) + out["lmhead"] - out["total"]) < 0.5
