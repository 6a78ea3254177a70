"""Pins of the oracle's int8 K/V cache (rml "The decoder", KV cache: each group
of channels stored as round(x / s) with one float32 scale s = max|x| / 127, the
group the largest power of two dividing head_dim, at most 32).

Closed forms on exactly representable groups, the rounding rule at halves,
invariants that any correct quantiser keeps, the page's worked example, and
the wiring into the forward pass.  No GPU.
"""

import json
import os

import numpy as np
import pytest

from oracle.decoder_ref import (Session, dequantize_int8_groups, kv_group_size, kv_int8_roundtrip,
                                quantize_int8_groups)
from tests.oracle_helpers import random_weights, toy_cfg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("hd,g", [(128, 32), (64, 32), (96, 32), (80, 16), (48, 16), (16, 16), (24, 8),
                                  (8, 8), (6, 2), (2, 2)])
def test_group_is_largest_power_of_two_dividing_head_dim_capped_at_32(hd, g):
    assert kv_group_size(hd) == g


def test_worked_example_scales_per_row():
    # Llama 3.1 8B (the page's worked example): 8 kv heads of 128, kv_size 1024 -> groups of 32,
    # 32 scales per cached row.
    gold = json.load(open(os.path.join(GOLDEN, "kv_row_size.json")))
    g = kv_group_size(gold["head_dim"])
    codes, scales = quantize_int8_groups(np.linspace(-1, 1, gold["kv_size"]), g)
    assert codes.size == gold["kv_size"] and scales.size == gold["kv_size"] // 32


def test_integer_group_with_max_127_is_stored_exactly():
    # max|x| = 127 gives s = 1 exactly: integers are their own codes and read back exactly.
    x = np.array([127, -127, 63, -1, 0, 5, 100, -50], np.float64)
    codes, scales = quantize_int8_groups(x, 8)
    assert scales.tolist() == [1.0]
    assert codes.tolist() == x.astype(int).tolist()
    assert np.array_equal(dequantize_int8_groups(codes, scales, 8), x)


def test_halves_round_away_from_zero():
    x = np.array([127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 0.0])
    codes, _ = quantize_int8_groups(x, 8)
    assert codes.tolist() == [127, 3, -3, 1, -1, 2, -2, 0]


def test_scaled_grid_is_exact_for_power_of_two_scales():
    # max|x| = 127 * 2^-3: s = 2^-3 exactly, so x = k * 2^-3 has code k.
    k = np.array([-127, -64, -3, 0, 1, 7, 64, 127] * 4, np.float64)
    x = k * 0.125
    codes, scales = quantize_int8_groups(x, 32)
    assert scales.tolist() == [0.125]
    assert codes.tolist() == k.astype(int).tolist()


def test_zero_group_and_single_spike():
    x = np.zeros(64)
    x[40] = -3.0
    codes, scales = quantize_int8_groups(x, 32)
    assert scales[0] == 0.0 and not codes[:32].any()
    assert codes[40] == -127 and np.count_nonzero(codes) == 1
    np.testing.assert_array_equal(dequantize_int8_groups(codes, scales, 32)[:32], 0.0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invariants_on_random_rows(seed):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, rng.uniform(0.01, 10), 256) * rng.choice([1, 1e-3], 256)
    codes, scales = quantize_int8_groups(x, 32)
    deq = dequantize_int8_groups(codes, scales, 32)
    xg, dg, cg = x.reshape(-1, 32), deq.reshape(-1, 32), codes.reshape(-1, 32)
    for i in range(xg.shape[0]):
        m = np.abs(xg[i]).max()
        # the largest element maps to +-127, and the scale spans it: 127 s = max|x| to f32 rounding
        assert np.abs(cg[i]).max() == 127
        assert abs(127 * float(scales[i]) - m) <= 1e-6 * m
        # round to nearest: each value within half a step (plus float32 rounding of x and s)
        assert np.all(np.abs(dg[i] - xg[i]) <= 0.5 * float(scales[i]) * (1 + 1e-5) + 1e-6 * m)
    # odd symmetry
    c2, s2 = quantize_int8_groups(-x, 32)
    assert np.array_equal(c2, -codes) and np.array_equal(s2, scales)


def test_groups_never_straddle_heads():
    # head_dim 24 -> groups of 8; changing head 1 leaves head 0's stored values alone.
    rng = np.random.default_rng(5)
    row = rng.normal(size=(2, 24))
    a = kv_int8_roundtrip(row, 24)
    row2 = row.copy()
    row2[1] *= 1000.0
    b = kv_int8_roundtrip(row2, 24)
    assert np.array_equal(a[0], b[0])
    assert not np.array_equal(a[1], b[1])


def _toks(cfg, n, seed):
    return list(np.random.default_rng(seed).integers(0, cfg.vocab, n))


def test_session_stores_the_int8_roundtrip_of_layer_zero_keys():
    # Layer 0's K/V do not depend on the cache, so the int8 session's layer-0 rows are
    # exactly the round trip of the exact session's.
    cfg = toy_cfg(head_dim=16)
    cfg8 = toy_cfg(head_dim=16, kv_int8=True)
    w = random_weights(cfg, seed=3)
    toks = _toks(cfg, 7, 4)
    a, b = Session(cfg, w), Session(cfg8, w)
    a.prefill(toks, 0)
    b.prefill(toks, 0)
    for p in range(7):
        assert np.array_equal(b.keys[0][p], kv_int8_roundtrip(a.keys[0][p], 16))
        assert np.array_equal(b.values[0][p], kv_int8_roundtrip(a.values[0][p], 16))


def test_int8_prefill_equals_per_token_bit_exact():
    cfg = toy_cfg(kv_int8=True, sliding_window=5)
    w = random_weights(cfg, seed=6)
    toks = _toks(cfg, 9, 7)
    a = Session(cfg, w)
    rows = a.prefill(toks, 0, all_logits=True)
    b = Session(cfg, w)
    assert np.array_equal(rows, np.stack([b.forward(t, p) for p, t in enumerate(toks)]))


def test_int8_cache_changes_logits_by_a_quantisation_sized_amount():
    cfg, cfg8 = toy_cfg(), toy_cfg(kv_int8=True)
    w = random_weights(cfg, seed=8)
    toks = _toks(cfg, 10, 9)
    exact = Session(cfg, w).prefill(toks, 0, all_logits=True)
    q8 = Session(cfg8, w).prefill(toks, 0, all_logits=True)
    d = np.abs(q8 - exact).max()
    assert 0 < d < 0.05 * np.abs(exact).max()
