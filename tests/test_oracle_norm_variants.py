"""Pins of the oracle's optional norms (rml "The decoder", One forward pass: step
4, QK-norm of each head or each whole row before RoPE; step 6, sandwich norms
on each block's output before the residual add).  Checked against an
independent forward built from torch's float64 library routines, closed
forms and invariants.  No GPU."""

import numpy as np
import pytest

from oracle import Session
from tests.oracle_helpers import random_weights, toy_cfg, torch_library_forward

CASES = {
    "qk_head": dict(qk_norm="head"),
    "qk_row": dict(qk_norm="row"),
    "sandwich": dict(sandwich_norms=True),
    "qk_head_sandwich_gqa_window": dict(qk_norm="head", sandwich_norms=True, n_kv_heads=1, sliding_window=4),
    "qk_row_bias": dict(qk_norm="row", qkv_bias=True),
    "moe_sandwich": dict(sandwich_norms=True, n_experts=4, n_experts_used=2),
}


def _toks(cfg, n, seed):
    return list(np.random.default_rng(seed).integers(0, cfg.vocab, n))


@pytest.mark.parametrize("case", sorted(CASES))
def test_forward_matches_torch_library(case):
    cfg = toy_cfg(**CASES[case])
    w = random_weights(cfg, seed=40)
    toks = _toks(cfg, 9, 41)
    ref = torch_library_forward(cfg, w, toks)
    got = Session(cfg, w).prefill(toks, 0, all_logits=True)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_equals_per_token_and_batched(case):
    cfg = toy_cfg(**CASES[case])
    w = random_weights(cfg, seed=42)
    toks = _toks(cfg, 8, 43)
    rows = Session(cfg, w).prefill(toks, 0, all_logits=True)
    b = Session(cfg, w)
    assert np.array_equal(rows, np.stack([b.forward(t, p) for p, t in enumerate(toks)]))
    batched = Session(cfg, w).prefill_batched(toks, 0, logits_rows=range(8))
    np.testing.assert_allclose(batched, rows, rtol=1e-12, atol=1e-12)


def test_qk_norm_head_gives_unit_rms_heads():
    # With k_norm weights 1, every cached key head has RMS sqrt(ms / (ms + eps)) before
    # RoPE, and RoPE keeps each pair's norm: so |k_head| = sqrt(hd * ms / (ms + eps)) ~ sqrt(hd).
    cfg = toy_cfg(qk_norm="head", rms_eps=1e-12)
    w = random_weights(cfg, seed=44)
    for l in range(cfg.n_layers):
        w._layers[l]["k_norm"] = np.ones(cfg.head_dim)
    s = Session(cfg, w)
    s.prefill(_toks(cfg, 6, 45), 0)
    for l in range(cfg.n_layers):
        for k in s.keys[l]:
            np.testing.assert_allclose(np.linalg.norm(k, axis=-1), np.sqrt(cfg.head_dim), rtol=1e-9)


def test_qk_norm_row_normalises_the_whole_row_not_each_head():
    cfg = toy_cfg(qk_norm="row", rms_eps=1e-12)
    w = random_weights(cfg, seed=46)
    for l in range(cfg.n_layers):
        w._layers[l]["k_norm"] = np.ones(cfg.n_kv_heads * cfg.head_dim)
    s = Session(cfg, w)
    s.prefill(_toks(cfg, 5, 47), 0)
    for k in s.keys[0]:
        assert abs(np.linalg.norm(k) - np.sqrt(k.size)) < 1e-9
        heads = np.linalg.norm(k, axis=-1)
        assert np.ptp(heads) > 1e-3     # heads are not each normalised


@pytest.mark.parametrize("mode", ["head", "row"])
def test_qk_norm_removes_the_scale_of_wq_and_wk(mode):
    cfg = toy_cfg(qk_norm=mode, rms_eps=1e-14)
    w = random_weights(cfg, seed=48)
    toks = _toks(cfg, 7, 49)
    a = Session(cfg, w).prefill(toks, 0, all_logits=True)
    for l in range(cfg.n_layers):
        w._layers[l]["wq"] = w._layers[l]["wq"] * 7.0
        w._layers[l]["wk"] = w._layers[l]["wk"] * 0.25
    b = Session(cfg, w).prefill(toks, 0, all_logits=True)
    np.testing.assert_allclose(b, a, rtol=1e-8, atol=1e-9)


def test_sandwich_with_zero_post_weights_passes_the_embedding_through():
    cfg = toy_cfg(sandwich_norms=True)
    w = random_weights(cfg, seed=50)
    for l in range(cfg.n_layers):
        w._layers[l]["post_attn_norm"] = np.zeros(cfg.hidden)
        w._layers[l]["post_ffn_norm"] = np.zeros(cfg.hidden)
    toks = _toks(cfg, 4, 51)
    got = Session(cfg, w).prefill(toks, 0, all_logits=True)
    x = w.embed_rows(toks)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    ref = (x / np.sqrt(ms + cfg.rms_eps) * w.out_norm()) @ w.lm_head().T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- per-layer RoPE base
@pytest.mark.parametrize("every", [0, 2, 3])
def test_per_layer_rope_base_matches_torch_library(every):
    cfg = toy_cfg(n_layers=3, rope_theta_local=50.0, rope_global_every=every)
    w = random_weights(cfg, seed=52)
    toks = _toks(cfg, 9, 53)
    ref = torch_library_forward(cfg, w, toks)
    got = Session(cfg, w).prefill(toks, 0, all_logits=True)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-11)
    b = Session(cfg, w).prefill_batched(toks, 0, logits_rows=range(9))
    np.testing.assert_allclose(b, got, rtol=1e-12, atol=1e-12)


def test_local_base_equal_to_global_is_the_plain_model():
    cfg = toy_cfg(n_layers=3)
    cfg2 = toy_cfg(n_layers=3, rope_theta_local=cfg.rope_theta, rope_global_every=3)
    w = random_weights(cfg, seed=54)
    toks = _toks(cfg, 7, 55)
    assert np.array_equal(Session(cfg, w).prefill(toks, 0, all_logits=True),
                          Session(cfg2, w).prefill(toks, 0, all_logits=True))


def test_global_layer_pattern():
    cfg = toy_cfg(n_layers=7, rope_theta_local=10.0, rope_global_every=3)
    assert [cfg.layer_is_global(l) for l in range(7)] == [False, False, True, False, False, True, False]
    assert not any(toy_cfg(n_layers=4, rope_theta_local=10.0).layer_is_global(l) for l in range(4))
    assert all(toy_cfg(n_layers=4).layer_is_global(l) for l in range(4))


def test_local_base_changes_only_local_layers_keys():
    # Layer 0's keys do not depend on the cache: with layer 0 global (every=1) they equal the
    # plain model's; with layer 0 local they are the plain keys rotated by the local base.
    cfg = toy_cfg(n_layers=2)
    w = random_weights(cfg, seed=56)
    toks = _toks(cfg, 5, 57)
    plain = Session(cfg, w)
    plain.prefill(toks, 0)
    glob = Session(toy_cfg(n_layers=2, rope_theta_local=50.0, rope_global_every=1), w)
    glob.prefill(toks, 0)
    loc = Session(toy_cfg(n_layers=2, rope_theta_local=50.0, rope_global_every=2), w)
    loc.prefill(toks, 0)
    for p in range(5):
        assert np.array_equal(glob.keys[0][p], plain.keys[0][p])
        if p > 0:
            assert not np.allclose(loc.keys[0][p], plain.keys[0][p])
        np.testing.assert_allclose(np.linalg.norm(loc.keys[0][p], axis=-1),
                                   np.linalg.norm(plain.keys[0][p], axis=-1), rtol=1e-12)
