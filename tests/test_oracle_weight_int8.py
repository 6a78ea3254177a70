"""Pins of the oracle's 8-bit projection weights (Pantheon "Llama Forward Pass",
weight modes: the projections and an untied output matrix stay quantised and are
expanded a block at a time; embeddings and norms stay f32).  Each weight row is
stored in groups of 32 input columns by the int8 rule the pages print for the
cache (rml "The decoder", KV cache), whose quantiser is pinned in
test_oracle_kv_int8.py; here: exact grids, the wiring into the forward pass, what
stays unquantised, and the size of the effect.  No GPU."""

import numpy as np
import pytest

from oracle import DictWeights, Session
from oracle.decoder_ref import WEIGHT_GROUP, weight_int8_roundtrip
from tests.oracle_helpers import random_weights, toy_cfg

PROJ = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def _toks(cfg, n, seed):
    return list(np.random.default_rng(seed).integers(0, cfg.vocab, n))


def test_group_is_32_input_columns_and_grids_are_exact():
    assert WEIGHT_GROUP == 32
    rng = np.random.default_rng(0)
    k = rng.integers(-127, 128, (5, 64)).astype(np.float64)
    k[:, 0], k[:, 32] = 127, -127            # each group spans [-127, 127]: s = 1 exactly
    assert np.array_equal(weight_int8_roundtrip(k), k)
    assert np.array_equal(weight_int8_roundtrip(k * 0.25), k * 0.25)   # s = 2^-2
    with pytest.raises(ValueError):
        weight_int8_roundtrip(np.ones((2, 48)))


def _quantised_copy(w, cfg):
    layers = []
    for l in range(cfg.n_layers):
        lw = dict(w.layer(l))
        for r in PROJ:
            if lw.get(r) is not None:
                lw[r] = weight_int8_roundtrip(lw[r])
        layers.append(lw)
    experts = None
    if cfg.n_experts:
        experts = [[tuple(weight_int8_roundtrip(m) for m in w.expert(l, e)) for e in range(cfg.n_experts)]
                   for l in range(cfg.n_layers)]
    head = None if w._lm_head is None else weight_int8_roundtrip(w._lm_head)
    return DictWeights(w._embd, w._out_norm, layers, lm_head=head, experts=experts)


@pytest.mark.parametrize("kw", [dict(), dict(qkv_bias=True), dict(n_experts=4, n_experts_used=2)])
def test_session_uses_the_read_back_projections(kw):
    cfg = toy_cfg(ffn=64, **kw)
    cfg8 = toy_cfg(ffn=64, weight_int8=True, **kw)
    w = random_weights(cfg, seed=60)
    toks = _toks(cfg, 8, 61)
    got = Session(cfg8, w).prefill(toks, 0, all_logits=True)
    ref = Session(cfg, _quantised_copy(w, cfg)).prefill(toks, 0, all_logits=True)
    assert np.array_equal(got, ref)


def test_embedding_norms_router_and_tied_head_stay_exact():
    cfg8 = toy_cfg(ffn=64, weight_int8=True, n_experts=4, n_experts_used=2)
    w = random_weights(cfg8, seed=62)
    tied = DictWeights(w._embd, w._out_norm, w._layers, lm_head=None, experts=w._experts)
    s = Session(cfg8, tied)
    assert np.array_equal(s.w.lm_head(), tied.lm_head())
    assert np.array_equal(s.w.embed_rows([3, 5]), tied.embed_rows([3, 5]))
    lw, raw = s.w.layer(0), tied.layer(0)
    for r in ("attn_norm", "ffn_norm", "router"):
        assert np.array_equal(lw[r], raw[r])
    assert not np.array_equal(lw["wq"], raw["wq"])
    untied = Session(cfg8, w)
    assert not np.array_equal(untied.w.lm_head(), w.lm_head())


def test_quantisation_moves_logits_by_a_small_amount():
    cfg, cfg8 = toy_cfg(ffn=64), toy_cfg(ffn=64, weight_int8=True)
    w = random_weights(cfg, seed=63)
    toks = _toks(cfg, 10, 64)
    exact = Session(cfg, w).prefill(toks, 0, all_logits=True)
    q8 = Session(cfg8, w).prefill(toks, 0, all_logits=True)
    d = np.abs(q8 - exact).max()
    assert 0 < d < 0.05 * np.abs(exact).max()
