"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a closed
form, an invariant, a worked example printed on a page (tests/golden/), or a
library routine that computes the same definition.  None needs a GPU.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import (DictWeights, OracleConfig, Session, attend_ref, kv_head_of, llama3_scale_inv_freq,
                    moe_ffn, rmsnorm, rope_inv_freq, rope_rotate, route_topk, silu, swiglu,
                    window_start)
from tests.oracle_helpers import random_weights, toy_cfg, torch_library_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("c,eps", [(1.0, 1e-5), (-3.0, 1e-6), (0.01, 1e-5), (0.0, 1e-5)])
def test_rmsnorm_constant_vector_closed_form(c, eps):
    # Pantheon "Llama Forward Pass", RMSNorm: for x = c*1, mean(x^2) = c^2.
    w = np.linspace(0.5, 1.5, 24)
    got = rmsnorm(np.full(24, c), w, eps)
    np.testing.assert_allclose(got, c / math.sqrt(c * c + eps) * w, rtol=1e-15, atol=0)


def test_rmsnorm_matches_torch_library():
    rng = np.random.default_rng(1)
    x, w = rng.normal(size=(5, 96)), rng.normal(size=96)
    ref = F.rms_norm(torch.tensor(x), (96,), weight=torch.tensor(w), eps=1e-6).numpy()
    np.testing.assert_allclose(rmsnorm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- SiLU / SwiGLU
def test_silu_closed_forms():
    assert silu(0.0) == 0.0
    assert abs(silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(silu(50.0) - 50.0) < 1e-15
    assert abs(silu(-50.0)) < 1e-19
    z = np.random.default_rng(2).normal(0, 4, 1000)
    np.testing.assert_allclose(silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-14, atol=1e-300)


def test_swiglu_identity_weights_closed_form():
    # With W_gate = W_up = W_down = I the FFN reduces to silu(n) * n.
    n = np.random.default_rng(3).normal(size=16)
    eye = np.eye(16)
    np.testing.assert_allclose(swiglu(n, eye, eye, eye), n / (1 + np.exp(-n)) * n, rtol=1e-15)


def test_swiglu_orientation_nonsquare():
    # Gate/up are [ffn, hidden], down is [hidden, ffn]: a transposed operand fails here.
    rng = np.random.default_rng(4)
    n, wg, wu, wd = rng.normal(size=8), rng.normal(size=(5, 8)), rng.normal(size=(5, 8)), rng.normal(size=(8, 5))
    g = sum(wg[:, i] * n[i] for i in range(8))
    u = sum(wu[:, i] * n[i] for i in range(8))
    a = g / (1 + np.exp(-g)) * u
    np.testing.assert_allclose(swiglu(n, wg, wu, wd), sum(wd[:, r] * a[r] for r in range(5)), rtol=1e-12)


# ---------------------------------------------------------------- RoPE
def test_rope_identity_at_position_zero():
    v = np.random.default_rng(5).normal(size=(3, 16))
    np.testing.assert_array_equal(rope_rotate(v, 0, rope_inv_freq(16, 10000.0)), v)


@pytest.mark.parametrize("i", [0, 1, 5, 7])
def test_rope_adjacent_pair_and_frequency(i):
    # sipllm "RoPE is adjacent-pair": pair i is (v[2i], v[2i+1]); rml "Rotary
    # embeddings": it turns theta^(-2i/head_dim) radians per position.
    hd, theta, pos = 16, 10000.0, 37
    v = np.zeros(hd)
    v[2 * i] = 1.0
    out = rope_rotate(v, pos, rope_inv_freq(hd, theta))
    ang = pos * theta ** (-2.0 * i / hd)
    expect = np.zeros(hd)
    expect[2 * i], expect[2 * i + 1] = math.cos(ang), math.sin(ang)
    np.testing.assert_allclose(out, expect, atol=1e-15)


def test_rope_pair_norms_preserved():
    v = np.random.default_rng(6).normal(size=(4, 32))
    out = rope_rotate(v, 1234, rope_inv_freq(32, 1e6))
    np.testing.assert_allclose(np.hypot(out[:, 0::2], out[:, 1::2]), np.hypot(v[:, 0::2], v[:, 1::2]), rtol=1e-14)


def test_rope_composition():
    inv = rope_inv_freq(16, 10000.0)
    v = np.random.default_rng(7).normal(size=16)
    np.testing.assert_allclose(rope_rotate(rope_rotate(v, 11, inv), 29, inv), rope_rotate(v, 40, inv), atol=1e-13)


def test_rope_relative_position_invariance():
    # rml "Rotary embeddings": q . k depends only on the distance between tokens.
    inv = rope_inv_freq(32, 10000.0)
    rng = np.random.default_rng(8)
    q, k = rng.normal(size=32), rng.normal(size=32)
    a = rope_rotate(q, 100, inv) @ rope_rotate(k, 93, inv)
    b = rope_rotate(q, 7, inv) @ rope_rotate(k, 0, inv)
    assert abs(a - b) < 1e-12


def test_rope_matches_complex_multiplication():
    hd, pos = 16, 523
    inv = rope_inv_freq(hd, 1e6)
    v = np.random.default_rng(9).normal(size=(2, hd))
    c = torch.view_as_complex(torch.tensor(v).reshape(2, hd // 2, 2))
    c = c * torch.polar(torch.ones(hd // 2, dtype=torch.float64), torch.tensor(pos * inv))
    np.testing.assert_allclose(rope_rotate(v, pos, inv), torch.view_as_real(c).reshape(2, hd).numpy(), atol=1e-14)


def test_rope_adjacent_equals_rotate_half_on_permuted_dims():
    # sipllm: adjacent-pair RoPE reproduces HF rotate_half only through a row
    # permutation (adjacent pair i <-> dims (i, i + hd/2)).  rotate_half is
    # written here independently: x * cos + rotate_half(x) * sin.
    hd, pos = 16, 77
    inv = rope_inv_freq(hd, 10000.0)
    x = np.random.default_rng(10).normal(size=hd)
    perm = np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])   # half layout <- adjacent layout
    xh = x[perm]
    ang = np.concatenate([pos * inv, pos * inv])
    rot_half = np.concatenate([-xh[hd // 2:], xh[:hd // 2]])
    yh = xh * np.cos(ang) + rot_half * np.sin(ang)
    y = np.empty(hd)
    y[perm] = yh
    np.testing.assert_allclose(rope_rotate(x, pos, inv), y, atol=1e-14)


def test_rope_half_style_is_rotate_half():
    # rml "Which dimensions pair": kHalf pairs dim i with i + head_dim/2, i.e. HF's
    # x * cos + rotate_half(x) * sin, written here independently.
    hd, pos = 16, 91
    inv = rope_inv_freq(hd, 10000.0)
    x = np.random.default_rng(11).normal(size=(3, hd))
    ang = np.concatenate([pos * inv, pos * inv])
    rot_half = np.concatenate([-x[:, hd // 2:], x[:, :hd // 2]], axis=1)
    np.testing.assert_allclose(rope_rotate(x, pos, inv, half=True), x * np.cos(ang) + rot_half * np.sin(ang),
                               atol=1e-14)


def test_rope_half_style_matches_complex_multiplication():
    hd, pos = 32, 1311
    inv = rope_inv_freq(hd, 1e6)
    v = np.random.default_rng(12).normal(size=hd)
    z = (v[:hd // 2] + 1j * v[hd // 2:]) * np.exp(1j * pos * inv)
    np.testing.assert_allclose(rope_rotate(v, pos, inv, half=True), np.concatenate([z.real, z.imag]), atol=1e-13)


@pytest.mark.parametrize("half", [False, True])
def test_partial_rotary_passes_the_tail_through(half):
    # sipllm partial-rotary (rope_rot): only the first rope_dim dims turn, the rest
    # pass through; the rotated part is a full rotation of a rope_dim-wide head.
    hd, rd, pos, theta = 32, 12, 57, 10000.0
    inv = rope_inv_freq(hd, theta, rope_dim=rd)
    assert inv.shape == (rd // 2,)
    v = np.random.default_rng(13).normal(size=(2, hd))
    out = rope_rotate(v, pos, inv, half=half, rope_dim=rd)
    np.testing.assert_array_equal(out[:, rd:], v[:, rd:])
    np.testing.assert_allclose(out[:, :rd], rope_rotate(v[:, :rd], pos, rope_inv_freq(rd, theta), half=half),
                               atol=1e-14)


def test_partial_rotary_frequencies_closed_form():
    # inv_freq[i] = theta^(-2i/rope_dim): with rope_dim 4 and theta 1e4 the two pairs
    # turn 1 and 1e-2 radians per position whatever head_dim is.
    np.testing.assert_allclose(rope_inv_freq(64, 1e4, rope_dim=4), [1.0, 1e-2], rtol=1e-15)


@pytest.mark.parametrize("half,rd", [(True, 0), (True, 12), (False, 12)])
def test_rope_variants_keep_relative_position_invariance(half, rd):
    hd = 32
    inv = rope_inv_freq(hd, 10000.0, rope_dim=rd)
    rng = np.random.default_rng(14)
    q, k = rng.normal(size=hd), rng.normal(size=hd)
    a = rope_rotate(q, 250, inv, half, rd) @ rope_rotate(k, 243, inv, half, rd)
    b = rope_rotate(q, 9, inv, half, rd) @ rope_rotate(k, 2, inv, half, rd)
    assert abs(a - b) < 1e-12


def test_half_style_model_equals_adjacent_model_on_permuted_qk_rows():
    # The same decoder with kHalf pairing and with adjacent pairing on q/k weight
    # rows permuted per head ((i, i + d/2) -> (2i, 2i+1)) gives the same logits:
    # attention sees only q . k, which the consistent permutation leaves unchanged.
    cfg_h = toy_cfg(rope_dim=8, rope_half=True)
    cfg_a = toy_cfg(rope_dim=8)
    w = random_weights(cfg_h, seed=21)
    hd, rd = cfg_h.head_dim, 8
    src = np.concatenate([np.stack([np.arange(rd // 2), np.arange(rd // 2) + rd // 2], 1).ravel(),
                          np.arange(rd, hd)])          # permuted row p <- original row src[p]

    def permute(m, heads):
        return np.concatenate([m[h * hd + src] for h in range(heads)])

    layers = []
    for l in range(cfg_h.n_layers):
        lw = w.layer(l)
        layers.append(dict(lw, wq=permute(lw["wq"], cfg_h.n_heads), wk=permute(lw["wk"], cfg_h.n_kv_heads)))
    wp = DictWeights(w.embed_rows(np.arange(cfg_h.vocab)), w.out_norm(), layers, lm_head=w.lm_head())
    toks = [3, 1, 4, 1, 5, 9, 2, 6]
    a = Session(cfg_h, w).prefill(toks, 0, all_logits=True)
    b = Session(cfg_a, wp).prefill(toks, 0, all_logits=True)
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_llama3_worked_example():
    g = _golden("llama3_rope_worked_example.json")
    p = g["params"]
    for case in g["cases"]:
        inv = np.array([2 * math.pi / case["wavelength"]])
        out = llama3_scale_inv_freq(inv, **p)
        assert abs(out[0] / inv[0] - case["ratio_to_original"]) < 1e-12, case


def test_llama3_scaling_applied_by_inv_freq():
    p = dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, orig_ctx=8192.0)
    plain = rope_inv_freq(128, 500000.0)
    scaled = rope_inv_freq(128, 500000.0, p)
    wl = 2 * math.pi / plain
    assert np.all(scaled[wl < 2048] == plain[wl < 2048])
    np.testing.assert_allclose(scaled[wl > 8192], plain[wl > 8192] / 8, rtol=1e-15)
    mid = (wl >= 2048) & (wl <= 8192)
    assert mid.any() and np.all(scaled[mid] <= plain[mid]) and np.all(scaled[mid] >= plain[mid] / 8)


# ---------------------------------------------------------------- attention
def test_attend_single_key_returns_its_value():
    rng = np.random.default_rng(11)
    q, k, v = rng.normal(size=(4, 8)), rng.normal(size=(1, 2, 8)), rng.normal(size=(1, 2, 8))
    out = attend_ref(q, k, v, 4, 2)
    for h in range(4):
        np.testing.assert_array_equal(out[h], v[0, h // 2])


def test_attend_equal_keys_is_mean_of_values():
    rng = np.random.default_rng(12)
    q = rng.normal(size=(4, 8))
    k = np.tile(rng.normal(size=(1, 2, 8)), (9, 1, 1))
    v = rng.normal(size=(9, 2, 8))
    out = attend_ref(q, k, v, 4, 2)
    for h in range(4):
        np.testing.assert_allclose(out[h], v[:, h // 2].mean(axis=0), rtol=1e-13)


def test_attend_dominant_key():
    # A key aligned with the query at large scale takes all the weight.
    q = np.zeros((1, 8))
    q[0, 0] = 1.0
    k = np.zeros((5, 1, 8))
    k[3, 0, 0] = 1e4
    v = np.arange(40.0).reshape(5, 1, 8)
    np.testing.assert_allclose(attend_ref(q, k, v, 1, 1)[0], v[3, 0], rtol=1e-15)


@pytest.mark.parametrize("nq,nkv", [(4, 2), (6, 6), (6, 1), (14, 2)])
def test_attend_matches_sdpa(nq, nkv):
    rng = np.random.default_rng(13)
    m, hd = 11, 8
    q, k, v = rng.normal(size=(nq, hd)), rng.normal(size=(m, nkv, hd)), rng.normal(size=(m, nkv, hd))
    ref = F.scaled_dot_product_attention(torch.tensor(q)[None, :, None, :],
                                         torch.tensor(k).transpose(0, 1)[None],
                                         torch.tensor(v).transpose(0, 1)[None], enable_gqa=True)
    np.testing.assert_allclose(attend_ref(q, k, v, nq, nkv), ref[0, :, 0, :].numpy(), rtol=1e-12, atol=1e-14)


def test_gqa_head_map_ratio_table():
    g = _golden("gqa_ratio_table.json")
    for m in g["models"]:
        nq, nkv = m["q_heads"], m["kv_heads"]
        assert nq // nkv == m["ratio"]
        # sipllm "h / gqa_group()" and Pantheon "h * n_kv_head / n_head" agree.
        assert [kv_head_of(h, nq, nkv) for h in range(nq)] == [h // m["ratio"] for h in range(nq)]
    assert [kv_head_of(h, 8, 8) for h in range(8)] == list(range(8))       # MHA
    assert [kv_head_of(h, 8, 1) for h in range(8)] == [0] * 8              # MQA


def test_kv_row_size_worked_example():
    g = _golden("kv_row_size.json")
    assert g["n_kv_heads"] * g["head_dim"] == g["kv_size"]
    # One cached position of one layer holds n_kv_heads * head_dim keys.
    cfg = toy_cfg(n_layers=1, hidden=16, n_heads=g["n_kv_heads"], n_kv_heads=g["n_kv_heads"],
                  head_dim=g["head_dim"], ffn=8, vocab=4)
    s = Session(cfg, random_weights(cfg, seed=30))
    s.prefill([1], 0)
    assert s.keys[0][0].size == g["kv_size"] and s.values[0][0].size == g["kv_size"]


@pytest.mark.parametrize("W", [1, 3, 8])
def test_window_readable_length(W):
    # Pantheon "Sliding Window": readable length min(pos + 1, max_seq).
    for pos in range(30):
        assert pos - window_start(pos, W) + 1 == min(pos + 1, W)
        assert window_start(pos, 0) == 0


# ---------------------------------------------------------------- MoE routing
def test_topk_tie_goes_to_lower_id():
    ids, w, _ = route_topk(np.array([0.5, 1.0, 1.0, 1.0, 0.2]), 2)
    assert ids == [1, 2]
    np.testing.assert_allclose(w, [0.5, 0.5], rtol=1e-15)
    ids, _, _ = route_topk(np.zeros(8), 3)
    assert ids == [0, 1, 2]


def test_topk_matches_stable_sort_and_weights_sum_to_one():
    rng = np.random.default_rng(14)
    for _ in range(200):
        r = np.round(rng.normal(size=8), 1)          # rounding makes ties common
        k = int(rng.integers(1, 9))
        ids, w, p = route_topk(r, k)
        assert ids == list(np.argsort(-r, kind="stable")[:k])
        assert abs(w.sum() - 1.0) <= 2.3e-16 * k
        np.testing.assert_allclose(p, scipy.special.softmax(r), rtol=1e-14)


def test_moe_with_all_experts_is_the_dense_softmax_mixture():
    rng = np.random.default_rng(15)
    h, f, E = 12, 7, 4
    router = rng.normal(size=(E, h))
    ex = [(rng.normal(size=(f, h)), rng.normal(size=(f, h)), rng.normal(size=(h, f))) for _ in range(E)]
    n = rng.normal(size=h)
    out, ids, wts, logits = moe_ffn(n, router, lambda e: ex[e], E)
    p = scipy.special.softmax(router @ n)
    ref = sum(p[e] * (ex[e][2] @ (F.silu(torch.tensor(ex[e][0] @ n)).numpy() * (ex[e][1] @ n))) for e in range(E))
    np.testing.assert_allclose(out, ref, rtol=1e-12)


def test_moe_equal_router_rows_pick_lowest_ids():
    rng = np.random.default_rng(16)
    router = np.tile(rng.normal(size=(1, 10)), (8, 1))
    ex = [(np.eye(10), np.eye(10), np.eye(10))] * 8
    _, ids, wts, _ = moe_ffn(rng.normal(size=10), router, lambda e: ex[e], 2)
    assert ids == [0, 1]
    np.testing.assert_allclose(wts, [0.5, 0.5], rtol=1e-15)


# ---------------------------------------------------------------- whole forward
CASES = {
    "dense": dict(),
    "bias_theta1e6": dict(qkv_bias=True, rope_theta=1e6, rms_eps=1e-6),
    "window3": dict(sliding_window=3),
    "moe": dict(n_experts=4, n_experts_used=2),
    "mha": dict(n_kv_heads=4),
    "mqa": dict(n_kv_heads=1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_whole_forward_matches_torch_library(case):
    cfg = toy_cfg(**CASES[case])
    w = random_weights(cfg, seed=20)
    toks = list(np.random.default_rng(21).integers(0, cfg.vocab, 9))
    ref = torch_library_forward(cfg, w, toks)
    s = Session(cfg, w)
    got = s.prefill(toks, 0, all_logits=True)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("case", sorted(CASES))
def test_single_pass_prefill_equals_per_token_bit_exact(case):
    # sipllm "Single-pass prefill": byte-for-byte identical to per-token forward.
    cfg = toy_cfg(**CASES[case])
    w = random_weights(cfg, seed=22)
    toks = list(np.random.default_rng(23).integers(0, cfg.vocab, 10))
    a = Session(cfg, w)
    all_rows = a.prefill(toks, 0, all_logits=True)
    b = Session(cfg, w)
    per_tok = np.stack([b.forward(t, p) for p, t in enumerate(toks)])
    assert np.array_equal(all_rows, per_tok)
    for l in range(cfg.n_layers):
        assert all(np.array_equal(x, y) for x, y in zip(a.keys[l], b.keys[l]))
        assert all(np.array_equal(x, y) for x, y in zip(a.values[l], b.values[l]))


@pytest.mark.parametrize("case", sorted(CASES))
def test_batched_order_matches_rowwise(case):
    cfg = toy_cfg(**CASES[case])
    w = random_weights(cfg, seed=24)
    toks = list(np.random.default_rng(25).integers(0, cfg.vocab, 12))
    a = Session(cfg, w)
    rowwise = a.prefill(toks, 0, all_logits=True)
    b = Session(cfg, w)
    batched = b.prefill_batched(toks, 0, logits_rows=range(12))
    np.testing.assert_allclose(batched, rowwise, rtol=1e-12, atol=1e-12)


def test_append_prefill_and_rewind():
    cfg = toy_cfg(sliding_window=4)
    w = random_weights(cfg, seed=26)
    toks = list(np.random.default_rng(27).integers(0, cfg.vocab, 14))
    full = Session(cfg, w).prefill(toks, 0)
    s = Session(cfg, w)
    s.prefill(toks[:5], 0)
    s.prefill(toks[5:9], 5)
    assert np.array_equal(s.prefill(toks[9:], 9), full)
    # A rewind to 6 then a different continuation equals a fresh run of that sequence.
    other = toks[:6] + [1, 2, 3]
    assert np.array_equal(s.prefill([1, 2, 3], 6), Session(cfg, w).prefill(other, 0))
    with pytest.raises(ValueError):
        s.prefill([1], 99)


def test_zero_layer_weights_reduce_to_head_of_embedding():
    cfg = toy_cfg()
    w = random_weights(cfg, seed=28, zero_layers=True)
    toks = [3, 17, 42]
    got = Session(cfg, w).prefill(toks, 0, all_logits=True)
    E = w.embed_rows(toks)
    ms = np.mean(E * E, axis=1, keepdims=True)
    ref = (E / np.sqrt(ms + cfg.rms_eps) * w.out_norm()) @ w.lm_head().T
    np.testing.assert_allclose(got, ref, rtol=1e-13)


def test_first_position_attention_is_the_value_path():
    # At position 0 the softmax has one key, so the attention half adds
    # Wo (Wv n + bv) whatever q, k and RoPE are.
    cfg = toy_cfg(n_layers=1, qkv_bias=True)
    w = random_weights(cfg, seed=29)
    lw = w.layer(0)
    x = w.embed_rows([7])[0]
    s = Session(cfg, w)
    y = s._attention_row(0, lw, x, 0)
    n = x / np.sqrt(np.mean(x * x) + cfg.rms_eps) * lw["attn_norm"]
    v = np.array([sum(lw["wv"][r, c] * n[c] for c in range(cfg.hidden)) for r in range(lw["wv"].shape[0])]) + lw["bv"]
    o = np.concatenate([v.reshape(cfg.n_kv_heads, cfg.head_dim)[h * cfg.n_kv_heads // cfg.n_heads]
                        for h in range(cfg.n_heads)])
    np.testing.assert_allclose(y, x + lw["wo"] @ o, rtol=1e-12)
