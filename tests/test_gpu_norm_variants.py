"""GPU parity of QK-norm and sandwich norms (rml "The decoder", One forward pass
steps 4 and 6) against the float64 oracle: prefill (tensor-core attention and
SIMT paths, chunked, wrapping), single-sequence decode (which runs the row
kernels for these models), batched decode, the kHalf permutation of the norm
weights, an int8 cache and a MoE FFN."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import (check_greedy_tokens, compare_logits, gpu_greedy, oracle_teacher_forced,
                               tolerances)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def _run(dec_mod, w, P, D, kv="f32", max_tokens=0, seed=0):
    d = dec_mod.Decoder(w, kv_dtype=kv, max_tokens=max_tokens)
    prompt = synthetic.prompt_tokens(w, P, seed=seed)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
    ref, _ = oracle_teacher_forced(dict(w, kv_int8=(kv == "i8")), prompt, taus, D)
    return rows, taus, ref


@pytest.mark.parametrize("kw", [dict(qk_norm="head"), dict(qk_norm="row"), dict(sandwich_norms=True),
                                dict(qk_norm="head", sandwich_norms=True, n_experts=4, n_experts_used=2),
                                dict(qk_norm="row", sandwich_norms=True, rope_half=True, rope_dim=8)])
def test_toy_norm_variants(dec_mod, kw):
    w = synthetic.workload("toy", **kw)
    rows, taus, ref = _run(dec_mod, w, 16, 12)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)
    assert [int(np.argmax(r)) for r in ref] == taus


def test_toy_qk_norm_window_chunked_prefill(dec_mod):
    w = synthetic.workload("toy", qk_norm="head", sandwich_norms=True, sliding_window=8, max_seq=8)
    rows, taus, ref = _run(dec_mod, w, 13, 9, max_tokens=5, seed=2)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)


def test_toy_qk_norm_int8_cache(dec_mod):
    w = synthetic.workload("toy", qk_norm="head")
    rows, taus, ref = _run(dec_mod, w, 16, 8, kv="i8", seed=3)
    compare_logits(rows, ref, *tolerances(w, "bf16"))


@pytest.mark.parametrize("kw", [dict(qk_norm="head", sandwich_norms=True), dict(qk_norm="row")])
def test_mistral_shape_norm_variants(dec_mod, kw):
    # bf16 weights: tensor-core GEMMs, and q reaches the tensor-core attention as planes.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=24, max_seq=24, **kw)
    rows, taus, ref = _run(dec_mod, w, 30, 6, seed=4)
    compare_logits(rows, ref, *tolerances(w))
    check_greedy_tokens(ref, taus, tolerances(w)[0])


def test_smollm2_shape_norm_variants_batched(dec_mod):
    w = synthetic.workload("smollm2-135m", n_layers=2, qk_norm="head", sandwich_norms=True, rope_half=True)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=95 + i)) for i, n in enumerate([11, 40, 2])]
    d = dec_mod.Decoder(w, n_seqs=3)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    rows = [[] for _ in prompts]
    taus = [[] for _ in prompts]
    for s_, p in enumerate(prompts):
        d.prefill(p, 0, lg, seq=s_)
        d.synchronize()
        rows[s_].append(lg.cpu().numpy().copy())
        taus[s_].append(int(np.argmax(rows[s_][-1])))
    tok = torch.tensor([t[0] for t in taus], dtype=torch.int32, device="cuda")
    out = torch.empty((3, V), device="cuda")
    for _ in range(5):
        d.decode_batch([2, 0, 1], [d.length_of(2), d.length_of(0), d.length_of(1)], tok[[2, 0, 1]].contiguous(),
                       out)
        d.synchronize()
        h = out.cpu().numpy()
        for i, s_ in enumerate([2, 0, 1]):
            rows[s_].append(h[i].copy())
            taus[s_].append(int(np.argmax(h[i])))
        tok = torch.tensor([t[-1] for t in taus], dtype=torch.int32, device="cuda")
    d.check()
    for s_, p in enumerate(prompts):
        ref, _ = oracle_teacher_forced(w, p, taus[s_], 5)
        compare_logits(np.stack(rows[s_]), ref, *tolerances(w))


@pytest.mark.parametrize("kw", [dict(rope_theta_local=50.0, rope_global_every=2),
                                dict(rope_theta_local=50.0, rope_global_every=0),
                                dict(rope_theta_local=500.0, rope_global_every=2, qk_norm="head",
                                     sandwich_norms=True)])
def test_toy_per_layer_rope_base(dec_mod, kw):
    w = synthetic.workload("toy", **kw)
    rows, taus, ref = _run(dec_mod, w, 16, 10, seed=5)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)


def test_gemma_like_combination_chunked_window(dec_mod):
    # Local base on layer 0, global on layer 1, QK-norm, sandwich norms, a window, chunked prefill.
    w = synthetic.workload("toy", rope_theta_local=20.0, rope_global_every=2, qk_norm="head",
                           sandwich_norms=True, sliding_window=8, max_seq=8)
    rows, taus, ref = _run(dec_mod, w, 13, 9, max_tokens=5, seed=6)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)


def test_qwen_shape_per_layer_base_batched(dec_mod):
    w = synthetic.workload("qwen2.5-0.5b", n_layers=3, rope_theta_local=10000.0, rope_global_every=3)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=97 + i)) for i, n in enumerate([6, 21])]
    d = dec_mod.Decoder(w, n_seqs=2)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    rows = [[] for _ in prompts]
    taus = [[] for _ in prompts]
    for s_, p in enumerate(prompts):
        d.prefill(p, 0, lg, seq=s_)
        d.synchronize()
        rows[s_].append(lg.cpu().numpy().copy())
        taus[s_].append(int(np.argmax(rows[s_][-1])))
    tok = torch.tensor([t[0] for t in taus], dtype=torch.int32, device="cuda")
    out = torch.empty((2, V), device="cuda")
    for _ in range(4):
        d.decode_batch([0, 1], [d.length_of(0), d.length_of(1)], tok, out, tok)
        d.synchronize()
        h = out.cpu().numpy()
        for s_ in range(2):
            rows[s_].append(h[s_].copy())
            taus[s_].append(int(np.argmax(h[s_])))
    d.check()
    for s_, p in enumerate(prompts):
        ref, _ = oracle_teacher_forced(w, p, taus[s_], 4)
        compare_logits(np.stack(rows[s_]), ref, *tolerances(w))


# Per-head QK-norm on the persistent decode step (bf16 weights, f32 cache, head_dim
# 64 / 128): the QKV phase leaves q and the new k unrotated, and the attention task
# normalises each head over head_dim, rotates it and stores the key.


def _persistent_qkn(dec_mod, w, P, D, seed):
    d = dec_mod.Decoder(w)
    d.set_fused("grid")
    assert d.fused_mode() == "grid"
    prompt = synthetic.prompt_tokens(w, P, seed=seed)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
    ref, _ = oracle_teacher_forced(w, prompt, taus, D)
    compare_logits(rows, ref, *tolerances(w))
    check_greedy_tokens(ref, taus, tolerances(w)[0])
    d.close()


def test_mistral_shape_qk_norm_persistent_window_wraps(dec_mod):
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=24, max_seq=24, qk_norm="head")
    _persistent_qkn(dec_mod, w, 30, 10, seed=41)


def test_qwen_shape_qk_norm_persistent_khalf(dec_mod):
    # head_dim 64, seven query heads per kv head, q/k biases, kHalf-permuted norm weights.
    w = synthetic.workload("qwen2.5-0.5b", n_layers=2, max_seq=96, qk_norm="head", rope_half=True)
    _persistent_qkn(dec_mod, w, 60, 8, seed=42)


def test_qk_norm_persistent_step_agrees_with_row_kernels(dec_mod):
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=0, max_seq=96, qk_norm="head")
    prompt = synthetic.prompt_tokens(w, 70, seed=43)
    out = {}
    weights = None
    for mode in ("grid", "off"):
        d = dec_mod.Decoder(w, weights=weights)
        weights = d.weights
        d.set_fused(mode)
        out[mode] = gpu_greedy(d, prompt, 8)
        d.close()
    assert out["grid"][1] == out["off"][1]
    np.testing.assert_allclose(out["grid"][0], out["off"][0], atol=2e-3, rtol=1e-4)


def test_qwen_shape_per_layer_base_persistent(dec_mod):
    # Per-layer RoPE base on the persistent step: the step builds both (cos, sin) tables
    # and each layer's QKV phase turns q and k with its own.
    w = synthetic.workload("qwen2.5-0.5b", n_layers=3, max_seq=96, rope_theta_local=10000.0,
                           rope_global_every=3)
    _persistent_qkn(dec_mod, w, 50, 8, seed=44)


def test_mistral_shape_qk_norm_per_layer_base_persistent(dec_mod):
    # QK-norm and a per-layer base together: the attention task rotates with the layer's table.
    w = synthetic.workload("mistral-7b", n_layers=2, max_seq=64, qk_norm="head", rope_theta_local=500.0,
                           rope_global_every=2)
    _persistent_qkn(dec_mod, w, 40, 8, seed=45)


def test_qk_norm_persistent_grid_and_cluster_agree(dec_mod):
    w = synthetic.workload("qwen2.5-0.5b", n_layers=2, max_seq=96, qk_norm="head", rope_theta_local=10000.0,
                           rope_global_every=2)
    prompt = synthetic.prompt_tokens(w, 40, seed=46)
    out = {}
    weights = None
    for mode in ("grid", "cluster"):
        d = dec_mod.Decoder(w, weights=weights)
        weights = d.weights
        if not d.fused_available(mode):
            assert mode == "cluster"
            d.close()
            continue
        d.set_fused(mode)
        out[mode] = gpu_greedy(d, prompt, 6)
        d.close()
    if "cluster" in out:
        assert out["grid"][1] == out["cluster"][1]
        np.testing.assert_allclose(out["grid"][0], out["cluster"][0], atol=2e-3, rtol=1e-4)
