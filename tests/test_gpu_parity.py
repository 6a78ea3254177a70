"""GPU parity: libdec.so (through the C ABI) against the float64 oracle on the
same seeded inputs.  Logits within the stated tolerances, greedy tokens
consistent with the oracle, KV slot positions exact, expert ids exact."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import (check_greedy_tokens, compare_logits, gpu_greedy, oracle_teacher_forced,
                               ring_positions, tolerances)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def _run_case(dec_mod, w, P, D, kv="f32", max_tokens=0, device_argmax=False, trace=False):
    d = dec_mod.Decoder(w, kv_dtype=kv, max_tokens=max_tokens)
    prompt = synthetic.prompt_tokens(w, P, seed=0)
    ids_t = logit_t = None
    if trace:
        cap = P + D
        ids_t = torch.full((w["n_layers"] * cap * w["n_experts_used"],), -1, dtype=torch.int32, device="cuda")
        logit_t = torch.zeros((w["n_layers"] * cap * w["n_experts"],), dtype=torch.float32, device="cuda")
        d.set_trace(ids_t, logit_t, cap)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=device_argmax)
    ref, sess = oracle_teacher_forced(w, prompt, taus, D, trace=trace)
    return d, prompt, rows, taus, ref, sess, ids_t, logit_t


def test_toy_full_workload(dec_mod):
    w = synthetic.workload("toy")
    d, prompt, rows, taus, ref, sess, *_ = _run_case(dec_mod, w, w["prompt"], w["decode"])
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)
    # The toy is fp32 throughout: the oracle's own greedy stream is the same.
    assert [int(np.argmax(r)) for r in ref] == taus


def test_toy_device_argmax_greedy(dec_mod):
    w = synthetic.workload("toy")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 16, 16, device_argmax=True)
    compare_logits(rows, ref, *tolerances(w))


def test_toy_bf16_kv(dec_mod):
    w = synthetic.workload("toy")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 16, 16, kv="bf16")
    compare_logits(rows, ref, *tolerances(w, "bf16"))


def test_toy_window_wraps_in_prefill_and_decode(dec_mod):
    # Window 8 = max_seq 8: the prompt of 12 already wraps the ring, decode wraps again.
    w = synthetic.workload("toy", sliding_window=8, max_seq=8)
    d, prompt, rows, taus, ref, sess, *_ = _run_case(dec_mod, w, 12, 10)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)
    length = 12 + 10
    assert d.length == length
    slots = ring_positions(length, w["max_seq"], w["sliding_window"])
    for l in range(w["n_layers"]):
        kc, vc = d.kv_layer(l)
        for s_, p in enumerate(slots):
            np.testing.assert_allclose(kc[s_].cpu().numpy(), sess.keys[l][p], atol=1e-5, rtol=1e-5)
            np.testing.assert_allclose(vc[s_].cpu().numpy(), sess.values[l][p], atol=1e-5, rtol=1e-5)


def test_toy_kv_slots_no_window(dec_mod):
    w = synthetic.workload("toy")
    d, prompt, rows, taus, ref, sess, *_ = _run_case(dec_mod, w, 16, 8)
    for l in range(w["n_layers"]):
        kc, vc = d.kv_layer(l)
        for p in range(24):
            np.testing.assert_allclose(kc[p].cpu().numpy(), sess.keys[l][p], atol=1e-5, rtol=1e-5)
            np.testing.assert_allclose(vc[p].cpu().numpy(), sess.values[l][p], atol=1e-5, rtol=1e-5)


def test_toy_moe_expert_ids_exact(dec_mod):
    w = synthetic.workload("toy", n_experts=4, n_experts_used=2)
    d, prompt, rows, taus, ref, sess, ids_t, logit_t = _run_case(dec_mod, w, 16, 8, trace=True)
    compare_logits(rows, ref, *tolerances(w))
    cap, k, E = 24, 2, 4
    ids = ids_t.view(w["n_layers"], cap, k).cpu().numpy()
    lg = logit_t.view(w["n_layers"], cap, E).cpu().numpy()
    for l in range(w["n_layers"]):
        for p in range(cap):
            np.testing.assert_allclose(lg[l, p], sess.trace.router_logits[(l, p)], atol=1e-5)
            assert list(ids[l, p]) == sess.trace.expert_ids[(l, p)], (l, p)


def test_toy_llama3_rope(dec_mod):
    w = synthetic.workload("toy", rope_llama3=dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0,
                                                   orig_ctx=64))
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 16, 8)
    compare_logits(rows, ref, *tolerances(w))


@pytest.mark.parametrize("kw", [dict(rope_half=True), dict(rope_dim=8), dict(rope_half=True, rope_dim=8)])
def test_toy_rope_pairing_and_partial_rotary(dec_mod, kw):
    # kHalf pairing (i, i + d/2) and partial rotary (first rope_dim dims only),
    # fp32 throughout: the same bound as the default adjacent-pair toy.
    w = synthetic.workload("toy", **kw)
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 12, 8)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)


@pytest.mark.parametrize("mode", ["off", "grid"])
def test_smollm2_shape_rope_half_partial(dec_mod, mode):
    # A SmolLM2-shaped bf16 model with kHalf pairing over the first 32 of 64 dims,
    # on the per-layer and the persistent decode schedules.
    w = synthetic.workload("smollm2-135m", n_layers=4, rope_half=True, rope_dim=32)
    d = dec_mod.Decoder(w)
    d.set_fused(mode)
    prompt = synthetic.prompt_tokens(w, 40, seed=0)
    rows, taus = gpu_greedy(d, prompt, 6)
    ref, _ = oracle_teacher_forced(w, prompt, taus, 6)
    compare_logits(rows, ref, *tolerances(w))


def test_toy_chunked_prefill(dec_mod):
    # max_tokens 5: a 16-token prompt runs as chunks 5+5+5+1.
    w = synthetic.workload("toy")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 16, 4, max_tokens=5)
    compare_logits(rows, ref, *tolerances(w))


def test_argument_errors_change_nothing(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w)
    logits = torch.empty(w["vocab"], device="cuda")
    d.prefill(synthetic.prompt_tokens(w, 10), 0, logits)
    cases = [
        (lambda: d.prefill([], 10, logits), dec_mod.DEC_EINVAL),
        (lambda: d.prefill([5, 256], 10, logits), dec_mod.DEC_EINVAL),
        (lambda: d.prefill([-1], 10, logits), dec_mod.DEC_EINVAL),
        (lambda: d.prefill([1], 11, logits), dec_mod.DEC_EINVAL),
        (lambda: d.decode(3, 12, logits), dec_mod.DEC_EINVAL),
        (lambda: d.prefill([1] * 23, 10, logits), dec_mod.DEC_ERANGE),
        (lambda: d.decode(300, 10, logits), dec_mod.DEC_EINVAL),
    ]
    for fn, status in cases:
        with pytest.raises(dec_mod.DecError) as ei:
            fn()
        assert ei.value.status == status
        assert d.length == 10
    d.check()


def test_device_token_out_of_range_reported(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w)
    logits = torch.empty(w["vocab"], device="cuda")
    d.prefill([1, 2, 3], 0, logits)
    bad = torch.tensor([999], dtype=torch.int32, device="cuda")
    d.decode_dev(bad, 3, logits)
    with pytest.raises(dec_mod.DecError) as ei:
        d.check()
    assert ei.value.status == dec_mod.DEC_EINVAL
    d.check()   # the error word was cleared


def test_rewind_then_append_matches_fresh(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w)
    a = torch.empty(w["vocab"], device="cuda")
    toks = synthetic.prompt_tokens(w, 14, seed=3)
    d.prefill(toks, 0, a)
    d.prefill([7, 8, 9], 6, a)
    d.synchronize()
    f = dec_mod.Decoder(w)
    b = torch.empty(w["vocab"], device="cuda")
    f.prefill(list(toks[:6]) + [7, 8, 9], 0, b)
    f.synchronize()
    assert d.length == 9
    np.testing.assert_allclose(a.cpu().numpy(), b.cpu().numpy(), atol=1e-6)


def test_runs_are_deterministic(dec_mod):
    w = synthetic.workload("smollm2-135m")
    outs = []
    for _ in range(2):
        d = dec_mod.Decoder(w)
        rows, taus = gpu_greedy(d, synthetic.prompt_tokens(w, 64), 8)
        outs.append((rows, taus))
        d.close()
    assert np.array_equal(outs[0][0], outs[1][0]) and outs[0][1] == outs[1][1]


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_smollm2_full_workload(dec_mod, kv):
    w = synthetic.workload("smollm2-135m")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, w["prompt"], w["decode"], kv=kv, device_argmax=True)
    tol_abs, tol_rel = tolerances(w, kv)
    compare_logits(rows, ref, tol_abs, tol_rel)
    check_greedy_tokens(ref, taus, tol_abs)


def test_qwen25_reduced(dec_mod):
    w = synthetic.workload("qwen2.5-0.5b")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 192, 16)
    compare_logits(rows, ref, *tolerances(w))
    check_greedy_tokens(ref, taus, tolerances(w)[0])


def test_mistral_reduced(dec_mod):
    w = synthetic.workload("mistral-7b")
    _, _, rows, taus, ref, *_ = _run_case(dec_mod, w, 40, 6)
    compare_logits(rows, ref, *tolerances(w))


def test_mistral_shape_window_wrap(dec_mod):
    # Mistral-shaped layers with a 24-slot window so that both prefill and decode wrap.
    w = synthetic.workload("mistral-7b", n_layers=4, sliding_window=24, max_seq=24)
    d, prompt, rows, taus, ref, sess, *_ = _run_case(dec_mod, w, 30, 10)
    compare_logits(rows, ref, *tolerances(w))
    slots = ring_positions(40, 24, 24)
    kc, vc = d.kv_layer(3)
    for s_, p in enumerate(slots):
        np.testing.assert_allclose(kc[s_].cpu().numpy(), sess.keys[3][p], atol=2e-3, rtol=2e-3)


def test_mixtral_reduced_expert_ids(dec_mod):
    # All 32 Mixtral-shaped layers at a short prompt.  The GPU's ids are the
    # definition's on its own router logits, bit for bit, and the oracle's.
    from oracle import route_topk
    w = synthetic.workload("mixtral-8x7b")
    P, D = 12, 3
    d, prompt, rows, taus, ref, sess, ids_t, logit_t = _run_case(dec_mod, w, P, D, trace=True)
    compare_logits(rows, ref, *tolerances(w))
    cap, k, E = P + D, 2, 8
    ids = ids_t.view(w["n_layers"], cap, k).cpu().numpy()
    lg = logit_t.view(w["n_layers"], cap, E).cpu().numpy()
    for l in range(w["n_layers"]):
        for p in range(cap):
            assert list(ids[l, p]) == route_topk(lg[l, p].astype(np.float64), k)[0], (l, p)
            assert list(ids[l, p]) == sess.trace.expert_ids[(l, p)], (l, p)


def test_toy_append_prefill_after_wrap(dec_mod):
    # Window 8: prefill 12 (wraps), decode 3, then append chunks of 5 and of 10 (> max_seq)
    # at the current length; each append's last logits match the oracle on the whole sequence.
    w = synthetic.workload("toy", sliding_window=8, max_seq=8)
    toks = list(synthetic.prompt_tokens(w, 30, seed=5))
    d = dec_mod.Decoder(w)
    lg = torch.empty(w["vocab"], device="cuda")
    d.prefill(toks[:12], 0, lg)
    for i in range(12, 15):
        d.decode(toks[i], i, lg)
    d.prefill(toks[15:20], 15, lg)
    d.synchronize()
    a = lg.cpu().numpy().copy()
    d.prefill(toks[20:30], 20, lg)
    d.synchronize()
    b = lg.cpu().numpy().copy()
    from tests.gpu_helpers import oracle_session
    s = oracle_session(w)
    ref = s.prefill_batched(toks, 0, logits_rows=[19, 29])
    tol = tolerances(w)[0]
    compare_logits(np.stack([a, b]), ref, tol, tol)
    slots = ring_positions(30, 8, 8)
    kc, _ = d.kv_layer(1)
    for s_, p in enumerate(slots):
        np.testing.assert_allclose(kc[s_].cpu().numpy(), s.keys[1][p], atol=1e-5, rtol=1e-5)


def _prefill_vs_decode_loop(dec_mod, w, P, extra):
    """Property at any size (sipllm: single-pass prefill == per-token forward): the prefill
    path (GEMMs + tiled attention) and the decode path (GEMVs + split-K attention) agree."""
    toks = synthetic.prompt_tokens(w, P + extra, seed=7)
    a = dec_mod.Decoder(w)
    la = torch.empty(w["vocab"], device="cuda")
    a.prefill(toks, 0, la)                      # one call over P + extra positions
    b = dec_mod.Decoder(w, weights=a.weights)
    lb = torch.empty(w["vocab"], device="cuda")
    b.prefill(toks[:P], 0, lb)
    for i in range(P, P + extra):               # the tail through the decode kernels
        b.decode(int(toks[i]), i, lb)
    a.synchronize()
    b.synchronize()
    x, y = la.cpu().numpy(), lb.cpu().numpy()
    compare_logits(x[None], y[None].astype(np.float64), *tolerances(w))
    return a, b


def test_smollm2_prefill_equals_decode_path_full_size(dec_mod):
    w = synthetic.workload("smollm2-135m")
    _prefill_vs_decode_loop(dec_mod, w, w["prompt"], 32)


@pytest.mark.slow
def test_mistral_full_prefill_then_wrapping_decode(dec_mod):
    # Full Mistral shape: 4096-token prefill fills the 4096-slot window; 48 more
    # positions wrap the ring.  Single-call prefill of all 4144 vs prefill 4096 + 48 decodes.
    w = synthetic.workload("mistral-7b")
    a, b = _prefill_vs_decode_loop(dec_mod, w, 4096, 48)
    assert a.length == b.length == 4144


@pytest.mark.parametrize("name,kw", [("toy", {}), ("toy", dict(n_experts=4, n_experts_used=2)),
                                     ("toy", dict(sliding_window=8, max_seq=8)), ("smollm2-135m", {}),
                                     ("mixtral-8x7b", dict(n_layers=2))])
def test_fused_step_matches_per_layer_kernels(dec_mod, name, kw):
    # The per-layer kernels and the persistent one-kernel decode step (over
    # every SM, or on one thread-block cluster) are schedules of the same
    # arithmetic: same greedy stream, logits to rounding.
    w = synthetic.workload(name, **kw)
    P = 12 if name == "toy" else 40
    prompt = synthetic.prompt_tokens(w, P, seed=9)
    runs = []
    weights = None
    for mode in ("off", "grid", "cluster"):
        d = dec_mod.Decoder(w, weights=weights)
        weights = d.weights
        if not d.fused_available(mode):
            assert mode == "cluster", f"schedule {mode} unavailable"
            d.close()
            continue
        d.set_fused(mode)
        runs.append((mode, gpu_greedy(d, prompt, 10)))
        d.close()
    (_, (ra, ta)) = runs[0]
    for mode, (rb, tb) in runs[1:]:
        assert ta == tb, mode
        np.testing.assert_allclose(ra, rb, atol=2e-4 if w["dtype"] == "f32" else 2e-3, rtol=1e-4, err_msg=mode)
