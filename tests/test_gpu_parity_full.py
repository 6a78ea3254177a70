"""GPU parity against the float64 oracle at the full prompt and decode lengths of the
large workloads, with fewer layers so the oracle finishes in seconds.

These take the paths the kernels take at full size: many 128-row tensor-core GEMM
tiles and grouped expert GEMMs with full tiles, the tensor-core prefill attention
over thousands of keys at head_dim 64 and 128, the persistent decode step's attention
over a 4096-slot ring that wraps (Pantheon "Llama Forward Pass", Sliding Window), and
the per-layer decode kernels.  Each case decodes greedily on the persistent schedule;
the oracle then runs prompt + those tokens in one single-pass prefill (exact by
sipllm "Transformer forward pass", Single-pass prefill), and the per-layer schedule is
fed the same tokens.  Logits: max|d| <= 2e-2 and relative RMS <= 1e-2 (bf16 weights,
fp32 accumulation)."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from oracle import route_topk
from tests.gpu_helpers import (check_greedy_tokens, compare_logits, gpu_greedy, gpu_teacher_forced,
                               oracle_teacher_forced, ring_positions, tolerances)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def _both_schedules(dec_mod, w, P, D, trace=False):
    """Greedy on the persistent step, then the per-layer kernels on the same tokens; the oracle
    on prompt + tokens.  Returns (oracle rows, oracle session, {mode: (handle, rows, ids, logits)})."""
    prompt = synthetic.prompt_tokens(w, P, seed=0)
    out = {}
    weights = None
    taus = None
    for mode in ("grid", "off"):
        d = dec_mod.Decoder(w, weights=weights)
        weights = d.weights
        d.set_fused(mode)
        ids_t = logit_t = None
        if trace:
            cap = P + D
            ids_t = torch.full((w["n_layers"] * cap * w["n_experts_used"],), -1, dtype=torch.int32,
                               device="cuda")
            logit_t = torch.zeros((w["n_layers"] * cap * w["n_experts"],), dtype=torch.float32, device="cuda")
            d.set_trace(ids_t, logit_t, cap)
        if taus is None:
            rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
        else:
            rows = gpu_teacher_forced(d, prompt, taus, D)
        out[mode] = (d, rows, ids_t, logit_t)
    ref, sess = oracle_teacher_forced(w, prompt, taus, D, trace=trace)
    check_greedy_tokens(ref, taus, tolerances(w)[0])
    for mode, (_, rows, _, _) in out.items():
        compare_logits(rows, ref, *tolerances(w))
    return ref, sess, out


def test_mistral_full_length_window_wraps(dec_mod):
    # 4096-token prompt fills the 4096-slot window; 48 decode steps wrap the ring.
    w = synthetic.workload("mistral-7b", n_layers=2)
    P, D = 4096, 48
    ref, sess, out = _both_schedules(dec_mod, w, P, D)
    slots = ring_positions(P + D, w["max_seq"], w["sliding_window"])
    assert slots.min() >= 0 and slots.max() == P + D - 1
    for mode, (d, *_rest) in out.items():
        assert d.length == P + D
        for l in range(w["n_layers"]):
            kc, vc = d.kv_layer(l)
            kr = np.stack([sess.keys[l][p] for p in slots])
            vr = np.stack([sess.values[l][p] for p in slots])
            np.testing.assert_allclose(kc.cpu().numpy(), kr, atol=2e-3, rtol=2e-3, err_msg=f"{mode} K layer {l}")
            np.testing.assert_allclose(vc.cpu().numpy(), vr, atol=2e-3, rtol=2e-3, err_msg=f"{mode} V layer {l}")


def test_qwen25_full_length(dec_mod):
    w = synthetic.workload("qwen2.5-0.5b", n_layers=4)
    _both_schedules(dec_mod, w, 2048, 32)


def test_mixtral_full_length_expert_ids(dec_mod):
    w = synthetic.workload("mixtral-8x7b", n_layers=2)
    P, D = 1024, 16
    ref, sess, out = _both_schedules(dec_mod, w, P, D, trace=True)
    cap, k, E = P + D, w["n_experts_used"], w["n_experts"]
    for mode, (_, _, ids_t, logit_t) in out.items():
        ids = ids_t.view(w["n_layers"], cap, k).cpu().numpy()
        lg = logit_t.view(w["n_layers"], cap, E).cpu().numpy()
        for l in range(w["n_layers"]):
            for p in range(cap):
                # The GPU's choice on its own router logits is the definition's, bit for bit
                # (prefill rows, and the decode kernels of this schedule).
                own, _, _ = route_topk(lg[l, p].astype(np.float64), k)
                assert list(ids[l, p]) == own, (mode, l, p)
                # And the same experts as the oracle's float64 forward pass.
                assert list(ids[l, p]) == sess.trace.expert_ids[(l, p)], (mode, l, p)
            err = max(np.abs(lg[l, p] - sess.trace.router_logits[(l, p)]).max() for p in range(cap))
            assert err < 2e-3, (mode, l, err)
