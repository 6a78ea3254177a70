"""GPU parity of 8-bit projection weights (weight_quant = 1) against the oracle's
weight_int8 mode.

Pantheon "Llama Forward Pass", weight modes: the projections (and an untied output
matrix) stay quantised and are expanded a block at a time; each weight row is held
in groups of 32 input columns by the int8 rule rml "The decoder" gives for the
cache.  The library quantises at dec_create; the quantiser alone is compared bit for
bit with the oracle's on the same values, then whole models (greedy decode, the
oracle teacher-forced on the GPU's tokens) within the tolerances of their weight
type: 1e-4 for the fp32 toy, 2e-2 / 1e-2 for bf16."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from oracle.decoder_ref import quantize_int8_groups
from tests.gpu_helpers import (check_greedy_tokens, compare_logits, gpu_greedy, gpu_teacher_forced,
                               oracle_teacher_forced, tolerances)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantiser_bit_exact_against_oracle(dec_mod, dtype):
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(96, 256, generator=g) * 0.02).to(dtype)
    w[3, 32:64] = 0                           # an all-zero group: s = 0, codes 0
    w[4, :32] = torch.arange(-16, 16, dtype=torch.float32).to(dtype)
    w[4, 0] = 127                             # s = 1: k + 0.5 ties round away from zero
    w[4, 1:5] = torch.tensor([2.5, -2.5, 0.5, -0.5]).to(dtype)
    codes, scales = dec_mod.weight_quantize_int8(w.cuda())
    torch.cuda.synchronize()
    c_gpu, s_gpu = codes.cpu().numpy(), scales.cpu().numpy()
    wf = w.float().numpy().astype(np.float64)
    for r in range(w.shape[0]):
        c_ref, s_ref = quantize_int8_groups(wf[r], 32)
        assert np.array_equal(c_gpu[r], c_ref), r
        assert np.array_equal(s_gpu[r].view(np.uint32), s_ref.astype(np.float32).view(np.uint32)), r
    assert list(c_gpu[4, 1:5]) == [3, -3, 1, -1]


def _case(dec_mod, w, P, D, mode=None):
    d = dec_mod.Decoder(w)
    if mode:
        d.set_fused(mode)
    prompt = synthetic.prompt_tokens(w, P, seed=0)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
    ref, _ = oracle_teacher_forced(w, prompt, taus, D)
    tol_abs, tol_rel = tolerances(w)
    compare_logits(rows, ref, tol_abs, tol_rel)
    check_greedy_tokens(ref, taus, tol_abs)
    return d, prompt, rows, taus, ref


def test_toy_int8_weights(dec_mod):
    # The toy shape with ffn 192 (a whole number of 32-column groups), fp32 base weights.
    w = synthetic.workload("toy", ffn=192, weight_int8=True)
    _, _, rows, taus, ref = _case(dec_mod, w, 16, 8)
    assert [int(np.argmax(r)) for r in ref] == taus


def test_toy_moe_int8_weights(dec_mod):
    w = synthetic.workload("toy", ffn=192, n_experts=4, n_experts_used=2, weight_int8=True)
    _case(dec_mod, w, 16, 6)


def test_int8_weights_differ_from_the_unquantised_model(dec_mod):
    # The quantisation is really applied: the int8 model's logits move away from the
    # bf16 model's by more than the tolerance, and match the oracle's int8 mode within it.
    base = synthetic.workload("smollm2-135m", n_layers=2)
    q = dict(base, weight_int8=True)
    _, _, rows_q, taus, ref_q = _case(dec_mod, q, 24, 2)
    dq = dec_mod.Decoder(base)
    rows_b = gpu_teacher_forced(dq, synthetic.prompt_tokens(base, 24, seed=0), taus, 2)
    assert np.abs(rows_b - rows_q).max() > tolerances(q)[0]


@pytest.mark.parametrize("mode", ["off", "grid"])
def test_smollm2_shape_int8_weights(dec_mod, mode):
    w = synthetic.workload("smollm2-135m", n_layers=4, weight_int8=True)
    _case(dec_mod, w, 64, 8, mode)


@pytest.mark.parametrize("mode", ["grid", "off"])
def test_qwen_shape_int8_weights_tied_head(dec_mod, mode):
    # q/k/v biases, a tied (bf16) head beside 8-bit projections; "grid" is the
    # persistent step reading int8 tiles, "off" the row kernels.
    w = synthetic.workload("qwen2.5-0.5b", n_layers=3, weight_int8=True)
    d, *_ = _case(dec_mod, w, 48, 6, mode)
    assert d.fused_mode() == mode


def test_mistral_shape_int8_weights_untied_head(dec_mod):
    w = synthetic.workload("mistral-7b", n_layers=2, weight_int8=True)
    d, *_ = _case(dec_mod, w, 40, 6)
    assert d.fused_mode() == "grid"   # the persistent step with int8 tiles, the head included


def test_mixtral_shape_int8_weights_grouped_experts(dec_mod):
    w = synthetic.workload("mixtral-8x7b", n_layers=2, weight_int8=True)
    d, *_ = _case(dec_mod, w, 20, 4)
    assert d.fused_mode() == "grid"


def test_batched_decode_int8_weights(dec_mod):
    w = synthetic.workload("smollm2-135m", n_layers=2, weight_int8=True)
    B, P = 3, 20
    d = dec_mod.Decoder(w, n_seqs=B)
    lg = torch.empty(w["vocab"], device="cuda")
    prompts = [synthetic.prompt_tokens(w, P, seed=40 + b) for b in range(B)]
    for b in range(B):
        d.prefill(prompts[b], 0, lg, seq=b)
    tok = torch.tensor([11, 12, 13], dtype=torch.int32, device="cuda")
    out = torch.empty((B, w["vocab"]), device="cuda")
    d.decode_batch(list(range(B)), [P] * B, tok, out)
    d.check()
    o = out.cpu().numpy()
    from tests.gpu_helpers import oracle_session
    for b in range(B):
        s = oracle_session(w)
        ref = s.prefill_batched(list(prompts[b]) + [11 + b], 0, logits_rows=[P])
        compare_logits(o[b][None], ref, *tolerances(w))
