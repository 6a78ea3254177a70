"""GPU parity of the persistent decode step's two FFN schedules against the oracle.

Pantheon "Llama Forward Pass", feed-forward block: down(silu(gate) * up); Mixture of
Experts: the selected experts' outputs weighted by their renormalised router scores.
With bf16 weights whose hidden size is a whole number of 128-column blocks and whose
ffn size is a multiple of 16, the persistent step runs the FFN as one phase over ffn
slices (each CTA: its gate/up rows, then its slice of the transposed down projection
into a partial sum over the hidden size) and a second phase that sums the partials
into the residual in CTA order.  Other shapes keep a gate/up phase and a down phase.
Both are compared with the float64 oracle, teacher-forced on the GPU's greedy
tokens, at the bf16 tolerances."""

import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import (check_greedy_tokens, compare_logits, gpu_greedy, oracle_teacher_forced,
                               tolerances)

pytestmark = pytest.mark.gpu

# A small bf16 shape (hidden 256 = two 128-column blocks).
BASE = dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, vocab=1024, max_seq=64)


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def _run(dec_mod, w, fused, P=24, D=6):
    d = dec_mod.Decoder(w)
    d.set_fused("grid")
    assert d.fused_mode() == "grid"
    assert d.ffn_fused() == fused
    prompt = synthetic.prompt_tokens(w, P, seed=3)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
    ref, _ = oracle_teacher_forced(w, prompt, taus, D)
    tol_abs, tol_rel = tolerances(w)
    compare_logits(rows, ref, tol_abs, tol_rel)
    check_greedy_tokens(ref, taus, tol_abs)
    d.close()


@pytest.mark.parametrize("ffn", [1360, 1352])
def test_dense_ffn_fused_and_two_phase(dec_mod, ffn):
    # 1360 = 85 * 16: one FFN phase over ffn slices; 1352 (8 past a multiple of 16):
    # the gate/up and down phases.
    _run(dec_mod, synthetic.workload("smollm2-135m", ffn=ffn, **BASE), fused=ffn % 16 == 0)


def test_moe_ffn_fused_slice_straddles_experts(dec_mod):
    # 2 of 4 experts, ffn 1360: 2720 (slot, ffn) tasks over the CTAs in 32-task
    # shares on a 152-SM GPU, so one CTA's share ends in the second slot's rows.
    w = synthetic.workload("smollm2-135m", ffn=1360, n_experts=4, n_experts_used=2, **BASE)
    _run(dec_mod, w, fused=True)


def test_qwen_shape_ffn_fused_with_bias(dec_mod):
    # hidden 896 = seven 128-column blocks (seven of the eight warps own one each).
    _run(dec_mod, synthetic.workload("qwen2.5-0.5b", n_layers=2, max_seq=64), fused=True, P=32, D=4)


def test_per_layer_schedule_reports_no_fused_ffn(dec_mod):
    w = synthetic.workload("smollm2-135m", ffn=1360, **BASE)
    d = dec_mod.Decoder(w)
    d.set_fused("off")
    assert not d.ffn_fused()
    d.close()
