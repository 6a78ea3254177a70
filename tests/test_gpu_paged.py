"""GPU parity of the paged K/V cache (rml "The decoder", KV cache: pages of
page_size positions from one arena reserved up front, taken by a sequence only
when a position first lands in them).  Logits against the float64 oracle, each
cached row against the oracle's K/V, page accounting, and running out of pages
as an error that changes nothing."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import compare_logits, gpu_greedy, oracle_teacher_forced, tolerances
from tests.test_gpu_batch import batch_greedy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def _check(w, prompts, rows, taus, D, kv="f32"):
    sessions = []
    for s_, p in enumerate(prompts):
        ref, sess = oracle_teacher_forced(dict(w, kv_int8=(kv == "i8")), p, taus[s_], D)
        compare_logits(rows[s_], ref, *tolerances(w, "bf16" if kv == "i8" else kv))
        sessions.append(sess)
    return sessions


def test_toy_paged_batch_uses_pages_as_sequences_grow(dec_mod):
    w = synthetic.workload("toy")                     # max_seq 32: two pages of 16 per sequence
    lens = [6, 20, 3]
    prompts = [list(synthetic.prompt_tokens(w, n, seed=110 + i)) for i, n in enumerate(lens)]
    d = dec_mod.Decoder(w, n_seqs=3, page_size=16, n_pages=5)
    assert d.pages_free == 5
    D = 11
    rows, taus = batch_greedy(d, prompts, D, order=[1, 2, 0])
    sessions = _check(w, prompts, rows, taus, D)
    # 17 positions -> 2 pages, 31 -> 2 pages, 14 -> 1 page: the whole arena.
    assert d.pages_free == 0
    for s_, sess in enumerate(sessions):
        for l in range(w["n_layers"]):
            for p in range(lens[s_] + D):
                k, v = d.kv_slot(l, s_, p)
                np.testing.assert_allclose(k.cpu().numpy(), sess.keys[l][p], atol=1e-5, rtol=1e-5)
                np.testing.assert_allclose(v.cpu().numpy(), sess.values[l][p], atol=1e-5, rtol=1e-5)
    # No page left: a call that needs one fails before anything changes.
    lg = torch.empty(w["vocab"], device="cuda")
    with pytest.raises(dec_mod.DecError) as ei:
        d.prefill(list(synthetic.prompt_tokens(w, 4, seed=1)), d.length_of(2), lg, seq=2)
    assert ei.value.status == dec_mod.DEC_ENOMEM
    assert d.length_of(2) == lens[2] + D and d.pages_free == 0
    # Returning a sequence's pages lets it (or another) grow again.
    d.kv_reset(1)
    assert d.pages_free == 2
    d.prefill(list(synthetic.prompt_tokens(w, 4, seed=1)), d.length_of(2), lg, seq=2)
    d.synchronize()
    d.check()
    assert d.pages_free == 1


def test_toy_paged_window_wraps_with_chunked_prefill(dec_mod):
    # Window 32 = max_seq 32 in pages of 16: the prompt of 40 wraps inside one call (chunks of 12).
    w = synthetic.workload("toy", sliding_window=32, max_seq=32)
    d = dec_mod.Decoder(w, max_tokens=12, page_size=16, n_pages=2)
    prompt = synthetic.prompt_tokens(w, 40, seed=7)
    rows, taus = gpu_greedy(d, prompt, 10)
    ref, _ = oracle_teacher_forced(w, prompt, taus, 10)
    tol, _ = tolerances(w)
    compare_logits(rows, ref, tol, tol)
    assert d.pages_free == 0


def test_toy_paged_int8_cache(dec_mod):
    w = synthetic.workload("toy")
    prompts = [list(synthetic.prompt_tokens(w, n, seed=120 + i)) for i, n in enumerate([9, 17])]
    d = dec_mod.Decoder(w, n_seqs=2, kv_dtype="i8", page_size=16, n_pages=4)
    rows, taus = batch_greedy(d, prompts, 8)
    _check(w, prompts, rows, taus, 8, "i8")


def test_mistral_shape_paged_window_batch(dec_mod):
    # Window 48 in pages of 16 (3 per sequence), tensor-core GEMMs and prefill attention.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=48, max_seq=48)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=130 + i)) for i, n in enumerate([30, 55])]
    d = dec_mod.Decoder(w, n_seqs=2, page_size=16, n_pages=6)
    rows, taus = batch_greedy(d, prompts, 5, order=[1, 0])
    _check(w, prompts, rows, taus, 5)
    assert d.pages_free == 0
