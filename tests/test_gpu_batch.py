"""GPU parity of batched multi-sequence decode (dec_decode_batch) against the
float64 oracle: every sequence of a batch, with its own prompt, length and
position, must give the logits the oracle gives for that sequence alone, and a
row's result must not depend on the rest of the batch."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from tests.gpu_helpers import check_greedy_tokens, compare_logits, oracle_teacher_forced, ring_positions, tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


def batch_greedy(d, prompts, D, order=None):
    """Prefill sequence i with prompts[i], then D greedy steps of all sequences as one batch
    (rows in ``order``, default 0..n-1), tokens fed back from the device argmax.
    Returns per sequence the logit rows [D+1, V] and the greedy tokens."""
    n, V = len(prompts), d.w["vocab"]
    order = list(range(n)) if order is None else list(order)
    rows = [[] for _ in range(n)]
    taus = [[] for _ in range(n)]
    lg = torch.empty(V, dtype=torch.float32, device="cuda")
    for s, p in enumerate(prompts):
        d.prefill(p, 0, lg, seq=s)
        d.synchronize()
        rows[s].append(lg.cpu().numpy().copy())
        taus[s].append(int(np.argmax(rows[s][-1])))
    B = len(order)
    d_tok = torch.tensor([taus[s][0] for s in order], dtype=torch.int32, device="cuda")
    d_arg = torch.empty(B, dtype=torch.int32, device="cuda")
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    for _ in range(D):
        pos = [d.length_of(s) for s in order]
        d.decode_batch(order, pos, d_tok, logits, d_arg)
        d.synchronize()
        host = logits.cpu().numpy()
        arg = d_arg.cpu().numpy()
        for i, s in enumerate(order):
            rows[s].append(host[i].copy())
            nxt = int(np.argmax(host[i]))
            assert int(arg[i]) == nxt, "device argmax differs from host argmax"
            taus[s].append(nxt)
        d_tok.copy_(d_arg)
    d.check()
    return [np.stack(r) for r in rows], taus


def _check_against_oracle(w, prompts, rows, taus, D, kv="f32"):
    tol_abs, tol_rel = tolerances(w, kv)
    sessions = []
    for s, p in enumerate(prompts):
        ref, sess = oracle_teacher_forced(w, p, taus[s], D)
        compare_logits(rows[s], ref, tol_abs, tol_rel)
        check_greedy_tokens(ref, taus[s], tol_abs)
        sessions.append(sess)
    return sessions


def test_toy_batch_ragged_prompts(dec_mod):
    w = synthetic.workload("toy")
    lens = [5, 9, 16, 2]
    prompts = [list(synthetic.prompt_tokens(w, n, seed=10 + i)) for i, n in enumerate(lens)]
    d = dec_mod.Decoder(w, n_seqs=len(prompts))
    D = 12
    rows, taus = batch_greedy(d, prompts, D)
    sessions = _check_against_oracle(w, prompts, rows, taus, D)
    # Each sequence's ring holds its own K/V at the slots of its own positions.
    for s, sess in enumerate(sessions):
        n = lens[s] + D
        assert d.length_of(s) == n
        for l in range(w["n_layers"]):
            kc, vc = d.kv_layer(l, seq=s)
            for p in range(n):
                np.testing.assert_allclose(kc[p].cpu().numpy(), sess.keys[l][p], atol=1e-5, rtol=1e-5)
                np.testing.assert_allclose(vc[p].cpu().numpy(), sess.values[l][p], atol=1e-5, rtol=1e-5)


def test_toy_batch_window_wraps(dec_mod):
    # Window 8 = max_seq 8: sequences at different phases of their rings, all wrapping while decoding.
    w = synthetic.workload("toy", sliding_window=8, max_seq=8)
    lens = [3, 8, 12]
    prompts = [list(synthetic.prompt_tokens(w, n, seed=20 + i)) for i, n in enumerate(lens)]
    d = dec_mod.Decoder(w, n_seqs=3)
    D = 10
    rows, taus = batch_greedy(d, prompts, D, order=[2, 0, 1])
    sessions = _check_against_oracle(w, prompts, rows, taus, D)
    for s, sess in enumerate(sessions):
        n = lens[s] + D
        slots = ring_positions(n, w["max_seq"], w["sliding_window"])
        for l in range(w["n_layers"]):
            kc, _ = d.kv_layer(l, seq=s)
            for sl, p in enumerate(slots):
                np.testing.assert_allclose(kc[sl].cpu().numpy(), sess.keys[l][p], atol=1e-5, rtol=1e-5)


def test_toy_moe_batch(dec_mod):
    w = synthetic.workload("toy", n_experts=4, n_experts_used=2)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=30 + i)) for i, n in enumerate([4, 11])]
    d = dec_mod.Decoder(w, n_seqs=2)
    rows, taus = batch_greedy(d, prompts, 8)
    _check_against_oracle(w, prompts, rows, taus, 8)


def test_mistral_shape_batch_window(dec_mod):
    # Mistral-shaped layers (GQA 32/8, tensor-core GEMMs), a 24-slot window, four sequences.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=24, max_seq=24)
    lens = [10, 20, 30, 5]
    prompts = [list(synthetic.prompt_tokens(w, n, seed=40 + i)) for i, n in enumerate(lens)]
    d = dec_mod.Decoder(w, n_seqs=4)
    D = 6
    rows, taus = batch_greedy(d, prompts, D, order=[1, 3, 0, 2])
    _check_against_oracle(w, prompts, rows, taus, D)


def test_toy_batch_bf16_kv(dec_mod):
    # bf16 K/V storage: the oracle keeps exact K/V, so the bf16 tolerance applies.
    w = synthetic.workload("toy")
    prompts = [list(synthetic.prompt_tokens(w, n, seed=45 + i)) for i, n in enumerate([7, 12, 1])]
    d = dec_mod.Decoder(w, n_seqs=3, kv_dtype="bf16")
    rows, taus = batch_greedy(d, prompts, 10)
    _check_against_oracle(w, prompts, rows, taus, 10, "bf16")


def test_qwen_shape_batch_bias(dec_mod):
    # q/k/v biases, 14/2 heads, head_dim 64, tied 151936-row head.
    w = synthetic.workload("qwen2.5-0.5b", n_layers=2)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=50 + i)) for i, n in enumerate([7, 33, 64])]
    d = dec_mod.Decoder(w, n_seqs=3)
    rows, taus = batch_greedy(d, prompts, 5)
    _check_against_oracle(w, prompts, rows, taus, 5)


def test_mixtral_shape_batch(dec_mod):
    w = synthetic.workload("mixtral-8x7b", n_layers=2)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=60 + i)) for i, n in enumerate([6, 13])]
    d = dec_mod.Decoder(w, n_seqs=2)
    rows, taus = batch_greedy(d, prompts, 3)
    _check_against_oracle(w, prompts, rows, taus, 3)


@pytest.mark.parametrize("name", ["toy", "smollm2-135m"])
def test_row_result_independent_of_batch(dec_mod, name):
    # The same three sequences stepped as one batch in one order, and on a second handle as
    # a batch of two in another order plus a batch of one: every row bit-identical.
    w = synthetic.workload(name, n_layers=2) if name != "toy" else synthetic.workload(name)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=70 + i)) for i, n in enumerate([6, 17, 3])]
    weights = dec_mod.DeviceWeights(w)
    a = dec_mod.Decoder(w, weights=weights, n_seqs=3)
    b = dec_mod.Decoder(w, weights=weights, n_seqs=3)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    first = []
    for s, p in enumerate(prompts):
        a.prefill(p, 0, lg, seq=s)
        b.prefill(p, 0, lg, seq=s)
        a.synchronize()
        b.synchronize()
        first.append(int(lg.argmax().item()))
    for step in range(3):
        tok = torch.tensor(first, dtype=torch.int32, device="cuda")
        out_a = torch.empty((3, V), device="cuda")
        a.decode_batch([0, 1, 2], [a.length_of(s) for s in range(3)], tok, out_a)
        out_b2 = torch.empty((2, V), device="cuda")
        b.decode_batch([2, 0], [b.length_of(2), b.length_of(0)], tok[[2, 0]].contiguous(), out_b2)
        out_b1 = torch.empty((1, V), device="cuda")
        b.decode_batch([1], [b.length_of(1)], tok[[1]].contiguous(), out_b1)
        a.synchronize()
        b.synchronize()
        assert torch.equal(out_a[0], out_b2[1])
        assert torch.equal(out_a[1], out_b1[0])
        assert torch.equal(out_a[2], out_b2[0])
        first = [int(x) for x in out_a.argmax(dim=1).tolist()]
    a.check()
    b.check()


def test_batch_matches_single_sequence_decode(dec_mod):
    # Sequence 0 stepped by dec_decode and a copy stepped inside a batch agree to rounding.
    w = synthetic.workload("toy")
    p = list(synthetic.prompt_tokens(w, 9, seed=80))
    d = dec_mod.Decoder(w, n_seqs=2)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    d.prefill(p, 0, lg, seq=0)
    d.prefill(p, 0, lg, seq=1)
    tok = int(lg.argmax().item())
    single = torch.empty(V, device="cuda")
    both = torch.empty((1, V), device="cuda")
    for i in range(5):
        d.decode(tok, 9 + i, single)
        d.decode_batch([1], [9 + i], torch.tensor([tok], dtype=torch.int32, device="cuda"), both)
        d.synchronize()
        compare_logits(both[0].cpu().numpy(), single.cpu().numpy().astype(np.float64), 1e-4, 1e-4)
        tok = int(single.argmax().item())


def test_batch_argument_errors_change_nothing(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w, n_seqs=3)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    d.prefill([1, 2, 3], 0, lg, seq=0)
    d.prefill([4, 5], 0, lg, seq=1)
    tok = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    out = torch.empty((2, V), device="cuda")
    cases = [
        ([0, 0], [3, 3]),        # a sequence twice
        ([0, 3], [3, 0]),        # sequence out of range
        ([0, 1], [4, 2]),        # position beyond the length
        ([0, 1], [3, -1]),       # negative position
    ]
    for seqs, pos in cases:
        with pytest.raises(dec_mod.DecError) as ei:
            d.decode_batch(seqs, pos, tok, out)
        assert ei.value.status == dec_mod.DEC_EINVAL
        assert (d.length_of(0), d.length_of(1), d.length_of(2)) == (3, 2, 0)
    with pytest.raises(dec_mod.DecError):
        d.decode_batch([], [], tok, out)
    with pytest.raises(dec_mod.DecError) as ei:
        d.prefill([1], 0, lg, seq=3)
    assert ei.value.status == dec_mod.DEC_EINVAL
    # Without a window, a full sequence reports DEC_ERANGE.
    full = list(synthetic.prompt_tokens(w, w["max_seq"], seed=1))
    d.prefill(full, 0, lg, seq=2)
    with pytest.raises(dec_mod.DecError) as ei:
        d.decode_batch([2], [w["max_seq"]], tok[:1].contiguous(), out[:1])
    assert ei.value.status == dec_mod.DEC_ERANGE
    d.decode_batch([0, 1], [3, 2], tok, out)
    d.check()
    assert (d.length_of(0), d.length_of(1)) == (4, 3)


def test_batch_device_token_out_of_range_reported(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w, n_seqs=2)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    d.prefill([1, 2], 0, lg, seq=0)
    d.prefill([3], 0, lg, seq=1)
    out = torch.empty((2, V), device="cuda")
    d.decode_batch([0, 1], [2, 1], torch.tensor([5, V + 7], dtype=torch.int32, device="cuda"), out)
    with pytest.raises(dec_mod.DecError) as ei:
        d.check()
    assert ei.value.status == dec_mod.DEC_EINVAL
    d.check()  # the flag was cleared by the report


def test_smollm2_shape_batch_bf16_kv(dec_mod):
    # bf16 rings with head_dim 64 take the compact-tile attention; 9 query heads over 3 kv heads.
    w = synthetic.workload("smollm2-135m", n_layers=4)
    prompts = [list(synthetic.prompt_tokens(w, n, seed=85 + i)) for i, n in enumerate([20, 77, 5])]
    d = dec_mod.Decoder(w, n_seqs=3, kv_dtype="bf16")
    rows, taus = batch_greedy(d, prompts, 6, order=[2, 0, 1])
    _check_against_oracle(w, prompts, rows, taus, 6, "bf16")
