"""GPU parity of the int8 K/V cache (kv_dtype DEC_I8) against the oracle's int8
cache (rml "The decoder", KV cache).

The quantiser itself is compared bit for bit: the same f32 rows go through the
library's kernel (dec_kv_quantize_int8) and the oracle, and codes and scales
must be identical.  End to end, the kernel quantises its own f32 K/V and the
oracle its float64 ones rounded to f32, so a code decided right at a rounding
boundary may differ by one step: logits are held to the bf16 tolerance and the
stored codes to "equal, or one step apart in a vanishing fraction"."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from oracle.decoder_ref import kv_group_size, quantize_int8_groups
from tests.gpu_helpers import TOL_BF16_ABS, TOL_BF16_REL, check_greedy_tokens, compare_logits, gpu_greedy
from tests.gpu_helpers import oracle_session

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


@pytest.mark.parametrize("nkv,hd", [(8, 128), (3, 64), (1, 16), (5, 16)])
def test_quantiser_bit_exact_against_oracle(dec_mod, nkv, hd):
    rng = np.random.default_rng(nkv * 100 + hd)
    n, kd = 37, nkv * hd
    x = rng.normal(0, 1, (n, kd)) * rng.choice([1.0, 1e-3, 30.0], (n, kd))
    x[0, :] = 0.0                                   # all-zero groups
    x[1, :] = 0.0
    x[1, 5] = -2.0                                  # a single spike
    g = kv_group_size(hd)
    x[2, :g] = np.r_[127.0, 2.5, -2.5, 0.5, -0.5, np.zeros(g - 5)]   # halves at s = 1
    x32 = x.astype(np.float32)
    out = dec_mod.kv_quantize_int8(torch.from_numpy(x32).cuda(), nkv, hd)
    torch.cuda.synchronize()
    scales, codes = dec_mod.split_int8_rows(out, nkv, hd)
    for r in range(n):
        ref_codes, ref_scales = quantize_int8_groups(x32[r], g)
        assert np.array_equal(codes[r].cpu().numpy(), ref_codes), f"row {r}"
        assert np.array_equal(scales[r].cpu().numpy(), ref_scales), f"row {r}"


def _oracle_int8(w, prompt, taus, D):
    s = oracle_session(dict(w, kv_int8=True))
    P = len(prompt)
    rows = s.prefill_batched(list(prompt) + list(taus[:D]), 0, logits_rows=list(range(P - 1, P + D)))
    return rows, s


def _check_ring_codes(d, dec_mod, w, sess, length, seq=0):
    """Stored codes/scales against the oracle's quantisation of its own K/V.

    f32 weights: K/V agree to ~1e-6, so scales to 2e-5 and almost every code.
    bf16 weights: the projection's bf16 rounding moves K/V by up to ~1e-3
    relative, so scales to 2e-3 and up to 5% of codes one step apart."""
    nkv, hd, ms = w["n_kv_heads"], w["head_dim"], w["max_seq"]
    f32 = w["dtype"] == "f32"
    rtol, frac = (2e-5, 1 / 2000) if f32 else (2e-3, 0.05)
    g = kv_group_size(hd)
    total = off_by_one = 0
    for l in range(w["n_layers"]):
        kr, vr = d.kv_layer(l, seq=seq)
        for rows, ref in ((kr, sess.keys[l]), (vr, sess.values[l])):
            sc, cd = dec_mod.split_int8_rows(rows, nkv, hd)
            sc, cd = sc.cpu().numpy(), cd.cpu().numpy().astype(np.int32)
            for p in range(max(0, length - ms), length):
                slot = p % ms if w["sliding_window"] else p
                # the oracle stores read-back values; re-quantising them gives its codes back
                rc, rs = quantize_int8_groups(np.asarray(ref[p]).reshape(-1), g)
                diff = np.abs(cd[slot] - rc.astype(np.int32))
                assert diff.max() <= 1, f"layer {l} pos {p}: codes differ by {diff.max()}"
                off_by_one += int(np.count_nonzero(diff))
                total += diff.size
                np.testing.assert_allclose(sc[slot], rs, rtol=rtol, atol=0)
    assert off_by_one <= max(2, int(total * frac)), f"{off_by_one} of {total} codes one step apart"


def test_toy_int8_cache_end_to_end(dec_mod):
    w = synthetic.workload("toy")
    d = dec_mod.Decoder(w, kv_dtype="i8")
    prompt = synthetic.prompt_tokens(w, 16, seed=0)
    rows, taus = gpu_greedy(d, prompt, 12, use_device_argmax=True)
    ref, sess = _oracle_int8(w, prompt, taus, 12)
    compare_logits(rows, ref, TOL_BF16_ABS, TOL_BF16_REL)
    check_greedy_tokens(ref, taus, TOL_BF16_ABS)
    _check_ring_codes(d, dec_mod, w, sess, 28)


def test_toy_int8_window_wraps_with_chunked_prefill(dec_mod):
    # Window 8 = max_seq 8, prompt of 13 in chunks of 5: history read back from the ring.
    w = synthetic.workload("toy", sliding_window=8, max_seq=8)
    d = dec_mod.Decoder(w, kv_dtype="i8", max_tokens=5)
    prompt = synthetic.prompt_tokens(w, 13, seed=3)
    rows, taus = gpu_greedy(d, prompt, 9)
    ref, sess = _oracle_int8(w, prompt, taus, 9)
    compare_logits(rows, ref, TOL_BF16_ABS, TOL_BF16_REL)
    _check_ring_codes(d, dec_mod, w, sess, 22)


def test_mistral_shape_int8_window(dec_mod):
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=24, max_seq=24)
    d = dec_mod.Decoder(w, kv_dtype="i8")
    prompt = synthetic.prompt_tokens(w, 30, seed=4)
    rows, taus = gpu_greedy(d, prompt, 6)
    ref, sess = _oracle_int8(w, prompt, taus, 6)
    compare_logits(rows, ref, TOL_BF16_ABS, TOL_BF16_REL)
    _check_ring_codes(d, dec_mod, w, sess, 36)


def test_qwen_shape_int8_batched(dec_mod):
    w = synthetic.workload("qwen2.5-0.5b", n_layers=2)
    lens = [9, 40, 3]
    prompts = [list(synthetic.prompt_tokens(w, n, seed=90 + i)) for i, n in enumerate(lens)]
    d = dec_mod.Decoder(w, kv_dtype="i8", n_seqs=3)
    V = w["vocab"]
    lg = torch.empty(V, device="cuda")
    rows = [[] for _ in lens]
    taus = [[] for _ in lens]
    for s_, p in enumerate(prompts):
        d.prefill(p, 0, lg, seq=s_)
        d.synchronize()
        rows[s_].append(lg.cpu().numpy().copy())
        taus[s_].append(int(np.argmax(rows[s_][-1])))
    tok = torch.tensor([t[0] for t in taus], dtype=torch.int32, device="cuda")
    out = torch.empty((3, V), device="cuda")
    for _ in range(5):
        d.decode_batch([0, 1, 2], [d.length_of(s_) for s_ in range(3)], tok, out, tok)
        d.synchronize()
        h = out.cpu().numpy()
        for s_ in range(3):
            rows[s_].append(h[s_].copy())
            taus[s_].append(int(np.argmax(h[s_])))
    d.check()
    for s_, p in enumerate(prompts):
        ref, sess = _oracle_int8(w, p, taus[s_], 5)
        compare_logits(np.stack(rows[s_]), ref, TOL_BF16_ABS, TOL_BF16_REL)
        _check_ring_codes(d, dec_mod, w, sess, lens[s_] + 5, seq=s_)


# The persistent decode step with an int8 cache (head_dim 128, bf16 weights): the
# warp attention reads each piece's codes and group scales by TMA and multiplies
# them back in registers; the task holding the current position quantises that row
# itself (the QKV phase leaves it in f32) with the cache's rule and writes it.


def _persistent_int8_case(dec_mod, w, P, D, seed):
    d = dec_mod.Decoder(w, kv_dtype="i8")
    d.set_fused("grid")
    assert d.fused_mode() == "grid"
    prompt = synthetic.prompt_tokens(w, P, seed=seed)
    rows, taus = gpu_greedy(d, prompt, D, use_device_argmax=True)
    ref, sess = _oracle_int8(w, prompt, taus, D)
    compare_logits(rows, ref, TOL_BF16_ABS, TOL_BF16_REL)
    check_greedy_tokens(ref, taus, TOL_BF16_ABS)
    _check_ring_codes(d, dec_mod, w, sess, P + D)
    return d, prompt, rows, taus


def test_mistral_shape_int8_persistent_long_prompt(dec_mod):
    # 300 keys per kv head: several 16-key pieces per warp and splits merged across CTAs.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=0, max_seq=320)
    _persistent_int8_case(dec_mod, w, 300, 8, seed=21)


def test_mistral_shape_int8_persistent_window_wraps(dec_mod):
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=40, max_seq=40)
    _persistent_int8_case(dec_mod, w, 36, 12, seed=22)


def test_mixtral_shape_int8_persistent(dec_mod):
    w = synthetic.workload("mixtral-8x7b", n_layers=2, max_seq=96)
    _persistent_int8_case(dec_mod, w, 64, 6, seed=23)


def test_int8_persistent_step_agrees_with_row_kernels(dec_mod):
    # The same model and prompt decoded by the persistent step and by the row kernels
    # (one row per step): the same tokens, logits within rounding.  The two paths
    # project K/V with different summation orders, so a channel at a code boundary
    # can land one int8 step apart (a step is 1/127 of its group's largest value):
    # the bound is looser than for the f32 cache.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=0, max_seq=96)
    prompt = synthetic.prompt_tokens(w, 70, seed=24)
    out = {}
    weights = None
    for mode in ("grid", "off"):
        d = dec_mod.Decoder(w, kv_dtype="i8", weights=weights)
        weights = d.weights
        d.set_fused(mode)
        out[mode] = gpu_greedy(d, prompt, 8)
        d.close()
    assert out["grid"][1] == out["off"][1]
    np.testing.assert_allclose(out["grid"][0], out["off"][0], atol=1e-2, rtol=1e-3)


def test_int8_persistent_grid_and_cluster_agree(dec_mod):
    # The one-cluster schedule runs the same int8-cache attention code on 16 (or 8) CTAs.
    w = synthetic.workload("mistral-7b", n_layers=2, sliding_window=0, max_seq=96)
    prompt = synthetic.prompt_tokens(w, 50, seed=25)
    out = {}
    weights = None
    for mode in ("grid", "cluster"):
        d = dec_mod.Decoder(w, kv_dtype="i8", weights=weights)
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
