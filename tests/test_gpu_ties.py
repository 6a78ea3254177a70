"""Tie rules on the GPU: equal router logits pick the lower expert id, equal maximum
logits make the greedy argmax return the lower token id.

rml "The decoder", Mixture of experts: top-k by repeated selection, ties to the lower
id; the same rule for the greedy argmax (the lower token id).  Ties are made exactly
by copying weight rows: two equal router rows give bit-equal router logits, a copied
LM-head row gives a bit-equal logit.  Every path that selects is checked: the
prefill router and argmax, the per-layer and persistent decode steps, and the
batched decode step's argmax."""

import numpy as np
import pytest
import torch

from decoder_only_forward_gb300 import synthetic
from oracle import OracleConfig, Session, route_topk
from tests.gpu_helpers import compare_logits, tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return dec


class _RouterCopies:
    """Oracle weight source whose router row e + E/2 is a copy of row e (e < E/2)."""

    def __init__(self, inner):
        self.inner = inner
        self.cfg = inner.cfg

    def layer(self, l):
        lw = dict(self.inner.layer(l))
        r = np.array(lw["router"], copy=True)
        half = r.shape[0] // 2
        r[half:] = r[:half]
        lw["router"] = r
        return lw

    def embed_rows(self, t):
        return self.inner.embed_rows(t)

    def out_norm(self):
        return self.inner.out_norm()

    def lm_head(self):
        return self.inner.lm_head()

    def expert(self, l, e):
        return self.inner.expert(l, e)


@pytest.mark.parametrize("name,kw,mode", [
    ("toy", dict(n_experts=4, n_experts_used=2), "off"),
    ("toy", dict(n_experts=4, n_experts_used=2), "grid"),
    ("mixtral-8x7b", dict(n_layers=2), "off"),
    ("mixtral-8x7b", dict(n_layers=2), "grid"),
])
def test_equal_router_rows_pick_lower_ids(dec_mod, name, kw, mode):
    w = synthetic.workload(name, **kw)
    weights = dec_mod.DeviceWeights(w)
    half = w["n_experts"] // 2
    for L in weights.layers:
        r = L["router"]
        r[half:].copy_(r[:half])      # every expert has a twin: logits e and e + E/2 are equal
    d = dec_mod.Decoder(w, weights=weights)
    d.set_fused(mode)
    P, D = 20, 6
    cap, k, E = P + D, w["n_experts_used"], w["n_experts"]
    ids_t = torch.full((w["n_layers"] * cap * k,), -1, dtype=torch.int32, device="cuda")
    lg_t = torch.zeros((w["n_layers"] * cap * E,), dtype=torch.float32, device="cuda")
    d.set_trace(ids_t, lg_t, cap)
    prompt = synthetic.prompt_tokens(w, P, seed=11)
    extra = synthetic.prompt_tokens(w, D, seed=12)
    logits = torch.empty(w["vocab"], device="cuda")
    d.prefill(prompt, 0, logits)                      # prefill router (row kernels)
    for i in range(D):
        d.decode(int(extra[i]), P + i, logits)        # decode router of this schedule
    d.check()
    ids = ids_t.view(w["n_layers"], cap, k).cpu().numpy()
    lg = lg_t.view(w["n_layers"], cap, E).cpu().numpy()
    src = synthetic.OracleWeightSource(w, device="cuda", cache=True)
    sess = Session(OracleConfig.from_dict(w), _RouterCopies(src), trace=True)
    ref = sess.prefill_batched(list(prompt) + list(extra), 0, logits_rows=[P + D - 1])
    compare_logits(logits.cpu().numpy()[None], ref, *tolerances(w))
    for l in range(w["n_layers"]):
        for p in range(cap):
            # Copied rows give bit-equal logits, so the tie is exact on the device...
            assert np.array_equal(lg[l, p, half:], lg[l, p, :half]), (l, p)
            got = list(ids[l, p])
            # ...the top two are the best expert of the first half and its twin, and the
            # lower id is taken first.
            e = int(np.argmax(lg[l, p, :half]))
            assert got == [e, e + half], (l, p, got)
            assert got == route_topk(lg[l, p].astype(np.float64), k)[0], (l, p)
            assert got == sess.trace.expert_ids[(l, p)], (l, p)


def _argmax_ties(dec_mod, mode):
    """Argmax over a logit vector whose maximum is shared by two rows."""
    w = synthetic.workload("toy")                     # untied head: the head's rows are free to edit
    weights = dec_mod.DeviceWeights(w)
    P, steps = 10, 3
    prompt = synthetic.prompt_tokens(w, P, seed=21)
    feed = [int(t) for t in synthetic.prompt_tokens(w, steps, seed=22)]

    def run(dw):
        d = dec_mod.Decoder(w, weights=dw)
        d.set_fused(mode)
        lg = torch.empty(w["vocab"], device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        rows, args = [], []
        d.prefill(prompt, 0, lg, am)
        d.synchronize()
        rows.append(lg.cpu().numpy().copy())
        args.append(int(am.item()))
        for i in range(steps):
            tok = torch.tensor([feed[i]], dtype=torch.int32, device="cuda")
            d.decode_dev(tok, P + i, lg, am)
            d.synchronize()
            rows.append(lg.cpu().numpy().copy())
            args.append(int(am.item()))
        d.check()
        d.close()
        return rows, args

    rows0, args0 = run(weights)
    tops = [int(np.argmax(r)) for r in rows0]
    assert args0 == tops
    # Copy each step's winning row into another row: the copy's logit equals the maximum.
    # Copies go to a lower id for some steps and a higher id for others.
    head = weights.lm_head
    used = set(tops)
    expect = []
    for s, t in enumerate(tops):
        cands = [c for c in (range(t) if s % 2 == 0 else range(w["vocab"] - 1, t, -1)) if c not in used]
        if not cands:
            cands = [c for c in range(w["vocab"]) if c not in used]
        a = cands[0]
        used.add(a)
        head[a].copy_(head[t])
        expect.append((a, t))
    rows1, args1 = run(weights)
    for s, (a, t) in enumerate(expect):
        r = rows1[s]
        assert r[a] == r[t] == r.max(), (s, a, t)
        assert args1[s] == min(a, t), (s, a, t, args1[s])
        assert int(np.argmax(r)) == min(a, t)
    return w, weights, prompt, expect


@pytest.mark.parametrize("mode", ["off", "grid"])
def test_equal_max_logits_argmax_takes_lower_id(dec_mod, mode):
    _argmax_ties(dec_mod, mode)


def test_batched_argmax_takes_lower_id(dec_mod):
    w = synthetic.workload("toy")
    weights = dec_mod.DeviceWeights(w)
    P = 10
    prompt = synthetic.prompt_tokens(w, P, seed=21)
    B = 3
    d = dec_mod.Decoder(w, weights=weights, n_seqs=B)
    lg1 = torch.empty(w["vocab"], device="cuda")
    for sq in range(B):
        d.prefill(prompt, 0, lg1, seq=sq)
    tok = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    out = torch.empty((B, w["vocab"]), device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    d.decode_batch(list(range(B)), [P] * B, tok, out, am)
    d.synchronize()
    t = int(np.argmax(out[0].cpu().numpy()))
    lower = [c for c in range(t)]
    a = lower[0] if lower else w["vocab"] - 1
    weights.lm_head[a].copy_(weights.lm_head[t])
    for sq in range(B):
        d.kv_reset(sq)
        d.prefill(prompt, 0, lg1, seq=sq)
    d.decode_batch(list(range(B)), [P] * B, tok, out, am)
    d.check()
    o = out.cpu().numpy()
    for b in range(B):
        assert o[b, a] == o[b, t] == o[b].max()
        assert int(am[b].item()) == min(a, t)
