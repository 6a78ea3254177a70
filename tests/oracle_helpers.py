"""Test-side helpers: small random models for the oracle pins, and an independent
float64 forward built from torch library routines (no code shared with the oracle).
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

from oracle import DictWeights, OracleConfig


def toy_cfg(**kw) -> OracleConfig:
    d = dict(n_layers=2, hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn=44, vocab=50,
             rms_eps=1e-5, rope_theta=10000.0)
    d.update(kw)
    return OracleConfig(**d)


def random_weights(cfg: OracleConfig, seed: int = 0, zero_layers: bool = False) -> DictWeights:
    rng = np.random.default_rng(seed)
    h, f = cfg.hidden, cfg.ffn
    qd, kd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim

    def mat(*shape, s=0.2):
        return np.zeros(shape) if zero_layers else rng.normal(0.0, s, shape)

    layers, experts = [], []
    for _ in range(cfg.n_layers):
        lw = dict(attn_norm=1 + rng.normal(0, 0.1, h), ffn_norm=1 + rng.normal(0, 0.1, h),
                  wq=mat(qd, h), wk=mat(kd, h), wv=mat(kd, h), wo=mat(h, qd))
        if cfg.qkv_bias:
            lw.update(bq=mat(qd), bk=mat(kd), bv=mat(kd))
        if cfg.qk_norm:
            nq_w, nk_w = (cfg.head_dim, cfg.head_dim) if cfg.qk_norm == "head" else (qd, kd)
            lw.update(q_norm=1 + rng.normal(0, 0.1, nq_w), k_norm=1 + rng.normal(0, 0.1, nk_w))
        if cfg.sandwich_norms:
            lw.update(post_attn_norm=1 + rng.normal(0, 0.1, h), post_ffn_norm=1 + rng.normal(0, 0.1, h))
        if cfg.n_experts:
            lw["router"] = mat(cfg.n_experts, h, s=0.5)
            experts.append([(mat(f, h), mat(f, h), mat(h, f)) for _ in range(cfg.n_experts)])
        else:
            lw.update(w_gate=mat(f, h), w_up=mat(f, h), w_down=mat(h, f))
        layers.append(lw)
    embd = rng.normal(0, 1.0, (cfg.vocab, h))
    head = rng.normal(0, 0.2, (cfg.vocab, h))
    return DictWeights(embd, 1 + rng.normal(0, 0.1, h), layers, lm_head=head,
                       experts=experts or None)


def torch_library_forward(cfg: OracleConfig, w: DictWeights, tokens) -> np.ndarray:
    """All-position logits from scratch, float64, through torch library routines.

    RMSNorm: F.rms_norm.  RoPE: complex multiplication of adjacent pairs by
    polar(1, pos * freq) (the complex form of the rotation).  Attention:
    F.scaled_dot_product_attention with an explicit boolean causal/window mask
    and enable_gqa (head h uses kv head h // group).  FFN: F.linear + F.silu.
    MoE: torch.softmax, torch.topk, division by the selected sum.  QK-norm and
    sandwich norms: F.rms_norm over each head / the row / the block output.
    """
    d = torch.float64
    T = lambda a: torch.as_tensor(np.asarray(a), dtype=d)
    n = len(tokens)
    h, nq, nkv, hd = cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    X = T(w.embed_rows(tokens))
    pos = torch.arange(n, dtype=d)
    def cis_of(theta):
        freq = theta ** (-torch.arange(0, hd, 2, dtype=d) / hd)
        return torch.polar(torch.ones(n, hd // 2, dtype=d), pos[:, None] * freq[None, :])

    cis_global = cis_of(cfg.rope_theta)
    cis_local = cis_of(cfg.rope_theta_local) if cfg.rope_theta_local else cis_global
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    allowed = j <= i
    if cfg.sliding_window > 0:
        allowed &= j >= i - cfg.sliding_window + 1

    def rope(Y, heads, cis):
        c = torch.view_as_complex(Y.reshape(n, heads, hd // 2, 2).contiguous())
        return torch.view_as_real(c * cis[:, None, :]).reshape(n, heads, hd)

    for l in range(cfg.n_layers):
        lw = {k: (None if v is None else T(v)) for k, v in w.layer(l).items()}
        N = F.rms_norm(X, (h,), weight=lw["attn_norm"], eps=cfg.rms_eps)
        Q = F.linear(N, lw["wq"], lw.get("bq"))
        K = F.linear(N, lw["wk"], lw.get("bk"))
        V = F.linear(N, lw["wv"], lw.get("bv"))
        if cfg.qk_norm == "head":
            Q = F.rms_norm(Q.reshape(n, nq, hd), (hd,), weight=lw["q_norm"], eps=cfg.rms_eps).reshape(n, -1)
            K = F.rms_norm(K.reshape(n, nkv, hd), (hd,), weight=lw["k_norm"], eps=cfg.rms_eps).reshape(n, -1)
        elif cfg.qk_norm == "row":
            Q = F.rms_norm(Q, (nq * hd,), weight=lw["q_norm"], eps=cfg.rms_eps)
            K = F.rms_norm(K, (nkv * hd,), weight=lw["k_norm"], eps=cfg.rms_eps)
        # Gemma-style base per layer: every rope_global_every-th layer (1-based) is global.
        is_global = not cfg.rope_theta_local or (cfg.rope_global_every and (l + 1) % cfg.rope_global_every == 0)
        cis = cis_global if is_global else cis_local
        Q, K = rope(Q, nq, cis), rope(K, nkv, cis)
        V = V.reshape(n, nkv, hd)
        O = F.scaled_dot_product_attention(Q.transpose(0, 1)[None], K.transpose(0, 1)[None],
                                           V.transpose(0, 1)[None], attn_mask=allowed,
                                           enable_gqa=True)
        A = F.linear(O[0].transpose(0, 1).reshape(n, nq * hd), lw["wo"])
        if cfg.sandwich_norms:
            A = F.rms_norm(A, (h,), weight=lw["post_attn_norm"], eps=cfg.rms_eps)
        X = X + A
        N2 = F.rms_norm(X, (h,), weight=lw["ffn_norm"], eps=cfg.rms_eps)
        if cfg.n_experts:
            probs = torch.softmax(F.linear(N2, lw["router"]), dim=-1)
            top = torch.topk(probs, cfg.n_experts_used, dim=-1)
            wts = top.values / top.values.sum(-1, keepdim=True)
            Fo = torch.zeros_like(X)
            for t in range(n):
                for s in range(cfg.n_experts_used):
                    wg, wu, wd = (T(a) for a in w.expert(l, int(top.indices[t, s])))
                    Fo[t] += wts[t, s] * F.linear(F.silu(F.linear(N2[t], wg)) * F.linear(N2[t], wu), wd)
        else:
            Fo = F.linear(F.silu(F.linear(N2, lw["w_gate"])) * F.linear(N2, lw["w_up"]), lw["w_down"])
        if cfg.sandwich_norms:
            Fo = F.rms_norm(Fo, (h,), weight=lw["post_ffn_norm"], eps=cfg.rms_eps)
        X = X + Fo
    Nf = F.rms_norm(X, (h,), weight=T(w.out_norm()), eps=cfg.rms_eps)
    return F.linear(Nf, T(w.lm_head())).numpy()
