"""Design study on the host: how much the logits move when an operand of a prefill
product is rounded to one bf16 instead of being carried exactly.

TEST AND DESIGN INFRASTRUCTURE ONLY, like the rest of ``oracle/``: nothing in the
library imports or runs it.  It restates the batched single-pass prefill of
``decoder_ref.Session.prefill_batched`` (sipllm "Transformer forward pass", Single-pass
prefill; Pantheon "Llama Forward Pass", Forward Pass Flow) in float64 with rounding
points at the inputs of the products a tensor-core kernel takes in bf16, and runs
several rounding variants side by side over the same weights, so each layer's
weights are drawn once for all of them.

Rounding points (what the GPU's tensor-core operands are):
  qkv     the normalised rows entering [Wq; Wk; Wv]
  o       the attention output entering Wo
  gateup  the normalised rows entering the gate/up (or expert gate/up) matrices
  down    silu(g) * u entering the down (or expert down) matrices
  attn    q, k and v entering the attention products, and the softmax weights
          entering P.V
Weights are bf16 already (rounding them is the identity).  A point is either exact
(float64), "hilo" (the value as the sum of two bf16, hi = bf16(x), lo = bf16(x - hi):
about 16 significant bits) or "bf16" (one bf16).  The error of a variant is measured
against the all-exact forward on the logits of the last ``rows`` positions.

    python -m oracle.precision_study mixtral-8x7b --prompt 256 --rows 16
"""

from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle.decoder_ref import (F64, kv_head_of, rmsnorm, rope_inv_freq, rope_pairs, route_topk, silu,
                                window_start)

POINTS = ("qkv", "o", "gateup", "down", "attn")


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as float64: float32 first, then
    the low 16 bits of the float32 pattern rounded away."""
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def apply(x, mode: str) -> np.ndarray:
    if mode == "exact":
        return x
    hi = bf16_round(x)
    if mode == "bf16":
        return hi
    if mode == "hilo":
        return hi + bf16_round(x - hi)
    raise ValueError(mode)


def variants_default() -> dict:
    """name -> {point: mode}.  The library today: every GEMM input hilo, attention hilo."""
    base = {p: "hilo" for p in POINTS}
    v = {"exact": {p: "exact" for p in POINTS}, "hilo_all": dict(base)}
    for p in ("qkv", "o", "gateup", "down", "attn"):
        d = dict(base)
        d[p] = "bf16"
        v[f"bf16_{p}"] = d
    v["bf16_gemms"] = dict(base, qkv="bf16", o="bf16", gateup="bf16", down="bf16")
    v["bf16_all"] = {p: "bf16" for p in POINTS}
    return v


class _Stream:
    """One variant's residual rows and K/V lists."""

    def __init__(self, X, n_layers):
        self.X = X.copy()
        self.K = [None] * n_layers
        self.V = [None] * n_layers


def study(w: dict, weights, P: int, rows: int, variants: dict, seed_prompt: int = 0, log=print) -> dict:
    """Runs every variant over the same weights; returns name -> (max |d|, relative RMS)."""
    from decoder_only_forward_gb300 import synthetic
    h, nq, nkv, hd = w["hidden"], w["n_heads"], w["n_kv_heads"], w["head_dim"]
    L, E, k = w["n_layers"], w["n_experts"], w["n_experts_used"]
    toks = synthetic.prompt_tokens(w, P, seed=seed_prompt)
    X0 = weights.embed_rows(toks)
    streams = {name: _Stream(X0, L) for name in variants}
    pos = np.arange(P)
    inv = rope_inv_freq(hd, w["rope_theta"])
    ang = pos[:, None].astype(F64) * inv[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    ia, ib = rope_pairs(hd)
    lo = np.array([window_start(int(p), w["sliding_window"]) for p in pos])
    j = np.arange(P)
    mask = (j[None, :] > pos[:, None]) | (j[None, :] < lo[:, None])
    scale = 1.0 / math.sqrt(hd)

    def rot(T):
        a, b = T[..., ia].copy(), T[..., ib].copy()
        out = T.copy()
        out[..., ia] = a * cos[:, None, :] - b * sin[:, None, :]
        out[..., ib] = a * sin[:, None, :] + b * cos[:, None, :]
        return out

    for l in range(L):
        t0 = time.perf_counter()
        lw = weights.layer(l)
        for name, s in streams.items():
            md = variants[name]
            N = apply(rmsnorm(s.X, lw["attn_norm"], w["rms_eps"]), md["qkv"])
            Q, K, V = N @ lw["wq"].T, N @ lw["wk"].T, N @ lw["wv"].T
            if w["qkv_bias"]:
                Q, K, V = Q + lw["bq"], K + lw["bk"], V + lw["bv"]
            Q = apply(rot(Q.reshape(P, nq, hd)), md["attn"])
            K = apply(rot(K.reshape(P, nkv, hd)), md["attn"])
            V = apply(V.reshape(P, nkv, hd), md["attn"])
            O = np.empty((P, nq, hd), F64)
            for hh in range(nq):
                g = kv_head_of(hh, nq, nkv)
                S = (Q[:, hh, :] @ K[:, g, :].T) * scale
                S[mask] = -np.inf
                Pm = np.exp(S - S.max(axis=1, keepdims=True))
                den = Pm.sum(axis=1, keepdims=True)
                # The kernel multiplies unnormalised weights (the running-max form) with V
                # and divides by their sum afterwards: the rounding point is the weight.
                O[:, hh, :] = (apply(Pm, md["attn"]) @ V[:, g, :]) / den
            s.X = s.X + apply(O.reshape(P, nq * hd), md["o"]) @ lw["wo"].T
            N2 = apply(rmsnorm(s.X, lw["ffn_norm"], w["rms_eps"]), md["gateup"])
            if E:
                # Routing on the variant's own router logits (the router stays f32 on the GPU).
                R = rmsnorm(s.X, lw["ffn_norm"], w["rms_eps"]) @ lw["router"].T
                s.routes = [route_topk(R[t], k) for t in range(P)]
            else:
                s.routes = None
            s.N2 = N2
            s.F = np.zeros((P, h), F64)
        if E:
            for e in range(E):
                wg, wu, wd = weights.expert(l, e)
                for name, s in streams.items():
                    md = variants[name]
                    sel = [(t, sl) for t in range(P) for sl, ee in enumerate(s.routes[t][0]) if ee == e]
                    if not sel:
                        continue
                    rr = np.array([t for t, _ in sel])
                    A = apply(silu(s.N2[rr] @ wg.T) * (s.N2[rr] @ wu.T), md["down"])
                    Y = A @ wd.T
                    for i, (t, sl) in enumerate(sel):
                        s.F[t] += s.routes[t][1][sl] * Y[i]
        else:
            for name, s in streams.items():
                md = variants[name]
                A = apply(silu(s.N2 @ lw["w_gate"].T) * (s.N2 @ lw["w_up"].T), md["down"])
                s.F = A @ lw["w_down"].T
        for s in streams.values():
            s.X = s.X + s.F
            s.N2 = s.F = None
        log(f"layer {l + 1}/{L} {time.perf_counter() - t0:.1f} s")
    head, wn = weights.lm_head(), weights.out_norm()
    logits = {name: rmsnorm(s.X[-rows:], wn, w["rms_eps"]) @ head.T for name, s in streams.items()}
    ref = logits["exact"]
    out = {}
    for name, lg in logits.items():
        d = lg - ref
        out[name] = (float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref)))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--prompt", type=int, default=256)
    ap.add_argument("--rows", type=int, default=16)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--out", default="")
    a = ap.parse_args()
    import torch
    from decoder_only_forward_gb300 import synthetic
    torch.set_num_threads(len(os.sched_getaffinity(0)))
    w = synthetic.workload(a.workload)
    if a.layers:
        w["n_layers"] = a.layers
    if w["sliding_window"] and a.prompt > w["max_seq"]:
        raise SystemExit("prompt longer than the window")
    src = synthetic.OracleWeightSource(w, device="cpu", cache=False)
    res = study(w, src, a.prompt, a.rows, variants_default(), log=lambda m: print(m, file=sys.stderr, flush=True))
    rec = {"workload": a.workload, "layers": w["n_layers"], "prompt": a.prompt, "rows": a.rows,
           "max_abs_and_rel_rms_vs_exact": {k: [round(v[0], 6), round(v[1], 7)] for k, v in res.items()}}
    line = json.dumps(rec)
    print(line)
    if a.out:
        with open(a.out, "a") as f:
            f.write(line + "\n")


if __name__ == "__main__":
    main()
