"""Shared pieces of the GPU parity tests: run the library, run the oracle on the
same seeded inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

from decoder_only_forward_gb300 import synthetic
from oracle import OracleConfig, Session

# Tolerances on logits (bf16 weights with fp32 accumulation / the fp32 toy).
TOL_BF16_ABS, TOL_BF16_REL = 2e-2, 1e-2
TOL_F32_ABS = 1e-4


def tolerances(w: dict, kv: str = "f32"):
    if w["dtype"] == "f32" and kv == "f32":
        return TOL_F32_ABS, TOL_F32_ABS
    return TOL_BF16_ABS, TOL_BF16_REL


def gpu_greedy(dec, prompt, n_decode: int, use_device_argmax: bool = False):
    """Prefill the prompt, then greedy-decode.  Returns (logit rows [n_decode+1, V], tokens)."""
    V = dec.w["vocab"]
    logits = torch.empty(V, dtype=torch.float32, device=dec.device)
    rows = []
    P = len(prompt)
    dec.prefill(prompt, 0, logits)
    dec.synchronize()
    rows.append(logits.cpu().numpy().copy())
    taus = [int(np.argmax(rows[-1]))]
    d_tok = torch.tensor([taus[0]], dtype=torch.int32, device=dec.device)
    d_arg = torch.empty(1, dtype=torch.int32, device=dec.device)
    for i in range(n_decode):
        if use_device_argmax:
            dec.decode_dev(d_tok, P + i, logits, d_arg)
        else:
            dec.decode(taus[-1], P + i, logits)
        dec.synchronize()
        rows.append(logits.cpu().numpy().copy())
        nxt = int(np.argmax(rows[-1]))
        if use_device_argmax:
            assert int(d_arg.item()) == nxt, "device argmax differs from host argmax"
            d_tok.copy_(d_arg)
        taus.append(nxt)
    dec.check()
    return np.stack(rows), taus


def gpu_teacher_forced(dec, prompt, taus, n_decode: int):
    """Prefill the prompt, then decode the given tokens (not the handle's own argmax).
    Returns the logit rows [n_decode + 1, V]: the prefill's last row and each step's."""
    V = dec.w["vocab"]
    logits = torch.empty(V, dtype=torch.float32, device=dec.device)
    P = len(prompt)
    dec.prefill(prompt, 0, logits)
    dec.synchronize()
    rows = [logits.cpu().numpy().copy()]
    for i in range(n_decode):
        dec.decode(int(taus[i]), P + i, logits)
        dec.synchronize()
        rows.append(logits.cpu().numpy().copy())
    dec.check()
    return np.stack(rows)


def oracle_session(w: dict, device: str = "cuda", trace: bool = False) -> Session:
    small = w["hidden"] <= 1024
    src = synthetic.OracleWeightSource(w, device=device, cache=small)
    return Session(OracleConfig.from_dict(w), src, trace=trace)


def oracle_teacher_forced(w: dict, prompt, taus, n_decode: int, device: str = "cuda", trace: bool = False):
    """Oracle logits for the prefill row and every decode step, in one single-pass run
    over prompt + the GPU's greedy tokens (valid because prefill == per-token)."""
    s = oracle_session(w, device, trace)
    P = len(prompt)
    toks = list(prompt) + list(taus[:n_decode])
    rows = s.prefill_batched(toks, 0, logits_rows=list(range(P - 1, P + n_decode)))
    return rows, s


def compare_logits(gpu: np.ndarray, ref: np.ndarray, tol_abs: float, tol_rel: float):
    d = np.abs(gpu.astype(np.float64) - ref)
    max_abs = float(d.max())
    rel = float(np.linalg.norm(gpu.astype(np.float64) - ref) / np.linalg.norm(ref))
    assert np.isfinite(gpu).all(), "non-finite logits"
    assert max_abs <= tol_abs, f"max|d| = {max_abs:.3e} > {tol_abs:.1e} (rel rms {rel:.2e})"
    assert rel <= tol_rel, f"relative rms {rel:.3e} > {tol_rel:.1e}"
    return max_abs, rel


def check_greedy_tokens(ref_rows: np.ndarray, taus, tol_abs: float):
    """Each GPU token is the oracle's argmax, or within 2*tol of the oracle's max (near-tie)."""
    for i, t in enumerate(taus[:len(ref_rows)]):
        r = ref_rows[i]
        if int(np.argmax(r)) != t:
            assert r.max() - r[t] <= 2 * tol_abs, f"step {i}: token {t} is {r.max() - r[t]:.3e} below the max"


def ring_positions(length: int, max_seq: int, sliding: int):
    """Position held by each slot after positions 0..length-1 were written (-1: never)."""
    slots = np.full(max_seq, -1, dtype=np.int64)
    for p in range(length):
        slots[(p % max_seq) if sliding > 0 else p] = p
    return slots
