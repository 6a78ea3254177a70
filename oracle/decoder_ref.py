"""Plain float64 definition of the decoder-only forward pass over a KV cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): the CUDA library never
imports, links or runs anything here.

What it computes, and where the pages define it (page title, section):

  [SIP]  "Transformer forward pass" (sipllm docs): Design / One block loop,
         Shared attention, RoPE is adjacent-pair, Single-pass prefill.
  [PAN]  "Llama Forward Pass" (Pantheon, docs/architecture/llama-forward.md):
         Forward Pass Flow; Key Operations: RMSNorm, RoPE, Grouped Query
         Attention, SwiGLU FFN, Sliding Window (Mistral), Mixture of Experts.
  [RML]  "The decoder" (rml): One forward pass, Attend, Rotary embeddings,
         Mixture of experts.
  [ZLLM] "The Algorithm Layer: From Attention and KV Cache to FFN and MoE":
         §2 Attention (the softmax(QK^T/sqrt(d_k)+mask)V definition), §4 FFN.

Per position p (absolute), per layer, pre-norm:
  n = x / sqrt(mean(x^2) + eps) * w_attn                      [PAN RMSNorm]
  q = Wq n (+bq), k = Wk n (+bk), v = Wv n (+bv)              [PAN Forward Pass Flow]
  q, k rotated pairwise on dims (2i, 2i+1) by p * theta^(-2i/hd),
       optionally with llama3 frequency scaling            [SIP RoPE; RML Rotary embeddings]
  (k, v) appended to a per-layer list indexed by absolute position
  o_h = softmax_j(q_h . K_j / sqrt(hd)) V_j over j in [lo, p],
       kv head of h = floor(h * n_kv / n_head),
       lo = 0, or p - W + 1 under a sliding window W       [PAN GQA, Sliding Window; RML Attend]
  x += Wo concat(o)
  n = rmsnorm(x, w_ffn)
  dense: x += Wd (silu(Wg n) * (Wu n))                        [PAN SwiGLU FFN]
  MoE:   P = softmax(Wr n); top-k by repeated selection (ties -> lower id);
         w_e = P_e / sum_sel P; x += sum_{e in selection order} w_e Wd_e(silu(Wg_e n) * (Wu_e n))
                                                              [PAN Mixture of Experts; RML Mixture of experts]
  logits = W_out rmsnorm(x, w_out)                             [PAN Forward Pass Flow]

Per-layer RoPE base (SIP RoPE, "per-layer base (Gemma 3)"; RML One forward pass
step 3 computes a global and a local table): with rope_theta_local set, layer l
rotates with rope_theta when it is one of every rope_global_every layers
((l + 1) % rope_global_every == 0) and with rope_theta_local otherwise; llama3
scaling, when on, applies to the global base only.

Optional norms (RML "The decoder", One forward pass, steps 4 and 6; SIP
Tradeoffs, optional weight roles):
  QK-norm: after the biases and before RoPE, q and k are RMS-normalised per
    head with a head_dim weight shared by the heads ("head"), or over the whole
    q / k row with a row-long weight ("row"), with the model's eps.
  Sandwich norms: each block's output (attention after Wo, FFN after down /
    the expert sum) is RMS-normalised with its post norm weight before it is
    added to the residual.

Optional 8-bit projection weights (PAN "Llama Forward Pass", weight modes: the
projection matrices Wq, Wk, Wv, Wo, W_gate, W_up, W_down and an untied W_output
stay quantised, expanded a block at a time; embeddings and norms stay f32): each
weight row is stored in groups of 32 input columns by the same rule the pages
print for the int8 cache, round(w / s) with s = max|w| / 127 in float32, and the
forward pass uses float32(code * s).  The router stays unquantised (not listed).

Optional int8 K/V cache (RML "The decoder", KV cache): every cached key and
value row is stored as groups of G channels (G the largest power of two that
divides head_dim, at most 32, so a group never spans two heads), each group as
round(x / s) with one float32 scale s = max|x| / 127; attention reads the
stored values back as code * s, the current position's included.

Readings taken where the pages are silent, garbled or disagree (each is listed
in the design notes as well):
  * RoPE pairs: pair i is dims (2i, 2i+1) with inv_freq_i = theta^(-2i/hd)
    (RML Rotary embeddings; SIP RoPE).  PAN's pseudo-code "(i, i+1) ...
    theta^(2i/hd)" is read the same way.  Rotation is counter-clockwise:
    (a, b) -> (a cos - b sin, a sin + b cos).
  * Sliding window W covers W positions including the query itself
    (RML Attend: "pos - window + 1"; PAN: readable min(pos+1, max_seq)).
  * Qwen2-style bias on q, k, v only (RML model config), not on the output.
  * Expert weights are always renormalised (every workload here does).
  * Argmax and top-k ties go to the lower index.
  * int8 K/V: the quantisation decision is taken in float32 (the precision a
    kernel holds K/V in): x rounded to float32, s = max|x| / 127 and x / s
    each one float32 operation, "round" = half away from zero (C round),
    codes clamped to [-127, 127], read back as float32(code * s).  An all-zero
    group stores s = 0 and codes 0.

Two execution orders are provided: ``Session.prefill`` (row-wise: layer-outer,
position-inner, one matrix-vector product per row, the single-pass prefill of
SIP) and ``Session.forward`` (one position through every layer).  Both call
the same per-row block, so they agree bit for bit.  ``Session.prefill_batched``
applies the same definition with matrix products over all rows; it agrees with
the row-wise order to rounding.

Parity pins (tests/test_oracle_*.py): closed forms for RMSNorm, SiLU, RoPE at
p=0, one-key and equal-key attention, GQA head maps; RoPE invariants (norm,
composition, relative position); the llama3 worked example of RML Rotary
embeddings; top-k tie rule, weights summing to one, k=E equals the dense
mixture; brute-force equality with torch's float64 library routines
(scaled_dot_product_attention with a causal/window mask and GQA, rms_norm,
complex-multiplication RoPE); prefill == per-token bit-exact; zero-weight
models that reduce to closed forms.  No page prints a numeric golden for a
whole model, so whole-model logits are pinned only through those parts.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------
# Configuration
# --------------------------------------------------------------------------

@dataclass
class OracleConfig:
    """Sizes and switches of one decoder (RML "The model config": one recipe plus switches)."""

    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_experts: int = 0
    n_experts_used: int = 0
    sliding_window: int = 0
    qkv_bias: bool = False
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    # llama3 scaling: dict(factor=, low_freq_factor=, high_freq_factor=, orig_ctx=) or None
    rope_llama3: Optional[dict] = None
    # Which dimensions pair (RML Rotary embeddings, "Which dimensions pair"): False =
    # adjacent (2i, 2i+1) (kInterleaved), True = (i, i + rope_dim/2) (kHalf, rotate_half).
    rope_half: bool = False
    # Rotary width (SIP partial-rotary rope_rot): only the first rope_dim dims of a head
    # turn, the rest pass through; 0 means head_dim.
    rope_dim: int = 0
    # int8 K/V cache with per-group float32 scales (RML "The decoder", KV cache).
    kv_int8: bool = False
    # QK-norm (RML One forward pass step 4): "" off, "head" per head (weights [hd]),
    # "row" over the whole q / k row (weights [nq*hd] / [nkv*hd]).
    qk_norm: str = ""
    # Sandwich norms (RML One forward pass step 6): post-attention / post-FFN RMSNorm of
    # each block's output before the residual add (weights post_attn_norm, post_ffn_norm).
    sandwich_norms: bool = False
    # 8-bit projection weights (PAN weight modes; groups of 32 input columns, see module notes).
    weight_int8: bool = False
    # Per-layer RoPE base (SIP RoPE, Gemma 3): 0 = one base for every layer; else local
    # layers use rope_theta_local and every rope_global_every-th layer the global base.
    rope_theta_local: float = 0.0
    rope_global_every: int = 0

    def layer_is_global(self, l: int) -> bool:
        """Whether layer l rotates with the global base (always, without a local base)."""
        if not self.rope_theta_local:
            return True
        return self.rope_global_every > 0 and (l + 1) % self.rope_global_every == 0

    @property
    def rotary_dim(self) -> int:
        return self.rope_dim if self.rope_dim else self.head_dim

    @classmethod
    def from_dict(cls, d: dict) -> "OracleConfig":
        names = cls.__dataclass_fields__.keys()
        return cls(**{k: d[k] for k in names if k in d})

    @property
    def is_moe(self) -> bool:
        return self.n_experts > 0


# --------------------------------------------------------------------------
# Elementary operations
# --------------------------------------------------------------------------

def rmsnorm(x, w, eps: float) -> np.ndarray:
    """rms = sqrt(mean(x^2) + eps); out = x / rms * w  (PAN Key Operations, RMSNorm).

    Works on the last axis; ``x`` may be one row or a stack of rows.
    """
    x = np.asarray(x, F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, F64)


def llama3_scale_inv_freq(inv_freq, factor: float, low_freq_factor: float,
                          high_freq_factor: float, orig_ctx: float) -> np.ndarray:
    """llama3 wavelength stretch (SIP RoPE variants; RML Rotary embeddings, worked example).

    With wavelength wl = 2*pi/inv: wl below orig/high keeps its frequency, wl
    above orig/low is slowed by ``factor``, and in between the two are blended
    with smooth = (orig/wl - low) / (high - low):
    inv' = (1 - smooth) * inv / factor + smooth * inv.
    """
    inv = np.asarray(inv_freq, F64)
    out = np.empty_like(inv)
    for i, f in enumerate(inv):
        wl = 2.0 * math.pi / f
        if wl < orig_ctx / high_freq_factor:
            out[i] = f
        elif wl > orig_ctx / low_freq_factor:
            out[i] = f / factor
        else:
            smooth = (orig_ctx / wl - low_freq_factor) / (high_freq_factor - low_freq_factor)
            out[i] = (1.0 - smooth) * f / factor + smooth * f
    return out


def rope_inv_freq(head_dim: int, theta: float, llama3: Optional[dict] = None, rope_dim: int = 0) -> np.ndarray:
    """inv_freq[i] = theta^(-2i/d) for pair i in [0, d/2), d the rotary width (RML Rotary
    embeddings; with partial rotary, SIP rope_rot, d = rope_dim)."""
    d = rope_dim if rope_dim else head_dim
    i = np.arange(d // 2, dtype=F64)
    inv = np.power(F64(theta), -2.0 * i / d)
    if llama3:
        inv = llama3_scale_inv_freq(inv, **llama3)
    return inv


def rope_pairs(head_dim: int, half: bool = False, rope_dim: int = 0):
    """Index arrays (a, b) of the rotated pairs of one head: pair i is (a[i], b[i]).

    Adjacent style (SIP "RoPE is adjacent-pair"; kInterleaved): (2i, 2i+1).  Half
    style (RML "Which dimensions pair"; kHalf): (i, i + d/2).  d = rope_dim or
    head_dim; dims >= d are not rotated (SIP partial-rotary).
    """
    d = rope_dim if rope_dim else head_dim
    i = np.arange(d // 2)
    return (i, i + d // 2) if half else (2 * i, 2 * i + 1)


def rope_rotate(vec, pos: int, inv_freq, half: bool = False, rope_dim: int = 0) -> np.ndarray:
    """Rotate each pair (v[a_i], v[b_i]) by angle pos*inv_freq[i]:
    (a, b) -> (a cos - b sin, a sin + b cos).

    ``vec`` is [..., head_dim]; each head is rotated independently.
    """
    v = np.array(vec, dtype=F64, copy=True)
    ia, ib = rope_pairs(v.shape[-1], half, rope_dim)
    ang = F64(pos) * np.asarray(inv_freq, F64)
    c, s = np.cos(ang), np.sin(ang)
    a = v[..., ia].copy()
    b = v[..., ib].copy()
    v[..., ia] = a * c - b * s
    v[..., ib] = a * s + b * c
    return v


# --------------------------------------------------------------------------
# int8 K/V cache (RML "The decoder", KV cache)
# --------------------------------------------------------------------------

def kv_group_size(head_dim: int) -> int:
    """Channels per int8 scale group: the largest power of two dividing head_dim, at most 32."""
    g = 1
    while g < 32 and head_dim % (2 * g) == 0:
        g *= 2
    return g


def round_half_away(x) -> np.ndarray:
    """C round(): to the nearest integer, halves away from zero."""
    x = np.asarray(x, F64)
    return np.sign(x) * np.floor(np.abs(x) + 0.5)


def quantize_int8_groups(row, group: int):
    """One cached row -> (codes int8 [n], scales float32 [n / group]).

    Each group of ``group`` channels becomes round(x / s) with s = max|x| / 127,
    the arithmetic in float32 (see the module notes); an all-zero group keeps
    s = 0 and codes 0.
    """
    x = np.asarray(row, F64).astype(np.float32).reshape(-1, group)
    m = np.abs(x).max(axis=1)
    s = (m / np.float32(127.0)).astype(np.float32)
    codes = np.zeros(x.shape, np.int8)
    nz = s > 0
    if nz.any():
        qf = (x[nz] / s[nz, None]).astype(np.float32)
        codes[nz] = np.clip(round_half_away(qf), -127, 127).astype(np.int8)
    return codes.reshape(-1), s


def dequantize_int8_groups(codes, scales, group: int) -> np.ndarray:
    """Stored row read back: float32(code * s), as float64."""
    c = np.asarray(codes, np.int8).astype(np.float32).reshape(-1, group)
    s = np.asarray(scales, np.float32)
    return (c * s[:, None]).astype(np.float32).astype(F64).reshape(-1)


def kv_int8_roundtrip(row, head_dim: int) -> np.ndarray:
    """The value an int8 cache gives back for a row of K or V (any shape, heads of head_dim)."""
    a = np.asarray(row, F64)
    g = kv_group_size(head_dim)
    codes, scales = quantize_int8_groups(a.reshape(-1), g)
    return dequantize_int8_groups(codes, scales, g).reshape(a.shape)


def qk_normalise(vec, weight, heads: int, mode: str, eps: float) -> np.ndarray:
    """QK-norm of q or k rows (last axis heads * hd): RMSNorm of each head with the
    shared [hd] weight ("head"), or of the whole row with a row-long weight ("row")."""
    v = np.asarray(vec, F64)
    if mode == "head":
        return rmsnorm(v.reshape(*v.shape[:-1], heads, v.shape[-1] // heads), weight, eps).reshape(v.shape)
    if mode == "row":
        return rmsnorm(v, weight, eps)
    raise ValueError(f"unknown qk_norm mode {mode!r}")


def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """Query head h reads kv head h * n_kv_head / n_head (PAN Grouped Query Attention)."""
    return (h * n_kv_heads) // n_heads


def window_start(pos: int, sliding_window: int) -> int:
    """First readable position: 0, or pos - window + 1 (RML Attend; PAN Sliding Window)."""
    if sliding_window <= 0:
        return 0
    return max(0, pos - sliding_window + 1)


def attend_ref(q, keys, values, n_heads: int, n_kv_heads: int) -> np.ndarray:
    """Brute-force attention of one query position (ZLLM §2; RML AttendRef).

    q: [n_heads, hd]; keys, values: [m, n_kv_heads, hd], the readable positions
    in order.  Every score is formed, softmaxed, and used for a weighted sum.
    """
    q = np.asarray(q, F64)
    keys = np.asarray(keys, F64)
    values = np.asarray(values, F64)
    hd = q.shape[-1]
    out = np.empty((n_heads, hd), F64)
    scale = 1.0 / math.sqrt(hd)
    for h in range(n_heads):
        g = kv_head_of(h, n_heads, n_kv_heads)
        s = (keys[:, g, :] @ q[h]) * scale
        e = np.exp(s - s.max())
        p = e / e.sum()
        out[h] = p @ values[:, g, :]
    return out


def silu(z) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, F64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(n, w_gate, w_up, w_down) -> np.ndarray:
    """W_down (silu(W_gate n) * (W_up n)) (PAN SwiGLU FFN; ZLLM §4)."""
    n = np.asarray(n, F64)
    return np.asarray(w_down, F64) @ (silu(np.asarray(w_gate, F64) @ n) * (np.asarray(w_up, F64) @ n))


def route_topk(router_logits, k: int):
    """Router softmax over all experts, top-k by repeated selection, renormalise.

    (PAN Mixture of Experts; RML Mixture of experts steps 1-3.)  Ties go to
    the lower expert id.  Returns (ids in selection order, weights, probs).
    """
    r = np.asarray(router_logits, F64)
    e = np.exp(r - r.max())
    p = e / e.sum()
    taken = np.zeros(len(p), dtype=bool)
    ids = []
    for _ in range(k):
        best = -1
        for j in range(len(p)):
            if taken[j]:
                continue
            if best < 0 or p[j] > p[best]:   # strict: an equal later id never displaces
                best = j
        taken[best] = True
        ids.append(best)
    total = F64(0.0)
    for j in ids:
        total += p[j]
    weights = np.array([p[j] / total for j in ids], F64)
    return ids, weights, p


def moe_ffn(n, router, expert: Callable[[int], tuple], k: int):
    """Weighted sum of the selected experts' SwiGLU outputs (PAN Mixture of Experts).

    ``expert(e)`` returns (W_gate_e, W_up_e, W_down_e).  Returns
    (ffn_out, ids, weights, router_logits).
    """
    n = np.asarray(n, F64)
    logits = np.asarray(router, F64) @ n
    ids, weights, _ = route_topk(logits, k)
    out = np.zeros(np.asarray(expert(ids[0])[2]).shape[0], F64)
    for e, w in zip(ids, weights):
        out += w * swiglu(n, *expert(e))
    return out, ids, weights, logits


# --------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------

class DictWeights:
    """In-memory weights, held as given and widened to float64 on use.

    Layer dicts carry: attn_norm, wq, wk, wv, (bq, bk, bv), wo, ffn_norm and
    either w_gate, w_up, w_down (dense) or router plus ``experts[l][e] =
    (w_gate, w_up, w_down)``.  ``lm_head=None`` means a tied head: the
    embedding matrix is reused (RML model config).
    """

    def __init__(self, tok_embd, out_norm, layers, lm_head=None, experts=None):
        self._embd = tok_embd
        self._out_norm = out_norm
        self._layers = layers
        self._lm_head = lm_head
        self._experts = experts

    def embed_rows(self, tokens) -> np.ndarray:
        return np.asarray(self._embd, F64)[np.asarray(tokens, np.int64)]

    def out_norm(self) -> np.ndarray:
        return np.asarray(self._out_norm, F64)

    def lm_head(self) -> np.ndarray:
        return np.asarray(self._embd if self._lm_head is None else self._lm_head, F64)

    def layer(self, l: int) -> dict:
        return {k: (None if v is None else np.asarray(v, F64)) for k, v in self._layers[l].items()}

    def expert(self, l: int, e: int):
        return tuple(np.asarray(t, F64) for t in self._experts[l][e])


# --------------------------------------------------------------------------
# Forward pass with a KV cache
# --------------------------------------------------------------------------

@dataclass
class Trace:
    """Optional per-(layer, position) record for layer-by-layer comparison (ZLLM §6 item 3)."""
    router_logits: dict = field(default_factory=dict)   # (l, pos) -> [E]
    expert_ids: dict = field(default_factory=dict)      # (l, pos) -> [k]
    expert_weights: dict = field(default_factory=dict)  # (l, pos) -> [k]
    hidden: dict = field(default_factory=dict)          # (l, pos) -> [h], after layer l


WEIGHT_GROUP = 32   # input columns per scale of an 8-bit weight row
_PROJECTIONS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def weight_int8_roundtrip(mat) -> np.ndarray:
    """A weight matrix [out, in] as its 8-bit storage gives it back: each row in groups of
    WEIGHT_GROUP input columns (in must be a multiple of it)."""
    m = np.asarray(mat, F64)
    if m.shape[-1] % WEIGHT_GROUP:
        raise ValueError(f"input width {m.shape[-1]} is not a multiple of {WEIGHT_GROUP}")
    out = np.empty_like(m)
    for r in range(m.shape[0]):
        codes, scales = quantize_int8_groups(m[r], WEIGHT_GROUP)
        out[r] = dequantize_int8_groups(codes, scales, WEIGHT_GROUP)
    return out


def _is_tied(weights) -> bool:
    """Whether a weight source's head is its embedding (same array, or the source says so)."""
    cfg = getattr(weights, "cfg", None)
    if isinstance(cfg, dict) and "tied" in cfg:
        return bool(cfg["tied"])
    return getattr(weights, "_lm_head", None) is None and hasattr(weights, "_embd")


class Int8ProjectionWeights:
    """A weight source whose projection matrices (and untied LM head) read back through
    8-bit storage; embeddings, norms, biases and the router pass through unchanged."""

    def __init__(self, inner, tied: bool):
        self.inner = inner
        self.tied = tied
        self._memo = {}

    def embed_rows(self, tokens):
        return self.inner.embed_rows(tokens)

    def out_norm(self):
        return self.inner.out_norm()

    def lm_head(self):
        if self.tied:
            return self.inner.lm_head()
        if "head" not in self._memo:
            self._memo["head"] = weight_int8_roundtrip(self.inner.lm_head())
        return self._memo["head"]

    def layer(self, l: int) -> dict:
        key = ("layer", l)
        if key not in self._memo:
            lw = dict(self.inner.layer(l))
            for r in _PROJECTIONS:
                if lw.get(r) is not None:
                    lw[r] = weight_int8_roundtrip(lw[r])
            self._memo[key] = lw
        return self._memo[key]

    def expert(self, l: int, e: int):
        key = ("expert", l, e)
        if key not in self._memo:
            self._memo[key] = tuple(weight_int8_roundtrip(m) for m in self.inner.expert(l, e))
        return self._memo[key]


class Session:
    """One sequence: a per-layer K/V list indexed by absolute position, plus the forward pass.

    The list is deliberately not a ring buffer: any circular storage in an
    implementation under test is checked against this plain record.
    """

    def __init__(self, cfg: OracleConfig, weights, trace: bool = False, trace_hidden: bool = False):
        self.cfg = cfg
        self.w = Int8ProjectionWeights(weights, getattr(weights, "tied", False) or
                                       _is_tied(weights)) if cfg.weight_int8 else weights
        self.inv_freq = rope_inv_freq(cfg.head_dim, cfg.rope_theta, cfg.rope_llama3, cfg.rope_dim)
        self.inv_freq_local = (rope_inv_freq(cfg.head_dim, cfg.rope_theta_local, None, cfg.rope_dim)
                               if cfg.rope_theta_local else self.inv_freq)
        self.keys = [[] for _ in range(cfg.n_layers)]
        self.values = [[] for _ in range(cfg.n_layers)]
        self.trace = Trace() if trace else None
        self.trace_hidden = trace_hidden

    # -- cache bookkeeping -------------------------------------------------
    @property
    def length(self) -> int:
        return len(self.keys[0]) if self.cfg.n_layers else 0

    def reset(self) -> None:
        for l in range(self.cfg.n_layers):
            self.keys[l].clear()
            self.values[l].clear()

    def _truncate(self, start_pos: int) -> None:
        """Appending at start_pos < length drops the later history (a rewind)."""
        if start_pos < 0 or start_pos > self.length:
            raise ValueError(f"start_pos {start_pos} outside [0, {self.length}]")
        for l in range(self.cfg.n_layers):
            del self.keys[l][start_pos:]
            del self.values[l][start_pos:]

    # -- one row through one layer ----------------------------------------
    def _attention_row(self, l: int, lw: dict, x: np.ndarray, pos: int) -> np.ndarray:
        c = self.cfg
        nq, nkv, hd = c.n_heads, c.n_kv_heads, c.head_dim
        n = rmsnorm(x, lw["attn_norm"], c.rms_eps)
        q = lw["wq"] @ n
        k = lw["wk"] @ n
        v = lw["wv"] @ n
        if c.qkv_bias:
            q = q + lw["bq"]
            k = k + lw["bk"]
            v = v + lw["bv"]
        if c.qk_norm:
            q = qk_normalise(q, lw["q_norm"], nq, c.qk_norm, c.rms_eps)
            k = qk_normalise(k, lw["k_norm"], nkv, c.qk_norm, c.rms_eps)
        inv = self.inv_freq if c.layer_is_global(l) else self.inv_freq_local
        q = rope_rotate(q.reshape(nq, hd), pos, inv, c.rope_half, c.rope_dim)
        k = rope_rotate(k.reshape(nkv, hd), pos, inv, c.rope_half, c.rope_dim)
        if len(self.keys[l]) != pos:
            raise AssertionError("positions must be appended in ascending order")
        v = v.reshape(nkv, hd)
        if c.kv_int8:
            k, v = kv_int8_roundtrip(k, hd), kv_int8_roundtrip(v, hd)
        self.keys[l].append(k)
        self.values[l].append(v)
        lo = window_start(pos, c.sliding_window)
        o = attend_ref(q, np.stack(self.keys[l][lo:pos + 1]),
                       np.stack(self.values[l][lo:pos + 1]), nq, nkv)
        out = lw["wo"] @ o.reshape(-1)
        if c.sandwich_norms:
            out = rmsnorm(out, lw["post_attn_norm"], c.rms_eps)
        return x + out

    def _ffn_row(self, l: int, lw: dict, x: np.ndarray, pos: int) -> np.ndarray:
        c = self.cfg
        n = rmsnorm(x, lw["ffn_norm"], c.rms_eps)
        if c.is_moe:
            out, ids, wts, logits = moe_ffn(n, lw["router"], lambda e: self.w.expert(l, e),
                                            c.n_experts_used)
            if self.trace is not None:
                self.trace.router_logits[(l, pos)] = logits
                self.trace.expert_ids[(l, pos)] = list(ids)
                self.trace.expert_weights[(l, pos)] = wts
        else:
            out = swiglu(n, lw["w_gate"], lw["w_up"], lw["w_down"])
        if c.sandwich_norms:
            out = rmsnorm(out, lw["post_ffn_norm"], c.rms_eps)
        return x + out

    def _block_row(self, l: int, lw: dict, x: np.ndarray, pos: int) -> np.ndarray:
        y = self._ffn_row(l, lw, self._attention_row(l, lw, x, pos), pos)
        if self.trace is not None and self.trace_hidden:
            self.trace.hidden[(l, pos)] = y.copy()
        return y

    def _logits_rows(self, X: np.ndarray) -> np.ndarray:
        """Final norm and head, one matrix-vector product per row (row-independent)."""
        head = self.w.lm_head()
        wn = self.w.out_norm()
        return np.stack([head @ rmsnorm(x, wn, self.cfg.rms_eps) for x in X])

    # -- drivers -------------------------------------------------------------
    def forward(self, token: int, pos: int) -> np.ndarray:
        """One position through every layer, returning its logits (SIP Transformer::forward)."""
        self._truncate(pos)
        x = self.w.embed_rows([token])[0]
        for l in range(self.cfg.n_layers):
            x = self._block_row(l, self.w.layer(l), x, pos)
        return self._logits_rows(x[None, :])[0]

    def prefill(self, tokens, start_pos: int, all_logits: bool = False) -> np.ndarray:
        """Single-pass prefill: each layer once, positions ascending (SIP Single-pass prefill).

        Returns the last row's logits, or every row's with ``all_logits``.
        """
        tokens = list(tokens)
        if not tokens:
            raise ValueError("empty input")
        self._truncate(start_pos)
        X = self.w.embed_rows(tokens)
        for l in range(self.cfg.n_layers):
            lw = self.w.layer(l)
            for t in range(len(tokens)):
                X[t] = self._block_row(l, lw, X[t], start_pos + t)
        rows = X if all_logits else X[-1:]
        out = self._logits_rows(rows)
        return out if all_logits else out[0]

    def prefill_batched(self, tokens, start_pos: int, logits_rows=None) -> np.ndarray:
        """The same definition with matrix products over all rows of a layer.

        ``logits_rows``: indices (into ``tokens``) whose logits are returned;
        default the last row.  Experts are visited one at a time, so a caller
        may stream their weights.
        """
        c = self.cfg
        tokens = list(tokens)
        n = len(tokens)
        if n == 0:
            raise ValueError("empty input")
        self._truncate(start_pos)
        nq, nkv, hd = c.n_heads, c.n_kv_heads, c.head_dim
        pos = start_pos + np.arange(n)
        X = self.w.embed_rows(tokens)
        tables = {}
        for name, inv in (("global", self.inv_freq), ("local", self.inv_freq_local)):
            ang = pos[:, None].astype(F64) * inv[None, :]
            tables[name] = (np.cos(ang), np.sin(ang))

        ia, ib = rope_pairs(hd, c.rope_half, c.rope_dim)

        def rot(T, l):  # T [n, heads, hd]; row t at position pos[t]; layer l's base
            cos, sin = tables["global" if c.layer_is_global(l) else "local"]
            a = T[..., ia].copy()
            b = T[..., ib].copy()
            out = T.copy()
            out[..., ia] = a * cos[:, None, :] - b * sin[:, None, :]
            out[..., ib] = a * sin[:, None, :] + b * cos[:, None, :]
            return out

        scale = 1.0 / math.sqrt(hd)
        for l in range(c.n_layers):
            lw = self.w.layer(l)
            N = rmsnorm(X, lw["attn_norm"], c.rms_eps)
            Q = N @ lw["wq"].T
            K = N @ lw["wk"].T
            V = N @ lw["wv"].T
            if c.qkv_bias:
                Q = Q + lw["bq"]
                K = K + lw["bk"]
                V = V + lw["bv"]
            if c.qk_norm:
                Q = qk_normalise(Q, lw["q_norm"], nq, c.qk_norm, c.rms_eps)
                K = qk_normalise(K, lw["k_norm"], nkv, c.qk_norm, c.rms_eps)
            Q = rot(Q.reshape(n, nq, hd), l)
            K = rot(K.reshape(n, nkv, hd), l)
            V = V.reshape(n, nkv, hd)
            for t in range(n):
                if c.kv_int8:
                    K[t], V[t] = kv_int8_roundtrip(K[t], hd), kv_int8_roundtrip(V[t], hd)
                self.keys[l].append(K[t])
                self.values[l].append(V[t])
            Kall = np.stack(self.keys[l])
            Vall = np.stack(self.values[l])
            j = np.arange(Kall.shape[0])
            lo = np.array([window_start(int(p), c.sliding_window) for p in pos])
            mask = (j[None, :] > pos[:, None]) | (j[None, :] < lo[:, None])
            O = np.empty((n, nq, hd), F64)
            for h in range(nq):
                g = kv_head_of(h, nq, nkv)
                S = (Q[:, h, :] @ Kall[:, g, :].T) * scale
                S[mask] = -np.inf
                E = np.exp(S - S.max(axis=1, keepdims=True))
                O[:, h, :] = (E / E.sum(axis=1, keepdims=True)) @ Vall[:, g, :]
            A = O.reshape(n, nq * hd) @ lw["wo"].T
            X = X + (rmsnorm(A, lw["post_attn_norm"], c.rms_eps) if c.sandwich_norms else A)
            N2 = rmsnorm(X, lw["ffn_norm"], c.rms_eps)
            if c.is_moe:
                R = N2 @ lw["router"].T
                routes = [route_topk(R[t], c.n_experts_used) for t in range(n)]
                outs = np.zeros((n, c.n_experts_used, c.hidden), F64)
                for e in range(c.n_experts):
                    sel = [(t, s) for t in range(n) for s, ee in enumerate(routes[t][0]) if ee == e]
                    if not sel:
                        continue
                    wg, wu, wd = self.w.expert(l, e)
                    rows = np.array([t for t, _ in sel])
                    Y = (silu(N2[rows] @ wg.T) * (N2[rows] @ wu.T)) @ wd.T
                    for i, (t, s) in enumerate(sel):
                        outs[t, s] = Y[i]
                F = np.zeros((n, c.hidden), F64)
                for s in range(c.n_experts_used):
                    F += np.array([routes[t][1][s] for t in range(n)])[:, None] * outs[:, s]
                X = X + (rmsnorm(F, lw["post_ffn_norm"], c.rms_eps) if c.sandwich_norms else F)
                if self.trace is not None:
                    for t in range(n):
                        p = int(pos[t])
                        self.trace.router_logits[(l, p)] = R[t]
                        self.trace.expert_ids[(l, p)] = list(routes[t][0])
                        self.trace.expert_weights[(l, p)] = routes[t][1]
            else:
                F = (silu(N2 @ lw["w_gate"].T) * (N2 @ lw["w_up"].T)) @ lw["w_down"].T
                X = X + (rmsnorm(F, lw["post_ffn_norm"], c.rms_eps) if c.sandwich_norms else F)
            if self.trace is not None and self.trace_hidden:
                for t in range(n):
                    self.trace.hidden[(l, int(pos[t]))] = X[t].copy()
        if logits_rows is None:
            logits_rows = [n - 1]
        rows = X[np.asarray(logits_rows, np.int64)]
        return rmsnorm(rows, self.w.out_norm(), c.rms_eps) @ self.w.lm_head().T


def greedy_argmax(logits) -> int:
    """Greedy choice; ties go to the lower token id (np.argmax returns the first maximum)."""
    return int(np.argmax(np.asarray(logits)))
