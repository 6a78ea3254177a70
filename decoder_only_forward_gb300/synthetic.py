"""Seeded synthetic inputs: workload shapes, random-init weights and prompts.

This module draws numbers and nothing else: it holds none of the forward
pass's arithmetic, so both the CUDA library's callers and the float64 oracle
can take their inputs from it.  Every tensor is drawn from its own seeded
torch generator (Philox on a GPU, the CPU generator on the host), so the same
(seed, layer, role, expert) always yields the same values on the same device.

Distributions: projection, head, embedding, router matrices and q/k/v biases
N(0, 0.02); norm weights 1 + N(0, 0.1) (kept in float32, as norm weights are
stored in f32 by the engines the pages describe); prompts uniform in [0, vocab).
"""

from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch

# Workload shapes.  ``prompt``/``decode`` are the token counts of one run,
# ``max_seq`` the KV capacity (min(sliding_window, n_ctx) under a window).
WORKLOADS = {
    "toy": dict(
        n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=172, vocab=256,
        tied=False, qkv_bias=False, rms_eps=1e-5, rope_theta=10000.0, sliding_window=0,
        n_experts=0, n_experts_used=0, dtype="f32", prompt=16, decode=16, max_seq=32),
    "smollm2-135m": dict(
        n_layers=30, hidden=576, n_heads=9, n_kv_heads=3, head_dim=64, ffn=1536, vocab=49152,
        tied=True, qkv_bias=False, rms_eps=1e-5, rope_theta=10000.0, sliding_window=0,
        n_experts=0, n_experts_used=0, dtype="bf16", prompt=512, decode=128, max_seq=640),
    "qwen2.5-0.5b": dict(
        n_layers=24, hidden=896, n_heads=14, n_kv_heads=2, head_dim=64, ffn=4864, vocab=151936,
        tied=True, qkv_bias=True, rms_eps=1e-6, rope_theta=1e6, sliding_window=0,
        n_experts=0, n_experts_used=0, dtype="bf16", prompt=2048, decode=256, max_seq=2304),
    "mistral-7b": dict(
        n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=14336, vocab=32000,
        tied=False, qkv_bias=False, rms_eps=1e-5, rope_theta=10000.0, sliding_window=4096,
        n_experts=0, n_experts_used=0, dtype="bf16", prompt=4096, decode=512, max_seq=4096),
    "mixtral-8x7b": dict(
        n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=14336, vocab=32000,
        tied=False, qkv_bias=False, rms_eps=1e-5, rope_theta=1e6, sliding_window=0,
        n_experts=8, n_experts_used=2, dtype="bf16", prompt=1024, decode=256, max_seq=1280),
}


def workload(name: str, **overrides) -> dict:
    """A copy of a named workload with fields replaced (for reduced-size parity cases)."""
    d = dict(WORKLOADS[name])
    d.update(overrides)
    d.setdefault("rope_llama3", None)
    return d


def tensor_seed(seed: int, layer: int, role: str, expert: int = -1) -> int:
    h = hashlib.blake2b(f"{seed}/{layer}/{role}/{expert}".encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & 0x7FFF_FFFF_FFFF_FFFF


def storage_dtype(cfg: dict) -> torch.dtype:
    return torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16


def role_shape(cfg: dict, role: str) -> tuple:
    h, f = cfg["hidden"], cfg["ffn"]
    qd = cfg["n_heads"] * cfg["head_dim"]
    kd = cfg["n_kv_heads"] * cfg["head_dim"]
    return {
        "tok_embd": (cfg["vocab"], h), "lm_head": (cfg["vocab"], h), "out_norm": (h,),
        "attn_norm": (h,), "ffn_norm": (h,),
        "wq": (qd, h), "wk": (kd, h), "wv": (kd, h), "bq": (qd,), "bk": (kd,), "bv": (kd,),
        "wo": (h, qd), "w_gate": (f, h), "w_up": (f, h), "w_down": (h, f),
        "router": (cfg["n_experts"], h),
        # QK-norm weights: one head_dim vector shared by the heads, or row-long ("row")
        "q_norm": (qd if cfg.get("qk_norm") == "row" else cfg["head_dim"],),
        "k_norm": (kd if cfg.get("qk_norm") == "row" else cfg["head_dim"],),
        "post_attn_norm": (h,), "post_ffn_norm": (h,),
    }[role]


_NORMS = {"out_norm", "attn_norm", "ffn_norm", "q_norm", "k_norm", "post_attn_norm", "post_ffn_norm"}
_BIASES = {"bq", "bk", "bv"}


def draw(cfg: dict, role: str, layer: int = -1, expert: int = -1, seed: int = 1234,
         device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """Draw one weight tensor in its stored dtype (norms and biases f32, matrices the config dtype).

    With ``out`` given, the values are written into that (possibly strided) view.
    """
    shape = role_shape(cfg, role)
    g = torch.Generator(device=device)
    g.manual_seed(tensor_seed(seed, layer, role, expert))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if role in _NORMS:
        t.mul_(0.1).add_(1.0)
        dt = torch.float32
    else:
        t.mul_(0.02)
        dt = torch.float32 if role in _BIASES else storage_dtype(cfg)
    t = t.to(dt)
    if out is not None:
        out.copy_(t)
        return out
    return t


def layer_roles(cfg: dict) -> list:
    roles = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm"]
    if cfg["qkv_bias"]:
        roles += ["bq", "bk", "bv"]
    if cfg.get("qk_norm"):
        roles += ["q_norm", "k_norm"]
    if cfg.get("sandwich_norms"):
        roles += ["post_attn_norm", "post_ffn_norm"]
    roles += ["router"] if cfg["n_experts"] > 0 else ["w_gate", "w_up", "w_down"]
    return roles


def prompt_tokens(cfg: dict, n: int, seed: int = 0) -> np.ndarray:
    """Prompt ids uniform in [0, vocab), from a CPU generator seeded with ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, cfg["vocab"], (n,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def _to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


@dataclass
class OracleWeightSource:
    """Hands the oracle float64 copies of freshly drawn tensors (same seeds, same device).

    Implements the oracle's weight interface (embed_rows, out_norm, lm_head,
    layer, expert).  Nothing is read back from buffers the library uses: each
    tensor is drawn again from its own generator.  ``cache=True`` keeps the
    float64 copies (for small models visited many times).
    """
    cfg: dict
    seed: int = 1234
    device: str = "cpu"
    cache: bool = False

    def __post_init__(self):
        self._memo = {}

    def _get(self, role, layer=-1, expert=-1):
        key = (role, layer, expert)
        if key in self._memo:
            return self._memo[key]
        a = _to_f64(draw(self.cfg, role, layer, expert, self.seed, self.device))
        if self.cache:
            self._memo[key] = a
        return a

    def embed_rows(self, tokens) -> np.ndarray:
        e = self._embedding()
        return np.array(e[np.asarray(tokens, np.int64)], copy=True)

    def _embedding(self) -> np.ndarray:
        # Used for every embed and, when tied, as the head: always kept.
        if ("tok_embd", -1, -1) not in self._memo:
            self._memo[("tok_embd", -1, -1)] = _to_f64(
                draw(self.cfg, "tok_embd", -1, -1, self.seed, self.device))
        return self._memo[("tok_embd", -1, -1)]

    def out_norm(self) -> np.ndarray:
        return self._get("out_norm")

    def lm_head(self) -> np.ndarray:
        return self._embedding() if self.cfg["tied"] else self._get("lm_head")

    def layer(self, l: int) -> dict:
        return {r: self._get(r, l) for r in layer_roles(self.cfg)}

    def expert(self, l: int, e: int):
        return tuple(self._get(r, l, e) for r in ("w_gate", "w_up", "w_down"))
