"""ctypes binding of libdec.so (declared in include/dec.h): argument marshalling only.

Every step of the forward pass runs in the library's CUDA kernels; this module
moves pointers and sizes across the C ABI and owns the torch tensors (device
memory, streams) the library is given.  Importing it raises if the library has
not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import synthetic

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdec.so")

DEC_OK, DEC_EINVAL, DEC_ERANGE, DEC_ECUDA, DEC_ETIMEOUT, DEC_ENOMEM = range(6)
DEC_F32, DEC_BF16, DEC_I8 = 0, 1, 2
KV_DTYPES = {"f32": DEC_F32, "bf16": DEC_BF16, "i8": DEC_I8}
DEC_FUSED_OFF, DEC_FUSED_GRID, DEC_FUSED_CLUSTER = 0, 1, 2
FUSED_MODES = {"off": DEC_FUSED_OFF, "grid": DEC_FUSED_GRID, "cluster": DEC_FUSED_CLUSTER}
STATUS_NAMES = {0: "DEC_OK", 1: "DEC_EINVAL", 2: "DEC_ERANGE", 3: "DEC_ECUDA", 4: "DEC_ETIMEOUT", 5: "DEC_ENOMEM"}

EXPORTED = ["dec_config_validate", "dec_workspace_bytes", "dec_create", "dec_prefill", "dec_decode",
            "dec_decode_dev", "dec_kv_reset", "dec_length", "dec_kv_layer", "dec_set_trace",
            "dec_check", "dec_timing_enable", "dec_timing_read", "dec_launch_count", "dec_destroy",
            "dec_last_error", "dec_attend_scratch_bytes", "dec_attend", "dec_attend_noalloc", "dec_gemm_bf16", "dec_set_graph", "dec_set_fused", "dec_fused_available", "dec_fused_mode", "dec_ffn_fused", "dec_phase_stamps",
            "dec_prefill_seq", "dec_kv_reset_seq", "dec_length_seq", "dec_decode_batch", "dec_kv_layer_seq",
            "dec_kv_quantize_int8", "dec_kv_slot", "dec_pages_free", "dec_selftest_wait_timeout",
            "dec_weight_quantize_int8"]
DEC_SITE_SELFTEST = 901

KERNEL_CLASSES = {"qkv": 1, "attn": 2, "oproj": 3, "gateup": 4, "down": 5, "lmhead": 6, "router": 7,
                  "pf_gemm": 8, "pf_attn": 9, "step": 10}


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "n_experts",
        "n_experts_used", "max_seq", "sliding_window", "max_tokens", "tied_embedding", "qkv_bias",
        "weight_dtype", "kv_dtype")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("rope_llama3", ctypes.c_int32),
        ("rope_factor", ctypes.c_float), ("rope_low_freq_factor", ctypes.c_float),
        ("rope_high_freq_factor", ctypes.c_float), ("rope_orig_ctx", ctypes.c_int32),
        ("rope_half", ctypes.c_int32), ("rope_dim", ctypes.c_int32), ("n_seqs", ctypes.c_int32),
        ("qk_norm", ctypes.c_int32), ("sandwich_norms", ctypes.c_int32),
        ("rope_theta_local", ctypes.c_float), ("rope_global_every", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("weight_quant", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wqkv", "bqkv", "wo", "ffn_norm", "w_gateup", "w_down", "router",
                 "q_norm", "k_norm", "post_attn_norm", "post_ffn_norm")]


class Weights(ctypes.Structure):
    _fields_ = [("tok_embd", ctypes.c_void_p), ("out_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights))]


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with decoder_only_forward_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "dec_config_validate": (I32, [ctypes.POINTER(Config), ctypes.c_char_p, SZ]),
        "dec_workspace_bytes": (SZ, [ctypes.POINTER(Config)]),
        "dec_create": (I32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), P, SZ, P, ctypes.POINTER(P)]),
        "dec_prefill": (I32, [P, ctypes.POINTER(I32), I32, I32, P, P]),
        "dec_launch_count": (ctypes.c_int64, [P]),
        "dec_decode": (I32, [P, I32, I32, P]),
        "dec_decode_dev": (I32, [P, P, I32, P, P]),
        "dec_kv_reset": (I32, [P]),
        "dec_length": (I32, [P]),
        "dec_kv_layer": (I32, [P, I32, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "dec_set_trace": (I32, [P, P, P, I32]),
        "dec_check": (I32, [P]),
        "dec_timing_enable": (I32, [P, I32, I32]),
        "dec_timing_read": (I32, [P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I32)]),
        "dec_destroy": (None, [P]),
        "dec_attend_scratch_bytes": (SZ, [I32, I32, I32, I32]),
        "dec_attend": (I32, [P, P, P, I32, I32, I32, I32, I32, I32, I32, P, P, SZ, P]),
        "dec_attend_noalloc": (I32, [P, P, P, I32, I32, I32, I32, I32, I32, I32, P, P]),
        "dec_gemm_bf16": (I32, [P, P, P, P, I32, I32, I32, P]),
        "dec_set_graph": (I32, [P, I32]),
        "dec_set_fused": (I32, [P, I32]),
        "dec_fused_available": (I32, [P, I32]),
        "dec_fused_mode": (I32, [P]),
        "dec_ffn_fused": (I32, [P]),
        "dec_phase_stamps": (I32, [P, P, I32]),
        "dec_last_error": (ctypes.c_char_p, [P]),
        "dec_prefill_seq": (I32, [P, I32, ctypes.POINTER(I32), I32, I32, P, P]),
        "dec_kv_reset_seq": (I32, [P, I32]),
        "dec_length_seq": (I32, [P, I32]),
        "dec_decode_batch": (I32, [P, I32, ctypes.POINTER(I32), ctypes.POINTER(I32), P, P, P]),
        "dec_kv_layer_seq": (I32, [P, I32, I32, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "dec_kv_quantize_int8": (I32, [P, I32, I32, I32, P, P]),
        "dec_kv_slot": (I32, [P, I32, I32, I32, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "dec_pages_free": (I32, [P]),
        "dec_selftest_wait_timeout": (I32, [P, I32]),
        "dec_weight_quantize_int8": (I32, [P, I32, ctypes.c_int64, I32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load_library()


class DecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def make_config(w: dict, kv_dtype: str = "f32", max_tokens: int = 0, n_seqs: int = 0, page_size: int = 0,
                n_pages: int = 0) -> Config:
    c = Config()
    for k in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
              "n_experts", "n_experts_used", "max_seq", "sliding_window"):
        setattr(c, k, int(w[k]))
    c.max_tokens = int(max_tokens)
    c.tied_embedding = int(bool(w["tied"]))
    c.qkv_bias = int(bool(w["qkv_bias"]))
    c.weight_dtype = DEC_F32 if w["dtype"] == "f32" else DEC_BF16
    c.kv_dtype = KV_DTYPES[kv_dtype]
    c.rms_eps = float(w["rms_eps"])
    c.rope_theta = float(w["rope_theta"])
    l3 = w.get("rope_llama3")
    if l3:
        c.rope_llama3 = 1
        c.rope_factor = l3["factor"]
        c.rope_low_freq_factor = l3["low_freq_factor"]
        c.rope_high_freq_factor = l3["high_freq_factor"]
        c.rope_orig_ctx = int(l3["orig_ctx"])
    c.rope_half = int(bool(w.get("rope_half", False)))
    c.rope_dim = int(w.get("rope_dim", 0))
    c.n_seqs = int(n_seqs)
    c.qk_norm = {None: 0, "": 0, "head": 1, "row": 2}[w.get("qk_norm")]
    c.sandwich_norms = int(bool(w.get("sandwich_norms", False)))
    c.rope_theta_local = float(w.get("rope_theta_local", 0.0) or 0.0)
    c.rope_global_every = int(w.get("rope_global_every", 0) or 0)
    c.page_size = int(page_size)
    c.n_pages = int(n_pages)
    c.weight_quant = 1 if w.get("weight_int8") else 0
    return c


def validate(c: Config) -> tuple:
    buf = ctypes.create_string_buffer(256)
    st = lib.dec_config_validate(ctypes.byref(c), buf, 256)
    return st, buf.value.decode()


def workspace_bytes(c: Config) -> int:
    return int(lib.dec_workspace_bytes(ctypes.byref(c)))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def attend(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, pos: int, sliding_window: int,
           out: torch.Tensor, scratch: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """dec_attend on torch device tensors: q [nq, hd] f32, k/v rings [max_seq, nkv, hd]."""
    max_seq, nkv, hd = k.shape
    nq = q.shape[0]
    kvd = DEC_F32 if k.dtype == torch.float32 else DEC_BF16
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.dec_attend(q.data_ptr(), k.data_ptr(), v.data_ptr(), nq, nkv, hd, max_seq, int(sliding_window), kvd,
                        int(pos), out.data_ptr(), scratch.data_ptr(), scratch.numel() * scratch.element_size(),
                        ctypes.c_void_p(s.cuda_stream))
    if st != DEC_OK:
        raise DecError(st, lib.dec_last_error(None).decode())


def gemm_bf16(a_hi: torch.Tensor, a_lo: Optional[torch.Tensor], b: torch.Tensor, c: torch.Tensor,
              stream: Optional[torch.cuda.Stream] = None) -> None:
    """c[m, n] = (a_hi + a_lo) @ b.T on the tensor-core kernel (bf16 in, f32 out)."""
    m, k = a_hi.shape
    n = b.shape[0]
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.dec_gemm_bf16(a_hi.data_ptr(), _ptr(a_lo), b.data_ptr(), c.data_ptr(), m, n, k,
                           ctypes.c_void_p(s.cuda_stream))
    if st != DEC_OK:
        raise DecError(st, lib.dec_last_error(None).decode())


def kv_int8_group(head_dim: int) -> int:
    """Channels per scale of the int8 cache rows (the library's rule, restated for views)."""
    g = 1
    while g < 32 and head_dim % (2 * g) == 0:
        g *= 2
    return g


def kv_int8_row_layout(n_kv_heads: int, head_dim: int) -> tuple:
    """(row bytes, code offset, group) of the DEC_I8 row format of dec.h."""
    kd = n_kv_heads * head_dim
    g = kv_int8_group(head_dim)
    sb = (kd // g * 4 + 15) // 16 * 16
    return sb + (kd + 15) // 16 * 16, sb, g


def split_int8_rows(rows: torch.Tensor, n_kv_heads: int, head_dim: int) -> tuple:
    """uint8 rows of the DEC_I8 format -> (scales f32 [n, kd/g], codes int8 [n, kd]) views."""
    kd = n_kv_heads * head_dim
    _, off, g = kv_int8_row_layout(n_kv_heads, head_dim)
    scales = rows[:, :kd // g * 4].contiguous().view(torch.float32)
    codes = rows[:, off:off + kd].contiguous().view(torch.int8)
    return scales, codes


def kv_quantize_int8(x: torch.Tensor, n_kv_heads: int, head_dim: int,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """dec_kv_quantize_int8: device f32 rows [n, n_kv_heads*head_dim] -> uint8 rows of the DEC_I8 format."""
    n = x.shape[0]
    rb, _, _ = kv_int8_row_layout(n_kv_heads, head_dim)
    out = torch.zeros((n, rb), dtype=torch.uint8, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.dec_kv_quantize_int8(x.data_ptr(), n, n_kv_heads, head_dim, out.data_ptr(),
                                  ctypes.c_void_p(s.cuda_stream))
    if st != DEC_OK:
        raise DecError(st, lib.dec_last_error(None).decode())
    return out


def weight_quantize_int8(w: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> tuple:
    """dec_weight_quantize_int8 on a device matrix [rows, cols] (f32 or bf16) -> (codes int8 [rows, cols],
    scales f32 [rows, cols / 32])."""
    rows, cols = w.shape
    codes = torch.empty((rows, cols), dtype=torch.int8, device=w.device)
    scales = torch.empty((rows, cols // 32), dtype=torch.float32, device=w.device)
    wd = DEC_F32 if w.dtype == torch.float32 else DEC_BF16
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib.dec_weight_quantize_int8(w.data_ptr(), wd, rows, cols, codes.data_ptr(), scales.data_ptr(),
                                      ctypes.c_void_p(s.cuda_stream))
    if st != DEC_OK:
        raise DecError(st, lib.dec_last_error(None).decode())
    return codes, scales


def attend_scratch_bytes(nq: int, nkv: int, hd: int, max_seq: int) -> int:
    return int(lib.dec_attend_scratch_bytes(nq, nkv, hd, max_seq))


class DeviceWeights:
    """Synthetic weights drawn straight into the library's device layouts.

    Layout only (no arithmetic): [Wq;Wk;Wv] rows concatenated, gate/up rows
    interleaved per output, experts stacked.
    """

    def __init__(self, w: dict, device="cuda", seed: int = 1234):
        self.w = w
        dt = synthetic.storage_dtype(w)
        h, f = w["hidden"], w["ffn"]
        qd, kd = w["n_heads"] * w["head_dim"], w["n_kv_heads"] * w["head_dim"]
        E = w["n_experts"]
        d = lambda role, l=-1, e=-1, out=None: synthetic.draw(w, role, l, e, seed, device, out)
        self.tok_embd = d("tok_embd")
        self.out_norm = d("out_norm")
        self.lm_head = None if w["tied"] else d("lm_head")
        self.layers = []
        for l in range(w["n_layers"]):
            L = {"attn_norm": d("attn_norm", l), "ffn_norm": d("ffn_norm", l), "wo": d("wo", l)}
            qkn, sw = w.get("qk_norm"), w.get("sandwich_norms")
            L["q_norm"] = d("q_norm", l) if qkn else None
            L["k_norm"] = d("k_norm", l) if qkn else None
            L["post_attn_norm"] = d("post_attn_norm", l) if sw else None
            L["post_ffn_norm"] = d("post_ffn_norm", l) if sw else None
            wqkv = torch.empty((qd + 2 * kd, h), dtype=dt, device=device)
            d("wq", l, out=wqkv[:qd])
            d("wk", l, out=wqkv[qd:qd + kd])
            d("wv", l, out=wqkv[qd + kd:])
            L["wqkv"] = wqkv
            L["bqkv"] = torch.cat([d("bq", l), d("bk", l), d("bv", l)]) if w["qkv_bias"] else None
            if E:
                L["router"] = d("router", l)
                gu = torch.empty((E, 2 * f, h), dtype=dt, device=device)
                dn = torch.empty((E, h, f), dtype=dt, device=device)
                for e in range(E):
                    v = gu[e].view(f, 2, h)
                    d("w_gate", l, e, out=v[:, 0, :])
                    d("w_up", l, e, out=v[:, 1, :])
                    d("w_down", l, e, out=dn[e])
                L["w_gateup"], L["w_down"] = gu, dn
            else:
                L["router"] = None
                gu = torch.empty((2 * f, h), dtype=dt, device=device)
                v = gu.view(f, 2, h)
                d("w_gate", l, out=v[:, 0, :])
                d("w_up", l, out=v[:, 1, :])
                L["w_gateup"], L["w_down"] = gu, d("w_down", l)
            self.layers.append(L)
        self._c_layers = (LayerWeights * w["n_layers"])()
        for i, L in enumerate(self.layers):
            for k in ("attn_norm", "wqkv", "bqkv", "wo", "ffn_norm", "w_gateup", "w_down", "router",
                      "q_norm", "k_norm", "post_attn_norm", "post_ffn_norm"):
                setattr(self._c_layers[i], k, _ptr(L[k]))
        self.c = Weights(self.tok_embd.data_ptr(), self.out_norm.data_ptr(), _ptr(self.lm_head),
                         ctypes.cast(self._c_layers, ctypes.POINTER(LayerWeights)))

    def nbytes(self) -> int:
        t = [self.tok_embd, self.out_norm, self.lm_head]
        for L in self.layers:
            t += list(L.values())
        return sum(x.numel() * x.element_size() for x in t if x is not None)


class Decoder:
    """A handle of the library: weights, workspace (KV cache + scratch) and a stream."""

    def __init__(self, w: dict, weights: Optional[DeviceWeights] = None, device="cuda", seed: int = 1234,
                 kv_dtype: str = "f32", max_tokens: int = 0, stream: Optional[torch.cuda.Stream] = None,
                 n_seqs: int = 0, page_size: int = 0, n_pages: int = 0):
        self.w = w
        self.device = torch.device(device)
        self.weights = weights if weights is not None else DeviceWeights(w, device, seed)
        self.cfg = make_config(w, kv_dtype, max_tokens, n_seqs, page_size, n_pages)
        st, msg = validate(self.cfg)
        if st != DEC_OK:
            raise DecError(st, msg)
        self.ws_bytes = workspace_bytes(self.cfg)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.stream = stream if stream is not None else torch.cuda.Stream(device=self.device)
        # dec_create may read the weights on the handle's stream (quantise, permute):
        # it must see them complete, so it waits for the stream they were drawn on.
        self.stream.wait_stream(torch.cuda.current_stream(self.device))
        self.kv_dtype = kv_dtype
        self.kv_torch_dtype = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.uint8}[kv_dtype]
        h = ctypes.c_void_p()
        st = lib.dec_create(ctypes.byref(self.cfg), ctypes.byref(self.weights.c), self.workspace.data_ptr(),
                            self.ws_bytes, ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        if st != DEC_OK:
            raise DecError(st, lib.dec_last_error(None).decode())
        self.h = h

    # -- calls -------------------------------------------------------------------
    def _raise(self, st: int):
        if st != DEC_OK:
            raise DecError(st, lib.dec_last_error(self.h).decode())

    def prefill(self, tokens, start_pos: int, logits: Optional[torch.Tensor],
                d_argmax: Optional[torch.Tensor] = None, seq: int = 0) -> None:
        """``tokens``: a host sequence of ids, or a pinned host int32 tensor (copied as is).
        ``seq``: the sequence whose KV rings are used (dec_prefill_seq)."""
        if isinstance(tokens, torch.Tensor):
            assert tokens.device.type == "cpu" and tokens.dtype == torch.int32 and tokens.is_contiguous()
            p, n = ctypes.cast(tokens.data_ptr(), ctypes.POINTER(ctypes.c_int32)), tokens.numel()
        else:
            a = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
            p, n = a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), a.size
        self._raise(lib.dec_prefill_seq(self.h, int(seq), p, int(n), int(start_pos), _ptr(logits), _ptr(d_argmax)))

    def decode_batch(self, seqs, positions, d_tokens: torch.Tensor, logits: torch.Tensor,
                     d_argmax: Optional[torch.Tensor] = None) -> None:
        """One batched decode step (dec_decode_batch): host ``seqs``/``positions`` (B each), device int32
        ``d_tokens`` [B], device f32 ``logits`` [B, vocab], optional device int32 ``d_argmax`` [B]."""
        sq = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        ps = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
        if sq.size != ps.size:
            raise ValueError("seqs and positions must have the same length")
        I32P = ctypes.POINTER(ctypes.c_int32)
        self._raise(lib.dec_decode_batch(self.h, int(sq.size), sq.ctypes.data_as(I32P), ps.ctypes.data_as(I32P),
                                         d_tokens.data_ptr(), logits.data_ptr(), _ptr(d_argmax)))

    @property
    def launch_count(self) -> int:
        return int(lib.dec_launch_count(self.h))

    def decode(self, token: int, pos: int, logits: Optional[torch.Tensor]) -> None:
        self._raise(lib.dec_decode(self.h, int(token), int(pos), _ptr(logits)))

    def decode_dev(self, d_token: torch.Tensor, pos: int, logits: Optional[torch.Tensor],
                   d_argmax: Optional[torch.Tensor] = None) -> None:
        self._raise(lib.dec_decode_dev(self.h, d_token.data_ptr(), int(pos), _ptr(logits), _ptr(d_argmax)))

    def set_fused(self, mode) -> None:
        """Decode schedule: "off" (per-layer kernels), "grid" (one persistent kernel over every SM) or
        "cluster" (one persistent kernel on one thread-block cluster); True means "grid", False "off"."""
        if isinstance(mode, bool):
            mode = DEC_FUSED_GRID if mode else DEC_FUSED_OFF
        elif isinstance(mode, str):
            mode = FUSED_MODES[mode]
        self._raise(lib.dec_set_fused(self.h, int(mode)))

    def fused_mode(self) -> str:
        """The schedule the next decode step takes: "off", "grid" or "cluster"."""
        m = int(lib.dec_fused_mode(self.h))
        return {v: k for k, v in FUSED_MODES.items()}[m]

    def ffn_fused(self) -> bool:
        """Whether the next decode step runs the FFN over ffn slices plus a partial-sum phase."""
        return int(lib.dec_ffn_fused(self.h)) == 1

    def fused_available(self, mode) -> int:
        """1 (or the cluster's CTA count) when the schedule can run on this handle, else 0."""
        if isinstance(mode, str):
            mode = FUSED_MODES[mode]
        return int(lib.dec_fused_available(self.h, int(mode)))

    def phase_stamps(self, stamps: Optional[torch.Tensor]) -> None:
        """Device int64 tensor receiving per-phase GPU timestamps of each fused decode step (None stops)."""
        self._raise(lib.dec_phase_stamps(self.h, _ptr(stamps), 0 if stamps is None else stamps.numel()))

    def set_graph(self, enable: bool) -> None:
        self._raise(lib.dec_set_graph(self.h, int(bool(enable))))

    def kv_reset(self, seq: int = 0) -> None:
        self._raise(lib.dec_kv_reset_seq(self.h, int(seq)))

    @property
    def length(self) -> int:
        return int(lib.dec_length(self.h))

    def length_of(self, seq: int) -> int:
        return int(lib.dec_length_seq(self.h, int(seq)))

    def kv_layer(self, layer: int, seq: int = 0):
        """(K, V) rings of a layer (of sequence ``seq``) as [max_seq, n_kv_heads, head_dim] views of the
        workspace; for an int8 cache, [max_seq, row_bytes] uint8 rows (see ``split_int8_rows``)."""
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        self._raise(lib.dec_kv_layer_seq(self.h, int(layer), int(seq), ctypes.byref(k), ctypes.byref(v)))
        base = self.workspace.data_ptr()
        ms, nkv, hd = self.w["max_seq"], self.w["n_kv_heads"], self.w["head_dim"]
        views = []
        for p in (k.value, v.value):
            off = p - base
            if self.kv_dtype == "i8":
                rb = kv_int8_row_layout(nkv, hd)[0]
                views.append(self.workspace[off:off + ms * rb].view(ms, rb))
            else:
                es = 4 if self.kv_torch_dtype == torch.float32 else 2
                views.append(self.workspace[off:off + ms * nkv * hd * es].view(self.kv_torch_dtype)
                             .view(ms, nkv, hd))
        return views[0], views[1]

    def kv_slot(self, layer: int, seq: int, slot: int):
        """(K, V) rows of one slot (either layout): [n_kv_heads, head_dim] views, or uint8 rows of the
        int8 format for an int8 cache."""
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        st = lib.dec_kv_slot(self.h, int(layer), int(seq), int(slot), ctypes.byref(k), ctypes.byref(v))
        if st != DEC_OK:
            raise DecError(st, f"no K/V row for layer {layer}, sequence {seq}, slot {slot}")
        base = self.workspace.data_ptr()
        nkv, hd = self.w["n_kv_heads"], self.w["head_dim"]
        out = []
        for p in (k.value, v.value):
            off = p - base
            if self.kv_dtype == "i8":
                rb = kv_int8_row_layout(nkv, hd)[0]
                out.append(self.workspace[off:off + rb].view(1, rb))
            else:
                es = 4 if self.kv_torch_dtype == torch.float32 else 2
                out.append(self.workspace[off:off + nkv * hd * es].view(self.kv_torch_dtype).view(nkv, hd))
        return out[0], out[1]

    @property
    def pages_free(self) -> int:
        return int(lib.dec_pages_free(self.h))

    def set_trace(self, ids: Optional[torch.Tensor], logits: Optional[torch.Tensor], capacity: int) -> None:
        self._raise(lib.dec_set_trace(self.h, _ptr(ids), _ptr(logits), int(capacity)))

    def check(self) -> None:
        self._raise(lib.dec_check(self.h))

    def selftest_wait_timeout(self, limit_us: int) -> None:
        """dec_selftest_wait_timeout: enqueue a bounded wait that runs out (see dec.h)."""
        self._raise(lib.dec_selftest_wait_timeout(self.h, int(limit_us)))

    def timing_enable(self, kernel_class: str, max_launches: int) -> None:
        cls = KERNEL_CLASSES.get(kernel_class, 0) if isinstance(kernel_class, str) else int(kernel_class)
        self._raise(lib.dec_timing_enable(self.h, cls, int(max_launches)))

    def timing_read(self) -> tuple:
        """(summed milliseconds, launches) of the timed kernel class in the most recent call."""
        ms, n = ctypes.c_float(), ctypes.c_int32()
        self._raise(lib.dec_timing_read(self.h, ctypes.byref(ms), ctypes.byref(n)))
        return float(ms.value), int(n.value)

    def synchronize(self) -> None:
        self.stream.synchronize()

    def close(self) -> None:
        if getattr(self, "h", None):
            lib.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
