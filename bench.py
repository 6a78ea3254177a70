"""Benchmark of the decoder forward pass: single-pass prefill + greedy decode at batch 1.

One step = prefill of the workload's prompt (P tokens) followed by D greedy
decode steps, through libdec.so.  ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the baseline arm).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload mixtral-8x7b] [--per-workload auto|none|a,b] [--kv f32|bf16|i8]

The main line measures one workload (default Mixtral-8x7B, the largest single-GPU
configuration); ``per_workload`` repeats the measurement, with fewer steps, for the
other named workloads in the same run.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from decoder_only_forward_gb300 import synthetic  # noqa: E402

METRIC = "prefill tok/s + decode tok/s at bs=1; decode % of HBM roofline"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2**20
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def max_over_ranks(values, device, world: int) -> list:
    """Each timing taken as the slowest rank's (replicas run in parallel; the job ends with the last)."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def replica_value(n_ranks: int, tokens_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes tokens_per_step per step; the step takes the
    slowest rank's time."""
    return n_ranks * tokens_per_step / (ms_per_step / 1e3)


def workload_of(args) -> dict:
    """The named workload, with the architecture variant flags applied."""
    kw = {}
    if getattr(args, "qk_norm", ""):
        kw["qk_norm"] = args.qk_norm
    if getattr(args, "sandwich", False):
        kw["sandwich_norms"] = True
    if getattr(args, "weights", "") == "i8":
        kw["weight_int8"] = True
    return synthetic.workload(args.workload, **kw)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- algorithmic work
def weight_bytes(w: dict) -> dict:
    """Bytes of each decode-path matrix (stored dtype), per layer / per launch."""
    es = 4 if w["dtype"] == "f32" else 2
    # 8-bit projections: one byte per weight plus an f32 scale per 32 columns.
    ps = 1 + 4 / 32 if w.get("weight_int8") else es
    h, f, hd = w["hidden"], w["ffn"], w["head_dim"]
    qd, kd = w["n_heads"] * hd, w["n_kv_heads"] * hd
    k = w["n_experts_used"] if w["n_experts"] else 1
    return {
        "qkv": (qd + 2 * kd) * h * ps,
        "oproj": h * qd * ps,
        "gateup": k * 2 * f * h * ps,
        "down": k * h * f * ps,
        "router": w["n_experts"] * h * es,
        "lmhead": w["vocab"] * h * (es if w["tied"] else ps),
        "embed_row": h * es,
    }


# DRAM bytes per launch of a roofline kernel, from one ncu capture each.  A figure holds only for the
# kernel source it measured: the source file's SHA-256 at capture time must
# match the current file, else the bench reports traffic as null.
TRAFFIC = {
    ("smollm2-135m", "down"): {
        "bytes": 1814336, "source": "decoder_only_forward_gb300/csrc/decode.cu",
        "sha256": "3d7213fecd5001252701110382d8e9dfd57676011ecc1ded9bf6666198c7ae34"},
    ("mixtral-8x7b", "step"): {
        "bytes": 25920759040, "source": "decoder_only_forward_gb300/csrc/decode_mk.cu",
        "sha256": "089d684fe53ae73b10b7d86dd4ca97ea9697d93c4a182b0a69e84d1ef790b4dd"},
}


def measured_traffic(workload: str, kernel: str):
    t = TRAFFIC.get((workload, kernel))
    if t is None:
        return None
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), t["source"])
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != t["sha256"]:
                return None
    except OSError:
        return None
    return t["bytes"]


def kv_bytes_per_element(w: dict, kv: str) -> float:
    """Stored bytes per K (or V) element: 4, 2, or for int8 rows (codes + per-group f32 scales) the
    row's bytes over its n_kv_heads * head_dim elements."""
    if kv != "i8":
        return 4 if kv == "f32" else 2
    from decoder_only_forward_gb300.dec import kv_int8_row_layout
    return kv_int8_row_layout(w["n_kv_heads"], w["head_dim"])[0] / (w["n_kv_heads"] * w["head_dim"])


def decode_bytes(w: dict, pos: int, kv_es: float) -> float:
    """Weights + KV read by one decode step at absolute position pos (the decode roofline's bytes)."""
    b = weight_bytes(w)
    per_layer = b["qkv"] + b["oproj"] + b["gateup"] + b["down"] + b["router"] + 2 * 4 * w["hidden"]
    m = min(pos + 1, w["max_seq"]) if w["sliding_window"] > 0 else pos + 1
    kv = 2 * w["n_kv_heads"] * w["head_dim"] * m * kv_es
    return w["n_layers"] * (per_layer + kv) + b["lmhead"] + b["embed_row"] + 4 * w["hidden"]


def batched_step_bytes(w: dict, positions, kv_es: int) -> float:
    """HBM bytes of one batched decode step: every weight matrix once (all experts for a MoE, an
    upper bound: a batch of rows usually touches every expert), the LM head, one embedding row and
    each row's readable K/V."""
    b = weight_bytes(w)
    E = w["n_experts"]
    ffn = (b["gateup"] + b["down"]) * (E // w["n_experts_used"] if E else 1)
    per_layer = b["qkv"] + b["oproj"] + ffn + b["router"] + 2 * 4 * w["hidden"]
    kv = 0
    for pos in positions:
        m = min(pos + 1, w["max_seq"]) if w["sliding_window"] > 0 else pos + 1
        kv += 2 * w["n_kv_heads"] * w["head_dim"] * m * kv_es
    return w["n_layers"] * per_layer + w["n_layers"] * kv + b["lmhead"] + len(positions) * b["embed_row"]


def prefill_flops(w: dict, P: int) -> float:
    h, f, hd = w["hidden"], w["ffn"], w["head_dim"]
    qd, kd = w["n_heads"] * hd, w["n_kv_heads"] * hd
    k = w["n_experts_used"] if w["n_experts"] else 1
    lin = (qd + 2 * kd) * h + h * qd + k * 3 * f * h + w["n_experts"] * h
    attn = 4 * hd * w["n_heads"] * P * (P + 1) / 2
    return w["n_layers"] * (2 * P * lin + attn) + 2 * w["vocab"] * h


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # nvidia-smi samples of this run; DEC_CLOCKS_DIR keeps them somewhere chosen.
        out_dir = os.environ.get("DEC_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
class _TimedSource:
    """Wraps a weight source and adds up the seconds spent drawing weights, so that the
    oracle's own arithmetic can be timed apart from input generation."""

    def __init__(self, inner):
        self.inner = inner
        self.cfg = inner.cfg
        self.fetch_s = 0.0

    def _t(self, fn, *a):
        t0 = time.perf_counter()
        try:
            return fn(*a)
        finally:
            self.fetch_s += time.perf_counter() - t0

    def embed_rows(self, tokens):
        return self._t(self.inner.embed_rows, tokens)

    def out_norm(self):
        return self._t(self.inner.out_norm)

    def lm_head(self):
        return self._t(self.inner.lm_head)

    def layer(self, l):
        return self._t(self.inner.layer, l)

    def expert(self, l, e):
        return self._t(self.inner.expert, l, e)


def oracle_sample_plan(w: dict) -> dict:
    """The bounded sample of a workload the float64 oracle is timed on: its first
    ``layers`` layers, a batched single-pass prefill of ``prefill`` prompt tokens, then
    ``decode`` per-token forwards; the time is scaled to the whole model by
    n_layers / layers (the head's share is scaled with it, which overstates the
    oracle's time by a few percent at most)."""
    if w["hidden"] >= 2048:
        return dict(layers=2, prefill=512, decode=4)
    return dict(layers=w["n_layers"], prefill=min(512, w["prompt"]), decode=4)


def oracle_sample(w: dict, plan: dict, device: str, src=None):
    """Times the float64 oracle on the bounded sample ``plan`` of workload ``w``.

    Weights are drawn once (on ``device``) and kept as float64 for the sampled layers;
    time spent drawing is excluded.  Returns (tok/s scaled to the whole model,
    seconds of oracle arithmetic, cores, the weight source for reuse)."""
    from oracle import OracleConfig, Session
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    ws = dict(w, n_layers=plan["layers"])
    if src is None:
        src = synthetic.OracleWeightSource(ws, device=device, cache=True)
    timed = _TimedSource(src)
    sess = Session(OracleConfig.from_dict(ws), timed)
    n_pf, n_dc = plan["prefill"], plan["decode"]
    toks = synthetic.prompt_tokens(w, n_pf + n_dc, seed=0)
    t0 = time.perf_counter()
    sess.prefill_batched(list(toks[:n_pf]), 0)
    for i in range(n_dc):
        sess.forward(int(toks[n_pf + i]), n_pf + i)
    dt = time.perf_counter() - t0 - timed.fetch_s
    scaled = dt * w["n_layers"] / plan["layers"]
    return (n_pf + n_dc) / scaled, dt, cores, src


def oracle_sample_text(name: str, w: dict, plan: dict, cores: int) -> str:
    what = (f"the first {plan['layers']} of {w['n_layers']} layers" if plan["layers"] < w["n_layers"]
            else f"all {w['n_layers']} layers")
    experts = f" (each with all {w['n_experts']} experts)" if w["n_experts"] else ""
    return (f"float64 oracle on {cores} host cores: {what}{experts} of the {name}-shaped model, batched "
            f"single-pass prefill of {plan['prefill']} prompt tokens + {plan['decode']} per-token forwards; "
            f"weights drawn beforehand (not timed); time scaled by {w['n_layers']}/{plan['layers']} layers")


# ---------------------------------------------------------------- our arm
PER_WORKLOAD_DEFAULT = ["smollm2-135m", "qwen2.5-0.5b", "mistral-7b", "mixtral-8x7b",
                        "mixtral-8x7b+int8_weights"]


def named_workload(name: str) -> dict:
    """A named workload, or one with a variant suffix ("+int8_weights": 8-bit projections)."""
    base, _, variant = name.partition("+")
    kw = {"weight_int8": True} if variant == "int8_weights" else {}
    if variant and not kw:
        raise ValueError(f"unknown workload variant {variant!r}")
    return synthetic.workload(base, **kw)


def gemm_flops(w: dict, P: int) -> float:
    """Algorithmic FLOPs of the prefill projection GEMMs (QKV, O, gate/up, down; MoE: the
    k selected experts per row): 2 * rows * active linear parameters."""
    h, f, hd = w["hidden"], w["ffn"], w["head_dim"]
    qd, kd = w["n_heads"] * hd, w["n_kv_heads"] * hd
    k = w["n_experts_used"] if w["n_experts"] else 1
    return w["n_layers"] * 2.0 * P * ((qd + 2 * kd) * h + h * qd + k * 3 * f * h)


def measure_workload(name, w, dev, args, steps, warmup, weights=None, want_e2e_steps=3,
                     attribution=True, world=1):
    """One workload: W untimed steps, then K timed steps of (kv reset, prefill of P tokens,
    D greedy decode steps), L2 flushed before each; then an end-to-end pass through the
    API with host buffers, and (optional) attribution passes after the timed region."""
    from decoder_only_forward_gb300 import dec
    P, D, V = w["prompt"], w["decode"], w["vocab"]
    kv_es = kv_bytes_per_element(w, args.kv)
    d = dec.Decoder(w, weights=weights, device=dev, kv_dtype=args.kv)
    if args.fused != "auto":
        d.set_fused(args.fused)
    s = d.stream
    prompt_np = synthetic.prompt_tokens(w, P, seed=0)
    prompt_pinned = torch.from_numpy(prompt_np).pin_memory()
    logits = torch.empty(V, dtype=torch.float32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    flush = torch.empty(max(2 * L2_BYTES, 256 * 2**20) // 4, dtype=torch.float32, device=dev)

    def step(evs=None):
        if evs is not None:
            with torch.cuda.stream(s):
                flush.zero_()
            evs[0].record(s)
        d.kv_reset()  # each step is a new sequence
        d.prefill(prompt_np, 0, logits, tok)
        if evs is not None:
            evs[1].record(s)
        for i in range(D):
            d.decode_dev(tok, P + i, logits, tok)
        if evs is not None:
            evs[2].record(s)

    for _ in range(warmup):
        step()
    d.check()
    torch.cuda.synchronize(dev)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    launches0 = d.launch_count
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index or 0) as clk:
        wall0 = time.perf_counter()
        for k in range(steps):
            step(events[k])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    launches = d.launch_count - launches0
    d.check()
    pre_ms = [e[0].elapsed_time(e[1]) for e in events]
    dec_ms = [e[1].elapsed_time(e[2]) for e in events]
    tot_ms = sum(p + q for p, q in zip(pre_ms, dec_ms))
    tot_ms, pre_sum, dec_sum = max_over_ranks([tot_ms, sum(pre_ms), sum(dec_ms)], dev, world)
    r = dict(d=d, P=P, D=D, V=V, kv_es=kv_es, steps=steps, warmup=warmup,
             ms_per_step=tot_ms / steps, pre_s=pre_sum / steps / 1e3, dec_s=dec_sum / steps / 1e3,
             launches=launches, wall=wall, clocks=clk.summary(), schedule=d.fused_mode(),
             weights_gb=d.weights.nbytes() / 1e9)
    r["dbytes"] = sum(decode_bytes(w, P + i, kv_es) for i in range(D))
    r["pflops"] = prefill_flops(w, P)

    # ---- end to end through the public API with host buffers ----
    if want_e2e_steps:
        tok_host = torch.empty(1, dtype=torch.int32).pin_memory()
        logits_host = torch.empty(V, dtype=torch.float32).pin_memory()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(want_e2e_steps):
            d.kv_reset()
            d.prefill(prompt_pinned, 0, logits, tok)
            for i in range(D):
                d.decode_dev(tok, P + i, logits, tok)
                with torch.cuda.stream(s):
                    tok_host.copy_(tok, non_blocking=True)
                s.synchronize()
            with torch.cuda.stream(s):
                logits_host.copy_(logits, non_blocking=True)
            s.synchronize()
        r["e2e_s"] = (time.perf_counter() - t0) / want_e2e_steps

    if attribution:
        # Prefill: each tensor-core kernel class timed alone in its own prefill (event pairs
        # around its launches; the launches are long, so the pairs barely perturb them).
        pk = {}
        for c in ("pf_gemm", "pf_attn"):
            d.timing_enable(c, 100000)
            d.kv_reset()
            d.prefill(prompt_np, 0, logits, tok)
            ms, n = d.timing_read()
            pk[c] = (ms, n)
        d.timing_enable("pf_gemm", 0)
        r["prefill_kernels"] = pk
        # Decode, persistent step: per-phase GPU timestamps of CTA 0 (one %globaltimer
        # store per grid barrier; the step is not otherwise changed).
        if r["schedule"] != "off":
            ppl_max = 6
            st = torch.zeros(w["n_layers"] * ppl_max + 2, dtype=torch.int64, device=dev)
            d.kv_reset()
            d.prefill(prompt_np, 0, logits, tok)
            d.phase_stamps(st)
            rows = []
            nst = min(D, 16)
            for i in range(nst):
                d.decode_dev(tok, P + i, logits, tok)
                d.synchronize()
                rows.append(st.cpu().numpy().astype(np.int64).copy())
            d.phase_stamps(None)
            d.check()
            r["phase_rows"] = rows
            r["ffn_fused"] = d.ffn_fused()
    return r


def phase_summary(w: dict, rows, merge_phase: bool, ffn_fused: bool = False) -> dict:
    """Per-phase µs per token (summed over layers) from the persistent step's stamps.  With
    the fused FFN the last two phases of a layer are the FFN over each CTA's ffn slice
    ("ffn") and the sum of the CTAs' down-projection partials into the residual ("ffn_sum")."""
    ppl = 6 if merge_phase else 5
    ffn = ["ffn", "ffn_sum"] if ffn_fused else ["gateup", "down"]
    names = (["qkv", "attn", "merge", "oproj"] if ppl == 6 else ["qkv", "attn", "oproj"]) + ffn
    n = w["n_layers"] * ppl + 1
    diffs = np.stack([np.diff(r[: n + 1]) for r in rows[2:]]) if len(rows) > 2 else \
        np.stack([np.diff(r[: n + 1]) for r in rows])
    med = np.median(diffs, axis=0)
    out = {nm: round(float(np.sum(med[:-1].reshape(w["n_layers"], ppl)[:, j])) / 1e3, 1)
           for j, nm in enumerate(names)}
    out["lmhead"] = round(float(med[-1]) / 1e3, 1)
    out["total"] = round(float(np.sum(med)) / 1e3, 1)
    return out


def workload_summary(name, w, r, n, hbm, tf, tf_sus) -> dict:
    """The prefill/decode figures of one measured workload."""
    P, D = r["P"], r["D"]
    out = {
        "workload": name, "prompt_tokens": P, "decode_tokens": D, "batch": 1, "steps": r["steps"],
        "warmup": r["warmup"], "decode_schedule": r["schedule"], "weights_gb": round(r["weights_gb"], 3),
        "step_tok_s": round(n * (P + D) / (r["ms_per_step"] / 1e3), 2), "ms_per_step": round(r["ms_per_step"], 4),
        "prefill": {"tok_s": round(n * P / r["pre_s"], 1), "ms": round(r["pre_s"] * 1e3, 4), "flops": r["pflops"],
                    "tensor_frac": round(r["pflops"] / r["pre_s"] / (tf * 1e12), 5),
                    "tensor_frac_sustained": round(r["pflops"] / r["pre_s"] / (tf_sus * 1e12), 5)},
        "decode": {"tok_s": round(n * D / r["dec_s"], 1), "ms": round(r["dec_s"] * 1e3, 4),
                   "bytes_per_token_avg": round(r["dbytes"] / D),
                   "hbm_frac": round(r["dbytes"] / r["dec_s"] / (hbm * 1e9), 4),
                   "hbm_frac_nominal_8tbs": round(r["dbytes"] / r["dec_s"] / (NOMINAL_HBM_GBS * 1e9), 4)},
        "clocks": r["clocks"],
    }
    if "e2e_s" in r:
        out["e2e_tok_s"] = round(n * (P + D) / r["e2e_s"], 2)
    return out


def run_ours(args, rank, world, local_rank):
    from decoder_only_forward_gb300 import build as dec_build
    if rank == 0:
        dec_build.build()
    if world > 1:
        torch.distributed.barrier()
    dec_build.build()

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workload_of(args)
    hbm, tf, tf_sus, peak_kind = peaks()
    r = measure_workload(args.workload, w, dev, args, args.steps, args.warmup,
                         want_e2e_steps=max(1, min(args.steps, 3)), world=world)
    d = r["d"]
    P, D, V = r["P"], r["D"], r["V"]
    n = world

    # ---- roofline of the dominant kernel: the decode step ----
    dec_share = r["dec_s"] / (r["ms_per_step"] / 1e3)
    if r["schedule"] != "off":
        # One persistent kernel per decode token: its launches are the decode region.
        per_launch_bytes = r["dbytes"] / D
        avg_launch_s = r["dec_s"] / D
        kname = "k_decode_step"
        traffic = measured_traffic(args.workload, "step")
        note = ("one launch per token; duration = the timed decode region / D (CUDA events on the "
                "library's stream), so launch gaps count against the kernel")
    else:
        per_launch_bytes = r["dbytes"] / D
        avg_launch_s = r["dec_s"] / D
        kname = "decode step (chain of per-layer kernels)"
        traffic = None
        note = "per-layer kernels chained by programmatic dependent launch; figure is per token, not per launch"
    achieved = per_launch_bytes / avg_launch_s / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_kind": peak_kind,
                "bytes_per_launch": int(per_launch_bytes), "avg_launch_us": round(avg_launch_s * 1e6, 3),
                "launches_per_step": D, "share_of_step": round(dec_share, 4), "note": note}
    pk = r.get("prefill_kernels", {})
    roofline_prefill = None
    if pk.get("pf_gemm", (0, 0))[1]:
        g_ms, g_n = pk["pf_gemm"]
        gf = gemm_flops(w, P)
        ach = gf / (g_ms / 1e3) / 1e12
        roofline_prefill = {
            "bound": "tensor", "kernel": "k_gemm_tc (prefill projection GEMMs)", "achieved": round(ach, 1),
            "peak": tf, "unit": "TFLOP/s", "frac": round(ach / tf, 4), "frac_sustained": round(ach / tf_sus, 4),
            "traffic": None, "peak_kind": peak_kind, "flops_per_launch": round(gf / g_n),
            "avg_launch_us": round(g_ms * 1e3 / g_n, 3), "launches_per_prefill": g_n,
            "ms_per_prefill": round(g_ms, 4), "share_of_prefill": round(g_ms / (r["pre_s"] * 1e3), 4),
            "note": "GEMM launches timed alone in one extra prefill (event pair around each launch)"}
    prefill_kernels = {c: {"ms": round(ms, 4), "launches": nl} for c, (ms, nl) in pk.items()}
    phases = None
    if "phase_rows" in r:
        # The step stores a start stamp, one per phase and one after the head: the count of
        # stored stamps gives the phases per layer (5, or 6 with a split-merge phase).
        nz = int(np.count_nonzero(r["phase_rows"][-1]))
        phases = phase_summary(w, r["phase_rows"], (nz - 2) // w["n_layers"] == 6, r.get("ffn_fused", False))

    out = None
    if rank == 0:
        value = replica_value(n, P + D, r["ms_per_step"])
        cpu = None
        if not args.no_cpu_baseline:
            plan = oracle_sample_plan(w)
            cv, secs, cores, _ = oracle_sample(w, plan, device=str(dev))
            cpu = {"value": round(cv, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                   "sample": oracle_sample_text(args.workload, w, plan, cores) + f"; {secs:.1f} s of arithmetic"}
        s = workload_summary(args.workload, w, r, n, hbm, tf, tf_sus)
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"] if w["dtype"] != "f32" else "f32",
            "data": "synthetic (random-init weights N(0,0.02), norms 1+N(0,0.1), uniform random prompt)",
            "config": {"workload": args.workload + (f"+qk_norm_{args.qk_norm}" if args.qk_norm else "")
                       + ("+sandwich" if args.sandwich else "") + ("+int8_weights" if args.weights == "i8" else ""),
                       "prompt_tokens": P, "decode_tokens": D, "batch": 1,
                       "decode_schedule": r["schedule"],
                       "kv_dtype": args.kv, "weights_gb": round(r["weights_gb"], 3),
                       "l2": "flushed before each step (write of a 258 MB buffer); weights also exceed L2",
                       "parallelism": f"replicas x{n}" if n > 1 else "single GPU"},
            "prefill": s["prefill"], "decode": s["decode"], "clocks": r["clocks"],
            "e2e": {"value": round(n * (P + D) / r["e2e_s"], 2), "unit": "tok/s",
                    "h2d_bytes_per_step": 4 * P, "d2h_bytes_per_step": 4 * D + 4 * V,
                    "note": "pinned prompt copied in by dec_prefill; each greedy token read back to the host; "
                            "final logits read back"},
            "gpu_launches": int(r["launches"] / args.steps) * args.steps,
            "gpu_launches_per_step": int(r["launches"] / args.steps),
            "roofline": roofline,
            "roofline_prefill": roofline_prefill,
            "prefill_kernels_ms": prefill_kernels,
            "decode_phases_us_per_token": phases,
            "cpu_baseline": cpu,
            "wall_s_timed": round(r["wall"], 3),
        }
    if rank == 0 and args.batch > 0:
        out["batched_decode"] = run_batched(args, w, d.weights, dev, r["kv_es"])
    d.close()
    del d, r
    if rank == 0 and args.per_workload != "none":
        names = PER_WORKLOAD_DEFAULT if args.per_workload == "auto" else args.per_workload.split(",")
        per = {}
        for nm in names:
            if nm == args.workload:
                per[nm] = {"same_as_main_line": True}
                continue
            torch.cuda.empty_cache()
            wn = named_workload(nm)
            rn = measure_workload(nm, wn, dev, args, args.per_workload_steps, 3, want_e2e_steps=1,
                                  attribution=False)
            per[nm] = workload_summary(nm, wn, rn, 1, hbm, tf, tf_sus)
            rn["d"].close()
            del rn
        out["per_workload"] = per
    return out


def run_batched(args, w, weights, dev, kv_es):
    """Batched multi-sequence decode: ``args.batch`` sequences, each prefilled with its own prompt of
    the workload's length, then greedy steps of all of them at once (dec_decode_batch, tokens fed
    back from the device argmax).  Inputs exceed L2 (weights and the sequences' K/V), so no flush."""
    from decoder_only_forward_gb300 import dec
    B, P, V = args.batch, w["prompt"], w["vocab"]
    if w["sliding_window"] == 0 and P + 3 + args.batch_steps > w["max_seq"]:
        return {"skipped": "the cache cannot hold the prompt plus the timed steps"}
    # A paged cache gets exactly the pages B sequences of max_seq positions need.
    ps = args.page_size
    n_pages = B * ((w["max_seq"] + ps - 1) // ps) if ps else 0
    d = dec.Decoder(w, weights=weights, device=dev, kv_dtype=args.kv, n_seqs=B, page_size=ps, n_pages=n_pages)
    lg = torch.empty(V, dtype=torch.float32, device=dev)
    for sq in range(B):
        d.prefill(synthetic.prompt_tokens(w, P, seed=100 + sq), 0, lg, seq=sq)
    seqs = list(range(B))
    tok = torch.zeros(B, dtype=torch.int32, device=dev)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)
    pos = P
    for _ in range(3):
        d.decode_batch(seqs, [pos] * B, tok, logits, tok)
        pos += 1
    d.check()
    K = args.batch_steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    launches0 = d.launch_count
    e0.record(d.stream)
    for i in range(K):
        d.decode_batch(seqs, [pos + i] * B, tok, logits, tok)
    e1.record(d.stream)
    torch.cuda.synchronize(dev)
    launches = d.launch_count - launches0
    ms = e0.elapsed_time(e1) / K
    nbytes = sum(batched_step_bytes(w, [pos + i] * B, kv_es) for i in range(K)) / K
    # Attribution: the attention kernels' share of one step.
    d.timing_enable("attn", 4 * w["n_layers"])
    d.decode_batch(seqs, [pos + K] * B, tok, logits, tok)
    attn_ms, n_attn = d.timing_read()
    d.timing_enable("attn", 0)
    d.check()
    hbm = peaks()[0]
    out = {"batch": B, "steps": K, "tok_s": round(B * 1e3 / ms, 1), "ms_per_step": round(ms, 4),
           "bytes_per_step": int(nbytes), "hbm_frac": round(nbytes / (ms / 1e3) / (hbm * 1e9), 4),
           "attn_ms_per_step": round(attn_ms, 4), "gpu_launches_per_step": int(launches / K),
           "kv_layout": f"paged, {ps} positions per page" if ps else "contiguous rings",
           "note": "each sequence prefilled with its own prompt; one CUDA graph per step; bytes count every "
                   "weight once plus each row's readable K/V"}
    d.close()
    return out


def run_profile(args):
    """A small fixed sequence for per-kernel profilers: prefill P + D decode steps."""
    from decoder_only_forward_gb300 import build as dec_build
    dec_build.build()
    from decoder_only_forward_gb300 import dec
    w = workload_of(args)
    if args.prompt:
        w["prompt"] = args.prompt
    if args.layers:
        w["n_layers"] = args.layers
    if args.profile_batch:
        run_profile_batched(args, w)
        return
    d = dec.Decoder(w, kv_dtype=args.kv)
    d.set_graph(False)
    if args.fused != "auto":
        d.set_fused(args.fused)
    P = w["prompt"]
    logits = torch.empty(w["vocab"], dtype=torch.float32, device="cuda")
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    d.prefill(synthetic.prompt_tokens(w, P, seed=0), 0, logits, tok)
    for i in range(args.profile):
        d.decode_dev(tok, P + i, logits, tok)
    d.check()
    print(f"profile run: {args.workload} prefill {P} + decode {args.profile}, {d.launch_count} kernel launches")
    d.close()


def run_profile_batched(args, w):
    """Batched decode for per-kernel profilers: args.profile_batch sequences prefilled with their own
    prompts, two untimed steps, then args.profile steps inside the NVTX range "batched_steps" (a
    profiler can keep to that range), kernels launched one by one."""
    from decoder_only_forward_gb300 import dec
    B, P, V = args.profile_batch, w["prompt"], w["vocab"]
    ps = args.page_size
    d = dec.Decoder(w, kv_dtype=args.kv, n_seqs=B, page_size=ps,
                    n_pages=B * ((w["max_seq"] + ps - 1) // ps) if ps else 0)
    d.set_graph(False)
    lg = torch.empty(V, dtype=torch.float32, device="cuda")
    for sq in range(B):
        d.prefill(synthetic.prompt_tokens(w, P, seed=100 + sq), 0, lg, seq=sq)
    seqs = list(range(B))
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, V), dtype=torch.float32, device="cuda")
    for i in range(2):
        d.decode_batch(seqs, [P + i] * B, tok, out, tok)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("batched_steps")
    for i in range(args.profile):
        d.decode_batch(seqs, [P + 2 + i] * B, tok, out, tok)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    d.check()
    print(f"profile run: {args.workload} batched decode of {B} sequences (prompt {P}), {args.profile} steps")
    d.close()


# ---------------------------------------------------------------- reference arm (oracle)
def run_reference(args):
    """The baseline arm: the float64 oracle as it stands on the host cores, on a bounded
    sample of the same workload each step (``oracle_sample_plan``), scaled to tok/s of
    the whole model.  Weights are drawn once (on the GPU when there is one, the same values
    the library gets) and kept as float64 for the sampled layers."""
    w = workload_of(args)
    plan = oracle_sample_plan(w)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    rates, secs = [], []
    cores = len(os.sched_getaffinity(0))
    src = None
    for i in range(args.warmup + args.steps):
        r, s_, cores, src = oracle_sample(w, plan, device=dev, src=src)
        if i >= args.warmup:
            rates.append(r)
            secs.append(s_)
    scale = w["n_layers"] / plan["layers"]
    tokens = plan["prefill"] + plan["decode"]
    value = tokens * len(secs) / (sum(secs) * scale)
    sample = oracle_sample_text(args.workload, w, plan, cores)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(secs) * scale / len(secs), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "prompt_tokens": w["prompt"], "decode_tokens": w["decode"],
                   "batch": 1, "sample": {"layers": plan["layers"], "prefill_tokens": plan["prefill"],
                                          "decode_tokens": plan["decode"], "time_scaled_by": scale}},
        "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral-8x7b", choices=sorted(synthetic.WORKLOADS),
                    help="the main line's workload (default: the largest single-GPU configuration)")
    ap.add_argument("--per-workload", default="auto",
                    help="also measure these workloads (comma list; auto: every named non-toy workload; none)")
    ap.add_argument("--per-workload-steps", type=int, default=3)
    ap.add_argument("--kv", default="f32", choices=["f32", "bf16", "i8"])
    ap.add_argument("--weights", default="", choices=["", "i8"],
                    help="i8: 8-bit projection weights (quantised by the library at create)")
    ap.add_argument("--prompt", type=int, default=0, help="override the prompt length (profiling only)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (with --profile only: small cases for profiler captures)")
    ap.add_argument("--fused", default="auto", choices=["auto", "off", "grid", "cluster"],
                    help="decode schedule: per-layer kernels, or the persistent one-kernel step over every SM "
                         "or on one thread-block cluster (default: the handle's own choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=16,
                    help="also time batched multi-sequence decode at this batch (0: skip)")
    ap.add_argument("--batch-steps", type=int, default=32)
    ap.add_argument("--qk-norm", default="", choices=["", "head", "row"],
                    help="architecture variant: QK-norm (adds q_norm/k_norm weights)")
    ap.add_argument("--sandwich", action="store_true", help="architecture variant: sandwich norms")
    ap.add_argument("--page-size", type=int, default=0,
                    help="batched decode on a paged cache of this page size (0: contiguous rings)")
    ap.add_argument("--profile", type=int, default=0, metavar="D",
                    help="profiling driver: one prefill + D decode steps, kernels launched one by one "
                         "(no graph, no timing passes, no JSON); for per-kernel profilers")
    ap.add_argument("--profile-batch", type=int, default=0, metavar="B",
                    help="with --profile D: D batched decode steps of B sequences instead")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.profile:
        run_profile(args)
        return
    if args.layers:
        ap.error("--layers changes the workload: it is for --profile runs only")
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
