"""Benchmark of the decoder forward pass: single-pass prefill + greedy decode at batch 1.

One step = prefill of the workload's prompt (P tokens) followed by D greedy
decode steps, through libdec.so.  ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the baseline arm).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload smollm2-135m] [--kv f32|bf16]
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
    h, f, hd = w["hidden"], w["ffn"], w["head_dim"]
    qd, kd = w["n_heads"] * hd, w["n_kv_heads"] * hd
    k = w["n_experts_used"] if w["n_experts"] else 1
    return {
        "qkv": (qd + 2 * kd) * h * es,
        "oproj": h * qd * es,
        "gateup": k * 2 * f * h * es,
        "down": k * h * f * es,
        "router": w["n_experts"] * h * es,
        "lmhead": w["vocab"] * h * es,
        "embed_row": h * es,
    }


# DRAM bytes per launch of a roofline kernel, from one ncu capture each (the
# summaries under profiles/ give the commands).  A figure holds only for the
# kernel source it measured: the source file's SHA-256 at capture time must
# match the current file, else the bench reports traffic as null.
TRAFFIC = {
    ("smollm2-135m", "down"): {
        "bytes": 1814336, "source": "decoder_only_forward_gb300/csrc/decode.cu",
        "sha256": "3d7213fecd5001252701110382d8e9dfd57676011ecc1ded9bf6666198c7ae34",
        "profile": "profiles/gemv_down_smollm2-135m_traffic.md"},
    ("mistral-7b", "step"): {
        "bytes": 15712395008, "source": "decoder_only_forward_gb300/csrc/decode_mk.cu",
        "sha256": "4bf7258819f5eaeff409afa95ceaa4deb2af4270224b2c6b5de9309906a0eb17",
        "profile": "profiles/decode_step_traffic_mistral-7b.md"},
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
def oracle_sample(w: dict, n_prefill: int, n_decode: int, device: str):
    """Times the float64 oracle on a bounded sample: batched single-pass prefill of
    n_prefill tokens + n_decode per-token forwards.  Returns (tok/s, seconds, cores)."""
    from oracle import OracleConfig, Session
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    src = synthetic.OracleWeightSource(w, device=device, cache=True)
    sess = Session(OracleConfig.from_dict(w), src)
    toks = synthetic.prompt_tokens(w, n_prefill + n_decode, seed=0)
    # Warm the float64 weight copies (drawing them is input generation, not the oracle).
    for l in range(w["n_layers"]):
        src.layer(l)
        if w["n_experts"]:
            for e in range(w["n_experts"]):
                src.expert(l, e)
    src.lm_head()
    src.out_norm()
    t0 = time.perf_counter()
    sess.prefill_batched(list(toks[:n_prefill]), 0)
    for i in range(n_decode):
        sess.forward(int(toks[n_prefill + i]), n_prefill + i)
    dt = time.perf_counter() - t0
    return (n_prefill + n_decode) / dt, dt, cores


def oracle_sample_size(w: dict):
    big = w["hidden"] >= 2048
    return (8, 1) if big else (48, 2)


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    from decoder_only_forward_gb300 import build as dec_build
    if rank == 0:
        dec_build.build()
    if world > 1:
        torch.distributed.barrier()
    dec_build.build()
    from decoder_only_forward_gb300 import dec

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workload_of(args)
    P, D = w["prompt"], w["decode"]
    kv_es = kv_bytes_per_element(w, args.kv)
    d = dec.Decoder(w, device=dev, kv_dtype=args.kv)
    if args.fused != "auto":
        d.set_fused(args.fused)
    s = d.stream
    prompt_np = synthetic.prompt_tokens(w, P, seed=0)
    prompt_pinned = torch.from_numpy(prompt_np).pin_memory()
    V = w["vocab"]
    logits = torch.empty(V, dtype=torch.float32, device=dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    flush = torch.empty(max(2 * L2_BYTES, 256 * 2**20) // 4, dtype=torch.float32, device=dev)

    def step():
        d.kv_reset()  # each step is a new sequence
        d.prefill(prompt_np, 0, logits, tok)
        for i in range(D):
            d.decode_dev(tok, P + i, logits, tok)

    def timed_step(evs):
        with torch.cuda.stream(s):
            flush.zero_()
        evs[0].record(s)
        d.kv_reset()  # each step is a new sequence
        d.prefill(prompt_np, 0, logits, tok)
        evs[1].record(s)
        for i in range(D):
            d.decode_dev(tok, P + i, logits, tok)
        evs[2].record(s)

    for _ in range(args.warmup):
        step()
    d.check()
    torch.cuda.synchronize(dev)

    # ---- timed region (device clocks) ----
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches0 = d.launch_count
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for k in range(args.steps):
            timed_step(events[k])
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
    ms_per_step = tot_ms / args.steps
    pre_s, dec_s = pre_sum / args.steps / 1e3, dec_sum / args.steps / 1e3

    hbm, tf, tf_sus, peak_kind = peaks()
    dbytes = sum(decode_bytes(w, P + i, kv_es) for i in range(D))
    pflops = prefill_flops(w, P)

    # ---- end to end through the public API with host buffers ----
    tok_host = torch.empty(1, dtype=torch.int32).pin_memory()
    logits_host = torch.empty(V, dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.steps, 3))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
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
    e2e_s = (time.perf_counter() - t0) / e2e_steps

    # ---- attribution: which kernel class dominates, and its roofline ----
    classes = ["step", "gateup", "down", "qkv", "oproj", "attn", "lmhead", "router"]
    per_class = {}
    for c in classes:
        d.timing_enable(c, 20000)
        d.kv_reset()  # each step is a new sequence
        d.prefill(prompt_np, 0, logits, tok)
        ms_pf, n_pf = d.timing_read()
        ms_dc, n_dc = 0.0, 0
        for i in range(D):
            d.decode_dev(tok, P + i, logits, tok)
            a, b = d.timing_read()
            ms_dc += a
            n_dc += b
        per_class[c] = dict(prefill_ms=ms_pf, prefill_launches=n_pf, decode_ms=ms_dc, decode_launches=n_dc)
    d.timing_enable("gateup", 0)
    dom = max(classes, key=lambda c: per_class[c]["prefill_ms"] + per_class[c]["decode_ms"])
    pc = per_class[dom]
    nl = pc["decode_launches"] + pc["prefill_launches"]
    wb = weight_bytes(w)
    if dom == "step":
        # The whole decode step is one kernel: its bytes are the step's weights + KV.
        per_launch_bytes = dbytes / D
    elif dom == "attn":
        per_launch_bytes = sum(2 * w["n_kv_heads"] * w["head_dim"] * kv_es *
                               (min(p + 1, w["max_seq"]) if w["sliding_window"] else p + 1)
                               for p in range(P + D)) / (P + D)
    else:
        per_launch_bytes = wb[dom] + 4 * w["hidden"] * 2
    avg_launch_s = (pc["prefill_ms"] + pc["decode_ms"]) / max(nl, 1) / 1e3
    achieved = per_launch_bytes / avg_launch_s / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": measured_traffic(args.workload, dom),
                "peak_kind": peak_kind,
                "bytes_per_launch": int(per_launch_bytes), "avg_launch_us": round(avg_launch_s * 1e6, 3),
                "launches_per_step": nl}

    out = None
    if rank == 0:
        n, k_steps = world, args.steps
        tokens_per_step = P + D
        value = replica_value(n, tokens_per_step, ms_per_step)
        cpu = None
        if not args.no_cpu_baseline:
            npf, ndc = oracle_sample_size(w)
            cv, secs, cores = oracle_sample(w, npf, ndc, device=str(dev))
            cpu = {"value": round(cv, 3), "unit": "tok/s", "cores": cores, "kind": "oracle",
                   "sample": f"float64 oracle: batched single-pass prefill of {npf} prompt tokens + {ndc} "
                             f"per-token forwards of the same {args.workload}-shaped model "
                             f"(weights preloaded as float64), {secs:.1f} s"}
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": n, "steps": k_steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"] if w["dtype"] != "f32" else "f32",
            "data": "synthetic (random-init weights N(0,0.02), norms 1+N(0,0.1), uniform random prompt)",
            "config": {"workload": args.workload + (f"+qk_norm_{args.qk_norm}" if args.qk_norm else "")
                       + ("+sandwich" if args.sandwich else ""), "prompt_tokens": P, "decode_tokens": D, "batch": 1,
                       "decode_schedule": d.fused_mode(),
                       "kv_dtype": args.kv, "weights_gb": round(d.weights.nbytes() / 1e9, 3),
                       "l2": "flushed before each step (write of a 258 MB buffer); weights also exceed L2",
                       "parallelism": f"replicas x{n}" if n > 1 else "single GPU"},
            "prefill": {"tok_s": round(n * P / pre_s, 1), "ms": round(pre_s * 1e3, 4),
                        "flops": pflops, "tensor_frac": round(pflops / pre_s / (tf * 1e12), 5),
                        "tensor_frac_sustained": round(pflops / pre_s / (tf_sus * 1e12), 5)},
            "decode": {"tok_s": round(n * D / dec_s, 1), "ms": round(dec_s * 1e3, 4),
                       "bytes_per_token_avg": round(dbytes / D), "hbm_frac": round(dbytes / dec_s / (hbm * 1e9), 4),
                       "hbm_frac_nominal_8tbs": round(dbytes / dec_s / (NOMINAL_HBM_GBS * 1e9), 4)},
            "clocks": clk.summary(),
            "e2e": {"value": round(n * tokens_per_step / e2e_s, 2), "unit": "tok/s",
                    "h2d_bytes_per_step": 4 * P, "d2h_bytes_per_step": 4 * D + 4 * V,
                    "note": "pinned prompt copied in by dec_prefill; each greedy token read back to the host; "
                            "final logits read back"},
            "gpu_launches": int(launches / args.steps) * args.steps,
            "gpu_launches_per_step": int(launches / args.steps),
            "roofline": roofline,
            "kernel_classes_ms_per_step": {c: round(v["prefill_ms"] + v["decode_ms"], 4) for c, v in per_class.items()},
            "cpu_baseline": cpu,
            "wall_s_timed": round(wall, 3),
        }
    if rank == 0 and args.batch > 0:
        out["batched_decode"] = run_batched(args, w, d.weights, dev, kv_es)
    d.close()
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
    w = workload_of(args)
    npf, ndc = oracle_sample_size(w)
    dev = "cpu"
    rates, secs = [], []
    cores = len(os.sched_getaffinity(0))
    for i in range(args.warmup + args.steps):
        r, s_, cores = oracle_sample(w, npf, ndc, device=dev)
        if i >= args.warmup:
            rates.append(r)
            secs.append(s_)
    value = (npf + ndc) * len(secs) / sum(secs)
    sample = (f"float64 oracle on {cores} host cores: batched single-pass prefill of {npf} prompt tokens + "
              f"{ndc} per-token forwards of the {args.workload}-shaped model per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(secs) / len(secs), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "prompt_tokens": npf, "decode_tokens": ndc, "batch": 1},
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
    ap.add_argument("--workload", default="smollm2-135m", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--kv", default="f32", choices=["f32", "bf16", "i8"])
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
