#!/usr/bin/env python3
"""Benchmark of the batched multi-session decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {dsb,reference}]
                    [--workload llama-68m|qwen3-14b] [--b B] [--T T]

Default workload: the llama-68m-shaped decode step (hidden 768, 12 heads,
head_dim 64, 2 layers, FFN 3072, vocab 32000, fp16 KV cache of
full_batch_size 8 at ctx 2048, seq_lens uniform in [128, 2048]) with a live
batch of b = 8 sessions advancing one token each -- the largest point of the
b in {1, 2, 4, 8} sweep the QAIC page runs on llama-68m.  Weights are random
N(0, 0.02) q8_0 of that shape (no trained weights), drawn on the device and
quantised by the library's own kernel.

One "step" is one replay of the captured decode-step graph (every kernel of
the hot path: embedding, RMSNorm+q8_0, narrow q8_0 matmuls, pos-vector RoPE,
KV write through batch_index, split-K attention + merge, SiLU-gate, head).
L2 is flushed (a 512 MiB write) before every timed step and each step is
timed on its stream with CUDA events.  Prints ONE JSON line on rank 0.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (sessions are independent: weak scaling, no collective on the
data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- distributed
def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _maybe_init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 100 ms; the
    summary keeps the samples stamped inside the region (between __enter__
    returning and __exit__), or all of them if the region was too short to
    catch one (``in_region`` says which)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 100

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_start = self.t_end = None

    def __enter__(self):
        import datetime
        fd, self.path = tempfile.mkstemp(prefix="dsb_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.2)
        self.t_start = datetime.datetime.now()
        return self

    def __exit__(self, *exc):
        import datetime
        self.t_end = datetime.datetime.now()
        time.sleep(2.0 * self.INTERVAL_MS / 1000.0)   # let a sample stamped before t_end reach the file
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def _stamp(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt)
            except ValueError:
                pass
        return None

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10 and parts[2].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0, "in_region": False}
        inside = [r for r in rows if self.t_start is not None and self.t_end is not None and
                  (lambda t: t is not None and self.t_start <= t <= self.t_end)(self._stamp(r[0]))]
        use = inside or rows
        sm = [float(r[2]) for r in use]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(use[0][3]), "reasons": reasons,
                "samples": len(use), "in_region": bool(inside)}


# ----------------------------------------------------------------- workloads
def _shape(name):
    from session_decode_step_dsb_gb300 import workloads
    return {"llama-68m": workloads.LLAMA68M, "llama-68m-spec": workloads.LLAMA68M_SPEC,
            "qwen3-14b": workloads.QWEN3_14B}[name]


def _make_model(ms, seed: int):
    """Random N(0, 0.02) q8_0 weights of the shape, drawn on the device and
    quantised by the library's kernel; caches N(0, 1) in the cache dtype."""
    import torch
    from session_decode_step_dsb_gb300 import dsb
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)

    def q8(rows, cols):
        out = torch.empty((rows, cols // 32 * 34), dtype=torch.uint8, device="cuda")
        step = max(1, (1 << 26) // cols)   # bound the float32 staging to 256 MiB
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            w = torch.randn((r1 - r0, cols), generator=g, device="cuda") * 0.02
            dsb.quantize_q8_0(w, out[r0:r1])
        return out

    w = {"wqkv": [], "wo": [], "wgu": [], "wdown": [], "attn_norm": [], "ffn_norm": []}
    for _ in range(ms.n_layers):
        w["wqkv"].append(q8(ms.qkv_rows, ms.hidden))
        w["wo"].append(q8(ms.hidden, ms.n_q_heads * ms.head_dim))
        w["wgu"].append(q8(2 * ms.ffn, ms.hidden))
        w["wdown"].append(q8(ms.hidden, ms.ffn))
        w["attn_norm"].append(torch.ones(ms.hidden, device="cuda"))
        w["ffn_norm"].append(torch.ones(ms.hidden, device="cuda"))
    w["embed"] = q8(ms.vocab, ms.hidden)
    w["head"] = q8(ms.vocab, ms.hidden)
    w["final_norm"] = torch.ones(ms.hidden, device="cuda")
    if ms.qk_norm:
        w["q_norm"] = [torch.ones(ms.head_dim, device="cuda") for _ in range(ms.n_layers)]
        w["k_norm"] = [torch.ones(ms.head_dim, device="cuda") for _ in range(ms.n_layers)]
    cdt = torch.float16 if ms.cache_dtype == "f16" else torch.bfloat16
    kc, vc = [], []
    for _ in range(ms.n_layers):
        shape = (ms.full_batch_size, ms.n_kv_heads, ms.ctx, ms.head_dim)
        kc.append(torch.randn(shape, generator=g, device="cuda").to(cdt).view(torch.int16))
        vc.append(torch.randn(shape, generator=g, device="cuda").to(cdt).view(torch.int16))
    model = dsb.DecodeModel(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, w,
                            kc, vc, 0 if ms.cache_dtype == "f16" else 1, ms.eps, ms.theta)
    return model


def _meta(ms, b, T, seed):
    from session_decode_step_dsb_gb300 import synth
    sid = synth.stream_id
    bi = synth.distinct_slots(seed, sid(synth.STREAM_META, 1), b, ms.full_batch_size)
    lens = synth.uniform_int(seed, sid(synth.STREAM_META, 2), max(128, T), ms.ctx, b)
    toks = synth.uniform_int(seed, sid(synth.STREAM_TOKENS, 0), 0, ms.vocab - 1, b * T)
    return bi, lens, toks


def step_bytes(ms, b, T, lens):
    """Algorithmic HBM bytes of one step: every q8_0 weight byte once, plus the
    K and V bytes attention must read (each kv head's rows once for its G*T
    query rows), plus the embedding rows and the logits."""
    nb = lambda cols: cols // 32 * 34
    per_layer = (ms.qkv_rows * nb(ms.hidden) + ms.hidden * nb(ms.n_q_heads * ms.head_dim) +
                 2 * ms.ffn * nb(ms.hidden) + ms.hidden * nb(ms.ffn))
    weights = ms.n_layers * per_layer + ms.vocab * nb(ms.hidden)
    e = 2
    kv = ms.n_layers * int(np.sum(lens)) * ms.n_kv_heads * ms.head_dim * 2 * e
    io = b * T * (nb(ms.hidden) + 4 * ms.vocab)
    return weights + kv + io, weights, kv


# ----------------------------------------------------------------- timing helpers
# GPU cycles of busy-wait enqueued before each start event, so that the host
# (Python, ctypes, argument checks, graph launch) has enqueued the timed work
# before the device reaches it: the events then bracket device time only.
HOST_SLACK_CYCLES = 200_000


def _time_device(fn, iters, flush, stream):
    """Median and mean device time (ms) of fn(), L2 flushed before each call."""
    import torch
    ts = []
    for _ in range(iters):
        flush.zero_()
        torch.cuda._sleep(HOST_SLACK_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts), sum(ts) / len(ts), ts


MATMUL_SHAPES = [(7168, 7168), (18432, 7168), (129280, 7168)]
MATMUL_NTOK = [1, 2, 3, 4, 8, 16]


def matmul_sweep(flush, stream, peak, iters=5):
    """Narrow q8_0 matmul GB/s on the DeepSeek-class dense-stage shapes at
    every n_tok the method targets (algorithmic bytes: weights once + q8_0
    activations + float32 outputs)."""
    import torch
    from session_decode_step_dsb_gb300 import dsb
    out = []
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    for rows, cols in MATMUL_SHAPES:
        w = torch.empty((rows, cols // 32 * 34), dtype=torch.uint8, device="cuda")
        step = max(1, (1 << 26) // cols)
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            dsb.quantize_q8_0(torch.randn((r1 - r0, cols), generator=g, device="cuda") * 0.02, w[r0:r1])
        x = dsb.quantize_q8_0(torch.randn((16, cols), generator=g, device="cuda"))
        for nt in MATMUL_NTOK:
            xs = x[:nt].contiguous()
            y = torch.empty((nt, rows), device="cuda")
            for _ in range(2):
                dsb.matmul_q8_0_narrow(w, rows, cols, xs, nt, y)
            med, mean, _ = _time_device(lambda: dsb.matmul_q8_0_narrow(w, rows, cols, xs, nt, y), iters, flush, stream)
            byts = 34 * rows * (cols // 32) + 34 * nt * (cols // 32) + 4 * nt * rows
            gbs = byts / (med * 1e-3) / 1e9
            out.append({"rows": rows, "cols": cols, "n_tok": nt, "us": round(med * 1e3, 2), "gbs": round(gbs, 1),
                        "frac": round(gbs / peak, 4)})
        del w, x
    return out


ATTN_CTX = [32768, 65536]


def attention_sweep(flush, stream, peak, iters=5):
    """Split-K decode attention on the long-context shapes (128 query and 128
    kv heads, head_dim 128, fp16 cache of full_batch_size 8), b = 1..4,
    seq_lens uniform in [16384, ctx]: GB/s over the K and V bytes it must read
    (each kv head's rows once) plus q, out and the split-K partials."""
    import torch
    from session_decode_step_dsb_gb300 import dsb, synth
    out = []
    F, H, D = 8, 128, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(99)
    for C in ATTN_CTX:
        kc = torch.empty((F, H, C, D), dtype=torch.float16, device="cuda")
        vc = torch.empty((F, H, C, D), dtype=torch.float16, device="cuda")
        for f in range(F):
            kc[f].normal_(generator=g)
            vc[f].normal_(generator=g)
        kv = dsb.kv_cache(kc.view(torch.int16), vc.view(torch.int16), dsb.DSB_F16)
        ws = dsb.Workspace(4, H, D, C)
        for b in (1, 2, 4):
            bi = synth.distinct_slots(5, synth.stream_id(synth.STREAM_META, 7), b, F)
            lens = synth.uniform_int(5, synth.stream_id(synth.STREAM_META, 8), 16384, C, b)
            q = torch.randn((b, H, D), generator=g, device="cuda")
            o = torch.empty_like(q)
            for _ in range(2):
                dsb.attention_decode_multi(q, kv, bi, 1, lens, ws, out=o)
            med, mean, _ = _time_device(lambda: dsb.attention_decode_multi(q, kv, bi, 1, lens, ws, out=o), iters,
                                        flush, stream)
            chunks = int(np.sum((lens + 127) // 128))
            byts = int(np.sum(lens)) * H * D * 2 * 2 + 2 * b * H * D * 4 + 2 * chunks * H * (D + 2) * 4
            gbs = byts / (med * 1e-3) / 1e9
            out.append({"ctx": C, "b": b, "seq_lens": [int(v) for v in lens], "us": round(med * 1e3, 1),
                        "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)})
        del kc, vc, kv, ws
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- dsb arm
def run_dsb(args):
    import torch
    from session_decode_step_dsb_gb300 import dsb
    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dist = _maybe_init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    ms = _shape(args.workload)
    b, T = args.b, args.T
    peak, peak_kind = _peaks()

    model = _make_model(ms, seed=1000 + rank)
    bi, lens, toks = _meta(ms, b, T, seed=7 + rank)
    n_tok = b * T
    ws = model.workspace(max(n_tok, 8))
    logits = torch.empty((n_tok, ms.vocab), dtype=torch.float32, device=dev)
    graph = model.graph(b, T, logits, ws)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    step = lambda: graph.launch(toks, bi, lens)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dsb.device_error()

    # ---- timed region: K steps, each after an L2 flush, device-timed
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        med, mean, ts = _time_device(step, args.steps, flush, stream)
    torch.cuda.synchronize()
    _barrier(dist)
    clocks = clk.summary()
    ms_step = _max_over_ranks(dist, mean, dev)
    dsb.device_error()

    # ---- b sweep (same model, fresh graphs), tokens/s per b
    sweep = {}
    b_list = {"llama-68m": (1, 2, 4, 8), "llama-68m-spec": (1, 4, 16, 64, 128),
              "qwen3-14b": (1, 2, 3, 4, 5, 8, 15, 16)}[args.workload]
    if world == 1 and T == 1:
        for bb in b_list:
            bi2, lens2, toks2 = _meta(ms, bb, 1, seed=7)
            lg = torch.empty((bb, ms.vocab), dtype=torch.float32, device=dev)
            g2 = model.graph(bb, 1, lg, ws)
            for _ in range(3):
                g2.launch(toks2, bi2, lens2)
            m2, mean2, _ = _time_device(lambda: g2.launch(toks2, bi2, lens2), 20, flush, stream)
            sweep[str(bb)] = {"ms_per_step": round(mean2, 4), "tokens_per_s": round(bb / (mean2 * 1e-3), 1)}
            g2.close()

    # ---- dominant kernel roofline: the narrow q8_0 matmul.  Its launches in
    # the step (the workload's own matrices at n_tok = b*T) are timed one by
    # one with CUDA events on the launching stream, L2 flushed before each.
    nbk = lambda cols: cols // 32 * 34
    mats = [(ms.qkv_rows, ms.hidden, model.w["wqkv"][0]), (ms.hidden, ms.n_q_heads * ms.head_dim, model.w["wo"][0]),
            (2 * ms.ffn, ms.hidden, model.w["wgu"][0]), (ms.hidden, ms.ffn, model.w["wdown"][0]),
            (ms.vocab, ms.hidden, model.w["head"])]
    tot_bytes = 0.0
    tot_ms = 0.0
    per_kernel = []
    nt = min(n_tok, 16)
    for rows, cols, wmat in mats:
        x = dsb.quantize_q8_0(torch.randn((nt, cols), device=dev))
        y = torch.empty((nt, rows), device=dev)
        for _ in range(2):
            dsb.matmul_q8_0_narrow(wmat, rows, cols, x, nt, y)
        m_, mean_, _ = _time_device(lambda: dsb.matmul_q8_0_narrow(wmat, rows, cols, x, nt, y), 10, flush, stream)
        byts = rows * nbk(cols) + nt * nbk(cols) + 4 * nt * rows
        reps = ms.n_layers if rows != ms.vocab else 1
        tot_bytes += byts * reps
        tot_ms += mean_ * reps
        per_kernel.append({"rows": rows, "cols": cols, "n_tok": nt, "us": round(mean_ * 1e3, 2),
                           "gbs": round(byts / (mean_ * 1e-3) / 1e9, 1)})
    achieved = tot_bytes / (tot_ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            traffic = json.load(f).get(f"{args.workload}:b{b}:T{T}")
    except Exception:
        traffic = None

    sweep_mm = matmul_sweep(flush, stream, peak) if (world == 1 and not args.no_matmul_sweep) else []
    sweep_attn = attention_sweep(flush, stream, peak) if (world == 1 and args.attn_sweep) else []

    # ---- end to end through the C ABI with host buffers: token ids, slots
    # and lengths from host arrays (staged by the library), logits copied back
    # to pinned host memory, every step inside the timed region.
    host_logits = torch.empty((n_tok, ms.vocab), dtype=torch.float32, pin_memory=True)
    e2e_steps = max(10, min(args.steps, 100))
    for _ in range(3):
        graph.launch(toks, bi, lens)
        host_logits.copy_(logits, non_blocking=True)
    torch.cuda.synchronize()
    _barrier(dist)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        graph.launch(toks, bi, lens)
        host_logits.copy_(logits, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = _max_over_ranks(dist, e2e_s, dev)
    meta_words = 2 * n_tok + 3 * b + 1
    e2e = {"value": round(world * n_tok / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 4 * meta_words,
           "d2h_bytes_per_step": 4 * n_tok * ms.vocab, "steps": e2e_steps,
           "note": "host int32 token ids/slots/seq_lens staged by the library; logits copied to pinned host"}

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "llama-68m":
        cpu = cpu_baseline(ms, b, T, budget_s=args.cpu_budget)
        cpu["cpu"] = _cpu_model()
        if args.cpu_all_core_budget > 0:
            cpu["all_cores"] = cpu_all_cores(args.workload, b, T, budget_s=args.cpu_all_core_budget)

    graph.close()
    total_bytes, wbytes, kvbytes = step_bytes(ms, b, T, lens)
    value = world * n_tok / (ms_step * 1e-3)
    if rank == 0:
        line = {
            "metric": "decode-step tokens/s and q8_0 narrow-matmul HBM GB/s (% of peak), n_tok=1..16",
            "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": f"int8xint8->int32 dot (q8_0), f32 accumulate; {ms.cache_dtype} KV",
            "data": "synthetic (seeded random weights/caches of the workload's shapes; no trained weights)",
            "config": {"workload": ms.name, "b": b, "tokens_per_seq": T, "n_tok": n_tok,
                       "full_batch_size": ms.full_batch_size, "ctx": ms.ctx, "seq_lens": [int(v) for v in lens],
                       "layers": ms.n_layers, "hidden": ms.hidden, "vocab": ms.vocab,
                       "l2": "flushed (512 MiB write) before every timed step", "parallelism": f"replicas x{world}",
                       "step_bytes": total_bytes, "weight_bytes": wbytes, "kv_bytes": kvbytes},
            "step_ms": {"p50": round(float(np.percentile(ts, 50)), 5), "p90": round(float(np.percentile(ts, 90)), 5),
                        "p95": round(float(np.percentile(ts, 95)), 5), "mean": round(float(mean), 5)},
            "step_roofline": {"bytes": total_bytes, "achieved_gbs": round(total_bytes / (ms_step * 1e-3) / 1e9, 1),
                              "peak_gbs": peak, "frac": round(total_bytes / (ms_step * 1e-3) / 1e9 / peak, 4)},
            "roofline": {"kernel": "matmul_q8_0_narrow_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "per": f"one step's matmul launches ({ms.n_layers} layers x 4 + head)",
                         "algorithmic_bytes": int(tot_bytes),
                         "peak_kind": f"{peak_kind} hbm_gbs", "launches": per_kernel},
            "b_sweep": sweep,
            "matmul_q8_0_narrow": sweep_mm,
            "attention_long_context": sweep_attn,
            "e2e": e2e,
            "gpu_launches": None,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        line["gpu_launches"] = args.steps * launches_per_step(ms)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def launches_per_step(ms) -> int:
    """Kernels of one step: embed + per layer (rmsnorm-q8, QKV, RoPE+KV write,
    attention partial, merge-q8, O, rmsnorm-q8, gate|up, silu-q8, down) +
    final rmsnorm-q8 + head."""
    return 1 + 10 * ms.n_layers + 2


# ----------------------------------------------------------------- CPU oracle
def _oracle_model(ms, seed):
    from oracle import q8_0 as oq
    from session_decode_step_dsb_gb300 import synth
    sid = synth.stream_id
    w = {"wqkv": [], "wo": [], "wgu": [], "wdown": []}
    for l in range(ms.n_layers):
        w["wqkv"].append(oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * l), ms.qkv_rows, ms.hidden, 0.02)))
        w["wo"].append(oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * l + 1), ms.hidden, ms.n_q_heads * ms.head_dim, 0.02)))
        w["wgu"].append(oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * l + 2), 2 * ms.ffn, ms.hidden, 0.02)))
        w["wdown"].append(oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_W, 10 * l + 3), ms.hidden, ms.ffn, 0.02)))
    w["head"] = oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_W, 999_000), ms.vocab, ms.hidden, 0.02))
    w["embed"] = oq.quantize_rows(synth.normal_rows(seed, sid(synth.STREAM_EMBED, 0), ms.vocab, ms.hidden, 0.02))
    w["attn_norm"] = [np.ones(ms.hidden, np.float32)] * ms.n_layers
    w["ffn_norm"] = [np.ones(ms.hidden, np.float32)] * ms.n_layers
    w["final_norm"] = np.ones(ms.hidden, np.float32)
    if ms.qk_norm:
        w["q_norm"] = [np.ones(ms.head_dim, np.float32)] * ms.n_layers
        w["k_norm"] = [np.ones(ms.head_dim, np.float32)] * ms.n_layers
    dims = (ms.full_batch_size, ms.n_kv_heads, ms.ctx, ms.head_dim)
    kc = [synth.cache_bits(seed, sid(synth.STREAM_KCACHE, l), dims, ms.cache_dtype) for l in range(ms.n_layers)]
    vc = [synth.cache_bits(seed, sid(synth.STREAM_VCACHE, l), dims, ms.cache_dtype) for l in range(ms.n_layers)]
    return w, kc, vc


def cpu_baseline(ms, b, T, budget_s=20.0):
    """The oracle's decode step (numpy, float64) timed on the host: one
    sequence of the b-sequence batch per sample (a bounded sample of the same
    workload), repeated until ~budget_s of CPU work."""
    from oracle import step as ostep
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    w, kc, vc = _oracle_model(ms, seed=0)
    bi, lens, toks = _meta(ms, b, T, seed=7)
    shape = ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, ms.eps,
                        ms.theta)
    n = 0
    t0 = time.perf_counter()
    while True:
        s = n % b
        ostep.decode_step(shape, w, kc, vc, ms.cache_dtype, toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * T / dt, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} single-sequence steps (1 of the {b} sessions each, {T} token(s)) of the {ms.name} "
                      f"workload, float64 numpy, {dt:.1f} s"}


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer / part codes), with the machine type."""
    import platform
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.startswith(key):
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                if key == "CPU part":
                    name = "Arm CPU part " + name
                break
    except OSError:
        pass
    return f"{name or 'unknown'} ({platform.machine()})"


def _oracle_worker(workload, b, T, budget_s, worker, start, ready, results):
    """One process of the all-core oracle run: builds the oracle model, reports
    ready, waits for the common start, then runs single-sequence oracle steps
    (sessions taken in turn from worker onwards) for budget_s seconds."""
    from oracle import step as ostep
    ms = _shape(workload)
    w, kc, vc = _oracle_model(ms, seed=0)
    bi, lens, toks = _meta(ms, b, T, seed=7)
    shape = ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, ms.eps,
                        ms.theta)
    ready.put(worker)
    start.wait(600)
    n = 0
    t0 = time.perf_counter()
    while True:
        s = (worker + n) % b
        ostep.decode_step(shape, w, kc, vc, ms.cache_dtype, toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    results.put((n, time.perf_counter() - t0))


def cpu_all_cores(workload, b, T, budget_s=8.0, max_workers=16):
    """The same oracle step on every host core at once: one spawned process
    per core (BLAS threads 1 each), all starting together after building
    their model; throughput = all steps' tokens / the longest process time."""
    import multiprocessing as mp
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    n = max(1, min(cores, max_workers))
    ctx = mp.get_context("spawn")
    start, ready, results = ctx.Event(), ctx.Queue(), ctx.Queue()
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
    os.environ["OMP_NUM_THREADS"] = os.environ["OPENBLAS_NUM_THREADS"] = "1"
    procs = [ctx.Process(target=_oracle_worker, args=(workload, b, T, budget_s, i, start, ready, results))
             for i in range(n)]
    try:
        for p in procs:
            p.start()
        for _ in procs:
            ready.get(timeout=600)
        start.set()
        res = [results.get(timeout=budget_s + 600) for _ in procs]
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    steps = sum(r[0] for r in res)
    dt = max(r[1] for r in res)
    return {"value": round(steps * T / dt, 3), "unit": "tokens/s", "cores": n, "host_cores": cores,
            "sample": f"{steps} single-sequence oracle steps over {n} processes in {dt:.1f} s"}


def run_reference(args):
    """The oracle timed as the reference arm: each step is one single-sequence
    oracle decode step of the workload (a bounded sample of the b-sequence
    step), on the host cores."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    from oracle import step as ostep
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    ms = _shape(args.workload)
    b, T = args.b, args.T
    if args.workload != "llama-68m":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm is timed on the llama-68m-shaped step; "
                          "drawing and quantising 40 Qwen3-14B-shaped layers in numpy takes tens of minutes"}))
        return
    w, kc, vc = _oracle_model(ms, seed=0)
    bi, lens, toks = _meta(ms, b, T, seed=7)
    shape = ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers, ms.eps,
                        ms.theta)

    def one(i):
        s = i % b
        ostep.decode_step(shape, w, kc, vc, ms.cache_dtype, toks[s * T:(s + 1) * T], bi[s:s + 1], T, lens[s:s + 1])

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    value = args.steps * T / dt
    line = {"impl": "reference", "metric": "decode-step tokens/s and q8_0 narrow-matmul HBM GB/s (% of peak), n_tok=1..16",
            "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": ms.name, "b": b, "tokens_per_seq": T,
                       "sample": f"one of the {b} sessions per step ({T} token(s))"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} single-sequence oracle steps of the {ms.name} workload"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PROBE_ATTENTION = {  # F, Hq, Hkv, ctx, D, cache dtype, b, T, shortest seq_len
    "qwen3-14b": (16, 40, 8, 4096, 128, 1, 16, 1, 1),
    "llama-68m": (8, 12, 12, 2048, 64, 0, 8, 1, 128),
}


def run_probe(spec: str):
    """A few launches of one kernel at one shape, for a profiler to capture
    (no timing, no JSON line): ``matmul:ROWS:COLS:NTOK[,NTOK...]`` runs the
    narrow matmul three times per n_tok on N(0, 0.02) weights;
    ``wide:ROWS:COLS:NTOK`` the tensor-core matmul three times;
    ``attention:WORKLOAD`` runs the decode attention four times on that
    workload's cache shape (b sequences, seq_lens uniform)."""
    import torch
    from session_decode_step_dsb_gb300 import dsb
    kind, *rest = spec.split(":")
    g = torch.Generator(device="cuda")
    g.manual_seed(4321)
    if kind == "matmul":
        rows, cols, nts = int(rest[0]), int(rest[1]), [int(v) for v in rest[2].split(",")]
        w = dsb.quantize_q8_0(torch.randn((rows, cols), generator=g, device="cuda") * 0.02)
        x = dsb.quantize_q8_0(torch.randn((16, cols), generator=g, device="cuda"))
        for nt in nts:
            xs = x[:nt].contiguous()
            for _ in range(3):
                dsb.matmul_q8_0_narrow(w, rows, cols, xs, nt)
    elif kind == "wide":
        rows, cols, nt = int(rest[0]), int(rest[1]), int(rest[2])
        w = dsb.quantize_q8_0(torch.randn((rows, cols), generator=g, device="cuda") * 0.02)
        x = dsb.quantize_q8_0(torch.randn((nt, cols), generator=g, device="cuda"))
        for _ in range(3):
            dsb.matmul_q8_0_wide(w, rows, cols, x, nt)
    elif kind == "attention":
        F, hq, hkv, C, D, dt, b, T, lo = PROBE_ATTENTION[rest[0]]
        cdt = torch.float16 if dt == 0 else torch.bfloat16
        kc = torch.randn((F, hkv, C, D), generator=g, device="cuda").to(cdt).view(torch.int16)
        vc = torch.randn((F, hkv, C, D), generator=g, device="cuda").to(cdt).view(torch.int16)
        kv = dsb.kv_cache(kc, vc, dt)
        rng = np.random.default_rng(3)
        bi = rng.permutation(F)[:b].astype(np.int32)
        lens = rng.integers(max(lo, T), C + 1, b).astype(np.int32)
        q = torch.randn((b * T, hq, D), generator=g, device="cuda")
        ws = dsb.Workspace(b * T, hq, D, C)
        out = torch.empty_like(q)
        for _ in range(4):
            dsb.attention_decode_multi(q, kv, bi, T, lens, ws, out=out)
    else:
        raise SystemExit(f"unknown probe {spec!r}")
    torch.cuda.synchronize()
    dsb.device_error()
    print("probe ok", spec)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["dsb", "reference"], default="dsb")
    ap.add_argument("--workload", choices=["llama-68m", "llama-68m-spec", "qwen3-14b"], default="llama-68m")
    ap.add_argument("--b", type=int, default=8)
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-all-core-budget", type=float, default=8.0,
                    help="seconds of the all-core oracle run beside the single-core one (0: skip)")
    ap.add_argument("--no-matmul-sweep", action="store_true")
    ap.add_argument("--attn-sweep", action="store_true",
                    help="also time the split-K attention at ctx 32768/65536 (allocates ~70 GB)")
    ap.add_argument("--probe", default=None,
                    help="run one kernel a few times for a profiler and exit: matmul:ROWS:COLS:NTOK[,..], "
                         "wide:ROWS:COLS:NTOK or attention:WORKLOAD")
    args = ap.parse_args(argv)
    if args.probe:
        run_probe(args.probe)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_dsb(args)


if __name__ == "__main__":
    main()
