#!/usr/bin/env python3
"""Benchmark of the batched multi-session decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {dsb,reference}]
                    [--workload qwen3-14b|llama-68m|llama-68m-spec] [--b B] [--T T]

Default workload: the Qwen3-14B-shaped decode step (hidden 5120, 40 query / 8
kv heads, head_dim 128 with the per-head q / k RMS norm, FFN 17408 SiLU-gated,
vocab 151936, 40 layers, bf16 KV cache [16, 8, 4096, 128], seq_lens uniform in
[1, 4096]) with the full live batch b = 16 advancing one token each -- the
largest single-GPU configuration of the method's workloads (the pypto page's
dynamic public batch 1..16).  Weights are random N(0, 0.02) q8_0 of that shape
(no trained weights), drawn on the device and quantised by the library's own
kernel.

One "step" is one replay of the captured decode-step graph (every kernel of
the hot path: embedding, RMSNorm+q8_0, narrow q8_0 matmuls, per-head norm +
pos-vector RoPE + KV write through batch_index, split-K attention + merge,
SiLU-gate, head).  L2 is flushed (a 512 MiB write, then half of it read back,
so no dirty line stays) before every timed step and
each step is timed on its stream with CUDA events.  Prints ONE JSON line on
rank 0; besides the headline it carries the b sweep, the narrow-matmul GB/s
sweep, the long-context attention GB/s, the llama-68m-shaped step and the
b x K speculative grid.

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


def _flush_l2(flush):
    """Evict L2 before a timed call: write the 512 MiB buffer, then read its
    first half back.  The write alone would leave L2 full of the buffer's dirty
    lines, and the timed call would pay for writing them back to HBM as its own
    reads evict them (129 MB: about 19 us of HBM time, a fifth of a small step);
    after the read, every line L2 holds is clean and none is the timed call's."""
    import torch
    flush.zero_()
    torch.count_nonzero(flush[: flush.numel() // 2])


def _time_device(fn, iters, flush, stream):
    """Median and mean device time (ms) of fn(), L2 flushed before each call."""
    import torch
    ts = []
    for _ in range(iters):
        _flush_l2(flush)
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


def matmul_sweep(flush, stream, peak, iters=15):
    """Narrow q8_0 matmul GB/s on the DeepSeek-class dense-stage shapes at
    every n_tok the method targets (algorithmic bytes: weights once + q8_0
    activations + float32 outputs): from q8_0 rows (dsb_matmul_q8_0_narrow)
    and from the staged layout the step's kernels write (staged_*).  Mean of
    the launches: the event clock here ticks in 2.048 us steps, and the mean
    over launches that start at random phases of it resolves below a tick."""
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
            _, t_row, _ = _time_device(lambda: dsb.matmul_q8_0_narrow(w, rows, cols, xs, nt, y), iters, flush, stream)
            byts = 34 * rows * (cols // 32) + 34 * nt * (cols // 32) + 4 * nt * rows
            gbs = byts / (t_row * 1e-3) / 1e9
            # the step's path: the same product from the staged layout
            stg = dsb.stage_q8_0(w, rows, cols, xs, nt)
            dsb.matmul_q8_0_staged(w, rows, cols, stg, nt, y)
            _, t_stg, _ = _time_device(lambda: dsb.matmul_q8_0_staged(w, rows, cols, stg, nt, y), iters, flush, stream)
            gbs_s = byts / (t_stg * 1e-3) / 1e9
            out.append({"rows": rows, "cols": cols, "n_tok": nt, "us": round(t_row * 1e3, 2), "gbs": round(gbs, 1),
                        "frac": round(gbs / peak, 4), "staged_us": round(t_stg * 1e3, 2),
                        "staged_frac": round(gbs_s / peak, 4)})
        del w, x
    return out


WIDE_CASES = [(18432, 7168, 32), (18432, 7168, 128), (18432, 7168, 256), (34816, 5120, 128)]


def wide_sweep(flush, stream, iters=15):
    """The wide q8_0 matmul on the tensor cores (dsb_matmul_q8_0_wide, the
    step's path past 32 token rows) on the DeepSeek-class 18432 x 7168 stage
    and the Qwen3-14B-shaped gate|up matrix: device time per call (mean of the
    launches, L2 flushed before each) and its useful q8_0 work as TOPS-eq
    (2 rows cols n_tok / time)."""
    import torch
    from session_decode_step_dsb_gb300 import dsb
    out = []
    g = torch.Generator(device="cuda")
    g.manual_seed(4321)
    for rows, cols, nt in WIDE_CASES:
        w = torch.empty((rows, cols // 32 * 34), dtype=torch.uint8, device="cuda")
        step = max(1, (1 << 26) // cols)
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            dsb.quantize_q8_0(torch.randn((r1 - r0, cols), generator=g, device="cuda") * 0.02, w[r0:r1])
        x = dsb.quantize_q8_0(torch.randn((nt, cols), generator=g, device="cuda"))
        y = torch.empty((nt, rows), device="cuda")
        scratch, _ = dsb._wide_scratch(nt, cols, w.device)
        for _ in range(2):
            dsb.matmul_q8_0_wide(w, rows, cols, x, nt, y=y, scratch=scratch)
        _, mean, _ = _time_device(lambda: dsb.matmul_q8_0_wide(w, rows, cols, x, nt, y=y, scratch=scratch), iters,
                                  flush, stream)
        out.append({"rows": rows, "cols": cols, "n_tok": nt, "us": round(mean * 1e3, 2),
                    "tops_eq": round(2.0 * rows * cols * nt / (mean * 1e-3) / 1e12, 1)})
        del w, x, y, scratch
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
B_SWEEP = {"llama-68m": (1, 2, 4, 8), "llama-68m-spec": (1, 4, 16, 64, 128),
           "qwen3-14b": (1, 2, 3, 4, 5, 8, 15, 16)}
DEFAULT_B = {"llama-68m": 8, "llama-68m-spec": 16, "qwen3-14b": 16}
# b x K points of the speculative grid (llama-68m shapes, full_batch_size 128,
# T = K + 1 draft tokens per sequence; the QAIC page's batch x K experiment)
SPEC_B = (1, 16, 128)
SPEC_K = (0, 7, 31)


def _step_graph_time(model, ms, b, T, seed, ws, flush, stream, iters, dev):
    """Median and mean device time (ms) of graph replays of one (b, T) step,
    the seq_lens drawn, and the per-replay times."""
    import torch
    bi, lens, toks = _meta(ms, b, T, seed)
    lg = torch.empty((b * T, ms.vocab), dtype=torch.float32, device=dev)
    g = model.graph(b, T, lg, ws)
    for _ in range(3):
        g.launch(toks, bi, lens)
    med, mean, ts = _time_device(lambda: g.launch(toks, bi, lens), iters, flush, stream)
    g.close()
    return med, mean, lens, ts


def llama_step(flush, stream, dev, steps):
    """The llama-68m-shaped step (the QAIC page's decode model) at b = 8 and
    its b sweep {1, 2, 4, 8}, T = 1."""
    import torch
    ms = _shape("llama-68m")
    model = _make_model(ms, seed=2000)
    ws = model.workspace(8)
    out = {"workload": ms.name, "layers": ms.n_layers, "ctx": ms.ctx, "full_batch_size": ms.full_batch_size}
    for b in (1, 2, 4, 8):
        med, mean, lens, _ = _step_graph_time(model, ms, b, 1, 7, ws, flush, stream, steps, dev)
        tb, wb, kb = step_bytes(ms, b, 1, lens)
        out[f"b{b}"] = {"ms_per_step": round(mean, 5), "tokens_per_s": round(b / (mean * 1e-3), 1),
                        "step_frac": round(tb / (mean * 1e-3) / 1e9 / _peaks()[0], 4)}
    del model, ws
    torch.cuda.empty_cache()
    return out


def spec_grid(flush, stream, dev, iters=10):
    """Dynamic batch x speculative decode on the llama-68m shapes with
    full_batch_size 128: tokens/s of the step at b in SPEC_B and K in SPEC_K
    (n_tok = b (K + 1); past 16 token rows the matmuls run on the tensor
    cores)."""
    import torch
    ms = _shape("llama-68m-spec")
    model = _make_model(ms, seed=3000)
    ws = model.workspace(max(SPEC_B) * (max(SPEC_K) + 1))
    out = []
    for b in SPEC_B:
        for K in SPEC_K:
            T = K + 1
            med, mean, _, _ = _step_graph_time(model, ms, b, T, 11, ws, flush, stream, iters, dev)
            out.append({"b": b, "K": K, "n_tok": b * T, "ms_per_step": round(mean, 5),
                        "tokens_per_s": round(b * T / (mean * 1e-3), 1)})
    del model, ws
    torch.cuda.empty_cache()
    return out


def run_dsb(args):
    import torch
    from session_decode_step_dsb_gb300 import dsb
    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dist = _maybe_init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    ms = _shape(args.workload)
    b = args.b if args.b else DEFAULT_B[args.workload]
    T = args.T
    peak, peak_kind = _peaks()

    model = _make_model(ms, seed=1000 + rank)
    bi, lens, toks = _meta(ms, b, T, seed=7 + rank)
    n_tok = b * T
    ws = model.workspace(max(n_tok, max(B_SWEEP[args.workload])))
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
    if world == 1 and T == 1:
        for bb in B_SWEEP[args.workload]:
            _, mean2, lens2, ts2 = _step_graph_time(model, ms, bb, 1, 7, ws, flush, stream, 20, dev)
            tb2, _, _ = step_bytes(ms, bb, 1, lens2)
            sweep[str(bb)] = {"ms_per_step": round(mean2, 4), "tokens_per_s": round(bb / (mean2 * 1e-3), 1),
                              "step_frac": round(tb2 / (mean2 * 1e-3) / 1e9 / peak, 4), "replays": len(ts2),
                              "ms_p50": round(float(np.percentile(ts2, 50)), 4),
                              "ms_p90": round(float(np.percentile(ts2, 90)), 4),
                              "ms_min": round(min(ts2), 4), "ms_max": round(max(ts2), 4)}

    # ---- dominant kernel roofline: the narrow q8_0 matmul, timed as it runs
    # in the step -- the step's own sequence of matmul launches (every layer's
    # matrices in order, then the head, at n_tok = b*T), captured once in a
    # CUDA graph and replayed after an L2 flush, CUDA events on the stream.
    # achieved = algorithmic bytes of the sequence / replay time.  Each shape
    # is also timed alone (L2 flushed before each launch) for reference.
    nbk = lambda cols: cols // 32 * 34
    nt = min(n_tok, 16)
    seq = []
    for l in range(ms.n_layers):
        seq += [(ms.qkv_rows, ms.hidden, model.w["wqkv"][l]), (ms.hidden, ms.n_q_heads * ms.head_dim, model.w["wo"][l]),
                (2 * ms.ffn, ms.hidden, model.w["wgu"][l]), (ms.hidden, ms.ffn, model.w["wdown"][l])]
    seq.append((ms.vocab, ms.hidden, model.w["head"]))
    # the step's matmul path: activations in the staged layout the producing
    # kernels write (staged once here, outside the timed graph)
    acts = {}
    for rows, cols, wmat in seq:
        if (rows, cols) not in acts:
            xq_ = dsb.quantize_q8_0(torch.randn((nt, cols), device=dev))
            acts[(rows, cols)] = (dsb.stage_q8_0(wmat, rows, cols, xq_, nt), torch.empty((nt, rows), device=dev))
    for rows, cols, wmat in seq:   # warm every launch's host caches before capture
        x, y = acts[(rows, cols)]
        dsb.matmul_q8_0_staged(wmat, rows, cols, x, nt, y)
    torch.cuda.synchronize()
    mm_graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(mm_graph, stream=cap_stream):
            for rows, cols, wmat in seq:
                x, y = acts[(rows, cols)]
                dsb.matmul_q8_0_staged(wmat, rows, cols, x, nt, y)
    stream.wait_stream(cap_stream)
    torch.cuda.synchronize()
    for _ in range(2):
        mm_graph.replay()
    _, mm_mean, _ = _time_device(mm_graph.replay, 10, flush, stream)
    tot_bytes = float(sum(rows * nbk(cols) + nt * nbk(cols) + 4 * nt * rows for rows, cols, _ in seq))
    achieved = tot_bytes / (mm_mean * 1e-3) / 1e9
    del mm_graph
    per_kernel = []
    for rows, cols, wmat in seq[:4] + seq[-1:]:
        x, y = acts[(rows, cols)]
        m_, mean_, _ = _time_device(lambda: dsb.matmul_q8_0_staged(wmat, rows, cols, x, nt, y), 10, flush, stream)
        byts = rows * nbk(cols) + nt * nbk(cols) + 4 * nt * rows
        per_kernel.append({"rows": rows, "cols": cols, "n_tok": nt, "us_alone": round(mean_ * 1e3, 2),
                           "gbs_alone": round(byts / (mean_ * 1e-3) / 1e9, 1)})
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            traffic = json.load(f).get(f"{args.workload}:b{b}:T{T}")
    except Exception:
        traffic = None

    sweep_mm = matmul_sweep(flush, stream, peak) if (world == 1 and not args.no_matmul_sweep) else []
    sweep_attn = attention_sweep(flush, stream, peak) if (world == 1 and not args.no_attn_sweep) else []
    sweep_wide = wide_sweep(flush, stream) if (world == 1 and not args.no_wide_sweep) else []

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
    graph.close()
    total_bytes, wbytes, kvbytes = step_bytes(ms, b, T, lens)
    del model, ws, graph
    torch.cuda.empty_cache()

    extra_llama = llama_step(flush, stream, dev, 50) if (world == 1 and args.workload != "llama-68m"
                                                         and not args.no_extra) else None
    extra_spec = spec_grid(flush, stream, dev) if (world == 1 and not args.no_extra) else []

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(ms, b, T, budget_s=args.cpu_budget)
        cpu["cpu"] = _cpu_model()
        if args.cpu_all_core_budget > 0 and args.workload == "llama-68m":
            cpu["all_cores"] = cpu_all_cores(args.workload, b, T, budget_s=args.cpu_all_core_budget)

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
                       "l2": "flushed before every timed step: 512 MiB written, then 256 MiB of it read back (clean cold L2)", "parallelism": f"replicas x{world}",
                       "step_bytes": total_bytes, "weight_bytes": wbytes, "kv_bytes": kvbytes},
            "step_ms": {"p50": round(float(np.percentile(ts, 50)), 5), "p90": round(float(np.percentile(ts, 90)), 5),
                        "p95": round(float(np.percentile(ts, 95)), 5), "mean": round(float(mean), 5)},
            "step_roofline": {"bytes": total_bytes, "achieved_gbs": round(total_bytes / (ms_step * 1e-3) / 1e9, 1),
                              "peak_gbs": peak, "frac": round(total_bytes / (ms_step * 1e-3) / 1e9 / peak, 4)},
            "roofline": {"kernel": "matmul_q8_0_narrow_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "per": f"one step's {len(seq)} matmul launches in step order ({ms.n_layers} layers x 4 + "
                                f"head, n_tok {nt}, activations staged as the step's kernels write them), "
                                f"graph-replayed after an L2 flush",
                         "ms_per_sequence": round(mm_mean, 4), "algorithmic_bytes": int(tot_bytes),
                         "peak_kind": f"{peak_kind} hbm_gbs", "launches_alone": per_kernel},
            "b_sweep": sweep,
            "matmul_q8_0_narrow": sweep_mm,
            "attention_long_context": sweep_attn,
            "matmul_q8_0_wide": sweep_wide,
            "llama_68m_step": extra_llama,
            "spec_grid": extra_spec,
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


# Models too large for the oracle to draw whole (the Qwen3-14B shapes: 40
# layers, a 151936-row head) are timed on a stated sample and scaled linearly:
# layer 0 of the model and the first HEAD_SAMPLE_ROWS rows of the head.  Every
# layer has the same shapes, and the head is a row-independent matmul, so the
# full step's time is n_layers x (one layer) + vocab / HEAD_SAMPLE_ROWS x (the
# head sample).
HEAD_SAMPLE_ROWS = 4096


def _oracle_sampler(ms, b, T):
    """(run_one(i) -> oracle seconds scaled to the full step for sequence
    i % b, description of the sample).  Small models run whole."""
    from oracle import matmul as omm
    from oracle import step as ostep
    bi, lens, toks = _meta(ms, b, T, seed=7)
    if ms.n_layers * ms.hidden * ms.ffn <= 64 * 1024 * 1024:
        w, kc, vc = _oracle_model(ms, seed=0)
        shape = ostep.Shape(ms.hidden, ms.n_q_heads, ms.n_kv_heads, ms.head_dim, ms.ffn, ms.vocab, ms.n_layers,
                            ms.eps, ms.theta)

        def run_one(i):
            s = i % b
            t0 = time.perf_counter()
            ostep.decode_step(shape, w, kc, vc, ms.cache_dtype, toks[s * T:(s + 1) * T], bi[s:s + 1], T,
                              lens[s:s + 1])
            return time.perf_counter() - t0
        return run_one, f"single-sequence steps (1 of the {b} sessions each, {T} token(s)) of the {ms.name} workload"
    hr = min(HEAD_SAMPLE_ROWS, ms.vocab)
    import dataclasses
    sub = dataclasses.replace(ms, n_layers=1, vocab=hr)
    w, kc, vc = _oracle_model(sub, seed=0)
    shape = ostep.Shape(sub.hidden, sub.n_q_heads, sub.n_kv_heads, sub.head_dim, sub.ffn, sub.vocab, 1, sub.eps,
                        sub.theta)
    toks_sub = toks % hr   # the embedding table of the sample holds hr rows

    def run_one(i):
        s = i % b
        tk = toks_sub[s * T:(s + 1) * T]
        t0 = time.perf_counter()
        ostep.decode_step(shape, w, kc, vc, sub.cache_dtype, tk, bi[s:s + 1], T, lens[s:s + 1])
        t1 = time.perf_counter()
        omm.matmul_q8_0(w["head"], ostep.quant(np.ones((T, sub.hidden))))
        th = time.perf_counter() - t1
        return ms.n_layers * max(t1 - t0 - th, 0.0) + (ms.vocab / hr) * th
    return run_one, (f"single-sequence steps (1 of the {b} sessions each, {T} token(s)) of the {ms.name} workload, "
                     f"timed on layer 0 of {ms.n_layers} and {hr} of {ms.vocab} head rows and scaled linearly "
                     f"(x{ms.n_layers} layers, x{ms.vocab / hr:.2f} head)")


def cpu_baseline(ms, b, T, budget_s=20.0):
    """The oracle's decode step (numpy, float64) timed on the host: one
    sequence of the b-sequence batch per sample (a bounded sample of the same
    workload), repeated until ~budget_s of CPU work."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    run_one, desc = _oracle_sampler(ms, b, T)
    n = 0
    scaled = 0.0
    t0 = time.perf_counter()
    while True:
        scaled += run_one(n)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * T / scaled, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} {desc}; float64 numpy, {dt:.1f} s of host time"}


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
    step; for the Qwen3-14B shapes one layer and part of the head, scaled
    linearly to the whole step), on the host cores."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    ms = _shape(args.workload)
    b = args.b if args.b else DEFAULT_B[args.workload]
    T = args.T
    run_one, desc = _oracle_sampler(ms, b, T)
    for i in range(args.warmup):
        run_one(i)
    scaled = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        scaled += run_one(i)
    host = time.perf_counter() - t0
    value = args.steps * T / scaled
    line = {"impl": "reference", "metric": "decode-step tokens/s and q8_0 narrow-matmul HBM GB/s (% of peak), n_tok=1..16",
            "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(scaled / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": ms.name, "b": b, "tokens_per_seq": T,
                       "sample": f"one of the {b} sessions per step ({T} token(s))"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} {desc}; {host:.1f} s of host time", "cpu": _cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PROBE_ATTENTION = {  # F, Hq, Hkv, ctx, D, cache dtype, b, T, shortest seq_len
    "qwen3-14b": (16, 40, 8, 4096, 128, 1, 16, 1, 1),
    "llama-68m": (8, 12, 12, 2048, 64, 0, 8, 1, 128),
}


def run_probe(spec: str):
    """A few launches of one kernel at one shape, for a profiler to capture
    (no timing, no JSON line): ``matmul:ROWS:COLS:NTOK[,NTOK...]`` runs the
    narrow matmul three times per n_tok on N(0, 0.02) weights;
    ``staged:ROWS:COLS:NTOK[,NTOK...]`` the same from the staged layout (the
    step's matmul path);
    ``wide:ROWS:COLS:NTOK`` the tensor-core matmul three times;
    ``attention:WORKLOAD`` runs the decode attention four times on that
    workload's cache shape (b sequences, seq_lens uniform); ``dp4a`` measures
    the dp4a issue rate and latency (one JSON line); ``mma`` the mma.sync
    f16 and s8 product rates (one JSON line); ``step:WORKLOAD[:B]``
    replays the workload's captured decode step four times."""
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
    elif kind == "staged":
        rows, cols, nts = int(rest[0]), int(rest[1]), [int(v) for v in rest[2].split(",")]
        w = dsb.quantize_q8_0(torch.randn((rows, cols), generator=g, device="cuda") * 0.02)
        x = dsb.quantize_q8_0(torch.randn((16, cols), generator=g, device="cuda"))
        for nt in nts:
            stg = dsb.stage_q8_0(w, rows, cols, x[:nt].contiguous(), nt)
            for _ in range(3):
                dsb.matmul_q8_0_staged(w, rows, cols, stg, nt)
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
    elif kind == "step":
        # the captured decode step of a workload (default live batch), replayed
        # three times after a warm-up replay: 1 + 10 * layers + 2 kernels each
        ms = _shape(rest[0])
        b = int(rest[1]) if len(rest) > 1 else DEFAULT_B[rest[0]]
        model = _make_model(ms, seed=1000)
        bi, lens, toks = _meta(ms, b, 1, seed=7)
        ws = model.workspace(b)
        logits = torch.empty((b, ms.vocab), dtype=torch.float32, device="cuda")
        graph = model.graph(b, 1, logits, ws)
        torch.cuda.synchronize()
        for _ in range(4):
            graph.launch(toks, bi, lens)
        torch.cuda.synchronize()
        graph.close()
        print(json.dumps({"probe": "step", "workload": ms.name, "b": b,
                          "kernels_per_step": launches_per_step(ms)}))
    elif kind == "dp4a":
        # the dp4a issue rate (many warps, independent chains) and latency
        # (one dependent chain), from which the narrow matmul's arithmetic
        # ceiling follows: 8 dp4a per q8_0 block and token
        props = torch.cuda.get_device_properties(0)
        sms = props.multi_processor_count
        out = torch.zeros(4, dtype=torch.int32, device="cuda")
        res = {}
        for blocks in (sms * 8, sms * 32):
            iters = 4096
            for _ in range(2):
                dsb.probe_dp4a(0, blocks, iters, out)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dsb.probe_dp4a(0, blocks, iters, out)
            e1.record()
            e1.synchronize()
            sec = e0.elapsed_time(e1) * 1e-3
            ops = blocks * 256 * 8 * iters
            res[f"rate_{blocks // sms}_ctas_per_sm"] = {"dp4a_per_s": ops / sec, "seconds": sec}
        dsb.probe_dp4a(1, 1, 1 << 16, out)
        torch.cuda.synchronize()
        cyc, it = int(out[1].item()) & 0xFFFFFFFF, int(out[2].item())
        res["latency_cycles"] = cyc / it
        with ClockSampler(0) as clk:
            dsb.probe_dp4a(0, sms * 32, 1 << 15, out)
            torch.cuda.synchronize()
        clocks = clk.summary()
        res["clocks"] = clocks
        mhz = clocks.get("sm_mhz") or 2070.0
        best = max(v["dp4a_per_s"] for k, v in res.items() if k.startswith("rate_"))
        res["dp4a_per_clk_per_sm"] = best / (sms * mhz * 1e6)
        res["sms"] = sms
        print(json.dumps({"probe": "dp4a", **res}))
    elif kind == "mma":
        # warp-level tensor-core products (mma.sync): m16n8k16 f16 -> f32 and
        # m16n8k32 s8 -> s32, 8 independent tiles per warp
        props = torch.cuda.get_device_properties(0)
        sms = props.multi_processor_count
        out = torch.zeros(4, dtype=torch.int32, device="cuda")
        res = {"sms": sms}
        with ClockSampler(0) as clk:
            for mode, name, ops_per in ((2, "f16_m16n8k16", 2 * 16 * 8 * 16), (3, "s8_m16n8k32", 2 * 16 * 8 * 32)):
                best = 0.0
                for blocks in (sms, sms * 2, sms * 4):
                    iters = 2048
                    dsb.probe_mma(mode, blocks, iters, out)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    dsb.probe_mma(mode, blocks, iters, out)
                    e1.record()
                    e1.synchronize()
                    sec = e0.elapsed_time(e1) * 1e-3
                    n = blocks * 8 * 8 * iters
                    res[f"{name}_{blocks // sms}_ctas_per_sm"] = {"tops": n * ops_per / sec / 1e12, "seconds": sec}
                    best = max(best, n / sec)
                res[f"{name}_per_clk_per_sm"] = best
        clocks = clk.summary()
        mhz = clocks.get("sm_mhz") or 2070.0
        for name in ("f16_m16n8k16", "s8_m16n8k32"):
            res[f"{name}_per_clk_per_sm"] = res[f"{name}_per_clk_per_sm"] / (sms * mhz * 1e6)
        res["clocks"] = clocks
        print(json.dumps({"probe": "mma", **res}))
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
    ap.add_argument("--workload", choices=["llama-68m", "llama-68m-spec", "qwen3-14b"], default="qwen3-14b")
    ap.add_argument("--b", type=int, default=0, help="live batch (default: 16 for qwen3-14b, 8 for llama-68m)")
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-all-core-budget", type=float, default=8.0,
                    help="seconds of the all-core oracle run beside the single-core one (0: skip)")
    ap.add_argument("--no-matmul-sweep", action="store_true")
    ap.add_argument("--no-wide-sweep", action="store_true", help="skip the wide tensor-core matmul timings")
    ap.add_argument("--no-attn-sweep", action="store_true",
                    help="skip the split-K attention at ctx 32768/65536 (allocates ~70 GB)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the llama-68m-shaped step and the b x K speculative grid")
    ap.add_argument("--probe", default=None,
                    help="run one kernel a few times for a profiler and exit: matmul:ROWS:COLS:NTOK[,..], "
                         "staged:ROWS:COLS:NTOKS, wide:ROWS:COLS:NTOK, attention:WORKLOAD, dp4a (the dp4a rate / latency probe) "
                         "or mma (the mma.sync rate probe)")
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
