"""Decode benchmark of the Qwen3-8B-shaped Q4_0 model (vocab 151936, hidden
4096, 36 layers, 32/8 heads, head_dim 128, FFN 12288, f16 KV cache) on one
GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Headline: batch-1 greedy decode after a 2048-token prompt.  One "step" is one
full decode step (embedding, 36 layers, final norm, tied LM head, argmax)
through the CUDA-graph replay of tq_decode_step; inputs are device-resident
and the model's 4.26 GB of weights exceed L2, so every step reads them from
HBM.  The same JSON line carries:

* `roofline`: the step's dominant kernel, the GEMV chain that follows each
  layer's attention (output projection, FFN, next layer's Q/K/V), launched as
  in the step (tq_decode_chain) for layers 0..34 in a CUDA graph and timed
  with CUDA events;
* `e2e`: the same step through the public API with the token copied in from
  pinned host memory and the argmax copied out, every step;
* `prefill`: the 2048-token prompt, timed warm with CUDA events, with the
  tensor-core GEMM's roofline (tq_gemm at 2048 rows over the 36 layers' gate
  matrices);
* `batched`: 32 sequences with seeded ragged contexts over a paged f16 cache,
  one decode step of the whole batch per graph replay, with the batched
  GEMM's roofline (tq_gemm at 32 rows over the 36 layers' down projections);
* `mixed`: one continuous-batching step (tq_step) of the same 32-sequence
  mix in which one sequence is still prefilling: 31 decode rows and a
  512-row prompt chunk, every projection a tensor-core GEMM over 543 rows;
* `sampling`: temperature / top-p sampling (tq_sample) of 151936-entry
  logit rows, 1 and 32 rows per call, L2 flushed between calls;
* `cpu_baseline` (also inside each sub-benchmark): the oracle timed on this
  host's cores on a bounded sample of each workload.

Under torchrun every rank runs an independent replica (the step does not
shard); `value` is the sum of tokens over all ranks divided by the slowest
rank's time.  `--impl reference` times the oracle alone on this host's cores.
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

METRIC = "decode tokens/s (B=1, Q4_0 Qwen3-8B shape) and achieved HBM GB/s vs peak"
PROMPT = 2048
N_SAMPLE_LAYERS = 2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true", help="skip the batched sub-benchmark")
    ap.add_argument("--batched-steps", type=int, default=30)
    ap.add_argument("--no-mixed", action="store_true", help="skip the continuous-batching sub-benchmark")
    ap.add_argument("--mixed-steps", type=int, default=10)
    ap.add_argument("--no-sampling", action="store_true", help="skip the sampling sub-benchmark")
    ap.add_argument("--prefill-reps", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling cases only: keep the first N layers of the workloads")
    ap.add_argument("--only", choices=["batched", "mixed", "sampling"], default=None,
                    help="profiling cases only: run just one sub-benchmark")
    ap.add_argument("--workload", default="qwen3_8b_q4_0",
                    help="decode workload of the headline (profiling cases may pick another)")
    ap.add_argument("--arch", default="qwen3", choices=["qwen3", "llama", "qwen2", "gemma3"],
                    help="layer recipe of the same shape (gemma3: window 512 on 5 of every 6 layers, "
                         "final logit softcap 30)")
    ap.add_argument("--wtype", default=None, choices=["q4_0", "q8_0", "affine4"],
                    help="weight format of the same shape")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": float(d["hbm_gbs"]), "tc": float(d["bf16_tflops"]),
                "tc_sust": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "kind": "measured"}
    return {"hbm": 6800.0, "tc": 1900.0, "tc_sust": 1700.0, "kind": "fallback"}


def dist_init():
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    return rank, world


def reduce_max(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing

class OracleSample:
    """The oracle (as it stands, float32) on bounded samples of the three
    workloads, over 2 of the 36 full-size layers (their layer time scaled to
    36) plus the full 151936 x 4096 LM head.  Weights are decoded once, before
    any timing."""

    def __init__(self):
        import numpy as np
        import synth
        from oracle import model as om
        from oracle import quant
        w = self.w = synth.QWEN3_8B_Q4
        weights = {}
        names = [f"blk.{i}.{t}" for i in range(N_SAMPLE_LAYERS) for t in synth.LAYER_TENSORS[:7]]
        for n in names + ["token_embd"]:
            weights[n] = quant.quantize(synth.host_tensor(w, n), w.wtype)
        for n in [f"blk.{i}.{t}" for i in range(N_SAMPLE_LAYERS) for t in synth.LAYER_TENSORS[7:]]:
            weights[n] = synth.host_tensor(w, n)
        weights["output_norm"] = synth.host_tensor(w, "output_norm")
        self.m = om.OracleModel(w, weights, dtype=np.float32)
        for n in names + ["token_embd"]:
            self.m.matrix(n)
        self.cores = len(os.sched_getaffinity(0))

    def _kv(self, stream, ctx):
        import numpy as np
        import synth
        w = self.w
        kv = synth.host_normal(w.seed, stream, 2 * w.n_kv_heads * ctx * w.head_dim, sigma=1.0)
        return kv.astype(np.float16).astype(np.float32).reshape(2, w.n_kv_heads, ctx, w.head_dim)

    def decode_step(self, ctx=PROMPT):
        """Seconds of one full batch-1 decode step at `ctx` cached positions."""
        import numpy as np
        import synth
        kv = self._kv(synth.KV_STREAM, ctx)
        cache = [(kv[0].copy(), kv[1].copy()) for _ in range(N_SAMPLE_LAYERS)]
        x = self.m.embed([1])
        t0 = time.perf_counter()
        for i in range(N_SAMPLE_LAYERS):
            x = self.m.block(i, x, cache, np.array([ctx]))
        t1 = time.perf_counter()
        self.m.head(x[-1])
        t2 = time.perf_counter()
        return (t1 - t0) / N_SAMPLE_LAYERS * self.w.n_layers + (t2 - t1)

    def decode_desc(self, ctx=PROMPT):
        return (f"oracle float32 batch-1 decode step at context {ctx}: {N_SAMPLE_LAYERS} of "
                f"{self.w.n_layers} full-size layers and the 151936x4096 LM head timed, the layer "
                f"time scaled to {self.w.n_layers} layers; weights decoded before timing")

    def batched_step(self, lens, n_seq=4):
        """Seconds of one batched decode step over len(lens) sequences, from
        `n_seq` of them (their layer time scaled to all sequences and 36 layers;
        the head for all sequences at once)."""
        import numpy as np
        import synth
        x_all = self.m.embed(list(range(1, len(lens) + 1)))
        t_layers = 0.0
        for b in range(n_seq):
            ctx = int(lens[b])
            kv = self._kv(synth.KV_STREAM + 2 + b, ctx)
            cache = [(kv[0].copy(), kv[1].copy()) for _ in range(N_SAMPLE_LAYERS)]
            x = x_all[b:b + 1]
            t0 = time.perf_counter()
            for i in range(N_SAMPLE_LAYERS):
                x = self.m.block(i, x, cache, np.array([ctx]))
            t_layers += time.perf_counter() - t0
        t0 = time.perf_counter()
        self.m.head(x_all)
        t_head = time.perf_counter() - t0
        return t_layers / n_seq * len(lens) / N_SAMPLE_LAYERS * self.w.n_layers + t_head

    def mixed_step(self, lens, cached, chunk, n_seq=4):
        """Seconds of one continuous-batching step: decode rows of len(lens)
        sequences (`n_seq` of them timed, scaled to all) and a `chunk`-row
        prompt chunk after `cached` positions, through 2 layers scaled to 36,
        plus the head for every sequence's last row."""
        import numpy as np
        import synth
        t_dec = self.batched_step(lens[:n_seq], n_seq) - self._head_time(n_seq)
        t_dec *= len(lens) / n_seq
        kv = self._kv(synth.KV_STREAM + 1, cached)
        cache = [(kv[0].copy(), kv[1].copy()) for _ in range(N_SAMPLE_LAYERS)]
        x = self.m.embed(self.w.prompt(n=chunk))
        t0 = time.perf_counter()
        for i in range(N_SAMPLE_LAYERS):
            x = self.m.block(i, x, cache, np.arange(cached, cached + chunk))
        t_chunk = (time.perf_counter() - t0) / N_SAMPLE_LAYERS * self.w.n_layers
        return t_dec + t_chunk + self._head_time(len(lens) + 1)

    def sampling(self, V, n=4):
        """Seconds of the oracle sampler on n seeded rows of V logits."""
        import numpy as np
        import synth
        from oracle import sample as osm
        rows = synth.host_normal(5, 7, n * V, sigma=2.0).astype(np.float64).reshape(n, V)
        us = synth.uniform_below(5, 8, n, 1 << 24).astype(np.float64) / float(1 << 24)
        t0 = time.perf_counter()
        for r in range(n):
            osm.sample(rows[r], 0.7, 0.9, float(us[r]))
        return time.perf_counter() - t0, n

    def _head_time(self, rows):
        x = self.m.embed(list(range(1, rows + 1)))
        t0 = time.perf_counter()
        self.m.head(x)
        return time.perf_counter() - t0

    def prefill(self, n=PROMPT):
        """Seconds of a full n-token prefill (36 layers scaled from 2, last-row head)."""
        import numpy as np
        x = self.m.embed(self.w.prompt(n=n))
        cache = self.m.new_cache()
        t0 = time.perf_counter()
        for i in range(N_SAMPLE_LAYERS):
            x = self.m.block(i, x, cache, np.arange(n))
        t1 = time.perf_counter()
        self.m.head(x[-1])
        t2 = time.perf_counter()
        return (t1 - t0) / N_SAMPLE_LAYERS * self.w.n_layers + (t2 - t1)


def run_reference(args, rank, world):
    if rank != 0:
        return
    o = OracleSample()
    for _ in range(args.warmup):
        o.decode_step()
    total = sum(o.decode_step() for _ in range(args.steps))
    value = args.steps / total
    desc = o.decode_desc()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 / value, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "qwen3_8b_q4_0 batch-1 greedy decode after a 2048-token prompt",
                       "sample": desc},
            "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": o.cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- helpers

def file_hash(*paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


CSRC = os.path.join(ROOT, "block_quantized_transformer_gb300", "csrc")


def traffic_of(name, *sources):
    """DRAM bytes per launch of a kernel from profiles/traffic.json (written
    from an ncu capture), if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    entry = json.load(open(p)).get(name)
    if not entry or entry.get("source_sha256_16") != file_hash(*[os.path.join(CSRC, s) for s in sources]):
        return None
    return int(entry["dram_bytes_per_launch"])


def time_graph(fn, n, stream, reps=3):
    """Mean time (ms) of one of the n launches that fn(i) enqueues, from a CUDA
    graph of all n, replayed `reps` times between CUDA events on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(n):                       # the first launches set kernel attributes
            fn(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
        g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / (reps * n)


# ----------------------------------------------------------------------------- GPU bench

def apply_variant(w, args):
    """The workload with the layer recipe and weight format the options name."""
    import dataclasses
    if args.arch == "qwen3" and (args.wtype is None or args.wtype == w.wtype):
        return w
    kw = {"arch": args.arch}
    if args.arch == "gemma3":
        kw.update(sliding_window=512, sliding_pattern=6, logit_softcap=30.0)
    if args.wtype is not None:
        kw["wtype"] = args.wtype
    return dataclasses.replace(w, name=f"{w.name}[{args.arch}, {kw.get('wtype', w.wtype)}]", **kw)


def q4_bytes(rows, cols):
    return rows * cols // 32 * 18


def run_gpu(args, rank, world):
    import numpy as np
    import torch
    import synth
    import block_quantized_transformer_gb300 as tq
    from block_quantized_transformer_gb300.synthetic import build_weights, build_model

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = {x.name: x for x in synth.WORKLOADS}[args.workload]
    import dataclasses
    if args.layers:
        w = dataclasses.replace(w, n_layers=args.layers)
    w = apply_variant(w, args)
    pk = peaks()
    K, W = args.steps, args.warmup
    P = w.prompt_len
    E = args.e2e_steps
    max_ctx = P + W + K + E + 16
    mats, gains = build_weights(w, dev)
    if args.only is not None:
        st = torch.cuda.Stream(device=dev)
        b = (run_batched(args, world, mats, gains, dev, st, pk) if args.only == "batched" else
             run_mixed(args, world, mats, gains, dev, st, pk) if args.only == "mixed" else
             run_sampling(dev, st, pk, w.vocab))
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    model = build_model(w, device=dev, max_ctx=max_ctx, max_prefill=P, weights=(mats, gains))
    torch.cuda.synchronize()
    weight_bytes = model.weight_bytes() + sum(g.numel() * 4 for g in gains.values())
    stream = torch.cuda.Stream(device=dev)
    prompt = torch.tensor(w.prompt(), dtype=torch.int32, device=dev)
    L = w.n_layers

    with torch.cuda.stream(stream):
        # ---- prefill, warm: one untimed call, then reps calls between CUDA events
        am = model.prefill(prompt)
        stream.synchronize()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(args.prefill_reps):
            am = model.prefill(prompt)
        p1.record(stream)
        stream.synchronize()
        prefill_ms = p0.elapsed_time(p1) / args.prefill_reps

        # ---- batch-1 decode: warm-up (graph capture on the first replay), timed region
        tok = torch.empty(1, dtype=torch.int32, device=dev)
        tok.copy_(am)
        pos = torch.full((1,), P, dtype=torch.int32, device=dev)
        for _ in range(W):
            model.decode_step(tok, pos, pos, argmax=tok, graph=True)
            pos.add_(1)
        stream.synchronize()
        ctx0 = int(pos.item())
        barrier(world)
        torch.cuda.synchronize()
        clocks = Clocks(local)
        clocks.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            model.decode_step(tok, pos, pos, argmax=tok, graph=True)
            pos.add_(1)
        e1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        clk = clocks.stop()
        barrier(world)
        assert model.status() == 0
    ms_max = reduce_max(ms, world)
    ms_step = ms_max / K
    value = world * K / (ms_max / 1e3)

    # algorithmic bytes per step: all weights + KV read at each step's context + KV write
    esz = 2 if w.kv == "f16" else 4
    kv_row = 2 * w.n_kv_heads * w.head_dim * esz * L              # bytes per cached position
    mean_ctx = ctx0 + (K - 1) / 2.0 + 1
    step_bytes = weight_bytes + kv_row * mean_ctx + kv_row

    # ---- dominant kernel: the GEMV chain after each attention, as launched in the step
    H, F, nq, nkv, hd = w.hidden, w.ffn, w.n_heads, w.n_kv_heads, w.head_dim
    chain_bytes = (q4_bytes(H, nq * hd) + 2 * q4_bytes(F, H) + q4_bytes(H, F)
                   + q4_bytes((nq + 2 * nkv) * hd, H))
    chain_act = 4 * (2 * H + 2 * nq * hd + 2 * H + F + 2 * H + F + H + (nq + 2 * nkv) * hd)
    n_chain = max(1, L - 1)
    chain_ms = time_graph(lambda i: model.decode_chain(i), n_chain, stream)
    chain_alg = chain_bytes + chain_act
    roofline = {"bound": "hbm", "achieved": round(chain_alg / (chain_ms / 1e3) / 1e9, 1), "peak": pk["hbm"],
                "unit": "GB/s", "frac": round(chain_alg / (chain_ms / 1e3) / 1e9 / pk["hbm"], 4),
                "traffic": traffic_of("gemv_chain_layer_qwen3_8b_q4_0", "gemv_impl.cuh", "gemv.cu", "gemv_q4.cu")
                if w.name == "qwen3_8b_q4_0" else None,
                "kernel": f"gemv_chain_kernel<{w.wtype.upper()}>: output projection + residual, RMSNorm + gate/up "
                          "+ SwiGLU, down projection + residual, next layer's RMSNorm + Q/K/V",
                "timing": f"tq_decode_chain for layers 0..{n_chain - 1} in one CUDA graph, CUDA events",
                "peak_kind": pk["kind"] + " copy bandwidth",
                "launch_ms": round(chain_ms, 5), "bytes_per_launch": int(chain_alg)}

    # ---- end to end: host token in, host argmax out, every step
    h_tok = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h_pos = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    d_tok = torch.empty(1, dtype=torch.int32, device=dev)
    d_pos = torch.empty(1, dtype=torch.int32, device=dev)
    d_out = torch.empty(1, dtype=torch.int32, device=dev)
    h_tok[0] = int(tok.item())
    p = ctx0 + K
    with torch.cuda.stream(stream):
        def e2e_step():
            nonlocal p
            h_pos[0] = p
            d_tok.copy_(h_tok, non_blocking=True)
            d_pos.copy_(h_pos, non_blocking=True)
            model.decode_step(d_tok, d_pos, d_pos, argmax=d_out, graph=True)
            h_out.copy_(d_out, non_blocking=True)
            stream.synchronize()
            h_tok[0] = int(h_out[0])
            p += 1
        e2e_step()                                  # graph capture with these buffers
        e2e_steps = min(E, max_ctx - p - 1)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(e2e_s, world)
    e2e = {"value": round(world * e2e_steps / e2e_s, 2), "unit": "tokens/s", "h2d_bytes_per_step": 8,
           "d2h_bytes_per_step": 4, "steps": e2e_steps}
    launches = model.launches_per_step * K
    model.close()

    # ---- prefill roofline: the tensor-core GEMM at 2048 rows (gate matrices of every layer)
    x = torch.randn(P, H, device=dev)
    y = torch.empty(P, F, device=dev)
    scr = torch.empty(tq.lib().tq_gemm_scratch_bytes(F, P, H) + 256, dtype=torch.uint8, device=dev)
    gemm_ms = time_graph(lambda i: tq.tq_gemm(mats[f"blk.{i}.ffn_gate"], x, out=y, scratch=scr), L, stream)
    gemm_flop = 2.0 * P * F * H
    prefill_flop = 2.0 * P * weight_count_layers(w) + attn_prefill_flop(w, P)
    prefill = {"tokens": P, "ms": round(prefill_ms, 3), "tokens_per_s": round(world * P / (prefill_ms / 1e3), 1),
               "timing": f"warm, {args.prefill_reps} calls between CUDA events",
               "tflops": round(prefill_flop / (prefill_ms / 1e3) / 1e12, 1),
               "frac_of_tensor_peak": round(prefill_flop / (prefill_ms / 1e3) / 1e12 / pk["tc_sust"], 4),
               "tensor_peak_tflops": pk["tc_sust"], "flop": prefill_flop,
               "roofline": {"bound": "tensor", "achieved": round(gemm_flop / (gemm_ms / 1e3) / 1e12, 1),
                            "peak": pk["tc"], "unit": "TFLOP/s",
                            "frac": round(gemm_flop / (gemm_ms / 1e3) / 1e12 / pk["tc"], 4),
                            "traffic": traffic_of("tcgemm_prefill_gate_qwen3_8b_q4_0", "tcgemm.cu")
                            if w.name == "qwen3_8b_q4_0" else None,
                            "kernel": f"tcgemm_kernel<{w.wtype.upper()}, 256> (tcgen05, fp16 operands, f32 TMEM) + "
                                      f"xprep16: gate projection {F}x{H} at {P} rows",
                            "timing": f"tq_gemm over the {L} layers' gate matrices in one CUDA graph",
                            "peak_kind": pk["kind"] + " bf16 dense burst (fp16 has the same rate)",
                            "launch_ms": round(gemm_ms, 5), "flop_per_launch": gemm_flop}}
    del x, y, scr

    batched = mixed = sampling = None
    if not args.no_batched and w.name.startswith("qwen3_8b_q4_0"):
        batched = run_batched(args, world, mats, gains, dev, stream, pk)
    if not args.no_mixed and w.name.startswith("qwen3_8b_q4_0"):
        mixed = run_mixed(args, world, mats, gains, dev, stream, pk)
    if not args.no_sampling:
        sampling = run_sampling(dev, stream, pk, w.vocab)

    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 (decode GEMVs: exact codes x 21-bit activations, f32 sums); prefill/batched "
                     "GEMMs: fp16 x fp16 -> f32 (tcgen05)",
            "data": "synthetic",
            "config": {"workload": f"{w.name} batch-1 greedy decode after a {P}-token prompt "
                                   f"(context {ctx0}..{ctx0 + K - 1})",
                       "weights": f"{w.wtype.upper()}, {weight_bytes / 1e9:.2f} GB, seeded N(0,0.02)", "kv_cache": "f16",
                       "l2": "inputs exceed L2 (4.3 GB of weights read every step)",
                       "parallelism": f"replicas x{world}"},
            "hbm": {"step_bytes": int(step_bytes), "achieved_gbs": round(step_bytes / (ms_step / 1e3) / 1e9, 1),
                    "frac_of_peak": round(step_bytes / (ms_step / 1e3) / 1e9 / pk["hbm"], 4),
                    "peak_gbs": pk["hbm"], "peak_kind": pk["kind"],
                    "roofline_tokens_per_s": round(pk["hbm"] * 1e9 / step_bytes, 1)},
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "prefill": prefill}
    if batched is not None:
        line["batched"] = batched
    if mixed is not None:
        line["mixed"] = mixed
    if sampling is not None:
        line["sampling"] = sampling
    if rank == 0 and not args.no_cpu_baseline and w.name == "qwen3_8b_q4_0" and not args.layers:
        o = OracleSample()
        o.decode_step()
        per_step = min(o.decode_step() for _ in range(3))
        line["cpu_baseline"] = {"value": round(1.0 / per_step, 5), "unit": "tokens/s", "cores": o.cores,
                                "kind": "oracle", "sample": o.decode_desc()}
        pf = o.prefill()
        line["prefill"]["cpu_baseline"] = {
            "value": round(PROMPT / pf, 3), "unit": "tokens/s", "cores": o.cores, "kind": "oracle",
            "sample": f"oracle float32 prefill of the {PROMPT}-token prompt: {N_SAMPLE_LAYERS} of "
                      f"{w.n_layers} full-size layers timed, scaled to {w.n_layers}, plus the last-row head"}
        if batched is not None:
            lens = synth.QWEN3_8B_Q4_BATCHED.context_lengths()
            bs = o.batched_step(lens)
            line["batched"]["cpu_baseline"] = {
                "value": round(len(lens) / bs, 4), "unit": "tokens/s", "cores": o.cores, "kind": "oracle",
                "sample": f"oracle float32 batched step: 4 of {len(lens)} sequences (their seeded "
                          f"contexts) through {N_SAMPLE_LAYERS} of {w.n_layers} full-size layers, scaled "
                          f"to all sequences and layers, plus the LM head for all {len(lens)}"}
        if mixed is not None:
            ml = synth.QWEN3_8B_Q4_BATCHED.context_lengths()[:-1]
            ts = o.mixed_step(ml, 1024, 512)
            line["mixed"]["cpu_baseline"] = {
                "value": round((len(ml) + 512) / ts, 4), "unit": "tokens/s", "cores": o.cores, "kind": "oracle",
                "sample": f"oracle float32 mixed step: decode rows of 4 of the {len(ml)} sequences and the "
                          f"512-row chunk after 1024 cached positions through {N_SAMPLE_LAYERS} of "
                          f"{w.n_layers} full-size layers, scaled to all rows and layers, plus the LM head "
                          f"for {len(ml) + 1} rows"}
        if sampling is not None:
            ts, n = o.sampling(w.vocab)
            line["sampling"]["cpu_baseline"] = {
                "value": round(n / ts, 3), "unit": "rows/s", "cores": o.cores, "kind": "oracle",
                "sample": f"oracle sampler (f64, sort-based) on {n} seeded {w.vocab}-entry rows, "
                          "temperature 0.7, top-p 0.9"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def weight_count_layers(w):
    """Weights multiplied per token in prefill: every layer's projections and the head row."""
    H, F, hd = w.hidden, w.ffn, w.head_dim
    per_layer = H * (w.n_heads + 2 * w.n_kv_heads) * hd + w.n_heads * hd * H + 3 * F * H
    return per_layer * w.n_layers


def attn_prefill_flop(w, T):
    """Causal attention of a T-token prompt: q.k and p.v over j <= i for every
    query head and layer."""
    pairs = T * (T + 1) / 2
    return 2.0 * 2.0 * pairs * w.n_heads * w.head_dim * w.n_layers


def run_batched(args, world, mats, gains, dev, stream, pk):
    """32 sequences of the batched serving mix over a paged f16 cache: cached
    lengths from the seeded length generator, pages handed out in a seeded
    shuffled order, the cache filled with seeded N(0, 1) values (no prefill:
    the step's cost does not depend on what the cache holds), then greedy
    decode steps of the whole batch, timed with CUDA events around graph
    replays."""
    import numpy as np
    import torch
    import synth
    import block_quantized_transformer_gb300 as tq
    from block_quantized_transformer_gb300.synthetic import build_model

    w = synth.QWEN3_8B_Q4_BATCHED
    if args.layers:
        import dataclasses
        w = dataclasses.replace(w, n_layers=args.layers)
    w = apply_variant(w, args)
    K, W = args.batched_steps, 3
    B, P = w.batch, w.page_size
    lens = w.context_lengths().astype(np.int64)
    need = lens + W + K + 1
    per_seq = int((need.max() + P - 1) // P)
    max_ctx = per_seq * P
    n_pages_seq = (need + P - 1) // P
    n_pages = int(n_pages_seq.sum())
    keys = synth.host_normal(w.length_seed, synth.LENGTH_STREAM + 1, n_pages, sigma=1.0)
    order = np.argsort(keys, kind="stable").astype(np.int32)        # seeded shuffle of the pool
    table = np.zeros((B, per_seq), dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :n_pages_seq[b]] = order[at:at + n_pages_seq[b]]
        at += n_pages_seq[b]
    model = build_model(w, device=dev, max_batch=B, max_ctx=max_ctx, max_prefill=B,
                        page_size=P, n_pages=n_pages, weights=(mats, gains))
    chunk = 1 << 26
    for cache, stream_id in ((model.k_cache, synth.KV_STREAM), (model.v_cache, synth.KV_STREAM + 1)):
        for i0 in range(0, cache.numel(), chunk):
            n = min(chunk, cache.numel() - i0)
            f = torch.empty(n, dtype=torch.float32, device=dev)
            synth.dev_normal(f, w.seed, stream_id, first=i0, sigma=1.0)
            cache[i0:i0 + n].copy_(f)
            del f
    torch.cuda.synchronize()
    weight_bytes = model.weight_bytes() + sum(g.numel() * 4 for g in gains.values())
    bt = torch.tensor(table, device=dev)
    tok = torch.tensor(synth.uniform_below(w.seed, synth.PROMPT_STREAM, B, w.vocab).astype(np.int32), device=dev)
    pos = torch.tensor(lens.astype(np.int32), device=dev)
    with torch.cuda.stream(stream):
        for _ in range(W):
            model.decode_step(tok, pos, pos, block_table=bt, argmax=tok, graph=True)
            pos.add_(1)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            model.decode_step(tok, pos, pos, block_table=bt, argmax=tok, graph=True)
            pos.add_(1)
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        barrier(world)
        assert model.status() == 0
    ms_max = reduce_max(ms, world)
    ms_step = ms_max / K
    kv_row = 2 * w.n_kv_heads * w.head_dim * 2 * w.n_layers
    ctx_sum = float((lens + W + 1).sum()) + B * (K - 1) / 2.0
    step_bytes = weight_bytes + kv_row * ctx_sum + kv_row * B
    launches = model.decode_launches(B) * K
    model.close()
    del model
    torch.cuda.empty_cache()

    # the batched GEMM as the step runs it: 32 rows, K split across CTAs (down projections)
    H, F, L = w.hidden, w.ffn, w.n_layers
    x = torch.randn(B, F, device=dev)
    y = torch.empty(B, H, device=dev)
    scr = torch.empty(tq.lib().tq_gemm_scratch_bytes(H, B, F) + 256, dtype=torch.uint8, device=dev)
    gemm_ms = time_graph(lambda i: tq.tq_gemm(mats[f"blk.{i}.ffn_down"], x, out=y, scratch=scr), L, stream)
    gemm_bytes = q4_bytes(H, F) + 4 * B * (F + H)
    return {"metric": f"decode tokens/s (B={B}, {w.wtype.upper()} Qwen3-8B shape, paged f16 KV)",
            "value": round(world * B * K / (ms_max / 1e3), 2), "unit": "tokens/s", "steps": K, "warmup": W,
            "ms_per_step": round(ms_step, 4),
            "config": {"workload": f"{w.name}: {B} sequences, cached lengths {int(lens.min())}..{int(lens.max())} "
                                   f"(sum {int(lens.sum())}), pages of {P} tokens in a seeded shuffled order",
                       "kv_cache": "f16, seeded N(0,1)", "l2": "inputs exceed L2"},
            "hbm": {"step_bytes": int(step_bytes), "achieved_gbs": round(step_bytes / (ms_step / 1e3) / 1e9, 1),
                    "frac_of_peak": round(step_bytes / (ms_step / 1e3) / 1e9 / pk["hbm"], 4),
                    "peak_gbs": pk["hbm"], "roofline_tokens_per_s": round(B * pk["hbm"] * 1e9 / step_bytes, 1)},
            "roofline": {"bound": "hbm", "achieved": round(gemm_bytes / (gemm_ms / 1e3) / 1e9, 1),
                         "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(gemm_bytes / (gemm_ms / 1e3) / 1e9 / pk["hbm"], 4),
                         "traffic": traffic_of("tcgemm_batched_down_qwen3_8b_q4_0", "tcgemm.cu")
                         if w.name == "qwen3_8b_q4_0_batched32_paged" else None,
                         "kernel": f"tcgemm_kernel<{w.wtype.upper()}, 32> (tcgen05) + xprep16: down projection "
                                   f"{H}x{F} at {B} rows, K split across CTAs as in the step",
                         "timing": f"tq_gemm over the {L} layers' down matrices in one CUDA graph",
                         "peak_kind": pk["kind"] + " copy bandwidth",
                         "launch_ms": round(gemm_ms, 5), "bytes_per_launch": int(gemm_bytes)},
            "gpu_launches": launches}


def run_mixed(args, world, mats, gains, dev, stream, pk):
    """Continuous batching: the 32-sequence serving mix with its last sequence
    still prefilling.  One tq_step carries a decode row of each of the first
    31 sequences (seeded ragged contexts) and a 512-row prompt chunk of the
    32nd after 1024 cached positions; the paged f16 cache holds seeded N(0, 1)
    values.  Every timed step repeats the same rows (same positions, so the
    same work), eager launches, CUDA events around the whole run."""
    import numpy as np
    import torch
    import synth
    from block_quantized_transformer_gb300.synthetic import build_model

    w = synth.QWEN3_8B_Q4_BATCHED
    if args.layers:
        import dataclasses
        w = dataclasses.replace(w, n_layers=args.layers)
    w = apply_variant(w, args)
    K, W = args.mixed_steps, 3
    B, P, H, V = w.batch, w.page_size, w.hidden, w.vocab
    CACHED, CHUNK = 1024, 512
    lens = w.context_lengths().astype(np.int64)
    lens[B - 1] = CACHED
    need = lens + 1
    need[B - 1] = CACHED + CHUNK
    per_seq = int((need.max() + P - 1) // P)
    n_pages_seq = (need + P - 1) // P
    n_pages = int(n_pages_seq.sum())
    keys = synth.host_normal(w.length_seed, synth.LENGTH_STREAM + 1, n_pages, sigma=1.0)
    order = np.argsort(keys, kind="stable").astype(np.int32)
    table = np.zeros((B, per_seq), dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :n_pages_seq[b]] = order[at:at + n_pages_seq[b]]
        at += n_pages_seq[b]
    n_rows = (B - 1) + CHUNK
    model = build_model(w, device=dev, max_batch=B, max_ctx=per_seq * P, max_prefill=n_rows,
                        page_size=P, n_pages=n_pages, weights=(mats, gains))
    chunk = 1 << 26
    for cache, stream_id in ((model.k_cache, synth.KV_STREAM), (model.v_cache, synth.KV_STREAM + 1)):
        for i0 in range(0, cache.numel(), chunk):
            n = min(chunk, cache.numel() - i0)
            f = torch.empty(n, dtype=torch.float32, device=dev)
            synth.dev_normal(f, w.seed, stream_id, first=i0, sigma=1.0)
            cache[i0:i0 + n].copy_(f)
            del f
    torch.cuda.synchronize()
    toks = synth.uniform_below(w.seed, synth.PROMPT_STREAM + 200, n_rows, w.vocab).astype(np.int32)
    seq = np.concatenate([np.arange(B - 1), np.full(CHUNK, B - 1)]).astype(np.int32)
    pos = np.concatenate([lens[:B - 1], CACHED + np.arange(CHUNK)]).astype(np.int32)
    last = np.concatenate([np.arange(B - 1), [n_rows - 1]]).astype(np.int32)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d_tok, d_seq, d_pos, d_last, bt = d(toks), d(seq), d(pos), d(last), d(table)
    am = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(W):
            model.step(d_tok, d_seq, d_pos, d_last, block_table=bt, argmax=am)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            model.step(d_tok, d_seq, d_pos, d_last, block_table=bt, argmax=am)
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        barrier(world)
        assert model.status() == 0
    weight_bytes = model.weight_bytes() + sum(g.numel() * 4 for g in gains.values())
    model.close()
    del model
    torch.cuda.empty_cache()
    ms_max = reduce_max(ms, world)
    ms_step = ms_max / K
    L, nq, hd = w.n_layers, w.n_heads, w.head_dim
    kv_row = 2 * w.n_kv_heads * hd * 2 * L
    keys_read = float((lens[:B - 1] + 1).sum()) + (CACHED + CHUNK)       # each decode row's context, the chunk's keys once
    step_bytes = weight_bytes + kv_row * keys_read + kv_row * n_rows
    pairs = float((lens[:B - 1] + 1).sum()) + CHUNK * CACHED + CHUNK * (CHUNK + 1) / 2.0
    flop = 2.0 * n_rows * weight_count_layers(w) + 2.0 * B * V * H + 4.0 * pairs * nq * hd * L
    s_step = ms_step / 1e3
    return {"metric": f"continuous-batching step rows/s ({B - 1} decode rows + a {CHUNK}-row prompt chunk, "
                      f"{w.wtype.upper()} Qwen3-8B shape, paged f16 KV)",
            "value": round(world * n_rows * K / (ms_max / 1e3), 1), "unit": "tokens/s", "steps": K, "warmup": W,
            "ms_per_step": round(ms_step, 4),
            "config": {"workload": f"{w.name}: decode rows of sequences 0..{B - 2} (cached lengths "
                                   f"{int(lens[:B - 1].min())}..{int(lens[:B - 1].max())}) and sequence {B - 1}'s "
                                   f"prompt rows {CACHED}..{CACHED + CHUNK - 1} in one tq_step ({n_rows} rows), "
                                   f"pages of {P} tokens in a seeded shuffled order",
                       "kv_cache": "f16, seeded N(0,1)", "l2": "inputs exceed L2",
                       "timing": f"{K} eager tq_step calls between CUDA events (the same rows each time)"},
            "tensor": {"flop": flop, "achieved_tflops": round(flop / s_step / 1e12, 1),
                       "frac_of_peak": round(flop / s_step / 1e12 / pk["tc_sust"], 4), "peak_tflops": pk["tc_sust"],
                       "peak_kind": pk["kind"] + " bf16 dense sustained"},
            "hbm": {"step_bytes": int(step_bytes), "achieved_gbs": round(step_bytes / s_step / 1e9, 1),
                    "frac_of_peak": round(step_bytes / s_step / 1e9 / pk["hbm"], 4), "peak_gbs": pk["hbm"]}}


def run_sampling(dev, stream, pk, V, reps=20):
    """tq_sample over seeded N(0, 2^2) logit rows of the vocabulary (temperature
    0.7, top-p 0.9, seeded u), 1 and 32 rows per call; a 256 MB write between
    calls flushes L2, and each call is timed alone with CUDA events."""
    import numpy as np
    import torch
    import synth
    import block_quantized_transformer_gb300 as tq

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for B in (1, 32):
        lg = torch.empty(B * V, dtype=torch.float32, device=dev)
        synth.dev_normal(lg, 5, 7, sigma=2.0)
        lg = lg.view(B, V)
        t = torch.full((B,), 0.7, dtype=torch.float32, device=dev)
        p = torch.full((B,), 0.9, dtype=torch.float32, device=dev)
        u = torch.from_numpy(synth.uniform_below(5, 8, B, 1 << 24).astype(np.float32) / float(1 << 24)).to(dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        times = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.fill_(i & 255)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                tq.tq_sample(lg, t, p, u, out=tok)
                e1.record(stream)
                stream.synchronize()
                if i >= 3:
                    times.append(e0.elapsed_time(e1))
        ms = statistics.mean(times)
        nbytes = B * V * 4
        out[f"rows_{B}"] = {"us_per_call": round(ms * 1e3, 2), "rows_per_s": round(B / (ms / 1e3), 1),
                            "bytes_per_call": nbytes, "achieved_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                            "frac_of_hbm_peak": round(nbytes / (ms / 1e3) / 1e9 / pk["hbm"], 4)}
    del flush
    r32 = out["rows_32"]
    return {"metric": f"temperature/top-p sampling of {V}-entry logit rows, rows/s", "value": r32["rows_per_s"],
            "unit": "rows/s",
            "config": {"workload": f"{V}-entry f32 logit rows, seeded N(0, 2^2); temperature 0.7, top-p 0.9, "
                                   "seeded u", "l2": "flushed before every call (256 MB write)",
                       "timing": f"{reps} calls after 3, each between CUDA events"},
            **out,
            "roofline": {"bound": "hbm", "achieved": r32["achieved_gbs"], "peak": pk["hbm"], "unit": "GB/s",
                         "frac": r32["frac_of_hbm_peak"], "traffic": None,
                         "kernel": "sample_kernel<4>, 32 rows (a 4-CTA cluster per row; the row is read once per pass)",
                         "bytes_per_launch": r32["bytes_per_call"], "launch_ms": round(r32["us_per_call"] / 1e3, 5),
                         "peak_kind": pk["kind"] + " copy bandwidth"}}


def main():
    args = parse()
    if args.impl == "reference":
        rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
        run_reference(args, rank, world)
        return
    rank, world = dist_init()
    run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
