#!/usr/bin/env python3
"""Decode benchmark: batch-1 speech-token decode tokens/s and achieved HBM GB/s.

Workload (default `gpt2m_q4`): GPT-2-Medium-shaped T3 (24 layers, d 1024,
16x64 heads, FFN 4096, vocab 6563) with Q4_0 weights, a 150-token prompt,
then sampled decode steps (temperature 0.8, top-k 1000, top-p 0.95) with
seeded Philox draws.  A "step" is one decode step of the whole hot path:
embedding, 24 layers (norm, quantised GEMVs with fused epilogues, RoPE/KV
append, split-KV attention), final norm, head GEMV, on-device sampler.

value: K steps with device-resident draws and device-side token feedback
(sd_decode_n), timed with CUDA events on the launching stream.
e2e:   the same metric through sd_step with host buffers (each step copies
its token and draw host->device and its token device->host).
roofline: the decode step is the unit: algorithmic bytes per step (quantised
weights + small fp32 tensors + KV cache read and written at that position) over
the event-timed step duration, against the measured HBM copy bandwidth.

Multi-GPU: batch-1 decode does not shard; `--gpus N` runs N independent
replicas (one process per GPU) and reports the aggregate tokens/s over the
slowest rank's time ("scaling": "weak").

`--impl reference` times the oracle (plain C, fp64 sums) on the host cores on
a bounded sample of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import PRESETS, get_preset, prompt_tokens, uniform_draws  # noqa: E402
from synth.presets import ARCH_QWEN_TTS  # noqa: E402
from synth import presets as P  # noqa: E402

METRIC = "decode tokens/s at batch 1 and achieved HBM GB/s vs ~8 TB/s roofline"
L2_BYTES = 129 * 2 ** 20


def workload_text(run) -> str:
    m = run.model
    s = run.sampler
    samp = "greedy" if s.greedy else f"T {s.temperature}, top-k {s.top_k}, top-p {s.top_p}"
    if m.arch == P.ARCH_QWEN_TTS:
        return (f"{run.name}: Talker {m.n_layer}x{m.d_model} ({m.n_head}/{m.n_kv_head} heads x {m.head_dim}, "
                f"FFN {m.d_ff}, codebook-0 vocab {m.vocab}) + code predictor {m.cp_layer}x{m.cp_d_model} "
                f"({m.n_codebooks - 1} passes per frame, vocab {m.cp_vocab}), {P.QUANT_NAMES[m.quant]} weights"
                f"{(' (code predictor ' + P.QUANT_NAMES[m.cp_quant] + ')') if m.cp_quant else ''}, "
                f"fp16 KV; prompt {run.prompt_len} + {run.n_steps} frames ({samp}), {m.batch} rows")
    return (f"{run.name}: {m.n_layer}x{m.d_model} {'GPT-2' if m.arch == P.ARCH_GPT2 else 'Llama'} T3, "
            f"{m.n_head}x{m.head_dim} heads, FFN {m.d_ff}, vocab {m.vocab}, {P.QUANT_NAMES[m.quant]} weights, "
            f"fp16 KV; prompt {run.prompt_len} + {run.n_steps} decode steps ({samp}), batch {m.batch}")


def step_bytes(m: P.ModelSpec, pos: int) -> int:
    """Algorithmic HBM bytes of one decode step at position `pos` (0-based)."""
    wq = int(m.quantised_params_per_step() * P.BYTES_PER_WEIGHT[m.quant])
    if m.arch == P.ARCH_QWEN_TTS and m.cp_quant:  # the code predictor's matrices in their own format
        cp = m.quantised_params_per_step() - m.talker_params()
        wq = int(m.talker_params() * P.BYTES_PER_WEIGHT[m.quant] + cp * P.BYTES_PER_WEIGHT[m.cp_quant])
    d, f = m.d_model, m.d_ff
    if m.arch == P.ARCH_GPT2:
        small = m.n_layer * (4 * d + m.qkv_rows + d + f + d) + 2 * d   # norm gains/offsets + biases
        small += 2 * d                                                  # token and position rows
    else:
        small = m.n_layer * 2 * d + d + d
    small *= 4
    kv = m.batch * m.kv_bytes_per_position() * (pos + 1) + m.batch * m.kv_bytes_per_position()  # read + write
    if m.arch == P.ARCH_QWEN_TTS:
        # code predictor: positions 0..15 of each frame read their prefix (the cache restarts per frame)
        cp_pos = 2 * m.cp_layer * m.cp_n_kv_head * m.cp_head_dim * 2
        kv += m.batch * cp_pos * sum(j + 1 for j in range(m.n_codebooks))
        small += 4 * m.batch * m.n_codebooks * m.d_model                   # code-embedding rows
    return wq + small + kv


def prefill_gemm_flops(m, P):
    """2 * weights * rows for the quantised matmuls of positions 0..P-2 (every
    layer, no head), plus the causal attention products (q.k and p.v)."""
    if m.arch == ARCH_QWEN_TTS:
        per_pos = m.talker_params() - m.vocab * m.d_model
    else:
        per_pos = m.quantised_params_per_step() - m.vocab * m.d_model
    n = P - 1
    att = 4 * m.n_layer * m.n_head * m.head_dim * (n * (n + 1) // 2)
    return m.batch * (2 * per_pos * n + att)


def mean_step_bytes(m, p0, n):
    return sum(step_bytes(m, p) for p in range(p0, p0 + n)) / n


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) >= 9:
                        rows.append(p)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks not sampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, ws):
    if ws > 1:
        dist.barrier()


def max_over_ranks(dist, ws, value: float, device=None) -> float:
    """Largest value over ranks (the slowest rank's time)."""
    if ws == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import autoregressive_speech_token_gb300 as sdpkg
    from autoregressive_speech_token_gb300 import build as sdbuild
    from synth.weights import build_model_blob

    ws, rank, local = dist_env()
    dist = init_dist(ws, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sdbuild.build()

    run = get_preset(args.config)
    m = run.model
    if m.arch == P.ARCH_QWEN_TTS:
        return run_gpu_frames(args, run, torch, sdpkg, build_model_blob, ws, rank, local, dist, dev)
    K, W = args.steps, args.warmup
    if run.prompt_len + max(K, W) > m.max_ctx:
        raise SystemExit(f"steps must keep prompt + steps <= {m.max_ctx}")
    blob, _ = build_model_blob(m, seed=run.weight_seed)
    stream = torch.cuda.current_stream(dev)
    dec = sdpkg.Decoder(m, blob, device=local, stream=stream.cuda_stream)
    del blob
    ladder = bool(args.ladder)
    if ladder:
        if m.batch != 2:
            raise SystemExit("--ladder needs a two-row configuration (conditional and unconditional rows)")
        dec.set_ladder(sdpkg.SamplerLadder.from_spec(P.MTL_LADDER))
    info = dec.info()
    prompt = prompt_tokens(run)
    s = sdpkg.Sampler.from_spec(run.sampler)
    B = m.batch
    tok_rows = 1 if ladder else B      # tokens produced per step
    n_dr = max(K, W)
    draws = uniform_draws(run.draw_seed, n_dr + 1, B)[..., 0]
    u_dev = torch.from_numpy(np.ascontiguousarray(draws[1:])).to(dev)
    out_dev = torch.zeros(n_dr, B, dtype=torch.int32, device=dev)

    # warm-up: W untimed steps after a fresh prefill
    dec.reset()
    dec.prefill(prompt, s, draws[0])
    dec.decode_n(W, s, u_dev, out_dev)
    torch.cuda.synchronize()

    # timed: K steps from position prompt_len, repeated; the median repetition is the result
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = []
    with ClockSampler(local) as clk:
        for r in range(args.repeats):
            dec.reset()
            dec.prefill(prompt, s, draws[0])
            barrier(dist, ws)
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("timed")
            ev0.record(stream)
            dec.decode_n(K, s, u_dev, out_dev)
            ev1.record(stream)
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
            barrier(dist, ws)
            reps.append(max_over_ranks(dist, ws, ev0.elapsed_time(ev1), dev))
    clocks = clk.summary()
    ms_max = sorted(reps)[len(reps) // 2]
    ms = ms_max
    value = ws * K * tok_rows / (ms_max / 1e3)

    # per-step time at the start and at the end of the run's position range (10 steps each)
    at_pos = {}
    nfix = min(10, K)
    for p0 in sorted({run.prompt_len, run.prompt_len + K - nfix}):
        dec.reset()
        dec.prefill(prompt, s, draws[0])
        if p0 > run.prompt_len:
            dec.decode_n(p0 - run.prompt_len, s, u_dev, out_dev)
        torch.cuda.synchronize()
        ev0.record(stream)
        dec.decode_n(nfix, s, u_dev, out_dev)
        ev1.record(stream)
        torch.cuda.synchronize()
        at_pos[f"pos_{p0}"] = round(ev0.elapsed_time(ev1) / nfix * 1e3, 1)

    # end to end through sd_step with host buffers
    dec.reset()
    tok = dec.prefill(prompt, s, draws[0])
    Ke = min(K, 64) if args.e2e_steps is None else args.e2e_steps
    for i in range(min(3, Ke)):                       # warm the host path
        tok = dec.step(tok, s, draws[1 + i])
    dec.reset()
    tok = dec.prefill(prompt, s, draws[0])
    barrier(dist, ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(Ke):
        tok = dec.step(tok, s, draws[1 + i])
    t1 = time.perf_counter()
    e2e_s = max_over_ranks(dist, ws, t1 - t0, dev)
    e2e = ws * Ke * tok_rows / e2e_s

    # prompt prefill: positions 0..P-2 as GEMMs, then the last position's step (CUDA events around sd_prefill)
    pf_ms = []
    for _ in range(3):
        dec.reset()
        torch.cuda.synchronize()
        ev0.record(stream)
        dec.prefill(prompt, s, draws[0])
        ev1.record(stream)
        torch.cuda.synchronize()
        pf_ms.append(ev0.elapsed_time(ev1))
    pf_ms = sorted(pf_ms)[1]
    pf_flops = prefill_gemm_flops(m, run.prompt_len)
    # the same prompt length given as input vectors (sd_prefill_embeds, a conditioning prefix)
    emb = (np.random.default_rng(7).standard_normal((B, run.prompt_len, m.d_model)) * 0.05).astype(np.float32)
    pe_ms = []
    for _ in range(3):
        dec.reset()
        torch.cuda.synchronize()
        ev0.record(stream)
        dec.prefill_embeds(emb, s, draws[0])
        ev1.record(stream)
        torch.cuda.synchronize()
        pe_ms.append(ev0.elapsed_time(ev1))
    pe_ms = sorted(pe_ms)[1]

    # roofline of the decode step
    peaks, peak_kind = load_peaks()
    bytes_step = mean_step_bytes(m, run.prompt_len, K)
    achieved = bytes_step / (ms / K / 1e3) / 1e9
    step_path = "cluster" if info.persistent_clusters else ("persistent" if info.persistent else "graph")
    if ladder:
        step_path = "ladder graph"
    traffic = load_traffic(args.config, step_path)
    dec.close()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": round(ms_max / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,0.02) weights, uniform prompt IDs, "
        "Philox draws)",
        "config": {"workload": workload_text(run), "batch": B, "prompt_len": run.prompt_len,
                   "positions": [run.prompt_len, run.prompt_len + K - 1], "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2: {bytes_step / 1e6:.1f} MB streamed per step vs "
                         f"{L2_BYTES / 2 ** 20:.0f} MiB L2",
                   "kernels_per_step": info.kernels_per_step, "attn_splits": info.attn_splits,
                   **({"sampler": "guided step: rows 0 / 1 conditional / unconditional, one token per step "
                                  "through the multilingual ladder (guidance 0.5, penalty 2, T 0.8, min_p 0.05, "
                                  "top-k 1000)"} if ladder else {})},
        "e2e": {"value": round(e2e, 2), "unit": "tokens/s", "h2d_bytes_per_step": int(info.step_h2d_bytes),
                "d2h_bytes_per_step": int(info.step_d2h_bytes), "steps": Ke},
        "roofline": {"bound": "hbm",
                     "kernel": (f"decode step with the sampler ladder ({info.kernels_per_step} kernels, one CUDA "
                                f"graph)" if ladder else
                                f"decode step (cluster persistent kernel k_cstep, {info.persistent_clusters} clusters "
                                f"x {info.cluster_size} CTAs, one launch per {K} steps)" if info.persistent_clusters
                                else f"decode step (persistent kernel, {info.persistent} CTAs, one launch per {K} steps)"
                                if info.persistent else f"decode step ({info.kernels_per_step} kernels, one CUDA graph)"),
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
                     "bytes_per_step": int(bytes_step),
                     "traffic": traffic},
        "prefill": {"ms": round(pf_ms, 3), "positions": run.prompt_len, "rows": B,
                    "gemm_gflop": round(pf_flops / 1e9, 2),
                    "gemm_tflops": round(pf_flops / (pf_ms / 1e3) / 1e12, 2),
                    "path": {0: "per-position step graphs", 1: "mma.sync GEMMs", 2: "tcgen05 GEMMs"}[info.prefill],
                    "note": "sd_prefill end to end (median of 3): positions 0..P-2 as GEMMs over all rows, "
                            "the last position through the step graph",
                    "embeds_ms": round(pe_ms, 3)},
        "repetitions": {"n": len(reps), "ms_per_step": [round(x / K, 5) for x in reps],
                        "spread_ms_per_step": round((max(reps) - min(reps)) / K, 5)},
        "us_per_step_at": at_pos,
        "gpu_launches": 1 if (info.persistent and not ladder) else int(info.kernels_per_step * K),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(run, seconds=args.cpu_seconds, single_core_steps=2)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_gpu_frames(args, run, torch, sdpkg, build_model_blob, ws, rank, local, dist, dev):
    """Talker + code predictor: a step is one frame (sd_frame: the Talker step,
    15 code-predictor passes and 16 samples per row); frames are host-driven
    calls, so the device-timed and end-to-end numbers both include the per-frame
    host round trip."""
    m = run.model
    K, W = args.steps, args.warmup
    if run.prompt_len + max(K, W) > m.max_ctx:
        raise SystemExit(f"frames must keep prompt + frames <= {m.max_ctx}")
    blob, _ = build_model_blob(m, seed=run.weight_seed)
    stream = torch.cuda.current_stream(dev)
    dec = sdpkg.Decoder(m, blob, device=local, stream=stream.cuda_stream)
    del blob
    info = dec.info()
    prompt = prompt_tokens(run)
    s = sdpkg.Sampler.from_spec(run.sampler)
    B = m.batch
    draws = uniform_draws(run.draw_seed, max(K, W) + 1, B, m.n_codebooks)
    dec.reset()
    codes = dec.prefill(prompt, s, draws[0])
    for i in range(W):
        codes = dec.frame(codes, s, s, draws[1 + i])
    dec.reset()
    codes = dec.prefill(prompt, s, draws[0])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        ev0.record(stream)
        for i in range(K):
            codes = dec.frame(codes, s, s, draws[1 + i])
        ev1.record(stream)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
    barrier(dist, ws)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(dist, ws, ms, dev)
    e2e_s = max_over_ranks(dist, ws, t1 - t0, dev)
    pf_ms = []
    for _ in range(3):
        dec.reset()
        torch.cuda.synchronize()
        ev0.record(stream)
        dec.prefill(prompt, s, draws[0])
        ev1.record(stream)
        torch.cuda.synchronize()
        pf_ms.append(ev0.elapsed_time(ev1))
    pf_ms = sorted(pf_ms)[1]
    pf_flops = prefill_gemm_flops(m, run.prompt_len)
    sh_ms = None
    if run.extra.get("shared_prompt") and B > 1:  # the rollouts' one prompt computed once (sd_prefill_shared)
        sh = []
        for _ in range(3):
            dec.reset()
            torch.cuda.synchronize()
            ev0.record(stream)
            dec.prefill_shared(prompt[0], s, draws[0])
            ev1.record(stream)
            torch.cuda.synchronize()
            sh.append(ev0.elapsed_time(ev1))
        sh_ms = sorted(sh)[1]
    dec.close()
    peaks, peak_kind = load_peaks()
    bytes_frame = mean_step_bytes(m, run.prompt_len, K)
    achieved = bytes_frame / (ms / K / 1e3) / 1e9
    unit = "row-frames/s" if B > 1 else "frames/s"
    line = {
        "metric": METRIC, "value": round(ws * K * B / (ms_max / 1e3), 2), "unit": unit, "n_gpus": ws, "steps": K,
        "warmup": W, "ms_per_step": round(ms_max / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) weights, uniform prompt IDs, Philox draws)",
        "config": {"workload": workload_text(run), "batch": B, "prompt_len": run.prompt_len,
                   "positions": [run.prompt_len, run.prompt_len + K - 1], "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2: {bytes_frame / 1e6:.1f} MB streamed per frame vs "
                         f"{L2_BYTES / 2 ** 20:.0f} MiB L2",
                   "kernels_per_step": info.kernels_per_step},
        "e2e": {"value": round(ws * K * B / e2e_s, 2), "unit": unit,
                "h2d_bytes_per_step": int(info.step_h2d_bytes), "d2h_bytes_per_step": int(info.step_d2h_bytes),
                "steps": K},
        "roofline": {"bound": "hbm", "kernel": f"frame ({info.kernels_per_step} kernels, one CUDA graph)",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
                     "bytes_per_step": int(bytes_frame), "traffic": None},
        "prefill": {"ms": round(pf_ms, 3), "positions": run.prompt_len, "rows": B,
                    "gemm_gflop": round(pf_flops / 1e9, 2),
                    "gemm_tflops": round(pf_flops / (pf_ms / 1e3) / 1e12, 2),
                    "path": {0: "per-position step graphs", 1: "mma.sync GEMMs", 2: "tcgen05 GEMMs"}[info.prefill],
                    **({"shared_ms": round(sh_ms, 3)} if sh_ms is not None else {})},
        "gpu_launches": int(info.kernels_per_step * K),
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def load_traffic(config, step_path):
    """Per-step DRAM bytes from the committed ncu summary of this workload and
    step path (graph or persistent kernel), if any."""
    path = os.path.join(ROOT, "profiles", f"traffic_{config}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d.get("dram_bytes_per_step") if d.get("path", "graph") == step_path else None
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle (CPU) arm

def cpu_baseline(run, seconds: float = 15.0, single_core_steps: int = 0):
    """The oracle as it stands on the host cores: prompt processed untimed,
    then decode steps timed until about `seconds` of CPU work."""
    import oracle
    from synth.weights import build_model_blob
    m = run.model
    blob, _ = build_model_blob(m, seed=run.weight_seed)
    cores = os.cpu_count() or 1
    model = oracle.Model(blob, threads=cores)
    prompt = prompt_tokens(run)
    draws = uniform_draws(run.draw_seed, run.n_steps + 1, m.batch)[..., 0]
    z = None
    for b in range(m.batch):
        for t in prompt[b]:
            z = model.token_forward(b, int(t), m.vocab)
    sa = dict(temperature=run.sampler.temperature, top_k=run.sampler.top_k, top_p=run.sampler.top_p,
              greedy=run.sampler.greedy)
    tok = [oracle.sample(z, u=float(draws[0][b]), **sa)[0] for b in range(m.batch)]
    n = 0
    t0 = time.perf_counter()
    while n < run.n_steps:
        for b in range(m.batch):
            z = model.token_forward(b, tok[b], m.vocab)
            tok[b] = oracle.sample(z, u=float(draws[n + 1][b]), **sa)[0]
        n += 1
        if time.perf_counter() - t0 > seconds and n >= 3:
            break
    dt = time.perf_counter() - t0
    threads = model.threads
    # the same oracle on one core, a few further steps (same arithmetic, bitwise the same results)
    single = None
    if single_core_steps > 0 and n + single_core_steps < run.n_steps:
        oracle.lib().orc_set_threads(1)
        t1 = time.perf_counter()
        for i in range(single_core_steps):
            for b in range(m.batch):
                z = model.token_forward(b, tok[b], m.vocab)
                tok[b] = oracle.sample(z, u=float(draws[n + 1 + i][b]), **sa)[0]
        single = round(single_core_steps * m.batch / (time.perf_counter() - t1), 3)
        oracle.lib().orc_set_threads(threads)
    model.close()
    out = {"value": round(n * m.batch / dt, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"{n} decode steps at positions {run.prompt_len}..{run.prompt_len + n - 1} after an untimed "
                     f"{run.prompt_len}-token prompt, batch {m.batch}, {threads} OpenMP threads"}
    if single is not None:
        out["single_core"] = {"value": single, "unit": "tokens/s", "cores": 1,
                              "sample": f"{single_core_steps} further decode steps on one thread"}
    return out


def run_reference(args):
    """The oracle as the reference arm: one model and one untimed prompt prefill,
    W untimed warm-up decode steps, then (after a reset and the same prompt) K
    timed decode steps at the positions the GPU arm times (prompt_len ..
    prompt_len + K - 1), each step one oracle forward per batch row plus its
    sampler draw.  Rank 0 only."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    run = get_preset(args.config)
    m = run.model
    if m.arch == P.ARCH_QWEN_TTS:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle's Talker prompt alone takes minutes on the "
                          "host cores for this configuration; its reference arm covers the T3 configurations"}),
              flush=True)
        return
    import oracle
    from synth.weights import build_model_blob
    K, W = args.steps, args.warmup
    if run.prompt_len + max(K, W) > m.max_ctx:
        raise SystemExit(f"steps must keep prompt + steps <= {m.max_ctx}")
    blob, _ = build_model_blob(m, seed=run.weight_seed)
    cores = os.cpu_count() or 1
    model = oracle.Model(blob, threads=cores)
    prompt = prompt_tokens(run)
    draws = uniform_draws(run.draw_seed, max(K, W) + 1, m.batch)[..., 0]
    sa = dict(temperature=run.sampler.temperature, top_k=run.sampler.top_k, top_p=run.sampler.top_p,
              greedy=run.sampler.greedy)

    ladder = bool(getattr(args, "ladder", False))
    if ladder and m.batch != 2:
        raise SystemExit("--ladder needs a two-row configuration (conditional and unconditional rows)")
    lad = P.MTL_LADDER
    seen = np.zeros(m.vocab, np.uint8)

    def pick(zs, u):  # the guided step's one token from the two rows' logits (the ladder)
        return oracle.sample_ladder(zs[0], zs[1], lad.cfg_weight, seen, lad.rep_penalty, lad.temperature,
                                    lad.min_p, lad.top_p, lad.top_k, u=u)[0]

    def prefill():
        model.reset()
        seen[:] = 0
        z = None
        toks, zs = [], []
        for b in range(m.batch):
            for t in prompt[b]:
                z = model.token_forward(b, int(t), m.vocab)
            zs.append(z)
            toks.append(oracle.sample(z, u=float(draws[0][b]), **sa)[0])
        if ladder:
            t = pick(zs, float(draws[0][0]))
            toks = [t] * m.batch
        return toks

    def step(tok, i):
        if ladder:
            seen[tok[0]] = 1
            zs = [model.token_forward(b, tok[b], m.vocab) for b in range(m.batch)]
            tok[:] = [pick(zs, float(draws[i + 1][0]))] * m.batch
            return
        for b in range(m.batch):
            z = model.token_forward(b, tok[b], m.vocab)
            tok[b] = oracle.sample(z, u=float(draws[i + 1][b]), **sa)[0]

    tok = prefill()
    for i in range(W):
        step(tok, i)
    tok = prefill()
    t0 = time.perf_counter()
    for i in range(K):
        step(tok, i)
    dt = time.perf_counter() - t0
    threads = model.threads
    model.close()
    value = round(K * (1 if ladder else m.batch) / dt, 3)
    sample = (f"{K} decode steps at positions {run.prompt_len}..{run.prompt_len + K - 1} after an untimed "
              f"{run.prompt_len}-token prompt, batch {m.batch}, {threads} OpenMP threads"
              + (", the guided step (one token per step through the sampler ladder)" if ladder else ""))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": round(dt * 1e3 / max(1, K), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,0.02) weights, uniform prompt IDs, Philox draws)",
            "config": {"workload": workload_text(run), "batch": m.batch, "prompt_len": run.prompt_len,
                       "wall_s": round(dt, 1)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=250)
    ap.add_argument("--warmup", type=int, default=25)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="gpt2m_q4", choices=sorted(PRESETS))
    ap.add_argument("--ladder", action="store_true",
                    help="two-row T3 configurations: the guided step (conditional row 0, unconditional row 1, "
                         "one token per step through the multilingual sampler ladder)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--repeats", type=int, default=5, help="timed repetitions (the median is reported)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
