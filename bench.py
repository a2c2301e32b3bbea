#!/usr/bin/env python3
"""Benchmark of the Llama decoder forward pass on one GB300 (or N replicas).

One step = the whole hot path over one synthetic job of the Llama-3-8B
shape: clear the sequence, prefill a 2048-token prompt in 4 ubatches of 512
(logits for the last position only), then 128 greedy decode steps at batch 1.
Weights (16 GB) and the prompt are drawn on the device before timing.

Reported (one JSON line from rank 0):
  value      decode tok/s at batch 1 (device-resident: llm_generate replays the
             captured decode graph with no host round trip per token)
  prefill    prefill tok/s and its fraction of the bf16/fp16 dense tensor peak
  roofline   the dominant kernel (by device time in a step) against HBM
  e2e        the same metric through the public host API: llm_decode with host
             token arrays and llm_get_argmax reading each token back
  cpu_baseline  the CPU oracle timed on the host cores on a bounded sample
Multi-GPU: replicas only (the pass has no data-path exchange); value is the
sum over ranks of tokens divided by the slowest rank's time.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "decode tok/s @bs1 (% HBM roofline); prefill tok/s (% bf16 tensor peak)"

WORKLOADS = {
    # the 8B-shape job: 2048-token prompt prefilled in 4 ubatches of 512, 128 decode steps at batch 1
    "llama8b": dict(shape=synth.LLAMA_8B, seed=2, prompt=2048, n_ubatch=512, n_ctx=4096, decode=128),
    # one layer of the same shapes, for profiling a kernel with a few GB on the device
    "llama8b_1layer": dict(shape=synth.scaled_shape(synth.LLAMA_8B, n_layer=1), seed=2, prompt=512, n_ubatch=512,
                           n_ctx=1024, decode=16),
    # two layers: layer 0 runs every prefill GEMM on all rows (the last one prunes to the output rows)
    "llama8b_2layer": dict(shape=synth.scaled_shape(synth.LLAMA_8B, n_layer=2), seed=2, prompt=512, n_ubatch=512,
                           n_ctx=1024, decode=16),
    # two layers with the full 2048-token prompt: the prefill attention of every ubatch (up to 2048 keys)
    "llama8b_2layer_2048": dict(shape=synth.scaled_shape(synth.LLAMA_8B, n_layer=2), seed=2, prompt=2048,
                                n_ubatch=512, n_ctx=4096, decode=16),
    "llama1b": dict(shape=synth.LLAMA_1B, seed=1, prompt=512, n_ubatch=512, n_ctx=4096, decode=256),
}

# The other full-size configurations of the forward pass, timed in the same run
# after the headline job (one JSON object each under "workloads").
EXTRA = {
    # ~1B shape (tied output): 512-token prompt in one ubatch, 256 greedy decode steps
    "llama1b": dict(shape=synth.LLAMA_1B, seed=1, prompt=512, n_ubatch=512, n_ctx=4096, decode=256, n_seq=1),
    # 8B shape, 32000-token prompt in ubatches of 512 (n_ctx 32768), then 64 decode steps
    "llama8b_long": dict(shape=synth.LLAMA_8B, seed=3, prompt=32000, n_ubatch=512, n_ctx=32768, decode=64, n_seq=1),
    # 8B shape, tied output: 8 sequences (lengths from seed 4) prefilled in mixed
    # 512-token ubatches, then 128 decode steps of 8 rows (one per sequence)
    "llama8b_multislot": dict(shape=synth.LLAMA_8B_TIED, seed=4, prompt=0, n_ubatch=512, n_ctx=8192, decode=128,
                              n_seq=8),
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ algorithmic work

def layer_matrix_params(s):
    q, kv = s.n_head * s.head_dim, s.n_head_kv * s.head_dim
    return (q + 2 * kv) * s.n_embd + s.n_embd * q + 3 * s.n_ff * s.n_embd


# bytes a matrix element takes in the decode GEMVs: fp16, or Q8_0 (32 one-byte
# codes and one fp16 scale a block)
WEIGHT_BYTES = {"f16": 2.0, "q8_0": 34 / 32}


def decode_bytes(s, positions, wb=2.0):
    """HBM bytes one decode token must move: every weight matrix once (wb B per
    element), one embedding row (fp16), the norm gains, K and V of positions
    0..p (read) and p (write), the logits row (fp32)."""
    kvrow = s.n_layer * s.n_head_kv * s.head_dim * 2 * 2
    fixed = round((s.n_layer * layer_matrix_params(s) + s.n_vocab * s.n_embd) * wb) + s.n_embd * 2
    fixed += (2 * s.n_layer + 1) * s.n_embd * 2 + s.n_vocab * 4
    return sum(fixed + kvrow * (p + 1) + kvrow for p in positions)


def decode_step_bytes(s, positions):
    """HBM bytes of one decode step over len(positions) rows (one per
    sequence): every weight matrix once for all rows, one embedding row and
    one fp32 logits row per row, and each row's K/V of positions 0..p read
    and p written."""
    kvrow = s.n_layer * s.n_head_kv * s.head_dim * 2 * 2
    fixed = (s.n_layer * layer_matrix_params(s) + s.n_vocab * s.n_embd) * 2 + (2 * s.n_layer + 1) * s.n_embd * 2
    return fixed + sum(s.n_embd * 2 + s.n_vocab * 4 + kvrow * (p + 1) + kvrow for p in positions)


def prefill_flops_seqs(s, lens, n_out):
    """prefill_flops for several sequences prefilled together."""
    per_tok = 2 * s.n_layer * layer_matrix_params(s)
    attn = 4 * s.n_head * s.head_dim * s.n_layer * sum(n * (n + 1) // 2 for n in lens)
    return per_tok * sum(lens) + attn + 2 * s.n_embd * s.n_vocab * n_out


def prefill_gemm_flops(s, n_tokens, n_last):
    """FLOPs of the prefill GEMMs alone: every layer's matrices over all rows,
    except the last layer's MLP and the LM head, over the n_last output rows."""
    d, q, kv, f = s.n_embd, s.n_head * s.head_dim, s.n_head_kv * s.head_dim, s.n_ff
    attn_mats = (q + 2 * kv) * d + d * q
    return 2 * (s.n_layer * attn_mats * n_tokens + (s.n_layer - 1) * 3 * f * d * n_tokens
                + 3 * f * d * n_last + s.n_vocab * d * n_last)


def prefill_flops(s, n_prompt, n_out=1):
    """2 * matrix params per token, 4 * H * hd per visible key per layer
    (QK^T and PV, causal), and the LM head only for output rows."""
    per_tok = 2 * s.n_layer * layer_matrix_params(s)
    attn = 4 * s.n_head * s.head_dim * s.n_layer * sum(p + 1 for p in range(n_prompt))
    return per_tok * n_prompt + attn + 2 * s.n_embd * s.n_vocab * n_out


def kernel_bytes(s, name, wb=2.0):
    """Algorithmic HBM bytes of one launch of a decode GEMV kernel at batch 1
    (weights at wb bytes an element)."""
    d, q, kv, f = s.n_embd, s.n_head * s.head_dim, s.n_head_kv * s.head_dim, s.n_ff
    b = {
        "gemv_qkv_rope_kv": ((q + 2 * kv) * d, d * 4 + 2 * kv * 2 + q * 4),
        "gemv_o_resid": (d * q, q * 2 + 2 * d * 4),
        "gemv_gateup_swiglu": (2 * f * d, d * 4 + f * 2),
        "gemv_down_resid": (d * f, f * 2 + 2 * d * 4),
        "gemv_lm_head": (s.n_vocab * d, d * 4 + s.n_vocab * 4),
    }.get(name)
    return None if b is None else round(b[0] * wb) + b[1]


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        busy = [v for v in sm if mx and v > 0.5 * max(mx)] or sm
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ replicas

def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks of the default process group (the
    job's time is its slowest replica's); the values themselves when world is 1.
    device: where the reduction tensor lives (cuda for NCCL, cpu for gloo)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_command(n, argv, script, port):
    """The torchrun command line that runs `script` with `argv` as n ranks on
    this node (rendezvous on 127.0.0.1:port)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), script] + list(argv)


def free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(n, argv, script=None):
    """Re-run `script` (this file by default) as n ranks under torchrun, one
    per GPU, and return the launcher's exit code: `bench.py --gpus N` started
    outside torchrun starts its own N replicas."""
    return subprocess.call(replica_command(n, argv, script or os.path.abspath(__file__), free_port()))


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput of `world` replicas that each processed
    `units_per_rank` units, over the slowest replica's time in milliseconds."""
    return world * units_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ our arm

def apply_options(ctx, args):
    """Context options given as --option key=value (the library's named
    settings: kernel choices, for comparing them on the same job)."""
    for kv in args.option:
        key, _, val = kv.partition("=")
        ctx.set_option(key, int(val))


def run_ours(args, rank, world, local_rank):
    import torch
    import llama_decoder_forward_02_gb300 as L

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = WORKLOADS[args.workload]
    s = wl["shape"]
    stream = torch.cuda.Stream(device=dev)
    st = stream.cuda_stream

    with torch.cuda.stream(stream):
        tensors = synth.make_weights(s, wl["seed"], dev)
    stream.synchronize()
    model = L.Model(s, tensors, stream=st)
    if args.wtype == "q8_0":
        model.quantize(stream=st)
    wb = WEIGHT_BYTES[args.wtype]
    del tensors
    torch.cuda.empty_cache()
    ctx = L.Context(model, wl["n_ctx"], 1, wl["n_ubatch"], stream=st)
    apply_options(ctx, args)

    prompt = synth.prompt(s.n_vocab, wl["seed"], wl["prompt"])
    prompt_dev = torch.tensor(prompt, dtype=torch.int32, device=dev)
    n_dec = wl["decode"]
    gen_out = torch.zeros(n_dec, dtype=torch.int32, device=dev)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(record):
        ctx.seq_clear(0)
        if record:
            ev[0].record(stream)
        ctx.decode(token_dev_ptr=prompt_dev.data_ptr(), n_tokens=wl["prompt"])
        if record:
            ev[1].record(stream)
        ctx.generate(0, n_dec, gen_out.data_ptr())
        if record:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step(False)
    ctx.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = ctx.kernel_launches()
    pre_ms, dec_ms = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(True)
        ev[2].synchronize()
        pre_ms.append(ev[0].elapsed_time(ev[1]))
        dec_ms.append(ev[1].elapsed_time(ev[2]))
    ctx.synchronize()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    clk = clocks.stop()
    launches = ctx.kernel_launches() - launches0
    tokens_out = gen_out.cpu().tolist()

    total_pre, total_dec, wall = max_over_ranks([sum(pre_ms), sum(dec_ms), wall], world, dev)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    dec_tps = job_rate(world, n_dec * args.steps, total_dec)
    pre_tps = job_rate(world, wl["prompt"] * args.steps, total_pre)
    dec_bytes = decode_bytes(s, range(wl["prompt"], wl["prompt"] + n_dec), wb)
    dec_gbs = dec_bytes * args.steps / (total_dec / 1e3) / 1e9
    pf = prefill_flops(s, wl["prompt"])
    pre_tfs = pf * args.steps / (total_pre / 1e3) / 1e12

    result = {
        "metric": METRIC, "value": round(dec_tps, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round((total_pre + total_dec) / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: Llama-3-8B shape (vocab {s.n_vocab}, d {s.n_embd}, {s.n_layer} layers, "
                               f"{s.n_head} heads / {s.n_head_kv} KV, head_dim {s.head_dim}, FFN {s.n_ff}), "
                               f"{wl['prompt']}-token prompt prefilled in ubatches of {wl['n_ubatch']} with logits for the "
                               f"last position, then {n_dec} greedy decode steps at batch 1",
                   "global_batch": world, "seq_len": wl["prompt"] + n_dec, "n_ctx": wl["n_ctx"],
                   "parallelism": f"replicas{world}",
                   "weights": "N(0,0.02) rounded to bf16, fp16 inside" if args.wtype == "f16" else
                              "N(0,0.02) rounded to bf16, re-encoded as Q8_0 blocks (32 one-byte codes, fp16 scale); "
                              "one-row GEMVs stream the Q8_0 rows, prefill reads f16(q*d)",
                   "l2": f"inputs larger than L2 ({dec_bytes / n_dec / 1e9:.1f} GB read per decode token)",
                   **({"options": list(args.option)} if args.option else {})},
        "decode": {"tok_per_s": round(dec_tps, 3), "ms_per_token": round(total_dec / args.steps / n_dec, 4),
                   "hbm_roofline": {"bytes_per_token": round(dec_bytes / n_dec), "achieved_gbs": round(dec_gbs, 1),
                                    "peak_gbs": hbm, "frac": round(dec_gbs / hbm, 4), "peak_kind": peak_kind}},
        "prefill": {"tok_per_s": round(pre_tps, 1), "ms": round(total_pre / args.steps, 3),
                    "tensor_roofline": {"flops_per_prompt": pf, "achieved_tflops": round(pre_tfs, 1),
                                        "peak_tflops_burst": tf_burst, "frac_burst": round(pre_tfs / tf_burst, 4),
                                        "peak_tflops_sustained": tf_sust, "frac_sustained": round(pre_tfs / tf_sust, 4),
                                        "peak_kind": peak_kind}},
        "gpu_launches": int(launches),
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
        "tokens_head": tokens_out[:8],
    }

    if not args.no_kernel_timing:
        result["kernels"], result["roofline"] = kernel_breakdown(ctx, step, s, hbm, peak_kind, args, wb)
        # the prefill GEMMs alone, and prefill attention alone, against the tensor peak
        gk = [k for k in result["kernels"] if k.startswith("gemm_")]
        g_ms = sum(result["kernels"][k]["total_ms"] for k in gk)
        g_fl = prefill_gemm_flops(s, wl["prompt"], 0)
        a_ms = result["kernels"].get("attn_prefill", {}).get("total_ms")
        a_fl = 4 * s.n_head * s.head_dim * s.n_layer * sum(p + 1 for p in range(wl["prompt"]))
        result["prefill"]["gemm_only"] = {
            "kernels": gk, "ms": round(g_ms, 3), "flops": g_fl, "achieved_tflops": round(g_fl / (g_ms / 1e3) / 1e12, 1),
            "frac_burst": round(g_fl / (g_ms / 1e3) / 1e12 / tf_burst, 4),
            "frac_sustained": round(g_fl / (g_ms / 1e3) / 1e12 / tf_sust, 4), "timing": "each launch alone"}
        if a_ms:
            result["prefill"]["attention_only"] = {
                "ms": round(a_ms, 3), "flops": a_fl, "achieved_tflops": round(a_fl / (a_ms / 1e3) / 1e12, 1),
                "frac_burst": round(a_fl / (a_ms / 1e3) / 1e12 / tf_burst, 4), "timing": "each launch alone"}
    if not args.no_kernel_timing:
        result["sampling"] = sampling_timing(ctx, s, dev)
    if not args.no_e2e:
        result["e2e"] = e2e(ctx, prompt, n_dec, wl, args, world, dev)
    ctx.free()
    model.free()
    del ctx, model
    torch.cuda.empty_cache()
    if not args.no_extra:
        result["workloads"] = {name: run_extra(name, cfg, args, world, dev, stream) for name, cfg in EXTRA.items()}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(s, wl, dev)
    return result


def run_extra(name, cfg, args, world, dev, stream):
    """One of the other full-size configurations: prefill the prompt(s) as the
    configuration says, then its greedy decode steps (one row per sequence),
    with CUDA events on the context stream around each phase.  Single-sequence
    jobs decode on the device (llm_generate); the 8-sequence job decodes 8
    rows a step through llm_decode, reading the 8 argmax tokens back each step."""
    import torch
    import llama_decoder_forward_02_gb300 as L
    s, st = cfg["shape"], stream.cuda_stream
    with torch.cuda.stream(stream):
        tensors = synth.make_weights(s, cfg["seed"], dev)
    stream.synchronize()
    model = L.Model(s, tensors, stream=st)
    del tensors
    torch.cuda.empty_cache()
    n_seq = cfg["n_seq"]
    ctx = L.Context(model, cfg["n_ctx"], n_seq, cfg["n_ubatch"], stream=st)
    apply_options(ctx, args)
    if n_seq == 1:
        lens = [cfg["prompt"]]
        seqs = [synth.prompt(s.n_vocab, cfg["seed"], cfg["prompt"])]
    else:
        lens = [int(n) for n in synth.multislot_lengths(cfg["seed"], n_seq)]
        seqs = [synth.prompt(s.n_vocab, cfg["seed"], n, stream=f"seq{i}") for i, n in enumerate(lens)]
    tokens = np.concatenate(seqs)
    seq_id = np.concatenate([np.full(n, i) for i, n in enumerate(lens)]).tolist()
    out = np.zeros(len(tokens), np.int8)
    out[np.cumsum(lens) - 1] = 1
    out = out.tolist()
    tok_dev = torch.tensor(tokens, dtype=torch.int32, device=dev)
    n_dec = cfg["decode"]
    gen = torch.zeros(n_dec, dtype=torch.int32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(record):
        for q in range(n_seq):
            ctx.seq_clear(q)
        if record:
            ev[0].record(stream)
        ctx.decode(token_dev_ptr=tok_dev.data_ptr(), n_tokens=len(tokens), seq_id=seq_id, output=out)
        if record:
            ev[1].record(stream)
        if n_seq == 1:
            ctx.generate(0, n_dec, gen.data_ptr())
        else:
            rows = list(range(n_seq))
            for _ in range(n_dec):
                ctx.decode(ctx.argmax(), seq_id=rows, output=[1] * n_seq)
        if record:
            ev[2].record(stream)

    steps, warm = max(1, min(args.steps, 2)), 1
    for _ in range(warm):
        step(False)
    ctx.synchronize()
    pre_ms, dec_ms = [], []
    for _ in range(steps):
        step(True)
        ev[2].synchronize()
        pre_ms.append(ev[0].elapsed_time(ev[1]))
        dec_ms.append(ev[1].elapsed_time(ev[2]))
    ctx.synchronize()
    ctx.free()
    model.free()
    torch.cuda.empty_cache()
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    pre, dec = sum(pre_ms) / steps, sum(dec_ms) / steps
    dbytes = sum(decode_step_bytes(s, [n + k for n in lens]) for k in range(n_dec))
    pflops = prefill_flops_seqs(s, lens, n_seq)
    return {
        "config": (f"{s.n_layer} layers, d {s.n_embd}, {s.n_head}/{s.n_head_kv} heads, head_dim {s.head_dim}, "
                   f"FFN {s.n_ff}, vocab {s.n_vocab}, {'tied' if s.tied_output else 'untied'} output; "
                   f"{n_seq} sequence(s) of {lens} prompt tokens in ubatches of {cfg['n_ubatch']} (n_ctx "
                   f"{cfg['n_ctx']} each), then {n_dec} greedy decode steps of {n_seq} row(s); seed {cfg['seed']}"),
        "steps": steps, "warmup": warm,
        "decode": {"tok_per_s": round(world * n_seq * n_dec / (dec / 1e3), 2), "ms_per_step": round(dec / n_dec, 4),
                   "hbm_roofline": {"bytes_per_step_avg": round(dbytes / n_dec), "achieved_gbs": round(dbytes / (dec / 1e3) / 1e9, 1),
                                    "peak_gbs": hbm, "frac": round(dbytes / (dec / 1e3) / 1e9 / hbm, 4),
                                    "peak_kind": peak_kind}},
        "prefill": {"tok_per_s": round(world * len(tokens) / (pre / 1e3), 1), "ms": round(pre, 3),
                    "tensor_roofline": {"flops": pflops, "achieved_tflops": round(pflops / (pre / 1e3) / 1e12, 1),
                                        "peak_tflops_burst": tf_burst,
                                        "frac_burst": round(pflops / (pre / 1e3) / 1e12 / tf_burst, 4),
                                        "peak_kind": peak_kind}},
    }


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/traffic.json), or None when there is none or the kernel's source
    has changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
        if not rec:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != rec["sha256_16"]:
                return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def kernel_breakdown(ctx, step, s, hbm, peak_kind, args, wb=2.0):
    """One step with every launch bracketed by CUDA events on the context
    stream (graphs and PDL bypassed so kernels run alone): device time per
    kernel class and the roofline of the dominant one."""
    ctx.kernel_timing(1)
    step(False)
    ctx.synchronize()
    times = ctx.kernel_times()
    ctx.kernel_timing(0)
    total = sum(v[0] for v in times.values())
    table = {k: {"launches": n, "total_ms": round(ms, 3), "avg_us": round(ms / n * 1e3, 2),
                 "share": round(ms / total, 4)} for k, (ms, n) in sorted(times.items(), key=lambda kv: -kv[1][0])}
    dom = max(times, key=lambda k: times[k][0])
    ms, n = times[dom]
    avg_s = ms / n / 1e3
    b = kernel_bytes(s, dom, wb)
    if b is not None:
        ach = b / avg_s / 1e9
        # the committed ncu traffic is of the fp16 kernels
        traffic = measured_traffic(dom) if wb == WEIGHT_BYTES["f16"] else None
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": traffic, "bytes_per_launch": b,
                "avg_launch_us": round(avg_s * 1e6, 2), "peak_kind": peak_kind + " (copy bandwidth)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None,
                "traffic": None}
    return table, roof


def sampling_timing(ctx, s, dev):
    """The sampling chain (llm_op_sample) on rows of real logits: the 8B step's
    last decode logits, tiled to 8 rows.  Device time per call with CUDA events;
    a call reads each row of n_vocab fp32 logits (its algorithmic bytes) ~6 times
    (4 radix-select passes, 2 gather passes) from L2."""
    import ctypes
    import torch
    import llama_decoder_forward_02_gb300 as L
    ctx.synchronize()
    ptr, n_out = ctx.logits_ptr()
    row = L.device_view(ptr, (n_out, s.n_vocab))[-1:].clone()
    res = {}
    for n in (1, 8):
        lg = row.repeat(n, 1).contiguous()
        u = torch.rand(n, device=dev) * 0.999
        hist = torch.randint(0, s.n_vocab, (64,), dtype=torch.int32, device=dev)
        out = torch.zeros(n, dtype=torch.int32, device=dev)
        sp = L.llm_sampling(0.8, 40, 0.95, 0.05, 1.1, 64)
        st = torch.cuda.current_stream().cuda_stream

        def call():
            assert L.llm_op_sample(lg.data_ptr(), n, s.n_vocab, ctypes.byref(sp), u.data_ptr(), hist.data_ptr(), 64,
                                   out.data_ptr(), st) == 0
        for _ in range(5):
            call()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(50):
            call()
        b.record()
        b.synchronize()
        us = a.elapsed_time(b) / 50 * 1e3
        res[f"rows_{n}"] = {"us_per_call": round(us, 2), "row_bytes": s.n_vocab * 4,
                            "achieved_gbs": round(n * s.n_vocab * 4 / us / 1e3, 1)}
    res["chain"] = "repeat penalty 1.1 over 64 tokens, top-k 40, temperature 0.8, top-p 0.95, min-p 0.05"
    return res


def e2e(ctx, prompt, n_dec, wl, args, world, dev):
    """The same job through the host API: host prompt array in, one host
    token array per decode step in, each argmax read back to the host."""
    import torch
    steps = max(1, args.steps)
    dec_times, pre_times = [], []
    prompt_list = [int(v) for v in prompt]
    for _ in range(steps + 1):
        ctx.seq_clear(0)
        ctx.synchronize()
        t0 = time.perf_counter()
        ctx.decode(prompt_list)
        tok = ctx.argmax()[-1]
        t1 = time.perf_counter()
        for _ in range(n_dec):
            ctx.decode([tok])
            tok = ctx.argmax()[-1]
        t2 = time.perf_counter()
        pre_times.append(t1 - t0)
        dec_times.append(t2 - t1)
    dec = sum(dec_times[1:]) / steps
    h2d = (len(prompt_list) + n_dec) * 4
    d2h = (1 + n_dec) * 4
    return {"value": round(world * n_dec / dec, 3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "prefill_tok_per_s": round(world * len(prompt_list) / (sum(pre_times[1:]) / steps), 1),
            "steps": steps, "api": "llm_decode (host tokens) + llm_get_argmax per token"}


class OracleTimer:
    """The CPU oracle as it stands (oracle.llama, float32, every layer of the
    full model) timed on the host cores on a bounded sample of the job: an
    n-token prompt prefilled, then batch-1 decode tokens chosen by its own
    greedy argmax.  Weights are drawn where the inputs are (synth gives the
    same tensors on any device) and handed to the oracle as host bf16."""

    def __init__(self, s, seed, device):
        from oracle import llama as O
        self.O, self.s, self.seed = O, s, seed
        host = {n: synth.bf16_bits(synth.make_tensor(s, seed, n, device)) for n in synth.tensor_names(s)}
        self.model = O.Model(O.Hparams.of(s), host, np.float32)
        self.ctx, self.tok, self.n_prompt = None, 0, 0

    def prefill_seconds(self, n):
        """Seconds for an n-token prompt (one ubatch) through the whole model."""
        self.ctx = self.O.Context(self.model, n_ctx=n + 512, n_seq_max=1, n_ubatch=512)
        prompt = synth.prompt(self.s.n_vocab, self.seed, n)
        t0 = time.perf_counter()
        assert self.ctx.decode(prompt) == 0
        dt = time.perf_counter() - t0
        self.tok = int(self.O.greedy_argmax(self.ctx.logits[-1])[0])
        self.n_prompt = n
        return dt

    def decode_seconds(self):
        """Seconds for one batch-1 decode token of the whole model."""
        t0 = time.perf_counter()
        assert self.ctx.decode([self.tok]) == 0
        dt = time.perf_counter() - t0
        self.tok = int(self.O.greedy_argmax(self.ctx.logits[-1])[0])
        return dt

    def describe(self, n_decode):
        s = self.s
        return (f"oracle.llama in float32, full model ({s.n_layer} layers, vocab {s.n_vocab}, d {s.n_embd}): a "
                f"{self.n_prompt}-token prompt prefilled, then {n_decode} batch-1 decode token(s) at positions "
                f"{self.n_prompt}..; every weight matrix widened and multiplied per call, as the oracle does")


def blas_threads():
    try:
        import torch
        return torch.get_num_threads()
    except Exception:
        return None


def cpu_baseline(s, wl, device, n_prefill=64, n_decode=2):
    smp = OracleTimer(s, wl["seed"], device)
    pre = smp.prefill_seconds(n_prefill)
    dec = [smp.decode_seconds() for _ in range(n_decode)]
    per_tok = sum(dec) / len(dec)
    return {"value": round(1.0 / per_tok, 5), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "blas_threads": blas_threads(), "decode_ms_per_token": round(1e3 * per_tok, 1),
            "prefill_ms_per_token": round(1e3 * pre / n_prefill, 2), "sample": smp.describe(n_decode),
            "sample_seconds": round(pre + sum(dec), 2)}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return None
    import torch
    wl = WORKLOADS[args.workload]
    s = wl["shape"]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    smp = OracleTimer(s, wl["seed"], dev)
    n_prefill = 64
    pre = smp.prefill_seconds(n_prefill)
    times = []
    for i in range(args.warmup + args.steps):
        dt = smp.decode_seconds()
        if i >= args.warmup:
            times.append(dt)
    v = len(times) / sum(times)
    desc = smp.describe(args.warmup + args.steps) + f"; each step is one decode token (the first {args.warmup} untimed)"
    return {"metric": METRIC, "value": round(v, 5), "unit": "tok/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{args.workload}: our arm's job and metric (decode tok/s at batch 1); {desc}"},
            "cpu_baseline": {"value": round(v, 5), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                             "blas_threads": blas_threads(), "decode_ms_per_token": round(1e3 * sum(times) / len(times), 1),
                             "prefill_ms_per_token": round(1e3 * pre / n_prefill, 2), "sample": desc},
            "e2e": {"value": round(v, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b")
    ap.add_argument("--wtype", choices=sorted(WEIGHT_BYTES), default="f16",
                    help="q8_0: re-encode the model as Q8_0 blocks before the run (the JSON says so)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other full-size configurations")
    ap.add_argument("--option", action="append", default=[], metavar="KEY=VALUE",
                    help="a context option (llm_set_option) for every context of the run; the JSON lists them")
    ap.add_argument("--prompt-len", type=int, default=0,
                    help="profiling only: shorter prompt than the workload's (the JSON says so)")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="profiling only: fewer decode steps than the workload's (the JSON says so)")
    args = ap.parse_args()
    if args.prompt_len or args.decode_steps:
        wl = dict(WORKLOADS[args.workload])
        wl["prompt"] = args.prompt_len or wl["prompt"]
        wl["decode"] = args.decode_steps or wl["decode"]
        WORKLOADS[args.workload + "_profile"] = wl
        args.workload = args.workload + "_profile"

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
