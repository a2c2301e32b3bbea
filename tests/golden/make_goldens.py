#!/usr/bin/env python3
"""Expected logits of the full-size workloads, written by the CPU oracle alone.

The oracle (``oracle/llama.py``, float32) runs each workload end to end on the
synthetic inputs of ``synth`` (weights, prompts and sequence lengths drawn by
its counter-based generator, which gives the same tensors on the CPU and on a
GPU), choosing every decode token by its own greedy argmax.  Nothing here
reads a GPU result: the stored values are the oracle's, and the GPU tests
drive the library along the stored tokens and compare its logits with them.

Workloads (the model shapes and job sizes of the forward pass's five
configurations; ``tiny`` runs its oracle inside the tests):

  llama1b            ~1B shape (tied output), 512-token prompt in one ubatch,
                     256 greedy decode steps, n_ctx 4096
  llama8b            8B shape, 2048-token prompt in 4 ubatches of 512 (logits
                     for the last position), 128 decode steps, n_ctx 4096
  llama8b_long       8B shape, 32000-token prompt in ubatches of 512, n_ctx
                     32768, 64 decode steps
  llama8b_multislot  8B shape with tied output, 8 sequences (lengths from
                     seed 4) prefilled together in mixed 512-token ubatches
                     with the last row of each sequence as output, then 128
                     decode steps of 8 rows (one per sequence), every row an
                     output

Stored per logits row (prefill outputs first, then each decode step's rows):
the argmax, the top-2 margin, the 32 largest logits with their ids, and the
logits at a fixed random set of 512 ids; for a few rows (``full_rows``) the
whole row.  Also stored: every token stream, per-tensor checksums of the
drawn weights (so a test can tell a different draw from a wrong result) and
the oracle's wall time per prefill token and per decode step on this host.

Usage: python tests/golden/make_goldens.py WORKLOAD [--out DIR] [--layers N]
(``--layers`` truncates the model, for checking this script quickly).
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import llama as O  # noqa: E402

N_TOP = 32
N_SAMPLE = 512


def checksum(bits: np.ndarray) -> tuple[int, int]:
    """Two integer sums of a tensor's bf16 bit patterns: plain, and weighted by
    (index mod 65521) + 1.  Exact in int64 for every tensor here."""
    b = bits.reshape(-1).astype(np.int64)
    w = (np.arange(b.size, dtype=np.int64) % 65521) + 1
    return int(b.sum()), int((b * w).sum())


def summarize(rows: np.ndarray, sample_ids: np.ndarray):
    """argmax, top-2 margin, top-N_TOP ids/values and the sampled values of
    each logits row (float32)."""
    rows = np.asarray(rows, dtype=np.float32)
    top = np.argsort(-rows, axis=1, kind="stable")[:, :N_TOP]
    top_vals = np.take_along_axis(rows, top, axis=1)
    srt = np.sort(rows, axis=1)
    return (np.argmax(rows, axis=1).astype(np.int32), (srt[:, -1] - srt[:, -2]).astype(np.float32),
            top.astype(np.int32), top_vals, rows[:, sample_ids])


def workload(name: str, layers: int | None):
    wl = {"llama1b": synth.WORKLOADS[1], "llama8b": synth.WORKLOADS[2], "llama8b_long": synth.WORKLOADS[3],
          "llama8b_multislot": synth.WORKLOADS[4]}[name]
    shape = wl.shape if not layers else synth.scaled_shape(wl.shape, n_layer=layers)
    return wl, shape


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("workload", choices=("llama1b", "llama8b", "llama8b_long", "llama8b_multislot"))
    ap.add_argument("--out", default=HERE)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--steps", type=int, default=0, help="fewer decode steps (checking this script)")
    args = ap.parse_args()
    wl, s = workload(args.workload, args.layers)
    steps = args.steps or wl.decode_steps
    log = lambda msg: print(f"[{time.strftime('%H:%M:%S')}] {args.workload}: {msg}", flush=True)

    t0 = time.time()
    names = synth.tensor_names(s)
    host, sums = {}, {}
    for n in names:
        bits = synth.bf16_bits(synth.make_tensor(s, wl.seed, n, "cpu"))
        host[n] = bits
        sums[n] = checksum(bits)
    log(f"weights drawn in {time.time() - t0:.0f} s")
    model = O.Model(O.Hparams.of(s), host, np.float32)
    ctx = O.Context(model, wl.n_ctx, wl.n_seq, wl.n_ubatch)

    if wl.n_seq == 1:
        prompt = synth.prompt(s.n_vocab, wl.seed, wl.prompt_len)
        seqs = [prompt]
        tokens, seq_id = prompt, np.zeros(len(prompt), np.int64)
        out = np.zeros(len(prompt), np.int8)
        out[-1] = 1
    else:
        lens = synth.multislot_lengths(wl.seed, wl.n_seq)
        seqs = [synth.prompt(s.n_vocab, wl.seed, int(n), stream=f"seq{i}") for i, n in enumerate(lens)]
        tokens = np.concatenate(seqs)
        seq_id = np.concatenate([np.full(len(x), i) for i, x in enumerate(seqs)])
        out = np.zeros(len(tokens), np.int8)
        out[np.cumsum([len(x) for x in seqs]) - 1] = 1

    t1 = time.time()
    assert ctx.decode(tokens, seq=seq_id, output=out) == O.OK
    prefill_s = time.time() - t1
    log(f"prefill of {len(tokens)} tokens in {prefill_s:.0f} s")
    rows = [ctx.logits.astype(np.float32).copy()]           # [n_seq][V]
    chosen = []                                             # [steps][n_seq]
    step_s = []
    for k in range(steps):
        nxt = O.greedy_argmax(rows[-1]).astype(np.int64)
        chosen.append(nxt)
        t2 = time.time()
        assert ctx.decode(nxt, seq=np.arange(wl.n_seq), output=np.ones(wl.n_seq, np.int8)) == O.OK
        step_s.append(time.time() - t2)
        rows.append(ctx.logits.astype(np.float32).copy())
        if k % 8 == 0 or k == steps - 1:
            log(f"decode step {k + 1}/{steps} ({step_s[-1]:.1f} s)")
    logits = np.concatenate(rows)                           # [(steps + 1) * n_seq][V]
    n = wl.n_seq
    # whole rows: the prefill outputs, the first and the last decode step
    full_rows = np.unique(np.concatenate([np.arange(n), n + np.arange(n), steps * n + np.arange(n)]))
    rng = np.random.default_rng(1000 + wl.seed)
    sample_ids = np.sort(rng.choice(s.n_vocab, N_SAMPLE, replace=False)).astype(np.int32)
    amax, margin, top_ids, top_vals, sample_vals = summarize(logits, sample_ids)

    path = os.path.join(args.out, f"{args.workload}{'_L%d' % args.layers if args.layers else ''}.npz")
    np.savez_compressed(
        path,
        workload=args.workload, seed=wl.seed, n_layer=s.n_layer, n_ctx=wl.n_ctx, n_ubatch=wl.n_ubatch,
        n_seq=n, steps=steps,
        seq_lens=np.array([len(x) for x in seqs], np.int32), prompt_tokens=tokens.astype(np.int32),
        seq_id=seq_id.astype(np.int32), out_flags=out,
        decode_tokens=np.array(chosen, np.int32).reshape(steps, n),
        argmax=amax, margin=margin, top_ids=top_ids, top_vals=top_vals,
        sample_ids=sample_ids, sample_vals=sample_vals,
        full_rows=full_rows.astype(np.int32), full=logits[full_rows],
        weight_names=np.array(names), weight_sums=np.array([sums[k] for k in names], np.int64),
        oracle_prefill_s_per_token=prefill_s / len(tokens),
        oracle_decode_s_per_step=float(np.mean(step_s)) if step_s else 0.0,
        oracle_host=f"{os.cpu_count()} cores, numpy {np.__version__}",
    )
    log(f"wrote {path} ({os.path.getsize(path) / 1e6:.1f} MB) after {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
