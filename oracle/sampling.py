"""Plain oracle of the token sampling chain (test infrastructure).

Sources, cited by page title and section:

* [EN] "Inside the inference engine: model architectures and forward pass",
  section "Token sampling pipeline": temperature 0 takes the argmax; otherwise
  Top-K (keep the K highest logits) -> Temperature (scale the logits) ->
  Softmax -> Top-P (keep the cumulative probability up to p) -> Min-P (keep the
  tokens above a threshold) -> weighted random sample; a fixed seed makes
  non-greedy output reproducible.
* [LC] "LLama.cpp — how it works", "Steps 14–15: logits and sampling" (the
  sampler chain): first a repeat penalty lowers the logits of tokens that
  already appeared, then temperature, top-p, and the draw.

The chain here is the two pages' steps in their order: repeat penalty ->
top-K -> temperature -> softmax -> top-P -> min-P -> draw.  Readings where the
pages leave a step open:

* repeat penalty: each distinct token among the last ``penalty_last_n`` of
  the history has its logit divided by the penalty if it is positive and
  multiplied by it otherwise (llama.cpp's rule; penalty 1 is off);
* top-K: the K largest logits, ties broken by the lower token id; the
  candidates are kept in that order (logit descending, id ascending);
* softmax subtracts the largest scaled logit;
* top-P: the shortest prefix of the candidates whose cumulative probability
  reaches p (so at least one token survives); p >= 1 is off;
* min-P: keep the candidates whose probability is at least min_p times the
  largest probability; min_p <= 0 is off;
* the draw: with u in [0, 1) given as an input, the first kept candidate (in
  order) whose running sum of probabilities exceeds u times the kept total;
  if rounding leaves none, the last kept candidate.

Arithmetic is float32 with sums taken one element at a time in candidate
order, the precision and order in which the GPU takes the same decisions;
``decide`` also reports how close the draw came to a neighbouring token.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Params:
    temperature: float = 0.8
    top_k: int = 40
    top_p: float = 0.95
    min_p: float = 0.05
    repeat_penalty: float = 1.0
    penalty_last_n: int = 64


def penalize(logits: np.ndarray, history, penalty: float, last_n: int) -> np.ndarray:
    """[LC] repeat penalty on the distinct tokens of the last ``last_n`` history entries."""
    out = np.array(logits, dtype=np.float32, copy=True)
    if penalty == 1.0 or last_n <= 0 or len(history) == 0:
        return out
    recent = np.unique(np.asarray(history, dtype=np.int64)[-last_n:])
    pen = np.float32(penalty)
    for t in recent:
        v = out[t]
        out[t] = v / pen if v > 0 else v * pen
    return out


def top_k(logits: np.ndarray, k: int):
    """[EN] Top-K: indices and logits of the K highest, logit descending, id ascending."""
    order = np.lexsort((np.arange(logits.size), -logits.astype(np.float64)))
    idx = order[:k]
    return idx, logits[idx]


def decide(logits: np.ndarray, p: Params, u: float, history=()):
    """Token chosen for one row of logits.  Returns (token, margin): margin is
    the distance of u * total from the nearest running-sum boundary of the
    kept candidates, relative to the total (0 means a tie)."""
    logits = np.asarray(logits, dtype=np.float32)
    if p.temperature <= 0:
        return int(np.argmax(logits)), 1.0               # [EN] temperature 0 -> greedy
    x = penalize(logits, history, p.repeat_penalty, p.penalty_last_n)
    idx, vals = top_k(x, p.top_k)
    t = np.float32(p.temperature)
    scaled = (vals / t).astype(np.float32)
    e = np.exp((scaled - scaled[0]).astype(np.float32)).astype(np.float32)
    z = np.float32(0)
    for v in e:                                            # sequential float32 sum
        z = np.float32(z + v)
    prob = (e / z).astype(np.float32)
    keep = len(prob)
    if p.top_p < 1.0:
        c = np.float32(0)
        for i, v in enumerate(prob):
            c = np.float32(c + v)
            if c >= np.float32(p.top_p):
                keep = i + 1
                break
    if p.min_p > 0:
        thr = np.float32(np.float32(p.min_p) * prob[0])
        m = 0
        while m < keep and prob[m] >= thr:
            m += 1
        keep = max(m, 1)
    kept = prob[:keep]
    total = np.float32(0)
    for v in kept:
        total = np.float32(total + v)
    target = np.float32(np.float32(u) * total)
    cums, c = [], np.float32(0)
    for v in kept:
        c = np.float32(c + v)
        cums.append(c)
    choice = keep - 1                                      # rounding left none: the last kept
    for i, ci in enumerate(cums):
        if ci > target:
            choice = i
            break
    lo = float(cums[choice - 1]) if choice > 0 else 0.0
    margin = min(abs(float(target) - lo), abs(float(cums[choice]) - float(target))) / max(float(total), 1e-30)
    return int(idx[choice]), margin


def sample_rows(logits: np.ndarray, p: Params, u, history=()):
    """One token per row of ``logits`` [n][V] with the uniforms ``u`` [n]."""
    out = [decide(row, p, float(ui), history) for row, ui in zip(np.atleast_2d(logits), np.atleast_1d(u))]
    return np.array([t for t, _ in out], np.int64), np.array([m for _, m in out])
