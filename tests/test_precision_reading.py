"""Why the library stores its KV cache (and tensor-core operands) in fp16.

The parity bar asks per-layer hidden max |d| <= 1e-2 * rms(hidden).  With
random N(0, 0.02) weights the MLP amplifies small perturbations of the
attention output roughly tenfold, so the storage rounding of the cache alone
decides whether any implementation can meet the bar.  These CPU tests run the
oracle with its exact cache and with the cache rounded as a bf16 / fp16 store
would round it, all other arithmetic exact (float64):

* bf16 storage already breaks the bar on a medium model — so no
  implementation with a bf16 cache can meet it, whatever its other precision;
* fp16 storage (same bytes, 3 more mantissa bits) stays well inside it.
"""
import numpy as np
import pytest

import synth
from oracle import llama as O
from gpu_model_util import MED64


def per_layer_rel_err(store, shape=MED64, n=64, seed=0):
    w = synth.host_weights(synth.make_weights(shape, seed, "cpu"))
    m = O.Model(O.Hparams.of(shape), w, np.float64)
    toks = synth.prompt(shape.n_vocab, seed, n)
    out = [1] * n
    ref = O.Context(m, n_ctx=n, n_ubatch=n)
    ref.decode(toks, output=out, keep_hidden=True)
    got = O.Context(m, n_ctx=n, n_ubatch=n, kv_store=store)
    got.decode(toks, output=out, keep_hidden=True)
    return [float(np.abs(g - r).max() / np.sqrt(np.mean(r ** 2)))
            for g, r in zip(got.hidden[0], ref.hidden[0])]


def test_round_to_bf16_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, 1.0078125, -3.0e38, 1e-40], np.float32)
    r = O.round_to_bf16(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: to even (1.0); 1 + 1.5*2^-8 rounds up
    assert list(r[:4]) == [1.0, 1.0, 1.0078125, 1.0078125]
    assert r[4] == np.float32(-2.9975083e38) or abs(r[4] / -3.0e38 - 1) < 2 ** -8
    import torch
    y = np.random.default_rng(0).normal(size=10000).astype(np.float32) * 10
    assert np.array_equal(O.round_to_bf16(y), torch.from_numpy(y).to(torch.bfloat16).float().numpy())


def test_bf16_cache_alone_breaks_the_hidden_bar():
    errs = per_layer_rel_err("bf16")
    assert max(errs) > 1e-2, errs


def test_fp16_cache_meets_the_hidden_bar_with_margin():
    errs = per_layer_rel_err("fp16")
    assert max(errs) < 0.3e-2, errs
