"""Parity at the full sizes of the 8B-shape workloads, through the C ABI.

* 8B, 2048-token prompt in 4 ubatches of 512 (the configuration bench.py
  times): the float32 oracle runs the whole model, so the logits of the prompt
  and of two decode steps (driven along the oracle's greedy tokens) are
  compared with the bar: max |dlogit| <= 5e-2 and top-1 agreement.
* 8B, 32k context (32000-token prompt in 63 ubatches, then decode), and
  8 sequences with separate caches prefilled in mixed 512-token ubatches, then
  decoded 8 rows at a time: the oracle cannot run these to full depth in a
  test, so it computes layer 0 for sampled rows (oracle.layer_rows: K/V of
  every row, Q, attention, O and MLP for the sampled ones) and the GPU's
  layer-0 hidden state of the same rows (llm_debug_hidden) must be within
  1e-2 * rms of it.  The samples reach every ubatch (positions up to 32k), the
  rows next to sequence boundaries inside mixed ubatches, and the decode rows,
  whose attention spans the whole cache.  At full depth the multi-sequence
  job checks a property: a sequence's decode logits in the batched step equal
  its logits decoded alone in a fresh context.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import llama as O
from gpu_model_util import LOGIT_TOL, HIDDEN_REL_TOL, compare_logits, top1_agreement

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LAYER0 = ("attn_norm", "attn_q", "attn_k", "attn_v", "attn_output", "ffn_norm", "ffn_gate", "ffn_up", "ffn_down")


@pytest.fixture(scope="module")
def lib():
    import llama_decoder_forward_02_gb300 as L
    return L


def stream():
    return torch.cuda.current_stream().cuda_stream


def build(lib, shape, seed, names=None):
    """The model on the GPU (weights drawn on the device) and host bf16 copies
    of `names` (all tensors when None) for the oracle."""
    t = synth.make_weights(shape, seed, "cuda")
    host = {k: synth.bf16_bits(v) for k, v in t.items() if names is None or k in names}
    model = lib.Model(shape, t, stream=stream())
    del t
    torch.cuda.empty_cache()
    return model, host


def layer0_names():
    return ["token_embd"] + [f"blk.0.{n}" for n in LAYER0]


def hidden_check(got, ref, what):
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    err = float(np.abs(got - ref).max())
    assert err <= HIDDEN_REL_TOL * rms, f"{what}: max |d| {err:.3e} > {HIDDEN_REL_TOL} * rms {rms:.3e}"
    return err / rms


def test_llama8b_2048_prompt_full_depth(lib):
    wl = synth.WORKLOADS[2]
    s = wl.shape
    model, host = build(lib, s, wl.seed)
    ctx = lib.Context(model, wl.n_ctx, 1, wl.n_ubatch, stream=stream())
    prompt = synth.prompt(s.n_vocab, wl.seed, wl.prompt_len)
    steps = 2
    oc = O.Context(O.Model(O.Hparams.of(s), host, np.float32), wl.n_ctx, 1, wl.n_ubatch)
    ref_tokens, ref_logits = O.generate_greedy(oc, prompt, steps)
    assert ctx.decode(prompt) == 0
    ctx.synchronize()
    got = [lib.logits_numpy(ctx, s.n_vocab)[-1]]
    for t in ref_tokens:
        assert ctx.decode([int(t)]) == 0
        ctx.synchronize()
        got.append(lib.logits_numpy(ctx, s.n_vocab)[-1])
    got = np.array(got)
    err = compare_logits(got, ref_logits)
    frac, _ = top1_agreement(got, ref_logits)
    assert frac >= 0.99
    print(f"8B 2048-token prompt + {steps} decode steps: max |dlogit| {err:.3e}, top-1 agreement {frac:.3f}")
    ctx.free()
    model.free()


def test_llama8b_32k_context_layer0_sampled(lib):
    wl = synth.WORKLOADS[3]
    s = wl.shape
    model, host = build(lib, s, wl.seed, layer0_names())
    ctx = lib.Context(model, wl.n_ctx, 1, wl.n_ubatch, stream=stream())
    prompt = synth.prompt(s.n_vocab, wl.seed, wl.prompt_len)
    n_ub = -(-wl.prompt_len // wl.n_ubatch)
    R = 2                                            # first rows of every ubatch
    dbg = torch.zeros((n_ub, s.n_layer, R, s.n_embd), dtype=torch.float32, device="cuda")
    ctx.debug_hidden(dbg.data_ptr(), R, n_ub)
    assert ctx.decode(prompt) == 0
    ctx.synchronize()
    gpu_rows = dbg[:, 0].cpu().numpy().reshape(n_ub * R, s.n_embd)
    rows = [u * wl.n_ubatch + r for u in range(n_ub) for r in range(R)]
    assert np.isfinite(lib.logits_numpy(ctx, s.n_vocab)).all()
    # two decode steps at positions 32000 and 32001, layer 0 of each
    toks = list(prompt)
    dec = torch.zeros((1, s.n_layer, 1, s.n_embd), dtype=torch.float32, device="cuda")
    gpu_dec = []
    for _ in range(2):
        tok = int(ctx.argmax()[-1])
        toks.append(tok)
        ctx.debug_hidden(dec.data_ptr(), 1, 1)
        assert ctx.decode([tok]) == 0
        ctx.synchronize()
        gpu_dec.append(dec[0, 0, 0].cpu().numpy().copy())
    ctx.debug_hidden(0, 0, 0)

    om = O.Model(O.Hparams.of(s), host, np.float32)
    h = om.embed_rows(np.array(toks))
    ref = O.layer_rows(om.hp, om.layer(0), h, np.arange(len(toks)), rows + [len(toks) - 2, len(toks) - 1])
    a = hidden_check(gpu_rows, ref[:len(rows)], "prefill rows, layer 0")
    b = hidden_check(np.array(gpu_dec), ref[len(rows):], "decode rows at 32000-32001, layer 0")
    print(f"8B 32k context, layer 0: prefill rows max|d|/rms {a:.2e}, decode rows {b:.2e}")
    ctx.free()
    model.free()


def test_llama8b_multislot_layer0_sampled_and_isolation(lib):
    wl = synth.WORKLOADS[4]
    s = wl.shape
    model, host = build(lib, s, wl.seed, layer0_names())
    lens = synth.multislot_lengths(wl.seed, wl.n_seq)
    seqs = [synth.prompt(s.n_vocab, wl.seed, int(n), stream=f"seq{i}") for i, n in enumerate(lens)]
    tokens = np.concatenate(seqs)
    seq_id = np.concatenate([np.full(len(x), i) for i, x in enumerate(seqs)])
    ends = np.cumsum(lens) - 1
    out = np.zeros(len(tokens), np.int8)
    out[ends] = 1
    ctx = lib.Context(model, wl.n_ctx, wl.n_seq, wl.n_ubatch, stream=stream())
    n_ub = -(-len(tokens) // wl.n_ubatch)
    dbg = torch.zeros((n_ub, s.n_layer, wl.n_ubatch, s.n_embd), dtype=torch.float32, device="cuda")
    ctx.debug_hidden(dbg.data_ptr(), wl.n_ubatch, n_ub)
    assert ctx.decode(tokens, seq_id=seq_id, output=out) == 0
    ctx.synchronize()
    gpu_l0 = dbg[:, 0].cpu().numpy().reshape(n_ub * wl.n_ubatch, s.n_embd)
    del dbg
    torch.cuda.empty_cache()
    prefill_logits = lib.logits_numpy(ctx, s.n_vocab)
    assert prefill_logits.shape == (wl.n_seq, s.n_vocab) and np.isfinite(prefill_logits).all()

    # one batched decode step: a row per sequence, logits for every row
    nxt = np.argmax(prefill_logits, axis=1)
    dec = torch.zeros((1, s.n_layer, wl.n_seq, s.n_embd), dtype=torch.float32, device="cuda")
    ctx.debug_hidden(dec.data_ptr(), wl.n_seq, 1)
    assert ctx.decode(nxt.tolist(), seq_id=list(range(wl.n_seq)), output=[1] * wl.n_seq) == 0
    ctx.synchronize()
    ctx.debug_hidden(0, 0, 0)
    gpu_dec = dec[0, 0].cpu().numpy()
    batched_logits = lib.logits_numpy(ctx, s.n_vocab)

    # layer 0 of sampled rows of every sequence: both ends, the ubatch borders
    # that fall inside it, and a few more
    om = O.Model(O.Hparams.of(s), host, np.float32)
    lw = om.layer(0)
    rng = np.random.default_rng(4)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    got, ref = [], []
    for i, x in enumerate(seqs):
        g0, n = int(starts[i]), len(x)
        cand = {0, n - 1, *rng.integers(0, n, 4).tolist()}
        cand |= {p for p in range(n) if (g0 + p) % wl.n_ubatch in (0, wl.n_ubatch - 1)}
        ps = sorted(cand)
        full = np.concatenate([x, [nxt[i]]])
        r = O.layer_rows(om.hp, lw, om.embed_rows(full), np.arange(n + 1), ps + [n])
        got.append(gpu_l0[[g0 + p for p in ps]])
        got.append(gpu_dec[i:i + 1])
        ref.append(r)
    a = hidden_check(np.concatenate(got), np.concatenate(ref), "multi-sequence rows, layer 0")
    print(f"8B 8 sequences, layer 0 of {sum(len(r) for r in ref)} sampled rows: max|d|/rms {a:.2e}")

    # full depth: a sequence decoded alone gives the logits it got in the batch
    for i in (int(np.argmin(lens)), int(np.argmax(lens))):
        alone = lib.Context(model, wl.n_ctx, 1, wl.n_ubatch, stream=stream())
        assert alone.decode(seqs[i]) == 0
        assert alone.decode([int(nxt[i])]) == 0
        alone.synchronize()
        e = compare_logits(lib.logits_numpy(alone, s.n_vocab), batched_logits[i:i + 1], tol=LOGIT_TOL)
        print(f"sequence {i} ({lens[i]} tokens) alone vs batched: max |dlogit| {e:.3e}")
        alone.free()
    ctx.free()
    model.free()
