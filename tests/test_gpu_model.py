"""End-to-end parity of the CUDA forward pass (through the C ABI) with the
CPU oracle on the same seeded inputs.

Bar: max |dlogit| <= 5e-2; per-layer hidden max |d| <= 1e-2 * rms(hidden);
identical greedy tokens on the tiny model; >= 99% top-1 agreement where the
oracle's top-2 margin exceeds 0.1.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import llama as O
from gpu_model_util import (Pair, MED64, MED128, compare_logits, top1_agreement, HIDDEN_REL_TOL)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import llama_decoder_forward_02_gb300 as L
    return L


@pytest.fixture(scope="module")
def tiny(lib):
    return lambda **kw: Pair(lib, synth.TINY, 0, **{"n_ctx": 64, **kw})


# ---------------------------------------------------------------- tiny model (16 + 16 greedy)

def test_tiny_greedy_tokens_identical(tiny):
    p = tiny(n_ubatch=16)
    prompt = synth.prompt(512, 0, 16)
    ref_tokens, ref_logits = O.generate_greedy(p.oc, prompt, 16)
    assert p.ctx.decode(prompt) == 0
    got_logits = [p.logits()[-1]]
    tokens = []
    for step in range(16):
        tok = p.ctx.argmax()[-1]
        tokens.append(tok)
        assert p.ctx.decode([tok]) == 0
        got_logits.append(p.logits()[-1])
    assert tokens == list(ref_tokens)
    compare_logits(np.array(got_logits), ref_logits)
    p.free()


def test_tiny_generate_on_device(tiny):
    p = tiny(n_ubatch=16)
    prompt = synth.prompt(512, 0, 16)
    ref_tokens, ref_logits = O.generate_greedy(p.oc, prompt, 16)
    out = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert p.ctx.decode(prompt) == 0
    assert p.ctx.generate(0, 16, out.data_ptr()) == 0
    p.ctx.synchronize()
    assert out.cpu().tolist() == list(ref_tokens)
    assert p.ctx.seq_pos_max(0) == 31
    compare_logits(p.logits(), ref_logits[-1:])
    # a second call continues from the last logits
    ref2, ref2_logits = O.generate_greedy(O.Context(p.om, 64), prompt, 24)
    assert p.ctx.generate(0, 8, out.data_ptr()) == 0
    p.ctx.synchronize()
    assert out[:8].cpu().tolist() == list(ref2[16:24])
    compare_logits(p.logits(), ref2_logits[-1:])
    p.free()


def test_tiny_hidden_states_per_layer(tiny):
    p = tiny(n_ubatch=16)
    prompt = synth.prompt(512, 0, 16)
    L, d = synth.TINY.n_layer, synth.TINY.n_embd
    buf = torch.zeros((1, L, 16, d), device="cuda")
    p.ctx.debug_hidden(buf.data_ptr(), 16, 1)
    out = [1] * 16
    assert p.ctx.decode(prompt, output=out) == 0
    p.ctx.synchronize()
    assert p.oc.decode(prompt, output=out, keep_hidden=True) == 0
    got = buf.cpu().double().numpy()[0]
    for layer in range(L):
        ref = p.oc.hidden[0][layer]
        rms = np.sqrt(np.mean(ref ** 2))
        err = np.abs(got[layer] - ref).max()
        assert err <= HIDDEN_REL_TOL * rms, (layer, err, rms)
    compare_logits(p.logits(), p.oc.logits)
    p.free()


@pytest.mark.parametrize("graphs,pdl", [(0, 0), (1, 0), (0, 1)])
def test_graphs_and_pdl_do_not_change_results(tiny, graphs, pdl):
    base, alt = tiny(n_ubatch=16), tiny(n_ubatch=16)
    alt.ctx.set_option("graphs", graphs)
    alt.ctx.set_option("pdl", pdl)
    prompt = synth.prompt(512, 0, 12)
    for q in (base, alt):
        assert q.ctx.decode(prompt) == 0
    for tok in (5, 77, 300, 12):
        for q in (base, alt):
            assert q.ctx.decode([tok]) == 0
        assert np.array_equal(base.logits(), alt.logits())
    base.free(); alt.free()


def test_decode_step_on_prefill_kernels(tiny):
    # ubatches of 1 row sent through the GEMM path must agree with the oracle too
    p = tiny(n_ubatch=16)
    p.ctx.set_option("gemv_path_max_rows", 0)
    prompt = synth.prompt(512, 0, 16)
    assert p.ctx.decode(prompt) == 0 and p.oc.decode(prompt) == 0
    for tok in (1, 2, 3):
        assert p.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        compare_logits(p.logits(), p.oc.logits)
    p.free()


# ---------------------------------------------------------------- ragged ubatches, pruning, sequences

@pytest.mark.parametrize("shape,n_ubatch", [(MED64, 64), (MED128, 100), (MED64, 7)])
def test_ragged_ubatches_and_output_rows(lib, shape, n_ubatch):
    p = Pair(lib, shape, 11, n_ctx=512, n_ubatch=n_ubatch)
    n = 150
    prompt = synth.prompt(shape.n_vocab, 11, n)
    out = np.zeros(n, np.int8)
    out[[0, 9, 63, 64, 99, 100, 149]] = 1
    assert p.ctx.decode(prompt, output=out) == 0
    assert p.oc.decode(prompt, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    # a few decode steps with the cache
    for tok in (3, 1000 % shape.n_vocab, 42):
        assert p.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        compare_logits(p.logits(), p.oc.logits)
    p.free()


def test_multi_sequence_prefill_and_batched_decode(lib):
    shape = MED64
    p = Pair(lib, shape, 4, n_ctx=256, n_seq=4, n_ubatch=64)
    lens = [70, 5, 130, 33]
    tokens, seq = [], []
    for s, n in enumerate(lens):
        tokens += list(synth.prompt(shape.n_vocab, 100 + s, n))
        seq += [s] * n
    out = np.zeros(len(tokens), np.int8)
    ends = np.cumsum(lens) - 1
    out[ends] = 1
    assert p.ctx.decode(tokens, seq_id=seq, output=out) == 0
    assert p.oc.decode(tokens, seq=seq, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    # batched decode: one row per sequence, in a shuffled order, 3 steps
    order = [2, 0, 3, 1]
    for step in range(3):
        toks = [(7 * step + 13 * s) % shape.n_vocab for s in order]
        assert p.ctx.decode(toks, seq_id=order, output=[1] * 4) == 0
        assert p.oc.decode(toks, seq=order, output=[1] * 4) == 0
        compare_logits(p.logits(), p.oc.logits)
    # interleaved rows of two sequences in one small ubatch (not all outputs)
    assert p.ctx.decode([1, 2, 3, 4], seq_id=[0, 1, 0, 1], output=[0, 1, 1, 0]) == 0
    assert p.oc.decode([1, 2, 3, 4], seq=[0, 1, 0, 1], output=[0, 1, 1, 0]) == 0
    compare_logits(p.logits(), p.oc.logits)
    for s in range(4):
        assert p.ctx.seq_pos_max(s) == p.oc.seq_pos_max(s)
    p.free()


def test_sequence_clear_and_reuse(lib):
    p = Pair(lib, MED64, 3, n_ctx=128, n_seq=2, n_ubatch=32)
    a = synth.prompt(MED64.n_vocab, 1, 40)
    assert p.ctx.decode(a) == 0
    first = p.logits()
    p.ctx.seq_clear(0)
    assert p.ctx.seq_pos_max(0) == -1
    assert p.ctx.decode(a) == 0
    assert np.array_equal(p.logits(), first)
    p.free()


# ---------------------------------------------------------------- error paths

def test_error_codes_leave_state_unchanged(lib):
    p = Pair(lib, MED64, 5, n_ctx=32, n_seq=2, n_ubatch=16)
    L = lib
    ctx = p.ctx
    with pytest.raises(L.LlmError):
        ctx.decode([MED64.n_vocab])                 # token out of range
    with pytest.raises(L.LlmError):
        ctx.decode([1], seq_id=[2])                 # sequence out of range
    with pytest.raises(L.LlmError):
        ctx.decode([1, 2], pos=[0, 2])              # gap
    assert ctx.decode(list(range(30))) == 0
    assert ctx.decode([1, 2, 3]) == L.LLM_NO_KV_ROOM  # 30, 31, 32 -> 32 >= n_ctx
    assert ctx.seq_pos_max(0) == 29
    assert ctx.decode([1, 2]) == 0
    assert ctx.seq_pos_max(0) == 31
    # device tokens out of range: the embedding kernel raises the error flag
    bad = torch.tensor([MED64.n_vocab + 5], dtype=torch.int32, device="cuda")
    assert ctx.decode(token_dev_ptr=bad.data_ptr(), n_tokens=1, seq_id=[1]) == 0
    with pytest.raises(L.LlmError):
        ctx.synchronize()
    ctx.synchronize()                               # flag was cleared
    p.free()


def test_fp16_activation_overflow_is_reported(lib):
    """An activation that cannot be stored as fp16 (here the first RMSNorm's
    x = h * gain, with the embedding scaled by 100 and that gain by 6e4) raises
    the error flag: llm_synchronize fails naming it, after a one-row decode step
    and after a prefill ubatch, and clean work afterwards reports nothing."""
    shape = synth.TINY
    st = torch.cuda.current_stream().cuda_stream
    t = synth.make_weights(shape, 81, "cpu")
    t["token_embd"] = (t["token_embd"].float() * 100).to(torch.bfloat16)
    t["blk.0.attn_norm"] = (t["blk.0.attn_norm"].float() * 6e4).to(torch.bfloat16)
    model = lib.Model(shape, {k: v.cuda() for k, v in t.items()}, stream=st)
    ctx = lib.Context(model, 64, 1, 16, stream=st)
    assert ctx.decode([5]) == 0
    with pytest.raises(lib.LlmError, match="fp16"):
        ctx.synchronize()
    ctx.synchronize()                                # cleared
    ctx.seq_clear(0)
    assert ctx.decode(synth.prompt(shape.n_vocab, 81, 12)) == 0
    with pytest.raises(lib.LlmError, match="fp16"):
        ctx.synchronize()
    ctx.free()
    model.free()


def test_device_tokens_match_host_tokens(lib):
    a, b = Pair(lib, MED64, 6, n_ctx=128, n_ubatch=32), Pair(lib, MED64, 6, n_ctx=128, n_ubatch=32)
    prompt = synth.prompt(MED64.n_vocab, 6, 50)
    dev = torch.tensor(prompt, dtype=torch.int32, device="cuda")
    assert a.ctx.decode(prompt) == 0
    assert b.ctx.decode(token_dev_ptr=dev.data_ptr(), n_tokens=50) == 0
    assert np.array_equal(a.logits(), b.logits())
    one = torch.tensor([17], dtype=torch.int32, device="cuda")
    assert a.ctx.decode([17]) == 0
    assert b.ctx.decode(token_dev_ptr=one.data_ptr(), n_tokens=1) == 0
    assert np.array_equal(a.logits(), b.logits())
    a.free(); b.free()


# ---------------------------------------------------------------- full-size 1B shape

@pytest.mark.slow
def test_llama1b_prefill_512_and_decode(lib):
    wl = synth.WORKLOADS[1]
    p = Pair(lib, wl.shape, wl.seed, n_ctx=wl.n_ctx, n_ubatch=wl.n_ubatch, dtype=np.float32, device_draw=True)
    prompt = synth.prompt(wl.shape.n_vocab, wl.seed, wl.prompt_len)
    steps = 6
    ref_tokens, ref_logits = O.generate_greedy(p.oc, prompt, steps)
    assert p.ctx.decode(prompt) == 0
    got = [p.logits()[-1]]
    for t in ref_tokens:                        # drive the GPU along the oracle's tokens
        assert p.ctx.decode([int(t)]) == 0
        got.append(p.logits()[-1])
    got = np.array(got)
    compare_logits(got, ref_logits)
    frac, n = top1_agreement(got, ref_logits)
    assert frac >= 0.99, (frac, n)
    p.free()


@pytest.mark.parametrize("gemm,attn", [(2, 0), (3, 1), (2, 2)])
@pytest.mark.parametrize("shape,n_ubatch", [(MED64, 64), (MED128, 100), (synth.TINY, 16)])
def test_prefill_on_both_gemm_kernels(lib, shape, n_ubatch, gemm, attn):
    """Prefill through each GEMM schedule (tcgen05 CTA pairs, persistent past
    one wave, the default; persistent pairs for every GEMM) and each prefill
    attention kernel (mma.sync; tcgen05 one CTA per head; tcgen05 CTA pairs,
    the default, where head_dim is 128 and the GQA group even)."""
    p = Pair(lib, shape, 21, n_ctx=512, n_ubatch=n_ubatch)
    p.ctx.set_option("gemm", gemm)
    p.ctx.set_option("attn_prefill", attn)
    n = 150
    prompt = synth.prompt(shape.n_vocab, 21, n)
    out = np.zeros(n, np.int8)
    out[[0, 40, 99, 100, 149]] = 1
    assert p.ctx.decode(prompt, output=out) == 0
    assert p.oc.decode(prompt, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    # every row an output: the LM head runs on the tensor-core GEMM too
    more = synth.prompt(shape.n_vocab, 22, 20)
    assert p.ctx.decode(more, output=[1] * 20) == 0
    assert p.oc.decode(more, output=[1] * 20) == 0
    compare_logits(p.logits(), p.oc.logits)
    p.free()


@pytest.mark.parametrize("gemm,resid_tma,split_k", [(2, 1, 1), (2, 1, 0), (2, 0, 1), (3, 1, 1), (4, 1, 1)])
def test_prefill_cta_pair_gemms(lib, gemm, resid_tma, split_k):
    """Every prefill GEMM of a layer (QKV + RoPE + KV append, O + residual,
    gate/up + SwiGLU, down + residual) on tcgen05 CTA pairs against the oracle,
    with a full 256-row ubatch and a ragged 44-row one; the residual epilogue
    through shared memory and TMA stores (default) and row by row, and the
    down projection (K = 8200 padded) with K split in two over 256-wide tiles
    (default) and not."""
    shape = synth.Shape(n_vocab=1024, n_embd=2048, n_layer=1, n_head=16, n_head_kv=4, head_dim=128, n_ff=8200,
                        rms_eps=1e-5, rope_theta=10000.0, tied_output=False)
    p = Pair(lib, shape, 43, n_ctx=512, n_ubatch=256, dtype=np.float32)
    p.ctx.set_option("gemm", gemm)
    p.ctx.set_option("gemm_resid_tma", resid_tma)
    p.ctx.set_option("gemm_split_k", split_k)
    prompt = synth.prompt(shape.n_vocab, 43, 300)
    out = np.zeros(300, np.int8)
    out[[0, 255, 256, 299]] = 1
    assert p.ctx.decode(prompt, output=out) == 0
    assert p.oc.decode(prompt, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    p.free()


def test_split_k_gemms_on_two_streams(lib):
    """Two contexts of one model prefill at the same time on two streams. The
    halves of the split-K down projection wait on each other (the launch is
    cooperative, so both are resident whatever else runs). Each context must
    give exactly the logits of the context prefilling alone, and those must
    match the oracle."""
    shape = synth.Shape(n_vocab=1024, n_embd=2048, n_layer=1, n_head=16, n_head_kv=4, head_dim=128, n_ff=8200,
                        rms_eps=1e-5, rope_theta=10000.0, tied_output=False)
    p = Pair(lib, shape, 47, n_ctx=512, n_ubatch=256, dtype=np.float32)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    c1 = lib.Context(p.model, 512, 1, 256, stream=s1.cuda_stream)
    c2 = lib.Context(p.model, 512, 1, 256, stream=s2.cuda_stream)
    prompt = synth.prompt(shape.n_vocab, 47, 300)
    out = np.zeros(300, np.int8)
    out[[0, 255, 299]] = 1
    # a first prefill on each context sizes its buffers (which synchronizes);
    # after clearing, the two prefills are only enqueued, and they overlap
    for c in (c1, c2):
        assert c.decode(prompt, output=out) == 0
        c.synchronize()
        c.seq_clear(0)
    assert c1.decode(prompt, output=out) == 0
    assert c2.decode(prompt, output=out) == 0
    c1.synchronize()
    c2.synchronize()
    assert p.ctx.decode(prompt, output=out) == 0
    ref = p.logits()
    assert np.array_equal(lib.logits_numpy(c1, shape.n_vocab), ref)
    assert np.array_equal(lib.logits_numpy(c2, shape.n_vocab), ref)
    assert p.oc.decode(prompt, output=out) == 0
    compare_logits(ref, p.oc.logits)
    c1.free()
    c2.free()
    p.free()


STREAM_SHAPE = synth.Shape(n_vocab=4096, n_embd=1024, n_layer=2, n_head=8, n_head_kv=2, head_dim=128, n_ff=3584,
                           rms_eps=1e-5, rope_theta=10000.0, tied_output=False)


@pytest.mark.parametrize("shape", [MED64, MED128, STREAM_SHAPE])
def test_batch1_streamed_gemvs(lib, shape):
    """One-row decode steps with the GEMVs streamed through shared memory (one
    CTA per SM; rows per stage 8 / 4, x slices of 1..8 groups per lane, the
    down projection's 7) against the oracle, and against the register-fragment
    GEMV path on the same steps."""
    p = Pair(lib, shape, 37, n_ctx=256, n_ubatch=64)
    q = Pair(lib, shape, 37, n_ctx=256, n_ubatch=64)
    q.ctx.set_option("gemv_stream", 0)
    prompt = synth.prompt(shape.n_vocab, 37, 40)
    for x in (p, q):
        assert x.ctx.decode(prompt) == 0
    assert p.oc.decode(prompt) == 0
    for tok in (5, 17 % shape.n_vocab, 1000 % shape.n_vocab, 3):
        assert p.ctx.decode([tok]) == 0 and q.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        got, alt = p.logits(), q.logits()
        compare_logits(got, p.oc.logits)
        assert np.abs(got - alt).max() <= 2e-2
    p.free(); q.free()


def test_batch1_decode_and_generate(lib):
    """One-row decode steps along the oracle's greedy tokens, then on-device
    greedy generation continuing from there."""
    shape = MED128
    p = Pair(lib, shape, 31, n_ctx=256, n_ubatch=64)
    prompt = synth.prompt(shape.n_vocab, 31, 40)
    ref_tokens, ref_logits = O.generate_greedy(p.oc, prompt, 12)
    assert p.ctx.decode(prompt) == 0
    got = [p.logits()[-1]]
    for t in ref_tokens:
        assert p.ctx.decode([int(t)]) == 0
        got.append(p.logits()[-1])
    compare_logits(np.array(got), ref_logits)
    # greedy generation on the device continues from there
    ref2, _ = O.generate_greedy(O.Context(p.om, 256), prompt, 12 + 10)
    out = torch.zeros(10, dtype=torch.int32, device="cuda")
    assert p.ctx.generate(0, 10, out.data_ptr()) == 0
    p.ctx.synchronize()
    assert out.cpu().tolist() == list(ref2[12:22])
    p.free()


# ---------------------------------------------------------------- sliding window and context shift

@pytest.mark.parametrize("shape,W,attn,n", [(MED64, 37, 1, 150), (MED128, 70, 1, 150), (MED128, 70, 2, 150),
                                            (MED128, 130, 2, 400), (MED128, 130, 1, 400), (MED64, 1, 1, 150)])
def test_sliding_window_prefill_and_decode(lib, shape, W, attn, n):
    """Sliding-window attention (a query at p sees keys p - W < k <= p) in the
    tiled prefill (windows crossing tiles and ragged ubatches, and with a
    400-token prompt key tiles wholly below the window skipped; the tcgen05
    kernel one CTA a head and on CTA pairs) and in one-row decode steps,
    against the oracle with the same window."""
    p = Pair(lib, shape, 51, n_ctx=512, n_ubatch=64 if n < 300 else 200)
    p.ctx.set_option("attn_prefill", attn)
    p.ctx.set_option("swa_window", W)
    p.oc.cache.window = W
    prompt = synth.prompt(shape.n_vocab, 51, n)
    out = np.zeros(n, np.int8)
    out[[0, 36, 63, 64, 100, 149, n - 1]] = 1
    assert p.ctx.decode(prompt, output=out) == 0
    assert p.oc.decode(prompt, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    for tok in (3, 900 % shape.n_vocab, 42, 7):
        assert p.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        compare_logits(p.logits(), p.oc.logits)
    # a two-row step: the multi-row decode kernels with the window
    assert p.ctx.decode([11, 12], output=[1, 1]) == 0 and p.oc.decode([11, 12], output=[1, 1]) == 0
    compare_logits(p.logits(), p.oc.logits)
    p.free()


@pytest.mark.parametrize("shape", [MED64, STREAM_SHAPE])
def test_context_shift(lib, shape):
    """llm_seq_shift: drop a middle span of the cache (later keys re-rotated by
    -n on the GPU), keep decoding, drop the oldest span, decode again; logits
    against the oracle doing the same shifts."""
    p = Pair(lib, shape, 53, n_ctx=256, n_ubatch=64)
    prompt = synth.prompt(shape.n_vocab, 53, 120)
    assert p.ctx.decode(prompt) == 0 and p.oc.decode(prompt) == 0
    p.ctx.seq_shift(0, 10, 50)
    p.oc.seq_discard(0, 10, 50)
    assert p.ctx.seq_pos_max(0) == p.oc.seq_pos_max(0) == 69
    for tok in (5, 17, 301 % shape.n_vocab):
        assert p.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        compare_logits(p.logits(), p.oc.logits)
    p.ctx.seq_shift(0, 0, 30)
    p.oc.seq_discard(0, 0, 30)
    more = synth.prompt(shape.n_vocab, 54, 20)
    assert p.ctx.decode(more) == 0 and p.oc.decode(more) == 0      # a prefill ubatch after the shift
    compare_logits(p.logits(), p.oc.logits)
    assert p.ctx.decode([9]) == 0 and p.oc.decode([9]) == 0
    compare_logits(p.logits(), p.oc.logits)
    with pytest.raises(lib.LlmError):
        p.ctx.seq_shift(0, 60, 40)                                  # past the sequence's end
    p.free()


# ---------------------------------------------------------------- FP8 E4M3 KV cache

@pytest.mark.parametrize("shape,n_ubatch", [(MED64, 64), (MED128, 100), (STREAM_SHAPE, 64)])
def test_fp8_kv_cache(lib, shape, n_ubatch):
    """The E4M3 KV cache (option kv_fp8): every QKV epilogue rounds K/V to E4M3,
    the attention kernels widen the staged bytes per tile; prefill across
    ubatches, one- and two-row decode steps and a context shift against the
    oracle whose cache rounds to E4M3 the same way."""
    p = Pair(lib, shape, 57, n_ctx=256, n_ubatch=n_ubatch)
    p.ctx.set_option("kv_fp8", 1)
    p.oc.cache.store = "e4m3"
    n = 150
    prompt = synth.prompt(shape.n_vocab, 57, n)
    out = np.zeros(n, np.int8)
    out[[0, 63, 64, 99, 149]] = 1
    assert p.ctx.decode(prompt, output=out) == 0 and p.oc.decode(prompt, output=out) == 0
    compare_logits(p.logits(), p.oc.logits)
    for tok in (3, 42):
        assert p.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        compare_logits(p.logits(), p.oc.logits)
    assert p.ctx.decode([5, 6], output=[1, 1]) == 0 and p.oc.decode([5, 6], output=[1, 1]) == 0
    compare_logits(p.logits(), p.oc.logits)
    p.ctx.seq_shift(0, 20, 40)
    p.oc.seq_discard(0, 20, 40)
    assert p.ctx.decode([7]) == 0 and p.oc.decode([7]) == 0
    compare_logits(p.logits(), p.oc.logits)
    # the element type changes only while the cache is empty
    with pytest.raises(lib.LlmError):
        p.ctx.set_option("kv_fp8", 0)
    p.ctx.seq_clear(0)
    p.ctx.set_option("kv_fp8", 0)
    p.free()


# ---------------------------------------------------------------- Q8_0 weights

@pytest.mark.parametrize("shape", [MED64, MED128, STREAM_SHAPE])
def test_q8_0_weights(lib, shape):
    """A model re-encoded as Q8_0 (llm_model_quantize) against the oracle's Q8_0
    model: prefill over two ubatches (tcgen05 GEMMs on the f16(q d) copies),
    one-row steps streaming the Q8_0 rows, a two-row step (register-fragment
    GEMVs on the copies); and the one-row steps against the same weights read
    from the fp16 copies (option gemv_q8 = 0)."""
    p = Pair(lib, shape, 61, n_ctx=256, n_ubatch=64, q8=True)
    q = Pair(lib, shape, 61, n_ctx=256, n_ubatch=64, q8=True)
    q.ctx.set_option("gemv_q8", 0)
    prompt = synth.prompt(shape.n_vocab, 61, 100)
    for x in (p, q):
        assert x.ctx.decode(prompt) == 0
    assert p.oc.decode(prompt) == 0
    compare_logits(p.logits(), p.oc.logits)
    for tok in (5, 17 % shape.n_vocab, 999 % shape.n_vocab, 3):
        assert p.ctx.decode([tok]) == 0 and q.ctx.decode([tok]) == 0 and p.oc.decode([tok]) == 0
        got, alt = p.logits(), q.logits()
        compare_logits(got, p.oc.logits)
        assert np.abs(got - alt).max() <= 2e-2
    assert p.ctx.decode([5, 6], output=[1, 1]) == 0 and p.oc.decode([5, 6], output=[1, 1]) == 0
    compare_logits(p.logits(), p.oc.logits)
    # encoded once, and only while the model has no context
    with pytest.raises(lib.LlmError):
        p.model.quantize()
    p.free(); q.free()
    if shape is MED64:
        r = Pair(lib, shape, 61, n_ctx=16)
        with pytest.raises(lib.LlmError):
            r.model.quantize()
        r.free()


# ---------------------------------------------------------------- failure paths

def test_injected_allocation_failure(lib):
    """llm_kv_alloc with one of its device allocations failing (the first, a
    middle one, the last) returns LLM_ERR_ALLOC with no context and nothing
    held against the model; a context made afterwards decodes as the oracle."""
    import ctypes
    shape = MED64
    st = torch.cuda.current_stream().cuda_stream
    t = synth.make_weights(shape, 71, "cpu")
    dev = {k: v.cuda() for k, v in t.items()}
    model = lib.Model(shape, dev, stream=st)
    del dev
    # every allocation in turn, until an index past the last one lets the call succeed
    n_failed = 0
    for n in range(64):
        assert lib.llm_debug_fail_alloc(n) == 0
        out = ctypes.c_void_p()
        rc = lib.llm_kv_alloc(model.handle, 64, 1, 16, ctypes.c_void_p(st), ctypes.byref(out))
        if rc == lib.LLM_OK:
            lib.llm_kv_free(out)
            break
        assert rc == lib.LLM_ERR_ALLOC and out.value is None, (n, rc)
        n_failed += 1
    assert n_failed >= 10, n_failed          # the cache, tables and every workspace
    # disarmed after one call: this one succeeds
    ctx = lib.Context(model, 64, 1, 16, stream=st)
    om = O.Model(O.Hparams.of(shape), synth.host_weights(t))
    oc = O.Context(om, 64, 1, 16)
    prompt = synth.prompt(shape.n_vocab, 71, 20)
    assert ctx.decode(prompt) == 0 and oc.decode(prompt) == 0
    ctx.synchronize()
    compare_logits(lib.logits_numpy(ctx, shape.n_vocab), oc.logits)
    ctx.free()
    # no failed call left a context counted against the model: quantising needs none
    model.quantize(stream=st)
    model.free()
