"""Pins of the CPU oracle against closed forms, invariants and brute force.

The pages print no worked numeric example, so each oracle function is pinned
by what the mathematics fixes: hand-computed values (RoPE angles, a two-key
softmax, SiLU at ln 3), invariants (unit RMS, norm preservation, relative
position, rows summing to one, causality, cache == recompute, pruning, ubatch
size independence, sequence isolation) and a pure-Python brute force of the
whole composition on tiny models.
"""
import math

import numpy as np
import pytest
import torch

import synth
import oracle
from oracle import llama as O
from brute_llama import BruteLlama

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------- widening

def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x4049], np.uint16)
    f = O.bf16_to_float(bits)
    assert f[0] == 1.0 and f[1] == -2.0
    assert f[2] == 2.0 ** -133          # smallest bf16 subnormal
    assert np.isinf(f[3])
    assert f[4] == 3.140625             # 0x4049 = 1.5703125 * 2


def test_bf16_widening_matches_torch():
    x = torch.randn(1000).to(torch.bfloat16)
    assert np.array_equal(O.bf16_to_float(synth.bf16_bits(x), np.float32), x.float().numpy())


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_rms_before_gain():
    x = RNG.normal(size=(7, 96)) * 3.0
    y = O.rms_norm(x, np.ones(96), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-12)
    g = 1 + 0.1 * RNG.normal(size=96)
    y2 = O.rms_norm(x, g, 0.0)
    assert np.allclose(np.sqrt(np.mean((y2 / g) ** 2, axis=1)), 1.0, atol=1e-12)


def test_rmsnorm_eps_inside_sqrt_closed_form():
    # constant row c: mean of squares is c^2, so the output is c / sqrt(c^2 + eps) * g
    c, eps = 0.01, 1e-5
    g = np.array([1.0, 2.0, -0.5, 3.0])
    y = O.rms_norm(np.full((1, 4), c), g, eps)
    assert np.allclose(y[0], c / math.sqrt(c * c + eps) * g, rtol=1e-14)
    # eps added outside the root would give c / (|c| + eps): different by ~5%
    assert not np.allclose(y[0], c / (abs(c) + eps) * g, rtol=1e-3)


# ----------------------------------------------------------------- RoPE

def test_rope_hand_values():
    # head_dim 2: one pair with frequency theta^0 = 1, so the angle is pos radians
    x = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    y = O.rope(x, np.array([1, 1]), 10000.0)
    assert np.allclose(y[0, 0], [math.cos(1), math.sin(1)])
    assert np.allclose(y[1, 0], [-math.sin(1), math.cos(1)])
    # head_dim 4, theta 10000: pair 1 has frequency 10000^(-2/4) = 1/100,
    # so at position 100 it turns by exactly 1 radian; pair 0 turns by 100 rad
    x = np.array([[[0.0, 0.0, 1.0, 0.0]], [[1.0, 0.0, 0.0, 0.0]]])
    y = O.rope(x, np.array([100, 100]), 10000.0)
    assert np.allclose(y[0, 0], [0, 0, math.cos(1), math.sin(1)])
    assert np.allclose(y[1, 0], [math.cos(100), math.sin(100), 0, 0])


def test_rope_pos0_identity_and_norm():
    x = RNG.normal(size=(5, 3, 64))
    assert np.allclose(O.rope(x, np.zeros(5, int), 500000.0), x, atol=0)
    y = O.rope(x, np.array([1, 7, 100, 4095, 32767]), 500000.0)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


@pytest.mark.parametrize("theta", [10000.0, 500000.0])
def test_rope_relative_position(theta):
    q = RNG.normal(size=(1, 1, 128))
    k = RNG.normal(size=(1, 1, 128))
    def dot(m, n):
        return float(np.sum(O.rope(q, np.array([m]), theta) * O.rope(k, np.array([n]), theta)))
    base = dot(10, 3)
    for shift in (1, 17, 1000, 30000):
        assert abs(dot(10 + shift, 3 + shift) - base) < 1e-9 * max(1.0, abs(base))
    assert abs(dot(11, 3) - base) > 1e-6          # and it does depend on the difference


# ----------------------------------------------------------------- attention

def test_attention_two_keys_closed_form():
    # hd 4 => scale 1/2.  q.k1 = 2 -> score 1, q.k2 = 0 -> score 0.
    q = np.array([[[2.0, 0, 0, 0]]])
    k = np.array([[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]])
    v = np.array([[[1.0, 2, 3, 4]], [[-1.0, 0, 5, 0]]])
    o = O.attention_one_seq(q, k, v, np.array([5]), np.array([0, 1]), 1)
    p1 = math.e / (math.e + 1.0)
    assert np.allclose(o[0, 0], p1 * v[0, 0] + (1 - p1) * v[1, 0], rtol=1e-14)


def test_attention_rows_sum_to_one_and_causal():
    tq, s, H, Hkv, hd = 6, 9, 4, 2, 8
    q = RNG.normal(size=(tq, H, hd))
    k = RNG.normal(size=(s, Hkv, hd))
    v = RNG.normal(size=(s, Hkv, hd))
    qpos = np.arange(3, 9)
    kpos = np.arange(9)
    o, p = O.attention_one_seq(q, k, v, qpos, kpos, Hkv, return_probs=True)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)
    future = kpos[None, :] > qpos[:, None]
    assert np.all(p[:, future] == 0.0)
    assert np.all(p[:, ~future] > 0.0)


def test_attention_single_visible_key_returns_v():
    q = RNG.normal(size=(1, 4, 8))
    k = RNG.normal(size=(3, 2, 8))
    v = RNG.normal(size=(3, 2, 8))
    o = O.attention_one_seq(q, k, v, np.array([0]), np.array([0, 1, 2]), 2)
    for h in range(4):
        assert np.allclose(o[0, h], v[0, h // 2], atol=1e-15)


def test_attention_zero_query_is_mean_of_visible_values():
    q = np.zeros((2, 2, 4))
    k = RNG.normal(size=(5, 1, 4))
    v = RNG.normal(size=(5, 1, 4))
    o = O.attention_one_seq(q, k, v, np.array([2, 4]), np.arange(5), 1)
    assert np.allclose(o[0, 0], v[:3, 0].mean(0)) and np.allclose(o[1, 1], v[:5, 0].mean(0))


def test_gqa_equals_mha_with_repeated_heads():
    tq, s, H, Hkv, hd = 4, 7, 8, 2, 16
    q = RNG.normal(size=(tq, H, hd))
    k = RNG.normal(size=(s, Hkv, hd))
    v = RNG.normal(size=(s, Hkv, hd))
    qpos, kpos = np.arange(3, 7), np.arange(7)
    gqa = O.attention_one_seq(q, k, v, qpos, kpos, Hkv)
    rep = H // Hkv
    mha = O.attention_one_seq(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), qpos, kpos, H)
    assert np.allclose(gqa, mha, atol=1e-14)


def test_attention_brute_force_loops():
    tq, s, H, Hkv, hd = 3, 5, 4, 2, 4
    q = RNG.normal(size=(tq, H, hd))
    k = RNG.normal(size=(s, Hkv, hd))
    v = RNG.normal(size=(s, Hkv, hd))
    qpos, kpos = np.array([2, 3, 4]), np.arange(5)
    o = O.attention_one_seq(q, k, v, qpos, kpos, Hkv)
    for t in range(tq):
        for h in range(H):
            j = h // 2
            sc = [sum(q[t, h, d] * k[c, j, d] for d in range(hd)) / 2.0 for c in range(s) if kpos[c] <= qpos[t]]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            ref = [sum(e[c] / sum(e) * v[c, j, d] for c in range(len(e))) for d in range(hd)]
            assert np.allclose(o[t, h], ref, atol=1e-13)


# ----------------------------------------------------------------- MLP

def test_silu_closed_form():
    # sigmoid(ln 3) = 3/4
    assert abs(O.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(-40.0)) < 1e-15


def test_swiglu_brute_force():
    d, f = 5, 7
    x = RNG.normal(size=(2, d))
    wg, wu, wd = RNG.normal(size=(f, d)), RNG.normal(size=(f, d)), RNG.normal(size=(d, f))
    y = O.swiglu_mlp(x, wg, wu, wd)
    for t in range(2):
        g = [sum(wg[i, c] * x[t, c] for c in range(d)) for i in range(f)]
        u = [sum(wu[i, c] * x[t, c] for c in range(d)) for i in range(f)]
        a = [g[i] / (1 + math.exp(-g[i])) * u[i] for i in range(f)]
        ref = [sum(wd[o, i] * a[i] for i in range(f)) for o in range(d)]
        assert np.allclose(y[t], ref, atol=1e-13)


# ----------------------------------------------------------------- whole model

MICRO = synth.Shape(n_vocab=11, n_embd=6, n_layer=2, n_head=4, n_head_kv=2, head_dim=4, n_ff=5,
                    rms_eps=1e-5, rope_theta=10000.0, tied_output=False)


def micro_weights(shape, seed, scale=0.5):
    """Larger-than-recipe weights so every term matters at this tiny size."""
    g = np.random.default_rng(seed)
    w = {}
    for n in synth.tensor_names(shape):
        dims = synth.tensor_shape(shape, n)
        w[n] = (1.0 + 0.2 * g.normal(size=dims)) if n.endswith("norm") else scale * g.normal(size=dims)
    return w


def as_lists(w):
    return {k: v.tolist() for k, v in w.items()}


@pytest.mark.parametrize("tied", [False, True])
def test_model_matches_brute_force_two_sequences(tied):
    shape = synth.scaled_shape(MICRO, tied_output=tied)
    w = micro_weights(shape, 7)
    hp = O.Hparams.of(shape)
    ctx = O.Context(O.Model(hp, w), n_ctx=16, n_seq_max=2, n_ubatch=3)
    brute = BruteLlama(hp, as_lists(w))
    # batch 1: two interleaved sequences, outputs on rows 2, 4 and 5
    tokens, seq = [3, 7, 1, 10, 0, 5], [0, 1, 0, 1, 1, 0]
    outputs = [0, 0, 1, 0, 1, 1]
    assert ctx.decode(tokens, seq=seq, output=outputs) == O.OK
    pos = [0, 0, 1, 1, 2, 2]
    ref = brute.batch(tokens, pos, seq, outputs)
    assert np.allclose(ctx.logits, np.array(ref), atol=1e-12)
    # batch 2: one decode token per sequence, continuing the caches
    assert ctx.decode([4, 9], seq=[1, 0], output=[1, 1]) == O.OK
    ref = brute.batch([4, 9], [3, 3], [1, 0], [1, 1])
    assert np.allclose(ctx.logits, np.array(ref), atol=1e-12)


def test_hidden_states_match_brute_force_layer_by_layer():
    shape = MICRO
    w = micro_weights(shape, 9)
    hp = O.Hparams.of(shape)
    ctx = O.Context(O.Model(hp, w), n_ctx=8)
    assert ctx.decode([1, 2, 3], output=[1, 1, 1], keep_hidden=True) == O.OK
    # one layer model built from the first layer: its output must equal hidden[0]
    one = synth.scaled_shape(shape, n_layer=1)
    w1 = {k: v for k, v in w.items() if not k.startswith("blk.1.")}
    b = BruteLlama(O.Hparams.of(one), as_lists(w1))
    lg = b.batch([1, 2, 3], [0, 1, 2], [0, 0, 0], [1, 1, 1])
    ctx1 = O.Context(O.Model(O.Hparams.of(one), w1), n_ctx=8)
    assert ctx1.decode([1, 2, 3], output=[1, 1, 1], keep_hidden=True) == O.OK
    assert np.allclose(ctx1.hidden[0][0], ctx.hidden[0][0], atol=0)
    assert np.allclose(ctx1.logits, lg, atol=1e-12)


def tiny_model(dtype=np.float64, shape=synth.TINY, seed=0):
    w = synth.host_weights(synth.make_weights(shape, seed, "cpu"))
    return O.Model(O.Hparams.of(shape), w, dtype)


@pytest.fixture(scope="module")
def tiny():
    return tiny_model()


def test_cache_decode_equals_full_recompute(tiny):
    toks = synth.prompt(512, 0, 12)
    step = O.Context(tiny, n_ctx=32)
    assert step.decode(toks[:8]) == O.OK
    for t in toks[8:]:
        assert step.decode([t]) == O.OK
    full = O.Context(tiny, n_ctx=32)
    assert full.decode(toks) == O.OK
    assert np.allclose(step.logits[-1], full.logits[-1], atol=1e-10)


def test_pruning_equals_all_rows_then_select(tiny):
    toks = synth.prompt(512, 0, 10)
    out = np.array([0, 1, 0, 0, 1, 0, 0, 0, 1, 1], np.int8)
    pos, seq = np.arange(10), np.zeros(10, int)
    a = O.forward_ubatch(tiny, O.KVCache(tiny.hp, 16, 1, np.float64), toks, pos, seq, out, prune=True)
    b = O.forward_ubatch(tiny, O.KVCache(tiny.hp, 16, 1, np.float64), toks, pos, seq, out, prune=False)
    assert a.shape == (4, 512)
    assert np.allclose(a, b, atol=1e-12)


def test_layer_rows_equals_layer_forward(tiny):
    """layer_rows (selected rows only, attention of the others skipped) gives
    exactly layer_forward's hidden state for those rows, in a prefill ubatch
    and for a later decode row that sees the whole cache."""
    toks = synth.prompt(512, 3, 21)
    ctx = O.Context(tiny, n_ctx=32)
    assert ctx.decode(toks[:20], keep_hidden=True) == O.OK
    full = ctx.hidden[0][0]                                  # layer 0, all 20 rows
    lw = tiny.layer(0)
    rows = [0, 7, 19]
    got = O.layer_rows(tiny.hp, lw, tiny.embed_rows(toks[:20]), np.arange(20), rows)
    assert np.allclose(got, full[rows], atol=1e-12)
    assert ctx.decode(toks[20:], keep_hidden=True) == O.OK     # decode row at position 20
    got = O.layer_rows(tiny.hp, lw, tiny.embed_rows(toks), np.arange(21), [20])
    assert np.allclose(got, ctx.hidden[0][0], atol=1e-12)
    # causal: row 7 does not see the rows after it (a mask slip would fail this)
    a = O.layer_rows(tiny.hp, lw, tiny.embed_rows(toks), np.arange(21), [7])
    b = O.layer_rows(tiny.hp, lw, tiny.embed_rows(toks[:8]), np.arange(8), [7])
    assert np.allclose(a, b, atol=1e-12, rtol=0)


def test_logits_independent_of_ubatch_size(tiny):
    toks = synth.prompt(512, 0, 16)
    out = np.zeros(16, np.int8)
    out[[3, 9, 15]] = 1
    res = []
    for nub in (1, 3, 16):
        ctx = O.Context(tiny, n_ctx=32, n_ubatch=nub)
        assert ctx.decode(toks, output=out) == O.OK
        res.append(ctx.logits)
    assert np.allclose(res[0], res[2], atol=1e-10) and np.allclose(res[1], res[2], atol=1e-10)


def test_sequence_isolation(tiny):
    a, b = synth.prompt(512, 0, 6), synth.prompt(512, 1, 4)
    mixed = O.Context(tiny, n_ctx=16, n_seq_max=2)
    tokens = np.concatenate([a, b])
    seq = np.array([0] * 6 + [1] * 4)
    out = np.zeros(10, np.int8)
    out[[5, 9]] = 1
    assert mixed.decode(tokens, seq=seq, output=out) == O.OK
    alone_a = O.Context(tiny, n_ctx=16)
    alone_a.decode(a)
    alone_b = O.Context(tiny, n_ctx=16)
    alone_b.decode(b)
    assert np.allclose(mixed.logits[0], alone_a.logits[-1], atol=1e-12)
    assert np.allclose(mixed.logits[1], alone_b.logits[-1], atol=1e-12)


def test_fp32_oracle_agrees_with_fp64():
    m64, m32 = tiny_model(np.float64), tiny_model(np.float32)
    toks = synth.prompt(512, 0, 16)
    c64, c32 = O.Context(m64, n_ctx=40), O.Context(m32, n_ctx=40)
    t64, l64 = O.generate_greedy(c64, toks, 16)
    t32, l32 = O.generate_greedy(c32, toks, 16, forced=t64)
    assert np.max(np.abs(l64 - l32)) < 1e-4


def test_tiny_logits_unit_order(tiny):
    ctx = O.Context(tiny, n_ctx=40)
    assert ctx.decode(synth.prompt(512, 0, 16)) == O.OK
    s = float(np.std(ctx.logits))
    assert 0.2 < s < 5.0


# ----------------------------------------------------------------- batch rules

def test_batch_rules(tiny):
    ctx = O.Context(tiny, n_ctx=8, n_seq_max=2)
    assert ctx.decode([]) == O.INVALID
    assert ctx.decode([512]) == O.INVALID                       # token out of range
    assert ctx.decode([-1]) == O.INVALID
    assert ctx.decode([1], seq=[2]) == O.INVALID                # seq out of range
    assert ctx.decode([1, 2], pos=[0, 2]) == O.INVALID          # gap
    assert ctx.decode([1], pos=[1]) == O.INVALID                # must continue at 0
    assert ctx.seq_pos_max(0) == -1
    assert ctx.decode([1, 2, 3]) == O.OK                        # default pos 0,1,2; last row out
    assert ctx.seq_pos_max(0) == 2 and ctx.logits.shape == (1, 512)
    assert ctx.logits_ith(2) is not None and ctx.logits_ith(1) is None
    assert ctx.decode([4], seq=[1]) == O.OK and ctx.seq_pos_max(1) == 0
    assert ctx.decode([1] * 6) == O.NO_KV_ROOM                  # pos 3..8, and 8 >= n_ctx
    assert ctx.seq_pos_max(0) == 2                              # nothing written
    assert ctx.decode([1] * 6, output=[1] * 6) == O.NO_KV_ROOM
    assert ctx.decode([1] * 4, output=[1, 0, 1, 0]) == O.OK     # pos 3..6
    assert ctx.logits.shape == (2, 512) and ctx.out_index == {0: 0, 2: 1}
    ctx.seq_clear(0)
    assert ctx.seq_pos_max(0) == -1


def test_greedy_ties_take_lowest_id():
    assert list(O.greedy_argmax(np.array([[0.0, 3.0, 1.0, 3.0], [5.0, 5.0, 5.0, 5.0]]))) == [1, 0]


def test_synth_is_deterministic():
    a = synth.make_tensor(synth.TINY, 0, "blk.1.ffn_up")
    b = synth.make_tensor(synth.TINY, 0, "blk.1.ffn_up")
    c = synth.make_tensor(synth.TINY, 1, "blk.1.ffn_up")
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert abs(float(a.float().std()) - 0.02) < 0.002
    gain = synth.make_tensor(synth.TINY, 0, "output_norm").float()
    assert abs(float(gain.mean()) - 1.0) < 0.01
    lens = synth.multislot_lengths()
    assert lens.shape == (8,) and lens.min() >= 256 and lens.max() <= 4096


# ----------------------------------------------------------------- sliding window and context shift

def test_window_brute_force_loops():
    # a key is visible iff 0 <= q_pos - k_pos < W: restate with explicit loops
    tq, s, H, Hkv, hd, W = 4, 9, 2, 1, 4, 3
    q = RNG.normal(size=(tq, H, hd))
    k = RNG.normal(size=(s, Hkv, hd))
    v = RNG.normal(size=(s, Hkv, hd))
    qpos, kpos = np.array([0, 2, 5, 8]), np.arange(9)
    o = O.attention_one_seq(q, k, v, qpos, kpos, Hkv, window=W)
    for t in range(tq):
        for h in range(H):
            keys = [c for c in range(s) if qpos[t] - W < kpos[c] <= qpos[t]]
            assert len(keys) == min(W, qpos[t] + 1)
            sc = [sum(q[t, h, d] * k[c, 0, d] for d in range(hd)) / 2.0 for c in keys]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            ref = [sum(e[i] / sum(e) * v[c, 0, d] for i, c in enumerate(keys)) for d in range(hd)]
            assert np.allclose(o[t, h], ref, atol=1e-13)


def test_window_limits():
    tq, s, H, hd = 3, 6, 2, 4
    q = RNG.normal(size=(tq, H, hd))
    k = RNG.normal(size=(s, H, hd))
    v = RNG.normal(size=(s, H, hd))
    qpos, kpos = np.array([1, 3, 5]), np.arange(6)
    # a window at least as long as the sequence is the full causal mask
    assert np.array_equal(O.attention_one_seq(q, k, v, qpos, kpos, H, window=6),
                          O.attention_one_seq(q, k, v, qpos, kpos, H))
    # a window of one: each query sees only its own position's value
    o1 = O.attention_one_seq(q, k, v, qpos, kpos, H, window=1)
    assert np.allclose(o1, v[qpos], atol=1e-15)


def test_window_model_sees_only_recent_tokens(tiny):
    # with window W, the last token's logits do not depend on tokens older than
    # W positions in layer 0's attention... over L layers information travels
    # L * (W - 1) positions, so tokens further back than that cannot matter
    W, L = 3, tiny.hp.n_layer
    toks = np.array(synth.prompt(512, 5, 16))
    a = O.Context(tiny, n_ctx=32, window=W)
    assert a.decode(toks) == O.OK
    far = L * (W - 1)
    other = toks.copy()
    other[: len(toks) - 1 - far] = (other[: len(toks) - 1 - far] + 7) % 512
    b = O.Context(tiny, n_ctx=32, window=W)
    assert b.decode(other) == O.OK
    assert np.allclose(a.logits[-1], b.logits[-1], atol=1e-12)
    # but the window does change the result against full attention
    c = O.Context(tiny, n_ctx=32)
    assert c.decode(toks) == O.OK
    assert not np.allclose(a.logits[-1], c.logits[-1], atol=1e-6)


@pytest.mark.parametrize("p0,n", [(4, 6), (0, 3), (9, 1)])
def test_discard_layer0_equals_prefill_of_the_kept_tokens(tiny, p0, n):
    # layer 0's K and V depend only on a token and its position, so after
    # dropping positions [p0, p0 + n) (later keys re-rotated by -n) layer 0 of
    # the cache equals a fresh prefill of the kept tokens at their new
    # positions; deeper layers keep what the dropped tokens contributed
    toks = synth.prompt(512, 6, 14)
    a = O.Context(tiny, n_ctx=32)
    assert a.decode(toks) == O.OK
    a.seq_discard(0, p0, n)
    assert a.seq_pos_max(0) == len(toks) - n - 1
    kept = list(toks[:p0]) + list(toks[p0 + n:])
    b = O.Context(tiny, n_ctx=32)
    assert b.decode(kept) == O.OK
    m = len(kept)
    assert np.allclose(a.cache.k[0, 0, :m], b.cache.k[0, 0, :m], atol=1e-12)
    assert np.array_equal(a.cache.v[0, 0, :m], b.cache.v[0, 0, :m])
    assert not a.cache.filled[0, m:].any()


@pytest.mark.parametrize("p0,n", [(4, 6), (0, 3)])
def test_discard_one_layer_model_equals_prefill_of_the_kept_tokens(p0, n):
    # with one layer the whole cache is layer 0, so the next token's logits
    # after the shift equal those after a fresh prefill of the kept tokens
    one = tiny_model(shape=synth.scaled_shape(synth.TINY, n_layer=1))
    toks = synth.prompt(512, 6, 14)
    a = O.Context(one, n_ctx=32)
    assert a.decode(toks) == O.OK
    a.seq_discard(0, p0, n)
    assert a.decode([77]) == O.OK
    kept = list(toks[:p0]) + list(toks[p0 + n:])
    b = O.Context(one, n_ctx=32)
    assert b.decode(kept + [77]) == O.OK
    assert np.allclose(a.logits[-1], b.logits[-1], atol=1e-10)


def test_discard_rejects_ranges_outside_the_sequence(tiny):
    a = O.Context(tiny, n_ctx=32)
    assert a.decode(synth.prompt(512, 6, 8)) == O.OK
    for p0, n in ((-1, 2), (6, 3), (0, 0)):
        with pytest.raises(ValueError):
            a.seq_discard(0, p0, n)


# ----------------------------------------------------------------- FP8 E4M3 KV cache elements

def test_e4m3_hand_values():
    x = np.array([0.0, 1.0, 0.3, -2.5, 0.06640625, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, 464.0,
                  1000.0, -1e9, 17.0, 19.0])
    want = np.array([0.0, 1.0, 0.3125, -2.5, 0.0625, 2.0 ** -9, 0.0, 2.0 ** -8, 448.0, 448.0,
                     448.0, -448.0, 16.0, 20.0])
    # 0.3 = 1.2 * 2^-2 -> 1.25 * 2^-2; 0.06640625 = 1.0625 * 2^-4 is a tie -> even 1.0;
    # 2^-10 is half the smallest subnormal -> 0 (even); 3 * 2^-10 -> 2^-8 (tie to even);
    # 464 saturates; 17 = 1.0625 * 16 -> 16 (tie to even), 19 = 1.1875 * 16 -> 1.25 * 16
    assert np.array_equal(O.round_to_e4m3(x), want)


def test_e4m3_matches_torch_in_range():
    x = torch.cat([torch.randn(20000) * 3, torch.randn(2000) * 1e-3, torch.linspace(-440, 440, 1001)])
    ref = x.to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.round_to_e4m3(x.double().numpy()), ref)


def test_e4m3_cache_holds_e4m3_values(tiny):
    # a context storing its cache as E4M3 keeps only E4M3 values, also after a
    # context shift re-rotates the keys, and still matches full recompute
    toks = synth.prompt(512, 8, 12)
    a = O.Context(tiny, n_ctx=32, kv_store="e4m3")
    assert a.decode(toks[:9]) == O.OK
    for t in toks[9:]:
        assert a.decode([t]) == O.OK
    filled = a.cache.filled[0]
    k, v = a.cache.k[0][:, filled], a.cache.v[0][:, filled]
    assert np.array_equal(O.round_to_e4m3(k), k) and np.array_equal(O.round_to_e4m3(v), v)
    b = O.Context(tiny, n_ctx=32, kv_store="e4m3")
    assert b.decode(toks) == O.OK
    assert np.allclose(a.logits[-1], b.logits[-1], atol=1e-10)
    a.seq_discard(0, 2, 4)
    filled = a.cache.filled[0]
    k = a.cache.k[0][:, filled]
    assert np.array_equal(O.round_to_e4m3(k), k)


# ----------------------------------------------------------------- Q8_0 weight blocks

def test_q8_0_hand_values():
    # max|w| = 127 * 2^-7, so d = 2^-7 exactly (an fp16 value too) and w / d is
    # the multiple of 2^-7 written below: halves go to the even neighbour
    u = 2.0 ** -7
    w = np.zeros((1, 32))
    w[0, :8] = np.array([127, 2.5, 3.5, -1.5, 0.4, -127, 0.5, -0.5]) * u
    q, d = O.quantize_q8_0(w)
    assert q.dtype == np.int8 and d.dtype == np.float16 and d.shape == (1, 1)
    assert d[0, 0] == np.float16(u)
    assert q[0, :8].tolist() == [127, 2, 4, -2, 0, -127, 0, 0]
    assert not q[0, 8:].any()
    assert np.array_equal(O.dequantize_q8_0(q, d), q.astype(np.float64) * u)
    # the dequantised block holds exact multiples of d with max|q| = 127: it encodes to itself
    q2, d2 = O.quantize_q8_0(O.dequantize_q8_0(q, d))
    assert np.array_equal(q2, q) and np.array_equal(d2, d)


def test_q8_0_scale_is_rounded_to_fp16():
    # max|w| = 1: d = fl32(1/127) = 0.0078740157..., stored as the fp16 value
    # 1032 * 2^-17 = 0.00787353515625 (the fp16 step at 2^-7 is 2^-17;
    # 1/127 / 2^-17 = 1032.06); the largest element dequantises to 127 times that
    w = np.zeros((1, 32))
    w[0, 3] = 1.0
    w[0, 5] = -0.25                       # 0.25 * 127 = 31.75 -> -32
    q, d = O.quantize_q8_0(w)
    assert float(d[0, 0]) == 1032 * 2.0 ** -17
    assert q[0, 3] == 127 and q[0, 5] == -32
    deq = O.dequantize_q8_0(q, d)
    assert deq[0, 3] == 127 * 1032 * 2.0 ** -17 == 0.99993896484375


def test_q8_0_blocks_are_independent_and_partial_last_block():
    # K = 40: a block of 32 and a last block of 8, each with its own scale
    w = np.zeros((2, 40))
    w[0, 31] = 2.0 * 127 * 2.0 ** -8      # block 0: d = 2^-7
    w[0, 32:] = np.arange(1, 9) * 2.0 ** -6  # block 1: max 8 * 2^-6 = 2^-3 -> d = 2^-3 / 127
    q, d = O.quantize_q8_0(w)
    assert d.shape == (2, 2) and q.shape == (2, 40)
    assert d[0, 0] == np.float16(2.0 ** -7) and q[0, 31] == 127 and not q[0, :31].any()
    assert q[0, 39] == 127 and np.all(np.diff(q[0, 32:].astype(int)) > 0)
    # an all-zero row: scale 0, codes 0, weights 0
    assert not d[1].any() and not q[1].any() and not O.dequantize_q8_0(q, d)[1].any()


def test_q8_0_error_bound_and_range():
    # |w - q d16| <= d/2 + 127 |d - d16| <= max|w| (1/254 + 2^-11): the nearest
    # integer is off by at most a half step, and the fp16 scale by 2^-11 relative
    rng = np.random.default_rng(7)
    w = rng.normal(0, 0.02, size=(64, 256)) * rng.uniform(0.01, 10, size=(64, 1))
    w = O.bf16_to_float(synth.bf16_bits(torch.from_numpy(w).float().to(torch.bfloat16)))
    q, d = O.quantize_q8_0(w)
    deq = O.dequantize_q8_0(q, d)
    amax = np.abs(w.reshape(64, 8, 32)).max(axis=2)
    bound = np.repeat(amax * (1 / 254 + 2.0 ** -11) * (1 + 1e-6), 32, axis=1)
    assert np.all(np.abs(w - deq) <= bound)
    assert np.abs(q.astype(int)).max() == 127
    # each block's largest element takes the code +-127
    qb = np.abs(q.astype(int)).reshape(64, 8, 32).max(axis=2)
    assert np.all(qb == 127)


def test_q8_0_sign_and_power_of_two_scaling():
    rng = np.random.default_rng(8)
    w = rng.normal(0, 1, size=(8, 96)).astype(np.float32)
    q, d = O.quantize_q8_0(w)
    qn, dn = O.quantize_q8_0(-w)
    assert np.array_equal(qn, -q) and np.array_equal(dn, d)
    q4, d4 = O.quantize_q8_0(w * 4)
    assert np.array_equal(q4, q) and np.array_equal(d4.astype(np.float64), 4 * d.astype(np.float64))


@pytest.mark.parametrize("tied", [False, True])
def test_q8_0_model_quantises_the_projections_only(tied):
    tiny = tiny_model(shape=synth.scaled_shape(synth.TINY, tied_output=tied))
    qm = tiny.quantized_q8_0()
    hp = tiny.hp
    assert hp.tied_output == tied
    for i in range(hp.n_layer):
        for t in O.Model.MATRICES:
            name = f"blk.{i}.{t}"
            a, b = tiny.get(name), qm.get(name)
            assert not np.array_equal(a, b)
            q, d = O.quantize_q8_0(b)       # a dequantised matrix is already on its grid
            assert np.max(np.abs(O.dequantize_q8_0(q, d) - b)) <= np.max(np.abs(b)) * 2.0 ** -10
        for t in ("attn_norm", "ffn_norm"):
            assert np.array_equal(tiny.get(f"blk.{i}.{t}"), qm.get(f"blk.{i}.{t}"))
    assert np.array_equal(tiny.get("output_norm"), qm.get("output_norm"))
    out_changed = not np.array_equal(tiny.get("output"), qm.get("output"))
    emb_changed = not np.array_equal(tiny.embed_rows(np.arange(8)), qm.embed_rows(np.arange(8)))
    assert out_changed and emb_changed == bool(hp.tied_output)


def test_q8_0_model_stays_close_to_the_original(tiny):
    # the encoding perturbs each weight by < 0.5 % of its block's largest; the
    # last-position logits move by a small fraction of their spread
    toks = synth.prompt(512, 10, 9)
    a = O.Context(tiny, n_ctx=32)
    b = O.Context(tiny.quantized_q8_0(), n_ctx=32)
    assert a.decode(toks) == O.OK and b.decode(toks) == O.OK
    la, lb = a.logits[-1], b.logits[-1]
    assert np.max(np.abs(la - lb)) < 0.05 * (la.max() - la.min())
    assert np.max(np.abs(la - lb)) > 0


def test_q8_0_scales_round_like_torch_half():
    # the stored scale is float32 max|w| / 127 rounded to fp16: compared with
    # torch's own float32 -> float16 conversion, over scales from the fp16
    # subnormal range to its largest normals
    rng = np.random.default_rng(9)
    mags = np.exp2(rng.uniform(-26, 15, size=(512, 1))).astype(np.float32)
    w = (rng.uniform(-1, 1, size=(512, 64)) * mags).astype(np.float32)
    _, d = O.quantize_q8_0(w)
    amax = np.abs(w.reshape(512, 2, 32)).max(axis=2)
    want = torch.from_numpy(amax / np.float32(127)).half().numpy()
    assert np.array_equal(d.view(np.uint16), want.view(np.uint16))
