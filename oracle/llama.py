"""Plain numpy oracle of the Llama decoder forward pass (test infrastructure).

Sources, cited by page title and section:

* [EN] "Inside the inference engine: model architectures and forward pass"
  (Ollama Go engine): section "Detailed explanation: Llama's forward pass in
  Go" (the per-layer sequence diagram and ``Model.Forward``), "KV Cache: memory
  for causal attention", "Token sampling pipeline", "Initialising the model
  with reflection" (``output,alt:token_embd`` tying).
* [LC] "LLama.cpp — how it works": "Step 10: the batch for one call"
  (``llama_batch``, ``llama_batch_allocr::init``), "Step 11: tokens become
  embeddings", "Steps 11–12: running the batch through the model"
  (``llama_decode``, ``init_batch`` ubatch split, return codes), "Steps 14–15:
  logits and sampling" (``llama_get_logits_ith``), "KV-cache and the Prefill /
  Decode stages".

Where the pages leave a step open, the reading taken is stated at the
function.  Arithmetic runs in ``dtype`` (float64 unless a caller asks for
float32); bf16 weights are widened exactly.  No blocking, fusion or reordering
beyond the definitions below.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

OK, NO_KV_ROOM, INVALID = 0, 1, -1


@dataclass(frozen=True)
class Hparams:
    """[LC] hparams read by the Llama graph, plus [EN] output tying."""
    n_vocab: int
    n_embd: int
    n_layer: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    rms_eps: float
    rope_theta: float
    tied_output: bool

    @staticmethod
    def of(shape) -> "Hparams":
        return Hparams(**{k: getattr(shape, k) for k in Hparams.__dataclass_fields__})


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned widened in the
    input's float type: the fp32 bits are rounded at bit 16."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.asarray(x).dtype)


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (1 sign, 4 exponent bits with bias
    7, 3 mantissa bits; ties to even), saturating at +-448, its largest finite
    value, and returned widened in the input's float type.  This is the
    quantised KV cache's element (the pages name more aggressive KV-cache
    quantisation without fixing a format; reading: E4M3 without a scale).
    The quantum of a value with exponent e is 2^(e - 3), with e no lower than
    -6, the smallest normal exponent (below it the values are subnormal, in
    steps of 2^-9)."""
    x = np.asarray(x)
    a = np.abs(x.astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = np.exp2(e - 3.0)
    r = np.round(a / q) * q                    # numpy rounds halves to even
    r = np.minimum(r, 448.0)
    return (np.sign(x) * r).astype(x.dtype)


def round_to(x: np.ndarray, store) -> np.ndarray:
    """Storage rounding of cached K/V: None keeps the values, "bf16" / "fp16"
    round to that type (nearest, ties to even), "e4m3" to FP8 E4M3
    (round_to_e4m3)."""
    if store is None:
        return x
    if store == "bf16":
        return round_to_bf16(x)
    if store == "fp16":
        return np.asarray(x).astype(np.float16).astype(np.asarray(x).dtype)
    if store == "e4m3":
        return round_to_e4m3(x)
    raise ValueError(store)


# --------------------------------------------------------------------------
# Q8_0 weights
# --------------------------------------------------------------------------

Q8_0_BLOCK = 32


def quantize_q8_0(w: np.ndarray):
    """Q8_0 encoding of a matrix, row by row.  [LC] "The GGUF format
    (reference)" lists Q8_0 among the tensor element types without giving its
    layout; the reading taken: each row is cut
    into blocks of 32 consecutive elements from its start (a last, shorter
    block keeps what is left); a block stores one scale and 32 signed bytes.
    In float32 arithmetic, with each operation rounded once:

        d = max|w| / 127            (the block's largest magnitude)
        q = nearest integer to w / d, ties to even   (|q| <= 127)

    and the stored scale is d rounded to fp16 (nearest, ties to even).  A block
    of zeros has d = 0 and q = 0.  ``w`` is widened to float32 first (exact for
    bf16 and fp16 values).  Returns (q int8 [N][K], d float16 [N][ceil(K/32)])."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    nb = (k + Q8_0_BLOCK - 1) // Q8_0_BLOCK
    blocks = np.zeros((n, nb * Q8_0_BLOCK), dtype=np.float32)
    blocks[:, :k] = w                              # zeros do not change a block's max|w|
    blocks = blocks.reshape(n, nb, Q8_0_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    d = amax / np.float32(127)                     # float32 / float32: one rounding
    safe = np.where(d > 0, d, np.float32(1)).astype(np.float32)
    q = np.rint(blocks / safe[:, :, None])         # numpy rounds halves to even
    q = np.where(d[:, :, None] > 0, q, 0).astype(np.int8)
    return q.reshape(n, nb * Q8_0_BLOCK)[:, :k].copy(), d.astype(np.float16)


def dequantize_q8_0(q: np.ndarray, d: np.ndarray, dtype=np.float64) -> np.ndarray:
    """The weights a Q8_0 matrix stands for: q times its block's stored (fp16)
    scale, exact in float64."""
    q = np.asarray(q)
    k = q.shape[1]
    scale = np.repeat(np.asarray(d).astype(dtype), Q8_0_BLOCK, axis=1)[:, :k]
    return q.astype(dtype) * scale


def bf16_to_float(bits: np.ndarray, dtype=np.float64) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16): a bf16 value is the top
    half of the fp32 value with the same bits."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        return bits.astype(dtype)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(dtype)


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm ([EN] "AttentionNorm (RMSNorm)", "MLPNorm (RMSNorm)",
    ``OutputNorm``): each row divided by sqrt(mean of its squares + eps), then
    multiplied elementwise by the gain.  Reading: eps inside the square root,
    mean over the model dimension, no bias."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope_angles(pos: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """Rotation angles [T][head_dim/2]: pos * theta^(-2i/head_dim) for pair i.
    [EN] "Q, K = RoPE(Q, positions), RoPE(K, positions)"; the pages name RoPE
    without a formula, so this is the standard rotary encoding with frequency
    scale 1 ([LC] context parameters leave rope scaling at its default)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate x [T][n_heads][head_dim] by position.  Reading: the pair i is the
    adjacent elements (2i, 2i+1); (a, b) -> (a cos - b sin, a sin + b cos)."""
    hd = x.shape[-1]
    ang = rope_angles(pos, hd, theta)                 # [T][hd/2]
    c = np.cos(ang)[:, None, :].astype(x.dtype)
    s = np.sin(ang)[:, None, :].astype(x.dtype)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def attention_one_seq(q, k, v, q_pos, k_pos, n_head_kv, return_probs=False, window=0):
    """Grouped-query scaled-dot-product attention of one sequence's queries
    against that sequence's cached keys ([EN] "attention =
    ScaledDotProduct(Q, K, V, cache)", GQA with fewer KV heads broadcast;
    "Full causal mask"; [LC] "Q is multiplied by all keys in the cache (and by
    itself), after mask and softmax by all values").

    q [Tq][H][hd], k/v [S][Hkv][hd], q_pos [Tq], k_pos [S].
    Readings: scale 1/sqrt(hd); query head h uses KV head h // (H/Hkv); key c
    is visible to query t iff k_pos[c] <= q_pos[t]; softmax subtracts the row
    maximum.  With window W > 0 (sliding-window attention, [EN] "KV Cache":
    each layer attends only to the most recent swaWindowSize tokens) key c is
    visible only if also q_pos[t] - k_pos[c] < W, i.e. the W latest positions
    up to and including the query's own.  Returns o [Tq][H][hd] (and the
    probabilities [H][Tq][S])."""
    tq, n_head, hd = q.shape
    group = n_head // n_head_kv
    scale = 1.0 / np.sqrt(hd)
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]   # [Tq][S]
    if window > 0:
        visible &= (np.asarray(q_pos)[:, None] - np.asarray(k_pos)[None, :]) < window
    out = np.empty_like(q)
    probs = [] if return_probs else None
    for h in range(n_head):
        j = h // group
        scores = (q[:, h, :] @ k[:, j, :].T) * scale                    # [Tq][S]
        scores = np.where(visible, scores, -np.inf)
        m = np.max(scores, axis=1, keepdims=True)
        e = np.exp(scores - m)
        p = e / np.sum(e, axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, j, :]
        if return_probs:
            probs.append(p)
    if return_probs:
        return out, np.stack(probs)
    return out


def silu(x):
    """SiLU(x) = x / (1 + exp(-x))."""
    return x / (1.0 + np.exp(-x))


def swiglu_mlp(x, w_gate, w_up, w_down):
    """[EN] MLP: Down(SiLU(Gate x) * Up x), weights [out][in]."""
    return (silu(x @ w_gate.T) * (x @ w_up.T)) @ w_down.T


# --------------------------------------------------------------------------
# Model, KV cache and one ubatch
# --------------------------------------------------------------------------

class Model:
    """Weights of a Llama model as host bf16 bit arrays (or float arrays),
    widened one tensor at a time on use.  Names follow the GGUF tags of the
    Llama struct ([EN] "Initialising the model with reflection"); ``output``
    falls back to ``token_embd`` when absent (``alt:token_embd``)."""

    def __init__(self, hp: Hparams, weights: dict, dtype=np.float64):
        self.hp, self.w, self.dtype = hp, weights, dtype

    def get(self, name):
        if name == "output" and (self.hp.tied_output or "output" not in self.w):
            name = "token_embd"
        return bf16_to_float(self.w[name], self.dtype)

    def layer(self, i):
        return {t: self.get(f"blk.{i}.{t}") for t in (
            "attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
            "ffn_norm", "ffn_gate", "ffn_up", "ffn_down")}

    def embed_rows(self, tokens):
        """[LC] Step 11: row ``token[i]`` of the embedding table becomes input
        row i (widened exactly)."""
        return bf16_to_float(np.asarray(self.w["token_embd"])[np.asarray(tokens)], self.dtype)

    # the matrices a layer multiplies by (GGUF tags)
    MATRICES = ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down")

    def quantized_q8_0(self) -> "Model":
        """The same model with its matrices stored as Q8_0 (quantize_q8_0) and
        used as the weights they stand for (dequantize_q8_0).  Reading: every
        matrix a projection multiplies by is quantised (the layers' Q, K, V,
        output, gate, up and down, and the output projection); the token
        embedding table is a lookup, kept as it is, unless it is also the
        output projection (tied), when the lookup reads the quantised table
        too.  Norm gains stay as they are."""
        w = dict(self.w)

        def q8(name):
            q, d = quantize_q8_0(bf16_to_float(self.w[name], np.float32))
            w[name] = dequantize_q8_0(q, d, np.float64)

        for i in range(self.hp.n_layer):
            for t in self.MATRICES:
                q8(f"blk.{i}.{t}")
        q8("token_embd" if self.hp.tied_output or "output" not in self.w else "output")
        return Model(self.hp, w, self.dtype)


class KVCache:
    """Per-sequence, per-layer cache of K and V by position ([EN] ``Causal``:
    per-layer keys/values plus position and sequence metadata per cell; [LC]
    "KV-cache and the Prefill / Decode stages").  Entries stay in ``dtype``
    unless ``store`` asks to round them as a lower-precision cache would."""

    def __init__(self, hp: Hparams, n_ctx: int, n_seq_max: int, dtype, store=None, window=0):
        self.hp, self.n_ctx, self.n_seq_max, self.store = hp, n_ctx, n_seq_max, store
        self.window = window          # sliding-window size, 0 = full causal
        shape = (n_seq_max, hp.n_layer, n_ctx, hp.n_head_kv, hp.head_dim)
        self.k = np.zeros(shape, dtype)
        self.v = np.zeros(shape, dtype)
        self.filled = np.zeros((n_seq_max, n_ctx), bool)

    def seq_pos_max(self, s):
        """[LC] ``memory->seq_pos_max(s)``: highest cached position, -1 if none."""
        idx = np.nonzero(self.filled[s])[0]
        return int(idx[-1]) if idx.size else -1

    def clear(self, s):
        self.filled[s] = False

    def discard(self, s, p0, n):
        """Context shift ([EN] "KV Cache": when the cache is full the model's
        Shift function adjusts the RoPE position encoding so the window slides
        forward without discarding the whole context).  Reading: positions
        [p0, p0 + n) of sequence s are dropped; every later cell moves to its
        position - n, its key re-rotated by the RoPE rotation of -n (rotations
        compose, so R(-n) R(p) = R(p - n)); values do not depend on position."""
        end = self.seq_pos_max(s) + 1
        if not (0 <= p0 and n >= 1 and p0 + n <= end):
            raise ValueError("discard range outside the sequence")
        hp = self.hp
        src = np.arange(p0 + n, end)
        for layer in range(hp.n_layer):
            k = self.k[s, layer, src]
            k = rope(k.astype(np.float64), np.full(src.size, -n), hp.rope_theta).astype(self.k.dtype)
            self.k[s, layer, src - n] = round_to(k, self.store)
            self.v[s, layer, src - n] = self.v[s, layer, src]
        self.filled[s, end - n:end] = False


def layer_forward(hp, lw, h, pos, seq, cache, layer, out_rows=None):
    """One decoder layer on the rows of a ubatch ([EN] sequence diagram of
    ``layer.Forward``): RMSNorm -> Q,K,V -> RoPE(Q,K) -> store K,V for the new
    positions -> attention over the cache -> output projection + residual ->
    (last layer only: keep the output rows) -> RMSNorm -> SwiGLU + residual.

    K/V of every row of the ubatch are stored before attention, so a token
    attends to itself and to earlier tokens of the same ubatch ([EN] "Store
    K,V for new positions" precedes "Build attention mask")."""
    t_rows = h.shape[0]
    H, Hkv, hd = hp.n_head, hp.n_head_kv, hp.head_dim
    x = rms_norm(h, lw["attn_norm"], hp.rms_eps)
    q = (x @ lw["attn_q"].T).reshape(t_rows, H, hd)
    k = (x @ lw["attn_k"].T).reshape(t_rows, Hkv, hd)
    v = (x @ lw["attn_v"].T).reshape(t_rows, Hkv, hd)
    q = rope(q, pos, hp.rope_theta)
    k = rope(k, pos, hp.rope_theta)
    for r in range(t_rows):
        cache.k[seq[r], layer, pos[r]] = round_to(k[r], cache.store)
        cache.v[seq[r], layer, pos[r]] = round_to(v[r], cache.store)
        cache.filled[seq[r], pos[r]] = True
    o = np.empty_like(q)
    for s in np.unique(seq):
        rows = np.nonzero(seq == s)[0]
        cells = np.nonzero(cache.filled[s])[0]
        o[rows] = attention_one_seq(q[rows], cache.k[s, layer, cells], cache.v[s, layer, cells],
                                    pos[rows], cells, Hkv, window=cache.window)
    h = h + o.reshape(t_rows, H * hd) @ lw["attn_output"].T
    if out_rows is not None:
        # [EN] Model.Forward: in the last layer the hidden state keeps only the
        # rows batch.Outputs selects, before the MLP.
        h = h[out_rows]
    x = rms_norm(h, lw["ffn_norm"], hp.rms_eps)
    return h + swiglu_mlp(x, lw["ffn_gate"], lw["ffn_up"], lw["ffn_down"])


def layer_rows(hp, lw, h, pos, rows):
    """One decoder layer for selected rows of one sequence whose rows
    [0, len(h)) sit at positions ``pos`` (in cache order): K and V of every
    row, then Q, attention over the keys with position <= the row's, output
    projection + residual and SwiGLU + residual for the rows ``rows`` only.
    This is ``layer_forward`` with the attention of the other rows skipped
    ([EN] Model.Forward keeps only the rows it needs; a row's output depends on
    the other rows only through their K and V), so the result for a selected
    row equals ``layer_forward``'s.  Returns the hidden state [len(rows)][d]."""
    H, Hkv, hd = hp.n_head, hp.n_head_kv, hp.head_dim
    rows = np.asarray(rows, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    x = rms_norm(h, lw["attn_norm"], hp.rms_eps)
    k = rope((x @ lw["attn_k"].T).reshape(-1, Hkv, hd), pos, hp.rope_theta)
    v = (x @ lw["attn_v"].T).reshape(-1, Hkv, hd)
    q = rope((x[rows] @ lw["attn_q"].T).reshape(-1, H, hd), pos[rows], hp.rope_theta)
    o = np.empty_like(q)
    for i, r in enumerate(rows):
        n = int(np.count_nonzero(pos <= pos[r]))      # keys with position <= the row's (cache order)
        o[i:i + 1] = attention_one_seq(q[i:i + 1], k[:n], v[:n], pos[r:r + 1], pos[:n], Hkv)
    hr = h[rows] + o.reshape(len(rows), H * hd) @ lw["attn_output"].T
    xr = rms_norm(hr, lw["ffn_norm"], hp.rms_eps)
    return hr + swiglu_mlp(xr, lw["ffn_gate"], lw["ffn_up"], lw["ffn_down"])


def forward_ubatch(model: Model, cache: KVCache, tokens, pos, seq, output, hidden_out=None,
                   prune=True):
    """[EN] ``Model.Forward`` on one ubatch: embed, every layer (the last one
    with the output rows), final RMSNorm, output projection.  Returns logits
    [n_outputs][n_vocab] for the rows with ``output != 0``, in batch order.

    ``prune=False`` keeps every row through the last layer and selects the
    output rows only before the final norm (used to pin the pruning)."""
    hp = model.hp
    tokens, pos, seq = (np.asarray(a, dtype=np.int64) for a in (tokens, pos, seq))
    out_rows = np.nonzero(np.asarray(output))[0]
    h = model.embed_rows(tokens)
    for i in range(hp.n_layer):
        last = i == hp.n_layer - 1
        h = layer_forward(hp, model.layer(i), h, pos, seq, cache, i,
                          out_rows if (last and prune) else None)
        if hidden_out is not None:
            hidden_out.append(h.copy())
    if not prune:
        h = h[out_rows]
    x = rms_norm(h, model.get("output_norm"), hp.rms_eps)
    return x @ model.get("output").T


# --------------------------------------------------------------------------
# The batch interface: llama_decode semantics
# --------------------------------------------------------------------------

class Context:
    """[LC] ``llama_context`` reduced to what decoding needs: a KV cache of
    ``n_ctx`` positions for each of ``n_seq_max`` sequences, the ubatch size,
    and the logits of the last ``decode`` call."""

    def __init__(self, model: Model, n_ctx: int, n_seq_max: int = 1, n_ubatch: int = 512, kv_store=None,
                 window: int = 0):
        self.model, self.n_ctx, self.n_seq_max, self.n_ubatch = model, n_ctx, n_seq_max, n_ubatch
        self.cache = KVCache(model.hp, n_ctx, n_seq_max, model.dtype, kv_store, window)
        self.logits = np.zeros((0, model.hp.n_vocab), model.dtype)
        self.out_index = {}          # batch index -> logits row
        self.hidden = None           # per ubatch: list of per-layer hidden states

    def seq_pos_max(self, s):
        return self.cache.seq_pos_max(s)

    def seq_clear(self, s):
        self.cache.clear(s)

    def seq_discard(self, s, p0, n):
        """Drop positions [p0, p0 + n) of sequence s and shift the rest down (KVCache.discard)."""
        self.cache.discard(s, p0, n)

    def fill_batch(self, tokens, pos=None, seq=None, output=None):
        """[LC] ``llama_batch_allocr::init``: reject empty batches and token ids
        outside [0, n_vocab); missing seq ids become 0; missing positions
        continue each sequence from seq_pos_max + 1; missing output flags ask
        for the last row only.  Readings: a seq id outside [0, n_seq_max) is
        invalid; each sequence's positions must continue its cache without gaps
        (p, p+1, ...); a position at or past n_ctx means the batch does not fit
        (return 1, the non-error code of ``llama_decode``).  Returns
        (code, tokens, pos, seq, output)."""
        tokens = np.asarray(tokens, dtype=np.int64)
        n = tokens.size
        if n <= 0:
            return INVALID, None, None, None, None
        if np.any(tokens < 0) or np.any(tokens >= self.model.hp.n_vocab):
            return INVALID, None, None, None, None
        seq = np.zeros(n, np.int64) if seq is None else np.asarray(seq, dtype=np.int64)
        if np.any(seq < 0) or np.any(seq >= self.n_seq_max):
            return INVALID, None, None, None, None
        nxt = {s: self.seq_pos_max(s) + 1 for s in range(self.n_seq_max)}
        if pos is None:
            pos = np.empty(n, np.int64)
            for i in range(n):
                pos[i] = nxt[int(seq[i])]
                nxt[int(seq[i])] += 1
        else:
            pos = np.asarray(pos, dtype=np.int64)
            for i in range(n):
                if pos[i] != nxt[int(seq[i])]:
                    return INVALID, None, None, None, None
                nxt[int(seq[i])] += 1
        if output is None:
            output = np.zeros(n, np.int8)
            output[-1] = 1
        output = np.asarray(output, dtype=np.int8)
        if np.any(pos >= self.n_ctx):
            return NO_KV_ROOM, None, None, None, None
        return OK, tokens, pos, seq, output

    def decode(self, tokens, pos=None, seq=None, output=None, keep_hidden=False):
        """[LC] ``llama_decode``: fill the batch, cut it into consecutive
        ubatches of at most n_ubatch tokens (``init_batch``), run each through
        the model, and keep the logits of every flagged row in batch order.
        Reading: the logits of all flagged rows are kept (not only the last
        one), and ``llama_get_logits_ith(i)`` finds row i's logits."""
        code, tokens, pos, seq, output = self.fill_batch(tokens, pos, seq, output)
        if code != OK:
            return code
        rows, self.out_index, self.hidden = [], {}, [] if keep_hidden else None
        for start in range(0, tokens.size, self.n_ubatch):
            sl = slice(start, start + self.n_ubatch)
            hid = [] if keep_hidden else None
            lg = forward_ubatch(self.model, self.cache, tokens[sl], pos[sl], seq[sl], output[sl], hid)
            if keep_hidden:
                self.hidden.append(hid)
            for r, i in enumerate(np.nonzero(output[sl])[0]):
                self.out_index[start + int(i)] = len(rows) + r
            rows.extend(list(lg))
        hp = self.model.hp
        self.logits = np.array(rows, dtype=self.model.dtype).reshape(-1, hp.n_vocab)
        return OK

    def logits_ith(self, i):
        """Logits of batch row i (negative i counts from the end of the
        output rows), or None if row i was not an output."""
        if i < 0:
            return self.logits[i] if -i <= len(self.logits) else None
        r = self.out_index.get(i)
        return None if r is None else self.logits[r]


def greedy_argmax(logits: np.ndarray) -> np.ndarray:
    """[EN] "Token sampling pipeline": temperature 0 takes the argmax.
    Reading: ties go to the lowest token id (``np.argmax`` returns the first)."""
    return np.argmax(np.atleast_2d(logits), axis=-1)


def generate_greedy(ctx: Context, prompt, n_steps: int, seq: int = 0, forced=None):
    """[LC] generation loop: decode the prompt with logits for its last row,
    take the argmax, decode that one token at the next position, repeat.
    ``forced`` (optional) replaces the chosen token at each step, so another
    implementation can be driven along the oracle's own choices.  Returns
    (tokens chosen, logits of each step [n_steps+1][n_vocab])."""
    n = len(prompt)
    out = np.zeros(n, np.int8)
    out[-1] = 1
    code = ctx.decode(prompt, seq=np.full(n, seq), output=out)
    assert code == OK, code
    chosen, logits = [], [ctx.logits[-1].copy()]
    for step in range(n_steps):
        tok = int(greedy_argmax(ctx.logits[-1])[0])
        if forced is not None:
            tok = int(forced[step])
        chosen.append(tok)
        code = ctx.decode([tok], seq=[seq])
        assert code == OK, code
        logits.append(ctx.logits[-1].copy())
    return np.array(chosen, np.int64), np.array(logits)
