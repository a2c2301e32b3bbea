"""Pure-Python brute-force Llama forward (explicit index loops, ``math`` only).

Used only to pin the numpy oracle on tiny models: it shares no code with the
oracle and spells every contraction out element by element, so a transposed
operand, a wrong head mapping, a dropped residual or a mask off by one in
either implementation makes the two disagree.
"""
import math


def _matvec(w, x):
    """w: list of rows [out][in]; y[o] = sum_i w[o][i] * x[i]."""
    return [sum(w[o][i] * x[i] for i in range(len(x))) for o in range(len(w))]


def _rmsnorm(x, g, eps):
    ms = sum(v * v for v in x) / len(x)
    inv = 1.0 / math.sqrt(ms + eps)
    return [x[i] * inv * g[i] for i in range(len(x))]


def _rotate(vec, pos, theta):
    hd = len(vec)
    out = list(vec)
    for i in range(hd // 2):
        ang = pos * math.pow(theta, -2.0 * i / hd)
        a, b = vec[2 * i], vec[2 * i + 1]
        out[2 * i] = a * math.cos(ang) - b * math.sin(ang)
        out[2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
    return out


class BruteLlama:
    """hp: object with the Llama hyper-parameters; w: dict of nested lists
    (matrices [out][in], vectors), names as the GGUF tags."""

    def __init__(self, hp, w):
        self.hp, self.w = hp, w
        self.cache = {}   # (seq, layer) -> list of (pos, [k per kv head], [v per kv head])

    def batch(self, tokens, pos, seq, outputs):
        hp, w = self.hp, self.w
        H, Hkv, hd = hp.n_head, hp.n_head_kv, hp.head_dim
        group = H // Hkv
        h = [list(w["token_embd"][t]) for t in tokens]
        rows = list(range(len(tokens)))
        for l in range(hp.n_layer):
            p = f"blk.{l}."
            qs = {}
            for t in rows:
                x = _rmsnorm(h[t], w[p + "attn_norm"], hp.rms_eps)
                q = _matvec(w[p + "attn_q"], x)
                k = _matvec(w[p + "attn_k"], x)
                v = _matvec(w[p + "attn_v"], x)
                qs[t] = [_rotate(q[a * hd:(a + 1) * hd], pos[t], hp.rope_theta) for a in range(H)]
                kh = [_rotate(k[a * hd:(a + 1) * hd], pos[t], hp.rope_theta) for a in range(Hkv)]
                vh = [v[a * hd:(a + 1) * hd] for a in range(Hkv)]
                self.cache.setdefault((seq[t], l), []).append((pos[t], kh, vh))
            for t in rows:
                o = []
                for a in range(H):
                    j = a // group
                    ents = [e for e in self.cache[(seq[t], l)] if e[0] <= pos[t]]
                    sc = [sum(qs[t][a][d] * e[1][j][d] for d in range(hd)) / math.sqrt(hd) for e in ents]
                    m = max(sc)
                    ex = [math.exp(s - m) for s in sc]
                    z = sum(ex)
                    o.extend(sum(ex[c] / z * ents[c][2][j][d] for c in range(len(ents))) for d in range(hd))
                y = _matvec(w[p + "attn_output"], o)
                h[t] = [h[t][i] + y[i] for i in range(len(y))]
            if l == hp.n_layer - 1:
                rows = [t for t in rows if outputs[t]]
            for t in rows:
                x = _rmsnorm(h[t], w[p + "ffn_norm"], hp.rms_eps)
                a = _matvec(w[p + "ffn_gate"], x)
                b = _matvec(w[p + "ffn_up"], x)
                u = [a[i] / (1.0 + math.exp(-a[i])) * b[i] for i in range(len(a))]
                y = _matvec(w[p + "ffn_down"], u)
                h[t] = [h[t][i] + y[i] for i in range(len(y))]
        wout = w["token_embd"] if hp.tied_output else w["output"]
        return [_matvec(wout, _rmsnorm(h[t], w["output_norm"], hp.rms_eps)) for t in rows]
