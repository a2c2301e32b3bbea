"""Seeded synthetic inputs for the Llama decoder forward pass.

This module only draws numbers: model shapes, bf16 weights, norm gains and
token streams.  It holds none of the forward pass's arithmetic, so both the
CUDA path (through the C ABI) and the CPU oracle can take their inputs from it
without sharing any computation.

Weights follow the workload recipe of the model shapes used here: every matrix
is N(0, 0.02) in fp32, rounded to bf16 (round to nearest even, which is what
``Tensor.to(torch.bfloat16)`` does); every RMSNorm gain is 1 + N(0, 0.02),
rounded the same way.  Each tensor has its own generator, seeded from the
config seed and the tensor's name, so a tensor does not change when another
one is added or skipped.  Prompts are uniform over [0, n_vocab).  Draws come
from a counter-based generator built from integer operations, so the CPU and
a GPU produce the same tensors (expected values computed on the CPU apply to
weights drawn on the GPU).

Tensor names follow the GGUF tags of the Llama model struct ("Inside the
inference engine: model architectures and forward pass", section "Initialising
the model with reflection"): ``token_embd``, ``output_norm``, ``output`` and
per layer ``blk.{i}.attn_norm / attn_q / attn_k / attn_v / attn_output /
ffn_norm / ffn_gate / ffn_up / ffn_down``.  Matrices are row-major [out][in].
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, asdict

import numpy as np
import torch


@dataclass(frozen=True)
class Shape:
    """Model hyper-parameters (the llama.cpp ``hparams`` fields that the
    Llama forward pass reads, plus the tied-output flag)."""
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

    def asdict(self):
        return asdict(self)


# The five workloads: tiny Llama, ~1B shape, Llama-3-8B shape, 8B long
# context, 8B multi-slot serving (tied output).
TINY = Shape(512, 128, 2, 4, 2, 32, 344, 1e-5, 10000.0, False)
LLAMA_1B = Shape(32000, 2048, 16, 32, 8, 64, 8192, 1e-5, 10000.0, True)
LLAMA_8B = Shape(128256, 4096, 32, 32, 8, 128, 14336, 1e-5, 500000.0, False)
LLAMA_8B_TIED = Shape(128256, 4096, 32, 32, 8, 128, 14336, 1e-5, 500000.0, True)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    seed: int
    n_ctx: int
    n_ubatch: int
    n_seq: int
    prompt_len: int          # per sequence (single-sequence workloads)
    decode_steps: int


WORKLOADS = {
    0: Workload("tiny", TINY, 0, 64, 16, 1, 16, 16),
    1: Workload("llama1b", LLAMA_1B, 1, 4096, 512, 1, 512, 256),
    2: Workload("llama8b", LLAMA_8B, 2, 4096, 512, 1, 2048, 128),
    3: Workload("llama8b_long", LLAMA_8B, 3, 32768, 512, 1, 32000, 64),
    4: Workload("llama8b_multislot", LLAMA_8B_TIED, 4, 8192, 512, 8, 0, 128),
}


def tensor_seed(seed: int, name: str) -> int:
    """A stable 63-bit key for one named tensor (or token stream) of one workload."""
    h = zlib.crc32(f"{seed}/{name}".encode()) & 0xFFFFFFFF
    return (seed * 0x9E3779B1 + h * 0x85EBCA77) & 0x7FFF_FFFF_FFFF_FFFF


# Counter-based generator: element i of a stream with key k is the splitmix64
# output of the state k + (i+1)*G (G the 64-bit golden-ratio increment),
# computed with wrapping int64 tensor arithmetic.  The same integer operations
# run on any device, so a CPU draw and a CUDA draw give the same words; a
# normal takes one float64 Box-Muller step on the word's two 32-bit halves,
# whose log / cos may differ by an ulp between devices, far below the bf16
# rounding that follows.
_G = -7046029254386353131          # 0x9E3779B97F4A7C15 as int64
_C1 = -4658895280553007687         # 0xBF58476D1CE4E5B9
_C2 = -7723592293110705685         # 0x94D049BB133111EB
_CHUNK = 1 << 24


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    """splitmix64 output function (bijective on 64-bit words)."""
    z = (z ^ _lsr(z, 30)) * _C1
    z = (z ^ _lsr(z, 27)) * _C2
    return z ^ _lsr(z, 31)


def _words(key: int, start: int, n: int, device) -> torch.Tensor:
    """Words of elements [start, start + n) of stream `key`."""
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix(i * _G + key)


def _normal_chunk(key: int, start: int, n: int, device) -> torch.Tensor:
    """Standard normals (float64) of elements [start, start + n): Box-Muller
    on u1 = (high half + 1/2) / 2^32 in (0, 1) and u2 = low half / 2^32."""
    w = _words(key, start, n, device)
    u1 = (_lsr(w, 32).double() + 0.5) * 2.0 ** -32
    u2 = (w & 0xFFFFFFFF).double() * 2.0 ** -32
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _below(key: int, n: int, bound: int) -> torch.Tensor:
    """n integers uniform in [0, bound) (bound < 2^31): the high 32 bits of a
    word times bound, shifted down 32 (exact in int64)."""
    return (_lsr(_words(key, 0, n, "cpu"), 32) * bound) >> 32


def make_tensor(shape: Shape, seed: int, name: str, device="cpu") -> torch.Tensor:
    """One bf16 tensor: N(0, 0.02) (norm gains 1 + N(0, 0.02)) in float64,
    rounded to float32 and then to bf16 (nearest, ties to even), drawn on
    ``device`` in chunks; CPU and CUDA draws agree."""
    dims = tensor_shape(shape, name)
    n = int(np.prod(dims))
    key = tensor_seed(seed, name)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s0 in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s0)
        x = _normal_chunk(key, s0, m, device) * 0.02
        if name.endswith("norm"):
            x = x + 1.0
        out[s0:s0 + m] = x.float().to(torch.bfloat16)
    return out.view(dims)


def make_weights(shape: Shape, seed: int, device="cpu") -> dict:
    """All tensors of a model as bf16 torch tensors on ``device`` (the same
    values on every device)."""
    return {n: make_tensor(shape, seed, n, device) for n in tensor_names(shape)}


def prompt(n_vocab: int, seed: int, n_tokens: int, stream: str = "prompt") -> np.ndarray:
    """``n_tokens`` token ids uniform over [0, n_vocab), int32."""
    return _below(tensor_seed(seed, stream), n_tokens, n_vocab).numpy().astype(np.int32)


def multislot_lengths(seed: int = 4, n_seq: int = 8, lo: int = 256, hi: int = 4096) -> np.ndarray:
    """Prompt lengths of the multi-slot workload: ``n_seq`` ints uniform in [lo, hi]."""
    return (lo + _below(tensor_seed(seed, "lengths"), n_seq, hi - lo + 1)).numpy().astype(np.int32)


def tensor_names(shape: Shape):
    names = ["token_embd", "output_norm"]
    if not shape.tied_output:
        names.append("output")
    for i in range(shape.n_layer):
        for t in ("attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
                  "ffn_norm", "ffn_gate", "ffn_up", "ffn_down"):
            names.append(f"blk.{i}.{t}")
    return names


def tensor_shape(shape: Shape, name: str):
    d, hd = shape.n_embd, shape.head_dim
    q, kv, f = shape.n_head * hd, shape.n_head_kv * hd, shape.n_ff
    leaf = name.split(".")[-1]
    return {
        "token_embd": (shape.n_vocab, d),
        "output": (shape.n_vocab, d),
        "output_norm": (d,),
        "attn_norm": (d,),
        "ffn_norm": (d,),
        "attn_q": (q, d),
        "attn_k": (kv, d),
        "attn_v": (kv, d),
        "attn_output": (d, q),
        "ffn_gate": (f, d),
        "ffn_up": (f, d),
        "ffn_down": (d, f),
    }[leaf]


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a tensor as a host uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_weights(weights: dict) -> dict:
    """bf16 tensors → dict of host uint16 bit arrays (for the oracle)."""
    return {k: bf16_bits(v) for k, v in weights.items()}


def scaled_shape(base: Shape, **kw) -> Shape:
    """A copy of ``base`` with some fields replaced (small test models)."""
    d = base.asdict()
    d.update(kw)
    return Shape(**d)
