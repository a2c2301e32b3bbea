"""The seeded input generator (synth): its integer stream is splitmix64 as
published (checked against a plain numpy uint64 restatement), its normals
have the stated mean and spread, its token draws are uniform and in range,
and a CUDA draw gives the same bf16 tensor as a CPU draw, which is what lets
expected values computed on the CPU apply to weights drawn on the GPU."""
import numpy as np
import pytest
import torch

import synth


def _splitmix_words(key, start, n):
    """Word i of a stream: the splitmix64 output of state key + (i + 1) * G
    (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    2014), in numpy uint64 arithmetic."""
    G = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + np.arange(start + 1, start + n + 1, dtype=np.uint64) * G
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def test_word_stream_is_splitmix64():
    for key in (0, 1, synth.tensor_seed(3, "blk.0.attn_q"), (1 << 63) - 1):
        got = synth._words(key, 1000, 257, "cpu").numpy().view(np.uint64)
        assert np.array_equal(got, _splitmix_words(key, 1000, 257))


def test_normals_and_weights_have_the_stated_distribution():
    z = synth._normal_chunk(synth.tensor_seed(0, "x"), 0, 1 << 20, "cpu").numpy()
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(np.abs(z) < 1.0) - 0.6827) < 3e-3          # one-sigma mass
    w = synth.make_tensor(synth.LLAMA_1B, 1, "blk.0.attn_q").float()
    assert abs(w.mean().item()) < 1e-4 and abs(w.std().item() - 0.02) < 1e-4
    g = synth.make_tensor(synth.LLAMA_1B, 1, "blk.0.attn_norm").float()
    assert abs(g.mean().item() - 1.0) < 3e-3 and abs(g.std().item() - 0.02) < 3e-3


def test_tokens_and_lengths_are_uniform_and_in_range():
    t = synth.prompt(1000, 7, 200000)
    assert t.min() == 0 and t.max() == 999 and t.dtype == np.int32
    counts = np.bincount(t, minlength=1000)
    assert abs(counts.mean() - 200) < 1e-9 and counts.std() < 3 * np.sqrt(200)
    lens = synth.multislot_lengths(4, 8)
    assert lens.shape == (8,) and lens.min() >= 256 and lens.max() <= 4096
    assert not np.array_equal(synth.prompt(1000, 7, 50), synth.prompt(1000, 8, 50))


@pytest.mark.gpu
def test_cuda_draws_equal_cpu_draws():
    for shape, seed, name in ((synth.LLAMA_8B, 3, "blk.5.ffn_down"), (synth.LLAMA_8B, 4, "token_embd"),
                              (synth.LLAMA_1B, 1, "blk.0.ffn_norm"), (synth.TINY, 0, "output")):
        a = synth.make_tensor(shape, seed, name, "cpu")
        b = synth.make_tensor(shape, seed, name, "cuda").cpu()
        diff = (a.view(torch.int16) != b.view(torch.int16)).sum().item()
        assert diff == 0, (name, diff)
