"""The stored full-depth expected values (tests/golden/*.npz, written by
tests/golden/make_goldens.py from the oracle alone) are internally
consistent: every row's argmax is its first top id, the 32 top logits are in
descending order with the stored margin their first gap, and where a whole
row is stored its top-32 values, its values at the 512 fixed ids and its
argmax agree with the per-row summaries.  The token streams have the
workload's sizes and every decode token is the oracle's argmax of the
previous row(s)."""
import glob
import os

import numpy as np
import pytest

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
FILES = sorted(glob.glob(os.path.join(HERE, "golden", "*.npz")))
WORKLOADS = {w.name: w for w in synth.WORKLOADS.values()}


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(p) for p in FILES])
def test_golden_file_is_consistent(path):
    g = np.load(path)
    name = str(g["workload"])
    wl = WORKLOADS[name]
    n_seq, steps = int(g["n_seq"]), int(g["steps"])
    rows = int(g["argmax"].shape[0])
    assert rows == n_seq * (steps + 1)
    assert int(g["seed"]) == wl.seed and int(g["n_layer"]) == wl.shape.n_layer and int(g["n_ctx"]) == wl.n_ctx
    top_ids, top_vals = g["top_ids"], g["top_vals"]
    assert top_ids.shape == (rows, 32) and top_vals.shape == (rows, 32)
    assert np.array_equal(g["argmax"], top_ids[:, 0])
    assert np.all(np.diff(top_vals, axis=1) <= 0)
    assert np.allclose(g["margin"], top_vals[:, 0] - top_vals[:, 1], rtol=0, atol=1e-6)
    assert np.all(g["margin"] >= 0)
    full, full_rows = g["full"], g["full_rows"]
    assert full.shape == (len(full_rows), wl.shape.n_vocab)
    for i, r in enumerate(full_rows):
        assert np.array_equal(full[i][top_ids[r]], top_vals[r])
        assert np.array_equal(full[i][g["sample_ids"]], g["sample_vals"][r])
        assert int(np.argmax(full[i])) == int(g["argmax"][r])
    # the prompt and the decode tokens: the oracle's own greedy choices
    seq_lens = np.asarray(g["seq_lens"])
    assert len(g["prompt_tokens"]) == int(seq_lens.sum()) and len(seq_lens) == n_seq
    assert g["decode_tokens"].shape == (steps, n_seq)
    am = g["argmax"].reshape(steps + 1, n_seq)
    assert np.array_equal(g["decode_tokens"], am[:steps])
    if n_seq == 1:
        assert np.array_equal(g["prompt_tokens"], synth.prompt(wl.shape.n_vocab, wl.seed, wl.prompt_len))
