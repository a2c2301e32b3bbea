"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, and its host-side batch rules (llm_batch_check, the same code
llm_decode runs) agree with the oracle's reading of llama_batch_allocr::init
and the ubatch split on random batches.  No GPU call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT

lib = pytest.importorskip("llama_decoder_forward_02_gb300")
from oracle import llama as O  # noqa: E402


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "llm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(llm_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 20
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
        assert hasattr(lib, n), f"binding lacks {n}"


def test_create_rejects_bad_arguments_without_gpu():
    out = ctypes.c_void_p(123)
    assert lib.llm_model_create(None, None, None, ctypes.byref(out)) == lib.LLM_ERR_INVALID
    assert out.value is None
    assert b"NULL" in lib.llm_last_error(None)
    hp = lib.llm_hparams(512, 128, 2, 4, 2, 48, 344, 1e-5, 1e4, 0)    # head_dim 48 unsupported
    w = lib.llm_weights()
    assert lib.llm_model_create(ctypes.byref(hp), ctypes.byref(w), None, ctypes.byref(out)) == lib.LLM_ERR_INVALID
    assert lib.llm_kv_alloc(None, 64, 1, 16, None, ctypes.byref(out)) == lib.LLM_ERR_INVALID
    assert lib.llm_decode(None, None) == lib.LLM_ERR_INVALID
    assert lib.llm_seq_pos_max(None, 0) == lib.LLM_ERR_INVALID
    # Q8_0 entry points: argument checks come before any device work
    assert lib.llm_model_quantize(None, lib.LLM_WTYPE_Q8_0, None) == lib.LLM_ERR_INVALID
    for n, k in ((0, 256), (4, 0), (4, 128), (4, 300)):
        assert lib.llm_op_quantize_q8_0(ctypes.c_void_p(16), n, k, ctypes.c_void_p(16), None) == lib.LLM_ERR_INVALID
    assert lib.llm_op_quantize_q8_0(None, 4, 256, ctypes.c_void_p(16), None) == lib.LLM_ERR_INVALID
    assert lib.llm_op_gemv_q8_0(None, None, None, 256, 256, None) == lib.LLM_ERR_INVALID
    # failure-path hooks: argument checks only
    assert lib.llm_op_wait_check(0, 0, ctypes.c_void_p(16), None) == lib.LLM_ERR_INVALID
    assert lib.llm_op_wait_check(0, 100, None, None) == lib.LLM_ERR_INVALID
    assert lib.llm_debug_fail_alloc(-2) == lib.LLM_ERR_INVALID
    assert lib.llm_debug_fail_alloc(3) == lib.LLM_OK and lib.llm_debug_fail_alloc(-1) == lib.LLM_OK


def test_attention_ops_check_shapes_before_any_device_work():
    """The standalone attention entry points refuse shapes their kernels do not
    cover (and prefill rows outside the cache, read from host arrays) before
    they touch the GPU; the reason is in llm_last_error(NULL)."""
    p = ctypes.c_void_p(256)                     # never dereferenced: the checks come first
    nb = lib.llm_op_attn_decode_scratch_bytes(1, 8, 64, 4)
    cases = [  # (T, H, Hkv, hd, n_ctx, n_seq, n_split, reason)
        (1, 12, 4, 64, 64, 1, 4, b"1, 2, 4 or 8"), (1, 8, 2, 64, 64, 1, 129, b"n_split"),
        (1, 8, 2, 64, 64, 1, 0, b"n_split"), (9, 8, 2, 64, 64, 1, 4, b"T must"), (1, 8, 2, 48, 64, 1, 4, b"head_dim"),
        (1, 8, 3, 64, 64, 1, 4, b"multiple"), (1, 8, 2, 64, 64, 0, 4, b"n_seq"),
    ]
    for T, H, Hkv, hd, n_ctx, n_seq, ns, why in cases:
        assert lib.llm_op_attn_decode(p, p, p, p, p, p, T, H, Hkv, hd, n_ctx, n_seq, ns, p, 1 << 30,
                                      None) == lib.LLM_ERR_INVALID
        assert why in lib.llm_last_error(None), (why, lib.llm_last_error(None))
        assert lib.llm_op_attn_decode_noalloc(p, p, p, p, p, p, T, H, Hkv, hd, n_ctx, n_seq, ns,
                                              None) == lib.LLM_ERR_INVALID
        assert why in lib.llm_last_error(None)
    assert lib.llm_op_attn_decode(p, p, p, p, p, p, 1, 8, 2, 64, 64, 1, 4, p, nb - 1, None) == lib.LLM_ERR_INVALID
    assert lib.llm_op_attn_decode(p, p, p, p, p, p, 1, 8, 2, 64, 64, 1, 4, None, nb, None) == lib.LLM_ERR_INVALID
    # prefill: rows past n_ctx, sequences past n_seq, gaps
    for pos, seq, why in (([62, 63, 64], [0, 0, 0], b"n_ctx"), ([-1, 0], [0, 0], b"n_ctx"),
                          ([0, 1], [1, 1], b"n_seq"), ([0, 2], [0, 0], b"consecutive")):
        ph = (ctypes.c_int32 * len(pos))(*pos)
        sh = (ctypes.c_int32 * len(seq))(*seq)
        assert lib.llm_op_attn_prefill(p, p, p, ph, sh, p, len(pos), 8, 2, 64, 64, 1, None) == lib.LLM_ERR_INVALID
        assert why in lib.llm_last_error(None), why


class _Stub:
    """Just enough of an oracle Model for Context.fill_batch."""
    def __init__(self, n_vocab):
        self.hp = O.Hparams(n_vocab, 8, 1, 1, 1, 8, 8, 1e-5, 1e4, False)
        self.dtype = np.float64


def check_host(n_vocab, n_ctx, n_seq, n_ub, spm, tokens, pos, seq, out):
    sp = (ctypes.c_int32 * n_seq)(*spm)
    b, keep = lib.batch(tokens, pos, seq, out)
    n = len(tokens)
    pos_o = (ctypes.c_int32 * max(n, 1))()
    idx_o = (ctypes.c_int32 * max(n, 1))()
    ubs = (ctypes.c_int32 * max(n, 1))()
    nub = ctypes.c_int32()
    rc = lib.llm_batch_check(n_vocab, n_ctx, n_seq, n_ub, sp, ctypes.byref(b), pos_o, idx_o, ubs, ctypes.byref(nub))
    return rc, list(pos_o[:n]), list(idx_o[:n]), list(ubs[:nub.value])


def test_batch_rules_match_oracle_on_random_batches():
    rng = np.random.default_rng(5)
    agree = {0: 0, 1: 0, -1: 0}
    for trial in range(400):
        n_vocab, n_ctx, n_seq, n_ub = 50, int(rng.integers(4, 20)), int(rng.integers(1, 4)), int(rng.integers(1, 6))
        ctx = O.Context(_Stub(n_vocab), n_ctx=n_ctx, n_seq_max=n_seq, n_ubatch=n_ub)
        spm = [int(rng.integers(-1, n_ctx // 2)) for _ in range(n_seq)]
        for s, pmax in enumerate(spm):
            ctx.cache.filled[s, :pmax + 1] = True
        n = int(rng.integers(0, 8))
        tokens = [int(v) for v in rng.integers(-2, n_vocab + 2 if trial % 5 == 0 else n_vocab, size=n)]
        seq = None if rng.random() < 0.4 else [int(v) for v in rng.integers(0, n_seq + (trial % 7 == 0), size=n)]
        out = None if rng.random() < 0.5 else [int(v) for v in rng.integers(0, 2, size=n)]
        pos = None
        if rng.random() < 0.5 and n:
            nxt = {s: spm[s] + 1 for s in range(n_seq)}
            pos = []
            for i in range(n):
                s = seq[i] if seq is not None else 0
                pos.append(nxt.get(s, 0) + (1 if rng.random() < 0.1 else 0))
                nxt[s] = nxt.get(s, 0) + 1
        code, t, p, s, o = ctx.fill_batch(tokens, pos, seq, out)
        rc, pos_o, idx_o, ubs = check_host(n_vocab, n_ctx, n_seq, n_ub, spm, tokens, pos, seq, out)
        assert rc == code, (tokens, pos, seq, out, spm, n_ctx)
        agree[code] += 1
        if code == O.OK:
            assert pos_o == list(p)
            rows = np.nonzero(o)[0]
            exp = [-1] * n
            for r, i in enumerate(rows):
                exp[i] = r
            assert idx_o == exp
            assert ubs == list(range(0, n, n_ub))
    assert all(v > 10 for v in agree.values()), agree
