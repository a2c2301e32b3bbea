"""The zero-allocation decode attention entry point.

llm_op_attn_decode_noalloc serves callers that cannot call cudaMalloc (hosts
whose caching allocator owns all device memory, fixed-footprint serving
processes, loops that must never enter the driver's allocator): its split
scratch is a static device array inside the library instead of memory the
caller passes.  These tests call it through the C ABI and check it

* against the oracle's attention (oracle.llama.attention_one_seq on the fp16
  cache values) and bit for bit against the allocating entry point,
  llm_op_attn_decode, which runs the same kernel with the same splits;
* on calls in a row whose shapes differ, a larger request before a smaller
  one, since the array keeps whatever the previous call left;
* on a row outside the cache, which must come back as LLM_ERR_COMPUTE (the
  array's own error word) and leave the next call clean;
* on a request larger than the array, which is refused before any work.

The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from oracle import llama as O

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _case(T, H, Hkv, hd, n_ctx, n_seq, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((T, H * hd), generator=g) * 1.5
    kc = torch.randn((n_seq, Hkv, n_ctx, hd), generator=g).to(torch.float16)
    vc = torch.randn((n_seq, Hkv, n_ctx, hd), generator=g).to(torch.float16)
    return q, kc, vc


def _oracle(q, kc, vc, pos, seq, Hkv):
    """Each row against its sequence's cached keys 0..pos (oracle attention on
    the fp16 cache values, float64)."""
    T = q.shape[0]
    hd = kc.shape[-1]
    H = q.shape[1] // hd
    out = np.zeros((T, H * hd))
    for t in range(T):
        k = kc[seq[t], :, :pos[t] + 1].double().numpy().transpose(1, 0, 2)     # [S][Hkv][hd]
        v = vc[seq[t], :, :pos[t] + 1].double().numpy().transpose(1, 0, 2)
        o = O.attention_one_seq(q[t].double().numpy().reshape(1, H, hd), k, v, [pos[t]], np.arange(pos[t] + 1), Hkv)
        out[t] = o.reshape(H * hd)
    return out


def _run(L, T, H, Hkv, hd, n_ctx, n_seq, n_split, pos, seq, seed):
    q, kc, vc = _case(T, H, Hkv, hd, n_ctx, n_seq, seed)
    qd, kd, vd = q.cuda(), kc.cuda(), vc.cuda()
    pos_d = torch.tensor(pos, dtype=torch.int32, device="cuda")
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    ref = torch.zeros((T, H * hd), dtype=torch.float16, device="cuda")
    nbytes = L.llm_op_attn_decode_scratch_bytes(T, H, hd, n_split)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    rc_ref = L.llm_op_attn_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos_d.data_ptr(), seq_d.data_ptr(),
                                  ref.data_ptr(), T, H, Hkv, hd, n_ctx, n_seq, n_split, scratch.data_ptr(), nbytes,
                                  _stream())
    got = torch.full((T, H * hd), float("nan"), dtype=torch.float16, device="cuda")
    rc = L.llm_op_attn_decode_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos_d.data_ptr(),
                                      seq_d.data_ptr(), got.data_ptr(), T, H, Hkv, hd, n_ctx, n_seq, n_split,
                                      _stream())
    torch.cuda.synchronize()
    return rc, rc_ref, got, ref, (q, kc, vc)


def test_noalloc_matches_oracle_and_allocating_entry_point_on_calls_in_a_row():
    import llama_decoder_forward_02_gb300 as L
    calls = [
        # (T, H, Hkv, hd, n_ctx, n_split, pos, seq): the largest request first, so
        # later, smaller calls find its partials and counters in the array
        (8, 32, 8, 128, 1000, 16, [999, 10, 500, 0, 63, 64, 700, 998], [0, 1, 1, 0, 1, 0, 0, 1]),
        (3, 32, 8, 128, 1000, 6, [999, 10, 500], [0, 1, 1]),
        (2, 8, 2, 64, 300, 3, [3, 299], [1, 0]),
        (3, 32, 8, 128, 1000, 6, [3, 700, 64], [1, 0, 0]),
    ]
    for i, (T, H, Hkv, hd, n_ctx, n_split, pos, seq) in enumerate(calls):
        n_seq = max(seq) + 1
        rc, rc_ref, got, ref, (q, kc, vc) = _run(L, T, H, Hkv, hd, n_ctx, n_seq, n_split, pos, seq, seed=11 + i)
        assert rc == 0 and rc_ref == 0, (i, rc, rc_ref, L.llm_last_error(None))
        # same kernel, same splits, merged in split order: identical bits
        assert torch.equal(got, ref), (i, (got.double() - ref.double()).abs().max().item())
        err = np.abs(got.cpu().double().numpy() - _oracle(q, kc, vc, pos, seq, Hkv)).max()
        assert err <= 1e-2, (i, err)


def test_noalloc_reports_a_row_outside_the_cache_then_runs_clean():
    import llama_decoder_forward_02_gb300 as L
    T, H, Hkv, hd, n_ctx, n_seq, n_split = 2, 8, 2, 64, 256, 2, 4
    rc, _, got, ref, _ = _run(L, T, H, Hkv, hd, n_ctx, n_seq, n_split, [100, n_ctx], [0, 1], seed=5)
    assert rc == L.LLM_ERR_COMPUTE
    assert b"outside" in L.llm_last_error(None)
    assert torch.all(got[1] == 0) and torch.equal(got[0], ref[0])
    rc, _, got, ref, _ = _run(L, T, H, Hkv, hd, n_ctx, n_seq, n_split, [100, 50], [0, 1], seed=6)
    assert rc == 0 and torch.equal(got, ref)


def test_noalloc_rejects_requests_beyond_its_array():
    import llama_decoder_forward_02_gb300 as L
    q = torch.zeros(64, device="cuda")
    p = q.data_ptr()
    # 8 * 64 * 64 * 130 floats > 1048576: refused before anything is launched
    rc = L.llm_op_attn_decode_noalloc(p, p, p, p, p, p, 8, 64, 8, 128, 4096, 1, 64, _stream())
    assert rc == L.LLM_ERR_INVALID
    assert b"static scratch" in L.llm_last_error(None)
