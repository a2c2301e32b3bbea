"""The zero-allocation decode attention entry point.

llm_op_attn_decode_noalloc serves callers that cannot call cudaMalloc (hosts
whose caching allocator owns all device memory, fixed-footprint serving
processes, loops that must never enter the driver's allocator): its split
scratch is a static device array inside the library instead of memory the
caller passes.  This test calls it through the C ABI and checks its output
against the allocating entry point, llm_op_attn_decode, on two calls in a
row with different inputs (the array keeps the previous call's contents),
and checks that a request larger than the array is refused.  The file is
named to be collected last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(T, H, Hkv, hd, n_ctx, pos, seq, seed):
    g = torch.Generator().manual_seed(seed)
    n_seq = max(seq) + 1
    q = (torch.randn((T, H * hd), generator=g) * 1.5).cuda()
    kc = torch.randn((n_seq, Hkv, n_ctx, hd), generator=g).to(torch.float16).cuda()
    vc = torch.randn((n_seq, Hkv, n_ctx, hd), generator=g).to(torch.float16).cuda()
    pos_d = torch.tensor(pos, dtype=torch.int32, device="cuda")
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    return q, kc, vc, pos_d, seq_d


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    import llama_decoder_forward_02_gb300 as L
    st = torch.cuda.current_stream().cuda_stream
    T, H, Hkv, hd, n_ctx, n_split = 3, 32, 8, 128, 1000, 6
    for call, (pos, seq) in enumerate([([999, 10, 500], [0, 1, 1]), ([3, 700, 64], [1, 0, 0])]):
        q, kc, vc, pos_d, seq_d = _case(T, H, Hkv, hd, n_ctx, pos, seq, seed=11 + call)
        ref = torch.zeros((T, H * hd), dtype=torch.float16, device="cuda")
        nbytes = L.llm_op_attn_decode_scratch_bytes(T, H, hd, n_split)
        scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        assert L.llm_op_attn_decode(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pos_d.data_ptr(), seq_d.data_ptr(),
                                    ref.data_ptr(), T, H, Hkv, hd, n_ctx, n_split, scratch.data_ptr(), nbytes,
                                    st) == 0
        got = torch.full((T, H * hd), float("nan"), dtype=torch.float16, device="cuda")
        assert L.llm_op_attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pos_d.data_ptr(),
                                            seq_d.data_ptr(), got.data_ptr(), T, H, Hkv, hd, n_ctx, n_split,
                                            st) == 0
        torch.cuda.synchronize()
        err = (got.double() - ref.double()).abs().max().item()
        assert np.isfinite(err) and err <= 1e-2, (call, err)


def test_noalloc_rejects_requests_beyond_its_array():
    import llama_decoder_forward_02_gb300 as L
    st = torch.cuda.current_stream().cuda_stream
    T, H, Hkv, hd, n_ctx = 8, 64, 8, 128, 4096
    q, kc, vc, pos_d, seq_d = _case(1, 8, 8, 32, 8, [0], [0], seed=3)
    # 8 * 64 * 64 * 130 floats > 1048576: refused before anything is launched
    rc = L.llm_op_attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pos_d.data_ptr(),
                                      seq_d.data_ptr(), q.data_ptr(), T, H, Hkv, hd, n_ctx, 64, st)
    assert rc == L.LLM_ERR_INVALID
    assert b"static scratch" in L.llm_last_error(None)
