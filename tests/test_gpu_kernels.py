"""Parity of each CUDA kernel, called through the C ABI, against the plain
definition of its operation on the same inputs (float64 on the host).

GEMV/GEMM: y = x W^T (fp16 inputs widened exactly, fp32 accumulation on the
GPU).  Attention: the oracle's attention_one_seq on the fp16 cache values.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import llama as O  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import llama_decoder_forward_02_gb300 as L
    return L


def stream():
    return torch.cuda.current_stream().cuda_stream


def f16_rand(shape, scale=1.0, gen=None):
    """fp16 operands: the library computes with fp16 tensor-core inputs."""
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * scale).to(torch.float16)


@pytest.mark.parametrize("N,K,T,ksplit", [
    (64, 128, 1, 1), (256, 384, 3, 3), (192, 1024, 8, 4), (4096, 4096, 1, 0), (6144, 4096, 8, 0),
    (1024, 14336, 2, 0), (128, 256, 5, 2),
])
def test_gemv(lib, N, K, T, ksplit):
    g = torch.Generator().manual_seed(N * 7 + K + T)
    W, x = f16_rand((N, K), 0.02, g), f16_rand((T, K), 1.0, g)
    ref = (x.double() @ W.double().T).numpy()
    Wd, xd = W.cuda(), x.cuda()
    y = torch.full((T, N), float("nan"), device="cuda")
    scratch = torch.zeros(64 * N * 8 * 4 + N, dtype=torch.uint8, device="cuda")
    for rep in range(2):    # second call reuses the counters the first one reset
        rc = lib.llm_op_gemv(Wd.data_ptr(), xd.data_ptr(), y.data_ptr(), N, K, T, ksplit,
                             scratch.data_ptr(), scratch.numel(), stream())
        assert rc == 0
        torch.cuda.synchronize()
        got = y.cpu().double().numpy()
        err = np.abs(got - ref).max()
        assert err <= 1e-4 * max(1.0, np.abs(ref).max()), err


def oracle_attention(q, kc, vc, pos, seq, Hkv):
    """q [T][H][hd] float64; caches [n_seq][Hkv][n_ctx][hd] float64."""
    out = np.zeros_like(q)
    for t in range(q.shape[0]):
        cells = np.arange(pos[t] + 1)
        k = kc[seq[t]][:, cells, :].transpose(1, 0, 2)   # [S][Hkv][hd]
        v = vc[seq[t]][:, cells, :].transpose(1, 0, 2)
        out[t:t + 1] = O.attention_one_seq(q[t:t + 1], k, v, np.array([pos[t]]), cells, Hkv)
    return out


@pytest.mark.parametrize("hd,H,Hkv,n_ctx,pos,seq,n_split", [
    (128, 32, 8, 2304, [2047], [0], 38),
    (128, 8, 2, 300, [0, 299, 150], [0, 1, 1], 5),
    (64, 32, 8, 640, [511, 600, 3, 64, 65, 127, 128, 639], [0, 1, 2, 3, 0, 1, 2, 3], 4),
    (32, 4, 2, 64, [15], [0], 1),
    (32, 4, 4, 96, [95, 40], [0, 0], 3),
    (128, 8, 1, 200, [199], [0], 16),
])
def test_attn_decode(lib, hd, H, Hkv, n_ctx, pos, seq, n_split):
    T, n_seq = len(pos), max(seq) + 1
    g = torch.Generator().manual_seed(hd + H + n_ctx)
    q = torch.randn((T, H * hd), generator=g) * 1.5
    kc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    vc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    o = torch.zeros((T, H * hd), dtype=torch.float16, device="cuda")
    pos_d = torch.tensor(pos, dtype=torch.int32, device="cuda")
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    nbytes = lib.llm_op_attn_decode_scratch_bytes(T, H, hd, n_split)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    qd, kd, vd = q.cuda(), kc.cuda(), vc.cuda()
    ref = oracle_attention(q.double().numpy().reshape(T, H, hd), kc.double().numpy(), vc.double().numpy(),
                           pos, seq, Hkv).reshape(T, H * hd)
    for rep in range(2):
        rc = lib.llm_op_attn_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos_d.data_ptr(), seq_d.data_ptr(),
                                    o.data_ptr(), T, H, Hkv, hd, n_ctx, n_seq, n_split, scratch.data_ptr(), nbytes,
                                    stream())
        assert rc == 0
        torch.cuda.synchronize()
        err = np.abs(o.cpu().double().numpy() - ref).max()
        assert err <= 1e-2, err


@pytest.mark.parametrize("bad", ["pos_past_ctx", "pos_negative", "seq_past_cache"])
def test_attn_decode_reports_rows_outside_the_cache(lib, bad):
    """A row whose position or sequence lies outside the cache it was given is
    skipped (its output is zero), the call returns LLM_ERR_COMPUTE and says
    why; the other rows are computed as usual and the next call is clean."""
    hd, H, Hkv, n_ctx, n_seq, n_split = 64, 8, 2, 256, 2, 4
    pos, seq = [100, 50], [0, 1]
    if bad == "pos_past_ctx":
        pos[1] = n_ctx
    elif bad == "pos_negative":
        pos[1] = -1
    else:
        seq[1] = n_seq
    T = 2
    g = torch.Generator().manual_seed(7)
    q = torch.randn((T, H * hd), generator=g)
    kc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    vc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    qd, kd, vd = q.cuda(), kc.cuda(), vc.cuda()
    o = torch.full((T, H * hd), 7.0, dtype=torch.float16, device="cuda")
    nbytes = lib.llm_op_attn_decode_scratch_bytes(T, H, hd, n_split)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

    def call(p, sq):
        pd = torch.tensor(p, dtype=torch.int32, device="cuda")
        sd = torch.tensor(sq, dtype=torch.int32, device="cuda")
        return lib.llm_op_attn_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pd.data_ptr(), sd.data_ptr(),
                                      o.data_ptr(), T, H, Hkv, hd, n_ctx, n_seq, n_split, scratch.data_ptr(), nbytes,
                                      stream())
    assert call(pos, seq) == lib.LLM_ERR_COMPUTE
    assert b"outside" in lib.llm_last_error(None)
    ref = oracle_attention(q[:1].double().numpy().reshape(1, H, hd), kc.double().numpy(), vc.double().numpy(),
                           [100], [0], Hkv).reshape(1, H * hd)
    got = o.cpu().double().numpy()
    assert np.abs(got[0] - ref[0]).max() <= 1e-2
    assert np.all(got[1] == 0.0)
    assert call([100, 50], [0, 1]) == 0


def test_attn_ops_reject_shapes_they_do_not_cover(lib):
    """Group sizes other than 1, 2, 4, 8, more than 128 splits, and prefill
    rows outside the cache are refused with LLM_ERR_INVALID before any work."""
    x = torch.zeros(4096, dtype=torch.float32, device="cuda")
    p = x.data_ptr()
    nb = lib.llm_op_attn_decode_scratch_bytes(1, 12, 64, 4)
    assert lib.llm_op_attn_decode(p, p, p, p, p, p, 1, 12, 4, 64, 64, 1, 4, p, nb, stream()) == lib.LLM_ERR_INVALID
    assert b"1, 2, 4 or 8" in lib.llm_last_error(None)
    nb = lib.llm_op_attn_decode_scratch_bytes(1, 8, 64, 129)
    assert lib.llm_op_attn_decode(p, p, p, p, p, p, 1, 8, 2, 64, 64, 1, 129, p, nb, stream()) == lib.LLM_ERR_INVALID
    assert b"n_split" in lib.llm_last_error(None)
    assert lib.llm_op_attn_decode_noalloc(p, p, p, p, p, p, 1, 12, 4, 64, 64, 1, 4, stream()) == lib.LLM_ERR_INVALID
    assert lib.llm_op_attn_decode_noalloc(p, p, p, p, p, p, 1, 8, 2, 64, 64, 1, 129, stream()) == lib.LLM_ERR_INVALID
    pos_h = (ctypes.c_int32 * 2)(63, 64)
    seq_h = (ctypes.c_int32 * 2)(0, 0)
    assert lib.llm_op_attn_prefill(p, p, p, pos_h, seq_h, p, 2, 8, 2, 64, 64, 1, stream()) == lib.LLM_ERR_INVALID
    pos_h = (ctypes.c_int32 * 2)(0, 1)
    seq_h = (ctypes.c_int32 * 2)(1, 1)
    assert lib.llm_op_attn_prefill(p, p, p, pos_h, seq_h, p, 2, 8, 2, 64, 64, 1, stream()) == lib.LLM_ERR_INVALID


@pytest.mark.parametrize("hd,H,Hkv,n_ctx,rows", [
    (128, 8, 2, 256, [(0, 0, 100)]),                    # (seq, pos0, n) segments
    (64, 8, 8, 700, [(0, 512, 130), (1, 0, 37)]),
    (32, 4, 2, 128, [(0, 0, 16)]),
    (128, 32, 8, 1200, [(0, 1000, 64), (2, 5, 1), (1, 300, 70)]),
    # several 128-key tiles, query tiles that straddle key tiles, ragged tails
    (128, 32, 8, 2304, [(0, 1536, 512)]),
    (64, 32, 8, 1024, [(0, 0, 512)]),
    (128, 8, 2, 600, [(0, 77, 300), (1, 0, 129)]),
    (64, 8, 1, 400, [(1, 255, 1), (0, 0, 257)]),
    (128, 6, 2, 400, [(0, 10, 250), (1, 0, 3)]),        # odd GQA group: one CTA per head
    (128, 4, 4, 300, [(0, 0, 200)]),
])
def test_attn_prefill(lib, hd, H, Hkv, n_ctx, rows):
    """Prefill attention through the C ABI (the tcgen05 kernel for head_dim
    64 and 128, the mma.sync kernel for 32) against the oracle's attention on
    the fp16 cache values."""
    n_seq = max(r[0] for r in rows) + 1
    pos = [p0 + i for s, p0, n in rows for i in range(n)]
    seq = [s for s, p0, n in rows for i in range(n)]
    T = len(pos)
    g = torch.Generator().manual_seed(hd * 3 + T)
    q = f16_rand((T, H * hd), 1.5, g)
    kc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    vc = f16_rand((n_seq, Hkv, n_ctx, hd), 1.0, g)
    o = torch.zeros((T, H * hd), dtype=torch.float16, device="cuda")
    pos_h = (ctypes.c_int32 * T)(*pos)
    seq_h = (ctypes.c_int32 * T)(*seq)
    qd, kd, vd = q.cuda(), kc.cuda(), vc.cuda()
    rc = lib.llm_op_attn_prefill(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), pos_h, seq_h,
                                 o.data_ptr(), T, H, Hkv, hd, n_ctx, n_seq, stream())
    assert rc == 0
    torch.cuda.synchronize()
    ref = oracle_attention(q.double().numpy().reshape(T, H, hd), kc.double().numpy(), vc.double().numpy(),
                           pos, seq, Hkv).reshape(T, H * hd)
    err = np.abs(o.cpu().double().numpy() - ref).max()
    assert err <= 2e-2, err


@pytest.mark.parametrize("M,N,K,kernel", [
    (1, 128, 64, 1), (256, 256, 128, 3), (130, 384, 320, 2), (512, 1024, 4096, 1), (300, 512, 192, 3),
    (512, 6144, 4096, 0), (77, 128, 14336, 1), (600, 4096, 4096, 0), (257, 28672, 512, 0), (16, 256, 128, 3),
    (129, 256, 1024, 0), (512, 28672, 4096, 0),
    # persistent pairs (double-buffered accumulators, several tiles per cluster)
    (1, 128, 64, 4), (512, 28672, 4096, 4), (300, 512, 192, 6), (130, 384, 320, 5), (600, 4096, 4096, 4),
    (2000, 8192, 256, 6), (77, 128, 14336, 4),
    # stream-K (equal K-stage runs per pair, split tiles finished in K order)
    (512, 4096, 4096, 7), (512, 6144, 4096, 7), (512, 4096, 14336, 7), (512, 28672, 4096, 7), (1, 256, 64, 7),
    (300, 512, 192, 7), (77, 256, 14336, 7), (2000, 8192, 256, 7), (130, 768, 320, 7), (17, 32000, 2048, 7),
    (512, 2048, 8192, 7),
])
def test_gemm_tcgen05_cta_pairs(lib, M, N, K, kernel):
    """The CTA-pair tcgen05 GEMM (cta_group::2, 256-row tiles, each CTA staging
    half of the weight tile) against the plain definition, including ragged M
    where the odd CTA's rows lie past M."""
    g = torch.Generator().manual_seed(M * 5 + N + K)
    A, W = f16_rand((M, K), 1.0, g), f16_rand((N, K), 0.02, g)
    ref = (A.double() @ W.double().T).numpy()
    C = torch.full((M, N), float("nan"), device="cuda")
    Ad, Wd = A.cuda(), W.cuda()
    rc = lib.llm_op_gemm(Ad.data_ptr(), Wd.data_ptr(), C.data_ptr(), M, N, K, kernel, stream())
    assert rc == 0
    torch.cuda.synchronize()
    got = C.cpu().double().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= 1e-4 * max(1.0, np.abs(ref).max()), err


# ---------------------------------------------------------------- Q8_0 weight rows

def q8_0_bytes(q, d):
    """The library's Q8_0 row layout of the oracle's encoding: each row's K
    codes, then its K/32 fp16 scales (little-endian)."""
    n = q.shape[0]
    return np.concatenate([q.view(np.uint8), d.astype(np.float16).view(np.uint8).reshape(n, -1)], axis=1)


def q8_test_matrix(N, K, seed, large=True):
    """fp16 weights N(0, 0.02) with hand-made blocks: exact ties of w / d (d =
    2^-7), a zero block, a block of fp16 subnormals and (large) a block near
    the fp16 range."""
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn((N, K), generator=g) * 0.02).to(torch.float16).float().numpy()
    w[0, :32] = np.array([127, 2.5, 3.5, -1.5, 0.5, -0.5, 126.5, -127] + [0] * 24) * 2.0 ** -7
    w[0, 32:64] = 0.0
    w[1, 64:96] = np.linspace(-1, 1, 32) * 2.0 ** -19
    if large:
        w[2, 96:128] = np.linspace(-60000, 50000, 32)
    return torch.from_numpy(w).to(torch.float16)


@pytest.mark.parametrize("N,K", [(3, 256), (300, 4096), (64, 14336), (1000, 2048)])
def test_quantize_q8_0_bit_exact(lib, N, K):
    W = q8_test_matrix(N, K, N + K)
    q, d = O.quantize_q8_0(W.float().numpy())
    want = q8_0_bytes(q, d)
    Wd = W.cuda()
    out = torch.zeros((N, K + K // 16), dtype=torch.uint8, device="cuda")
    assert lib.llm_op_quantize_q8_0(Wd.data_ptr(), N, K, out.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)
    assert torch.equal(Wd.cpu(), W)            # the matrix is only read
    assert lib.llm_op_quantize_q8_0(Wd.data_ptr(), N, 384, out.data_ptr(), stream()) == lib.LLM_ERR_INVALID


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 14336), (1000, 2048), (461, 256), (3000, 8192)])
def test_gemv_q8_0(lib, N, K):
    """The streamed one-row GEMV on Q8_0 rows written from the oracle's encoding
    (ragged row counts over the SMs; 1..8 rows a stage) against the float64
    product with the weights the blocks stand for."""
    W = q8_test_matrix(N, K, 3 * N + K, large=False)
    q, d = O.quantize_q8_0(W.float().numpy())
    g = torch.Generator().manual_seed(N + 5 * K)
    x = f16_rand((K,), 1.0, g)
    ref = O.dequantize_q8_0(q, d) @ x.double().numpy()
    Wq = torch.from_numpy(q8_0_bytes(q, d)).cuda()
    xd = x.cuda()
    y = torch.full((N,), float("nan"), device="cuda")
    assert lib.llm_op_gemv_q8_0(Wq.data_ptr(), xd.data_ptr(), y.data_ptr(), N, K, stream()) == 0
    torch.cuda.synchronize()
    got = y.cpu().double().numpy()
    err = np.abs(got - ref).max()
    assert err <= 1e-4 * max(1.0, np.abs(ref).max()), err
    assert lib.llm_op_gemv_q8_0(Wq.data_ptr(), xd.data_ptr(), y.data_ptr(), N, K + 128, stream()) == lib.LLM_ERR_INVALID


# ---------------------------------------------------------------- bounded waits

def test_bounded_wait_times_out_and_reports(lib):
    """The bounded mbarrier wait of the pipelined kernels: a phase that completes
    leaves the error word alone; one that never does (nothing arrives) gives up
    after the given polls, sets the time-out bit (4) and returns, and the device
    stays usable (a GEMV right after is exact)."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.llm_op_wait_check(1, 1000, err.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    assert err.item() == 0
    assert lib.llm_op_wait_check(0, 1000, err.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    assert err.item() == 4
    g = torch.Generator().manual_seed(11)
    W, x = f16_rand((256, 512), 0.02, g), f16_rand((1, 512), 1.0, g)
    ref = (x.double() @ W.double().T).numpy()
    Wd, xd = W.cuda(), x.cuda()
    y = torch.full((1, 256), float("nan"), device="cuda")
    scratch = torch.zeros(64 * 256 * 8 * 4 + 256, dtype=torch.uint8, device="cuda")
    assert lib.llm_op_gemv(Wd.data_ptr(), xd.data_ptr(), y.data_ptr(), 256, 512, 1, 0,
                           scratch.data_ptr(), scratch.numel(), stream()) == 0
    torch.cuda.synchronize()
    assert np.abs(y.cpu().double().numpy() - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())
