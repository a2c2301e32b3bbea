// Internal interface between the host orchestrator and the sm_103a kernels.
// Host-compilable (no device code); every launcher returns a cudaError_t.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace llm {

typedef __nv_bfloat16 bf16;   // type of the weights handed to llm_model_create
typedef __half f16;           // type of the weights, activations and KV cache inside

// How a kernel is put on the stream: programmatic dependent launch on/off,
// and a host counter of launches (for reporting).
struct Launch {
    cudaStream_t stream;
    bool pdl;
    int64_t *count;
    bool cooperative = false;    // all CTAs co-resident (CTAs that wait on one another)
};

// Interleave granularity of the fused gate/up weight: rows [16b, 16b+8) of
// the packed matrix are gate rows [8b, 8b+8), rows [16b+8, 16b+16) the up
// rows with the same indices.
constexpr int GU_GROUP = 8;

// Per-row layout of the KV cache of one layer, shared by all kernels that
// read or write it: element (seq, kv_head, pos, d) lives at
//   base + seq * seq_stride + (kv_head * n_ctx + pos) * head_dim + d.
struct KvView {
    f16 *k, *v;               // this layer's base (seq 0, head 0, pos 0), fp16 cache
    long long seq_stride;      // elements between sequences
    int n_ctx, n_seq, head_dim, n_kv_head;
    // FP8 E4M3 cache (one byte an element, same element offsets) when not null;
    // k and v are then unused
    uint8_t *k8 = nullptr, *v8 = nullptr;
};

// ------------------------------------------------------------------ decode GEMV
enum GemvPro { PRO_BF16 = 0, PRO_NORM = 1 };
enum GemvEpi { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3 };

struct GemvArgs {
    const f16 *W;             // [N][K]
    int N, K, T, ksplit;
    // prologue PRO_BF16: x f16 [T][ldx]
    const f16 *x; int ldx;
    // prologue PRO_NORM: x = f16(h[row] * r[row] * gain); r from the
    // per-64-column partial sums of squares ss_part[(K/64)][8] when given,
    // else computed from h.
    const float *h; int ldh; const int *row_map;
    const float *ss_part; const float *gain; float eps;
    // split-K scratch: part fp32 [ksplit][N][8], counters uint32 [N/64]
    float *part; unsigned *counters;
    // EPI_STORE: out[t*ldo + n]
    float *out; int ldo;
    // EPI_RESID: hres[t*ldh_res + n] += y; ss_out[(N/64)][8] partial sums
    float *hres; int ldh_res; float *ss_out;
    // EPI_QKV: rows [0,n_q) -> RoPE -> q_out fp32 [T][n_q]; [n_q, n_q+n_kv) -> RoPE
    // -> K cache; [n_q+n_kv, n_q+2n_kv) -> V cache.  rope: float2 [n_ctx][hd/2].
    int n_q, n_kv; const float2 *rope; float *q_out; KvView kv;
    const int *pos, *seq;
    // EPI_SWIGLU: u_out f16 [T][ldu]
    f16 *u_out; int ldu;
    uint32_t *err;
    // streamed GEMV only: once its own stages are issued, CTA b prefetches into
    // L2 the first pf_bytes of the rows CTA b of the next streamed GEMV will
    // read (weights pf_W [pf_N][pf_K], row groups of pf_unit); pf_W may be null
    const f16 *pf_W; int pf_N, pf_K, pf_unit; int pf_bytes;
    // ... and a second such target after it (the GEMV after next: the QKV GEMV
    // warms the gate/up weights while decode attention leaves HBM idle)
    const f16 *pf2_W; const uint8_t *pf2_W8; int pf2_N, pf2_K, pf2_unit; int pf2_bytes;
    // streamed GEMV only, handing the next RMSNorm its input:
    // EPI_RESID with xg_out: also writes xg_out[n] = f16(h_new[n] * gain_next[n])
    // and its CTA's sum of h_new^2 over its rows to ss_cta[blockIdx.x];
    // PRO_NORM with xg: x = xg (fp16 [K]) and sum(h^2) = the n_ss_in partials
    // ss_in summed in order (h, gain and ss_part are then not read)
    const f16 *xg; const float *ss_in; int n_ss_in;
    const float *gain_next; f16 *xg_out; float *ss_cta;
    // streamed GEMV only: when W8 is set the weights are the Q8_0 rows W8
    // (K codes, then K/32 fp16 scales, K + K/16 bytes a row) and W is not
    // read; pf_W8 likewise replaces pf_W for the prefetch
    const uint8_t *W8, *pf_W8;
};
cudaError_t launch_gemv(int pro, int epi, const GemvArgs &a, const Launch &l);
// One-row GEMV streamed through shared memory, one CTA per SM (T == 1 only;
// same arguments; ss_part / ss_out / part / counters are not used).
bool gemv_stream_ok(int epi, int N, int K, int num_sms, int smem_kb = 0, bool q8 = false);
int gemv_stream_unit(int epi);      // rows kept together in one CTA
// smem_kb: shared-memory cap of the CTA (0 = as much as helps, ~200 KB);
// stage_kb: largest ring stage when warps take several rows each (0 = the
// default: one row a warp for fp16 rows, up to 96 KB stages for Q8_0 rows)
cudaError_t launch_gemv_stream(int pro, int epi, const GemvArgs &a, int num_sms, int smem_kb, const Launch &l,
                               int stage_kb = 0);
// Host-side choice of the K split for an N x K GEMV over T rows.
int gemv_pick_split(int N, int K, int T, int num_sms);
size_t gemv_smem_bytes(int K, int ksplit, int T);

// ------------------------------------------------------------------ decode attention
struct AttnDecodeArgs {
    const float *q;            // [T][H*hd] fp32, after RoPE
    KvView kv;
    const int *pos, *seq;      // [T]
    f16 *o;                   // [T][H*hd]
    int T, H, n_split;
    float *part;               // [T][H][n_split][hd+2]
    unsigned *counters;        // [T][Hkv]
    uint32_t *err;
    int window = 0;            // sliding window: keys with pos - W < key <= pos (0 = all)
};
// Most sequence splits per (row, kv head) the decode-attention kernel takes.
constexpr int ATTN_DECODE_MAX_SPLIT = 128;
cudaError_t launch_attn_decode(const AttnDecodeArgs &a, const Launch &l);
size_t attn_decode_scratch_floats(int T, int H, int hd, int n_split);

// ------------------------------------------------------------------ prefill attention
// One tile = consecutive rows of one sequence with consecutive positions (up
// to 64 rows for the mma.sync kernel, 128 for the tcgen05 kernel); keys below
// kv_ready were in the cache before this ubatch (the first position the
// ubatch writes for that sequence).
struct AttnTile { int row0, n_rows, seq, pos0, kv_ready; };
struct AttnPrefillArgs {
    const f16 *q;             // [T][H*hd] f16, after RoPE
    KvView kv;
    const AttnTile *tiles; int n_tiles;
    f16 *o;                   // [T][H*hd]
    int H;
    uint32_t *err;
    int window = 0;           // sliding window: keys with pos - W < key <= pos (0 = all)
};
cudaError_t launch_attn_prefill(const AttnPrefillArgs &a, const Launch &l);
// The tcgen05 prefill attention (128 query rows of one sequence and one head
// a CTA, S = Q K^T and O += P V on the tensor cores, accumulators in TMEM).
// Q arrives by TMA from q [rows][H*hd] (map mQ, boxes of 128 rows x 64), K and
// V from the caches viewed as [n_seq*n_layer*Hkv*n_ctx][hd] (maps mK, mV, same
// boxes); fp16 cache, head_dim 64 or 128.
struct AttnPrefillTcArgs {
    const AttnTile *tiles; int n_tiles;     // tiles of at most 128 rows
    int H, Hkv, head_dim, n_layer, layer, n_ctx, n_seq;
    f16 *o; int ldo;                        // o [rows][ldo], head h at column h*hd
    uint32_t *err;
    int window;                             // sliding window (0 = all earlier positions)
};
struct TmaMap;
bool attn_prefill_tc_ok(int head_dim, bool fp8_cache);
cudaError_t launch_attn_prefill_tc(const AttnPrefillTcArgs &a, const TmaMap &mQ, const TmaMap &mK, const TmaMap &mV,
                                   const Launch &l);
// The same on CTA pairs (cta_group::2, the two query heads of a GQA group on
// two SMs, each staging half of every K/V tile): head_dim 128, H / Hkv even;
// mK64 reads the K cache in boxes of 64 rows x 64 columns.
bool attn_prefill_pair_ok(int head_dim, int H, int Hkv, bool fp8_cache);
cudaError_t launch_attn_prefill_pair(const AttnPrefillTcArgs &a, const TmaMap &mQ, const TmaMap &mK64,
                                     const TmaMap &mV, const Launch &l);
// Context shift of sequence seq (all layers; kv0 is layer 0's view): drop
// positions [p0, p0 + n), move rows [p0 + n, end) down by n with keys
// re-rotated by RoPE(-n) (rope: float2 [n_ctx][hd/2] cos, sin).
cudaError_t launch_kv_shift(const KvView &kv0, int n_layer, int seq, int p0, int n, int end, const float2 *rope,
                            const Launch &l);

// ------------------------------------------------------------------ prefill GEMM
struct GemmArgs {
    const f16 *A;             // [M][K]
    const f16 *W;             // [N][K]
    int M, N, K;
    float *C; int ldc;                          // EPI_STORE
    float *hres; int ldh;                       // EPI_RESID
    int n_q, n_kv; const float2 *rope; f16 *q_out; KvView kv;   // EPI_QKV (q_out [M][n_q])
    // EPI_QKV on the tensor-core GEMMs: the RoPE table position-minor,
    // rope_t[i * rope_n + pos] = rope[pos * (head_dim / 2) + i], so that a
    // warp's rows (consecutive positions) read one pair index in one request;
    // null = read rope
    const float2 *rope_t; int rope_n;
    const int *pos, *seq;
    f16 *u_out; int ldu;                       // EPI_SWIGLU
    uint32_t *err;
    // RMSNorm fused across GEMMs (prefill).  Producer (EPI_RESID with x_next):
    // also writes x_next[row][col] = f16(h_new * gain_next[col]) and, per 32
    // columns, the partial sum of h_new^2 to ss_next[row * (N / 32) + col / 32].
    // Consumer (row_ss set): every accumulator row is first multiplied by
    // 1 / sqrt(sum_g row_ss[row * n_ss + g] / (32 * n_ss) + eps), the row's
    // RMSNorm scale, its gain having been applied to A already.
    const float *gain_next; f16 *x_next; float *ss_next;
    const float *row_ss; int n_ss; float eps;
    // EPI_RESID on one-tile CTA pairs: 1 = h is read into shared memory by TMA
    // while the last MMAs run and h, x_next are written back by TMA stores
    // (the maps of hres and x_next are handed to the launcher)
    int tma_epi;
    // EPI_RESID through shared memory on one-tile 256-wide pairs, K split in
    // two: the pairs with blockIdx.z = z compute half z of the K stages, park
    // the other half's columns of their fp32 accumulator in part (slot
    // 2 * cta + z, column-major [BN / 2][128]), release flags[2 * cta + z] =
    // epoch, wait (bounded) for the partner's flag, add its parked half of
    // their own columns and apply the epilogue to columns [z BN/2, (z+1) BN/2).
    // All CTAs of both halves must be resident at once (the caller checks the
    // pair count).
    int split_k; float *part; unsigned *flags; unsigned epoch;
};

// A TMA descriptor (CUtensorMap: 128 bytes, 64-byte aligned) of one fp16
// operand [rows][cols], boxes of box_rows x 64 with 128-byte swizzle.
struct alignas(64) TmaMap { uint64_t opaque[16]; };
bool make_operand_map(TmaMap *m, const f16 *ptr, int rows, int cols, int box_rows);
// The tcgen05/TMEM GEMM on CTA pairs (cta_group::2): 256 x bn tiles, bn in
// {128, 192, 256}; mA boxes 128 x 64 over A [>=M][K], mB boxes of bn / 2 x 64
// over W [N][K].
int gemm_pair_pick_bn(int M, int N, int max_clusters);
int gemm_pair_max_clusters();
cudaError_t launch_gemm_pair(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, int bn,
                             const Launch &l, const TmaMap *mH = nullptr, const TmaMap *mX = nullptr);
// fp32 [rows][cols] in boxes of 128 rows x 32 columns with 128-byte swizzle
// (the residual tiles of the pair GEMM's TMA epilogue)
bool make_f32_tile_map(TmaMap *m, const float *ptr, int rows, int cols);
cudaError_t init_gemm_pair_attributes();
// Persistent variant: one cluster per resident pair slot loops over the tiles,
// the accumulator double-buffered in tensor memory so each tile's epilogue
// overlaps the next tile's MMAs.  Same arguments.
cudaError_t launch_gemm_pair_persist(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, int bn,
                                     const Launch &l);
// Stream-K variant (256-wide tiles, N % 256 == 0): every resident pair takes
// an equal run of 128-deep K stages across the tiles; a tile split between
// pairs is finished by the pair holding its first stages, which adds the
// others' parked partials in K order.  ws: fp32 [gemm_pair_sk_ws_floats]
// (contents need not be initialised); flags: uint32 [2 * max clusters], zero
// before the first launch and written with `epoch`, which must differ from the
// previous launch's that used the same flags (and be nonzero).
int gemm_pair_sk_clusters(int M, int N, int K);
size_t gemm_pair_sk_ws_floats(int max_clusters);
cudaError_t launch_gemm_pair_sk(int epi, const GemmArgs &a, const TmaMap &mA, const TmaMap &mB, float *ws,
                                unsigned *flags, unsigned epoch, const Launch &l);

// ------------------------------------------------------------------ sampling chain
struct SampleParams {
    float temperature;      // <= 0: greedy argmax
    int top_k;              // 1..1024 (and <= V) when temperature > 0
    float top_p;            // >= 1: off
    float min_p;            // <= 0: off
    float repeat_penalty;   // 1: off
    int penalty_last_n;     // history entries considered
};
// out[r] = the token the chain picks from logits row r (fp32 [n_rows][V]) with
// the uniform u[r]; history [n_hist] (device) are the earlier tokens.
// Largest vocabulary the sampling chain takes (a cluster of 8 CTAs holds a row
// in shared memory, 32768 keys each).
constexpr int SAMPLE_MAX_VOCAB = 262144;
cudaError_t launch_sample(const float *logits, int n_rows, int V, const SampleParams &p, const float *u,
                          const int *history, int n_hist, int *out, const Launch &l);

// ------------------------------------------------------------------ small kernels
// h[t][:] = float(E[tok[t]][:]); for T <= 8 also the per-64-column partial
// sums of squares ss_part[(d/64)][8].  With gain (prefill): also
// x[t][:] = f16(h[t][:] * gain) and the per-32-column partial sums of squares
// ss32[t][d/32] that the first QKV GEMM's fused RMSNorm reads.
cudaError_t launch_embed(const f16 *E, const int *tok, int T, int d, int n_vocab, float *h,
                         float *ss_part, uint32_t *err, const Launch &l, const float *gain = nullptr,
                         f16 *x = nullptr, float *ss32 = nullptr);
// dst[r][:] = src[rows[r]][:] (fp32 rows of length d); ss rows likewise when
// given (decode layout [(d/64)][8]); with x_src also the fp16 rows x_dst[r] =
// x_src[rows[r]] and the per-32-column partials ss32_dst[r] = ss32_src[rows[r]].
cudaError_t launch_gather_rows(const float *src, const int *rows, int n_rows, int d, float *dst,
                               const float *ss_src, float *ss_dst, const Launch &l, const f16 *x_src = nullptr,
                               f16 *x_dst = nullptr, const float *ss32_src = nullptr, float *ss32_dst = nullptr);
// out[r] = argmax_v logits[r][v], lowest index on ties.
cudaError_t launch_argmax(const float *logits, int n_rows, int n_vocab, int *out,
                          const Launch &l);
// Greedy feedback for on-device generation: tok = argmax(logits row);
// tokens_out[*step] = tok if *step < *n_steps; next_tok[0] = tok;
// pos[0] += advance; (*step)++.
cudaError_t launch_argmax_feed(const float *logits, int n_vocab, int *tokens_out, int *step,
                               const int *n_steps, int *next_tok, int *pos, int advance,
                               const Launch &l);
// Model set-up helpers (not on the hot path).
cudaError_t launch_widen_bf16(const bf16 *src, float *dst, int n, cudaStream_t st);
// dst[r*dst_ld + c] = fp16(src[r*src_ld + c]) for r < rows, c < cols; values
// beyond the fp16 range raise ERRF_BAD_INDEX in *err.
cudaError_t launch_convert_rows(const bf16 *src, int src_ld, f16 *dst, int dst_ld, int rows, int cols,
                                uint32_t *err, cudaStream_t st);
cudaError_t launch_repack_gate_up(const bf16 *gate, const bf16 *up, int F, int F_pad, int d, f16 *dst,
                                  uint32_t *err, cudaStream_t st);
// Copy the hidden state rows into the diagnostic buffer.
cudaError_t launch_copy_f32(const float *src, float *dst, size_t n, const Launch &l);
// Q8_0 encoding of the fp16 matrix w [N][K] (K % 32 == 0): into q8 (rows of
// q8_0_row_bytes(K) bytes, K % 256 == 0) when not null, and with write_back
// w itself replaced by the weights the blocks stand for, f16(q * d).
size_t q8_0_row_bytes(int K);
// The bounded shared-memory mbarrier wait on its own (one thread): arrive
// (when asked) on a fresh one-arrival barrier, then poll its phase at most
// `polls` times; a wait that never completes raises ERRF_WAIT_TIMEOUT in *err.
cudaError_t launch_wait_check(int arrive, uint32_t polls, uint32_t *err, cudaStream_t st);
cudaError_t launch_quantize_q8_0(f16 *w, int N, int K, uint8_t *q8, bool write_back, cudaStream_t st);

}  // namespace llm
