// C ABI of the Llama forward pass: model set-up, context (KV cache,
// workspaces, decode graphs), and the ubatch orchestrator.
//
// The forward pass follows "Inside the inference engine: model architectures
// and forward pass", section "Detailed explanation: Llama's forward pass in
// Go" (Model.Forward: embed, layers with the output rows kept before the last
// MLP, OutputNorm, Output), and the batch handling of "LLama.cpp — how it
// works", "Steps 11–12" (llama_decode: fill the batch, loop over ubatches,
// keep the flagged rows' logits) and "Steps 14–15" (llama_get_logits_ith).
// Graph reuse for same-shaped decode steps (the "graph is built once at the
// first one-token decode and reused" passage of Step 13) becomes CUDA-graph
// capture of one decode step.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "sched.h"
#include "../../include/llm.h"

namespace llm {
void set_global_error(const char *msg);
cudaError_t init_gemv_attributes();
cudaError_t init_attn_prefill_attributes();
cudaError_t init_attn_decode_attributes();
cudaError_t init_attn_prefill_tc_attributes();
cudaError_t init_sample_attributes();
cudaError_t init_gemv_stream_attributes();

// Kernel attributes (dynamic shared-memory limits, carveouts) take effect on
// the device that is current when they are set, so they are set once per
// device, the first time an entry point runs with that device current.
cudaError_t init_kernel_attributes() {
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static bool done[MAX_DEV] = {false};
    static cudaError_t status[MAX_DEV];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= MAX_DEV) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = init_gemv_attributes();
        if (!e) e = init_attn_prefill_attributes();
        if (!e) e = init_gemm_pair_attributes();
        if (!e) e = init_attn_decode_attributes();
        if (!e) e = init_attn_prefill_tc_attributes();
        if (!e) e = init_sample_attributes();
        if (!e) e = init_gemv_stream_attributes();
        status[dev] = e;
        done[dev] = true;
    }
    return status[dev];
}
}  // namespace llm

using namespace llm;

static thread_local std::string g_create_error = "no error";

void llm::set_global_error(const char *msg) { g_create_error = msg; }

// A weight matrix as the tcgen05 GEMM reads it: TMA map + tile width.
struct WMap {
    TmaMap map128, map256;       // boxes of 128 or 256 rows (one-CTA tile width; pair width 256)
    TmaMap map64, map96;         // boxes of 64 or 96 rows (half of a 128- or 192-wide pair tile)
    bool has256 = false, has96 = false;
};

struct LayerW {
    f16 *wqkv, *wo, *wgu, *wdown;
    float *attn_norm, *ffn_norm;
    WMap mqkv, mo, mgu, mdown;
    // Q8_0 rows of the same matrices (llm_model_quantize), or null
    const uint8_t *q_qkv = nullptr, *q_o = nullptr, *q_gu = nullptr, *q_down = nullptr;
};

struct llm_model {
    llm_hparams hp;
    int d, H, Hkv, hd, n_q, n_kv, n_qkv, F, F_pad, V, L;
    f16 *wbuf = nullptr;
    float *fbuf = nullptr;
    f16 *token_embd = nullptr, *output = nullptr;
    float *output_norm = nullptr;
    WMap mout;
    std::vector<LayerW> layers;
    int wtype = 0;                     // LLM_WTYPE_* of llm_model_quantize (0: as created)
    uint8_t *qbuf = nullptr;           // Q8_0 rows of every decode matrix
    const uint8_t *q_out = nullptr;    // Q8_0 rows of the output projection
    int num_sms = 0;
    int device = 0;
    int n_contexts = 0;
};

// Kernel classes for the optional per-kernel event timing.
enum KId {
    K_EMBED, K_GATHER, K_GEMV_QKV, K_ATTN_DECODE, K_GEMV_O, K_GEMV_GATEUP, K_GEMV_DOWN,
    K_GEMV_LMHEAD, K_GEMM_QKV, K_ATTN_PREFILL, K_GEMM_O, K_GEMM_GATEUP, K_GEMM_DOWN, K_GEMM_LMHEAD,
    K_ARGMAX, K_COPY, K_COUNT
};
static const char *const KNAME[K_COUNT] = {
    "embed", "gather_rows", "gemv_qkv_rope_kv", "attn_decode", "gemv_o_resid", "gemv_gateup_swiglu",
    "gemv_down_resid", "gemv_lm_head", "gemm_qkv_rope_kv", "attn_prefill", "gemm_o_resid", "gemm_gateup_swiglu",
    "gemm_down_resid", "gemm_lm_head", "argmax", "copy"};

struct KtRec { int id; cudaEvent_t a, b; };

struct llm_ctx {
    llm_model *m = nullptr;
    cudaStream_t stream = nullptr;
    bool own_stream = false;      // created here because the caller passed the legacy stream
    int n_ctx = 0, n_seq_max = 0, n_ubatch = 0;
    // cache and tables
    f16 *kc = nullptr, *vc = nullptr;
    size_t kv_elems = 0;                      // elements of each of kc, vc
    bool kv_fp8 = false;                      // kc, vc hold FP8 E4M3 (one byte an element)
    float2 *rope = nullptr;
    float2 *rope_t = nullptr;      // the same table position-minor [hd / 2][n_ctx] (prefill QKV epilogue)
    // workspaces
    float *h = nullptr, *h2 = nullptr, *ss = nullptr, *ss2 = nullptr, *qf = nullptr;
    f16 *xg = nullptr;                        // one-row steps: f16(h * the next norm gain) [d]
    float *ss_cta = nullptr;                  // one-row steps: per-CTA sums of h^2 [num_sms]
    f16 *x = nullptr, *qb = nullptr, *o = nullptr, *u = nullptr;
    float *gemv_part = nullptr; unsigned *gemv_cnt = nullptr;
    size_t gemv_part_floats = 0, gemv_cnt_n = 0;
    TmaMap ax, ao, au;             // activation operands of the tcgen05 GEMM
    f16 *x2 = nullptr; TmaMap ax2; // prefill: the output rows' f16(h * gain) after the last layer's gather
    TmaMap ah, ah2;                // the residual streams h, h2 (fp32) for the GEMMs' residual epilogue
    bool resid_tma = true;         // option "gemm_resid_tma": that epilogue through shared memory and TMA
    bool split_k = true;           // option "gemm_split_k": residual GEMMs on 256-wide tiles with K split in two
    float *ss32 = nullptr, *ss32b = nullptr;   // prefill: per-32-column sums of h^2 of x / x2
    TmaMap aq, akc, avc, akc64;    // q and the fp16 caches, as the tcgen05 prefill attention reads them
    float *attn_part = nullptr; unsigned *attn_cnt = nullptr;
    size_t attn_part_floats = 0;
    int attn_split[9] = {0};
    int attn_split_cap = 0;        // largest one-row split the scratch holds
    // metadata
    int *meta_dev = nullptr; size_t meta_cap = 0;         // ints
    int *meta_host[2] = {nullptr, nullptr}; size_t meta_host_cap[2] = {0, 0};
    cudaEvent_t meta_ev[2] = {nullptr, nullptr}; int meta_slot = 0;
    int *dec_dev = nullptr;        // decode-graph metadata (see DEC_* offsets)
    int *dec_host[4] = {nullptr}; cudaEvent_t dec_ev[4] = {nullptr}; int dec_slot = 0;
    // outputs
    float *logits = nullptr; int logits_cap = 0;
    int *argmax_dev = nullptr; int *argmax_host = nullptr; int argmax_cap = 0;
    void *samp_dev = nullptr; size_t samp_cap = 0;   // uniforms and history of llm_sample
    int *gen_tokens = nullptr; int gen_cap = 0;
    uint32_t *err_dev = nullptr;
    // graphs: [T] decode step, [0] unused; gen = decode T=1 + feed
    cudaGraphExec_t graph[9] = {nullptr};
    int64_t graph_kernels[9] = {0};
    cudaGraphExec_t gen_graph = nullptr; int64_t gen_graph_kernels = 0;
    // host state
    std::vector<int32_t> seq_next;
    std::vector<int32_t> out_index;
    int n_outputs = 0;
    // options
    bool use_graphs = true;
    // programmatic dependent launch, per kernel family: the decode GEMVs run
    // faster without it (a one-wave grid placed beside the previous kernel's
    // CTAs ends up unevenly spread over the SMs); decode attention uses it to
    // stream its cached K/V while the QKV kernel runs; prefill keeps it
    bool use_pdl = false, use_pdl_attn = true, use_pdl_prefill = true;
    int gemm_kernel = 2, gemv_max_rows = 8;   // gemm: 2 CTA pairs (persistent past one wave), 3 persistent, 4 stream-K
    float *sk_ws = nullptr; unsigned *sk_flags = nullptr;   // stream-K partial slots and their flags
    unsigned sk_epoch = 0;                                  // per stream-K launch (nonzero)
    int swa_window = 0;                       // sliding-window attention: last W positions (0 = all)
    int attn_mode = 1;                        // prefill attention: 1 tcgen05 one CTA a head, 2 CTA pairs where they apply, 0 mma.sync
    bool attn_tc_ok = false;                  // tcgen05 applies: fp16 cache, head_dim 64 or 128, maps made
    bool attn_pair_ok = false;                // ... and the CTA pairs: head_dim 128, an even GQA group
    int ksplit_opt[5] = {0, 0, 0, 0, 0};      // GEMV K splits (qkv, o, gate/up, down, lm head); 0 = auto
    int64_t launches = 0;
    float *dbg = nullptr; int dbg_rows = 0, dbg_ub = 0;
    bool stream_ok = false, use_stream = true;    // one-row GEMVs streamed through shared memory
    bool stream_q8 = false, use_q8 = true;        // ... reading the model's Q8_0 rows (when it has them)
    int stream_pf_kb = 128;                       // L2 prefetch of the next streamed GEMV (KB per CTA)
    int stream_pf2_kb = 256;                      // ... of the gate/up GEMV by the QKV GEMV (KB per CTA)
    int stream_attn_kb = 136;                     // smem cap of the GEMVs beside decode attention (0 = none)
    int stream_stage_kb = 0;                      // largest ring stage of the streamed GEMVs (0 = their default)
    // per-kernel timing (diagnostic): events around every launch, eager only
    bool ktime = false;
    std::vector<KtRec> kt_pending;
    std::vector<cudaEvent_t> kt_pool;
    double kt_ms[K_COUNT] = {0};
    int64_t kt_n[K_COUNT] = {0};
    std::string last_error = "no error";
};

// Captured decode graphs bake in the options and buffers they were captured
// with: a change of either drops them, and the next step captures afresh.
static void drop_graphs(llm_ctx *c) {
    for (int t = 0; t < 9; ++t)
        if (c->graph[t]) { cudaGraphExecDestroy(c->graph[t]); c->graph[t] = nullptr; }
    if (c->gen_graph) { cudaGraphExecDestroy(c->gen_graph); c->gen_graph = nullptr; }
}

// decode-graph metadata layout (ints)
enum { DEC_TOK = 0, DEC_POS = 8, DEC_SEQ = 16, DEC_STEP = 24, DEC_NSTEPS = 25, DEC_INTS = 32 };

#define CK(call)                                                                      \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) return fail(c, LLM_ERR_COMPUTE, #call, e_);             \
    } while (0)

static int32_t fail(llm_ctx *c, int32_t code, const char *what, cudaError_t e = cudaSuccess) {
    std::string msg = what;
    if (e != cudaSuccess) { msg += ": "; msg += cudaGetErrorString(e); }
    if (c) c->last_error = msg; else g_create_error = msg;
    return code;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ============================================================== model

extern "C" int32_t llm_model_create(const llm_hparams *hp, const llm_weights *w, void *stream,
                                    llm_model **out) {
    llm_ctx *c = nullptr;
    if (!out) return fail(c, LLM_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!hp || !w) return fail(c, LLM_ERR_INVALID, "hparams or weights is NULL");
    const int d = hp->n_embd, H = hp->n_head, Hkv = hp->n_head_kv, hd = hp->head_dim;
    if (hp->n_vocab <= 0 || d <= 0 || hp->n_layer <= 0 || H <= 0 || Hkv <= 0 || hp->n_ff <= 0)
        return fail(c, LLM_ERR_INVALID, "non-positive hyper-parameter");
    if (H % Hkv) return fail(c, LLM_ERR_INVALID, "n_head must be a multiple of n_head_kv");
    if (hd != 32 && hd != 64 && hd != 128) return fail(c, LLM_ERR_INVALID, "head_dim must be 32, 64 or 128");
    if (d % 128 || (H * hd) % 128 || (Hkv * hd) % 64 || hp->n_vocab % 128)
        return fail(c, LLM_ERR_INVALID, "n_embd, n_head*head_dim and n_vocab must be multiples of 128, n_head_kv*head_dim of 64");
    if ((w->output == nullptr) != (hp->tied_output != 0))
        return fail(c, LLM_ERR_INVALID, "output must be NULL iff tied_output");
    if (!w->token_embd || !w->output_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
        !w->ffn_norm || !w->w_gate || !w->w_up || !w->w_down)
        return fail(c, LLM_ERR_INVALID, "missing weight pointer");
    for (int l = 0; l < hp->n_layer; ++l)
        if (!w->attn_norm[l] || !w->wq[l] || !w->wk[l] || !w->wv[l] || !w->wo[l] || !w->ffn_norm[l] ||
            !w->w_gate[l] || !w->w_up[l] || !w->w_down[l])
            return fail(c, LLM_ERR_INVALID, "missing per-layer weight pointer");

    cudaError_t e = init_kernel_attributes();
    if (e) return fail(c, LLM_ERR_COMPUTE, "kernel attributes", e);

    llm_model *m = new llm_model();
    m->hp = *hp;
    m->d = d; m->H = H; m->Hkv = Hkv; m->hd = hd;
    m->n_q = H * hd; m->n_kv = Hkv * hd; m->n_qkv = m->n_q + 2 * m->n_kv;
    m->F = hp->n_ff; m->F_pad = (int)align_up(hp->n_ff, 128);
    m->V = hp->n_vocab; m->L = hp->n_layer;
    cudaGetDevice(&m->device);
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);

    const size_t per_layer = (size_t)m->n_qkv * d + (size_t)d * m->n_q + (size_t)2 * m->F_pad * d + (size_t)d * m->F_pad;
    const size_t n_emb = (size_t)m->V * d;
    const size_t total = n_emb * (hp->tied_output ? 1 : 2) + per_layer * m->L;
    if (cudaMalloc(&m->wbuf, total * sizeof(f16)) != cudaSuccess ||
        cudaMalloc(&m->fbuf, (size_t)d * (1 + 2 * m->L) * sizeof(float)) != cudaSuccess) {
        cudaGetLastError();
        if (m->wbuf) cudaFree(m->wbuf);
        delete m;
        return fail(c, LLM_ERR_ALLOC, "weight allocation failed");
    }
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *flag = nullptr;
    if (cudaMalloc(&flag, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(m->wbuf);
        cudaFree(m->fbuf);
        delete m;
        return fail(c, LLM_ERR_ALLOC, "weight allocation failed");
    }
    f16 *p = m->wbuf;
    e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), st);
    m->token_embd = p; p += n_emb;
    if (!e) e = launch_convert_rows((const bf16 *)w->token_embd, d, m->token_embd, d, m->V, d, flag, st);
    if (!hp->tied_output) {
        m->output = p; p += n_emb;
        if (!e) e = launch_convert_rows((const bf16 *)w->output, d, m->output, d, m->V, d, flag, st);
    } else {
        m->output = m->token_embd;
    }
    m->output_norm = m->fbuf;
    if (!e) e = launch_widen_bf16((const bf16 *)w->output_norm, m->output_norm, d, st);
    m->layers.resize(m->L);
    for (int l = 0; l < m->L && !e; ++l) {
        LayerW &lw = m->layers[l];
        lw.wqkv = p; p += (size_t)m->n_qkv * d;
        lw.wo = p; p += (size_t)d * m->n_q;
        lw.wgu = p; p += (size_t)2 * m->F_pad * d;
        lw.wdown = p; p += (size_t)d * m->F_pad;
        lw.attn_norm = m->fbuf + d * (1 + 2 * l);
        lw.ffn_norm = lw.attn_norm + d;
        e = launch_convert_rows((const bf16 *)w->wq[l], d, lw.wqkv, d, m->n_q, d, flag, st);
        if (!e) e = launch_convert_rows((const bf16 *)w->wk[l], d, lw.wqkv + (size_t)m->n_q * d, d, m->n_kv, d, flag, st);
        if (!e) e = launch_convert_rows((const bf16 *)w->wv[l], d, lw.wqkv + (size_t)(m->n_q + m->n_kv) * d, d, m->n_kv, d, flag, st);
        if (!e) e = launch_convert_rows((const bf16 *)w->wo[l], m->n_q, lw.wo, m->n_q, d, m->n_q, flag, st);
        if (!e) e = launch_repack_gate_up((const bf16 *)w->w_gate[l], (const bf16 *)w->w_up[l], m->F, m->F_pad, d, lw.wgu, flag, st);
        if (!e) e = cudaMemsetAsync(lw.wdown, 0, (size_t)d * m->F_pad * sizeof(f16), st);
        if (!e) e = launch_convert_rows((const bf16 *)w->w_down[l], m->F, lw.wdown, m->F_pad, d, m->F, flag, st);
        if (!e) e = launch_widen_bf16((const bf16 *)w->attn_norm[l], lw.attn_norm, d, st);
        if (!e) e = launch_widen_bf16((const bf16 *)w->ffn_norm[l], lw.ffn_norm, d, st);
    }
    uint32_t flag_h = 0;
    if (!e) e = cudaMemcpyAsync(&flag_h, flag, sizeof flag_h, cudaMemcpyDeviceToHost, st);
    bool maps_ok = true;
    auto wmap = [&](WMap &wm, const f16 *ptr, int rows, int cols) {
        maps_ok = maps_ok && make_operand_map(&wm.map128, ptr, rows, cols, 128);
        maps_ok = maps_ok && make_operand_map(&wm.map64, ptr, rows, cols, 64);
        wm.has256 = rows % 256 == 0;
        if (wm.has256) maps_ok = maps_ok && make_operand_map(&wm.map256, ptr, rows, cols, 256);
        wm.has96 = rows % 192 == 0;
        if (wm.has96) maps_ok = maps_ok && make_operand_map(&wm.map96, ptr, rows, cols, 96);
    };
    for (int l = 0; l < m->L; ++l) {
        LayerW &lw = m->layers[l];
        wmap(lw.mqkv, lw.wqkv, m->n_qkv, d);
        wmap(lw.mo, lw.wo, d, m->n_q);
        wmap(lw.mgu, lw.wgu, 2 * m->F_pad, d);
        wmap(lw.mdown, lw.wdown, d, m->F_pad);
    }
    wmap(m->mout, m->output, m->V, d);
    if (!maps_ok) {
        cudaStreamSynchronize(st);
        cudaFree(flag);
        cudaFree(m->wbuf);
        cudaFree(m->fbuf);
        delete m;
        return fail(c, LLM_ERR_COMPUTE, "TMA descriptor creation failed");
    }
    if (!e) e = cudaStreamSynchronize(st);
    cudaFree(flag);
    if (e || flag_h) {
        cudaFree(m->wbuf);
        cudaFree(m->fbuf);
        delete m;
        if (e) return fail(c, LLM_ERR_COMPUTE, "weight copy", e);
        return fail(c, LLM_ERR_INVALID, "a weight lies outside the fp16 range (|w| > 65504)");
    }
    *out = m;
    return LLM_OK;
}

extern "C" void llm_model_free(llm_model *m) {
    if (!m) return;
    cudaFree(m->qbuf);
    cudaFree(m->wbuf);
    cudaFree(m->fbuf);
    delete m;
}

// Q8_0 weights: every matrix a projection multiplies by is encoded in place
// (its fp16 copy, which the prefill GEMMs and the 2-8-row GEMVs read, becomes
// f16(q * d)), and, where its rows suit the streamed GEMV (K % 256 == 0 for
// every decode matrix), its Q8_0 rows are kept beside it for the one-row
// decode GEMVs, which then stream about half the bytes.
extern "C" int32_t llm_model_quantize(llm_model *m, int32_t wtype, void *stream) {
    llm_ctx *c = nullptr;
    if (!m) return fail(c, LLM_ERR_INVALID, "model is NULL");
    if (wtype != LLM_WTYPE_Q8_0) return fail(c, LLM_ERR_INVALID, "unknown weight type");
    if (m->wtype) return fail(c, LLM_ERR_INVALID, "the model is already quantised");
    if (m->n_contexts) return fail(c, LLM_ERR_INVALID, "the model has live contexts");
    const int d = m->d;
    struct Mat { f16 *w; int N, K; const uint8_t **q; };
    std::vector<Mat> mats;
    for (LayerW &lw : m->layers) {
        mats.push_back({lw.wqkv, m->n_qkv, d, &lw.q_qkv});
        mats.push_back({lw.wo, d, m->n_q, &lw.q_o});
        mats.push_back({lw.wgu, 2 * m->F_pad, d, &lw.q_gu});
        mats.push_back({lw.wdown, d, m->F_pad, &lw.q_down});
    }
    mats.push_back({m->output, m->V, d, &m->q_out});    // the embedding table too when tied
    const bool rows = d % 256 == 0 && m->n_q % 256 == 0 && m->F_pad % 256 == 0;
    size_t total = 0;
    if (rows)
        for (const Mat &mt : mats) total += align_up((size_t)mt.N * q8_0_row_bytes(mt.K), 256);
    uint8_t *qb = nullptr;
    if (total && cudaMalloc(&qb, total) != cudaSuccess) {
        cudaGetLastError();
        return fail(c, LLM_ERR_ALLOC, "Q8_0 allocation failed");
    }
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    size_t off = 0;
    for (const Mat &mt : mats) {
        uint8_t *q = qb ? qb + off : nullptr;
        if (qb) off += align_up((size_t)mt.N * q8_0_row_bytes(mt.K), 256);
        if (!e) e = launch_quantize_q8_0(mt.w, mt.N, mt.K, q, true, st);
        *mt.q = q;
    }
    if (!e) e = cudaStreamSynchronize(st);
    if (e) {
        for (const Mat &mt : mats) *mt.q = nullptr;
        cudaFree(qb);
        m->wtype = -1;     // the fp16 copies may be partly rewritten
        return fail(c, LLM_ERR_COMPUTE, "Q8_0 encoding failed; the model's weights are undefined", e);
    }
    m->qbuf = qb;
    m->wtype = wtype;
    return LLM_OK;
}

// The one-row GEMVs can read the model's Q8_0 rows with this context's caps.
static bool q8_plans_ok(const llm_ctx *c) {
    const llm_model *m = c->m;
    const int d = m->d, n = m->num_sms;
    return m->qbuf && gemv_stream_ok(EPI_QKV, m->n_qkv, d, n, c->stream_attn_kb, true) &&
           gemv_stream_ok(EPI_RESID, d, m->n_q, n, c->stream_attn_kb, true) &&
           gemv_stream_ok(EPI_SWIGLU, 2 * m->F_pad, d, n, 0, true) && gemv_stream_ok(EPI_RESID, d, m->F_pad, n, 0, true) &&
           gemv_stream_ok(EPI_STORE, m->V, d, n, 0, true);
}

// ============================================================== context

static void ctx_release(llm_ctx *c) {
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    drop_graphs(c);
    void *dev[] = {c->kc, c->vc, c->rope, c->rope_t, c->h, c->h2, c->ss, c->ss2, c->qf, c->x, c->qb, c->o, c->u,
                   c->gemv_part, c->gemv_cnt, c->sk_ws, c->sk_flags, c->attn_part, c->attn_cnt, c->meta_dev, c->dec_dev,
                   c->logits, c->argmax_dev, c->gen_tokens, c->err_dev,
                   c->samp_dev, c->xg, c->ss_cta, c->x2, c->ss32, c->ss32b};
    for (void *p : dev) if (p) cudaFree(p);
    for (int i = 0; i < 2; ++i) {
        if (c->meta_host[i]) cudaFreeHost(c->meta_host[i]);
        if (c->meta_ev[i]) cudaEventDestroy(c->meta_ev[i]);
    }
    for (int i = 0; i < 4; ++i) {
        if (c->dec_host[i]) cudaFreeHost(c->dec_host[i]);
        if (c->dec_ev[i]) cudaEventDestroy(c->dec_ev[i]);
    }
    if (c->argmax_host) cudaFreeHost(c->argmax_host);
    for (auto &r : c->kt_pending) { c->kt_pool.push_back(r.a); c->kt_pool.push_back(r.b); }
    for (cudaEvent_t ev : c->kt_pool) cudaEventDestroy(ev);
    if (c->own_stream) cudaStreamDestroy(c->stream);
    if (c->m) c->m->n_contexts--;
    delete c;
}

// TMA maps of the tcgen05 prefill attention: q [n_ubatch][n_q] and the fp16
// caches viewed as [n_seq * n_layer * Hkv * n_ctx][hd]; remade whenever the
// cache is reallocated.  Without them (FP8 cache, head_dim 32, more cache
// rows than a map addresses) prefill attention runs on the mma.sync kernel.
static void make_attn_maps(llm_ctx *c) {
    const llm_model *m = c->m;
    const long long rows = (long long)c->n_seq_max * m->L * m->Hkv * c->n_ctx;
    const int nub = c->n_ubatch < 8 ? 8 : c->n_ubatch;
    c->attn_tc_ok = !c->kv_fp8 && attn_prefill_tc_ok(m->hd, false) && rows < (1ll << 31) &&
                    make_operand_map(&c->aq, c->qb, nub, m->n_q, 128) &&
                    make_operand_map(&c->akc, c->kc, (int)rows, m->hd, 128) &&
                    make_operand_map(&c->avc, c->vc, (int)rows, m->hd, 128);
    c->attn_pair_ok = c->attn_tc_ok && attn_prefill_pair_ok(m->hd, m->H, m->Hkv, false) &&
                      make_operand_map(&c->akc64, c->kc, (int)rows, m->hd, 64);
}

static int attn_pick_split(const llm_model *m, int T, int n_ctx) {
    // the kernel uses only the splits a sequence needs (whole 64-key tiles each)
    const int mx = (n_ctx + 63) / 64;
    int s;
    if (T == 1) {
        // one-row steps: ~1.7 sqrt(key tiles of the context), the balance of
        // the splits' merge against their parallelism (measured on the 8B
        // shape: 14 at n_ctx 4096 and 38 at 32768, where one CTA per SM, 19,
        // was 1.5% and 1.8% slower)
        s = (int)lrint(1.7 * std::sqrt((double)mx));
    } else {
        // multi-row steps: about two CTAs per SM at full context (8 rows of the
        // 8B shape at n_ctx 8192: 4 splits 1801 tok/s, 2 splits 1661)
        s = 2 * m->num_sms / (T * m->Hkv);
    }
    if (s > 128) s = 128;
    if (s > mx) s = mx;
    return s < 1 ? 1 : s;
}

// Allocation-failure injection for tests (llm_debug_fail_alloc): the device
// allocation of that index in the next llm_kv_alloc fails; -1 = none.
static int g_fail_alloc = -1;

extern "C" int32_t llm_debug_fail_alloc(int32_t n) {
    if (n < -1) return LLM_ERR_INVALID;
    g_fail_alloc = n;
    return LLM_OK;
}

extern "C" int32_t llm_kv_alloc(llm_model *m, int32_t n_ctx, int32_t n_seq_max, int32_t n_ubatch, void *stream,
                                llm_ctx **out) {
    llm_ctx *nc = nullptr;
    const int inject = g_fail_alloc;      // armed for this call only
    g_fail_alloc = -1;
    if (!out) return fail(nc, LLM_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!m || n_ctx < 1 || n_seq_max < 1 || n_ubatch < 1 || n_ubatch > 4096)
        return fail(nc, LLM_ERR_INVALID, "invalid context arguments");
    llm_ctx *c = new llm_ctx();
    c->m = m;
    m->n_contexts++;
    c->stream = (cudaStream_t)stream;
    if (!c->stream) {
        // The legacy default stream cannot be captured into a graph.  A blocking
        // stream stays ordered with it, so callers on stream 0 see no difference.
        if (cudaStreamCreate(&c->stream) != cudaSuccess) {
            cudaGetLastError();
            c->stream = nullptr;
            ctx_release(c);
            return fail(nc, LLM_ERR_ALLOC, "stream creation failed");
        }
        c->own_stream = true;
    }
    c->n_ctx = n_ctx; c->n_seq_max = n_seq_max; c->n_ubatch = n_ubatch;
    c->seq_next.assign(n_seq_max, 0);
    const int d = m->d, hd = m->hd;
    const int nub = n_ubatch < 8 ? 8 : n_ubatch;
    bool ok = true;
    int n_alloc = 0;
    auto dmal = [&](void **p, size_t bytes) {
        if (!ok) return;
        if (n_alloc++ == inject) { ok = false; return; }
        if (cudaMalloc(p, bytes ? bytes : 16) != cudaSuccess) { ok = false; cudaGetLastError(); }
    };
    const size_t kv_elems = (size_t)n_seq_max * m->L * m->Hkv * n_ctx * hd;
    c->kv_elems = kv_elems;
    dmal((void **)&c->kc, kv_elems * sizeof(f16));
    dmal((void **)&c->vc, kv_elems * sizeof(f16));
    dmal((void **)&c->rope, (size_t)n_ctx * (hd / 2) * sizeof(float2));
    dmal((void **)&c->rope_t, (size_t)n_ctx * (hd / 2) * sizeof(float2));
    dmal((void **)&c->h, (size_t)nub * d * sizeof(float));
    dmal((void **)&c->h2, (size_t)nub * d * sizeof(float));
    dmal((void **)&c->xg, (size_t)d * sizeof(f16));
    dmal((void **)&c->ss_cta, (size_t)m->num_sms * sizeof(float));
    dmal((void **)&c->ss, (size_t)(d / 64) * 8 * sizeof(float));
    dmal((void **)&c->ss2, (size_t)(d / 64) * 8 * sizeof(float));
    dmal((void **)&c->qf, (size_t)8 * m->n_q * sizeof(float));
    dmal((void **)&c->x, (size_t)nub * d * sizeof(f16));
    dmal((void **)&c->x2, (size_t)nub * d * sizeof(f16));
    dmal((void **)&c->ss32, (size_t)nub * (d / 32) * sizeof(float));
    dmal((void **)&c->ss32b, (size_t)nub * (d / 32) * sizeof(float));
    dmal((void **)&c->qb, (size_t)nub * m->n_q * sizeof(f16));
    dmal((void **)&c->o, (size_t)nub * m->n_q * sizeof(f16));
    dmal((void **)&c->u, (size_t)nub * m->F_pad * sizeof(f16));
    // split-K scratch: the largest ksplit * N over the GEMVs and row counts
    const int shapes[5][2] = {{m->n_qkv, d}, {d, m->n_q}, {2 * m->F_pad, d}, {d, m->F_pad}, {m->V, d}};
    size_t part = 0, cnt = 0;
    for (int T = 1; T <= 8; ++T)
        for (auto &s : shapes) {
            const int ks = gemv_pick_split(s[0], s[1], T, m->num_sms);
            part = std::max(part, (size_t)ks * s[0] * 8);
            if (s[0] != m->V)     // room for tuning the split of the layer GEMVs
                part = std::max(part, (size_t)std::min(32, s[1] / 128) * s[0] * 8);
            cnt = std::max(cnt, (size_t)s[0] / 64);
        }
    c->gemv_part_floats = part; c->gemv_cnt_n = cnt;
    dmal((void **)&c->gemv_part, part * sizeof(float));
    const int max_pairs = gemm_pair_max_clusters();
    dmal((void **)&c->sk_ws, gemm_pair_sk_ws_floats(max_pairs) * sizeof(float));
    dmal((void **)&c->sk_flags, (size_t)2 * max_pairs * sizeof(unsigned));
    dmal((void **)&c->gemv_cnt, cnt * sizeof(unsigned));
    size_t ap = 0;
    c->attn_split_cap = std::min(128, (n_ctx + 63) / 64);
    for (int T = 1; T <= 8; ++T) {
        c->attn_split[T] = attn_pick_split(m, T, n_ctx);
        ap = std::max(ap, attn_decode_scratch_floats(T, m->H, hd, c->attn_split_cap));   // any split up to the cap
    }
    c->attn_part_floats = ap;
    dmal((void **)&c->attn_part, ap * sizeof(float));
    dmal((void **)&c->attn_cnt, (size_t)8 * m->Hkv * sizeof(unsigned));
    dmal((void **)&c->dec_dev, DEC_INTS * sizeof(int));
    dmal((void **)&c->err_dev, sizeof(uint32_t));
    if (ok) {
        for (int i = 0; i < 4 && ok; ++i) {
            if (cudaHostAlloc((void **)&c->dec_host[i], DEC_INTS * sizeof(int), cudaHostAllocDefault) != cudaSuccess ||
                cudaEventCreateWithFlags(&c->dec_ev[i], cudaEventDisableTiming) != cudaSuccess)
                ok = false;
        }
        for (int i = 0; i < 2 && ok; ++i)
            if (cudaEventCreateWithFlags(&c->meta_ev[i], cudaEventDisableTiming) != cudaSuccess) ok = false;
    }
    if (!ok) {
        ctx_release(c);
        return fail(nc, LLM_ERR_ALLOC, "context allocation failed");
    }
    if (!make_operand_map(&c->ax, c->x, nub, d, 128) || !make_operand_map(&c->ax2, c->x2, nub, d, 128) ||
        !make_f32_tile_map(&c->ah, c->h, nub, d) || !make_f32_tile_map(&c->ah2, c->h2, nub, d) ||
        !make_operand_map(&c->ao, c->o, nub, m->n_q, 128) ||
        !make_operand_map(&c->au, c->u, nub, m->F_pad, 128)) {
        ctx_release(c);
        return fail(nc, LLM_ERR_COMPUTE, "TMA descriptor creation failed");
    }
    make_attn_maps(c);
    // RoPE table: angle = pos * theta^(-2i/hd), in double precision
    std::vector<float2> tab((size_t)n_ctx * (hd / 2));
    for (int pidx = 0; pidx < n_ctx; ++pidx)
        for (int i = 0; i < hd / 2; ++i) {
            const double ang = (double)pidx * std::pow((double)m->hp.rope_theta, -2.0 * i / hd);
            tab[(size_t)pidx * (hd / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    std::vector<float2> tab_t(tab.size());
    for (int pidx = 0; pidx < n_ctx; ++pidx)
        for (int i = 0; i < hd / 2; ++i) tab_t[(size_t)i * n_ctx + pidx] = tab[(size_t)pidx * (hd / 2) + i];
    cudaError_t e = cudaMemcpyAsync(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, c->stream);
    if (!e) e = cudaMemcpyAsync(c->rope_t, tab_t.data(), tab_t.size() * sizeof(float2), cudaMemcpyHostToDevice, c->stream);
    if (!e) e = cudaMemsetAsync(c->gemv_cnt, 0, cnt * sizeof(unsigned), c->stream);
    if (!e) e = cudaMemsetAsync(c->sk_flags, 0, (size_t)2 * gemm_pair_max_clusters() * sizeof(unsigned), c->stream);
    if (!e) e = cudaMemsetAsync(c->attn_cnt, 0, (size_t)8 * m->Hkv * sizeof(unsigned), c->stream);
    if (!e) e = cudaMemsetAsync(c->err_dev, 0, sizeof(uint32_t), c->stream);
    if (!e) e = cudaMemsetAsync(c->dec_dev, 0, DEC_INTS * sizeof(int), c->stream);
    // one-row steps: every GEMV shape has a streamed plan
    c->stream_ok = gemv_stream_ok(EPI_QKV, m->n_qkv, d, m->num_sms, c->stream_attn_kb) &&
                   gemv_stream_ok(EPI_RESID, d, m->n_q, m->num_sms, c->stream_attn_kb) &&
                   gemv_stream_ok(EPI_SWIGLU, 2 * m->F_pad, d, m->num_sms) &&
                   gemv_stream_ok(EPI_RESID, d, m->F_pad, m->num_sms) && gemv_stream_ok(EPI_STORE, m->V, d, m->num_sms);
    c->stream_q8 = q8_plans_ok(c);
    if (!e) e = cudaMemsetAsync(c->kc, 0, kv_elems * sizeof(f16), c->stream);
    if (!e) e = cudaMemsetAsync(c->vc, 0, kv_elems * sizeof(f16), c->stream);
    if (!e) e = cudaStreamSynchronize(c->stream);
    if (e) {
        ctx_release(c);
        return fail(nc, LLM_ERR_COMPUTE, "context initialisation", e);
    }
    *out = c;
    return LLM_OK;
}

extern "C" void llm_kv_free(llm_ctx *c) { ctx_release(c); }

// ============================================================== the forward pass

namespace {

struct UbDev {
    const int *tok, *pos, *seq;
    const int *out_rows;      // rows of the ubatch that are outputs (n_out entries), or NULL = all
    const AttnTile *tiles;    // up to 64 rows each (mma.sync prefill attention)
    int n_tiles;
    const AttnTile *tiles128; // up to 128 rows each (tcgen05 prefill attention)
    int n_tiles128;
    int T, n_out;
    int out_base;             // first logits row of this ubatch
    int ub_index;
};

Launch lnch(llm_ctx *c) { return Launch{c->stream, c->use_pdl && !c->ktime, &c->launches}; }
Launch lnch_attn(llm_ctx *c) { return Launch{c->stream, c->use_pdl_attn && !c->ktime, &c->launches}; }
// the streamed GEMVs always overlap their start with the previous kernel's tail
Launch lnch_stream(llm_ctx *c) { return Launch{c->stream, !c->ktime, &c->launches}; }
Launch lnch_prefill(llm_ctx *c) { return Launch{c->stream, c->use_pdl_prefill && !c->ktime, &c->launches}; }

cudaEvent_t kt_event(llm_ctx *c) {
    if (!c->kt_pool.empty()) {
        cudaEvent_t ev = c->kt_pool.back();
        c->kt_pool.pop_back();
        return ev;
    }
    cudaEvent_t ev = nullptr;
    cudaEventCreate(&ev);
    return ev;
}

// Runs a launcher; with timing on, brackets it with events on the context stream.
template <typename F>
cudaError_t timed(llm_ctx *c, int kid, F &&f) {
    if (!c->ktime) return f();
    cudaEvent_t a = kt_event(c), b = kt_event(c);
    cudaEventRecord(a, c->stream);
    const cudaError_t e = f();
    cudaEventRecord(b, c->stream);
    c->kt_pending.push_back(KtRec{kid, a, b});
    return e;
}

KvView kv_view(llm_ctx *c, int layer) {
    const llm_model *m = c->m;
    const size_t per_layer = (size_t)m->Hkv * c->n_ctx * m->hd;
    KvView v;
    if (c->kv_fp8) {
        v.k = v.v = nullptr;
        v.k8 = reinterpret_cast<uint8_t *>(c->kc) + layer * per_layer;
        v.v8 = reinterpret_cast<uint8_t *>(c->vc) + layer * per_layer;
    } else {
        v.k = c->kc + layer * per_layer;
        v.v = c->vc + layer * per_layer;
    }
    v.seq_stride = (long long)(per_layer * m->L);
    v.n_ctx = c->n_ctx; v.n_seq = c->n_seq_max; v.head_dim = m->hd; v.n_kv_head = m->Hkv;
    return v;
}

enum { GV_QKV, GV_O, GV_GU, GV_DOWN, GV_LM };

GemvArgs gemv_base(llm_ctx *c, const f16 *W, int N, int K, int T, int cls) {
    GemvArgs a;
    memset(&a, 0, sizeof a);
    a.W = W; a.N = N; a.K = K; a.T = T;
    a.ksplit = gemv_pick_split(N, K, T, c->m->num_sms);
    const int ko = c->ksplit_opt[cls];
    if (ko > 0 && K % (128 * ko) == 0 && (size_t)ko * N * 8 <= c->gemv_part_floats &&
        gemv_smem_bytes(K, ko, T) <= 100 * 1024)
        a.ksplit = ko;
    a.part = c->gemv_part; a.counters = c->gemv_cnt;
    a.eps = c->m->hp.rms_eps;
    a.err = c->err_dev;
    return a;
}

cudaError_t debug_copy(llm_ctx *c, const UbDev &u, int layer, const float *h, int rows) {
    if (!c->dbg || u.ub_index >= c->dbg_ub) return cudaSuccess;
    const int d = c->m->d;
    const int n = rows < c->dbg_rows ? rows : c->dbg_rows;
    float *dst = c->dbg + (((size_t)u.ub_index * c->m->L + layer) * c->dbg_rows) * d;
    return timed(c, K_COPY, [&] { return launch_copy_f32(h, dst, (size_t)n * d, lnch(c)); });
}

// Decode-sized ubatch (1..8 rows): GEMV kernels and split attention.
cudaError_t run_small(llm_ctx *c, const UbDev &u) {
    const llm_model *m = c->m;
    const int d = m->d, T = u.T;
    const Launch L = lnch(c);
    // one-row steps stream their GEMVs (one CTA per SM, overlapped launches)
    const bool stream = T == 1 && c->stream_ok && c->use_stream;
    // kb: shared-memory cap of a streamed GEMV; the ones before and after
    // decode attention leave room for an attention CTA on the same SM
    auto gv = [&](int pro, int epi, const GemvArgs &a, int kb) {
        return stream ? launch_gemv_stream(pro, epi, a, m->num_sms, kb, lnch_stream(c), c->stream_stage_kb)
                      : launch_gemv(pro, epi, a, L);
    };
    const int akb = c->stream_attn_kb;
    // the streamed GEMV that follows: its first weight bytes per CTA go to L2
    // while this one drains (all of them when `all`)
    // one-row steps of a Q8_0 model stream its Q8_0 rows
    const bool q8 = stream && c->stream_q8 && c->use_q8;
    auto wq = [&](GemvArgs &a, const uint8_t *q) { if (q8) a.W8 = q; };
    auto prefetch = [&](GemvArgs &a, const f16 *W, const uint8_t *Wq, int N, int K, int epi, bool all) {
        if (c->stream_pf_kb <= 0) return;
        a.pf_W = W; a.pf_N = N; a.pf_K = K; a.pf_unit = gemv_stream_unit(epi);
        if (q8) a.pf_W8 = Wq;
        a.pf_bytes = all ? (1 << 30) : c->stream_pf_kb * 1024;
    };
    // a residual GEMV hands the next RMSNorm GEMV its input: f16(h * gain) and
    // per-CTA sums of h^2 (read back in order), so that GEMV reads 8 KB, not h
    const bool handoff = stream && m->num_sms <= 256;
    auto give_x = [&](GemvArgs &a, const float *gain) {
        if (handoff) { a.gain_next = gain; a.xg_out = c->xg; a.ss_cta = c->ss_cta; }
    };
    auto take_x = [&](GemvArgs &a) {
        if (handoff) { a.xg = c->xg; a.ss_in = c->ss_cta; a.n_ss_in = m->num_sms; }
    };
    cudaError_t e = timed(c, K_EMBED, [&] { return launch_embed(m->token_embd, u.tok, T, d, m->V, c->h, c->ss, c->err_dev, L); });
    if (e) return e;
    float *hcur = c->h, *sscur = c->ss;
    int Tc = T;
    for (int l = 0; l < m->L; ++l) {
        const LayerW &w = m->layers[l];
        const KvView kv = kv_view(c, l);
        GemvArgs a = gemv_base(c, w.wqkv, m->n_qkv, d, T, GV_QKV);
        wq(a, w.q_qkv);
        a.h = c->h; a.ldh = d; a.ss_part = c->ss; a.gain = w.attn_norm;
        if (stream) {
            prefetch(a, w.wo, w.q_o, d, m->n_q, EPI_RESID, true);     // all of Wo, read during attention
            if (c->stream_pf2_kb > 0) {
                // and the first KB of each gate/up slab: HBM is idle while attention runs
                a.pf2_W = w.wgu; a.pf2_N = 2 * m->F_pad; a.pf2_K = d; a.pf2_unit = gemv_stream_unit(EPI_SWIGLU);
                if (q8) a.pf2_W8 = w.q_gu;
                a.pf2_bytes = c->stream_pf2_kb * 1024;
            }
        }
        if (stream && l > 0) take_x(a);                                // h * attn_norm from the down GEMV
        a.n_q = m->n_q; a.n_kv = m->n_kv; a.rope = c->rope; a.q_out = c->qf; a.kv = kv;
        a.pos = u.pos; a.seq = u.seq;
        if ((e = timed(c, K_GEMV_QKV, [&] { return gv(PRO_NORM, EPI_QKV, a, akb); }))) return e;
        AttnDecodeArgs at;
        at.q = c->qf; at.kv = kv; at.pos = u.pos; at.seq = u.seq; at.o = c->o; at.T = T; at.H = m->H;
        at.n_split = c->attn_split[T]; at.part = c->attn_part; at.counters = c->attn_cnt; at.err = c->err_dev;
        at.window = c->swa_window;
        if ((e = timed(c, K_ATTN_DECODE, [&] { return launch_attn_decode(at, lnch_attn(c)); }))) return e;
        a = gemv_base(c, w.wo, d, m->n_q, T, GV_O);
        wq(a, w.q_o);
        a.x = c->o; a.ldx = m->n_q; a.hres = c->h; a.ldh_res = d; a.ss_out = c->ss;
        if (stream) {
            prefetch(a, w.wgu, w.q_gu, 2 * m->F_pad, d, EPI_SWIGLU, false);
            give_x(a, w.ffn_norm);                                     // x of the gate/up GEMV
        }
        if ((e = timed(c, K_GEMV_O, [&] { return gv(PRO_BF16, EPI_RESID, a, akb); }))) return e;
        if (l == m->L - 1 && u.out_rows) {
            // keep only the output rows before the last MLP
            if ((e = timed(c, K_GATHER, [&] { return launch_gather_rows(c->h, u.out_rows, u.n_out, d, c->h2, c->ss, c->ss2, L); }))) return e;
            hcur = c->h2; sscur = c->ss2; Tc = u.n_out;
        }
        if (Tc == 0) break;
        a = gemv_base(c, w.wgu, 2 * m->F_pad, d, Tc, GV_GU);
        wq(a, w.q_gu);
        a.h = hcur; a.ldh = d; a.ss_part = sscur; a.gain = w.ffn_norm; a.u_out = c->u; a.ldu = m->F_pad;
        if (stream) prefetch(a, w.wdown, w.q_down, d, m->F_pad, EPI_RESID, false);
        if (stream && hcur == c->h) take_x(a);
        if ((e = timed(c, K_GEMV_GATEUP, [&] { return gv(PRO_NORM, EPI_SWIGLU, a, 0); }))) return e;
        a = gemv_base(c, w.wdown, d, m->F_pad, Tc, GV_DOWN);
        wq(a, w.q_down);
        a.x = c->u; a.ldx = m->F_pad; a.hres = hcur; a.ldh_res = d; a.ss_out = sscur;
        if (stream) {
            if (l + 1 < m->L) prefetch(a, m->layers[l + 1].wqkv, m->layers[l + 1].q_qkv, m->n_qkv, d, EPI_QKV, false);
            else prefetch(a, m->output, m->q_out, m->V, d, EPI_STORE, false);
            if (hcur == c->h) give_x(a, l + 1 < m->L ? m->layers[l + 1].attn_norm : m->output_norm);
        }
        if ((e = timed(c, K_GEMV_DOWN, [&] { return gv(PRO_BF16, EPI_RESID, a, 0); }))) return e;
        if ((e = debug_copy(c, u, l, hcur, Tc))) return e;
    }
    if (Tc == 0) return cudaSuccess;
    GemvArgs a = gemv_base(c, m->output, m->V, d, Tc, GV_LM);
    wq(a, m->q_out);
    a.h = hcur; a.ldh = d; a.ss_part = sscur; a.gain = m->output_norm;
    a.out = c->logits + (size_t)u.out_base * m->V; a.ldo = m->V;
    if (stream && hcur == c->h) take_x(a);                             // h * output_norm from the last down
    return timed(c, K_GEMV_LMHEAD, [&] { return gv(PRO_NORM, EPI_STORE, a, 0); });
}

cudaError_t gemm(llm_ctx *c, int epi, const GemmArgs &g, const TmaMap &ma, const WMap &mw) {
    if (c->gemm_kernel == 4 && g.N % 256 == 0) {
        // stream-K over 256-wide pair tiles: every pair gets the same share of K stages
        if (++c->sk_epoch == 0) c->sk_epoch = 1;
        return launch_gemm_pair_sk(epi, g, ma, mw.map128, c->sk_ws, c->sk_flags, c->sk_epoch, lnch_prefill(c));
    }
    const int bn = gemm_pair_pick_bn(g.M, g.N, gemm_pair_max_clusters());
    if (!bn || (bn == 192 && !mw.has96)) return cudaErrorInvalidValue;
    const TmaMap &mb = bn == 128 ? mw.map64 : bn == 192 ? mw.map96 : mw.map128;
    // more tiles than resident pairs: the persistent kernel overlaps each
    // tile's epilogue with the next tile's MMAs (measured: gate/up 98 -> 88 us);
    // one wave runs faster without its extra warps
    if (c->gemm_kernel == 3 || (long long)((g.M + 255) / 256) * (g.N / bn) > gemm_pair_max_clusters())
        return launch_gemm_pair_persist(epi, g, ma, mb, bn, lnch_prefill(c));
    // the residual epilogue through shared memory when both of its buffers have maps
    const TmaMap *mh = nullptr, *mx = nullptr;
    if (epi == EPI_RESID && c->resid_tma) {
        mh = g.hres == c->h ? &c->ah : g.hres == c->h2 ? &c->ah2 : nullptr;
        mx = g.x_next == c->x ? &c->ax : g.x_next == c->x2 ? &c->ax2 : nullptr;
        if (g.x_next && !mx) mh = nullptr;
    }
    GemmArgs gt = g;
    gt.tma_epi = mh != nullptr;
    // a residual GEMM with a long K (down) on 256-wide tiles with K split in
    // two: as many pairs as the 128-wide tiles, each stage carrying twice the
    // MMA work for 4/3 of the bytes an SM takes in; the halves exchange their
    // partials through L2 (measured: down 61.5 -> 54.7 us; O, K 4096, lost
    // more to the exchange than it gained: 28.6 -> 30.9); both halves must be
    // resident
    if (epi == EPI_RESID && c->split_k && mh && g.N % 256 == 0 && g.K >= 8192) {
        const long long units = (long long)((g.M + 255) / 256) * (g.N / 256) * 2;
        if (units <= gemm_pair_max_clusters()) {
            gt.split_k = 1; gt.part = c->sk_ws; gt.flags = c->sk_flags;
            if (++c->sk_epoch == 0) c->sk_epoch = 1;
            gt.epoch = c->sk_epoch;
            return launch_gemm_pair(epi, gt, ma, mw.map128, 256, lnch_prefill(c), mh, mx);
        }
    }
    return launch_gemm_pair(epi, gt, ma, mb, bn, lnch_prefill(c), mh, mx);
}

GemmArgs gemm_base(llm_ctx *c, const f16 *A, const f16 *W, int M, int N, int K) {
    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.A = A; g.W = W; g.M = M; g.N = N; g.K = K; g.err = c->err_dev;
    return g;
}

// Prefill-sized ubatch: tensor-core GEMMs and tiled causal attention.  Each
// RMSNorm is fused across two GEMMs: the kernel that last updates h (the
// embedding, or a residual GEMM's epilogue) also writes f16(h * gain) as the
// next GEMM's A operand and per-32-column sums of h^2; that GEMM scales its
// accumulator rows by 1 / sqrt(mean(h^2) + eps) before its own epilogue.
cudaError_t run_large(llm_ctx *c, const UbDev &u) {
    const llm_model *m = c->m;
    const int d = m->d, T = u.T;
    const Launch L = lnch_prefill(c);
    const float eps = m->hp.rms_eps;
    cudaError_t e = timed(c, K_EMBED, [&] {
        return launch_embed(m->token_embd, u.tok, T, d, m->V, c->h, nullptr, c->err_dev, L, m->layers[0].attn_norm,
                            c->x, c->ss32);
    });
    if (e) return e;
    float *hcur = c->h, *sscur = c->ss32;
    f16 *xcur = c->x;
    const TmaMap *axcur = &c->ax;
    int Tc = T;
    // the fused RMSNorm of a GEMM's rows (consumer) / of the next GEMM (producer)
    auto norm_in = [&](GemmArgs &g) { g.row_ss = sscur; g.n_ss = d / 32; g.eps = eps; };
    auto norm_out = [&](GemmArgs &g, const float *gain) { g.gain_next = gain; g.x_next = xcur; g.ss_next = sscur; };
    for (int l = 0; l < m->L; ++l) {
        const LayerW &w = m->layers[l];
        const KvView kv = kv_view(c, l);
        GemmArgs g = gemm_base(c, c->x, w.wqkv, T, m->n_qkv, d);
        norm_in(g);
        g.n_q = m->n_q; g.n_kv = m->n_kv; g.rope = c->rope; g.q_out = c->qb; g.kv = kv; g.pos = u.pos; g.seq = u.seq;
        g.rope_t = c->rope_t; g.rope_n = c->n_ctx;
        if ((e = timed(c, K_GEMM_QKV, [&] { return gemm(c, EPI_QKV, g, c->ax, w.mqkv); }))) return e;
        if (c->attn_tc_ok && c->attn_mode > 0) {
            AttnPrefillTcArgs at;
            at.tiles = u.tiles128; at.n_tiles = u.n_tiles128; at.H = m->H; at.Hkv = m->Hkv; at.head_dim = m->hd;
            at.n_layer = m->L; at.layer = l; at.n_ctx = c->n_ctx; at.n_seq = c->n_seq_max;
            at.o = c->o; at.ldo = m->n_q; at.err = c->err_dev; at.window = c->swa_window;
            const bool pair = c->attn_pair_ok && c->attn_mode == 2;
            if ((e = timed(c, K_ATTN_PREFILL, [&] {
                     return pair ? launch_attn_prefill_pair(at, c->aq, c->akc64, c->avc, L)
                                 : launch_attn_prefill_tc(at, c->aq, c->akc, c->avc, L);
                 })))
                return e;
        } else {
            AttnPrefillArgs at;
            at.q = c->qb; at.kv = kv; at.tiles = u.tiles; at.n_tiles = u.n_tiles; at.o = c->o; at.H = m->H;
            at.err = c->err_dev; at.window = c->swa_window;
            if ((e = timed(c, K_ATTN_PREFILL, [&] { return launch_attn_prefill(at, L); }))) return e;
        }
        g = gemm_base(c, c->o, w.wo, T, d, m->n_q);
        g.hres = c->h; g.ldh = d;
        norm_out(g, w.ffn_norm);                       // x and sums of squares of the MLP's RMSNorm
        if ((e = timed(c, K_GEMM_O, [&] { return gemm(c, EPI_RESID, g, c->ao, w.mo); }))) return e;
        if (l == m->L - 1 && u.out_rows) {
            if ((e = timed(c, K_GATHER, [&] {
                     return launch_gather_rows(c->h, u.out_rows, u.n_out, d, c->h2, nullptr, nullptr, L, c->x, c->x2,
                                               c->ss32, c->ss32b);
                 })))
                return e;
            hcur = c->h2; xcur = c->x2; sscur = c->ss32b; axcur = &c->ax2; Tc = u.n_out;
        }
        if (Tc == 0) break;
        const float *gain_next = l + 1 < m->L ? m->layers[l + 1].attn_norm : m->output_norm;
        if (Tc > 8) {
            g = gemm_base(c, xcur, w.wgu, Tc, 2 * m->F_pad, d);
            norm_in(g);
            g.u_out = c->u; g.ldu = m->F_pad;
            if ((e = timed(c, K_GEMM_GATEUP, [&] { return gemm(c, EPI_SWIGLU, g, *axcur, w.mgu); }))) return e;
            g = gemm_base(c, c->u, w.wdown, Tc, d, m->F_pad);
            g.hres = hcur; g.ldh = d;
            norm_out(g, gain_next);
            if ((e = timed(c, K_GEMM_DOWN, [&] { return gemm(c, EPI_RESID, g, c->au, w.mdown); }))) return e;
        } else {
            // a few rows (the output rows of the last layer): GEMVs with the
            // RMSNorm computed from h in their prologue
            GemvArgs a = gemv_base(c, w.wgu, 2 * m->F_pad, d, Tc, GV_GU);
            a.h = hcur; a.ldh = d; a.gain = w.ffn_norm; a.u_out = c->u; a.ldu = m->F_pad;
            if ((e = timed(c, K_GEMV_GATEUP, [&] { return launch_gemv(PRO_NORM, EPI_SWIGLU, a, L); }))) return e;
            a = gemv_base(c, w.wdown, d, m->F_pad, Tc, GV_DOWN);
            a.x = c->u; a.ldx = m->F_pad; a.hres = hcur; a.ldh_res = d;
            if ((e = timed(c, K_GEMV_DOWN, [&] { return launch_gemv(PRO_BF16, EPI_RESID, a, L); }))) return e;
        }
        if ((e = debug_copy(c, u, l, hcur, Tc))) return e;
    }
    if (Tc == 0) return cudaSuccess;
    float *lg = c->logits + (size_t)u.out_base * m->V;
    if (Tc > 8) {
        GemmArgs g = gemm_base(c, xcur, m->output, Tc, m->V, d);
        norm_in(g);
        g.C = lg; g.ldc = m->V;
        return timed(c, K_GEMM_LMHEAD, [&] { return gemm(c, EPI_STORE, g, *axcur, m->mout); });
    }
    GemvArgs a = gemv_base(c, m->output, m->V, d, Tc, GV_LM);
    a.h = hcur; a.ldh = d; a.gain = m->output_norm; a.out = lg; a.ldo = m->V;
    return timed(c, K_GEMV_LMHEAD, [&] { return launch_gemv(PRO_NORM, EPI_STORE, a, L); });
}

cudaError_t run_ubatch(llm_ctx *c, const UbDev &u) {
    return u.T <= c->gemv_max_rows ? run_small(c, u) : run_large(c, u);
}

int32_t ensure_logits(llm_ctx *c, int rows) {
    if (rows <= c->logits_cap) return LLM_OK;
    int cap = c->logits_cap ? c->logits_cap : 8;
    while (cap < rows) cap *= 2;
    cudaStreamSynchronize(c->stream);
    if (c->logits) cudaFree(c->logits);
    if (c->argmax_dev) cudaFree(c->argmax_dev);
    if (c->argmax_host) cudaFreeHost(c->argmax_host);
    c->logits = nullptr; c->argmax_dev = nullptr; c->argmax_host = nullptr; c->logits_cap = 0;
    if (cudaMalloc(&c->logits, (size_t)cap * c->m->V * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&c->argmax_dev, (size_t)cap * sizeof(int)) != cudaSuccess ||
        cudaHostAlloc((void **)&c->argmax_host, (size_t)cap * sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        return fail(c, LLM_ERR_ALLOC, "logits allocation failed");
    }
    c->logits_cap = cap;
    // captured graphs wrote to the old logits buffer
    drop_graphs(c);
    return LLM_OK;
}

int *staging(llm_ctx *c, size_t ints) {
    const int s = c->meta_slot;
    c->meta_slot ^= 1;
    cudaEventSynchronize(c->meta_ev[s]);
    if (c->meta_host_cap[s] < ints) {
        if (c->meta_host[s]) cudaFreeHost(c->meta_host[s]);
        size_t cap = align_up(ints, 4096);
        if (cudaHostAlloc((void **)&c->meta_host[s], cap * sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
            c->meta_host[s] = nullptr; c->meta_host_cap[s] = 0;
            return nullptr;
        }
        c->meta_host_cap[s] = cap;
    }
    return c->meta_host[s];
}

// Capture (once) and launch the decode graph for T rows whose metadata sits in dec_dev.
cudaError_t launch_decode_graph(llm_ctx *c, int T) {
    if (!c->graph[T]) {
        UbDev u;
        memset(&u, 0, sizeof u);
        u.tok = c->dec_dev + DEC_TOK; u.pos = c->dec_dev + DEC_POS; u.seq = c->dec_dev + DEC_SEQ;
        u.T = T; u.n_out = T; u.out_base = 0; u.ub_index = 1 << 30;
        cudaGraph_t gr = nullptr;
        const int64_t before = c->launches;
        cudaError_t e = cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal);
        if (e) return e;
        cudaError_t er = run_small(c, u);
        e = cudaStreamEndCapture(c->stream, &gr);
        if (er) { if (gr) cudaGraphDestroy(gr); return er; }
        if (e) return e;
        e = cudaGraphInstantiate(&c->graph[T], gr, 0);
        cudaGraphDestroy(gr);
        if (e) { c->graph[T] = nullptr; return e; }
        c->graph_kernels[T] = c->launches - before;
        c->launches = before;
    }
    c->launches += c->graph_kernels[T];
    return cudaGraphLaunch(c->graph[T], c->stream);
}

// The attention tiles of ubatch rows [s0, s1): runs of at most max_rows rows
// of one sequence (consecutive positions); kv_ready is the sequence's first
// position in the ubatch, below which its keys were cached before it.
int build_tiles(const std::vector<int32_t> &seq, const std::vector<int32_t> &pos, int s0, int s1, int max_rows,
                AttnTile *out) {
    int t = 0;
    for (int i = s0; i < s1;) {
        int j = i;
        while (j < s1 && seq[j] == seq[i] && j - i < max_rows) ++j;
        int ready = pos[i];
        for (int q = s0; q < i; ++q)
            if (seq[q] == seq[i]) { ready = pos[q]; break; }
        if (out) out[t] = AttnTile{i - s0, j - i, seq[i], pos[i], ready};
        ++t;
        i = j;
    }
    return t;
}

}  // namespace

extern "C" int32_t llm_decode(llm_ctx *c, const llm_batch *b) {
    if (!c || !b) return fail(c, LLM_ERR_INVALID, "ctx or batch is NULL");
    const llm_model *m = c->m;
    BatchPlan p;
    const int rc = plan_batch(*b, m->V, c->n_ctx, c->n_seq_max, c->n_ubatch, c->seq_next, p);
    if (rc != LLM_OK) { c->last_error = p.error; return rc; }
    if (ensure_logits(c, p.n_outputs) != LLM_OK) return LLM_ERR_ALLOC;
    const bool dev_tok = (b->flags & LLM_BATCH_TOKENS_ON_DEVICE) != 0;

    // decode step: replay the captured graph
    if (c->use_graphs && !c->dbg && !c->ktime && p.n <= c->gemv_max_rows && p.n_outputs == p.n) {
        const int T = p.n;
        const int s = c->dec_slot;
        c->dec_slot = (s + 1) & 3;
        CK(cudaEventSynchronize(c->dec_ev[s]));
        int *hs = c->dec_host[s];
        for (int i = 0; i < T; ++i) {
            hs[DEC_TOK + i] = dev_tok ? 0 : p.tok[i];
            hs[DEC_POS + i] = p.pos[i];
            hs[DEC_SEQ + i] = p.seq[i];
        }
        CK(cudaMemcpyAsync(c->dec_dev + DEC_POS, hs + DEC_POS, 16 * sizeof(int), cudaMemcpyHostToDevice, c->stream));
        if (dev_tok) CK(cudaMemcpyAsync(c->dec_dev + DEC_TOK, b->token, T * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
        else CK(cudaMemcpyAsync(c->dec_dev + DEC_TOK, hs + DEC_TOK, T * sizeof(int), cudaMemcpyHostToDevice, c->stream));
        CK(cudaEventRecord(c->dec_ev[s], c->stream));
        CK(launch_decode_graph(c, T));
    } else {
        // metadata of every ubatch in one upload: tok | pos | seq | out_rows | tiles
        const int nub = (int)p.ub_start.size() - 1;
        std::vector<size_t> off_tok(nub), off_rows(nub), off_tiles(nub), off_tiles128(nub);
        std::vector<int> n_tiles(nub), n_tiles128(nub), n_out(nub);
        constexpr size_t TILE_INTS = sizeof(AttnTile) / sizeof(int);
        size_t ints = 3 * (size_t)p.n;
        for (int k = 0; k < nub; ++k) {
            const int s0 = p.ub_start[k], s1 = p.ub_start[k + 1];
            int no = 0;
            for (int i = s0; i < s1; ++i) no += p.out[i];
            n_out[k] = no;
            n_tiles[k] = build_tiles(p.seq, p.pos, s0, s1, 64, nullptr);
            n_tiles128[k] = build_tiles(p.seq, p.pos, s0, s1, 128, nullptr);
            off_rows[k] = ints; ints += no;
            ints = align_up(ints, 4);
            off_tiles[k] = ints; ints += (size_t)n_tiles[k] * TILE_INTS;
            off_tiles128[k] = ints; ints += (size_t)n_tiles128[k] * TILE_INTS;
        }
        if (c->meta_cap < ints) {
            CK(cudaStreamSynchronize(c->stream));
            if (c->meta_dev) cudaFree(c->meta_dev);
            c->meta_dev = nullptr;
            const size_t cap = align_up(ints, 4096);
            if (cudaMalloc(&c->meta_dev, cap * sizeof(int)) != cudaSuccess) {
                cudaGetLastError();
                c->meta_cap = 0;
                return fail(c, LLM_ERR_ALLOC, "metadata allocation failed");
            }
            c->meta_cap = cap;
        }
        int *hs = staging(c, ints);
        if (!hs) return fail(c, LLM_ERR_ALLOC, "pinned staging allocation failed");
        const int slot = c->meta_slot ^ 1;
        const int n = p.n;
        for (int i = 0; i < n; ++i) {
            hs[i] = dev_tok ? 0 : p.tok[i];
            hs[n + i] = p.pos[i];
            hs[2 * n + i] = p.seq[i];
        }
        for (int k = 0; k < nub; ++k) {
            const int s0 = p.ub_start[k], s1 = p.ub_start[k + 1];
            int *rows = hs + off_rows[k];
            int r = 0;
            for (int i = s0; i < s1; ++i) if (p.out[i]) rows[r++] = i - s0;
            build_tiles(p.seq, p.pos, s0, s1, 64, reinterpret_cast<AttnTile *>(hs + off_tiles[k]));
            build_tiles(p.seq, p.pos, s0, s1, 128, reinterpret_cast<AttnTile *>(hs + off_tiles128[k]));
        }
        CK(cudaMemcpyAsync(c->meta_dev, hs, ints * sizeof(int), cudaMemcpyHostToDevice, c->stream));
        CK(cudaEventRecord(c->meta_ev[slot], c->stream));
        int out_base = 0;
        for (int k = 0; k < nub; ++k) {
            const int s0 = p.ub_start[k], s1 = p.ub_start[k + 1];
            UbDev u;
            u.tok = dev_tok ? b->token + s0 : c->meta_dev + s0;
            u.pos = c->meta_dev + n + s0;
            u.seq = c->meta_dev + 2 * n + s0;
            u.T = s1 - s0;
            u.n_out = n_out[k];
            u.out_rows = (n_out[k] == u.T) ? nullptr : c->meta_dev + off_rows[k];
            u.tiles = reinterpret_cast<const AttnTile *>(c->meta_dev + off_tiles[k]);
            u.n_tiles = n_tiles[k];
            u.tiles128 = reinterpret_cast<const AttnTile *>(c->meta_dev + off_tiles128[k]);
            u.n_tiles128 = n_tiles128[k];
            u.out_base = out_base;
            u.ub_index = k;
            out_base += n_out[k];
            CK(run_ubatch(c, u));
        }
    }
    for (int i = 0; i < p.n; ++i) c->seq_next[p.seq[i]] = p.pos[i] + 1;
    c->out_index = p.out_index;
    c->n_outputs = p.n_outputs;
    return LLM_OK;
}

extern "C" const float *llm_get_logits(llm_ctx *c, int32_t *n_outputs) {
    if (!c) return nullptr;
    if (n_outputs) *n_outputs = c->n_outputs;
    return c->n_outputs ? c->logits : nullptr;
}

extern "C" const float *llm_get_logits_ith(llm_ctx *c, int32_t i) {
    if (!c || c->n_outputs == 0) return nullptr;
    int r;
    if (i < 0) {
        r = c->n_outputs + i;
        if (r < 0) return nullptr;
    } else {
        if (i >= (int)c->out_index.size()) return nullptr;
        r = c->out_index[i];
        if (r < 0) return nullptr;
    }
    return c->logits + (size_t)r * c->m->V;
}

extern "C" int32_t llm_get_argmax(llm_ctx *c, int32_t *out, int32_t capacity) {
    if (!c || !out) return fail(c, LLM_ERR_INVALID, "ctx or out is NULL");
    if (capacity < c->n_outputs) return fail(c, LLM_ERR_INVALID, "capacity below n_outputs");
    if (c->n_outputs == 0) return 0;
    CK(launch_argmax(c->logits, c->n_outputs, c->m->V, c->argmax_dev, lnch(c)));
    CK(cudaMemcpyAsync(c->argmax_host, c->argmax_dev, c->n_outputs * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    memcpy(out, c->argmax_host, c->n_outputs * sizeof(int));
    return c->n_outputs;
}

static bool sampling_ok(const llm_sampling *s, int V) {
    return s && (s->temperature <= 0.f ||
                 (s->top_k >= 1 && s->top_k <= 1024 && s->top_k <= V && s->repeat_penalty > 0.f &&
                  s->penalty_last_n >= 0 && s->top_p > 0.f && s->min_p < 1.f));
}

static SampleParams sample_params(const llm_sampling *s) {
    return SampleParams{s->temperature, s->top_k, s->top_p, s->min_p, s->repeat_penalty, s->penalty_last_n};
}

extern "C" int32_t llm_sample(llm_ctx *c, const llm_sampling *s, const float *u, const int32_t *history,
                              int32_t n_history, int32_t *out, int32_t capacity) {
    if (!c || !s || !out || n_history < 0 || (n_history > 0 && !history))
        return fail(c, LLM_ERR_INVALID, "invalid sample arguments");
    if (!sampling_ok(s, c->m->V)) return fail(c, LLM_ERR_INVALID, "invalid sampling parameters");
    if (c->m->V > SAMPLE_MAX_VOCAB) return fail(c, LLM_ERR_INVALID, "n_vocab too large for sampling");
    const int n = c->n_outputs;
    if (capacity < n) return fail(c, LLM_ERR_INVALID, "capacity below n_outputs");
    if (n == 0) return 0;
    if (s->temperature > 0.f && !u) return fail(c, LLM_ERR_INVALID, "uniforms are NULL");
    for (int i = 0; s->temperature > 0.f && i < n; ++i)
        if (!(u[i] >= 0.f && u[i] < 1.f)) return fail(c, LLM_ERR_INVALID, "uniforms must lie in [0, 1)");
    const size_t need = align_up((size_t)n * sizeof(float), 256) + (size_t)(n_history + 1) * sizeof(int32_t);
    if (need > c->samp_cap) {
        CK(cudaStreamSynchronize(c->stream));
        if (c->samp_dev) cudaFree(c->samp_dev);
        c->samp_dev = nullptr; c->samp_cap = 0;
        if (cudaMalloc(&c->samp_dev, need) != cudaSuccess) {
            cudaGetLastError();
            return fail(c, LLM_ERR_ALLOC, "sampling buffer allocation failed");
        }
        c->samp_cap = need;
    }
    float *u_dev = static_cast<float *>(c->samp_dev);
    int *h_dev = reinterpret_cast<int *>(static_cast<char *>(c->samp_dev) + align_up((size_t)n * sizeof(float), 256));
    if (s->temperature > 0.f) CK(cudaMemcpyAsync(u_dev, u, n * sizeof(float), cudaMemcpyHostToDevice, c->stream));
    if (n_history > 0)
        CK(cudaMemcpyAsync(h_dev, history, n_history * sizeof(int32_t), cudaMemcpyHostToDevice, c->stream));
    CK(launch_sample(c->logits, n, c->m->V, sample_params(s), u_dev, h_dev, n_history, c->argmax_dev, lnch(c)));
    CK(cudaMemcpyAsync(c->argmax_host, c->argmax_dev, n * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    memcpy(out, c->argmax_host, n * sizeof(int));
    return n;
}

extern "C" int32_t llm_generate(llm_ctx *c, int32_t seq_id, int32_t n_steps, int32_t *tokens_out) {
    if (!c || !tokens_out || n_steps < 1) return fail(c, LLM_ERR_INVALID, "invalid generate arguments");
    if (seq_id < 0 || seq_id >= c->n_seq_max) return fail(c, LLM_ERR_INVALID, "invalid seq_id");
    if (c->n_outputs < 1) return fail(c, LLM_ERR_INVALID, "no logits to start from");
    if (c->seq_next[seq_id] + n_steps > c->n_ctx) { c->last_error = "sequence would pass n_ctx"; return LLM_NO_KV_ROOM; }
    if (c->gemv_max_rows < 1) return fail(c, LLM_ERR_INVALID, "decode kernels disabled");
    if (n_steps > c->gen_cap) {
        CK(cudaStreamSynchronize(c->stream));
        if (c->gen_tokens) cudaFree(c->gen_tokens);
        c->gen_tokens = nullptr;
        c->gen_cap = 0;
        if (c->gen_graph) { cudaGraphExecDestroy(c->gen_graph); c->gen_graph = nullptr; }
        int cap = 256;
        while (cap < n_steps) cap *= 2;
        if (cudaMalloc(&c->gen_tokens, cap * sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return fail(c, LLM_ERR_ALLOC, "generate buffer allocation failed");
        }
        c->gen_cap = cap;
    }
    const llm_model *m = c->m;
    const int s = c->dec_slot;
    c->dec_slot = (s + 1) & 3;
    CK(cudaEventSynchronize(c->dec_ev[s]));
    int *hs = c->dec_host[s];
    memset(hs, 0, DEC_INTS * sizeof(int));
    hs[DEC_POS] = c->seq_next[seq_id];
    hs[DEC_SEQ] = seq_id;
    hs[DEC_STEP] = 0;
    hs[DEC_NSTEPS] = n_steps;
    CK(cudaMemcpyAsync(c->dec_dev, hs, DEC_INTS * sizeof(int), cudaMemcpyHostToDevice, c->stream));
    CK(cudaEventRecord(c->dec_ev[s], c->stream));
    const Launch L = lnch(c);
    int *step = c->dec_dev + DEC_STEP, *nst = c->dec_dev + DEC_NSTEPS;
    int *tok = c->dec_dev + DEC_TOK, *pos = c->dec_dev + DEC_POS;
    // the first token comes from the last output row of the previous decode
    CK(launch_argmax_feed(c->logits + (size_t)(c->n_outputs - 1) * m->V, m->V, c->gen_tokens, step, nst, tok, pos,
                          0, L));
    UbDev u;
    memset(&u, 0, sizeof u);
    u.tok = tok; u.pos = pos; u.seq = c->dec_dev + DEC_SEQ;
    u.T = 1; u.n_out = 1; u.out_base = 0; u.ub_index = 1 << 30;
    if (c->use_graphs && !c->ktime) {
        if (!c->gen_graph) {
            // one step = decode the fed token (logits row 0) + feed its argmax back
            cudaGraph_t gr = nullptr;
            const int64_t before = c->launches;
            CK(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
            cudaError_t er = run_small(c, u);
            if (!er) er = launch_argmax_feed(c->logits, m->V, c->gen_tokens, step, nst, tok, pos, 1, L);
            const cudaError_t e2 = cudaStreamEndCapture(c->stream, &gr);
            if (er || e2) {
                if (gr) cudaGraphDestroy(gr);
                return fail(c, LLM_ERR_COMPUTE, "generate capture", er ? er : e2);
            }
            const cudaError_t e3 = cudaGraphInstantiate(&c->gen_graph, gr, 0);
            cudaGraphDestroy(gr);
            if (e3) { c->gen_graph = nullptr; return fail(c, LLM_ERR_COMPUTE, "generate instantiate", e3); }
            c->gen_graph_kernels = c->launches - before;
            c->launches = before;
        }
        for (int i = 0; i < n_steps; ++i) {
            c->launches += c->gen_graph_kernels;
            CK(cudaGraphLaunch(c->gen_graph, c->stream));
        }
    } else {
        for (int i = 0; i < n_steps; ++i) {
            CK(run_small(c, u));
            CK(timed(c, K_ARGMAX, [&] { return launch_argmax_feed(c->logits, m->V, c->gen_tokens, step, nst, tok, pos, 1, L); }));
        }
    }
    c->n_outputs = 1;
    CK(cudaMemcpyAsync(tokens_out, c->gen_tokens, n_steps * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
    c->seq_next[seq_id] += n_steps;
    c->out_index.assign(1, 0);
    return LLM_OK;
}

extern "C" int32_t llm_seq_pos_max(llm_ctx *c, int32_t seq_id) {
    if (!c || seq_id < 0 || seq_id >= c->n_seq_max) return LLM_ERR_INVALID;
    return c->seq_next[seq_id] - 1;
}

extern "C" int32_t llm_seq_clear(llm_ctx *c, int32_t seq_id) {
    if (!c || seq_id < 0 || seq_id >= c->n_seq_max) return LLM_ERR_INVALID;
    c->seq_next[seq_id] = 0;
    return LLM_OK;
}

extern "C" int32_t llm_seq_shift(llm_ctx *c, int32_t seq_id, int32_t p0, int32_t n_discard) {
    if (!c || seq_id < 0 || seq_id >= c->n_seq_max) return fail(c, LLM_ERR_INVALID, "bad context or sequence");
    const int end = c->seq_next[seq_id];
    if (p0 < 0 || n_discard < 1 || p0 + n_discard > end)
        return fail(c, LLM_ERR_INVALID, "shift range outside the sequence's positions");
    const llm_model *m = c->m;
    CK(launch_kv_shift(kv_view(c, 0), m->L, seq_id, p0, n_discard, end, c->rope, Launch{c->stream, false, &c->launches}));
    c->seq_next[seq_id] = end - n_discard;
    return LLM_OK;
}

extern "C" int32_t llm_synchronize(llm_ctx *c) {
    if (!c) return LLM_ERR_INVALID;
    CK(cudaStreamSynchronize(c->stream));
    uint32_t flag = 0;
    CK(cudaMemcpy(&flag, c->err_dev, sizeof flag, cudaMemcpyDeviceToHost));
    if (flag) {
        CK(cudaMemset(c->err_dev, 0, sizeof(uint32_t)));
        std::string msg = "kernel error flag 0x" + [&] { char b[16]; snprintf(b, sizeof b, "%x", flag); return std::string(b); }() +
                          " raised:";
        if (flag & ERRF_BAD_TOKEN) msg += " a token id outside [0, n_vocab);";
        if (flag & ERRF_BAD_INDEX) msg += " a sequence, position or row index out of range;";
        if (flag & ERRF_WAIT_TIMEOUT) msg += " a bounded wait timed out;";
        if (flag & ERRF_F16_RANGE) msg += " an activation narrowed to fp16 was not finite or beyond +-65504;";
        c->last_error = msg;
        return LLM_ERR_COMPUTE;
    }
    return LLM_OK;
}

extern "C" const char *llm_last_error(const llm_ctx *c) {
    return c ? c->last_error.c_str() : g_create_error.c_str();
}

extern "C" int32_t llm_debug_hidden(llm_ctx *c, float *dst, int32_t max_rows, int32_t max_ubatches) {
    if (!c) return LLM_ERR_INVALID;
    if (dst && (max_rows < 1 || max_ubatches < 1)) return fail(c, LLM_ERR_INVALID, "invalid debug buffer");
    c->dbg = dst; c->dbg_rows = max_rows; c->dbg_ub = max_ubatches;
    return LLM_OK;
}

extern "C" int32_t llm_set_option(llm_ctx *c, const char *key, int32_t value) {
    if (!c || !key) return LLM_ERR_INVALID;
    if (!strcmp(key, "graphs")) { c->use_graphs = value != 0; return LLM_OK; }
    if (!strcmp(key, "pdl") || !strcmp(key, "pdl_attn") || !strcmp(key, "pdl_prefill")) {
        (!strcmp(key, "pdl") ? c->use_pdl : !strcmp(key, "pdl_attn") ? c->use_pdl_attn : c->use_pdl_prefill) = value != 0;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemm")) {
        if (value < 2 || value > 4)
            return fail(c, LLM_ERR_INVALID,
                        "gemm kernel must be 2 (CTA pairs, persistent past one wave), 3 (persistent) or 4 (stream-K)");
        c->gemm_kernel = value;
        return LLM_OK;
    }
    static const char *const ks_keys[5] = {"ksplit_qkv", "ksplit_o", "ksplit_gateup", "ksplit_down", "ksplit_lm"};
    for (int i = 0; i < 5; ++i)
        if (!strcmp(key, ks_keys[i])) {
            if (value < 0 || value > 64) return fail(c, LLM_ERR_INVALID, "ksplit must be 0..64");
            c->ksplit_opt[i] = value;
            drop_graphs(c);
            return LLM_OK;
        }
    if (!strcmp(key, "attn_split")) {    // one-row decode attention splits; 0 = auto
        if (value < 0 || value > c->attn_split_cap) return fail(c, LLM_ERR_INVALID, "attn_split out of range");
        c->attn_split[1] = value ? value : attn_pick_split(c->m, 1, c->n_ctx);
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "attn_split_rows")) {  // decode attention splits of 2-8-row steps; 0 = auto
        if (value < 0 || value > c->attn_split_cap) return fail(c, LLM_ERR_INVALID, "attn_split_rows out of range");
        for (int T = 2; T <= 8; ++T) c->attn_split[T] = value ? value : attn_pick_split(c->m, T, c->n_ctx);
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "kv_fp8")) {
        // the cache element type; only while every sequence is empty
        for (int s = 0; s < c->n_seq_max; ++s)
            if (c->seq_next[s] != 0) return fail(c, LLM_ERR_INVALID, "kv_fp8 needs an empty cache (llm_seq_clear)");
        const bool want = value != 0;
        if (want == c->kv_fp8) return LLM_OK;
        const size_t bytes = c->kv_elems * (want ? 1 : sizeof(f16));
        cudaStreamSynchronize(c->stream);
        cudaFree(c->kc); cudaFree(c->vc);
        c->kc = c->vc = nullptr;
        if (cudaMalloc((void **)&c->kc, bytes) != cudaSuccess || cudaMalloc((void **)&c->vc, bytes) != cudaSuccess ||
            cudaMemsetAsync(c->kc, 0, bytes, c->stream) != cudaSuccess ||
            cudaMemsetAsync(c->vc, 0, bytes, c->stream) != cudaSuccess) {
            cudaGetLastError();
            return fail(c, LLM_ERR_ALLOC, "KV cache reallocation failed");
        }
        c->kv_fp8 = want;
        make_attn_maps(c);
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "attn_prefill")) {
        if (value < 0 || value > 2)
            return fail(c, LLM_ERR_INVALID, "attn_prefill must be 0 (mma.sync), 1 (tcgen05, one CTA) or 2 (tcgen05, CTA pairs)");
        c->attn_mode = value;
        return LLM_OK;
    }
    if (!strcmp(key, "swa_window")) {
        if (value < 0) return fail(c, LLM_ERR_INVALID, "swa_window must be >= 0");
        c->swa_window = value;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemm_split_k")) {
        if (value < 0 || value > 1) return fail(c, LLM_ERR_INVALID, "gemm_split_k must be 0 or 1");
        c->split_k = value != 0;
        return LLM_OK;
    }
    if (!strcmp(key, "gemm_resid_tma")) {
        if (value < 0 || value > 1) return fail(c, LLM_ERR_INVALID, "gemm_resid_tma must be 0 or 1");
        c->resid_tma = value != 0;
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_prefetch2_kb")) {
        if (value < 0 || value > 4096) return fail(c, LLM_ERR_INVALID, "gemv_prefetch2_kb must be 0..4096");
        c->stream_pf2_kb = value;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_prefetch_kb")) {
        if (value < 0 || value > 4096) return fail(c, LLM_ERR_INVALID, "gemv_prefetch_kb must be 0..4096");
        c->stream_pf_kb = value;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_attn_smem_kb")) {
        if (value != 0 && (value < 120 || value > 224)) return fail(c, LLM_ERR_INVALID, "gemv_attn_smem_kb must be 0 or 120..224");
        if (value && !(gemv_stream_ok(EPI_QKV, c->m->n_qkv, c->m->d, c->m->num_sms, value) &&
                       gemv_stream_ok(EPI_RESID, c->m->d, c->m->n_q, c->m->num_sms, value)))
            return fail(c, LLM_ERR_INVALID, "gemv_attn_smem_kb too small for these shapes");
        c->stream_attn_kb = value;
        c->stream_q8 = q8_plans_ok(c);
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_stage_kb")) {
        if (value != 0 && (value < 16 || value > 128)) return fail(c, LLM_ERR_INVALID, "gemv_stage_kb must be 0 or 16..128");
        c->stream_stage_kb = value;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_q8")) {
        c->use_q8 = value != 0;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_stream")) {
        c->use_stream = value != 0;
        drop_graphs(c);
        return LLM_OK;
    }
    if (!strcmp(key, "gemv_path_max_rows")) {
        if (value < 0 || value > 8) return fail(c, LLM_ERR_INVALID, "gemv_path_max_rows must be 0..8");
        c->gemv_max_rows = value;
        return LLM_OK;
    }
    return fail(c, LLM_ERR_INVALID, "unknown option");
}

extern "C" int64_t llm_kernel_launches(const llm_ctx *c) { return c ? c->launches : 0; }

static void kt_collect(llm_ctx *c) {
    if (c->kt_pending.empty()) return;
    cudaStreamSynchronize(c->stream);
    for (auto &r : c->kt_pending) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
            c->kt_ms[r.id] += ms;
            c->kt_n[r.id] += 1;
        }
        c->kt_pool.push_back(r.a);
        c->kt_pool.push_back(r.b);
    }
    c->kt_pending.clear();
    cudaGetLastError();
}

extern "C" int32_t llm_kernel_timing(llm_ctx *c, int32_t enable) {
    if (!c) return LLM_ERR_INVALID;
    kt_collect(c);
    c->ktime = enable != 0;
    for (int k = 0; k < K_COUNT; ++k) { c->kt_ms[k] = 0.0; c->kt_n[k] = 0; }
    return LLM_OK;
}

extern "C" int32_t llm_kernel_time(llm_ctx *c, int32_t kernel, double *total_ms, int64_t *count,
                                   const char **name) {
    if (!c || kernel < 0 || kernel >= K_COUNT) return LLM_ERR_INVALID;
    kt_collect(c);
    if (total_ms) *total_ms = c->kt_ms[kernel];
    if (count) *count = c->kt_n[kernel];
    if (name) *name = KNAME[kernel];
    return LLM_OK;
}

// ============================================================== single-kernel entry points

extern "C" int32_t llm_op_gemv(const void *W, const void *x, float *y, int32_t N, int32_t K, int32_t T,
                               int32_t ksplit, void *scratch, int64_t scratch_bytes, void *stream) {
    if (!W || !x || !y || !scratch || T < 1 || T > 8 || N < 64 || N % 64 || K < 128 || K % 128)
        return LLM_ERR_INVALID;
    cudaError_t e = init_kernel_attributes();
    if (e) return LLM_ERR_COMPUTE;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ksplit <= 0) ksplit = gemv_pick_split(N, K, T, sms);
    if (K % (128 * ksplit)) return LLM_ERR_INVALID;
    const size_t need = (size_t)ksplit * N * 8 * sizeof(float) + (size_t)(N / 64) * sizeof(unsigned);
    if ((size_t)scratch_bytes < need) return LLM_ERR_INVALID;
    GemvArgs a;
    memset(&a, 0, sizeof a);
    a.W = (const f16 *)W; a.N = N; a.K = K; a.T = T; a.ksplit = ksplit;
    a.x = (const f16 *)x; a.ldx = K;
    a.part = (float *)scratch;
    a.counters = (unsigned *)((char *)scratch + (size_t)ksplit * N * 8 * sizeof(float));
    a.out = y; a.ldo = N;
    e = launch_gemv(PRO_BF16, EPI_STORE, a, Launch{(cudaStream_t)stream, false, nullptr});
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int32_t llm_op_quantize_q8_0(const void *W, int32_t N, int32_t K, void *out, void *stream) {
    if (!W || !out || N < 1 || K < 256 || K % 256) return LLM_ERR_INVALID;
    // write_back is off: W is only read
    const cudaError_t e = launch_quantize_q8_0((f16 *)W, N, K, (uint8_t *)out, false, (cudaStream_t)stream);
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int32_t llm_op_wait_check(int32_t arrive, int32_t polls, uint32_t *err, void *stream) {
    if (!err || polls < 1) return LLM_ERR_INVALID;
    return launch_wait_check(arrive, (uint32_t)polls, err, (cudaStream_t)stream) ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int32_t llm_op_gemv_q8_0(const void *Wq, const void *x, float *y, int32_t N, int32_t K, void *stream) {
    if (!Wq || !x || !y) return LLM_ERR_INVALID;
    if (init_kernel_attributes()) return LLM_ERR_COMPUTE;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (!gemv_stream_ok(EPI_STORE, N, K, sms, 0, true)) return LLM_ERR_INVALID;
    GemvArgs a;
    memset(&a, 0, sizeof a);
    a.W8 = (const uint8_t *)Wq; a.N = N; a.K = K; a.T = 1;
    a.x = (const f16 *)x; a.ldx = K;
    a.out = y; a.ldo = N;
    const cudaError_t e = launch_gemv_stream(PRO_BF16, EPI_STORE, a, sms, 0, Launch{(cudaStream_t)stream, false, nullptr});
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int32_t llm_op_gemm(const void *A, const void *W, float *C, int32_t M, int32_t N, int32_t K,
                               int32_t kernel, void *stream) {
    if (!A || !W || !C || M < 1 || N % 128 || K % 64 || K < 64 || kernel < 0 || kernel > 7) return LLM_ERR_INVALID;
    if (init_kernel_attributes()) return LLM_ERR_COMPUTE;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.A = (const f16 *)A; g.W = (const f16 *)W; g.M = M; g.N = N; g.K = K; g.C = C; g.ldc = N;
    const Launch L{(cudaStream_t)stream, false, nullptr};
    const int mc = gemm_pair_max_clusters();
    if (kernel == 7 || (kernel == 0 && N % 256 == 0)) {
        // stream-K: partial slots and flags for this call only
        if (N % 256) return LLM_ERR_INVALID;
        static unsigned epoch = 0;
        if (++epoch == 0) epoch = 1;
        TmaMap ma, mb;
        if (!make_operand_map(&ma, (const f16 *)A, M, K, 128) || !make_operand_map(&mb, (const f16 *)W, N, K, 128))
            return LLM_ERR_COMPUTE;
        cudaStream_t st = (cudaStream_t)stream;
        float *ws = nullptr;
        unsigned *flags = nullptr;
        if (cudaMallocAsync((void **)&ws, gemm_pair_sk_ws_floats(mc) * sizeof(float), st) != cudaSuccess ||
            cudaMallocAsync((void **)&flags, (size_t)2 * mc * sizeof(unsigned), st) != cudaSuccess) {
            cudaGetLastError();
            if (ws) cudaFreeAsync(ws, st);
            return LLM_ERR_ALLOC;
        }
        cudaError_t e = cudaMemsetAsync(flags, 0, (size_t)2 * mc * sizeof(unsigned), st);
        if (!e) e = launch_gemm_pair_sk(EPI_STORE, g, ma, mb, ws, flags, epoch, L);
        cudaFreeAsync(ws, st);
        cudaFreeAsync(flags, st);
        return e ? LLM_ERR_COMPUTE : LLM_OK;
    }
    const int bn = kernel == 0 ? gemm_pair_pick_bn(M, N, mc) : 64 * ((kernel - 1) % 3 + 2);
    if (!bn || N % bn) return LLM_ERR_INVALID;
    TmaMap ma, mb;
    if (!make_operand_map(&ma, (const f16 *)A, M, K, 128) || !make_operand_map(&mb, (const f16 *)W, N, K, bn / 2))
        return LLM_ERR_COMPUTE;
    const bool persist = kernel >= 4 || (kernel == 0 && (long long)((M + 255) / 256) * (N / bn) > mc);
    const cudaError_t e = persist ? launch_gemm_pair_persist(EPI_STORE, g, ma, mb, bn, L)
                                  : launch_gemm_pair(EPI_STORE, g, ma, mb, bn, L);
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int32_t llm_op_sample(const float *logits, int32_t n_rows, int32_t n_vocab, const llm_sampling *s,
                                 const float *u, const int32_t *history, int32_t n_history, int32_t *out,
                                 void *stream) {
    if (!logits || !out || n_rows < 1 || n_vocab < 4 || n_vocab % 4 || (reinterpret_cast<uintptr_t>(logits) & 15u) ||
        n_history < 0 || (n_history > 0 && !history) ||
        !sampling_ok(s, n_vocab) || (s->temperature > 0.f && !u) || n_vocab > SAMPLE_MAX_VOCAB)
        return LLM_ERR_INVALID;
    if (init_kernel_attributes()) return LLM_ERR_COMPUTE;
    const cudaError_t e = launch_sample(logits, n_rows, n_vocab, sample_params(s), u, history, n_history, out,
                                        Launch{(cudaStream_t)stream, false, nullptr});
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}

extern "C" int64_t llm_op_attn_decode_scratch_bytes(int32_t T, int32_t H, int32_t hd, int32_t n_split) {
    // split partials, then 8 * H counters, then one error word
    return (int64_t)(attn_decode_scratch_floats(T, H, hd, n_split) * sizeof(float) +
                     ((size_t)8 * H + 1) * sizeof(unsigned));
}

namespace llm {
// Shape checks shared by the standalone decode-attention entry points; null
// when the arguments are acceptable, else the reason.
const char *attn_decode_args_error(const void *q, const void *k, const void *v, const void *pos, const void *seq,
                                   const void *o, int T, int H, int Hkv, int hd, int n_ctx, int n_seq, int n_split) {
    if (!q || !k || !v || !pos || !seq || !o) return "a pointer is NULL";
    if (T < 1 || T > 8) return "T must be 1..8";
    if (hd != 32 && hd != 64 && hd != 128) return "head_dim must be 32, 64 or 128";
    if (Hkv < 1 || H < 1 || H % Hkv) return "n_head must be a positive multiple of n_head_kv";
    const int G = H / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return "n_head / n_head_kv must be 1, 2, 4 or 8";
    if (n_ctx < 1 || n_seq < 1) return "n_ctx and n_seq must be positive";
    if (n_split < 1 || n_split > ATTN_DECODE_MAX_SPLIT) return "n_split must be 1..128";
    return nullptr;
}

// Reads the kernel's error word after the stream has run the launch: a row
// whose position lies outside [0, n_ctx) or whose sequence lies outside
// [0, n_seq) was skipped and is reported as LLM_ERR_COMPUTE.
int32_t attn_decode_check(const char *who, uint32_t *err_dev, cudaStream_t st) {
    uint32_t flag = 0;
    cudaError_t e = cudaMemcpyAsync(&flag, err_dev, sizeof flag, cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    std::string msg = who;
    if (e) {
        msg += ": launch failed: ";
        msg += cudaGetErrorString(e);
        set_global_error(msg.c_str());
        return LLM_ERR_COMPUTE;
    }
    if (flag) {
        msg += ": a row's position is outside [0, n_ctx) or its sequence outside [0, n_seq); that row's output is zero";
        set_global_error(msg.c_str());
        return LLM_ERR_COMPUTE;
    }
    return LLM_OK;
}
}  // namespace llm

extern "C" int32_t llm_op_attn_decode(const float *q, const void *k_cache, const void *v_cache, const int32_t *pos,
                                      const int32_t *seq, void *o, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                      int32_t n_ctx, int32_t n_seq, int32_t n_split, void *scratch,
                                      int64_t scratch_bytes, void *stream) {
    if (const char *why = attn_decode_args_error(q, k_cache, v_cache, pos, seq, o, T, H, Hkv, hd, n_ctx, n_seq, n_split)) {
        set_global_error((std::string("llm_op_attn_decode: ") + why).c_str());
        return LLM_ERR_INVALID;
    }
    if (!scratch || scratch_bytes < llm_op_attn_decode_scratch_bytes(T, H, hd, n_split)) {
        set_global_error("llm_op_attn_decode: scratch is NULL or smaller than llm_op_attn_decode_scratch_bytes");
        return LLM_ERR_INVALID;
    }
    if (init_kernel_attributes()) return LLM_ERR_COMPUTE;
    const size_t part_bytes = attn_decode_scratch_floats(T, H, hd, n_split) * sizeof(float);
    unsigned *counters = (unsigned *)((char *)scratch + part_bytes);
    uint32_t *err = counters + (size_t)8 * H;
    cudaStream_t st = (cudaStream_t)stream;
    AttnDecodeArgs at;
    at.q = q;
    at.kv.k = (f16 *)k_cache; at.kv.v = (f16 *)v_cache;
    at.kv.seq_stride = (long long)Hkv * n_ctx * hd;
    at.kv.n_ctx = n_ctx; at.kv.n_seq = n_seq; at.kv.head_dim = hd; at.kv.n_kv_head = Hkv;
    at.pos = pos; at.seq = seq; at.o = (f16 *)o; at.T = T; at.H = H; at.n_split = n_split;
    at.part = (float *)scratch;
    at.counters = counters;
    at.err = err;
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), st);
    if (!e) e = launch_attn_decode(at, Launch{st, false, nullptr});
    if (e) {
        set_global_error("llm_op_attn_decode: launch failed");
        return LLM_ERR_COMPUTE;
    }
    return attn_decode_check("llm_op_attn_decode", err, st);
}

extern "C" int32_t llm_op_attn_prefill(const void *q, const void *k_cache, const void *v_cache, const int32_t *pos,
                                       const int32_t *seq, void *o, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                       int32_t n_ctx, int32_t n_seq, void *stream) {
    auto bad = [](const char *why) {
        set_global_error((std::string("llm_op_attn_prefill: ") + why).c_str());
        return LLM_ERR_INVALID;
    };
    if (!q || !k_cache || !v_cache || !pos || !seq || !o) return bad("a pointer is NULL");
    if (T < 1 || Hkv < 1 || H < 1 || H % Hkv || n_ctx < 1 || n_seq < 1) return bad("invalid shape");
    if (hd != 32 && hd != 64 && hd != 128) return bad("head_dim must be 32, 64 or 128");
    std::vector<AttnTile> tiles;
    for (int i = 0; i < T;) {
        int j = i;
        while (j < T && seq[j] == seq[i] && j - i < 64) {
            if (pos[j] < 0 || pos[j] >= n_ctx) return bad("a position is outside [0, n_ctx)");
            if (j > i && pos[j] != pos[j - 1] + 1) return bad("positions of a sequence's rows must be consecutive");
            ++j;
        }
        if (seq[i] < 0 || seq[i] >= n_seq) return bad("a sequence id is outside [0, n_seq)");
        tiles.push_back(AttnTile{i, j - i, seq[i], pos[i], pos[i]});
        i = j;
    }
    if (init_kernel_attributes()) return LLM_ERR_COMPUTE;
    // the tcgen05 kernel where it applies (as in the forward pass): 128-row tiles
    const long long cache_rows = (long long)n_seq * Hkv * n_ctx;
    const bool tc = attn_prefill_tc_ok(hd, false) && cache_rows < (1ll << 31);
    if (tc) {
        std::vector<int32_t> sv(seq, seq + T), pv(pos, pos + T);
        tiles.resize(T);
        tiles.resize(build_tiles(sv, pv, 0, T, 128, tiles.data()));
    }
    AttnTile *dtiles = nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMallocAsync((void **)&dtiles, tiles.size() * sizeof(AttnTile), st) != cudaSuccess) return LLM_ERR_ALLOC;
    cudaError_t e = cudaMemcpyAsync(dtiles, tiles.data(), tiles.size() * sizeof(AttnTile), cudaMemcpyHostToDevice, st);
    if (tc) {
        // CTA pairs where they apply, as in the forward pass
        const bool pair = attn_prefill_pair_ok(hd, H, Hkv, false);
        TmaMap mq, mk, mv;
        if (!make_operand_map(&mq, (const f16 *)q, T, H * hd, 128) ||
            !make_operand_map(&mk, (const f16 *)k_cache, (int)cache_rows, hd, pair ? 64 : 128) ||
            !make_operand_map(&mv, (const f16 *)v_cache, (int)cache_rows, hd, 128)) {
            cudaFreeAsync(dtiles, st);
            cudaStreamSynchronize(st);
            return LLM_ERR_COMPUTE;
        }
        AttnPrefillTcArgs at;
        at.tiles = dtiles; at.n_tiles = (int)tiles.size(); at.H = H; at.Hkv = Hkv; at.head_dim = hd;
        at.n_layer = 1; at.layer = 0; at.n_ctx = n_ctx; at.n_seq = n_seq;
        at.o = (f16 *)o; at.ldo = H * hd; at.err = nullptr; at.window = 0;
        if (!e) e = pair ? launch_attn_prefill_pair(at, mq, mk, mv, Launch{st, false, nullptr})
                         : launch_attn_prefill_tc(at, mq, mk, mv, Launch{st, false, nullptr});
    } else {
        AttnPrefillArgs at;
        at.q = (const f16 *)q;
        at.kv.k = (f16 *)k_cache; at.kv.v = (f16 *)v_cache;
        at.kv.seq_stride = (long long)Hkv * n_ctx * hd;
        at.kv.n_ctx = n_ctx; at.kv.n_seq = n_seq; at.kv.head_dim = hd; at.kv.n_kv_head = Hkv;
        at.tiles = dtiles; at.n_tiles = (int)tiles.size(); at.o = (f16 *)o; at.H = H; at.err = nullptr;
        if (!e) e = launch_attn_prefill(at, Launch{st, false, nullptr});
    }
    cudaFreeAsync(dtiles, st);
    if (!e) e = cudaStreamSynchronize(st);
    return e ? LLM_ERR_COMPUTE : LLM_OK;
}
