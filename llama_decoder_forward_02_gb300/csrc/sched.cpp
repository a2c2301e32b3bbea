#include "sched.h"

#include <cstdio>

namespace llm {

int plan_batch(const llm_batch &b, int n_vocab, int n_ctx, int n_seq_max, int n_ubatch,
               const std::vector<int32_t> &seq_next, BatchPlan &p) {
    char buf[160];
    p = BatchPlan();
    if (b.n_tokens <= 0) { p.error = "batch has no tokens"; return LLM_ERR_INVALID; }
    if (!b.token) { p.error = "batch has no token array"; return LLM_ERR_INVALID; }
    const int n = b.n_tokens;
    p.n = n;
    if (!(b.flags & LLM_BATCH_TOKENS_ON_DEVICE)) {
        p.tok.assign(b.token, b.token + n);
        for (int i = 0; i < n; ++i)
            if (p.tok[i] < 0 || p.tok[i] >= n_vocab) {
                snprintf(buf, sizeof buf, "invalid token[%d] = %d", i, p.tok[i]);
                p.error = buf;
                return LLM_ERR_INVALID;
            }
    }
    p.seq.assign(n, 0);
    if (b.seq_id) p.seq.assign(b.seq_id, b.seq_id + n);
    for (int i = 0; i < n; ++i)
        if (p.seq[i] < 0 || p.seq[i] >= n_seq_max) {
            snprintf(buf, sizeof buf, "invalid seq_id[%d] = %d (n_seq_max %d)", i, p.seq[i], n_seq_max);
            p.error = buf;
            return LLM_ERR_INVALID;
        }
    std::vector<int32_t> nxt = seq_next;
    p.pos.resize(n);
    for (int i = 0; i < n; ++i) {
        const int s = p.seq[i];
        if (b.pos && b.pos[i] != nxt[s]) {
            snprintf(buf, sizeof buf, "pos[%d] = %d but sequence %d continues at %d", i, b.pos[i], s, nxt[s]);
            p.error = buf;
            return LLM_ERR_INVALID;
        }
        p.pos[i] = nxt[s]++;
    }
    p.out.assign(n, 0);
    if (b.output) {
        for (int i = 0; i < n; ++i) p.out[i] = b.output[i] ? 1 : 0;
    } else {
        p.out[n - 1] = 1;
    }
    for (int i = 0; i < n; ++i)
        if (p.pos[i] >= n_ctx) {
            snprintf(buf, sizeof buf, "position %d of sequence %d does not fit n_ctx %d", p.pos[i], p.seq[i], n_ctx);
            p.error = buf;
            return LLM_NO_KV_ROOM;
        }
    p.out_index.assign(n, -1);
    for (int i = 0; i < n; ++i)
        if (p.out[i]) p.out_index[i] = p.n_outputs++;
    for (int s = 0; s < n; s += n_ubatch) p.ub_start.push_back(s);
    p.ub_start.push_back(n);
    return LLM_OK;
}

}  // namespace llm

extern "C" int32_t llm_batch_check(int32_t n_vocab, int32_t n_ctx, int32_t n_seq_max, int32_t n_ubatch,
                                   const int32_t *seq_pos_max, const llm_batch *b, int32_t *pos_out,
                                   int32_t *out_index, int32_t *ubatch_starts, int32_t *n_ubatches) {
    if (!b || !seq_pos_max || n_seq_max < 1 || n_ubatch < 1) return LLM_ERR_INVALID;
    std::vector<int32_t> nxt(n_seq_max);
    for (int s = 0; s < n_seq_max; ++s) nxt[s] = seq_pos_max[s] + 1;
    llm::BatchPlan p;
    const int rc = llm::plan_batch(*b, n_vocab, n_ctx, n_seq_max, n_ubatch, nxt, p);
    if (rc != LLM_OK) return rc;
    for (int i = 0; i < p.n; ++i) {
        if (pos_out) pos_out[i] = p.pos[i];
        if (out_index) out_index[i] = p.out_index[i];
    }
    const int nub = (int)p.ub_start.size() - 1;
    if (ubatch_starts)
        for (int i = 0; i < nub; ++i) ubatch_starts[i] = p.ub_start[i];
    if (n_ubatches) *n_ubatches = nub;
    return LLM_OK;
}
