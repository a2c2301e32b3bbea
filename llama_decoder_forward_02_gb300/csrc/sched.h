// Host-side batch scheduler: the rules of "LLama.cpp — how it works",
// "Step 10" (llama_batch_allocr::init fills missing seq ids, positions and
// output flags, and rejects bad token ids) and "Steps 11–12" (init_batch cuts
// the batch into consecutive ubatches of at most n_ubatch tokens).  Pure C++,
// no CUDA, so it runs and is tested without a GPU.
#pragma once
#include <stdint.h>
#include <string>
#include <vector>

#include "../../include/llm.h"

namespace llm {

struct BatchPlan {
    int n = 0;
    std::vector<int32_t> tok;        // host copy of the token ids (empty if on device)
    std::vector<int32_t> pos, seq;
    std::vector<int8_t> out;
    std::vector<int32_t> out_index;  // batch index -> logits row, or -1
    int n_outputs = 0;
    std::vector<int32_t> ub_start;   // ubatch i covers [ub_start[i], ub_start[i+1])
    std::string error;
};

// Validates `b` against the cache state `seq_next` (next free position of
// every sequence, i.e. seq_pos_max + 1) and fills `p`.  Returns LLM_OK,
// LLM_NO_KV_ROOM or LLM_ERR_INVALID (with p.error set).
int plan_batch(const llm_batch &b, int n_vocab, int n_ctx, int n_seq_max, int n_ubatch,
               const std::vector<int32_t> &seq_next, BatchPlan &p);

}  // namespace llm
