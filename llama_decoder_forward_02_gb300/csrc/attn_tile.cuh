// Shared-memory tiles of K/V rows for the attention kernels: rows of head_dim
// fp16 values, 16-byte chunks XOR-swizzled so that ldmatrix over 8
// consecutive rows is free of bank conflicts, filled with cp.async.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace llm {

template <int HD>
struct Swz {
    static constexpr int CH = HD / 8;                      // 16-byte chunks per row
    __device__ static __forceinline__ int chunk(int r, int c) {
        return CH >= 8 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & (CH - 1)));
    }
    __device__ static __forceinline__ int off(int r, int c) { return r * HD + chunk(r, c) * 8; }
};

// rows [0, rows_valid) of src (row stride HD) into a ROWS x HD swizzled tile;
// the remaining rows are zero-filled.
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows(f16 *dst, const f16 *src, int rows_valid, int tid) {
    constexpr int CH = HD / 8;
    for (int i = tid; i < ROWS * CH; i += THREADS) {
        const int r = i / CH, c = i - r * CH;
        const bool pv = r < rows_valid;
        cp_async16(dst + Swz<HD>::off(r, c), src + (size_t)(pv ? r : 0) * HD + c * 8, pv);
    }
}

// rows [r_lo, r_hi) of src (row stride HD) into a ROWS x HD swizzled tile,
// rows [r_zero, ROWS) zero-filled, every other row left untouched (so that a
// later call can fill it: two cp.async writes to one address are unordered).
template <int HD, int ROWS, int THREADS>
__device__ __forceinline__ void load_rows_span(f16 *dst, const f16 *src, int r_lo, int r_hi, int r_zero, int tid) {
    constexpr int CH = HD / 8;
    for (int i = tid; i < ROWS * CH; i += THREADS) {
        const int r = i / CH, c = i - r * CH;
        const bool copy = r >= r_lo && r < r_hi;
        if (copy || r >= r_zero)
            cp_async16(dst + Swz<HD>::off(r, c), src + (size_t)(copy ? r : 0) * HD + c * 8, copy);
    }
}

}  // namespace llm
