// Decode attention with the cache split along the sequence (flash-decoding):
// for each decode row t and query head h, o = softmax(q K^T / sqrt(hd)) V over
// the cached positions c <= pos[t] of sequence seq[t] ("Inside the inference
// engine: model architectures and forward pass", sections "Detailed
// explanation: Llama's forward pass in Go" (GQA, ScaledDotProduct with the
// cache) and "KV Cache: memory for causal attention" (full causal mask);
// "LLama.cpp — how it works", "KV-cache and the Prefill / Decode stages": the
// new token's Q meets every cached K and V).
//
// Bound by HBM reads of K and V.  One CTA per (split, kv head, row) reads its
// span of keys once for all G = H/Hkv query heads of the group (the GQA
// sharing): the G heads are the rows of one m16 tile, so QK^T and PV run on
// mma.sync.  The span streams through double-buffered 64-key K/V tiles in
// swizzled shared memory (cp.async), so a short span has all its loads in
// flight at once; the four warps take 16 keys of each tile with their own
// online softmax (base 2, q pre-scaled by log2(e)/sqrt(hd)) and are combined
// at the end.  Each CTA writes (max, sum, unnormalised output) for its split;
// the CTA that arrives last at the (row, kv head) counter merges all splits
// in split order, so the result is deterministic and nothing spins.
#include <mutex>
#include <string>

#include "attn_decode_unit.cuh"
#include "attn_tile.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "../../include/llm.h"

namespace llm {

namespace {

using namespace attn_dec;

struct BlockSync {
    __device__ static __forceinline__ void sync() { __syncthreads(); }
};

struct GridDep {
    __device__ static __forceinline__ void wait() {
        pdl_wait();
        pdl_trigger();
    }
};

// At most 128 registers a thread: a CTA then fits on an SM beside one CTA of a
// streamed one-row GEMV (9 warps of 128 registers put 3 warps, 12 K registers,
// on one of the SM's four 16 K-register sub-partitions), so it can be resident
// and stream its cached K/V while the QKV GEMV still runs.
template <int HD, int G, bool F8>
__global__ void __launch_bounds__(THREADS, 4) attn_decode_kernel(const AttnDecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    attn_decode_unit<HD, G, BlockSync, GridDep, F8>(a, blockIdx.x, blockIdx.y, blockIdx.z, threadIdx.x, smem_raw);
}

}  // namespace

size_t attn_decode_scratch_floats(int T, int H, int hd, int n_split) {
    return (size_t)T * H * n_split * (hd + 2);
}

#define ATTN_DEC_CASE(HDV, GV)                                                                        \
    if (a.kv.head_dim == HDV && G == GV)                                                              \
        return a.kv.k8 ? launch_kernel(attn_decode_kernel<HDV, GV, true>, grid, dim3(THREADS), decode_smem_bytes<HDV>(), l, a) \
                       : launch_kernel(attn_decode_kernel<HDV, GV, false>, grid, dim3(THREADS), decode_smem_bytes<HDV>(), l, a);

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, const Launch &l) {
    if (a.T < 1 || a.T > 8 || a.n_split < 1 || a.n_split > MAX_SPLIT || a.kv.n_kv_head < 1 || a.H % a.kv.n_kv_head)
        return cudaErrorInvalidValue;
    const int G = a.H / a.kv.n_kv_head;
    const dim3 grid(a.n_split, a.kv.n_kv_head, a.T);
    ATTN_DEC_CASE(32, 1) ATTN_DEC_CASE(32, 2) ATTN_DEC_CASE(32, 4) ATTN_DEC_CASE(32, 8)
    ATTN_DEC_CASE(64, 1) ATTN_DEC_CASE(64, 2) ATTN_DEC_CASE(64, 4) ATTN_DEC_CASE(64, 8)
    ATTN_DEC_CASE(128, 1) ATTN_DEC_CASE(128, 2) ATTN_DEC_CASE(128, 4) ATTN_DEC_CASE(128, 8)
    return cudaErrorInvalidValue;
}

cudaError_t init_attn_decode_attributes() {
    cudaError_t e = cudaSuccess;
#define ATTN_DEC_ATTR1(HDV, GV, F)                                                                   \
    if (!e) e = allow_smem(attn_decode_kernel<HDV, GV, F>, decode_smem_bytes<HDV>());                \
    if (!e) e = cudaFuncSetAttribute(attn_decode_kernel<HDV, GV, F>, cudaFuncAttributePreferredSharedMemoryCarveout, \
                                     cudaSharedmemCarveoutMaxShared);
#define ATTN_DEC_ATTR(HDV, GV) ATTN_DEC_ATTR1(HDV, GV, false) ATTN_DEC_ATTR1(HDV, GV, true)
    ATTN_DEC_ATTR(32, 1) ATTN_DEC_ATTR(32, 2) ATTN_DEC_ATTR(32, 4) ATTN_DEC_ATTR(32, 8)
    ATTN_DEC_ATTR(64, 1) ATTN_DEC_ATTR(64, 2) ATTN_DEC_ATTR(64, 4) ATTN_DEC_ATTR(64, 8)
    ATTN_DEC_ATTR(128, 1) ATTN_DEC_ATTR(128, 2) ATTN_DEC_ATTR(128, 4) ATTN_DEC_ATTR(128, 8)
#undef ATTN_DEC_ATTR
    return e;
}

}  // namespace llm

// ---------------------------------------------------------------------------
// Zero-allocation variant of the decode attention entry point.
//
// Some callers cannot call cudaMalloc at all: host code under a caching
// allocator that owns all device memory and forbids outside allocations, a
// serving process with a fixed device-memory footprint, or real-time loops
// that must never block in the driver's allocator (cudaMalloc can
// synchronize the device).  For them the split partials and split counters live in one
// file-scope device array instead of caller- or library-allocated memory.
// Every GPU that loads this library holds that array (4 MiB + 2 KiB) until
// the process exits.
// ---------------------------------------------------------------------------
namespace llm {
namespace {

constexpr size_t NOALLOC_PART_FLOATS = (size_t)1 << 20;    // 4 MiB of split partials
constexpr size_t NOALLOC_COUNTERS = 512;                    // (row, kv head) counters
// partials first, then the counters (as 32-bit words), then one error word
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_PART_FLOATS + NOALLOC_COUNTERS + 1];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[256] = {nullptr};   // per device: the array's device address

}  // namespace

// Records the message llm_last_error(NULL) reports (defined with the C ABI).
void set_global_error(const char *msg);
const char *attn_decode_args_error(const void *q, const void *k, const void *v, const void *pos, const void *seq,
                                   const void *o, int T, int H, int Hkv, int hd, int n_ctx, int n_seq, int n_split);
int32_t attn_decode_check(const char *who, uint32_t *err_dev, cudaStream_t st);

}  // namespace llm

extern "C" int32_t llm_op_attn_decode_noalloc(const float *q, const void *k_cache, const void *v_cache,
                                              const int32_t *pos, const int32_t *seq, void *o, int32_t T,
                                              int32_t H, int32_t Hkv, int32_t hd, int32_t n_ctx, int32_t n_seq,
                                              int32_t n_split, void *stream) {
    using namespace llm;
    if (const char *why = attn_decode_args_error(q, k_cache, v_cache, pos, seq, o, T, H, Hkv, hd, n_ctx, n_seq, n_split)) {
        set_global_error((std::string("llm_op_attn_decode_noalloc: ") + why).c_str());
        return LLM_ERR_INVALID;
    }
    const size_t need = attn_decode_scratch_floats(T, H, hd, n_split);
    if (need > NOALLOC_PART_FLOATS || (size_t)T * Hkv > NOALLOC_COUNTERS) {
        set_global_error("llm_op_attn_decode_noalloc: T*H*n_split*(head_dim+2) exceeds the 1048576-float "
                         "static scratch (or T*n_head_kv exceeds 512); use llm_op_attn_decode");
        return LLM_ERR_INVALID;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) {
        set_global_error("llm_op_attn_decode_noalloc: no current device");
        return LLM_ERR_COMPUTE;
    }
    void *base = nullptr;
    {
        // once per device, with that device current: the host-side name of
        // the array is not a device address, so ask the runtime for it
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                set_global_error("llm_op_attn_decode_noalloc: cudaGetSymbolAddress failed");
                return LLM_ERR_COMPUTE;
            }
            g_noalloc_addr[dev] = p;
        }
        base = g_noalloc_addr[dev];
    }
    float *part = static_cast<float *>(base);
    unsigned *counters = reinterpret_cast<unsigned *>(part + NOALLOC_PART_FLOATS);
    uint32_t *err = counters + NOALLOC_COUNTERS;
    cudaStream_t st = (cudaStream_t)stream;
    // the counters and the error word must start at zero; the array keeps
    // whatever the last call left
    cudaError_t e = cudaMemsetAsync(counters, 0, (NOALLOC_COUNTERS + 1) * sizeof(unsigned), st);
    AttnDecodeArgs at;
    at.q = q;
    at.kv.k = (f16 *)k_cache; at.kv.v = (f16 *)v_cache;
    at.kv.seq_stride = (long long)Hkv * n_ctx * hd;
    at.kv.n_ctx = n_ctx; at.kv.n_seq = n_seq; at.kv.head_dim = hd; at.kv.n_kv_head = Hkv;
    at.pos = pos; at.seq = seq; at.o = (f16 *)o; at.T = T; at.H = H; at.n_split = n_split;
    at.part = part; at.counters = counters; at.err = err;
    if (!e) e = init_kernel_attributes();
    if (!e) e = launch_attn_decode(at, Launch{st, false, nullptr});
    if (e) {
        set_global_error("llm_op_attn_decode_noalloc: launch failed");
        return LLM_ERR_COMPUTE;
    }
    return attn_decode_check("llm_op_attn_decode_noalloc", err, st);
}
