// Host-side creation of the TMA descriptors (CUtensorMap) that the tcgen05
// kernels load their fp16 operand tiles with: a row-major [rows][cols] matrix
// read in boxes of box_rows x 64 elements with 128-byte swizzle, the layout
// the kernels' shared-memory matrix descriptors expect.  The driver entry
// point is looked up once through the runtime, so the library links no
// driver library directly.
#include <cuda.h>
#include <mutex>

#include "gemm_tc_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool make_operand_map(TmaMap *m, const f16 *ptr, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !ptr || cols % 64 || rows < 1 || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "TmaMap must hold a CUtensorMap");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tcg::BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(m), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void *)ptr, dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_f32_tile_map(TmaMap *m, const float *ptr, int rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !ptr || cols % 32 || rows < 1 || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(m), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void *)ptr, dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace llm
