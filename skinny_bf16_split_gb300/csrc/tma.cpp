// tma.cpp -- TMA tensor-map encoding through the driver entry point.
//
// cuTensorMapEncodeTiled is a pure host function of the driver API.  It is
// looked up once through the runtime (cudaGetDriverEntryPointByVersion), so the
// library links only the CUDA runtime.
#include "internal.h"

namespace dep {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace

CUresult encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};  // bytes between rows
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// A [outer, inner] BF16 matrix (inner a multiple of 64) viewed in three
// dimensions {64 columns, outer rows, inner / 64 column blocks}: the block
// dimension steps 128 bytes along a row, so a box {64, box_rows, blocks}
// lands in shared memory as `blocks` consecutive [box_rows x 64] slices, the
// image of that many 2-D boxes {64, box_rows} at consecutive 64-column offsets
// (with the 128-byte swizzle, rows past `outer` filled with zeros), from one
// copy instruction instead of `blocks`.  Columns past `inner` would alias into
// the next row, which is why inner % 64 == 0 is required.
CUresult encode_bf16_3d_blocks(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                               uint32_t box_rows, uint32_t blocks)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    if (inner % 64 != 0)
        return CUDA_ERROR_INVALID_VALUE;
    const cuuint64_t dims[3] = {64, outer, inner / 64};
    const cuuint64_t strides[2] = {inner * 2, 128};  // bytes between rows, between column blocks
    const cuuint32_t box[3] = {64, box_rows, blocks};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace dep
