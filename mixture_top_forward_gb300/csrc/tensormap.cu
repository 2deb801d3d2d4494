// Host side of the TMA loads: tensor maps for bf16 row matrices [rows x 64]
// (128-byte rows) read as boxes of `box_rows` rows in the 128-byte swizzle.
// cuTensorMapEncodeTiled is taken from the driver through the runtime's
// entry-point query, so the library links no driver library itself.
#include <cudaTypedefs.h>

#include <mutex>

#include "tensormap.cuh"

namespace mita {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
}  // namespace

static bool load_encoder() {
    std::call_once(g_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

bool make_row_tmap(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    if (!load_encoder() || rows == 0 || box_rows == 0 || box_rows > 256) return false;
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_head_tmap(CUtensorMap* map, const void* base, uint64_t rows_per_head, uint64_t heads,
                    uint64_t row_stride_rows, uint64_t head_stride_rows, uint32_t box_rows) {
    if (!load_encoder() || rows_per_head == 0 || heads == 0 || box_rows == 0 || box_rows > 256) return false;
    const cuuint64_t dims[3] = {64, rows_per_head, heads};
    const cuuint64_t strides[2] = {row_stride_rows * 128, head_stride_rows * 128};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mita
