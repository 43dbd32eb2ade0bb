// Host-side 2-D TMA tensor maps.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "tmap.h"

namespace slmoe {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::mutex g_encode_mu;

static int get_encode() {
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (g_encode) return SLMOE_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(SLMOE_ECUDA, "cuTensorMapEncodeTiled not available");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return SLMOE_OK;
}

int tmap_encode_2d(CUtensorMap *m, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                   long long rows, long long cols, long long pitch, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle) {
    int rc = get_encode();
    if (rc) return rc;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch * elem_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SLMOE_ECUDA, "cuTensorMapEncodeTiled failed (%d): rows %lld cols %lld pitch %lld box %d x %d",
                    (int)r, rows, cols, pitch, box_cols, box_rows);
    return SLMOE_OK;
}

int tmap_encode_fp4(CUtensorMap *m, const void *base, long long rows, long long K) {
    int rc = get_encode();
    if (rc) return rc;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SLMOE_ECUDA, "cuTensorMapEncodeTiled (FP4) failed (%d): rows %lld K %lld", (int)r, rows, K);
    return SLMOE_OK;
}

}  // namespace slmoe
