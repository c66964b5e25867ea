// Error state, version string and device queries for libdspark.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace dspark {

static thread_local char g_last_error[512] = "";

dspark_status fail(dspark_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

dspark_status cuda_fail(cudaError_t e, const char *what) {
    return fail(DSPARK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

void clear_error() { g_last_error[0] = '\0'; }

int current_sm_count(int *sm_count) {
    static int cached[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(cuda_fail(e, "cudaGetDevice"));
    if (dev >= 0 && dev < 64 && cached[dev] > 0) {
        *sm_count = cached[dev];
        return DSPARK_OK;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(cuda_fail(e, "cudaDeviceGetAttribute(SM count)"));
    if (dev >= 0 && dev < 64) cached[dev] = n;
    *sm_count = n;
    return DSPARK_OK;
}

namespace {

dspark_status encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle, const void *base,
                           uint32_t rank, const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(DSPARK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, dtype, rank, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSPARK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return DSPARK_OK;
}

dspark_status encode_tiled_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                              CUtensorMapSwizzle swizzle, const void *base, uint64_t rows, uint64_t cols,
                              uint32_t box_rows, uint32_t box_cols) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    return encode_tiled(map, dtype, swizzle, base, 2, dims, strides, box);
}

}  // namespace

dspark_status make_tmap_2d(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols) {
    return encode_tiled_2d(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                           CU_TENSOR_MAP_SWIZZLE_128B, base, rows, cols, box_rows, box_cols);
}

dspark_status make_tmap_kblocks(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_kblocks) {
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_kblocks};
    return encode_tiled(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        CU_TENSOR_MAP_SWIZZLE_128B, base, 3, dims, strides, box);
}

dspark_status make_tmap_rows_f32(CUtensorMap *map, const float *base, uint64_t planes, uint64_t rows, uint64_t cols,
                                 uint32_t box_planes, uint32_t box_cols) {
    const cuuint64_t dims[3] = {cols, rows, planes};
    const cuuint64_t strides[2] = {cols * 4, rows * cols * 4};
    const cuuint32_t box[3] = {box_cols, 1, box_planes};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, base, 3, dims, strides, box);
}

dspark_status make_tmap_kblocks_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                                  uint32_t box_katoms) {
    const cuuint64_t dims[3] = {128, rows, cols / 128};
    const cuuint64_t strides[2] = {cols, 128};
    const cuuint32_t box[3] = {128, box_rows, box_katoms};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B, base, 3, dims, strides, box);
}

}  // namespace dspark

extern "C" const char *dspark_last_error(void) { return dspark::g_last_error; }

extern "C" const char *dspark_version(void) { return "libdspark 0.1 sm_103a"; }
