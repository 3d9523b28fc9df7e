// tma_host.cu -- host-side helpers for the TMA kernels: tensor-map encoding
// (through the driver entry point, so the library needs no libcuda link) and
// the device's SM count.
#include <cudaTypedefs.h>

#include "tma.cuh"

namespace pa {

namespace {
// The driver's encoder, resolved once (a function-local static: thread-safe initialisation).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return nullptr;
    }();
    return fn;
}
}  // namespace

int make_tensor_map_3d(CUtensorMap *map, const void *base, pa_dtype dtype, int dim0, int dim1,
                       int64_t dim2, int box0, int box1, int box2, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    CUtensorMapDataType dt = dtype == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                             : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int eb = dtype == PA_F32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)dim0, (cuuint64_t)dim1, (cuuint64_t)dim2};
    cuuint64_t strides[2] = {(cuuint64_t)dim0 * eb, (cuuint64_t)dim0 * eb * dim1};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, (cuuint32_t)box2};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_block_map(CUtensorMap *map, const void *base, pa_dtype dtype, int head_dim, int num_kv_heads,
                      int64_t rows, int block_size) {
    auto fn = encode_fn();
    if (!fn || head_dim % 64 != 0 || rows % 8 != 0 || block_size % 8 != 0) return PA_ERR_CUDA;
    CUtensorMapDataType dt = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t row_bytes = (cuuint64_t)num_kv_heads * head_dim * 2;
    // (column in a 64-wide slice, row in a group of 8, slice, group, kv head)
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)head_dim / 64, (cuuint64_t)rows / 8, (cuuint64_t)num_kv_heads};
    cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, (cuuint64_t)head_dim * 2};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)head_dim / 64, (cuuint32_t)block_size / 8, 1};
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, dt, 5, const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_tensor_map(CUtensorMap *map, const void *base, pa_dtype dtype, int head_dim,
                       int num_kv_heads, int64_t rows, int box_heads, int box_rows) {
    return make_tensor_map_3d(map, base, dtype, head_dim, num_kv_heads, rows, head_dim, box_heads,
                              box_rows, false);
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace pa
