// tmap.cu -- host helpers: TMA tensor-map encoding through the driver entry
// point (no link-time dependency on libcuda) and cached device properties.
#include <cudaTypedefs.h>
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode()
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

int make_tmap_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                 uint64_t inner, uint64_t rows, uint64_t outer, uint64_t row_stride_bytes,
                 uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle)
{
    std::call_once(g_encode_once, load_encode);
    if (!g_encode)
        return MOE_ERR_CUDA;
    const cuuint64_t dims[3] = {inner, rows, outer};
    const cuuint64_t strides[2] = {row_stride_bytes, outer_stride_bytes};
    const cuuint32_t box[3] = {box_inner, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    (void)elem_bytes;
    const CUresult r = g_encode(m, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, uint64_t inner, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    std::call_once(g_encode_once, load_encode);
    if (!g_encode)
        return MOE_ERR_CUDA;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(m, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int make_tmap_nd(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle)
{
    std::call_once(g_encode_once, load_encode);
    if (!g_encode)
        return MOE_ERR_CUDA;
    if (rank < 1 || rank > 5)
        return MOE_ERR_INVALID_ARG;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; i++) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; i++)
        st[i] = strides_bytes[i];
    const CUresult r = g_encode(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int sm_count(int device)
{
    static std::atomic<int> cache[64];   // 0 = not yet queried
    if (device < 0 || device >= 64)
        return 0;
    int n = cache[device].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
            return 0;
        cache[device].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace moe
