// tc_host.cu -- host helpers of the tensor-core kernels: TMA tensor maps.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc.cuh"

namespace llsa {

namespace {
std::mutex g_enc_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lk(g_enc_mu);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

int make_tmap_bf16(CUtensorMap* map, const void* base, long long rows, int cols, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return LLSA_ERR_CUDA;
    cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LLSA_OK : LLSA_ERR_CUDA;
}

int make_tmap_tokens(CUtensorMap* map, const void* base, const Shape& s) {
    if (!s.raster) return make_tmap_bf16(map, base, s.slices * (long long)s.n, s.d, 16);
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return LLSA_ERR_CUDA;
    const cuuint64_t row = (cuuint64_t)s.d * 2;
    cuuint64_t gdim[4] = {(cuuint64_t)s.d, (cuuint64_t)s.side, (cuuint64_t)s.side, (cuuint64_t)s.slices};
    cuuint64_t gstride[3] = {row, row * s.side, row * s.side * s.side};
    cuuint32_t box[4] = {64, 4, 4, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LLSA_OK : LLSA_ERR_CUDA;
}

}  // namespace llsa
