// TMA tensor-map encoding through the driver entry point (looked up once;
// no link-time dependency on the driver library).
#include "ssd_tmap.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace ssd {
namespace {
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000 *out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}
}  // namespace

cudaError_t make_tmap_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                           const uint64_t *strides, const uint32_t *box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank),
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ssd
