// tmap.cu -- encoding of 2-D TMA tensor maps through the driver entry point
// (looked up once through the runtime, so the library needs no -lcuda).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qmm_internal.h"

namespace qmm {

int encode_tmap_2d(void *out128, int dtype, const void *base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return -1;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {cuuint64_t(dim0), cuuint64_t(dim1)};
    const cuuint64_t strides[1] = {cuuint64_t(stride1_bytes)};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = encode(reinterpret_cast<CUtensorMap *>(out128), CUtensorMapDataType(dtype), 2,
                        const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CUtensorMapSwizzle(swizzle),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

} // namespace qmm
