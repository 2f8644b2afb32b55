// tmap.cu -- encoding of TMA tensor maps through the driver entry point
// (looked up once through the runtime, so the library needs no -lcuda).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qmm_internal.h"

namespace qmm {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return encode;
}

} // namespace

int encode_tmap_2d(void *out128, int dtype, const void *base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1, int swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode)
        return -1;
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

int encode_tmap_3d(void *out128, int dtype, const void *base, uint64_t dim0, uint64_t dim1,
                   uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                   uint32_t box1, uint32_t box2, int swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode)
        return -1;
    const cuuint64_t dims[3] = {cuuint64_t(dim0), cuuint64_t(dim1), cuuint64_t(dim2)};
    const cuuint64_t strides[2] = {cuuint64_t(stride1_bytes), cuuint64_t(stride2_bytes)};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = encode(reinterpret_cast<CUtensorMap *>(out128), CUtensorMapDataType(dtype), 3,
                        const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CUtensorMapSwizzle(swizzle),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

// A Q4_K (Q5_K) matrix of N rows seen as a 3-D tensor of uint64 words: (18
// (22) words = one 144 (176)-byte super-block, N rows, NB super-blocks),
// strides row_bytes and the super-block size.  A box (words, 16, ks) is then
// one 16-row tile of ks consecutive super-blocks, landing in shared memory as
// ks units of 16 rows (super-block major), every row one super-block after
// the previous one.
int make_column_map(void *out128, const void *w, int64_t N, int64_t row_bytes, int ks,
                    int sb_bytes)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode)
        return -1;
    const cuuint32_t words = cuuint32_t(sb_bytes / 8);
    const cuuint64_t dims[3] = {words, cuuint64_t(N), cuuint64_t(row_bytes / sb_bytes)};
    const cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(sb_bytes)};
    const cuuint32_t box[3] = {words, 16u, cuuint32_t(ks)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = encode(reinterpret_cast<CUtensorMap *>(out128), CU_TENSOR_MAP_DATA_TYPE_UINT64, 3,
                        const_cast<void *>(w), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

} // namespace qmm
