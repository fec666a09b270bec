// TMA tensor map encoding shared by the tensor-core kernels.
#include <cudaTypedefs.h>

#include "launch.h"
#include "tmap.h"

namespace mhc {

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    // looked up once (thread-safe static initialisation)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
    }();
    return fn;
}

static bool tmap_encode(CUtensorMap *m, CUtensorMapDataType dtype, const void *base, int rank,
                        const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                        CUtensorMapSwizzle sw)
{
    auto fn = encode_tiled();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    return fn(m, dtype, cuuint32_t(rank), const_cast<void *>(base), d,
              st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
               const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle sw)
{
    return tmap_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box, sw);
}

bool tmap_f32_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols, CUtensorMapSwizzle sw)
{
    const uint64_t dims[2] = {cols, rows};
    const uint64_t strides[1] = {cols * 4};
    const uint32_t box[2] = {box_cols, box_rows};
    return tmap_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, 2, dims, strides, box, sw);
}

}  // namespace mhc
