// TMA tensor maps (cuTensorMapEncodeTiled, reached through the runtime's
// driver entry point so the library does not link the driver directly).
#include <mutex>

#include "rsa_internal.h"

namespace rsa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

}  // namespace

namespace {

bool make_map_sw128(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, int rank, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || rank < 1 || rank > 5)
        return false;
    cuuint64_t d[5];
    cuuint64_t st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank)
            st[i] = strides_bytes[i];
    }
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool make_bf16_map_sw128(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims,
                         const uint64_t *strides_bytes, const uint32_t *box)
{
    return make_map_sw128(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides_bytes, box);
}

bool make_f32_map_sw128(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims,
                        const uint64_t *strides_bytes, const uint32_t *box)
{
    return make_map_sw128(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, rank, dims, strides_bytes, box);
}

}  // namespace rsa
