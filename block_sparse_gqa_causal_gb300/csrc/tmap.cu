// tmap.cu -- host-side creation of TMA tensor maps (CUtensorMap) through the
// driver entry point, so the library needs no link-time libcuda.
#include <cudaTypedefs.h>

#include "msa_internal.h"

namespace msa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}
}  // namespace

cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const unsigned long long *dims,
                           const unsigned long long *strides_bytes, const unsigned *box)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    cuuint64_t d[5], str[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) str[i] = strides_bytes[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), d, str, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_bf16_3d(CUtensorMap *map, const void *base, unsigned long long d0, unsigned long long d1,
                              unsigned long long d2, unsigned long long stride1_bytes,
                              unsigned long long stride2_bytes, unsigned box0, unsigned box1)
{
    const unsigned long long dims[3] = {d0, d1, d2};
    const unsigned long long strides[2] = {stride1_bytes, stride2_bytes};
    const unsigned box[3] = {box0, box1, 1};
    return make_tmap_bf16(map, base, 3, dims, strides, box);
}

}  // namespace msa
