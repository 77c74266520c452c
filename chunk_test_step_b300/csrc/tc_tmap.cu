// Host-side TMA tensor maps for the tensor-core kernels: cuTensorMapEncodeTiled
// reached through the runtime's driver entry-point query (no link against
// libcuda).
#include "lact_internal.cuh"

#include <cudaTypedefs.h>

namespace lact {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}
}  // namespace

bool tmap_available() { return tmap_encoder() != nullptr; }

bool make_tmap_bf16(CUtensorMap* m, const void* p, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                    const uint32_t* box) {
    auto enc = tmap_encoder();
    if (!enc || rank < 1 || rank > 3) return false;
    cuuint64_t gd[3], gs[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(p), gd, gs, bx, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2D fp32 (f32 = true) or bf16 map, 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* m, const void* p, bool f32, const uint64_t* dims, const uint64_t* strides_bytes,
                  const uint32_t* box) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t gd[2] = {dims[0], dims[1]}, gs[1] = {strides_bytes[0]};
    cuuint32_t bx[2] = {box[0], box[1]}, es[2] = {1, 1};
    CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void*>(p), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lact
