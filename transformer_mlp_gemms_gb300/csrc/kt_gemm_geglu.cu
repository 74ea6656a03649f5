// kt_gemm_geglu.cu -- kernel instantiations: the up projection with the GEGLU epilogue (value and gate accumulators).
#include "kt_gemm.cuh"

namespace kt {

#define KT_LAUNCH(E, D)                                                                     \
    return p.pair == 2 ? launch_one<E, D, 2>(a, b, c, p, grid, smem, stream, pdl, why) \
                       : launch_one<E, D, 1>(a, b, c, p, grid, smem, stream, pdl, why)

kt_status launch_gemm_geglu(int dtype, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                            const GemmParams& p, int grid, int smem, void* stream, bool pdl, const char** why) {
    if (dtype == KT_F16) KT_LAUNCH(EPI_GEGLU, KT_F16);
    KT_LAUNCH(EPI_GEGLU, KT_BF16);
}

#undef KT_LAUNCH

}  // namespace kt
