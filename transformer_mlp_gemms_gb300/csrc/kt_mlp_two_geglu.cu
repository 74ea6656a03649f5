// kt_mlp_two_geglu.cu -- kernel instantiations: both projections in one launch, the up
// projection with the GEGLU epilogue.
#include "kt_gemm.cuh"

namespace kt {

#define KT_LAUNCH(E, D)                                                                                            \
    return up.pair == 2 ? launch_one<E, D, 2, true>(m[0], m[1], m[2], up, m[3], m[4], m[5], down, grid, smem, stream, \
                                                    pdl, why)                                                     \
                        : launch_one<E, D, 1, true>(m[0], m[1], m[2], up, m[3], m[4], m[5], down, grid, smem, stream, \
                                                    pdl, why)

kt_status launch_mlp_two_geglu(int dtype, const CUtensorMap* const* m, const GemmParams& up, const GemmParams& down,
                               int grid, int smem, void* stream, bool pdl, const char** why) {
    if (dtype == KT_F16) KT_LAUNCH(EPI_GEGLU, KT_F16);
    KT_LAUNCH(EPI_GEGLU, KT_BF16);
}

#undef KT_LAUNCH

}  // namespace kt
