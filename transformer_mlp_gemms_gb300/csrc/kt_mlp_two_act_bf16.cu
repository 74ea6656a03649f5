// kt_mlp_two_act_bf16.cu -- kernel instantiations: both projections in one launch, the up
// projection with an elementwise activation, bf16 inputs and outputs.
#include "kt_gemm.cuh"

namespace kt {

#define KT_LAUNCH(E, D)                                                                                            \
    return up.pair == 2 ? launch_one<E, D, 2, true>(m[0], m[1], m[2], up, m[3], m[4], m[5], down, grid, smem, stream, \
                                                    pdl, why)                                                     \
                        : launch_one<E, D, 1, true>(m[0], m[1], m[2], up, m[3], m[4], m[5], down, grid, smem, stream, \
                                                    pdl, why)

kt_status launch_mlp_two_act_bf16(int epi, const CUtensorMap* const* m, const GemmParams& up, const GemmParams& down,
                                 int grid, int smem, void* stream, bool pdl, const char** why) {
    switch (epi) {
        case EPI_GELU_ERF: KT_LAUNCH(EPI_GELU_ERF, KT_BF16);
        case EPI_GELU_TANH: KT_LAUNCH(EPI_GELU_TANH, KT_BF16);
        case EPI_GELU_SIGMOID: KT_LAUNCH(EPI_GELU_SIGMOID, KT_BF16);
        case EPI_SILU: KT_LAUNCH(EPI_SILU, KT_BF16);
        case EPI_NONE: KT_LAUNCH(EPI_NONE, KT_BF16);
    }
    *why = "unknown epilogue kind";
    return KT_ERR_INVALID;
}

#undef KT_LAUNCH

}  // namespace kt
