// kt_gemm_act.cu -- kernel instantiations: the up projection with an elementwise activation (GELU erf / tanh / sigmoid, SiLU, none).
#include "kt_gemm.cuh"

namespace kt {

#define KT_LAUNCH(E, D)                                                                     \
    return p.pair == 2 ? launch_one<E, D, 2>(a, b, c, p, grid, smem, stream, pdl, why) \
                       : launch_one<E, D, 1>(a, b, c, p, grid, smem, stream, pdl, why)

kt_status launch_gemm_act(int epi, int dtype, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                          const GemmParams& p, int grid, int smem, void* stream, bool pdl, const char** why) {
    if (dtype == KT_F16) {
        switch (epi) {
            case EPI_GELU_ERF: KT_LAUNCH(EPI_GELU_ERF, KT_F16);
            case EPI_GELU_TANH: KT_LAUNCH(EPI_GELU_TANH, KT_F16);
            case EPI_GELU_SIGMOID: KT_LAUNCH(EPI_GELU_SIGMOID, KT_F16);
            case EPI_SILU: KT_LAUNCH(EPI_SILU, KT_F16);
            case EPI_NONE: KT_LAUNCH(EPI_NONE, KT_F16);
        }
    } else {
        switch (epi) {
            case EPI_GELU_ERF: KT_LAUNCH(EPI_GELU_ERF, KT_BF16);
            case EPI_GELU_TANH: KT_LAUNCH(EPI_GELU_TANH, KT_BF16);
            case EPI_GELU_SIGMOID: KT_LAUNCH(EPI_GELU_SIGMOID, KT_BF16);
            case EPI_SILU: KT_LAUNCH(EPI_SILU, KT_BF16);
            case EPI_NONE: KT_LAUNCH(EPI_NONE, KT_BF16);
        }
    }
    *why = "unknown epilogue kind";
    return KT_ERR_INVALID;
}

#undef KT_LAUNCH

}  // namespace kt
