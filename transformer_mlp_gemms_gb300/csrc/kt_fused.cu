// kt_fused.cu -- the H-on-chip variant: one kernel computes both projections for
// blocks of 128 tokens and never writes H to memory (the handoff the KohakuTPU page
// could not make, "SDXL as a requirements inventory", section 6.3, H9).
//
// It applies where an F-slice of H and the whole Y accumulator fit tensor memory
// together: D <= 256.  Per CTA and row block (persistent over row blocks):
//
//   X[128 x D] is loaded once into shared memory (K-major, 128-byte swizzle);
//   for each slice j of 64 hidden columns:
//     up MMA:   Hacc[b] = X . W_up[:, slice j] (+ the gate slice for GEGLU), fp32 TMEM
//     epilogue: H = round(act(Hacc[b] + b_up)) written into shared memory in the
//               K-major swizzled layout the next MMA reads (two buffers, b = j % 2)
//     down MMA: Yacc += H[b] . W_down[slice j, :]                 fp32 TMEM
//   Y = round(Yacc + b_down (+ R)), TMA tensor stores.
//
// The MMAs are issued in the order up(0), up(1), down(0), up(2), down(1), ... so the
// epilogue of slice j runs while the tensor pipe computes up(j+1).  The weight slices
// stream through one stage ring in exactly that order.  Every wait is bounded as in
// the two-kernel path.
#include "kt_gemm.cuh"

namespace kt {

namespace {

constexpr int kFS = kFusedSlice;  // hidden columns per slice
constexpr uint32_t kHaccCol = 256;  // TMEM column of the H accumulators (Y uses 0 .. Dk-1)

template <int EPI, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    kt_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWu,
                    const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    constexpr int NB = EPI == EPI_GEGLU ? 2 : 1;  // B boxes per up slice (value, gate)
    const uint32_t sX = base;
    const uint32_t sH = sX + p.x_bytes;                 // two 128 x 64 H buffers, 16 KB each
    const uint32_t sRing = sH + 2u * 16384u;
    const uint32_t staging = sRing + (uint32_t)p.stages * p.stage_bytes;
    const uint32_t bars = staging + (uint32_t)kStagingBytes;
    const uint32_t bar_full = bars;                     // [stages]
    const uint32_t bar_empty = bar_full + 8u * kMaxStages;
    const uint32_t bar_xfull = bar_empty + 8u * kMaxStages;
    const uint32_t bar_xempty = bar_xfull + 8u;
    const uint32_t bar_hacc_full = bar_xempty + 8u;     // [2]
    const uint32_t bar_hacc_empty = bar_hacc_full + 16u;
    const uint32_t bar_hs_full = bar_hacc_empty + 16u;  // [2]
    const uint32_t bar_hs_empty = bar_hs_full + 16u;
    const uint32_t bar_yfull = bar_hs_empty + 16u;
    const uint32_t bar_yempty = bar_yfull + 8u;
    const uint32_t bar_drain = bar_yempty + 8u;
    uint32_t* slots = reinterpret_cast<uint32_t*>(base_ptr + (bar_drain + 8u - base));
    uint32_t* tmem_slot = slots;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slots + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar_xfull, 1);
        mbar_init(bar_xempty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_hacc_full + 8u * b, 1);
            mbar_init(bar_hacc_empty + 8u * b, kEpiWarps);
            mbar_init(bar_hs_full + 8u * b, kEpiWarps);
            mbar_init(bar_hs_empty + 8u * b, 1);
        }
        mbar_init(bar_yfull, 1);
        mbar_init(bar_yempty, kEpiWarps);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmWu);
        prefetch_tmap(&tmWd);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.pdl_wait) asm volatile("griddepcontrol.wait;" ::: "memory");

    const int n = p.n_slices;
    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            auto next_stage = [&](uint32_t bytes) -> int {  // returns the stage, or -1 on abort
                if (!wait_phase(bar_empty + 8u * stage, phase ^ 1u, abort_flag, p.error, DEV_TIMEOUT_PRODUCER,
                                p.wait_limit_ns))
                    return -1;
                const int s = (int)stage;
                mbar_arrive_expect_tx(bar_full + 8u * stage, bytes);
                armed |= 1u << stage;
                armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == (uint32_t)p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return s;
            };
            auto load_up = [&](int j) -> bool {  // W_up columns [64 j, 64 j + 64) (+ gate), all Dk rows
                const int s = next_stage(p.wup_bytes);
                if (s < 0) return false;
                const uint32_t dst = sRing + (uint32_t)s * p.stage_bytes;
                tma_load_2d(dst, &tmWu, bar_full + 8u * s, kFS * j, 0);
                if (NB == 2) tma_load_2d(dst + (uint32_t)p.Dk * 128u, &tmWu, bar_full + 8u * s, p.gate_col + kFS * j, 0);
                return true;
            };
            auto load_dn = [&](int j) -> bool {  // W_down rows [64 j, 64 j + 64), Dk columns in 64-column boxes
                const int s = next_stage(p.wdn_bytes);
                if (s < 0) return false;
                const uint32_t dst = sRing + (uint32_t)s * p.stage_bytes;
                for (int ch = 0; ch < p.Dk / 64; ++ch)
                    tma_load_2d(dst + (uint32_t)ch * (uint32_t)kFS * 128u, &tmWd, bar_full + 8u * s, 64 * ch, kFS * j);
                return true;
            };
            int rbi = 0;
            int x_last = -1;  // row-block index of the last X load issued
            for (int tm = blockIdx.x; tm < p.tiles_m && ok; tm += gridDim.x, ++rbi) {
                if (!wait_phase(bar_xempty, (uint32_t)(rbi & 1) ^ 1u, abort_flag, p.error, DEV_TIMEOUT_PRODUCER,
                                p.wait_limit_ns))
                    break;
                mbar_arrive_expect_tx(bar_xfull, p.x_bytes);
                x_last = rbi;
                for (int a = 0; a < p.Dk / 64; ++a) tma_load_2d(sX + 16384u * a, &tmX, bar_xfull, 64 * a, tm * kBM);
                for (int j = 0; j < n && ok; ++j) {
                    ok = load_up(j);
                    if (ok && j >= 1) ok = load_dn(j - 1);
                }
                if (ok) ok = load_dn(n - 1);
            }
            if (*abort_flag) {
                // no copy may still be landing in shared memory that is about to be released
                for (int s = 0; s < p.stages; ++s)
                    if (armed & (1u << s)) wait_drain(bar_full + 8u * s, (armed_phase >> s) & 1u, 100000000ull);
                if (x_last >= 0) wait_drain(bar_xfull, (uint32_t)(x_last & 1), 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool issued = false;
            bool ok = true;
            const uint64_t ax0 = smem_desc(sX, 16u, 1024u);
            auto take_stage = [&]() -> int {
                if (!wait_phase(bar_full + 8u * stage, phase, abort_flag, p.error, DEV_TIMEOUT_MMA, p.wait_limit_ns))
                    return -1;
                tc_fence_after();
                const int s = (int)stage;
                if (++stage == (uint32_t)p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return s;
            };
            int rbi = 0;
            for (int tm = blockIdx.x; tm < p.tiles_m && ok; tm += gridDim.x, ++rbi) {
                if (!wait_phase(bar_xfull, (uint32_t)(rbi & 1), abort_flag, p.error, DEV_TIMEOUT_MMA, p.wait_limit_ns))
                    break;
                tc_fence_after();
                for (int j = 0; j <= n && ok; ++j) {
                    if (j < n) {
                        const uint32_t c = (uint32_t)(rbi * n + j), b = c & 1u, use = c >> 1;
                        if (!wait_phase(bar_hacc_empty + 8u * b, (use & 1u) ^ 1u, abort_flag, p.error, DEV_TIMEOUT_MMA,
                                        p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        const int s = take_stage();
                        if (s < 0) {
                            ok = false;
                            break;
                        }
                        const uint32_t sB = sRing + (uint32_t)s * p.stage_bytes;
                        const uint64_t bd0 = smem_desc(sB, (uint32_t)p.Dk * 128u, 1024u);
                        const uint64_t gd0 = smem_desc(sB + (uint32_t)p.Dk * 128u, (uint32_t)p.Dk * 128u, 1024u);
                        const uint32_t d = tmem_base + kHaccCol + b * (uint32_t)(NB * kFS);
                        for (int k = 0; k < p.Dk / 16; ++k) {
                            const uint64_t ad = ax0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2);
                            mma_f16(d, ad, bd0 + (uint64_t)(k * 128), p.idesc_up, k > 0 ? 1u : 0u);
                            if (NB == 2) mma_f16(d + kFS, ad, gd0 + (uint64_t)(k * 128), p.idesc_up, k > 0 ? 1u : 0u);
                        }
                        issued = true;
                        mma_commit(bar_empty + 8u * s);
                        mma_commit(bar_hacc_full + 8u * b);
                        if (j == n - 1) mma_commit(bar_xempty);
                    }
                    if (j >= 1) {
                        const int jj = j - 1;
                        const uint32_t c = (uint32_t)(rbi * n + jj), b = c & 1u, use = c >> 1;
                        if (!wait_phase(bar_hs_full + 8u * b, use & 1u, abort_flag, p.error, DEV_TIMEOUT_MMA,
                                        p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        if (jj == 0 && !wait_phase(bar_yempty, (uint32_t)(rbi & 1) ^ 1u, abort_flag, p.error,
                                                   DEV_TIMEOUT_MMA, p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        const int s = take_stage();
                        if (s < 0) {
                            ok = false;
                            break;
                        }
                        const uint32_t sB = sRing + (uint32_t)s * p.stage_bytes;
                        const uint64_t hd0 = smem_desc(sH + b * 16384u, 16u, 1024u);
                        const uint64_t bd0 = smem_desc(sB, (uint32_t)kFS * 128u, 1024u);
                        for (int k = 0; k < kFS / 16; ++k)
                            mma_f16(tmem_base, hd0 + (uint64_t)(k * 2), bd0 + (uint64_t)(k * 128), p.idesc_dn,
                                    (jj > 0 || k > 0) ? 1u : 0u);
                        mma_commit(bar_empty + 8u * s);
                        mma_commit(bar_hs_empty + 8u * b);
                    }
                }
                if (ok) mma_commit(bar_yfull);
            }
            if (*abort_flag && issued) {
                mma_commit(bar_drain);
                wait_drain(bar_drain, 0u, 100000000ull);
            }
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;    // TMEM lane quadrant of this warp
        const int half = ew >> 2;  // which 32-column group(s)
        const int row = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const uint32_t stg = staging + (uint32_t)ew * 2048u;
        int rbi = 0;
        bool live = true;
        for (int tm = blockIdx.x; tm < p.tiles_m && live; tm += gridDim.x, ++rbi) {
            for (int j = 0; j < n; ++j) {
                const uint32_t c = (uint32_t)(rbi * n + j), b = c & 1u, use = c >> 1;
                bool got = wait_phase(bar_hacc_full + 8u * b, use & 1u, abort_flag, p.error, DEV_TIMEOUT_EPILOGUE,
                                      p.wait_limit_ns);
                got = got && wait_phase(bar_hs_empty + 8u * b, (use & 1u) ^ 1u, abort_flag, p.error,
                                        DEV_TIMEOUT_EPILOGUE, p.wait_limit_ns);
                if (!epi_all(got)) {
                    live = false;
                    break;
                }
                tc_fence_after();
                // this warp's 32 rows x 32 hidden columns of the slice
                const int g = half;
                const int col = kFS * j + 32 * g;
                uint32_t r[32];
                tmem_ld32(tmem_base + lanes + kHaccCol + b * (uint32_t)(NB * kFS) + 32u * g, r);
                float v[32];
                if constexpr (EPI == EPI_GEGLU) {
                    uint32_t gr[32];
                    tmem_ld32(tmem_base + lanes + kHaccCol + b * (uint32_t)(NB * kFS) + kFS + 32u * g, gr);
                    tmem_wait_ld_only();
                    reg_fence32(r);
                    reg_fence32(gr);
                    float bv[32], bg[32];
                    if (p.bias_up) {
                        load_bias32<DT>(p.bias_up, col, p.F, bv);
                        load_bias32<DT>(p.bias_up, p.gate_col + col, p.gate_col + p.F, bg);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) bv[i] = bg[i] = 0.0f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        f2_split(geglu_f2<true>(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), f2(bv[i], bv[i + 1]),
                                          f2(__uint_as_float(gr[i]), __uint_as_float(gr[i + 1])), f2(bg[i], bg[i + 1])),
                                 v[i], v[i + 1]);
                } else {
                    tmem_wait_ld_only();
                    reg_fence32(r);
                    float bb[32];
                    if (p.bias_up) {
                        load_bias32<DT>(p.bias_up, col, p.F, bb);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) bb[i] = 0.0f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        f2_split(act_f2<EPI, true>(f2_add<true>(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                                    f2(bb[i], bb[i + 1]))),
                                 v[i], v[i + 1]);
                }
                // hidden columns past F meet zero rows of W_down; keep them exactly zero
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (col + i >= p.F) v[i] = 0.0f;
                // H[row][32 g + 8 i ..] -> 16-byte chunk 4 g + i of the row, 128-byte swizzle
                const uint32_t hrow = sH + b * 16384u + (uint32_t)row * 128u;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t chunk = (uint32_t)(4 * g + i) ^ ((uint32_t)row & 7u);
                    st_shared_v4(hrow + (chunk << 4), pack2<DT>(v[8 * i], v[8 * i + 1]),
                                 pack2<DT>(v[8 * i + 2], v[8 * i + 3]), pack2<DT>(v[8 * i + 4], v[8 * i + 5]),
                                 pack2<DT>(v[8 * i + 6], v[8 * i + 7]));
                }
                fence_async_smem();  // the tensor pipe reads H through the async proxy
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_hacc_empty + 8u * b);
                    mbar_arrive(bar_hs_full + 8u * b);
                }
            }
            if (!live) break;
            const bool got = wait_phase(bar_yfull, (uint32_t)(rbi & 1), abort_flag, p.error, DEV_TIMEOUT_EPILOGUE,
                                        p.wait_limit_ns);
            if (!epi_all(got)) break;
            tc_fence_after();
            const int y0 = tm * kBM + q * 32;
            const bool rows_live = y0 < p.M;
            for (int g = half; g < p.Dk / 32; g += 2) {
                uint32_t r[32];
                tmem_ld32(tmem_base + lanes + 32u * g, r);
                tmem_wait_ld_only();
                reg_fence32(r);
                const int col = 32 * g;
                if (col < p.D && rows_live) {
                    float v[32], bb[32];
                    if (p.bias_dn) {
                        load_bias32<DT>(p.bias_dn, col, p.D, bb);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) bb[i] = 0.0f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) + bb[i];
                    if (p.residual) add_residual32<DT>(p.residual, y0 + lane, p.M, col, p.D, v);
                    stage_and_store<DT>(&tmY, stg, lane, v, col, y0);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_yempty);
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, kTmemCols);
    }
}

template <int EPI, int DT>
kt_status launch_fused_t(const CUtensorMap* tx, const CUtensorMap* twu, const CUtensorMap* twd, const CUtensorMap* ty,
                         const FusedParams& p, int grid, int smem, void* stream, bool pdl, const char** why) {
    auto kern = kt_fused_kernel<EPI, DT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, *tx, *twu, *twd, *ty, p);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

}  // namespace

kt_status launch_fused(int epi, int dtype, const void* tx, const void* twu, const void* twd, const void* ty,
                       const FusedParams& p, int grid, int smem, void* stream, bool pdl, const char** why) {
    const CUtensorMap* a = reinterpret_cast<const CUtensorMap*>(tx);
    const CUtensorMap* b = reinterpret_cast<const CUtensorMap*>(twu);
    const CUtensorMap* c = reinterpret_cast<const CUtensorMap*>(twd);
    const CUtensorMap* d = reinterpret_cast<const CUtensorMap*>(ty);
    if (p.Dk < 64 || p.Dk > 256 || p.Dk % 64 != 0 || p.n_slices < 1 || p.stages < 2 || p.stages > kMaxStages) {
        *why = "inconsistent fused launch";
        return KT_ERR_INVALID;
    }
#define KT_FUSED(E)                                                                                 \
    return dtype == KT_BF16 ? launch_fused_t<E, KT_BF16>(a, b, c, d, p, grid, smem, stream, pdl, why) \
                            : launch_fused_t<E, KT_F16>(a, b, c, d, p, grid, smem, stream, pdl, why)
    switch (epi) {
        case EPI_GELU_ERF: KT_FUSED(EPI_GELU_ERF);
        case EPI_GELU_TANH: KT_FUSED(EPI_GELU_TANH);
        case EPI_GEGLU: KT_FUSED(EPI_GEGLU);
        case EPI_NONE: KT_FUSED(EPI_NONE);
        case EPI_GELU_SIGMOID: KT_FUSED(EPI_GELU_SIGMOID);
        case EPI_SILU: KT_FUSED(EPI_SILU);
    }
#undef KT_FUSED
    *why = "unknown epilogue kind";
    return KT_ERR_INVALID;
}

}  // namespace kt
