// kt_mlp_kernels.cu -- host side of the sm_103a kernels: tensor-map encoding, the
// instruction descriptor, the launch dispatch over the kernel instantiations (which
// live in kt_gemm_act.cu, kt_gemm_geglu.cu and kt_gemm_down.cu), the allocation-free
// down projection, and the small elementwise / test kernels.
#include "kt_gemm.cuh"

#include <climits>

namespace kt {

__global__ void kt_timestamp_kernel(unsigned long long* dst) { *dst = global_ns(); }

// Copy n16 16-byte words from src to dst (either may be pinned host memory mapped into the
// device's address space: the host-buffer entry point moves X in and Y out with SM loads
// and stores over the CPU-GPU link instead of copy-engine transfers).  A programmatic
// dependent of the previous kernel: lets its own dependent start at once, and waits for
// the previous kernel to complete before it reads.
__global__ void __launch_bounds__(256) kt_copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                        size_t n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four independent 16-byte loads in flight per thread
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

// Elementwise evaluation of the epilogue's fp32 activations (test hook), through the
// same pair functions the epilogues call, in the paired-instruction form (P) or the
// scalar one: elements 2j and 2j + 1 form one pair (an odd last element is paired with
// itself).  GEGLU adds -0 as both biases, which keeps every value's bits.
template <bool P>
__device__ __forceinline__ f32x2 activation_pair(int act, f32x2 x, f32x2 gate) {
    if (act == KT_ACT_GELU_ERF) return gelu_erf_f2<P>(x);
    if (act == KT_ACT_GELU_TANH) return gelu_tanh_f2<P>(x);
    if (act == KT_ACT_GEGLU) return geglu_f2<P>(x, f2(-0.0f), gate, f2(-0.0f));
    if (act == KT_ACT_GELU_SIGMOID) return gelu_sigmoid_f2<P>(x);
    if (act == KT_ACT_SILU) return silu_f2<P>(x);
    return x;
}
__global__ void kt_activation_kernel(int act, bool paired, const float* __restrict__ z,
                                     const float* __restrict__ g, float* __restrict__ out, int64_t n) {
    const int64_t pairs = (n + 1) / 2;
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < pairs; j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = 2 * j, i1 = 2 * j + 1 < n ? 2 * j + 1 : 2 * j;
        const f32x2 x = f2(z[i0], z[i1]);
        const f32x2 gate = act == KT_ACT_GEGLU ? f2(g[i0], g[i1]) : f2(0.0f);
        const f32x2 y = paired ? activation_pair<true>(act, x, gate) : activation_pair<false>(act, x, gate);
        out[i0] = y.x;
        if (i1 != i0) out[i1] = y.y;
    }
}

// LayerNorm prologue ("SDXL as a requirements inventory", section 1.3: the block's
// feed-forward reads LayerNorm(x)).  One warp per row: the row is read once (kept in
// registers as packed 16-bit vectors when D <= 2048, re-read from L1 / L2 beyond),
// mean and biased variance over D in fp32 (two passes: the variance is a sum of
// squared deviations from the mean, no cancellation), then (x - mean) / sqrt(var + eps) * gamma +
// beta rounded once to the dtype.  HBM-bound: 2 * M * D * 2 bytes.
constexpr int kLnWarps = 8;
constexpr int kLnCache = 8;  // 16-byte vectors per lane kept in registers: D <= 32 * 8 * 8

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int DT>
__global__ void __launch_bounds__(kLnWarps * 32) kt_layernorm_kernel(const uint4* __restrict__ X,
                                                                      const uint4* __restrict__ gamma,
                                                                      const uint4* __restrict__ beta, float eps,
                                                                      uint4* __restrict__ Xn, int M, int D) {
    // X may be the previous kernel's output: wait for it (no-op without a dependency)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int row = (int)blockIdx.x * kLnWarps + (threadIdx.x >> 5);
    const int nv = D >> 3;  // 16-byte vectors per row
    const bool cached = nv <= 32 * kLnCache;
    // gamma and beta, shared by the CTA's rows, staged once in shared memory (rows that fit
    // in registers); the loads overlap the rows' own
    __shared__ uint4 s_gamma[32 * kLnCache], s_beta[32 * kLnCache];
    if (cached) {
        for (int j = threadIdx.x; j < nv; j += kLnWarps * 32) {
            s_gamma[j] = gamma[j];
            s_beta[j] = beta[j];
        }
    }
    const uint4* xr = X + (size_t)(row < M ? row : 0) * (size_t)nv;
    // Statistics of the deviations from the row's first element x0: x - x0 is exact in
    // fp32 for 16-bit inputs, and the sums then carry rounding errors relative to the
    // spread of the row rather than to its mean (a row far from zero with a small spread
    // would otherwise lose the normalised value's low bits).  A row that fits in
    // registers is loaded in one go; x0 comes from lane 0's first vector.
    float x0 = 0.0f;
    uint4 c[kLnCache];
    float s = 0.0f;
    if (cached) {
#pragma unroll
        for (int i = 0; i < kLnCache; ++i) {
            const int j = lane + 32 * i;
            if (j < nv && row < M) c[i] = xr[j];
        }
        __syncthreads();  // gamma and beta staged (every thread of the CTA reaches this)
        if (row >= M) return;
        {
            float f[8];
            unpack8<DT>(c[0], f);
            x0 = __shfl_sync(0xffffffffu, f[0], 0);
        }
#pragma unroll
        for (int i = 0; i < kLnCache; ++i) {
            if (lane + 32 * i < nv) {
                float f[8];
                unpack8<DT>(c[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) s += f[e] - x0;
            }
        }
    } else {
        if (row >= M) return;
        {
            float f[8];
            unpack8<DT>(xr[0], f);
            x0 = f[0];
        }
        for (int j = lane; j < nv; j += 32) {
            float f[8];
            unpack8<DT>(xr[j], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) s += f[e] - x0;
        }
    }
    const float dmean = warp_sum(s) / (float)D;  // mean - x0
    float q = 0.0f;
    if (cached) {
#pragma unroll
        for (int i = 0; i < kLnCache; ++i) {
            if (lane + 32 * i < nv) {
                float f[8];
                unpack8<DT>(c[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float dv = (f[e] - x0) - dmean;
                    q += dv * dv;
                }
            }
        }
    } else {
        for (int j = lane; j < nv; j += 32) {
            float f[8];
            unpack8<DT>(xr[j], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dv = (f[e] - x0) - dmean;
                q += dv * dv;
            }
        }
    }
    const float var = warp_sum(q) / (float)D;
    const float rstd = 1.0f / sqrtf(var + eps);
    uint4* yr = Xn + (size_t)row * (size_t)nv;
    auto emit = [&](int j, const uint4& w, const uint4& gw, const uint4& bw) {
        float f[8], g[8], b[8], y[8];
        unpack8<DT>(w, f);
        unpack8<DT>(gw, g);
        unpack8<DT>(bw, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = ((f[e] - x0) - dmean) * rstd * g[e] + b[e];
        uint4 o;
        o.x = pack2<DT>(y[0], y[1]);
        o.y = pack2<DT>(y[2], y[3]);
        o.z = pack2<DT>(y[4], y[5]);
        o.w = pack2<DT>(y[6], y[7]);
        yr[j] = o;
    };
    if (cached) {
#pragma unroll
        for (int i = 0; i < kLnCache; ++i)
            if (lane + 32 * i < nv) emit(lane + 32 * i, c[i], s_gamma[lane + 32 * i], s_beta[lane + 32 * i]);
    } else {
        for (int j = lane; j < nv; j += 32) emit(j, xr[j], gamma[j], beta[j]);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

uint32_t make_idesc(int dtype, int n, int m, int b_kmajor) {
    uint32_t d = 0;
    d |= 1u << 4;                                   // D (accumulator) format: f32
    d |= (dtype == KT_BF16 ? 1u : 0u) << 7;         // A format: f16 = 0, bf16 = 1
    d |= (dtype == KT_BF16 ? 1u : 0u) << 10;        // B format
    /* bit 15 = 0: A is K-major */
    d |= (b_kmajor ? 0u : 1u) << 16;                // B: MN-major (1) or K-major (0)
    d |= (uint32_t)(n >> 3) << 17;                  // N >> 3
    d |= (uint32_t)(m >> 4) << 24;                  // M >> 4 (256 for a CTA pair)
    return d;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace


// ---------------------------------------------------------------------------
// Allocation-free down projection (kt_down_proj_noalloc)
// ---------------------------------------------------------------------------
// Scratch of the allocation-free entry point, laid out as [error word, padded to
// 256 B][split-K tile counters, padded to 256 B][fp32 split-K partials].  It is
// file-scope device memory: every GPU that loads this library holds these bytes
// until the process exits.  Host code must not use the symbol itself (on the host it
// is only a stand-in); it uses the device address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char* g_noalloc_ptr[kNoAllocMaxDevices] = {};  // device address of the scratch, per device
int g_noalloc_sms[kNoAllocMaxDevices] = {};
thread_local char g_noalloc_msg[192];
}  // namespace

kt_status noalloc_down_proj(int64_t M, int64_t F, int64_t D, int dtype, const void* H, const void* W_down,
                            const void* b_down, void* Y, void* stream, const char** why) {
    if (M < 1 || F < 1 || D < 1) {
        *why = "M, F and D must be positive";
        return KT_ERR_INVALID;
    }
    if (dtype != KT_F16 && dtype != KT_BF16) {
        *why = "unknown dtype";
        return KT_ERR_INVALID;
    }
    auto misaligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
    if (!H || !W_down || !Y || misaligned(H) || misaligned(W_down) || misaligned(Y) || misaligned(b_down)) {
        *why = "H, W_down and Y must be non-NULL, and all pointers 16-byte aligned";
        return KT_ERR_INVALID;
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    if (dev < 0 || dev >= kNoAllocMaxDevices) {
        *why = "device ordinal beyond the allocation-free entry point's table";
        return KT_ERR_UNSUPPORTED;
    }
    unsigned char* scratch = nullptr;
    int sms = 0;
    {
        // once per device, with that device current: its SM count and the device
        // address of the static scratch
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_ptr[dev]) {
            int major = 0, minor = 0, count = 0;
            if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
                (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
                *why = cudaGetErrorString(e);
                return KT_ERR_CUDA;
            }
            if (major != 10 || minor != 3) {
                *why = "this library is built for sm_103a (GB300)";
                return KT_ERR_UNSUPPORTED;
            }
            void* addr = nullptr;
            if ((e = cudaGetSymbolAddress(&addr, g_noalloc_scratch)) != cudaSuccess || !addr) {
                *why = e != cudaSuccess ? cudaGetErrorString(e) : "cudaGetSymbolAddress returned NULL";
                return KT_ERR_CUDA;
            }
            g_noalloc_sms[dev] = count;
            g_noalloc_ptr[dev] = static_cast<unsigned char*>(addr);
        }
        scratch = g_noalloc_ptr[dev];
        sms = g_noalloc_sms[dev];
    }
    // the tile plan of the MLP's down projection, with the split-K reduction through this
    // entry point's scratch (not through a cluster's shared memory)
    PlanChoice pc;
    kt_status st = plan_choose(M, D, F, KT_ACT_NONE, sms, &pc, why, /*allow_cluster_sk=*/false, KT_W_IN_OUT,
                               KT_H_MEMORY, /*allow_one_launch=*/false);
    if (st != KT_OK) return st;
    const GemmConfig& g = pc.down;
    const size_t n_counters = (size_t)g.tiles_m * (size_t)g.tiles_n * (size_t)g.pair;
    const size_t counter_bytes = (n_counters * 4 + 255) / 256 * 256;
    const size_t part_bytes =
        g.split_k > 1 ? (size_t)g.split_k * g.tiles_m * g.pair * kBM * (size_t)g.tiles_n * g.BN * sizeof(float) : 0;
    const size_t need = 256 + counter_bytes + part_bytes;
    if (need > kNoAllocScratchBytes) {
        std::snprintf(g_noalloc_msg, sizeof(g_noalloc_msg),
                      "this problem needs %zu bytes of scratch; the allocation-free entry point has %zu",
                      need, (size_t)kNoAllocScratchBytes);
        *why = g_noalloc_msg;
        return KT_ERR_UNSUPPORTED;
    }
    // the error word and the tile counters must start at zero
    if ((e = cudaMemsetAsync(scratch, 0, 256 + counter_bytes, static_cast<cudaStream_t>(stream))) != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    alignas(64) CUtensorMap tmA, tmB, tmC;
    if (!encode_tmap(&tmA, H, dtype, M, F, kBM, kAtomK, 128, why) ||
        !encode_tmap(&tmB, W_down, dtype, F, D, g.bk, b_box_cols(g.BN, g.pair), 2 * b_box_cols(g.BN, g.pair), why) ||
        !encode_tmap(&tmC, Y, dtype, M, D, 32, kStoreCols, 64, why))
        return KT_ERR_CUDA;
    GemmParams q;
    std::memset(&q, 0, sizeof(q));
    q.M = (int)M;
    q.N = (int)D;
    q.K = (int)F;
    q.BN = g.BN;
    q.stages = g.stages;
    q.split_k = g.split_k;
    q.tiles_m = g.tiles_m;
    q.tiles_n = g.tiles_n;
    q.kblocks = g.kblocks;
    q.kblocks_per_split = g.kblocks_per_split;
    q.num_tiles = g.tiles_m * g.tiles_n * g.split_k;
    q.pair = g.pair;
    q.cluster_sk = 0;
    q.idesc = make_idesc(dtype, g.BN, kBM * g.pair);
    q.bk = g.bk;
    q.dbl_staging = g.dbl_staging;
    q.a_bytes = kBM * g.bk * 2;
    q.b_bytes = (uint32_t)b_tile_bytes(g.BN, g.pair, g.bk, 0);
    q.stage_bytes = (uint32_t)stage_bytes(g.BN, 1, g.pair, g.bk);
    q.acc_bufs = 2u;
    q.bias = b_down;
    q.error = reinterpret_cast<int*>(scratch);
    q.counters = reinterpret_cast<int*>(scratch + 256);
    q.partials = reinterpret_cast<float*>(scratch + 256 + counter_bytes);
    q.wait_limit_ns = 4000000000ull;
    return launch_gemm(EPI_DOWN, dtype, &tmA, &tmB, &tmC, q, g.grid, g.smem_bytes, stream, false, why);
}

kt_status launch_copy16(const void* src, void* dst, size_t bytes, int grid, void* stream, const char** why) {
    if (bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u)) {
        *why = "copy: 16-byte aligned pointers and a multiple of 16 bytes";
        return KT_ERR_INVALID;
    }
    if (bytes == 0) return KT_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max(1, grid), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kt_copy16_kernel, reinterpret_cast<const uint4*>(src),
                                       reinterpret_cast<uint4*>(dst), bytes / 16);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

kt_status launch_timestamp(void* dst, void* stream, const char** why) {
    kt_timestamp_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<unsigned long long*>(dst));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

kt_status launch_layernorm(int dtype, const void* X, const void* gamma, const void* beta, float eps, void* Xn,
                           int64_t M, int64_t D, void* stream, const char** why) {
    if (M < 1 || D < 8 || D % 8 != 0 || M > INT32_MAX || D > INT32_MAX) {
        *why = "LayerNorm: M >= 1 and D a positive multiple of 8";
        return KT_ERR_INVALID;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + kLnWarps - 1) / kLnWarps), 1, 1);
    cfg.blockDim = dim3(kLnWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint4* x = static_cast<const uint4*>(X);
    const uint4* g = static_cast<const uint4*>(gamma);
    const uint4* b = static_cast<const uint4*>(beta);
    uint4* y = static_cast<uint4*>(Xn);
    cudaError_t e = dtype == KT_BF16
                        ? cudaLaunchKernelEx(&cfg, kt_layernorm_kernel<KT_BF16>, x, g, b, eps, y, (int)M, (int)D)
                        : cudaLaunchKernelEx(&cfg, kt_layernorm_kernel<KT_F16>, x, g, b, eps, y, (int)M, (int)D);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

kt_status launch_activation(int act, bool paired, const float* z, const float* g, float* out, int64_t n,
                            void* stream, const char** why) {
    const int64_t blocks = n == 0 ? 0 : std::min<int64_t>((n + 255) / 256, 4096);
    if (blocks > 0)
        kt_activation_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(act, paired, z, g, out, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

bool encode_tmap(void* tmap128, const void* base, int dtype, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, int swizzle_bytes, const char** why) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) {
        *why = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(tmap128),
                    dtype == KT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_bytes == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                    : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected the tensor (alignment, stride or box)";
        return false;
    }
    return true;
}

kt_status launch_gemm(int epi, int dtype, const void* tmA, const void* tmB, const void* tmC, const GemmParams& p,
                      int grid, int smem_bytes, void* stream, bool pdl, const char** why) {
    const CUtensorMap* a = reinterpret_cast<const CUtensorMap*>(tmA);
    const CUtensorMap* b = reinterpret_cast<const CUtensorMap*>(tmB);
    const CUtensorMap* c = reinterpret_cast<const CUtensorMap*>(tmC);
    if (p.pair == 2 && (grid % 2) != 0) {
        *why = "a CTA-pair launch needs an even grid";
        return KT_ERR_INVALID;
    }
    if (p.cluster_sk && (p.pair != 1 || epi != EPI_DOWN || p.split_k < 2 || p.split_k > 8 ||
                         grid != p.num_tiles || grid % p.split_k != 0 ||
                         (uint64_t)p.stages * p.stage_bytes < (uint64_t)kBM * (uint64_t)p.BN * 4u)) {
        *why = "inconsistent cluster split-K launch";
        return KT_ERR_INVALID;
    }
    switch (epi) {
        case EPI_GELU_ERF:
        case EPI_GELU_TANH:
        case EPI_GELU_SIGMOID:
        case EPI_SILU:
        case EPI_NONE: return launch_gemm_act(epi, dtype, a, b, c, p, grid, smem_bytes, stream, pdl, why);
        case EPI_GEGLU: return launch_gemm_geglu(dtype, a, b, c, p, grid, smem_bytes, stream, pdl, why);
        case EPI_DOWN: return launch_gemm_down(dtype, a, b, c, p, grid, smem_bytes, stream, pdl, why);
    }
    *why = "unknown epilogue kind";
    return KT_ERR_INVALID;
}

kt_status launch_mlp_two(int epi, int dtype, const void* const* maps, const GemmParams& up, const GemmParams& down,
                         int grid, int smem_bytes, void* stream, bool pdl, const char** why) {
    const CUtensorMap* m[6];
    for (int i = 0; i < 6; ++i) m[i] = reinterpret_cast<const CUtensorMap*>(maps[i]);
    // the down projection's K splits (if any) are summed by the last CTA of each tile
    // through the partials and tile counters
    if (up.pair != down.pair || (up.pair == 2 && grid % 2 != 0) || down.split_k < 1 || up.split_k != 1 ||
        (down.split_k > 1 && (down.partials == nullptr || down.counters == nullptr)) ||
        up.cluster_sk || down.cluster_sk || up.stages != down.stages || up.stage_bytes != down.stage_bytes ||
        up.dbl_staging != down.dbl_staging || up.sched == nullptr || grid / up.pair > up.num_tiles + down.num_tiles) {
        *why = "inconsistent one-launch configuration";
        return KT_ERR_INVALID;
    }
    switch (epi) {
        case EPI_GEGLU: return launch_mlp_two_geglu(dtype, m, up, down, grid, smem_bytes, stream, pdl, why);
        case EPI_GELU_ERF:
        case EPI_GELU_TANH:
        case EPI_GELU_SIGMOID:
        case EPI_SILU:
        case EPI_NONE:
            return dtype == KT_F16 ? launch_mlp_two_act_f16(epi, m, up, down, grid, smem_bytes, stream, pdl, why)
                                   : launch_mlp_two_act_bf16(epi, m, up, down, grid, smem_bytes, stream, pdl, why);
    }
    *why = "unknown epilogue kind";
    return KT_ERR_INVALID;
}

}  // namespace kt
