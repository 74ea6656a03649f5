// kt_mlp_abi.cpp -- the extern "C" boundary: validation, plan ownership, launches.
//
// A plan binds a problem (M, D, F, act, dtype, bias and the kt_mlp_options flags)
// to the device current at plan time, holds the planner's choice and owns the
// device workspace: the intermediate H[M][F], the split-K fp32 partials, the
// split-K tile counters, the device error word and, with a LayerNorm prologue, the
// normalised Xn[M][D].  A run encodes (and caches, per pointer set) the TMA tensor
// maps and enqueues on the caller's stream: the LayerNorm kernel (if any), the up
// projection with its fused epilogue, then the down projection, each a
// programmatic dependent launch of the one before.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kt_internal.h"

namespace {

thread_local std::string g_last_error;

kt_status fail(kt_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

kt_status ok() {
    g_last_error.clear();
    return KT_OK;
}

kt_status cuda_fail(const char* what, cudaError_t e) {
    return fail(KT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

const char* act_name(int a) {
    switch (a) {
        case KT_ACT_GELU_ERF: return "gelu_erf";
        case KT_ACT_GELU_TANH: return "gelu_tanh";
        case KT_ACT_GEGLU: return "geglu";
        case KT_ACT_NONE: return "none";
        case KT_ACT_GELU_SIGMOID: return "gelu_sigmoid";
        case KT_ACT_SILU: return "silu";
    }
    return "?";
}

kt_status validate_problem(int64_t M, int64_t D, int64_t F, int act, int dtype, int bias) {
    if (M < 1 || D < 1 || F < 1) return fail(KT_ERR_INVALID, "M, D and F must be positive");
    if (act < KT_ACT_GELU_ERF || act > KT_ACT_SILU) return fail(KT_ERR_INVALID, "unknown activation");
    if (dtype != KT_F16 && dtype != KT_BF16) return fail(KT_ERR_INVALID, "unknown dtype");
    if (bias != 0 && bias != 1) return fail(KT_ERR_INVALID, "bias must be 0 or 1");
    return KT_OK;
}

kt_status validate_options(const kt_mlp_options* o) {
    if (!o) return fail(KT_ERR_INVALID, "options is NULL");
    kt_status s = validate_problem(o->M, o->D, o->F, o->act, o->dtype, o->bias);
    if (s != KT_OK) return s;
    if ((o->residual != 0 && o->residual != 1) || (o->layernorm != 0 && o->layernorm != 1))
        return fail(KT_ERR_INVALID, "residual and layernorm must be 0 or 1");
    if (o->weight_layout != KT_W_IN_OUT && o->weight_layout != KT_W_OUT_IN)
        return fail(KT_ERR_INVALID, "unknown weight layout");
    if (o->layernorm && !(o->ln_eps > 0.0f && o->ln_eps < 3.0e38f))
        return fail(KT_ERR_INVALID, "ln_eps must be positive and finite");
    if (o->launches != KT_LAUNCH_AUTO && o->launches != KT_LAUNCH_ONE && o->launches != KT_LAUNCH_TWO)
        return fail(KT_ERR_INVALID, "launches must be KT_LAUNCH_AUTO, KT_LAUNCH_ONE or KT_LAUNCH_TWO");
    if (o->h_path != KT_H_AUTO && o->h_path != KT_H_MEMORY && o->h_path != KT_H_ON_CHIP)
        return fail(KT_ERR_INVALID, "unknown H path");
    return KT_OK;
}

kt_mlp_options base_options(int64_t M, int64_t D, int64_t F, int act, int dtype, int bias) {
    kt_mlp_options o;
    std::memset(&o, 0, sizeof(o));
    o.M = M; o.D = D; o.F = F;
    o.act = act; o.dtype = dtype; o.bias = bias;
    o.weight_layout = KT_W_IN_OUT;
    o.h_path = KT_H_MEMORY;
    return o;
}

}  // namespace

struct kt_mlp_plan_s {
    int64_t M, D, F, F_up;
    int act, dtype, bias;
    int residual = 0, layernorm = 0, w_layout = KT_W_IN_OUT;
    float ln_eps = 0.0f;
    int device, num_sms;
    kt::PlanChoice choice;
    // device workspace (one allocation each)
    void* H = nullptr;          // [M][F]
    float* partials = nullptr;  // [SK][tiles_m*128][tiles_n*BN] when the down GEMM splits K
    int* flags = nullptr;       // [0] error word, [2..] split-K tile counters, then row-block counters
    unsigned* ready = nullptr;  // per up-projection row block: CTA tiles of H stored (inside flags)
    unsigned* readers = nullptr;  // per row block: the down projection's waits done this run (inside flags)
    unsigned* ready_expect = nullptr;  // per row block: the down projection's waits per run (own allocation)
    int* sched = nullptr;       // one-launch plans: the work-item counters (inside flags)
    size_t flag_bytes = 0;
    void* xn = nullptr;         // [M][D] LayerNorm output (layernorm plans)
    void* x_stage = nullptr;    // [M][D] for kt_mlp_run_host
    void* y_stage = nullptr;    // [M][D]
    int64_t workspace_bytes = 0;
    // tensor maps, cached by pointer set
    alignas(64) CUtensorMap tm_x, tm_wu, tm_h, tm_wd, tm_hs, tm_ys;  // loads, then H / Y stores
    alignas(64) CUtensorMap tm_fwu, tm_fwd;  // the fused kernel's weight maps (H-on-chip plans)
    const void* c_x = nullptr;
    const void* c_wu = nullptr;
    const void* c_h = nullptr;
    const void* c_wd = nullptr;
    const void* c_y = nullptr;
    bool cache_valid = false;
    void* last_stream = nullptr;
    cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};  // timed runs, created on first use
    int inject_stall = 0;
    int64_t stall_limit_us = 0;
    unsigned long long* trace_up = nullptr;    // caller-owned device buffers, or null
    unsigned long long* trace_down = nullptr;
};

namespace {

void free_plan(kt_mlp_plan_s* p) {
    if (!p) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != p->device) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    for (cudaEvent_t e : p->ev)
        if (e) cudaEventDestroy(e);
    cudaFree(p->H);
    cudaFree(p->xn);
    cudaFree(p->ready_expect);
    cudaFree(p->partials);
    cudaFree(p->flags);
    cudaFree(p->x_stage);
    cudaFree(p->y_stage);
    if (prev >= 0 && prev != p->device) cudaSetDevice(prev);
    delete p;
}

kt::GemmParams make_params(const kt_mlp_plan_s* P, const kt::GemmConfig& g, int epi) {
    kt::GemmParams q;
    std::memset(&q, 0, sizeof(q));
    q.M = (int)g.M;
    q.N = (int)g.N;
    q.K = (int)g.K;
    q.BN = g.BN;
    q.pair = g.pair;
    q.cluster_sk = g.cluster_sk;
    q.stages = g.stages;
    q.split_k = g.split_k;
    q.tiles_m = g.tiles_m;
    q.tiles_n = g.tiles_n;
    q.kblocks = g.kblocks;
    q.kblocks_per_split = g.kblocks_per_split;
    q.num_tiles = g.tiles_m * g.tiles_n * g.split_k;
    q.gate_col = epi == kt::EPI_GEGLU ? (int)P->F : 0;
    q.b_kmajor = g.b_kmajor;
    q.dbl_staging = g.dbl_staging;
    q.idesc = kt::make_idesc(P->dtype, g.BN * g.n_b, kt::kBM * g.pair, g.b_kmajor);  // GEGLU: N = 2 BN
    q.bk = g.bk;
    q.a_bytes = kt::kBM * g.bk * 2;
    q.b_bytes = (uint32_t)kt::b_tile_bytes(g.BN, g.pair, g.bk, g.b_kmajor);
    q.b_atom_bytes = g.b_kmajor ? (uint32_t)(g.BN / g.pair) * 128u : 0u;
    q.stage_bytes = (uint32_t)kt::stage_bytes(g.BN, g.n_b, g.pair, g.bk, g.b_kmajor);
    q.acc_bufs = 2u;
    q.geglu_share = epi == kt::EPI_GEGLU ? (uint32_t)(g.BN / g.pair) : 0u;
    q.error = P->flags;
    q.wait_limit_ns = 4000000000ull;  // 4 s: far beyond any legitimate wait
    q.stall_limit_ns = (unsigned long long)P->stall_limit_us * 1000ull;
    return q;
}

kt_status run_impl(kt_mlp_plan_t P, const kt_mlp_tensors& t, void* H, void* stream, bool timed = false) {
    if (!P) return fail(KT_ERR_INVALID, "plan is NULL");
    if (!t.X || !t.W_up || !t.W_down || !t.Y || !H) return fail(KT_ERR_INVALID, "X, W_up, W_down, Y (and H) must be non-NULL");
    if (P->bias && (!t.b_up || !t.b_down)) return fail(KT_ERR_INVALID, "plan has bias = 1: b_up and b_down are required");
    if (!P->bias && (t.b_up || t.b_down)) return fail(KT_ERR_INVALID, "plan has bias = 0: b_up and b_down must be NULL");
    if (P->residual != (t.R != nullptr)) return fail(KT_ERR_INVALID, "R must be given iff the plan has residual = 1");
    if (P->layernorm != (t.ln_gamma != nullptr) || P->layernorm != (t.ln_beta != nullptr))
        return fail(KT_ERR_INVALID, "ln_gamma and ln_beta must be given iff the plan has layernorm = 1");
    if (!aligned16(t.X) || !aligned16(t.W_up) || !aligned16(t.W_down) || !aligned16(t.Y) || !aligned16(H) ||
        !aligned16(t.b_up) || !aligned16(t.b_down) || !aligned16(t.R) || !aligned16(t.ln_gamma) ||
        !aligned16(t.ln_beta))
        return fail(KT_ERR_INVALID, "device pointers must be 16-byte aligned");
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != P->device) return fail(KT_ERR_INVALID, "the current device is not the plan's device");

    const char* why = "";
    if (P->choice.h_on_chip && t.H_out)
        return fail(KT_ERR_INVALID, "an H-on-chip plan keeps H on chip: H_out must be NULL");
    const void* A_up = P->layernorm ? P->xn : t.X;
    if (!P->cache_valid || P->c_x != A_up || P->c_wu != t.W_up || P->c_h != H || P->c_wd != t.W_down ||
        P->c_y != t.Y) {
        // A operands: [rows][K] K-major, box 128 rows x 64 columns, 128-byte swizzle.
        // B operands [K][N] (N-major): box bk rows (K) x 64 columns (N), 128-byte swizzle,
        // or x 32 columns, 64-byte swizzle (b_box_cols); [N][K] (K-major): box (BN / pair)
        // rows (N) x 64 columns (K), 128-byte swizzle.
        // Stores of H and Y: box 32 rows x 32 columns, 64-byte swizzle.
        const kt::GemmConfig& u = P->choice.up;
        const kt::GemmConfig& d = P->choice.down;
        const bool km = P->w_layout == KT_W_OUT_IN;
        bool good =
            kt::encode_tmap(&P->tm_x, A_up, P->dtype, P->M, P->D, kt::kBM, kt::kAtomK, 128, &why) &&
            (km ? kt::encode_tmap(&P->tm_wu, t.W_up, P->dtype, P->F_up, P->D, u.BN / u.pair, 64, 128, &why)
                : kt::encode_tmap(&P->tm_wu, t.W_up, P->dtype, P->D, P->F_up, u.bk, kt::b_box_cols(u.BN, u.pair),
                                  2 * kt::b_box_cols(u.BN, u.pair), &why)) &&
            kt::encode_tmap(&P->tm_h, H, P->dtype, P->M, P->F, kt::kBM, kt::kAtomK, 128, &why) &&
            (km ? kt::encode_tmap(&P->tm_wd, t.W_down, P->dtype, P->D, P->F, d.BN / d.pair, 64, 128, &why)
                : kt::encode_tmap(&P->tm_wd, t.W_down, P->dtype, P->F, P->D, d.bk, kt::b_box_cols(d.BN, d.pair),
                                  2 * kt::b_box_cols(d.BN, d.pair), &why)) &&
            kt::encode_tmap(&P->tm_hs, H, P->dtype, P->M, P->F, 32, kt::kStoreCols, 64, &why) &&
            kt::encode_tmap(&P->tm_ys, t.Y, P->dtype, P->M, P->D, 32, kt::kStoreCols, 64, &why) &&
            (!P->choice.h_on_chip ||
             (kt::encode_tmap(&P->tm_fwu, t.W_up, P->dtype, P->D, P->F_up, P->choice.fused.Dk, 64, 128, &why) &&
              kt::encode_tmap(&P->tm_fwd, t.W_down, P->dtype, P->F, P->D, kt::kFusedSlice, 64, 128, &why)));
        if (!good) {
            P->cache_valid = false;
            return fail(KT_ERR_CUDA, std::string("tensor map: ") + why);
        }
        P->c_x = A_up;
        P->c_wu = t.W_up;
        P->c_h = H;
        P->c_wd = t.W_down;
        P->c_y = t.Y;
        P->cache_valid = true;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (timed) cudaEventRecord(P->ev[0], st);
    kt_status s;
    if (P->layernorm) {
        s = kt::launch_layernorm(P->dtype, t.X, t.ln_gamma, t.ln_beta, P->ln_eps, P->xn, P->M, P->D, stream, &why);
        if (s != KT_OK) return fail(s, std::string("LayerNorm launch: ") + why);
    }
    if (timed) cudaEventRecord(P->ev[1], st);

    const int epi_up = kt::up_epilogue(P->act);
    if (P->choice.h_on_chip) {
        // one kernel: H stays on chip
        const kt::FusedConfig& f = P->choice.fused;
        kt::FusedParams fp;
        std::memset(&fp, 0, sizeof(fp));
        fp.M = (int)P->M; fp.D = (int)P->D; fp.F = (int)P->F;
        fp.Dk = f.Dk; fp.n_slices = f.n_slices; fp.tiles_m = f.tiles_m; fp.stages = f.stages;
        fp.gate_col = P->act == KT_ACT_GEGLU ? (int)P->F : 0;
        fp.idesc_up = kt::make_idesc(P->dtype, kt::kFusedSlice, kt::kBM, 0);
        fp.idesc_dn = kt::make_idesc(P->dtype, f.Dk, kt::kBM, 0);
        fp.x_bytes = f.x_bytes; fp.stage_bytes = f.stage_bytes; fp.wup_bytes = f.wup_bytes; fp.wdn_bytes = f.wdn_bytes;
        fp.bias_up = P->bias ? t.b_up : nullptr;
        fp.bias_dn = P->bias ? t.b_down : nullptr;
        fp.residual = t.R;
        fp.error = P->flags;
        fp.wait_limit_ns = 4000000000ull;
        fp.pdl_wait = 1;
        s = kt::launch_fused(epi_up, P->dtype, &P->tm_x, &P->tm_fwu, &P->tm_fwd, &P->tm_ys, fp, f.grid, f.smem_bytes,
                             stream, !timed, &why);
        if (s != KT_OK) return fail(s, std::string("fused launch: ") + why);
        if (timed) {
            cudaEventRecord(P->ev[2], st);
            cudaEventRecord(P->ev[3], st);
        }
        P->last_stream = stream;
        return ok();
    }
    // the down projection's producer waits on per-row-block counters of stored H tiles
    // (instead of the whole up grid); its last reader of a row block resets them
    const unsigned per_block = (unsigned)(P->choice.up.tiles_n * P->choice.up.pair);
    kt::GemmParams up = make_params(P, P->choice.up, epi_up);
    up.bias = P->bias ? t.b_up : nullptr;
    up.inject_stall = P->inject_stall;
    up.pdl_wait = 1;
    up.trace = P->trace_up;
    up.ready = P->ready;

    kt::GemmParams dn = make_params(P, P->choice.down, kt::EPI_DOWN);
    dn.bias = P->bias ? t.b_down : nullptr;
    dn.residual = t.R;
    dn.partials = P->partials;
    dn.counters = P->flags + 2;  // 8-byte aligned: the reduce-scatter's counters are 64-bit
    dn.pdl_wait = 1;
    dn.trace = P->trace_down;
    dn.ready = P->ready;
    dn.ready_readers = P->readers;
    dn.ready_expect = P->ready_expect;
    dn.ready_target = per_block;
    dn.ready_rows = kt::kBM * P->choice.up.pair;
    if (P->choice.one_launch) {
        // both projections in one launch: one shared-memory ring, tiles from one queue; a
        // down projection split along K reduce-scatters its partials among the splits (GEGLU:
        // the last split to arrive sums them)
        up.stage_bytes = dn.stage_bytes = (uint32_t)P->choice.one_slot;
        dn.rs_sk = dn.split_k > 1 && P->act != KT_ACT_GEGLU ? 1 : 0;
        up.sched = dn.sched = P->sched;
        up.pdl_wait = dn.pdl_wait = 1;
        const void* maps[6] = {&P->tm_x, &P->tm_wu, &P->tm_hs, &P->tm_h, &P->tm_wd, &P->tm_ys};
        s = kt::launch_mlp_two(epi_up, P->dtype, maps, up, dn, P->choice.one_grid, P->choice.one_smem, stream, !timed,
                               &why);
        if (s != KT_OK) return fail(s, std::string("one-launch MLP: ") + why);
        if (timed) {
            cudaEventRecord(P->ev[2], st);
            cudaEventRecord(P->ev[3], st);
        }
        P->last_stream = stream;
        return ok();
    }
    s = kt::launch_gemm(epi_up, P->dtype, &P->tm_x, &P->tm_wu, &P->tm_hs, up, P->choice.up.grid,
                        P->choice.up.smem_bytes, stream, !timed, &why);
    if (s != KT_OK) return fail(s, std::string("up projection launch: ") + why);
    if (timed) cudaEventRecord(P->ev[2], st);
    s = kt::launch_gemm(kt::EPI_DOWN, P->dtype, &P->tm_h, &P->tm_wd, &P->tm_ys, dn, P->choice.down.grid,
                        P->choice.down.smem_bytes, stream, !timed, &why);
    if (s != KT_OK) return fail(s, std::string("down projection launch: ") + why);
    if (timed) cudaEventRecord(P->ev[3], st);
    P->last_stream = stream;
    return ok();
}

kt_mlp_tensors base_tensors(const void* X, const void* W_up, const void* W_down, const void* b_up,
                            const void* b_down, void* Y) {
    kt_mlp_tensors t;
    std::memset(&t, 0, sizeof(t));
    t.X = X; t.W_up = W_up; t.W_down = W_down; t.b_up = b_up; t.b_down = b_down; t.Y = Y;
    return t;
}

kt_status timed_impl(kt_mlp_plan_t plan, const kt_mlp_tensors& t, void* stream, float* ms3) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    for (cudaEvent_t& e : plan->ev) {
        if (!e) {
            cudaError_t ce = cudaEventCreate(&e);
            if (ce != cudaSuccess) return cuda_fail("cudaEventCreate", ce);
        }
    }
    kt_status s = run_impl(plan, t, t.H_out ? t.H_out : plan->H, stream, true);
    if (s != KT_OK) return s;
    cudaError_t e = cudaEventSynchronize(plan->ev[3]);
    if (e != cudaSuccess) return cuda_fail("cudaEventSynchronize", e);
    for (int i = 0; i < 3; ++i) {
        ms3[i] = 0.0f;
        cudaEventElapsedTime(&ms3[i], plan->ev[i], plan->ev[i + 1]);
    }
    return ok();
}

kt_status create_plan(const kt_mlp_options& o, kt_mlp_plan_t* out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDeviceProperties", e);
    if (prop.major != 10 || prop.minor != 3) {
        char buf[160];
        std::snprintf(buf, sizeof(buf), "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev,
                      prop.major, prop.minor);
        return fail(KT_ERR_UNSUPPORTED, buf);
    }
    kt_mlp_plan_s* P = new (std::nothrow) kt_mlp_plan_s();
    if (!P) return fail(KT_ERR_NOMEM, "host allocation of the plan failed");
    const int64_t M = o.M, D = o.D, F = o.F;
    P->M = M; P->D = D; P->F = F;
    P->F_up = o.act == KT_ACT_GEGLU ? 2 * F : F;
    P->act = o.act; P->dtype = o.dtype; P->bias = o.bias;
    P->residual = o.residual; P->layernorm = o.layernorm; P->w_layout = o.weight_layout;
    P->ln_eps = o.layernorm ? o.ln_eps : 0.0f;
    P->device = dev;
    P->num_sms = prop.multiProcessorCount;
    const char* why = "";
    kt_status s = kt::plan_choose(M, D, F, o.act, P->num_sms, &P->choice, &why, true, o.weight_layout, o.h_path,
                                  true, o.launches);
    if (s != KT_OK) {
        delete P;
        return fail(s, why);
    }
    const kt::GemmConfig& dn = P->choice.down;
    const kt::GemmConfig& up = P->choice.up;
    size_t h_bytes = (size_t)M * (size_t)F * 2;
    // two per 128-row half tile: split-K arrivals, and (reduce-scatter) splits done reading
    size_t n_counters = 2 * (size_t)dn.tiles_m * dn.tiles_n * dn.pair;
    size_t n_ready = (size_t)up.tiles_m;                               // one per up row block
    // [0] error word, [1] padding, [2 ..) split-K counters, readiness counters, work counters
    size_t flag_bytes = 4 * (2 + n_counters + 2 * n_ready + 2);
    size_t part_bytes = dn.split_k > 1
                            ? (size_t)dn.split_k * dn.tiles_m * dn.pair * kt::kBM * (size_t)dn.tiles_n * dn.BN * 4
                            : 0;
    size_t io_bytes = (size_t)M * (size_t)D * 2;
    size_t xn_bytes = o.layernorm ? io_bytes : 0;
    if ((e = cudaMalloc(&P->H, h_bytes)) != cudaSuccess ||
        (e = cudaMalloc(reinterpret_cast<void**>(&P->flags), flag_bytes)) != cudaSuccess ||
        (part_bytes && (e = cudaMalloc(reinterpret_cast<void**>(&P->partials), part_bytes)) != cudaSuccess) ||
        (xn_bytes && (e = cudaMalloc(&P->xn, xn_bytes)) != cudaSuccess) ||
        (e = cudaMalloc(&P->x_stage, io_bytes)) != cudaSuccess ||
        (e = cudaMalloc(&P->y_stage, io_bytes)) != cudaSuccess) {
        free_plan(P);
        cudaGetLastError();
        return fail(KT_ERR_NOMEM, std::string("workspace allocation: ") + cudaGetErrorString(e));
    }
    if ((e = cudaMemset(P->flags, 0, flag_bytes)) != cudaSuccess) {
        free_plan(P);
        return cuda_fail("cudaMemset", e);
    }
    P->ready = reinterpret_cast<unsigned*>(P->flags + 2 + n_counters);
    P->readers = P->ready + n_ready;
    P->sched = P->flags + 2 + n_counters + 2 * n_ready;
    P->flag_bytes = flag_bytes;
    {
        // how many times this plan's down projection waits on each up row block per run:
        // every tile (and split) of a 128-row CTA share waits on the row blocks it covers
        std::vector<unsigned> expect(n_ready, 0u);
        const int64_t rows_up = (int64_t)kt::kBM * up.pair;
        for (int64_t tm = 0; tm < dn.tiles_m; ++tm)
            for (int r = 0; r < dn.pair; ++r) {
                const int64_t m0 = tm * kt::kBM * dn.pair + (int64_t)r * kt::kBM;
                if (m0 >= M) continue;
                const int64_t m1 = std::min<int64_t>(m0 + kt::kBM, M) - 1;
                for (int64_t rb = m0 / rows_up; rb <= m1 / rows_up; ++rb)
                    expect[(size_t)rb] += (unsigned)(dn.tiles_n * dn.split_k);
            }
        if ((e = cudaMalloc(reinterpret_cast<void**>(&P->ready_expect), 4 * n_ready)) != cudaSuccess ||
            (e = cudaMemcpy(P->ready_expect, expect.data(), 4 * n_ready, cudaMemcpyHostToDevice)) != cudaSuccess) {
            free_plan(P);
            cudaGetLastError();
            return fail(KT_ERR_NOMEM, std::string("workspace allocation: ") + cudaGetErrorString(e));
        }
    }
    P->workspace_bytes =
        (int64_t)(h_bytes + flag_bytes + 4 * n_ready + part_bytes + xn_bytes + 2 * io_bytes);
    *out = P;
    return ok();
}

void fill_one_launch(const kt::PlanChoice& c, kt_plan_info* out) {
    out->one_launch = c.one_launch;
    if (c.one_launch) {
        out->one_launch_grid = c.one_grid;
        out->one_launch_stages = c.one_stages;
        out->one_launch_smem_bytes = c.one_smem;
        out->one_launch_est_us = c.one_est_us;
    }
}

kt_status info_impl(const kt_mlp_options& o, int num_sms, kt_plan_info* out) {
    kt::PlanChoice c;
    const char* why = "";
    kt_status s = kt::plan_choose(o.M, o.D, o.F, o.act, num_sms, &c, &why, true, o.weight_layout, o.h_path, true,
                                  o.launches);
    if (s != KT_OK) return fail(s, why);
    std::memset(out, 0, sizeof(*out));
    out->M = o.M; out->D = o.D; out->F = o.F;
    out->act = o.act; out->dtype = o.dtype; out->bias = o.bias;
    out->num_sms = num_sms;
    out->residual = o.residual; out->layernorm = o.layernorm; out->weight_layout = o.weight_layout;
    out->ln_eps = o.layernorm ? o.ln_eps : 0.0f;
    out->h_on_chip = c.h_on_chip;
    if (c.h_on_chip) {
        out->fused_grid = c.fused.grid;
        out->fused_stages = c.fused.stages;
        out->fused_smem_bytes = c.fused.smem_bytes;
        out->fused_est_us = c.fused.est_us;
    }
    fill_one_launch(c, out);
    kt::plan_fill_info(c.up, &out->up);
    kt::plan_fill_info(c.down, &out->down);
    // H, error word and split-K counters, three words per up row block, host staging
    int64_t ws = o.M * o.F * 2 + 4 * (2 + 2 * (int64_t)c.down.tiles_m * c.down.tiles_n * c.down.pair) +
                 4 * 3 * (int64_t)c.up.tiles_m + 8 + 2 * 2 * o.M * o.D;
    if (c.down.split_k > 1)
        ws += (int64_t)c.down.split_k * c.down.tiles_m * c.down.pair * kt::kBM * (int64_t)c.down.tiles_n * c.down.BN * 4;
    if (o.layernorm) ws += 2 * o.M * o.D;
    out->workspace_bytes = ws;
    return ok();
}

}  // namespace

extern "C" {

int kt_mlp_abi_version(void) { return KT_MLP_ABI_VERSION; }

const char* kt_last_error(void) { return g_last_error.c_str(); }

kt_status kt_mlp_plan_info(int64_t M, int64_t D, int64_t F, kt_act act, kt_dtype dtype, int bias,
                           int num_sms, kt_plan_info* out) {
    if (!out) return fail(KT_ERR_INVALID, "out is NULL");
    kt_status s = validate_problem(M, D, F, act, dtype, bias);
    if (s != KT_OK) return s;
    return info_impl(base_options(M, D, F, act, dtype, bias), num_sms, out);
}

kt_status kt_mlp_plan_info_ex(const kt_mlp_options* options, int num_sms, kt_plan_info* out) {
    if (!out) return fail(KT_ERR_INVALID, "out is NULL");
    kt_status s = validate_options(options);
    if (s != KT_OK) return s;
    return info_impl(*options, num_sms, out);
}

kt_status kt_mlp_plan(int64_t M, int64_t D, int64_t F, kt_act act, kt_dtype dtype, int bias,
                      kt_mlp_plan_t* out) {
    if (!out) return fail(KT_ERR_INVALID, "out is NULL");
    *out = nullptr;
    kt_status s = validate_problem(M, D, F, act, dtype, bias);
    if (s != KT_OK) return s;
    return create_plan(base_options(M, D, F, act, dtype, bias), out);
}

kt_status kt_mlp_plan_ex(const kt_mlp_options* options, kt_mlp_plan_t* out) {
    if (!out) return fail(KT_ERR_INVALID, "out is NULL");
    *out = nullptr;
    kt_status s = validate_options(options);
    if (s != KT_OK) return s;
    return create_plan(*options, out);
}

kt_status kt_mlp_run(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                     const void* b_up, const void* b_down, void* Y, void* stream) {
    return run_impl(plan, base_tensors(X, W_up, W_down, b_up, b_down, Y), plan ? plan->H : nullptr, stream);
}

kt_status kt_mlp_run_with_h(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                            const void* b_up, const void* b_down, void* Y, void* H_out, void* stream) {
    if (!H_out) return fail(KT_ERR_INVALID, "H_out is NULL");
    if (plan && plan->choice.h_on_chip)
        return fail(KT_ERR_INVALID, "an H-on-chip plan keeps H on chip: it cannot return H");
    return run_impl(plan, base_tensors(X, W_up, W_down, b_up, b_down, Y), H_out, stream);
}

kt_status kt_mlp_run_ex(kt_mlp_plan_t plan, const kt_mlp_tensors* tensors, void* stream) {
    if (!plan || !tensors) return fail(KT_ERR_INVALID, "plan and tensors must be non-NULL");
    return run_impl(plan, *tensors, tensors->H_out ? tensors->H_out : plan->H, stream);
}

kt_status kt_mlp_run_ex_timed(kt_mlp_plan_t plan, const kt_mlp_tensors* tensors, void* stream, float* ms) {
    if (!plan || !tensors || !ms) return fail(KT_ERR_INVALID, "plan, tensors and ms must be non-NULL");
    return timed_impl(plan, *tensors, stream, ms);
}

kt_status kt_mlp_run_timed(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                           const void* b_up, const void* b_down, void* Y, void* stream,
                           float* ms_up, float* ms_down) {
    float ms[3] = {0.f, 0.f, 0.f};
    kt_status s = timed_impl(plan, base_tensors(X, W_up, W_down, b_up, b_down, Y), stream, ms);
    if (s != KT_OK) return s;
    if (ms_up) *ms_up = ms[1];
    if (ms_down) *ms_down = ms[2];
    return ok();
}

kt_status kt_mlp_run_host(kt_mlp_plan_t plan, const void* X_host, const void* W_up, const void* W_down,
                          const void* b_up, const void* b_down, void* Y_host, void* stream) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    if (!X_host || !Y_host) return fail(KT_ERR_INVALID, "X_host and Y_host must be non-NULL");
    if (plan->residual || plan->layernorm)
        return fail(KT_ERR_INVALID, "kt_mlp_run_host takes plans without residual / layernorm");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    size_t bytes = (size_t)plan->M * (size_t)plan->D * 2;
    // Pinned host buffers mapped into the device's address space are moved by copy
    // kernels (SM loads and stores over the CPU-GPU link, chained to the MLP's kernels by
    // programmatic dependent launch: no copy-engine submission on the path); any other host
    // memory goes through cudaMemcpyAsync.
    const void* x_dev = nullptr;
    void* y_dev = nullptr;
    auto mapped = [](const void* h) -> const void* {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
        return a.devicePointer;
    };
    x_dev = mapped(X_host);
    y_dev = const_cast<void*>(mapped(Y_host));
    const bool by_kernel = x_dev && y_dev && bytes % 16 == 0 && aligned16(x_dev) && aligned16(y_dev);
    const int copy_grid = std::max(1, std::min(plan->num_sms, (int)((bytes / 16 + 1023) / 1024)));
    const char* why = "";
    cudaError_t e = cudaSuccess;
    if (by_kernel) {
        kt_status s = kt::launch_copy16(x_dev, plan->x_stage, bytes, copy_grid, stream, &why);
        if (s != KT_OK) return fail(s, std::string("copy of X to the device: ") + why);
    } else {
        e = cudaMemcpyAsync(plan->x_stage, X_host, bytes, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_fail("copy of X to the device", e);
    }
    kt_status s = run_impl(plan, base_tensors(plan->x_stage, W_up, W_down, b_up, b_down, plan->y_stage), plan->H,
                           stream);
    if (s != KT_OK) return s;
    if (by_kernel) {
        s = kt::launch_copy16(plan->y_stage, y_dev, bytes, copy_grid, stream, &why);
        if (s != KT_OK) return fail(s, std::string("copy of Y to the host: ") + why);
    } else {
        e = cudaMemcpyAsync(Y_host, plan->y_stage, bytes, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_fail("copy of Y to the host", e);
    }
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    return ok();
}

kt_status kt_mlp_status(kt_mlp_plan_t plan) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(plan->last_stream));
    if (e != cudaSuccess) return cuda_fail("stream", e);
    int word = 0;
    e = cudaMemcpy(&word, plan->flags, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("reading the error word", e);
    if (word != kt::DEV_OK) {
        // clear the word and the counters an aborted run may have left behind
        cudaMemset(plan->flags, 0, plan->flag_bytes);
        cudaDeviceSynchronize();
        const char* where = word == kt::DEV_TIMEOUT_PRODUCER ? "producer"
                          : word == kt::DEV_TIMEOUT_MMA ? "MMA issuer"
                          : word == kt::DEV_TIMEOUT_EPILOGUE ? "epilogue"
                          : word == kt::DEV_INJECTED_STALL ? "injected stall" : "unknown";
        return fail(KT_ERR_TIMEOUT, std::string("a bounded device wait ran out (") + where + ")");
    }
    return ok();
}

kt_status kt_mlp_destroy(kt_mlp_plan_t plan) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    free_plan(plan);
    return ok();
}

kt_status kt_mlp_get_info(kt_mlp_plan_t plan, kt_plan_info* out) {
    if (!plan || !out) return fail(KT_ERR_INVALID, "plan and out must be non-NULL");
    std::memset(out, 0, sizeof(*out));
    out->M = plan->M; out->D = plan->D; out->F = plan->F;
    out->act = plan->act; out->dtype = plan->dtype; out->bias = plan->bias;
    out->num_sms = plan->num_sms;
    out->residual = plan->residual; out->layernorm = plan->layernorm; out->weight_layout = plan->w_layout;
    out->ln_eps = plan->ln_eps;
    out->h_on_chip = plan->choice.h_on_chip;
    if (plan->choice.h_on_chip) {
        out->fused_grid = plan->choice.fused.grid;
        out->fused_stages = plan->choice.fused.stages;
        out->fused_smem_bytes = plan->choice.fused.smem_bytes;
        out->fused_est_us = plan->choice.fused.est_us;
    }
    fill_one_launch(plan->choice, out);
    kt::plan_fill_info(plan->choice.up, &out->up);
    kt::plan_fill_info(plan->choice.down, &out->down);
    out->workspace_bytes = plan->workspace_bytes;
    return ok();
}

kt_status kt_mlp_describe(kt_mlp_plan_t plan, char* buf, size_t len) {
    if (!plan || !buf || len == 0) return fail(KT_ERR_INVALID, "plan and buf must be non-NULL, len > 0");
    const kt::GemmConfig& u = plan->choice.up;
    const kt::GemmConfig& d = plan->choice.down;
    std::snprintf(buf, len,
                  "M=%lld D=%lld F=%lld act=%s dtype=%s bias=%d residual=%d layernorm=%d weights=%s sms=%d | up: %dx%d tiles %dx%d (grid %d, %d "
                  "wave%s, %d stages, useful %.3f, model %.2f us) | down: %dx%d tiles %dx%d split_k %d (grid %d, "
                  "%d wave%s, %d stages, %s, useful %.3f, model %.2f us) | workspace %lld B",
                  (long long)plan->M, (long long)plan->D, (long long)plan->F, act_name(plan->act),
                  plan->dtype == KT_BF16 ? "bf16" : "f16", plan->bias, plan->residual, plan->layernorm,
                  plan->w_layout == KT_W_OUT_IN ? "out_in" : "in_out", plan->num_sms, kt::kBM * u.pair, u.BN, u.tiles_m, u.tiles_n,
                  u.grid, u.waves, u.waves == 1 ? "" : "s", u.stages, u.useful_over_padded, u.est_us,
                  kt::kBM * d.pair, d.BN,
                  d.tiles_m, d.tiles_n, d.split_k, d.grid, d.waves, d.waves == 1 ? "" : "s", d.stages,
                  d.split_k == 1 ? "no reduction" : d.cluster_sk ? "cluster reduction" : "global reduction",
                  d.useful_over_padded, d.est_us, (long long)plan->workspace_bytes);
    if (plan->choice.one_launch) {
        const size_t used = std::strlen(buf);
        std::snprintf(buf + used, len - used,
                      " | RUNS both in one launch (grid %d, %d shared stages of %d B, model %.2f us)",
                      plan->choice.one_grid, plan->choice.one_stages, plan->choice.one_slot, plan->choice.one_est_us);
    }
    if (plan->choice.h_on_chip) {
        const kt::FusedConfig& f = plan->choice.fused;
        const size_t used = std::strlen(buf);
        std::snprintf(buf + used, len - used,
                      " | RUNS H on chip: one kernel, 128-row blocks x %d slices of 64 (grid %d, %d stages, model %.2f us)",
                      f.n_slices, f.grid, f.stages, f.est_us);
    }
    return ok();
}

kt_status kt_mlp_debug_trace(kt_mlp_plan_t plan, void* trace_up, void* trace_down) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    if ((trace_up && !aligned16(trace_up)) || (trace_down && !aligned16(trace_down)))
        return fail(KT_ERR_INVALID, "trace buffers must be 16-byte aligned");
    plan->trace_up = static_cast<unsigned long long*>(trace_up);
    plan->trace_down = static_cast<unsigned long long*>(trace_down);
    return ok();
}

kt_status kt_debug_activation(kt_act act_and_form, const float* z, const float* gate, float* out, int64_t n,
                              void* stream) {
    const int form = (int)act_and_form & ~0xff;
    const int act = (int)act_and_form & 0xff;
    if (form != 0 && form != KT_ACTIVATION_SCALAR_FORM) return fail(KT_ERR_INVALID, "unknown activation form");
    if (act < KT_ACT_GELU_ERF || act > KT_ACT_SILU) return fail(KT_ERR_INVALID, "unknown activation");
    if (n < 0 || (n > 0 && (!z || !out || (act == KT_ACT_GEGLU && !gate))))
        return fail(KT_ERR_INVALID, "z and out (and gate for GEGLU) must be non-NULL, n >= 0");
    const char* why = "";
    kt_status s = kt::launch_activation(act, form == 0, z, gate, out, n, stream, &why);
    if (s != KT_OK) return fail(s, why);
    return ok();
}

kt_status kt_down_proj_noalloc(int64_t M, int64_t F, int64_t D, kt_dtype dtype, const void* H,
                               const void* W_down, const void* b_down, void* Y, void* stream) {
    const char* why = "";
    kt_status s = kt::noalloc_down_proj(M, F, D, dtype, H, W_down, b_down, Y, stream, &why);
    if (s != KT_OK) return fail(s, why);
    return ok();
}

kt_status kt_debug_timestamp(void* dst, void* stream) {
    if (!dst || (reinterpret_cast<uintptr_t>(dst) & 7u)) return fail(KT_ERR_INVALID, "dst must be an aligned device uint64");
    const char* why = "";
    kt_status s = kt::launch_timestamp(dst, stream, &why);
    if (s != KT_OK) return fail(s, why);
    return ok();
}

kt_status kt_mlp_debug_stall(kt_mlp_plan_t plan, int enable, int64_t limit_us) {
    if (!plan) return fail(KT_ERR_INVALID, "plan is NULL");
    if (enable && (limit_us < 1 || limit_us > 10000000))
        return fail(KT_ERR_INVALID, "limit_us must be in [1, 10 000 000]");
    plan->inject_stall = enable ? 1 : 0;
    plan->stall_limit_us = enable ? limit_us : 0;
    return ok();
}

}  // extern "C"
