/*
 * kt_mlp.h -- C ABI of the fused transformer MLP library for one GB300 (sm_103a).
 *
 *   Y = act(X . W_up [+ b_up]) . W_down [+ b_down]
 *
 * The operation is the transformer feed-forward block in the two forms the pages
 * work on:
 *   - the plain GELU MLP: up projection, GELU, down projection -- the F16 SigLIP
 *     MLP [1,729,1152] -> [1,729,4304] -> [1,729,1152] without biases
 *     ("MLP layout sweep and remaining representation limits", opening paragraph;
 *     its "ISA review" section computes GELU through tanh);
 *   - SDXL's GEGLU FeedForward: one projection to 2F, split along the last axis
 *     into value (first half) and gate (SECOND half), value * gelu_erf(gate),
 *     then the projection back ("SDXL as a requirements inventory",
 *     section 1.3 FeedForward; section 9.3 for the erf form and the half order).
 *
 * Options of the transformer block around the feed-forward (kt_mlp_plan_ex /
 * kt_mlp_run_ex), from "SDXL as a requirements inventory": a LayerNorm of X before
 * the up projection and the residual add after the down projection (section 1.3,
 * BasicTransformerBlock: x = ff(LayerNorm(x)) + x; section 3, rows 3 and 9-10); the
 * sigmoid GELU x * sigmoid(1.702 x) (section 9.3) and SiLU (section 1.3, timestep
 * embedding; section 3 row 4) as further activations; weights in PyTorch's
 * nn.Linear order [out][in] (section 1.4; section 3 row 1).
 *
 * Numerics: operands in the 16-bit I/O dtype, products accumulated in fp32 in
 * tensor memory, bias added to the fp32 accumulator, the activation evaluated
 * in fp32, and exactly ONE rounding (to nearest even) of H to the I/O dtype
 * before the down projection reads it ("The software stack", section 2.3: the
 * accumulator is a resident format, never a memory word).  Y is rounded once.
 *
 * Layouts (all row-major, contiguous, 16-byte aligned device pointers, dtype dt):
 *   X[M][D], W_up[D][F_up], W_down[F][D], b_up[F_up], b_down[D], Y[M][D],
 *   H[M][F];  F_up = F for GELU, 2F for GEGLU.  Weights are [in][out]; a PyTorch
 *   nn.Linear weight ([out][in]) is passed as weight.t().contiguous().
 *
 * Requirements: M >= 1; D >= 8 and F >= 8, both multiples of 8 (16-byte row
 * pitch for the tensor-memory-accelerator copies).  Anything else returns
 * KT_ERR_UNSUPPORTED or KT_ERR_INVALID and launches nothing.
 *
 * Errors: every call returns a kt_status; kt_last_error() gives a message for
 * the calling thread's last non-OK status.  Device-side waits are bounded: a
 * wait that runs out sets the plan's error word, the kernel returns, and
 * kt_mlp_status() reports KT_ERR_TIMEOUT.  There is no CPU fallback: without a
 * usable sm_103a device kt_mlp_plan() fails.
 */
#ifndef KT_MLP_H
#define KT_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KT_MLP_ABI_VERSION 3

typedef enum {
    KT_ACT_GELU_ERF = 0,  /* gelu(z) = z * Phi(z) = 0.5 z (1 + erf(z / sqrt 2))                 */
    KT_ACT_GELU_TANH = 1, /* 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))                   */
    KT_ACT_GEGLU = 2,     /* P[:, :F] * gelu_erf(P[:, F:]), F_up = 2F                          */
    KT_ACT_NONE = 3,      /* no activation (two chained linear layers); checks the GEMMs alone */
    KT_ACT_GELU_SIGMOID = 4, /* z * sigmoid(1.702 z): the sigmoid approximation of GELU        */
    KT_ACT_SILU = 5       /* z * sigmoid(z) (SiLU / swish)                                      */
} kt_act;

/*
 * Where the intermediate H lives.  KT_H_MEMORY: two kernels, H written once (to L2 /
 * HBM) by the up projection and read by the down projection.  KT_H_ON_CHIP: one kernel
 * that keeps H in shared memory, one 64-column slice at a time, and accumulates Y in
 * tensor memory; it applies only where Y[128 x D] fits tensor memory beside the slices
 * (D <= 256, D <= 192 for GEGLU) and to [in][out] weights.  KT_H_AUTO: the planner's
 * choice between the two.  kt_mlp_plan uses KT_H_MEMORY.
 */
typedef enum { KT_H_AUTO = 0, KT_H_MEMORY = 1, KT_H_ON_CHIP = 2 } kt_h_path;

/* How the two projections are launched when H goes through memory.  KT_LAUNCH_TWO: two
 * persistent kernels, the down projection's CTAs starting as the up projection's finish
 * (programmatic dependent launch) and loading rows of H as they are stored; a down
 * projection split along K reduces inside clusters or through global memory.
 * KT_LAUNCH_ONE: one persistent kernel that takes up tiles, then down items, from one work
 * queue (a down item once its rows of H are stored); down items may be K splits of a tile,
 * reduce-scattered among the splits through global memory (GEGLU: summed by the last split
 * to arrive).  KT_LAUNCH_AUTO is the planner's choice: one launch wherever a one-launch
 * plan exists (measured faster on every benchmark shape), else two. */
typedef enum { KT_LAUNCH_AUTO = 0, KT_LAUNCH_ONE = 1, KT_LAUNCH_TWO = 2 } kt_launches;

/* Memory order of W_up and W_down. */
typedef enum {
    KT_W_IN_OUT = 0, /* W_up[D][F_up], W_down[F][D]: the layer computes X . W               */
    KT_W_OUT_IN = 1  /* W_up[F_up][D], W_down[D][F]: PyTorch nn.Linear order, X . W^T; GEGLU's
                        value rows are W_up[0:F], its gate rows W_up[F:2F]                   */
} kt_weight_layout;

typedef enum { KT_F16 = 0, KT_BF16 = 1 } kt_dtype;

typedef enum {
    KT_OK = 0,
    KT_ERR_INVALID = 1,     /* bad argument: null pointer, negative size, unknown enum  */
    KT_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels support          */
    KT_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed (message says which)  */
    KT_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (see kt_mlp_status)    */
    KT_ERR_NOMEM = 5        /* device or host allocation failed                          */
} kt_status;

typedef struct kt_mlp_plan_s* kt_mlp_plan_t;

/* What the planner chose for one of the two GEMMs (host-side description). */
typedef struct {
    int32_t BM, BN, BK;        /* CTA tile: BM x BN output, BK-deep k-blocks              */
    int32_t stages;            /* shared-memory pipeline depth                            */
    int32_t split_k;           /* SK: CTAs sharing one output tile along K                */
    int32_t tiles_m, tiles_n;  /* output tiles: ceil(M/BM) x ceil(N/BN)                   */
    int32_t kblocks;           /* ceil(K/BK)                                              */
    int32_t grid;              /* persistent CTAs launched (<= SM count)                  */
    int32_t waves;             /* ceil(tiles_m * tiles_n * split_k / SMs)                 */
    int32_t smem_bytes;        /* dynamic shared memory per CTA                           */
    int32_t tmem_cols;         /* tensor-memory columns allocated per CTA                 */
    int32_t cluster_sk;        /* 1: the split_k CTAs of a tile form a thread-block cluster and
                                  reduce through distributed shared memory; 0: through global
                                  memory (or no split)                                     */
    int32_t b_kmajor;          /* 1: the weight operand is [N][K] (PyTorch order), K-major  */
    int64_t M, N, K;           /* the GEMM: [M,K] x [K,N]                                 */
    double useful_over_padded; /* M*N*K / (padded M * padded N * padded K)                */
    double est_us;             /* the planner's modelled time (a model, not a measurement) */
} kt_gemm_plan_info;

typedef struct {
    int64_t M, D, F;
    int32_t act, dtype, bias;
    int32_t num_sms;
    kt_gemm_plan_info up;      /* X[M,D] . W_up[D,F_up] with the fused epilogue -> H[M,F] */
    kt_gemm_plan_info down;    /* H[M,F] . W_down[F,D] (+ b_down) -> Y[M,D]               */
    int64_t workspace_bytes;   /* device bytes the plan owns (H, split-K partials, flags) */
    int32_t residual, layernorm, weight_layout;  /* the kt_mlp_options of the plan (0 for kt_mlp_plan) */
    float ln_eps;
    int32_t h_on_chip;         /* 1: the fused H-on-chip kernel runs (up / down describe the
                                  two-kernel alternative); its tile facts follow           */
    int32_t fused_grid, fused_stages, fused_smem_bytes;
    double fused_est_us;
    int32_t one_launch;        /* 1: both projections run in ONE persistent launch: up and down
                                  tiles taken from one work queue (up tiles first), a down tile
                                  as soon as its rows of H are stored; up / down describe the
                                  two GEMMs in it, sharing one shared-memory ring            */
    int32_t one_launch_grid, one_launch_stages, one_launch_smem_bytes;
    double one_launch_est_us;
} kt_plan_info;

/*
 * Problem description for kt_mlp_plan_ex.  Zero-initialise it and set the fields;
 * with residual = layernorm = 0 and weight_layout = KT_W_IN_OUT it describes the same
 * problem as kt_mlp_plan(M, D, F, act, dtype, bias).
 */
typedef struct {
    int64_t M, D, F;        /* rows (tokens), model dim, hidden dim                          */
    int32_t act;            /* kt_act                                                        */
    int32_t dtype;          /* kt_dtype: the I/O dtype of every tensor                       */
    int32_t bias;           /* 1: b_up[F_up] and b_down[D]                                   */
    int32_t residual;       /* 1: Y = R + FF(.), R[M][D] added to the fp32 result before the
                               one rounding of Y                                             */
    int32_t layernorm;      /* 1: the up projection reads LayerNorm(X) instead of X:
                               (x - mean) / sqrt(var + ln_eps) * gamma + beta per row, mean
                               and biased variance over D in fp32, rounded once to dtype     */
    int32_t weight_layout;  /* kt_weight_layout                                              */
    float ln_eps;           /* LayerNorm epsilon (> 0; PyTorch's default is 1e-5)            */
    int32_t h_path;         /* kt_h_path: where H lives between the two projections          */
    int32_t launches;       /* kt_launches: one or two kernel launches (H through memory)    */
} kt_mlp_options;

/*
 * Device tensors of one kt_mlp_run_ex call (row-major, contiguous, 16-byte aligned,
 * the plan's dtype).  Pointers the plan does not use must be NULL.
 */
typedef struct {
    const void* X;          /* [M][D]                                                        */
    const void* W_up;       /* [D][F_up] (KT_W_IN_OUT) or [F_up][D] (KT_W_OUT_IN)            */
    const void* W_down;     /* [F][D]    (KT_W_IN_OUT) or [D][F]    (KT_W_OUT_IN)            */
    const void* b_up;       /* [F_up], iff bias                                              */
    const void* b_down;     /* [D], iff bias                                                 */
    const void* R;          /* [M][D], iff residual; may be X itself, and may equal Y
                               (in-place update of a residual stream)                        */
    const void* ln_gamma;   /* [D], iff layernorm                                            */
    const void* ln_beta;    /* [D], iff layernorm                                            */
    void* Y;                /* [M][D]; may equal X and / or R, must not partially overlap them */
    void* H_out;            /* [M][F] to receive the rounded intermediate, or NULL (the plan's
                               workspace is used); must be NULL for an H-on-chip plan        */
} kt_mlp_tensors;

/*
 * kt_mlp_plan -- validate the problem, choose tiles / pipeline depth / split-K
 * with the padding-aware planner, and allocate the plan's device workspace on the
 * CURRENT device (H[M][F], fp32 split-K partials, tile counters, error word).
 *   M, D, F  : rows (tokens), model dim, hidden dim.
 *   act      : kt_act.     dtype: kt_dtype.     bias: 0 = no biases, 1 = b_up and b_down.
 *   out      : receives the plan handle (owned by the caller; free with kt_mlp_destroy).
 * Errors: INVALID (null out, non-positive size, bad enum), UNSUPPORTED (D or F not a
 * multiple of 8, device not sm_103, sizes past the 32-bit tile index range),
 * CUDA / NOMEM (device query or allocation failed).  On error *out is NULL.
 */
kt_status kt_mlp_plan(int64_t M, int64_t D, int64_t F, kt_act act, kt_dtype dtype, int bias,
                      kt_mlp_plan_t* out);

/*
 * kt_mlp_run -- enqueue the MLP on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  The plan's launch schedule (kt_plan_info.one_launch): either one persistent
 * kernel running both projections, or two -- the up GEMM with the fused
 * bias/activation/rounding epilogue writing H into the plan's workspace, then the down GEMM
 * (programmatic dependent launch) writing Y.  All pointers are device pointers owned by the
 * caller, 16-byte aligned, laid out as described at the top of this file.  b_up /
 * b_down must be non-NULL iff the plan has bias = 1.  Asynchronous: returns after
 * enqueueing.  A plan must not run concurrently on two streams (one workspace).
 * Every launch parameter is the same from call to call, so the call may be captured
 * into a CUDA graph (stream capture) and replayed; replays read and write the
 * captured pointers.  The same holds for kt_mlp_run_ex.
 * Errors: INVALID (null / misaligned pointer, bias mismatch), CUDA (launch failed).
 */
kt_status kt_mlp_run(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                     const void* b_up, const void* b_down, void* Y, void* stream);

/*
 * kt_mlp_plan_ex -- kt_mlp_plan for a problem with the options of kt_mlp_options: a
 * LayerNorm prologue, a residual add, the sigmoid GELU / SiLU activations, the
 * [out][in] weight order and the H path.  A layernorm plan also owns a workspace
 * Xn[M][D] for the normalised X.  Errors as kt_mlp_plan, plus INVALID for a flag
 * outside {0, 1}, an unknown weight layout or H path, or ln_eps <= 0 (or not finite)
 * with layernorm = 1; UNSUPPORTED for KT_H_ON_CHIP where it does not apply.
 */
kt_status kt_mlp_plan_ex(const kt_mlp_options* options, kt_mlp_plan_t* out);

/* kt_mlp_plan_info_ex -- kt_mlp_plan_info for a kt_mlp_options problem (host only). */
kt_status kt_mlp_plan_info_ex(const kt_mlp_options* options, int num_sms, kt_plan_info* out);

/*
 * kt_mlp_run_ex -- enqueue the block on `stream`: with layernorm, a LayerNorm kernel
 * writes Xn (one warp per row); the up GEMM (fused epilogue, programmatic dependent
 * launch) writes H; the down GEMM adds b_down and R to the fp32 result, rounds once
 * and writes Y.  Any plan may be run with it (a kt_mlp_plan plan takes the tensors
 * of kt_mlp_run).  Asynchronous.  Errors: INVALID (null tensors, a pointer present or
 * absent against the plan's options, misaligned pointer), CUDA (launch failed).
 */
kt_status kt_mlp_run_ex(kt_mlp_plan_t plan, const kt_mlp_tensors* tensors, void* stream);

/*
 * kt_mlp_run_ex_timed -- kt_mlp_run_ex with CUDA events around each kernel, no
 * programmatic overlap between them; waits and writes the device times in ms to
 * ms[0] (LayerNorm, 0 without it), ms[1] (up GEMM) and ms[2] (down GEMM).
 */
kt_status kt_mlp_run_ex_timed(kt_mlp_plan_t plan, const kt_mlp_tensors* tensors, void* stream, float* ms);

/*
 * kt_mlp_run_with_h -- as kt_mlp_run, but the rounded intermediate H[M][F] is
 * written to the caller's device buffer H_out (16-byte aligned) instead of the
 * plan's workspace, so that it can be inspected.  Same kernels, same results.
 * INVALID for an H-on-chip plan (it never writes H).
 */
kt_status kt_mlp_run_with_h(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                            const void* b_up, const void* b_down, void* Y, void* H_out, void* stream);

/*
 * kt_mlp_run_host -- end-to-end call with HOST activations: copies X_host[M][D] to
 * the device (plan-owned staging), runs the MLP, copies Y back into Y_host[M][D]
 * and synchronises `stream`.  Weights and biases stay device pointers (resident
 * model parameters).  Pinned host memory (mapped into the device's address space) is
 * moved by two copy kernels chained to the MLP by programmatic dependent launch;
 * any other host memory by cudaMemcpyAsync, which works but is slower.  Returns after
 * Y_host is filled.
 */
kt_status kt_mlp_run_host(kt_mlp_plan_t plan, const void* X_host, const void* W_up,
                          const void* W_down, const void* b_up, const void* b_down,
                          void* Y_host, void* stream);

/*
 * kt_mlp_run_timed -- as kt_mlp_run, with CUDA events recorded on `stream` before,
 * between and after the two kernels; waits for the last event and writes each
 * kernel's device time in milliseconds to *ms_up / *ms_down (either may be NULL).
 * The down kernel is launched without the programmatic dependency here, so the two
 * kernels do not overlap and each time is that kernel's alone.  For measurement.
 */
kt_status kt_mlp_run_timed(kt_mlp_plan_t plan, const void* X, const void* W_up, const void* W_down,
                           const void* b_up, const void* b_down, void* Y, void* stream,
                           float* ms_up, float* ms_down);

/*
 * kt_mlp_status -- synchronise the plan's last stream and read its device error
 * word.  KT_OK, or KT_ERR_TIMEOUT when a bounded wait ran out in an earlier run
 * (the word is then cleared), or KT_ERR_CUDA if the stream reported an error.
 */
kt_status kt_mlp_status(kt_mlp_plan_t plan);

/* kt_mlp_destroy -- free the plan's workspace (after synchronising its device). */
kt_status kt_mlp_destroy(kt_mlp_plan_t plan);

/* kt_mlp_describe -- write a one-line text description of the plan into buf. */
kt_status kt_mlp_describe(kt_mlp_plan_t plan, char* buf, size_t len);

/* kt_mlp_get_info -- copy the plan's chosen configuration into *out. */
kt_status kt_mlp_get_info(kt_mlp_plan_t plan, kt_plan_info* out);

/*
 * kt_mlp_plan_info -- run the planner alone, on the host, for a device with
 * `num_sms` SMs.  Touches no GPU; used to inspect and test tile choices.
 * Same validation and errors as kt_mlp_plan (except CUDA / NOMEM).
 */
kt_status kt_mlp_plan_info(int64_t M, int64_t D, int64_t F, kt_act act, kt_dtype dtype, int bias,
                           int num_sms, kt_plan_info* out);

/*
 * kt_mlp_debug_stall -- failure-injection hook for tests.  With enable = 1 the next
 * runs of this plan make the up kernel's producer wait on a barrier nobody
 * signals, bounded by `limit_us` microseconds; the wait runs out, the kernel
 * records KT_ERR_TIMEOUT in the plan's error word and returns without computing.
 * enable = 0 restores normal runs.  No GPU fault is involved.
 */
kt_status kt_mlp_debug_stall(kt_mlp_plan_t plan, int enable, int64_t limit_us);

/*
 * kt_mlp_debug_trace -- timeline tracing for tests and profiling.  With non-NULL
 * device buffers, the next runs of this plan write, per CTA of the up / down kernel,
 * 32 uint64 slots: %globaltimer (ns) at CTA entry, set-up done, first copy issued,
 * first stage landed, first tile's main loop done, epilogue start / done, exit;
 * then the SM id, the number of tiles, the last tile's main-loop / epilogue end,
 * four epilogue sub-phase marks of the first epilogue warp, and ten marks of the
 * CTA's second tile (epilogue sub-phases, its main loop's start and end, its first
 * copy); with both projections in one launch (trace_up then holds the one kernel's
 * CTAs), slots 26-30: first down item taken, its rows of H stored, up and down items
 * processed (counts), last up tile's main loop done; slot 31: past the wait for the
 * previous kernel in the stream.  Each buffer must hold 32 * grid uint64 (grid from
 * kt_mlp_get_info); the caller owns them.  NULL buffers switch tracing off.
 */
kt_status kt_mlp_debug_trace(kt_mlp_plan_t plan, void* trace_up, void* trace_down);

/*
 * kt_debug_activation -- evaluate the epilogue's fp32 activation elementwise on
 * device arrays: out[i] = gelu_erf(z[i]) / gelu_tanh(z[i]) / z[i] * gelu_erf(gate[i])
 * (GEGLU) / z[i] (none) / gelu_sigmoid(z[i]) / silu(z[i]), for i < n, enqueued on
 * `stream`.  The same device
 * functions as the fused epilogue; exposed so that their accuracy can be tested
 * against the oracle on their own.  gate is read only for GEGLU.  The epilogues
 * evaluate the activations on pairs of values with the paired fp32 instructions
 * (add / mul / fma .rn.f32x2); `act` alone selects that form, `act |
 * KT_ACTIVATION_SCALAR_FORM` the same steps as two scalar instructions each, which
 * must give the same bits.  Any other flag: KT_ERR_INVALID.
 */
#define KT_ACTIVATION_SCALAR_FORM 0x100
kt_status kt_debug_activation(kt_act act, const float* z, const float* gate, float* out, int64_t n,
                              void* stream);

/*
 * kt_debug_timestamp -- enqueue a one-thread kernel on `stream` that writes
 * %globaltimer (ns) to the device uint64 at dst.  Brackets launches in traces.
 */
kt_status kt_debug_timestamp(void* dst, void* stream);

/*
 * kt_down_proj_noalloc -- the down projection on its own, Y[M][D] = round(H[M][F] .
 * W_down[F][D] (+ b_down[D])), fp32 accumulation, that allocates no device memory.
 * The pages have no counterpart to this entry point; it exists for callers of the
 * library that cannot allocate: for example a host framework's plugin hook that is
 * handed only input / output pointers and a stream and must not allocate there, or
 * a latency-critical serving loop that must never call cudaMalloc / cudaFree
 * (cudaFree synchronises the whole device, cudaMalloc can block).
 *   H, W_down, Y : device pointers (16-byte aligned, row-major, dtype); the caller
 *                  owns them.  b_down: device pointer or NULL (no bias).
 * It runs the same kernel as the two-launch down projection of kt_mlp_run, with the
 * tile plan the planner chooses without the cluster split-K reduction (its split-K
 * partials go through global memory; for SigLIP's 729 x 4304 -> 1152 that plan can
 * differ from kt_mlp_run's, which reduces inside clusters).  Instead of a plan's
 * workspace, its split-K partials, tile counters and
 * error word live in one static device array of 16 MiB that the library holds on
 * every GPU that loads it, until the process exits.  A problem whose plan needs
 * more scratch than that is rejected with KT_ERR_UNSUPPORTED and a message giving
 * both sizes; nothing is launched.  Each call clears the counters and error word
 * (cudaMemsetAsync on `stream`) before its kernel; otherwise the array keeps the
 * last call's contents.  All calls on a device share the array, so calls that
 * overlap on the GPU (on two streams, or from two host threads) race and give wrong
 * results.  The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and the SM count; make that first
 * call before any stream capture.  There is no status word to read afterwards: a
 * device-side wait that runs out (never in normal operation) leaves Y incomplete.
 * Errors: INVALID (NULL / misaligned pointer, bad size or dtype), UNSUPPORTED (not
 * sm_103, D or F not a multiple of 8, scratch too small), CUDA (a runtime call or
 * the launch failed).
 */
kt_status kt_down_proj_noalloc(int64_t M, int64_t F, int64_t D, kt_dtype dtype, const void* H,
                               const void* W_down, const void* b_down, void* Y, void* stream);

/* Thread-local message for the calling thread's last non-OK status ("" if none). */
const char* kt_last_error(void);

/* KT_MLP_ABI_VERSION of the loaded library. */
int kt_mlp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KT_MLP_H */
