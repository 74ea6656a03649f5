// kt_internal.h -- shared between the host ABI layer, the planner and the kernels.
// Not part of the public interface (that is include/kt_mlp.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "kt_mlp.h"

#ifdef __CUDACC__
#define KT_HOST_DEVICE __host__ __device__
#else
#define KT_HOST_DEVICE
#endif

namespace kt {

// Fixed tile geometry of the sm_103a kernels.
constexpr int kBM = 128;          // tcgen05 M (one CTA, cta_group::1): TMEM lane i = tile row i
constexpr int kAtomK = 64;        // 64 16-bit elements = one 128-byte swizzle row (the A box width)
constexpr int kEpiWarps = 8;      // epilogue warps (two per TMEM lane quadrant)
constexpr int kThreads = (2 + kEpiWarps) * 32;  // producer warp + MMA warp + epilogue
constexpr int kTmemCols = 512;    // whole tensor memory of the SM (one CTA per SM)
constexpr int kAccSlot = 256;     // TMEM columns reserved per accumulator buffer
constexpr int kSmemBudget = 227 * 1024;  // opt-in dynamic shared memory per CTA
// barriers, TMEM slot and flags (1 KB), 1024-byte alignment slack (1 KB), and a 16 KB
// guard band past the ring so that no descriptor stride can reach beyond the allocation
constexpr int kStoreCols = 32;    // columns per epilogue TMA store box (32 rows x 32 columns)
constexpr int kStagingBytes = kEpiWarps * 32 * kStoreCols * 2;  // one 2 KB buffer per epilogue warp
// output staging, barriers / TMEM slot / flags, the epilogue's two bias slices (2 KB)
// and 1024-byte alignment slack (1 KB)
constexpr int kBarrierBytes = 512;
constexpr int kBiasSmemBytes = 2048;
constexpr int kSmemReserve = kStagingBytes + kBarrierBytes + kBiasSmemBytes + 1024;

// Epilogue warps per kernel kind: 8 for every kind (two per TMEM lane quadrant).  GEGLU's
// 128-column tiles split into 4 column groups evenly over 8 warps; 12 warps measured no
// faster and cost a third more output staging.
constexpr int epi_warps(int epi) { return epi == 2 /* EPI_GEGLU */ ? 8 : kEpiWarps; }
constexpr int smem_reserve(int epi) {
    return epi_warps(epi) * 32 * kStoreCols * 2 + kBarrierBytes + kBiasSmemBytes + 1024;
}
constexpr int kMaxStages = 8;
constexpr int kItemRing = 4;  // work items published ahead when both projections run in one launch
constexpr int kRsMaxSplit = 4;  // largest split along K of the one-launch down projection (reduce-scatter)

// Epilogue kinds (one kernel instantiation each, times two dtypes).
enum Epi : int {
    EPI_GELU_ERF = 0,   // H = round(gelu_erf(acc + b))
    EPI_GELU_TANH = 1,  // H = round(gelu_tanh(acc + b))
    EPI_GEGLU = 2,      // H = round((acc_v + b_v) * gelu_erf(acc_g + b_g))
    EPI_NONE = 3,       // H = round(acc + b)
    EPI_DOWN = 4,       // Y = round(sum_s partial_s + b [+ R])   (split-K when SK > 1)
    EPI_GELU_SIGMOID = 5,  // H = round(z * sigmoid(1.702 z)),  z = acc + b
    EPI_SILU = 6           // H = round(z * sigmoid(z))
};

// Device error word values (first writer wins).
enum DevError : int { DEV_OK = 0, DEV_TIMEOUT_PRODUCER = 1, DEV_TIMEOUT_MMA = 2,
                      DEV_TIMEOUT_EPILOGUE = 3, DEV_INJECTED_STALL = 4 };

// One GEMM's launch configuration, chosen by the planner.
struct GemmConfig {
    int64_t M, N, K;       // output rows, output columns, reduction length
    int BN;                // N tile (H columns for GEGLU, whose MMA N is 2 BN), multiple of 32, 32..256
    int stages;
    int split_k;
    int tiles_m, tiles_n, kblocks, kblocks_per_split;
    int grid;
    int waves;
    int smem_bytes;
    int n_b;               // B operand tiles per stage: 1, or 2 for GEGLU (value + gate)
    int pair;              // 1: one CTA per 128-row tile; 2: a CTA pair per 256-row tile (cta_group::2)
    int bk;                // k-block depth per pipeline stage: 64 or 128
    int cluster_sk;        // 1: split-K partials reduce-scattered through L2 inside a cluster
    int b_kmajor;          // 1: the weight is stored [N][K] (PyTorch order) and loaded K-major
    int dbl_staging;       // 1: shared memory left over for a second set of output staging buffers
    double useful_over_padded;
    double est_us;
    double t_tile_us;      // model: one tile's main loop on one CTA (pair), and its epilogue
    double t_epi_us;
    double t_x_us;         // model: the split-K exchange of one tile (0 without split-K)
};

// The H-on-chip variant (kt_fused.cu): both projections in one kernel, H in shared
// memory one 64-column slice at a time; applies for D <= 256 with [in][out] weights.
constexpr int kFusedSlice = 64;
struct FusedConfig {
    int Dk;                // D rounded up to 64: K of the up GEMM, N of the down GEMM
    int n_b;               // up-projection B boxes per slice (2 for GEGLU)
    int n_slices;          // ceil(F / 64)
    int tiles_m;           // ceil(M / 128)
    int grid, waves, stages, smem_bytes;
    uint32_t x_bytes, stage_bytes, wup_bytes, wdn_bytes;
    double est_us;
};

struct PlanChoice {
    GemmConfig up, down;
    int h_on_chip;         // 1: run the fused kernel (`fused`) instead of up + down
    FusedConfig fused;
    // 1: both projections in one persistent launch (kt_gemm_kernel<..., TWO = true>): up and
    // down tiles from one dynamic work queue, down tiles as soon as their rows of H are
    // stored; one shared-memory ring of `one_stages` stages of `one_slot` bytes
    int one_launch;
    int one_grid, one_stages, one_slot, one_smem, one_dbl;
    double one_est_us;
    GemmConfig one_up, one_down;  // the two GEMMs' configurations in that launch
};

// Columns of one box of an N-major ([K][N]) B tile: 64 (128-byte rows, 128-byte swizzle)
// when the CTA's column share (BN, or BN/2 in a CTA pair; a multiple of 16) is a multiple
// of 64, else 32 (64-byte rows, 64-byte swizzle) when it is a multiple of 32, else 16
// (32-byte rows, 32-byte swizzle), so that no column is loaded in vain.  The box's row
// bytes are also its swizzle span.
KT_HOST_DEVICE inline int b_box_cols(int BN, int pair) {
    const int share = BN / pair;
    return share % 64 == 0 ? 64 : share % 32 == 0 ? 32 : 16;
}

// Bytes of one pipeline stage in one CTA: its 128-row A tile (bk/64 swizzle atoms of
// 128 x 64) + n_b B tiles holding its share of the columns: in b_box_cols-wide boxes of
// bk rows for a [K][N] weight (N-major), or in bk/64 atoms of (share) rows x 64 for a
// [N][K] weight (K-major).
inline int b_tile_bytes(int BN, int pair, int bk, int b_kmajor) {
    (void)b_kmajor;
    return (BN / pair) * bk * 2;
}
inline int stage_bytes(int BN, int n_b, int pair, int bk, int b_kmajor = 0) {
    return kBM * bk * 2 + n_b * b_tile_bytes(BN, pair, bk, b_kmajor);
}

// Planner (host only, no GPU): returns KT_OK and fills `out`, or an error status.
// w_layout: KT_W_IN_OUT ([in][out] weights, N-major B) or KT_W_OUT_IN ([out][in], K-major B).
// h_path: KT_H_AUTO (the fused H-on-chip kernel where it applies and the model prefers
// it), KT_H_MEMORY (always two kernels) or KT_H_ON_CHIP (the fused kernel, or
// KT_ERR_UNSUPPORTED where it does not apply).
kt_status plan_choose(int64_t M, int64_t D, int64_t F, int act, int num_sms, PlanChoice* out,
                      const char** why, bool allow_cluster_sk = true, int w_layout = KT_W_IN_OUT,
                      int h_path = KT_H_MEMORY, bool allow_one_launch = true, int launches = KT_LAUNCH_AUTO);

// The up projection's epilogue kind for a kt_act.
int up_epilogue(int act);

// Fill the public description from a choice.
void plan_fill_info(const GemmConfig& g, kt_gemm_plan_info* out);

// Launch parameters shared by host and device.
struct GemmParams {
    int M, N, K;
    int BN, stages, split_k;
    int pair;                // 1 or 2 (CTA pair, tiles of 256 rows); tiles_m counts pair-tiles
    int bk;                  // k-block depth per stage (64 or 128)
    int cluster_sk;          // 1: the split_k CTAs of a tile form a cluster and reduce on chip
    int rs_sk;               // 1 (both projections in one launch): the split_k CTAs of a tile
                             // reduce-scatter their fp32 partials through global memory, each
                             // summing the 32 x 32 units it owns; splits of a tile are adjacent
                             // work items (all of them run at once: no item waits on a later one)
    int tiles_m, tiles_n, kblocks, kblocks_per_split, num_tiles;
    int gate_col;            // GEGLU: first gate column (row, K-major) of W_up (= F); else 0
    int b_kmajor;            // 1: B is [N][K] in memory, loaded in 64-deep K-major atoms
    uint32_t b_atom_bytes;   // K-major B: bytes of one 64-deep atom of this CTA's column share
    uint32_t idesc;          // tcgen05 instruction descriptor
    uint32_t stage_bytes, a_bytes, b_bytes;  // per stage / A tile / one B operand tile
    uint32_t acc_bufs;       // accumulator buffers in TMEM (1 or 2)
    uint32_t geglu_share;    // GEGLU: H columns per CTA share (BN / pair); the accumulator holds,
                             // per share, its value columns then its gate columns
    const void* bias;        // b_up (GEGLU: value then gate halves) / b_down / null
    const void* residual;    // down projection: R[M][N] added before the rounding, or null
    float* partials;         // split-K: [split_k][tiles_m*BM][tiles_n*BN] fp32 (rs_sk: [half tile][unit]
                             // [sending split][8][32 rows][4])
    int* counters;           // split-K: per 128-row half tile, arrival counters (zero between runs);
                             // rs_sk: one 64-bit arrival counter per half tile (8-byte aligned),
                             // growing by split_k per run
    int* error;              // device error word
    int inject_stall;        // failure-injection hook (producer waits on a silent barrier)
    unsigned long long wait_limit_ns;   // bound of every device-side wait
    unsigned long long stall_limit_ns;  // bound of the injected wait
    int pdl_wait;            // 1: griddepcontrol.wait before the first global access (see ready)
    int dbl_staging;         // 1: two output staging buffers per epilogue warp
    unsigned* ready;         // up: per row-block counters of stored tiles (incremented per CTA tile);
                             // down: the same counters, waited on before loading rows of H; or null
    unsigned* ready_readers; // down: per row block, how many of this run's waits on it are done
    const unsigned* ready_expect;  // down: per row block, how many waits this run makes on it
    unsigned ready_target;   // down: counter value meaning "every tile of this row block stored"
    int ready_rows;          // down: rows per up-projection row block (128 x its CTA pairing)
    unsigned long long* trace;  // optional per-CTA timeline (kTraceSlots u64 per CTA) or null
    int* sched;              // both projections in one launch: [0] next work item, [1] units done
                             // (zero between runs; the last unit to finish resets both)
};

// Per-CTA trace slots (globaltimer ns unless noted), written when GemmParams::trace is set.
enum TraceSlot : int {
    TR_ENTRY = 0,        // first instruction of the CTA
    TR_SETUP = 1,        // barriers initialised, TMEM allocated
    TR_FIRST_TMA = 2,    // producer issued its first copy
    TR_FIRST_FULL = 3,   // MMA issuer saw the first stage land
    TR_MAIN_DONE = 4,    // MMA issuer committed the last k-block of its first tile
    TR_EPI_START = 5,    // epilogue saw the first accumulator ready
    TR_EPI_DONE = 6,     // epilogue finished its first tile
    TR_EXIT = 7,         // after the teardown barrier
    TR_SMID = 8,         // %smid
    TR_TILES = 9,        // tiles this CTA processed
    TR_LAST_MAIN = 10,   // MMA issuer committed its last tile
    TR_LAST_EPI = 11,    // epilogue finished its last tile
    TR_EPI_LD = 12,      // first epilogue warp: first accumulator group in registers
    TR_EPI_MATH = 13,    //   ... its bias / activation done
    TR_EPI_STORE = 14,   //   ... its first store issued
    TR_EPI_DRAIN = 15,   //   ... all its stores complete
    // steady state: the CTA's second tile
    TR_S_ACC = 16,       // first epilogue warp: accumulator ready
    TR_S_SIG = 17,       //   ... the previous tile's rows counted (up projection)
    TR_S_G0M = 18,       //   ... its first column group computed
    TR_S_G0S = 19,       //   ... its first column group's store issued
    TR_S_G1M = 20,       //   ... its second column group computed
    TR_S_G1S = 21,       //   ... its second column group's store issued
    TR_S_ARR = 22,       //   ... accumulator released
    TR_S_MMA0 = 23,      // MMA issuer: the tile's accumulator free, main loop starts
    TR_S_MMA1 = 24,      // MMA issuer: the tile's last k-block committed
    TR_S_LD0 = 25,       // producer: the tile's first copy issued
    // both projections in one launch
    TR_T_DN_TAKEN = 26,  // producer: first down-projection tile taken
    TR_T_DN_READY = 27,  // producer: its rows of H stored (readiness wait done)
    TR_T_UP_ITEMS = 28,  // MMA issuer: up-projection tiles processed (a count)
    TR_T_DN_ITEMS = 29,  // MMA issuer: down-projection tiles processed (a count)
    TR_T_LAST_UP = 30,   // MMA issuer: last up-projection tile's main loop committed
    TR_PDL = 31,         // thread 0 past the wait for the predecessor grid
    kTraceSlots = 32
};

// Launch parameters of the fused kernel.
struct FusedParams {
    int M, D, F, Dk, n_slices, tiles_m, stages;
    int gate_col;            // GEGLU: F (first gate column of W_up); else 0
    uint32_t idesc_up, idesc_dn;
    uint32_t x_bytes, stage_bytes, wup_bytes, wdn_bytes;
    const void* bias_up;
    const void* bias_dn;
    const void* residual;
    int* error;
    unsigned long long wait_limit_ns;
    int pdl_wait;
};

// tx: X [M][D] (box 128 x 64); twu: W_up [D][F_up] (box Dk rows x 64); twd: W_down [F][D]
// (box 64 x 64); ty: Y store map (box 32 x 32).
kt_status launch_fused(int epi, int dtype, const void* tx, const void* twu, const void* twd, const void* ty,
                       const FusedParams& p, int grid, int smem, void* stream, bool pdl, const char** why);

// Allocation-free down projection (kt_mlp_kernels.cu): its split-K partials, tile
// counters and error word live in a static device array of this many bytes.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
kt_status noalloc_down_proj(int64_t M, int64_t F, int64_t D, int dtype, const void* H, const void* W_down,
                            const void* b_down, void* Y, void* stream, const char** why);

// LayerNorm of each row of X[M][D] into Xn[M][D] (kt_mlp_kernels.cu): fp32 statistics,
// biased variance, one rounding to the dtype.  Launched as a programmatic dependent.
kt_status launch_layernorm(int dtype, const void* X, const void* gamma, const void* beta, float eps, void* Xn,
                           int64_t M, int64_t D, void* stream, const char** why);

// Elementwise activation test kernel (kt_mlp_kernels.cu).
kt_status launch_activation(int act, bool paired, const float* z, const float* g, float* out, int64_t n,
                            void* stream, const char** why);

// One-thread kernel writing %globaltimer to dst (kt_mlp_kernels.cu).
kt_status launch_timestamp(void* dst, void* stream, const char** why);

// Copy `bytes` (a multiple of 16, both pointers 16-byte aligned; device memory or mapped
// pinned host memory) with `grid` CTAs, as a programmatic dependent of the previous kernel
// on `stream` (kt_mlp_kernels.cu).
kt_status launch_copy16(const void* src, void* dst, size_t bytes, int grid, void* stream, const char** why);

// Host launch wrappers (kt_mlp_kernels.cu).  tmA / tmB / tmC point to 128-byte
// CUtensorMaps: the A operand, the B operand and the output (H or Y) store map.
kt_status launch_gemm(int epi, int dtype, const void* tmA, const void* tmB, const void* tmC, const GemmParams& p,
                      int grid, int smem_bytes, void* stream, bool pdl, const char** why);

// Both projections in one launch: maps[0..2] the up projection's A, B and H store maps,
// maps[3..5] the down projection's; up.stages / stage_bytes / dbl_staging equal down's.
kt_status launch_mlp_two(int epi, int dtype, const void* const* maps, const GemmParams& up, const GemmParams& down,
                         int grid, int smem_bytes, void* stream, bool pdl, const char** why);

// Encode a 2-D tiled tensor map over a row-major [rows][cols] 16-bit matrix with a
// box of box_cols x box_rows and a 128- or 64-byte swizzle.  Returns false on failure.
bool encode_tmap(void* tmap128, const void* base, int dtype, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, int swizzle_bytes, const char** why);

// tcgen05 instruction descriptor for kind::f16 with fp32 accumulation, A K-major,
// B MN-major (b_kmajor = 0) or K-major (1), M = m (128, or 256 for a CTA pair), N = n.
uint32_t make_idesc(int dtype, int n, int m, int b_kmajor = 0);

}  // namespace kt
