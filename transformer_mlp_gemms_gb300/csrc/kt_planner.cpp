// kt_planner.cpp -- padding-aware, wave-aware tile planner (host only, no GPU).
//
// Principle ("The software stack", section 2.1): candidates are ranked by the
// work they do, discounted by the padding they add, not by raw tile size; and
// section 2.2: the grid is (ceil(M/BM), ceil(N/BN), SK), SK > 1 needs a
// reduction, and every output element must be produced exactly once.  Section
// 6 of the same page: the choice is analytic -- no autotuning; measurements are
// the second opinion.  The KohakuTPU residency limits are replaced by the
// sm_103a ones: TMEM columns per accumulator (<= 256 per buffer), shared memory
// per CTA (227 KB), tcgen05 N a multiple of 16 up to 256 (here of 32: the epilogue
// stores whole 32 x 32 boxes), one CTA per SM.
//
// Model, per candidate (PAIR, BN, SK), PAIR = 2 being a CTA pair on a 256-row tile:
//   tiles   = ceil(M/(128 PAIR)) * ceil(N/BN) * SK,  waves = ceil(PAIR tiles / SMs)
//   per k-block (depth BK = 64 or 128) and CTA: t_kb = max(MMA time of 128 x BN x BK,
//                          the MMA thread's issue chain, its stage bytes / its share of
//                          the L2 feed, load latency / stages)
//   t_main  = kblocks_per_split * t_kb + t_fill
//   t_epi   = 128 * BN * c_epi          (per-element epilogue cost of the kind)
//           + (SK > 1) the fp32 partial write and the last CTA's read of SK partials
//   t_cta   = t_main + (waves-1) * max(t_main, t_epi) + t_epi   (two TMEM buffers)
// and the candidate with the smallest t_cta wins; ties go to the larger
// tile (fewer, more intense tiles).  All constants are a model; est_us is never
// reported as a measurement.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "kt_internal.h"

namespace kt {
namespace {

constexpr double kClk = 2.0e9;             // SM clock of short kernels on GB300 (measured 1.9-2.07 GHz)
constexpr double kRsm = 8192.0 * kClk;    // dense 16-bit FLOP/s per SM: 4096 MAC per clock
// The single MMA-issuing thread (measured with clock64 on GB300): about 80 cycles per
// tcgen05.mma instruction, and about 200 cycles per stage for the full-barrier wait,
// the commit and the loop.
constexpr double kIssuePerMma = 80.0 / kClk;
constexpr double kIssuePerStage = 200.0 / kClk;
constexpr double kL2Feed = 20e12;         // aggregate L2 -> SM bytes/s (model)
constexpr double kSmFeedMax = 240e9;      // one SM's fill bandwidth (model)
constexpr double kTFill = 0.35e-6;        // pipeline fill + drain latency per tile (model)
// Load latency that the stages in flight must cover (all but the one the MMAs read), and
// a fixed cost per k-block that nothing overlaps (calibrated on GB300 with a measured
// sweep of tile shapes: the main loop runs at about max(MMA, issue, feed,
// 1.2 us / (stages - 1)) + 0.17 us per k-block, so that deep k-blocks of large TMA
// boxes beat more, shallower stages holding the same bytes, given three stages or more).
constexpr double kLoadLatency = 1.2e-6;
constexpr double kStageCost = 0.17e-6;
// The fused H-on-chip kernel's ring (two stages per 64-column slice) was calibrated
// against the two-kernel path with a load latency of 2.0 us per ring pass.
constexpr double kFusedLoadLatency = 2.0e-6;
// Launch, set-up, first loads and drain of one kernel, as CUDA events around a single
// launch see them (calibrated; shifts every candidate equally, so it does not change
// the ranking).
constexpr double kKernelOverhead = 8.5e-6;
// Split-K exchange rates of one SM (measured on GB300 with a probe of 120 CTAs moving
// 96 KB each): stores out of the SM ~40-50 GB/s (per-thread or bulk copies), reads of
// L2-resident data ~70 GB/s; a partial is written once and read once.
constexpr double kSmStoreRate = 32e9;
constexpr double kSmReadRate = 70e9;
// Clusters of SK CTAs that can be resident at once on a 152-SM GB300 (measured with
// cudaOccupancyMaxActiveClusters at one CTA per SM); sizes not listed are not used.
int max_active_clusters(int size, int num_sms) {
    int cap = 0;
    switch (size) {
        case 2: cap = 76; break;
        case 3: cap = 46; break;
        case 4: cap = 36; break;
        case 6: cap = 23; break;
        case 8: cap = 15; break;
        default: return 0;
    }
    return (int)((int64_t)cap * num_sms / 152);
}
// Extra cost of a CTA pair (calibrated): once per kernel for cluster launch, paired
// tensor-memory allocation and cluster barriers, and per tile for the cross-CTA
// barrier traffic of the main loop and epilogue.
constexpr double kPairKernelCost = 3.0e-6;
constexpr double kPairTileCost = 0.3e-6;
// Splits along K of the one-launch down projection's tiles considered by the planner, and
// the fixed cost of their reduce-scatter (the arrival handshake of the splits) beside its
// partial traffic.
constexpr int kOneLaunchMaxSplit = kRsMaxSplit;
constexpr double kOneLaunchSplitCost = 1.0e-6;
// GEGLU's one-launch splits are summed by the last split to arrive (all partials through
// global memory, read back by one CTA): calibrated on GB300 at 7 us over the modelled exchange.
constexpr double kOneLaunchLastArriverCost = 7.0e-6;

double epi_cost_per_elem(int epi) {      // seconds per output element per SM (model)
    switch (epi) {
        case EPI_GELU_ERF: return 0.11e-9;
        case EPI_GELU_TANH: return 0.07e-9;
        case EPI_GEGLU: return 0.13e-9;
        case EPI_NONE: return 0.03e-9;
        case EPI_GELU_SIGMOID:
        case EPI_SILU: return 0.07e-9;
        default: return 0.03e-9;
    }
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int max_stages(int BN, int n_b, int pair, int bk, int kmaj, int epi) {
    int s = (kSmemBudget - smem_reserve(epi)) / stage_bytes(BN, n_b, pair, bk, kmaj);
    return std::min(s, kMaxStages);
}

bool evaluate(int64_t M, int64_t N, int64_t K, int BN, int SK, int n_b, int epi, int num_sms, int pair,
              int bk, GemmConfig* g, bool cluster_sk = false, int kmaj = 0, int force_stages = 0) {
    // GEGLU: value and gate columns form one MMA operand of N = 2 BN (at most 256, one
    // accumulator buffer of tensor memory); an N-major share must be whole 64-column boxes
    // (its epilogue pairs each 32-column group of value columns with the gate columns one
    // share further on: a share must hold whole 32-column groups)
    if (n_b == 2 && (n_b * BN > kAccSlot || (!kmaj && (BN / pair) % 64 != 0) || (BN / pair) % 32 != 0)) return false;
    int stages = max_stages(BN, n_b, pair, bk, kmaj, epi);
    if (force_stages > 0) {  // a ring shared with another GEMM (one launch for both projections)
        if (force_stages > stages) return false;
        stages = force_stages;
    }
    if (stages < 2) return false;
    if (pair == 2 && num_sms < 2) return false;
    const int64_t bm = (int64_t)kBM * pair;  // rows per tile (a pair's tile spans two CTAs)
    int64_t tm = cdiv(M, bm), tn = cdiv(N, BN), kb = cdiv(K, bk);
    int64_t kps = cdiv(kb, SK);
    int64_t sk_eff = cdiv(kb, kps);  // no empty split
    if (sk_eff != SK) return false;
    int64_t tiles = tm * tn * SK;
    if (tiles > (int64_t)1 << 29) return false;
    const int64_t slots = (num_sms / pair) * pair;  // CTAs resident at once (pairs need two SMs)
    int64_t ctas = tiles * pair;
    int64_t grid = std::min<int64_t>(ctas, slots);
    int64_t waves = cdiv(ctas, slots);
    if (cluster_sk) {
        // the SK CTAs of a tile form a cluster: one tile per CTA, all clusters resident at
        // once, and the idle stage ring stages the tile's fp32 partial for its bulk copies
        if (epi != EPI_DOWN || pair != 1 || SK < 2 || SK > 8) return false;
        if (tm * tn > max_active_clusters(SK, num_sms)) return false;
        if ((int64_t)stages * stage_bytes(BN, n_b, pair, bk, kmaj) < (int64_t)kBM * BN * 4) return false;
        grid = ctas;
        waves = 1;
    }

    // per CTA and k-block: the MMA time of its 128 rows, the issue chain of the one MMA
    // thread (in a pair it issues for both CTAs), the time to stream its share of the
    // operands, and the load latency the ring of `stages` k-blocks has to cover
    double t_mma = n_b * 2.0 * kBM * BN * bk / kRsm;
    double t_issue = kIssuePerStage + (bk / 16) * kIssuePerMma;
    double bytes_kb = (double)stage_bytes(BN, n_b, pair, bk, kmaj);
    double feed = std::min(kSmFeedMax, kL2Feed / (double)grid);
    double t_kb = std::max(std::max(t_mma, t_issue), std::max(bytes_kb / feed, kLoadLatency / (stages - 1))) +
                  kStageCost;
    double t_main = (double)kps * t_kb + kTFill + (pair == 2 ? kPairTileCost : 0.0);
    double t_epi = (double)kBM * BN * epi_cost_per_elem(epi);
    // split-K (calibrated on GB300): writing the fp32 partial, then the last CTA reading
    // all SK partials, both latency-bound at a few tens of GB/s per SM; in a cluster: the
    // (SK-1)/SK of the partial other CTAs own written, a cluster-wide handshake, the
    // owner's reads of its 1/SK of the tile from every other split
    // The exchange moves partials through the same SM ports the main loop loads through,
    // so it does not hide under the next tile's main loop: it is paid once per wave.
    const double part = kBM * BN * 4.0;  // one fp32 partial tile
    double t_x = 0.0;
    if (SK > 1 && !cluster_sk) t_x = part / kSmStoreRate + SK * part / kSmReadRate;
    if (SK > 1 && cluster_sk) t_x = 0.5e-6 + (SK - 1.0) / SK * part * (1.0 / kSmStoreRate + 1.0 / kSmReadRate);
    double t_cta = t_main + (waves - 1) * std::max(t_main, t_epi) + t_epi + waves * t_x;

    g->M = M; g->N = N; g->K = K;
    g->BN = BN; g->stages = stages; g->split_k = SK;
    g->tiles_m = (int)tm; g->tiles_n = (int)tn; g->kblocks = (int)kb;
    g->kblocks_per_split = (int)kps;
    g->grid = (int)grid; g->waves = (int)waves;
    g->smem_bytes = stages * stage_bytes(BN, n_b, pair, bk, kmaj) + smem_reserve(epi);
    // a second set of output staging buffers where it costs no pipeline stage: a warp's
    // next store then need not wait for its previous one to be read out
    g->dbl_staging = g->smem_bytes + epi_warps(epi) * 2048 <= kSmemBudget ? 1 : 0;
    if (g->dbl_staging) g->smem_bytes += epi_warps(epi) * 2048;
    g->b_kmajor = kmaj;
    g->n_b = n_b;
    g->pair = pair;
    g->bk = bk;
    g->cluster_sk = cluster_sk ? 1 : 0;
    g->useful_over_padded = (double)M * N * K /
                            ((double)(tm * bm) * (double)(tn * BN) * (double)(kb * bk));
    g->est_us = (t_cta + kKernelOverhead + (pair == 2 ? kPairKernelCost : 0.0)) * 1e6;
    g->t_tile_us = t_main * 1e6;
    g->t_epi_us = t_epi * 1e6;
    g->t_x_us = t_x * 1e6;
    return true;
}

// N-major weight boxes of 16 columns (a CTA share that is an odd multiple of 16) move 32-byte
// rows: four times the L2 requests per byte of 64-column boxes.  Measured on GB300 they lose
// (SDXL level 2's down projection as 256 x 160 pair tiles, 16-column boxes: 75.8 us; as
// 256 x 192, 32-column boxes: 73.7 us), so the planner's own search leaves them out; a
// forced plan (KT_FORCE_UP / KT_FORCE_DOWN) may still use them.
bool narrow_boxes(int BN, int pair, int kmaj) { return !kmaj && b_box_cols(BN, pair) < 32; }

bool better(const GemmConfig& a, const GemmConfig& b) {
    // a strictly better than b?
    if (a.est_us < b.est_us * (1.0 - 1e-9)) return true;
    if (b.est_us < a.est_us * (1.0 - 1e-9)) return false;
    if (a.BN != b.BN) return a.BN > b.BN;
    if (a.pair != b.pair) return a.pair > b.pair;
    if (a.bk != b.bk) return a.bk > b.bk;
    return a.split_k < b.split_k;
}

bool choose(int64_t M, int64_t N, int64_t K, int n_b, int epi, int max_sk, int num_sms,
            GemmConfig* best, bool allow_cluster_sk, int kmaj) {
    bool found = false;
    for (int pair = 1; pair <= 2; ++pair) {
        for (int BN = 32; BN <= 256; BN += 32) {  // whole 32-column store boxes
            // (a pair splits the columns into two shares, multiples of 16: whole 16-column
            // weight boxes; the epilogue stores 32-column boxes of the whole tile)
            if (narrow_boxes(BN, pair, kmaj)) continue;
            for (int bk = 64; bk <= 128; bk += 64) {
                for (int SK = 1; SK <= max_sk; ++SK) {
                    for (int cl = 0; cl <= (allow_cluster_sk ? 1 : 0); ++cl) {
                        GemmConfig g;
                        if (!evaluate(M, N, K, BN, SK, n_b, epi, num_sms, pair, bk, &g, cl == 1, kmaj)) continue;
                        if (!found || better(g, *best)) {
                            *best = g;
                            found = true;
                        }
                    }
                }
            }
        }
    }
    return found;
}

}  // namespace

// The fused H-on-chip kernel: feasibility (tensor memory: Y[128 x Dk] beside two slice
// accumulators; shared memory: X tile, two H slices and a ring of >= 2 weight stages) and
// its modelled time.  Per CTA and row block, each 64-column slice costs the larger of its
// MMAs (up and down), its weight bytes at the SM's load rate, its epilogue and the load
// latency its two ring stages must cover; the slices pipeline, so the row block costs
// n_slices of those plus one X load and the Y epilogue.
static bool plan_fused(int64_t M, int64_t D, int64_t F, int act, int num_sms, FusedConfig* f) {
    const int n_b = act == KT_ACT_GEGLU ? 2 : 1;
    if (D < 1 || D > 256 || num_sms < 1) return false;
    const int Dk = (int)((D + 63) / 64 * 64);
    if (Dk + 2 * n_b * kFusedSlice > kTmemCols) return false;
    const uint32_t x_bytes = (uint32_t)(Dk / 64) * 16384u;
    const uint32_t wup = (uint32_t)(n_b * Dk) * 128u, wdn = (uint32_t)Dk * 128u;
    const uint32_t stage = std::max(wup, wdn);
    const int fixed = (int)x_bytes + 2 * 16384 + kSmemReserve;
    const int stages = std::min(kMaxStages, (kSmemBudget - fixed) / (int)stage);
    if (stages < 2) return false;
    const int64_t tiles_m = cdiv(M, kBM);
    const int64_t n_slices = cdiv(F, kFusedSlice);
    if (tiles_m > ((int64_t)1 << 29) || n_slices > ((int64_t)1 << 20)) return false;
    f->Dk = Dk;
    f->n_b = n_b;
    f->n_slices = (int)n_slices;
    f->tiles_m = (int)tiles_m;
    f->grid = (int)std::min<int64_t>(tiles_m, num_sms);
    f->waves = (int)cdiv(tiles_m, num_sms);
    f->stages = stages;
    f->smem_bytes = fixed + stages * (int)stage;
    f->x_bytes = x_bytes;
    f->stage_bytes = stage;
    f->wup_bytes = wup;
    f->wdn_bytes = wdn;
    const double t_mma = (n_b + 1) * 2.0 * kBM * kFusedSlice * Dk / kRsm;
    const double t_load = (double)(wup + wdn) / 100e9;
    const double t_epi = (double)kBM * kFusedSlice * epi_cost_per_elem(up_epilogue(act));
    // each slice takes two ring stages (its W_up and its W_down slices): the ring must
    // cover the load latency as in the two-kernel main loop
    const double t_lat = 2.0 * kFusedLoadLatency / stages;
    const double t_slice = std::max(std::max(t_mma, t_load), std::max(t_epi, t_lat));
    const double t_rb =
        (double)n_slices * t_slice + kFusedLoadLatency / 2 + (double)kBM * Dk * epi_cost_per_elem(EPI_DOWN);
    f->est_us = ((double)f->waves * t_rb + kKernelOverhead) * 1e6;
    return true;
}

// Both projections in one persistent launch, tiles from one dynamic queue (up tiles first):
// the down projection's candidates with the up projection's CTA pairing, whole tiles or
// split along K (each split a work item; the last CTA to finish a tile sums the partials
// through global memory), the two GEMMs sharing one shared-memory ring (its stage the
// larger of their k-blocks).  Modelled time: the up tiles spread over the units, then the
// down items in whole rounds of one item per unit (a down item is long: a round a few
// items short of the units' count still costs a full item), at least the total work spread
// over the units, plus the last epilogue (with the split-K exchange) and the launch.
static void plan_one_launch(int64_t M, int64_t D, int64_t F, int act, int num_sms, int kmaj, PlanChoice* out,
                            const GemmConfig* forced_up, const GemmConfig* forced_down) {
    out->one_launch = 0;
    out->one_est_us = 0.0;
    const int epi_up = up_epilogue(act);
    const int n_b = act == KT_ACT_GEGLU ? 2 : 1;
    // the up projection's candidates: the forced one, or the best tile of each CTA pairing
    // (the down projection runs with the same pairing in one launch)
    GemmConfig ups[2];
    int n_ups = 0;
    if (forced_up) {
        ups[n_ups++] = *forced_up;
    } else {
        for (int pair = 1; pair <= 2; ++pair) {
            bool got = false;
            for (int BN = 32; BN <= 256; BN += 32)
                for (int bk = 64; bk <= 128; bk += 64) {
                    if (narrow_boxes(BN, pair, kmaj)) continue;
                    GemmConfig g;
                    if (!evaluate(M, F, D, BN, 1, n_b, epi_up, num_sms, pair, bk, &g, false, kmaj)) continue;
                    if (!got || better(g, ups[n_ups])) {
                        ups[n_ups] = g;
                        got = true;
                    }
                }
            if (got) ++n_ups;
        }
    }
    bool found = false;
    for (int iu = 0; iu < n_ups; ++iu) {
    const GemmConfig& u0 = ups[iu];
    const int pair = u0.pair;
    const int units = num_sms / pair;
    for (int BN = 32; BN <= 256; BN += 32)
      for (int bk = 64; bk <= 128; bk += 64)
        for (int SK = 1; SK <= kOneLaunchMaxSplit; ++SK) {
            if (forced_down && (forced_down->BN != BN || forced_down->bk != bk || forced_down->pair != pair ||
                                forced_down->split_k != SK || forced_down->cluster_sk))
                continue;
            if (!forced_down && narrow_boxes(BN, pair, kmaj)) continue;
            GemmConfig d0;
            if (!evaluate(M, D, F, BN, SK, 1, EPI_DOWN, num_sms, pair, bk, &d0, false, kmaj)) continue;
            const int slot = std::max(stage_bytes(u0.BN, n_b, pair, u0.bk, kmaj), stage_bytes(BN, 1, pair, bk, kmaj));
            const int stages = std::min((kSmemBudget - smem_reserve(epi_up)) / slot, kMaxStages);
            GemmConfig u, d;
            if (stages < 2 || !evaluate(M, F, D, u0.BN, 1, n_b, epi_up, num_sms, pair, u0.bk, &u, false, kmaj, stages) ||
                !evaluate(M, D, F, BN, SK, 1, EPI_DOWN, num_sms, pair, bk, &d, false, kmaj, stages))
                continue;
            const double up_tiles = (double)u.tiles_m * u.tiles_n;
            const double dn_items = (double)d.tiles_m * d.tiles_n * SK;
            // a split is worth its exchange only while all the items run in one round
            if (SK > 1 && !forced_down && dn_items > units) continue;
            const int grid = (int)std::min<int64_t>((int64_t)units, (int64_t)(up_tiles + dn_items)) * pair;
            const double n = grid / pair;
            const double work = (up_tiles * u.t_tile_us + dn_items * d.t_tile_us) / n;
            const double rounds = up_tiles * u.t_tile_us / n + std::ceil(dn_items / n) * d.t_tile_us;
            // the splits of a tile reduce-scatter their partials: each writes the (SK - 1) / SK
            // of its fp32 partial that other splits own and reads as much back
            const double part = kBM * BN * 4.0;
            const double t_x = SK == 1 ? 0.0
                               : act == KT_ACT_GEGLU
                                   ? d.t_x_us + kOneLaunchLastArriverCost * 1e6
                                   : ((SK - 1.0) / SK * part * (1.0 / kSmStoreRate + 1.0 / kSmReadRate) +
                                      kOneLaunchSplitCost) * 1e6;
            const double t = std::max(work, rounds) + std::max(u.t_epi_us, d.t_epi_us + t_x) +
                             kKernelOverhead * 1e6 + (pair == 2 ? kPairKernelCost * 1e6 : 0.0);
            if (!found || t < out->one_est_us) {
                found = true;
                out->one_est_us = t;
                out->one_grid = grid;
                out->one_stages = stages;
                out->one_slot = slot;
                const int smem = stages * slot + smem_reserve(epi_up);
                out->one_dbl = smem + epi_warps(epi_up) * 2048 <= kSmemBudget ? 1 : 0;
                out->one_smem = smem + (out->one_dbl ? epi_warps(epi_up) * 2048 : 0);
                u.dbl_staging = d.dbl_staging = out->one_dbl;
                u.stages = d.stages = stages;
                u.smem_bytes = d.smem_bytes = out->one_smem;
                d.t_x_us = t_x;
                out->one_up = u;
                out->one_down = d;
            }
        }
    }
    if (found) out->one_launch = 1;
}

kt_status plan_choose(int64_t M, int64_t D, int64_t F, int act, int num_sms, PlanChoice* out,
                      const char** why, bool allow_cluster_sk, int w_layout, int h_path, bool allow_one_launch,
                      int launches) {
    if (M < 1 || D < 1 || F < 1) { *why = "M, D and F must be positive"; return KT_ERR_INVALID; }
    if (act < KT_ACT_GELU_ERF || act > KT_ACT_SILU) { *why = "unknown activation"; return KT_ERR_INVALID; }
    if (w_layout != KT_W_IN_OUT && w_layout != KT_W_OUT_IN) { *why = "unknown weight layout"; return KT_ERR_INVALID; }
    if (h_path != KT_H_AUTO && h_path != KT_H_MEMORY && h_path != KT_H_ON_CHIP) {
        *why = "unknown H path";
        return KT_ERR_INVALID;
    }
    out->h_on_chip = 0;
    const int kmaj = w_layout == KT_W_OUT_IN ? 1 : 0;
    if (num_sms < 1) { *why = "num_sms must be positive"; return KT_ERR_INVALID; }
    if (D % 8 != 0 || F % 8 != 0) {
        *why = "D and F must be multiples of 8 (16-byte row pitch for TMA)";
        return KT_ERR_UNSUPPORTED;
    }
    const int64_t lim = (int64_t)1 << 30;
    int64_t F_up = act == KT_ACT_GEGLU ? 2 * F : F;
    if (M >= lim || D >= lim || F_up >= lim || M * F >= ((int64_t)1 << 40) ||
        M * D >= ((int64_t)1 << 40)) {
        *why = "sizes beyond the supported index range";
        return KT_ERR_UNSUPPORTED;
    }
    int epi_up = up_epilogue(act);
    int n_b = act == KT_ACT_GEGLU ? 2 : 1;
    if (!choose(M, F, D, n_b, epi_up, 1, num_sms, &out->up, false, kmaj)) {
        *why = "no feasible tile for the up projection";
        return KT_ERR_UNSUPPORTED;
    }
    if (!choose(M, D, F, 1, EPI_DOWN, 16, num_sms, &out->down, allow_cluster_sk, kmaj)) {
        *why = "no feasible tile for the down projection";
        return KT_ERR_UNSUPPORTED;
    }
    // Measurement overrides (planner calibration sweeps): KT_FORCE_UP="BN[,PAIR[,BK]]" and
    // KT_FORCE_DOWN="BN,SK[,PAIR[,BK[,CLUSTER]]]".  An infeasible override is an error, never ignored.
    if (const char* e = std::getenv("KT_FORCE_UP")) {
        int bn = 0, pr = 1, bk = 64;
        GemmConfig g;
        int nf = std::sscanf(e, "%d,%d,%d", &bn, &pr, &bk);
        if (nf < 1 || (pr != 1 && pr != 2) || (bk != 64 && bk != 128) || bn % 32 != 0 || bn < 32 ||
            bn > 256 || !evaluate(M, F, D, bn, 1, n_b, epi_up, num_sms, pr, bk, &g, false, kmaj)) {
            *why = "KT_FORCE_UP must be a feasible \"BN[,PAIR[,BK]]\" (BN a multiple of 32; BK 64 or "
                   "128; GEGLU: BN <= 128, and BN / PAIR a multiple of 64 for [in][out] weights)";
            return KT_ERR_INVALID;
        }
        out->up = g;
    }
    if (const char* e = std::getenv("KT_FORCE_DOWN")) {
        int bn = 0, sk = 0, pr = 1, bk = 64, cl = 0;
        GemmConfig g;
        int nf = std::sscanf(e, "%d,%d,%d,%d,%d", &bn, &sk, &pr, &bk, &cl);
        if (nf < 2 || (pr != 1 && pr != 2) || (bk != 64 && bk != 128) || bn % 32 != 0 || bn < 32 ||
            bn > 256 || sk < 1 || sk > 64 || (cl && !allow_cluster_sk) ||
            !evaluate(M, D, F, bn, sk, 1, EPI_DOWN, num_sms, pr, bk, &g, cl != 0, kmaj)) {
            *why = "KT_FORCE_DOWN must be a feasible \"BN,SK[,PAIR[,BK[,CLUSTER]]]\" (no empty split)";
            return KT_ERR_INVALID;
        }
        out->down = g;
    }
    // the H path: the fused kernel where it applies ([in][out] weights, D small enough)
    // and is asked for, or, in KT_H_AUTO, where the model prefers it to two kernels
    if (h_path != KT_H_MEMORY) {
        const bool fits = w_layout == KT_W_IN_OUT && plan_fused(M, D, F, act, num_sms, &out->fused);
        if (h_path == KT_H_ON_CHIP && !fits) {
            *why = "the H-on-chip kernel needs [in][out] weights and D <= 256 (<= 192 for GEGLU)";
            return KT_ERR_UNSUPPORTED;
        }
        if (fits && (h_path == KT_H_ON_CHIP || out->fused.est_us < out->up.est_us + out->down.est_us))
            out->h_on_chip = 1;
    }
    // Both projections in one launch (KT_LAUNCH_ONE), where H goes through memory.  The
    // planner's own choice (KT_LAUNCH_AUTO) is one launch wherever a one-launch plan exists:
    // the second kernel's launch, its CTAs' set-up and the partial waves at the boundary
    // between the projections cost more than one launch's work queue now that the queue
    // hands items on without cluster-scope release-ordered arrivals (GB300, CUDA events,
    // 256 MiB scrub between calls; one launch against two: SigLIP 32.3 against 37.7 us,
    // M = 256 24.6 against 29.6, M = 1000 35.1 against 38.2, M = 4096 69.7 against 77.6,
    // SDXL level 2 69.2 against 70.7, SDXL level 1 81.5 against 84.0, M = 16384 227.6
    // against 229.6 us); the tiny case keeps H on chip.
    // Override: KT_FORCE_LAUNCHES=1|2.
    out->one_launch = 0;
    if (launches != KT_LAUNCH_AUTO && launches != KT_LAUNCH_ONE && launches != KT_LAUNCH_TWO) {
        *why = "unknown launches option";
        return KT_ERR_INVALID;
    }
    const char* fl = std::getenv("KT_FORCE_LAUNCHES");
    if (fl) {
        const int v = std::atoi(fl);
        if (v != 1 && v != 2) {
            *why = "KT_FORCE_LAUNCHES must be 1 or 2";
            return KT_ERR_INVALID;
        }
        launches = v == 1 ? KT_LAUNCH_ONE : KT_LAUNCH_TWO;
    }
    const bool forced_dn = std::getenv("KT_FORCE_DOWN") != nullptr;
    const bool auto_one = launches == KT_LAUNCH_AUTO && !forced_dn;
    const int force_launches = launches == KT_LAUNCH_ONE ? 1 : auto_one ? 0 : 2;
    if (allow_one_launch && !out->h_on_chip && force_launches != 2) {
        plan_one_launch(M, D, F, act, num_sms, kmaj, out, std::getenv("KT_FORCE_UP") ? &out->up : nullptr,
                        forced_dn ? &out->down : nullptr);
        if (out->one_launch) {  // the configurations that launch runs
            out->up = out->one_up;
            out->down = out->one_down;
        }
    }
    if (allow_one_launch && force_launches == 1 && !out->one_launch) {
        *why = "one launch: no configuration applies (H stays on chip, or no whole-tile down projection fits)";
        return KT_ERR_UNSUPPORTED;
    }
    return KT_OK;
}

int up_epilogue(int act) {
    switch (act) {
        case KT_ACT_GELU_ERF: return EPI_GELU_ERF;
        case KT_ACT_GELU_TANH: return EPI_GELU_TANH;
        case KT_ACT_GEGLU: return EPI_GEGLU;
        case KT_ACT_GELU_SIGMOID: return EPI_GELU_SIGMOID;
        case KT_ACT_SILU: return EPI_SILU;
    }
    return EPI_NONE;
}

void plan_fill_info(const GemmConfig& g, kt_gemm_plan_info* o) {
    o->BM = kBM * g.pair; o->BN = g.BN; o->BK = g.bk;
    o->stages = g.stages; o->split_k = g.split_k;
    o->tiles_m = g.tiles_m; o->tiles_n = g.tiles_n; o->kblocks = g.kblocks;
    o->grid = g.grid; o->waves = g.waves;
    o->smem_bytes = g.smem_bytes; o->tmem_cols = kTmemCols;
    o->cluster_sk = g.cluster_sk; o->b_kmajor = g.b_kmajor;
    o->M = g.M; o->N = g.N; o->K = g.K;
    o->useful_over_padded = g.useful_over_padded;
    o->est_us = g.est_us;
}

}  // namespace kt
