// kt_gemm.cuh -- the sm_103a GEMM kernel template of the fused MLP (device code
// and its launch helper), included by the translation units that instantiate it.
//
// One persistent, warp-specialised kernel template serves both projections, on one
// CTA per 128-row tile (PAIR = 1) or on a CTA pair per 256-row tile (PAIR = 2,
// tcgen05 cta_group::2: each CTA loads its 128 rows of A and half of the B columns):
//
//   warp 0      A producer: TMA (cp.async.bulk.tensor, 128-byte swizzle) loads of the
//               A tile (128 x 64 K-major boxes, one per 64-deep atom of a BK = 64 or
//               128 k-block) into an S-stage shared-memory ring, one mbarrier pair
//               (full / empty) per stage; its arrival on the full barrier carries the
//               stage's byte count.  The down projection's A producer first waits for
//               the up projection's per-row-block counters of stored H tiles.
//   warp 10     B producer: the B tile(s) of the same stages -- N-major boxes of an
//               [in][out] weight, 64, 32 or 16 columns wide (128-, 64- or 32-byte swizzle:
//               the widest that divides the CTA's column share), or (BN / PAIR)-row
//               K-major boxes of an [out][in] weight.  Two issuing threads take in about
//               twice the bytes per second of one.
//   warp 1      MMA issuer: one thread of the leader CTA issues tcgen05.mma kind::f16
//               (M = 128 or 256, N = BN, K = 16, fp32 accumulation in tensor memory),
//               BK / 16 per k-block, and tcgen05.commit hands the stage back.  Two
//               TMEM accumulator buffers let tile i+1's main loop run under tile i's
//               epilogue.  GEGLU loads the value and the gate columns of its tile as
//               one B operand, so one MMA of N = 2 BN fills both accumulators.
//   warps 2-9   epilogue: tcgen05.ld moves the fp32 accumulator to registers (TMEM
//               lane = tile row), adds the bias (staged per tile in shared memory),
//               applies the activation (GELU erf / tanh / sigmoid, SiLU, GEGLU
//               value * gelu(gate)), rounds ONCE to the I/O dtype, stages each warp's
//               32 x 32 block in swizzled shared memory and writes it with a TMA
//               tensor store (clipped at the ragged edges).  The up projection then
//               counts the stored tile for the down projection.  The down projection
//               adds b_down and the residual and stores Y; with split-K its CTAs
//               either reduce-scatter their fp32 partials through L2 inside a
//               cluster (each 32 x 32 unit summed by its owner CTA, its own partial
//               still in TMEM) or write them to global memory for the last CTA to
//               arrive on the tile; partials are always summed in split order.
//
// TWO = true runs both projections in one launch: the up projection's tiles, then the
// down projection's (whole tiles, or K splits whose partials the last CTA to finish a
// tile sums through global memory), taken from one global work counter by the leader
// CTA's producer and published to every role of the CTA (pair) through a small ring of
// item indices in shared memory; a down tile's producer waits for the counters of its
// rows of H as above.  Each role's per-tile work is a lambda over one projection's
// parameters (the epilogue's also over its epilogue kind), shared by both modes.
//
// Sources: "SDXL as a requirements inventory", section 1.3 (FeedForward: value =
// first half, gate = second half) and 9.3 (erf GELU); "MLP layout sweep and
// remaining representation limits" (the SigLIP MLP, tanh GELU, K-partitioned
// down projection with a reduction); "The software stack", sections 2.2 (3-D grid,
// split-K needs a reduction, every output element produced exactly once), 2.3
// (epilogue folding; the accumulator is never a memory word) and 2.4 (B resident,
// A double-buffered -> here a multi-stage ring).
//
// Every device-side wait is bounded by %globaltimer; on expiry the kernel records
// an error code, raises a CTA-wide abort flag, drains its own in-flight copies and
// MMAs (again bounded), frees tensor memory and returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "kt_internal.h"

namespace kt {

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void trace_mark(unsigned long long* tr, int slot) {
    if (tr) tr[(size_t)blockIdx.x * kTraceSlots + slot] = global_ns();
}
// As trace_mark, keeping the latest of several threads' marks.
__device__ __forceinline__ void trace_max(unsigned long long* tr, int slot) {
    if (tr) atomicMax(tr + (size_t)blockIdx.x * kTraceSlots + slot, global_ns());
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Non-blocking test of the phase of parity `parity` (no suspension: the fast path of a
// wait whose phase has usually completed already).
__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// As mbar_try_wait, acquiring at cluster scope: for barriers whose phase completes on
// data written by other CTAs of the cluster (remote asynchronous stores).
__device__ __forceinline__ uint32_t mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Wait for the phase of parity `parity` of barrier `bar` to complete.  Returns
// false if the CTA is aborting or if `limit_ns` passed (then raises the abort
// flag and records `code` in the error word, first writer wins).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err, int code, unsigned long long limit_ns) {
    auto try_wait = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_wait()) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_wait()) return true;
        if ((i & 31u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, code);
                return false;
            }
        }
    }
}

// Wait until the counter at `ctr` reaches `target` (wrap-around compare), acquiring at
// GPU scope.  Gives up, with the abort flag raised, when the error word shows that an
// earlier kernel failed, when this CTA aborts, or after limit_ns (error code recorded).
__device__ __forceinline__ bool wait_counter(const unsigned* ctr, unsigned target, volatile int* abort_flag, int* err,
                                             unsigned long long limit_ns, int code = DEV_TIMEOUT_PRODUCER) {
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if ((int)(v - target) >= 0) return true;
        if ((i & 15u) == 15u) {
            if (*abort_flag || *reinterpret_cast<volatile int*>(err) != 0) {
                *abort_flag = 1;
                return false;
            }
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, code);
                return false;
            }
        }
        __nanosleep(32);
    }
}

// As wait_counter, on a 64-bit counter that only grows (no wrap-around within a run's
// reach): waits until it reaches `target`; a time-out records DEV_TIMEOUT_EPILOGUE.
__device__ __forceinline__ bool wait_counter64(const unsigned long long* ctr, unsigned long long target,
                                               volatile int* abort_flag, int* err, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((i & 15u) == 15u) {
            if (*abort_flag || *reinterpret_cast<volatile int*>(err) != 0) {
                *abort_flag = 1;
                return false;
            }
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, DEV_TIMEOUT_EPILOGUE);
                return false;
            }
        }
        __nanosleep(32);
    }
}

// Drain wait used on the abort path: ignores the abort flag, bounded by limit_ns.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Tensor-memory allocation.  With PAIR = 2 (cta_group::2) one warp of each CTA of the
// pair performs the allocation collectively; the same columns are allocated in both.
template <int PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    if constexpr (PAIR == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <int PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (PAIR == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same rendezvous without release ordering, for the kernel's start: what the peers
// must see of this CTA's set-up (its barriers' initialisation) is already published by
// fence.mbarrier_init.release.cluster.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster shared window, of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its cluster-window address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrivals without release ordering (a release-ordered arrival costs its thread several
// tenths of a microsecond): for a thread whose earlier accesses the waiter depends on are
// complete by other means: a load that an acquire orders before the arrival (the work
// queue's slots), or tensor-memory loads that tcgen05.wait::ld has completed (an epilogue
// handing its accumulator back to the MMA issuer).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Hand a 32-bit value to the waiters of a cluster peer's barrier (both addresses in the
// peer's shared memory): the arrival announces 4 bytes, and an asynchronous store of the
// value completes them, so the phase completes only once the value is in place.
__device__ __forceinline__ void post_index(uint32_t slot_cluster, uint32_t bar_cluster, int value) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], 4;" ::"r"(bar_cluster)
                 : "memory");
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(slot_cluster),
                 "r"(value), "r"(bar_cluster)
                 : "memory");
}

// TMA load whose completion is signalled on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar_cluster, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading-dimension and
// stride-dimension byte offsets (all >> 4), descriptor version 1 (bits 46-48 =
// 0b001), base offset 0 (tiles are 1024-byte aligned), swizzle mode in bits 61-63:
// 128-byte swizzle (= 2) by default, 64-byte swizzle (= 4).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz = 2u) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// M = 256 across the CTA pair: this CTA's smem holds A rows [0,128) and B columns
// [0, N/2) of its half; the peer's the other halves (same offsets).
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this offset in both CTAs of the pair once all prior MMAs finish.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"((unsigned short)3)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns; thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// tcgen05.wait::ld, with the loaded registers threaded through so that no use
// of them can be scheduled before the wait.  (tmem_f16cols below: 16 columns as fp32.)
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&r)[16], uint32_t (&s)[16]) {
    tmem_wait_ld(r);
    asm volatile(""
                 : "+r"(s[0]), "+r"(s[1]), "+r"(s[2]), "+r"(s[3]), "+r"(s[4]), "+r"(s[5]),
                   "+r"(s[6]), "+r"(s[7]), "+r"(s[8]), "+r"(s[9]), "+r"(s[10]), "+r"(s[11]),
                   "+r"(s[12]), "+r"(s[13]), "+r"(s[14]), "+r"(s[15])
                 :
                 : "memory");
}

// 16 consecutive fp32 accumulator columns of this lane's row (TMEM lane), waited for.
__device__ __forceinline__ void tmem_f16cols(uint32_t taddr, float* v) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Pass 32 registers through an empty asm so that no use of them is scheduled
// before the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
    asm volatile(""
                 : "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld_only() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// TMA tensor store of a box from shared memory (clipped at the tensor's bounds).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
// Untiled bulk copy of `bytes` (a multiple of 16) from shared to global memory.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int NEPI = kEpiWarps>
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NEPI * 32) : "memory");
}

// Barrier over the epilogue warps that also ANDs a predicate across them, so that
// all of them take the same branch after a bounded wait (no warp is left behind
// at a later named barrier).
template <int NEPI = kEpiWarps>
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(NEPI * 32)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------
// Epilogue arithmetic (fp32)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2_approx(float x) {  // 2^x, hardware approximation (ftz)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {  // 1/x, hardware approximation (ftz)
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of fp32 values, and their arithmetic in two forms: P = true issues the
// sm_100-family paired instructions (add / sub / mul / fma .rn.f32x2 on the two values
// as one 64-bit register pair), P = false two scalar .rn instructions.  Both round each
// lane exactly as one scalar .rn instruction does (and neither form is contracted
// into a different fma), so the two forms give the same bits; the paired one issues
// about half the instructions.  The hardware approximations (ex2, rcp) and the sign
// selects are per lane in both.  The epilogues use the paired form; the scalar one
// serves the test hook, which checks that the two agree bit for bit.
struct f32x2 {
    float x, y;
};
__device__ __forceinline__ f32x2 f2(float a, float b) { return f32x2{a, b}; }
__device__ __forceinline__ f32x2 f2(float a) { return f32x2{a, a}; }
__device__ __forceinline__ void f2_split(f32x2 v, float& a, float& b) {
    a = v.x;
    b = v.y;
}
#define KT_F2_BINARY(name, op, scalar)                                                                  \
    template <bool P>                                                                                 \
    __device__ __forceinline__ f32x2 name(f32x2 a, f32x2 b) {                                         \
        if constexpr (P) {                                                                            \
            f32x2 o;                                                                                  \
            asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" op      \
                ".rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"                                   \
                : "=f"(o.x), "=f"(o.y)                                                                \
                : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                            \
            return o;                                                                                 \
        } else {                                                                                      \
            return f32x2{scalar(a.x, b.x), scalar(a.y, b.y)};                                         \
        }                                                                                             \
    }
KT_F2_BINARY(f2_add, "add", __fadd_rn)
KT_F2_BINARY(f2_sub, "sub", __fsub_rn)
KT_F2_BINARY(f2_mul, "mul", __fmul_rn)
#undef KT_F2_BINARY
template <bool P>
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    if constexpr (P) {
        f32x2 o;
        asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
            "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
            : "=f"(o.x), "=f"(o.y)
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
        return o;
    } else {
        return f32x2{__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y)};
    }
}
__device__ __forceinline__ f32x2 f2_ex2(f32x2 v) { return f32x2{ex2_approx(v.x), ex2_approx(v.y)}; }
__device__ __forceinline__ f32x2 f2_rcp(f32x2 v) { return f32x2{rcp_approx(v.x), rcp_approx(v.y)}; }

// gelu_erf(z) = z * Phi(z), and Phi(-|z|) = erfc(a) / 2 with a = |z| / sqrt 2.
// erfc(a), a >= 0, by the Chebyshev fit of Numerical Recipes in C (2nd ed., section
// 6.2, "erfcc"): erfc(a) = t * exp(-a^2 + P(t)), t = 1 / (1 + a/2), P of degree 9,
// fractional error below 1.2e-7 for every a >= 0.  Evaluated in fp32 with the hardware
// exp2 and reciprocal, constants folded: with t' = t / 2 = 1 / (2 + a) and
// u = a sqrt(log2 e),  erfc(a) / 2 = t' * 2^(Q(t') - u^2),  Q(t') = log2(e) P(2 t')
// (coefficient i of the fit times 2^i log2 e; Horner's rule).  Then gelu = z Phi(-|z|)
// for z < 0 and z - z Phi(-|z|) for z >= 0: no cancellation for z < 0, no branches.
namespace erfc_fit {
constexpr double kL = 1.4426950408889634;  // log2(e)
constexpr float kQ9 = (float)(0.17087277 * 512.0 * kL), kQ8 = (float)(-0.82215223 * 256.0 * kL);
constexpr float kQ7 = (float)(1.48851587 * 128.0 * kL), kQ6 = (float)(-1.13520398 * 64.0 * kL);
constexpr float kQ5 = (float)(0.27886807 * 32.0 * kL), kQ4 = (float)(-0.18628806 * 16.0 * kL);
constexpr float kQ3 = (float)(0.09678418 * 8.0 * kL), kQ2 = (float)(0.37409196 * 4.0 * kL);
constexpr float kQ1 = (float)(1.00002368 * 2.0 * kL), kQ0 = (float)(-1.26551223 * kL);
constexpr float kU = 0.84932180028801907f;  // sqrt(log2(e) / 2): u = |z| kU
constexpr float kA = 0.83255461115769776f;  // 1 / sqrt(log2 e):  a = u kA
}  // namespace erfc_fit

template <bool P>
__device__ __forceinline__ f32x2 gelu_erf_f2(f32x2 z) {
    using namespace erfc_fit;
    const f32x2 az = f2(fabsf(z.x), fabsf(z.y));
    const f32x2 u = f2_mul<P>(az, f2(kU)), nu = f2_mul<P>(az, f2(-kU));  // u and -u, both exact
    const f32x2 tp = f2_rcp(f2_fma<P>(u, f2(kA), f2(2.0f)));             // t' = 1 / (2 + a)
    f32x2 q = f2_fma<P>(f2(kQ9), tp, f2(kQ8));
    q = f2_fma<P>(q, tp, f2(kQ7));
    q = f2_fma<P>(q, tp, f2(kQ6));
    q = f2_fma<P>(q, tp, f2(kQ5));
    q = f2_fma<P>(q, tp, f2(kQ4));
    q = f2_fma<P>(q, tp, f2(kQ3));
    q = f2_fma<P>(q, tp, f2(kQ2));
    q = f2_fma<P>(q, tp, f2(kQ1));
    q = f2_fma<P>(q, tp, f2(kQ0));
    const f32x2 zh = f2_mul<P>(z, f2_mul<P>(tp, f2_ex2(f2_fma<P>(nu, u, q))));  // z Phi(-|z|)
    const f32x2 r = f2_sub<P>(z, zh);
    return f2(z.x >= 0.0f ? r.x : zh.x, z.y >= 0.0f ? r.y : zh.y);
}

// gelu_tanh(z) = 0.5 z (1 + tanh(u)) = z / (1 + exp(-2u)),  u = sqrt(2/pi)(z + 0.044715 z^3);
// exp(-2u) = 2^(z (c1 + c2 z^2)), c1 = -2 sqrt(2/pi) log2(e), c2 = 0.044715 c1.
template <bool P>
__device__ __forceinline__ f32x2 gelu_tanh_f2(f32x2 z) {
    const f32x2 x = f2_mul<P>(z, f2_fma<P>(f2(-0.1029432395800235f), f2_mul<P>(z, z), f2(-2.302208198144325f)));
    return f2_mul<P>(z, f2_rcp(f2_add<P>(f2(1.0f), f2_ex2(x))));
}

// z * sigmoid(a z) = z / (1 + exp(-a z)) = z / (1 + 2^(c z)),  c = -a log2(e):
// a = 1.702 for the sigmoid form of GELU, a = 1 for SiLU.  For z -> -inf the power
// overflows to +inf and the reciprocal to 0, so the result goes to -0 (no NaN).
template <bool P>
__device__ __forceinline__ f32x2 gelu_sigmoid_f2(f32x2 z) {
    return f2_mul<P>(z, f2_rcp(f2_add<P>(f2(1.0f), f2_ex2(f2_mul<P>(z, f2(-2.4554669595930157f))))));
}
template <bool P>
__device__ __forceinline__ f32x2 silu_f2(f32x2 z) {
    return f2_mul<P>(z, f2_rcp(f2_add<P>(f2(1.0f), f2_ex2(f2_mul<P>(z, f2(-1.4426950408889634f))))));
}

template <int EPI, bool P>
__device__ __forceinline__ f32x2 act_f2(f32x2 z) {
    if constexpr (EPI == EPI_GELU_ERF) return gelu_erf_f2<P>(z);
    else if constexpr (EPI == EPI_GELU_TANH) return gelu_tanh_f2<P>(z);
    else if constexpr (EPI == EPI_GELU_SIGMOID) return gelu_sigmoid_f2<P>(z);
    else if constexpr (EPI == EPI_SILU) return silu_f2<P>(z);
    else return z;
}

// GEGLU on a pair: (value + b_value) * gelu_erf(gate + b_gate).
template <bool P>
__device__ __forceinline__ f32x2 geglu_f2(f32x2 v, f32x2 bv, f32x2 g, f32x2 bg) {
    return f2_mul<P>(f2_add<P>(v, bv), gelu_erf_f2<P>(f2_add<P>(g, bg)));
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (DT == KT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int DT>
__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (DT == KT_BF16) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&u[i]);
            float2 t = __bfloat1622float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        } else {
            __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}

// 32 bias values starting at column `col` (groups of 8 at or past `limit` read as 0).
template <int DT>
__device__ __forceinline__ void load_bias32(const void* bias, int col, int limit, float* b) {
    const uint16_t* ptr = reinterpret_cast<const uint16_t*>(bias) + col;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col + 8 * g < limit) {
            uint4 w = __ldg(reinterpret_cast<const uint4*>(ptr + 8 * g));
            unpack8<DT>(w, b + 8 * g);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) b[8 * g + i] = 0.0f;
        }
    }
}

// n (a multiple of 4) fp32 bias values from the tile's bias slice staged in shared
// memory (bsm: the first of them; columns past N were staged as zeros).  Every lane
// reads the same addresses: broadcast reads.
template <int n>
__device__ __forceinline__ void bias_from_smem(uint32_t bsm, float* b) {
#pragma unroll
    for (int g = 0; g < n / 4; ++g)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b[4 * g]), "=f"(b[4 * g + 1]), "=f"(b[4 * g + 2]), "=f"(b[4 * g + 3])
                     : "r"(bsm + 16u * g));
}

// Add n (16 or 32) values of row `row` of the residual R[M][N], starting at column
// `col`, to v (rows past M and groups of 8 at or past N are skipped: those results are
// never stored).  Plain loads: R may be the output Y itself, whose other blocks other
// threads are writing meanwhile.
template <int DT, int n = 32>
__device__ __forceinline__ void add_residual32(const void* R, int row, int M, int col, int N, float* v) {
    if (row >= M) return;
    const uint16_t* ptr = reinterpret_cast<const uint16_t*>(R) + (size_t)row * (size_t)N + col;
#pragma unroll
    for (int g = 0; g < n / 8; ++g) {
        if (col + 8 * g < N) {
            const uint4 w = *reinterpret_cast<const uint4*>(ptr + 8 * g);
            float f[8];
            unpack8<DT>(w, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * g + i] += f[i];
        }
    }
}

// Stage a warp's 32 x 32 block, already rounded to the I/O dtype (this lane's row: 32
// values packed in pairs in w), in the warp's 2 KB shared-memory buffer in the 64-byte
// swizzled layout the output tensor map expects (16-byte chunk c of row r lands at
// chunk c ^ ((r >> 1) & 3)), and store it with one TMA tensor store at (x, y).  Rows
// and columns past the tensor's bounds are clipped by the TMA unit.
__device__ __forceinline__ void stage_and_store_packed(const CUtensorMap* tmC, uint32_t stg, int lane,
                                                       const uint32_t* w, int x, int y, bool two_buffers = false) {
    // the previous store from this buffer has read it (with two buffers per warp, the
    // store from the other buffer may still be reading)
    if (lane == 0) {
        if (two_buffers) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        else bulk_wait_read0();
    }
    __syncwarp();
    const uint32_t row_base = stg + (uint32_t)lane * 64u;
    const uint32_t sw = ((uint32_t)lane >> 1) & 3u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(row_base + ((c ^ sw) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmC, stg, x, y);
        bulk_commit();
    }
}

// As stage_and_store_packed, rounding 32 fp32 values (round to nearest even) first.
template <int DT>
__device__ __forceinline__ void stage_and_store(const CUtensorMap* tmC, uint32_t stg, int lane, const float* v,
                                                int x, int y, bool two_buffers = false) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack2<DT>(v[2 * i], v[2 * i + 1]);
    stage_and_store_packed(tmC, stg, lane, w, x, y, two_buffers);
}

// The MMAs of one k-block: NK steps of K = 16 (4 for a 64-deep stage, 8 for 128).
// Descriptor start addresses move in 16-byte units.  A (K-major): +32 bytes per step
// inside a 64-deep swizzle atom, +16 KB per atom.  B N-major (KB = 0): +16 rows per
// step, b_step16 units (2 KB for 128-byte rows, 1 KB for 64-byte rows, 512 B for 32-byte rows).  B K-major
// (KB = 1): as A, with atoms of b_atom16 units.
// GEGLU needs no second MMA: its B operand holds the value and the gate columns of
// the tile side by side, so one MMA of N = 2 BN fills both accumulators.
template <int PAIR, int NK, int KB>
__device__ __forceinline__ void issue_kblock(uint32_t d, uint64_t ad0, uint64_t bd0, uint32_t idesc, uint32_t acc0,
                                             uint32_t b_atom16, uint32_t b_step16 = 128u) {
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        const uint64_t ad = ad0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2);
        const uint64_t boff = KB ? (uint64_t)((k >> 2) * b_atom16 + (k & 3) * 2) : (uint64_t)(k * b_step16);
        const uint64_t bd = bd0 + boff;
        const uint32_t acc = k == 0 ? acc0 : 1u;
        if constexpr (PAIR == 2) mma_f16_pair(d, ad, bd, idesc, acc);
        else mma_f16(d, ad, bd, idesc, acc);
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// The t-th work item of the kernel: a tile, which of its split_k partial sums this CTA
// accumulates (`split`) and that split's k-blocks [kb0, kb1).  The SK splits of one tile
// are consecutive items with a reduction in which the splits wait on one another (inside
// a cluster, or the reduce-scatter of one launch), otherwise split-major.
struct TileCoord {
    int split, tm, tn, mn;
    int kb0, kb1;
};

__device__ __forceinline__ TileCoord decode_tile(int t, const GemmParams& p) {
    TileCoord c;
    const int per_split = p.tiles_m * p.tiles_n;
    if (p.cluster_sk || p.rs_sk) {
        c.split = t % p.split_k;
        c.mn = t / p.split_k;
    } else {
        c.split = t / per_split;
        c.mn = t - c.split * per_split;
    }
    c.tm = c.mn / p.tiles_n;
    c.tn = c.mn - c.tm * p.tiles_n;
    c.kb0 = c.split * p.kblocks_per_split;
    c.kb1 = min(c.kb0 + p.kblocks_per_split, p.kblocks);
    return c;
}

// This CTA's part of a tile's operands (CTA r of the pair): its first row of A (m_r),
// its first B column (nb_r) and how many B boxes it loads per k-block (chunks_r; N-major
// B: boxes of bw columns, the widest of 64, 32 and 16 that divides the share; K-major:
// one box of the share's rows per 64-deep atom).  Boxes entirely past the tensor are not
// loaded: they would only feed accumulator rows / columns that are never stored.
// Returns the bytes this CTA's copies of one k-block bring in.
template <int PAIR>
__device__ __forceinline__ uint32_t cta_share(const GemmParams& p, const TileCoord& c, uint32_t r, int n_b, int& m_r,
                                              int& nb_r, int& chunks_r) {
    const int bcols = p.BN / PAIR;
    const int bw = b_box_cols(p.BN, PAIR);
    m_r = c.tm * (kBM * PAIR) + (int)r * kBM;
    nb_r = c.tn * p.BN + (int)r * bcols;
    const uint32_t a_b = m_r < p.M ? p.a_bytes : 0u;
    if (p.b_kmajor) {
        chunks_r = nb_r < p.N ? 1 : 0;
        return a_b + (uint32_t)(n_b * chunks_r) * p.b_bytes;
    }
    chunks_r = 0;  // boxes of the share that start inside [0, N)
    for (int ch = 0; ch * bw < bcols; ++ch)
        if (nb_r + bw * ch < p.N) chunks_r = ch + 1;
    return a_b + (uint32_t)(n_b * chunks_r) * ((uint32_t)p.bk * (uint32_t)bw * 2u);
}

// The copies of one k-block (starting at K = k0) into the stage at sA with full barrier
// fb.  A role: the stage's byte count (tx; with CTA pairs, both CTAs' bytes, counted on
// the leader's barrier) and the A boxes; B role: the B boxes.  The B copies may complete
// on the barrier before the A thread's arrival: its transaction count then runs negative
// until the arrival, and the phase cannot complete before it.
template <int PAIR>
__device__ __forceinline__ void issue_kblock_copies(const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                                    int n_b, bool a_role, bool leader, uint32_t fb, uint32_t sA,
                                                    int k0, int m_me, int nb_me, int chunks, uint32_t tx) {
    const uint32_t sB = sA + p.a_bytes;
    const int bw = b_box_cols(p.BN, PAIR);
    // N-major B: box j is bw columns x bk rows at column nb + bw j, row k0.
    // K-major B: box j is bcols rows x 64 at row nb, column k0 + 64 j.
    const uint32_t box_bytes = p.b_kmajor ? p.b_atom_bytes : (uint32_t)p.bk * (uint32_t)bw * 2u;
    const int nbox = p.b_kmajor ? (chunks ? p.bk / kAtomK : 0) : chunks;
    // shared-memory slots of value box j and gate box j: N-major, the gate chunks follow
    // all value chunks at the same pitch; K-major, each 64-deep atom holds this CTA's
    // value rows, then its gate rows
    auto vslot = [&](int j) { return sB + box_bytes * (uint32_t)(p.b_kmajor ? n_b * j : j); };
    auto gslot = [&](int j) {
        return p.b_kmajor ? sB + box_bytes * (uint32_t)(2 * j + 1) : sB + p.b_bytes + box_bytes * (uint32_t)j;
    };
    auto bx = [&](int j) { return p.b_kmajor ? k0 + kAtomK * j : nb_me + bw * j; };
    auto by = [&](int j, int row0) { return p.b_kmajor ? row0 + nb_me : k0; };
    auto gx = [&](int j) { return p.b_kmajor ? k0 + kAtomK * j : p.gate_col + nb_me + bw * j; };
    if constexpr (PAIR == 2) {
        const uint32_t fb_leader = mapa_rank(fb, 0);
        if (a_role) {
            if (leader) mbar_arrive_expect_tx(fb, tx);
            if (m_me < p.M)
                for (int a = 0; a < p.bk / kAtomK; ++a)
                    tma_load_2d_pair(sA + 16384u * a, &tmA, fb_leader, k0 + kAtomK * a, m_me);
        } else {
            for (int j = 0; j < nbox; ++j) tma_load_2d_pair(vslot(j), &tmB, fb_leader, bx(j), by(j, 0));
            if (n_b == 2)
                for (int j = 0; j < nbox; ++j) tma_load_2d_pair(gslot(j), &tmB, fb_leader, gx(j), by(j, p.gate_col));
        }
    } else {
        if (a_role) {
            mbar_arrive_expect_tx(fb, tx);
            if (m_me < p.M)
                for (int a = 0; a < p.bk / kAtomK; ++a) tma_load_2d(sA + 16384u * a, &tmA, fb, k0 + kAtomK * a, m_me);
        } else {
            for (int j = 0; j < nbox; ++j) tma_load_2d(vslot(j), &tmB, fb, bx(j), by(j, 0));
            if (n_b == 2)
                for (int j = 0; j < nbox; ++j) tma_load_2d(gslot(j), &tmB, fb, gx(j), by(j, p.gate_col));
        }
    }
}

// PAIR = 1: one CTA per 128 x BN tile (cta_group::1).  PAIR = 2: a cluster pair per
// 256 x BN tile (cta_group::2): each CTA loads its 128 rows of A and half of the B
// columns; the even CTA (the leader) issues the MMAs, which write each CTA's 128
// rows of the accumulator into that CTA's tensor memory; each CTA's epilogue stores
// its own rows.
template <int EPI, int DT, int PAIR, bool TWO>
__global__ void __launch_bounds__((3 + epi_warps(EPI)) * 32, 1)
    kt_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmParams p,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC2, const __grid_constant__ GemmParams p2) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle tiles want 1024-byte alignment
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t tiles_bytes = (uint32_t)p.stages * p.stage_bytes;
    constexpr int EPI_UP = EPI;            // the up projection's epilogue (epi_item's EPI is per item)
    constexpr int NEPI = epi_warps(EPI);   // epilogue warps
    constexpr int NPART = NEPI / 4;        // epilogue warps per TMEM lane quadrant
    constexpr int kWarpB = 2 + NEPI;       // the B operand's producer (after the epilogue warps)
    // NEPI x 2 KB output staging buffers, twice over when the plan has room for a second set
    const uint32_t kStaging = (uint32_t)NEPI * 2048u * (p.dbl_staging ? 2u : 1u);
    const uint32_t staging = base + tiles_bytes;
    const uint32_t bar_full = staging + kStaging;
    const uint32_t bar_empty = bar_full + 8u * kMaxStages;
    const uint32_t bar_accf = bar_empty + 8u * kMaxStages;
    const uint32_t bar_acce = bar_accf + 16u;
    const uint32_t bar_stall = bar_acce + 16u;
    const uint32_t bar_drain = bar_stall + 8u;
    const uint32_t bar_pready = bar_drain + 8u;  // cluster split-K: every CTA's partials are written
    uint32_t* slots = reinterpret_cast<uint32_t*>(base_ptr + tiles_bytes + kStaging + 8u * (2 * kMaxStages + 8));
    // the epilogue's bias slices, two tiles deep: [2][value 256 | gate 256] in the I/O dtype
    const uint32_t bias_smem = staging + kStaging + kBarrierBytes;
    uint32_t* tmem_slot = slots;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slots + 1);
    volatile int* last_flag = reinterpret_cast<volatile int*>(slots + 2);
    // reduce-scatter split-K: the run's arrival target, shared by the epilogue warps
    volatile unsigned long long* rs_target = reinterpret_cast<volatile unsigned long long*>(slots + 4);
    // TWO (both projections in one launch): the work-item ring, kItemRing deep: item
    // indices and their full / empty barriers (in the barrier area, past the slots)
    const uint32_t item_idx = staging + kStaging + 256u;
    const uint32_t item_full = item_idx + 16u;
    const uint32_t item_empty = item_full + 8u * kItemRing;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned long long* const tr = p.trace;
    if (threadIdx.x == 0) trace_mark(tr, TR_ENTRY);
    const uint32_t rank = PAIR == 2 ? (cluster_ctarank() & 1u) : 0u;  // position in the CTA pair
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / PAIR;        // first tile of this CTA (or pair)
    const int unit_step = (int)gridDim.x / PAIR;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_accf + 8u * b, 1);
            mbar_init(bar_acce + 8u * b, NEPI * PAIR);  // both CTAs' epilogues (leader's copy)
        }
        mbar_init(bar_stall, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_pready, (uint32_t)(p.split_k * NEPI));
        if constexpr (TWO) {
            // consumers of an item: the MMA issuer, the B producer and the epilogue warps of
            // the leader CTA, and both producers and the epilogue warps of its peer
            for (int i = 0; i < kItemRing; ++i) {
                mbar_init(item_full + 8u * i, 1);
                mbar_init(item_empty + 8u * i, PAIR == 2 ? 4 + 2 * NEPI : 2 + NEPI);
            }
        }
        *abort_flag = 0;
        *last_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
        if constexpr (TWO) {
            prefetch_tmap(&tmA2);
            prefetch_tmap(&tmB2);
            prefetch_tmap(&tmC2);
        }
    }
    if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    if (PAIR == 2 || p.cluster_sk) cluster_sync_relaxed();  // peers' barriers initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) trace_mark(tr, TR_SETUP);

    // Programmatic dependent launch: let the next kernel in the stream get its CTAs
    // resident (and through their set-up) as SMs free up; every kernel here waits for
    // its predecessor's completion before its first global-memory access.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // With row-block readiness counters (down projection after the up projection), only
    // the epilogue waits for the predecessor grid to complete (before it reads the bias
    // or the residual and writes Y); the A producer waits on the counters of the rows of H
    // it reads, the B producer reads only the weights, and the MMA warp touches no global
    // memory.
    const bool ready_mode = EPI == EPI_DOWN && p.ready != nullptr;
    if (p.pdl_wait && (!ready_mode || (warp >= 2 && warp < kWarpB))) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) trace_mark(tr, TR_PDL);

    const int n_b = (EPI == EPI_GEGLU) ? 2 : 1;

    // Work items.  One projection: tiles unit0, unit0 + unit_step, ... (static).  TWO: items
    // 0 .. p.num_tiles - 1 are up-projection tiles, the next p2.num_tiles down-projection
    // items (tiles, or K splits of tiles).  Unit u's first item is item u; the rest are
    // handed out dynamically: the leader CTA's producer takes the next index (unit_step +
    // a global counter) and publishes it in the item ring of both CTAs of the pair; every
    // role consumes the same sequence.  Indices go out in increasing order and up tiles
    // wait on nothing, so a down item waiting for its rows of H always waits on up tiles
    // held by units that run or will run once the SMs the previous kernel holds are free
    // (the grid fits the GPU); the split-K reduction waits on nothing: the last CTA to
    // finish a tile sums it.
    const int total = p.num_tiles + (TWO ? p2.num_tiles : 0);
    // While up tiles remain for every unit, the leader's producer takes each index one item
    // ahead (the counter's round trip then overlaps the previous item's loads); down tiles
    // are taken on demand, so that none waits on a unit still busy with an earlier tile.
    int next_idx = -1;
    // Item k >= 1 goes through ring slot (k - 1) % kItemRing; item 0 is unit0 for every
    // role and never enters the ring, so that no role waits for another before its first
    // item (at a kernel's start that wait would be the publisher's whole first code path).
    auto publish = [&](uint32_t k) -> int {  // leader CTA's producer, k >= 1
        const uint32_t r = k - 1u, slot = r % kItemRing, par = (r / kItemRing) & 1u;
        if (!wait_phase(item_empty + 8u * slot, par ^ 1u, abort_flag, p.error, DEV_TIMEOUT_PRODUCER,
                        p.wait_limit_ns))
            return INT_MAX;
        const int idx = next_idx >= 0 ? next_idx : unit_step + atomicAdd(p.sched, 1);
        next_idx = idx + 2 * unit_step < p.num_tiles ? unit_step + atomicAdd(p.sched, 1) : -1;
        // the pair's peer gets the index by an asynchronous store that completes on its slot's
        // full barrier, as copies do (no cluster-scope release-ordered arrival)
        if constexpr (PAIR == 2) post_index(mapa_rank(item_idx + 4u * slot, 1), mapa_rank(item_full + 8u * slot, 1), idx);
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(item_idx + 4u * slot), "r"(idx) : "memory");
        mbar_arrive(item_full + 8u * slot);
        return idx;
    };
    auto consume = [&](uint32_t k) -> int {  // one thread per consuming warp, k >= 1
        const uint32_t r = k - 1u, slot = r % kItemRing, par = (r / kItemRing) & 1u;
        if (!wait_phase<PAIR == 2>(item_full + 8u * slot, par, abort_flag, p.error, DEV_TIMEOUT_EPILOGUE,
                                   p.wait_limit_ns))
            return INT_MAX;
        // the slot is free for the publisher's next index once this read is done: the
        // acquire orders the arrival after it, so the arrival itself need not release
        int idx;
        asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(idx) : "r"(item_idx + 4u * slot) : "memory");
        if constexpr (PAIR == 2) mbar_arrive_cluster_relaxed(mapa_rank(item_empty + 8u * slot, 0));
        else mbar_arrive_relaxed(item_empty + 8u * slot);
        return idx;
    };
    // item k for a role: the static first item, else the ring's
    auto item_of = [&](uint32_t k, bool publisher) -> int {
        if (k == 0) {
            if (publisher)  // one index taken ahead while up tiles remain for every unit
                next_idx = unit0 + 2 * unit_step < p.num_tiles ? unit_step + atomicAdd(p.sched, 1) : -1;
            return unit0 < total ? unit0 : total;
        }
        return publisher ? publish(k) : consume(k);
    };

    if (warp == 0 || warp == kWarpB) {
        // ------------------------------ producers ------------------------------
        // Two threads in two warps fill the ring: warp 0 the A operand (X, or H with its
        // readiness waits) and the stage's byte count, warp kWarpB the B operand (weights),
        // which never waits for H and so runs ahead by up to the ring's depth.  One issuing
        // thread per stage takes in about half the bytes per second that two do.
        const bool a_role = warp == 0;
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0, armed_phase = 0;  // per-stage bits: loads issued / their phase
            if (a_role && p.inject_stall) {
                // failure injection: a barrier nobody arrives on, bounded wait
                wait_phase(bar_stall, 0, abort_flag, p.error, DEV_INJECTED_STALL, p.stall_limit_ns);
            }
            // one work item of one projection (p: its parameters, tmA / tmB: its operands);
            // its first `skip` k-blocks were issued already (the early copies below)
            auto produce = [&](const GemmParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, const int n_b,
                               const bool ready_mode, const int t, const int local, const int skip) -> bool {
                const TileCoord c = decode_tile(t, p);
                const int kb0 = c.kb0, kb1 = c.kb1;
                int m_me, nb_me, chunks;
                uint32_t tx = cta_share<PAIR>(p, c, rank, n_b, m_me, nb_me, chunks);
                if (PAIR == 2) {  // the leader's full barrier counts the bytes of both CTAs
                    int m_o, nb_o, ch_o;
                    tx += cta_share<PAIR>(p, c, rank ^ 1u, n_b, m_o, nb_o, ch_o);
                }
                if (a_role && ready_mode && m_me < p.M) {
                    // the up projection's row blocks that hold this CTA's 128 rows of H
                    const int r1 = min(m_me + kBM, p.M) - 1;
                    bool got = true;
                    for (int rb = m_me / p.ready_rows; rb <= r1 / p.ready_rows && got; ++rb) {
                        got = wait_counter(p.ready + rb, p.ready_target, abort_flag, p.error, p.wait_limit_ns);
                        // the last of this run's waits on the row block resets its counters
                        // for the next run (whose up projection starts only after this grid
                        // has completed): every launch parameter stays the same from run to
                        // run, so a captured CUDA graph can replay the pair of kernels
                        if (got && atomicAdd(p.ready_readers + rb, 1u) == p.ready_expect[rb] - 1u) {
                            atomicExch(p.ready + rb, 0u);
                            atomicExch(p.ready_readers + rb, 0u);
                        }
                    }
                    if (!got) return false;
                    asm volatile("fence.proxy.async.global;" ::: "memory");  // H was written by TMA stores
                    if (TWO && tr && local >= 0 && tr[(size_t)blockIdx.x * kTraceSlots + TR_T_DN_READY] == 0)
                        trace_mark(tr, TR_T_DN_READY);
                }
                bool ok = true;
                for (int kb = kb0 + skip; kb < kb1; ++kb) {
                    if (!wait_phase(bar_empty + 8u * stage, phase ^ 1u, abort_flag, p.error,
                                    DEV_TIMEOUT_PRODUCER, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (a_role && tr && armed == 0) trace_mark(tr, TR_FIRST_TMA);
                    if (a_role && tr && kb == kb0 && local == 1) trace_mark(tr, TR_S_LD0);
                    issue_kblock_copies<PAIR>(p, tmA, tmB, n_b, a_role, leader, bar_full + 8u * stage,
                                              base + stage * p.stage_bytes, kb * p.bk, m_me, nb_me, chunks, tx);
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == (uint32_t)p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return ok;
            };
            // Early copies: the first item of a unit is static (item unit0).  When it waits on
            // nothing (an up-projection tile, or a tile of a projection without readiness
            // counters), its first k-blocks go out here, one per stage of the fresh ring, before
            // the item ring and the general path: at a kernel's start every code region runs
            // for the first time and waits for its instruction fetch, and the general path's
            // regions (item ring, tile decode, ring waits) put ~1.5 us before the first copy.
            int pre = 0;  // k-blocks of the first item issued here
            const bool first_free = TWO ? unit0 < p.num_tiles : (unit0 < p.num_tiles && !ready_mode);
            if (first_free && !p.inject_stall) {
                const TileCoord c = decode_tile(unit0, p);
                int m_me, nb_me, chunks;
                uint32_t tx = cta_share<PAIR>(p, c, rank, n_b, m_me, nb_me, chunks);
                if (PAIR == 2) {
                    int m_o, nb_o, ch_o;
                    tx += cta_share<PAIR>(p, c, rank ^ 1u, n_b, m_o, nb_o, ch_o);
                }
                pre = min(p.stages, c.kb1 - c.kb0);
                if (a_role && tr) trace_mark(tr, TR_FIRST_TMA);
                for (int s = 0; s < pre; ++s)
                    issue_kblock_copies<PAIR>(p, tmA, tmB, n_b, a_role, leader, bar_full + 8u * s,
                                              base + (uint32_t)s * p.stage_bytes, (c.kb0 + s) * p.bk, m_me, nb_me,
                                              chunks, tx);
                armed = (pre >= 32 ? 0xffffffffu : (1u << pre) - 1u);
                stage = (uint32_t)(pre % p.stages);
                phase = pre == p.stages ? 1u : 0u;
            }
            if constexpr (TWO) {
                bool done = false;  // this unit took the end-of-work index
                for (uint32_t k = 0; !*abort_flag; ++k) {
                    const int idx = item_of(k, leader && a_role);
                    if (idx >= total) {
                        done = idx != INT_MAX;
                        break;
                    }
                    if (a_role && tr && idx == p.num_tiles + (int)blockIdx.x / PAIR) trace_mark(tr, TR_T_DN_TAKEN);
                    const bool ok = idx >= p.num_tiles
                                        ? produce(p2, tmA2, tmB2, 1, p2.ready != nullptr, idx - p.num_tiles, (int)k, 0)
                                        : produce(p, tmA, tmB, n_b, false, idx, (int)k, k == 0 ? pre : 0);
                    if (!ok) break;
                }
                if (done && leader && a_role) {
                    // the last unit to finish resets the counter for the next run
                    __threadfence();
                    if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x / PAIR - 1) {
                        __threadfence();
                        atomicExch(p.sched, 0);
                        atomicExch(p.sched + 1, 0);
                    }
                }
            } else {
                int local = 0;
                for (int t = unit0; t < p.num_tiles && !*abort_flag; t += unit_step, ++local)
                    if (!produce(p, tmA, tmB, n_b, ready_mode, t, local, local == 0 ? pre : 0)) break;
            }
            if (*abort_flag && leader && a_role) {
                // do not leave copies in flight into shared memory we are about to release
                // (the leader's full barriers count the peer's copies, and the B thread's, too)
                for (int s = 0; s < p.stages; ++s)
                    if (armed & (1u << s)) wait_drain(bar_full + 8u * s, (armed_phase >> s) & 1u, 100000000ull);
            }
            if (*abort_flag && !a_role) {
                // the B thread's copies of a stage the A thread never armed complete on no
                // phase: give them 100 us to land (a copy takes a few microseconds)
                const unsigned long long t0 = global_ns();
                while (global_ns() - t0 < 100000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0;
            bool issued_any = false;
            // one work item of one projection (p: its parameters)
            auto mma_item = [&](const GemmParams& p, const int n_b, const int t, const int local) -> bool {
                const TileCoord c = decode_tile(t, p);
                const uint32_t buf = p.acc_bufs == 2 ? (uint32_t)(local & 1) : 0u;
                const uint32_t use = p.acc_bufs == 2 ? (uint32_t)(local >> 1) : (uint32_t)local;
                if (!wait_phase(bar_acce + 8u * buf, (use & 1u) ^ 1u, abort_flag, p.error, DEV_TIMEOUT_MMA,
                                p.wait_limit_ns))
                    return false;
                tc_fence_after();
                if (tr && local == 1) trace_mark(tr, TR_S_MMA0);
                const uint32_t d = tmem_base + buf * (uint32_t)kAccSlot;
                const int kb0 = c.kb0, kb1 = c.kb1;
                // Descriptors of stage 0, computed once per tile: a stage's descriptors are
                // those of stage 0 with the start address moved by the stage offset (the
                // 14-bit address field cannot carry: shared addresses stay below 256 KB), and
                // the K steps only move it by constant offsets (issue_kblock), so that the
                // issuing thread does little work between two k-blocks.  128-byte swizzle,
                // 8-row groups 1 KB apart; N-major B in chunks of bw columns (the box width:
                // 64, 32 or 16), each row 2 bw bytes with a swizzle of that span (128, 64 or
                // 32 bytes: descriptor modes 2, 4 and 6), chunks bk x 2 bw bytes apart, 8-row
                // groups 16 bw bytes apart.  GEGLU: the gate chunks follow the value chunks
                // (N-major: at the same chunk pitch; K-major: inside every 64-deep atom), one
                // operand of 2 BN.
                const uint32_t brow = 2u * (uint32_t)b_box_cols(p.BN, PAIR);  // bytes per N-major B row
                const uint32_t b_lbo = p.b_kmajor ? 16u : (uint32_t)p.bk * brow;
                const uint32_t b_sbo = p.b_kmajor ? 1024u : 8u * brow;
                const uint32_t b_swz = p.b_kmajor || brow == 128u ? 2u : brow == 64u ? 4u : 6u;
                const uint64_t ad_s0 = smem_desc(base, 16u, 1024u);
                const uint64_t bd_s0 = smem_desc(base + p.a_bytes, b_lbo, b_sbo, b_swz);
                const uint32_t stage16 = p.stage_bytes >> 4;
                const uint32_t b_step16 = brow;  // 16 rows of brow bytes, in 16-byte units
                const uint32_t batom16 = (p.b_atom_bytes * (uint32_t)n_b) >> 4;
                const int variant = (p.b_kmajor ? 2 : 0) + (p.bk == 64 ? 0 : 1);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t fb = bar_full + 8u * stage;
                    if (!mbar_test_wait(fb, phase) &&
                        !wait_phase(fb, phase, abort_flag, p.error, DEV_TIMEOUT_MMA, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (tr && !issued_any) trace_mark(tr, TR_FIRST_FULL);
                    const uint64_t soff = (uint64_t)(stage * stage16);
                    const uint64_t ad0 = ad_s0 + soff, bd0 = bd_s0 + soff;
                    const uint32_t acc0 = kb > kb0 ? 1u : 0u;
                    switch (variant) {
                        case 0: issue_kblock<PAIR, 4, 0>(d, ad0, bd0, p.idesc, acc0, 0u, b_step16); break;
                        case 1: issue_kblock<PAIR, 8, 0>(d, ad0, bd0, p.idesc, acc0, 0u, b_step16); break;
                        case 2: issue_kblock<PAIR, 4, 1>(d, ad0, bd0, p.idesc, acc0, batom16); break;
                        default: issue_kblock<PAIR, 8, 1>(d, ad0, bd0, p.idesc, acc0, batom16); break;
                    }
                    issued_any = true;
                    // stage free (in both CTAs of a pair) once these MMAs completed
                    if constexpr (PAIR == 2) mma_commit_pair(bar_empty + 8u * stage);
                    else mma_commit(bar_empty + 8u * stage);
                    if (++stage == (uint32_t)p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) return false;
                // accumulator ready for the epilogue (of both CTAs of a pair)
                if constexpr (PAIR == 2) mma_commit_pair(bar_accf + 8u * buf);
                else mma_commit(bar_accf + 8u * buf);
                if (tr) {
                    if (local == 0) trace_mark(tr, TR_MAIN_DONE);
                    if (local == 1) trace_mark(tr, TR_S_MMA1);
                    trace_mark(tr, TR_LAST_MAIN);
                    tr[(size_t)blockIdx.x * kTraceSlots + TR_TILES] = (unsigned long long)(local + 1);
                }
                return true;
            };
            if constexpr (TWO) {
                unsigned long long n_up = 0, n_dn = 0;
                for (uint32_t k = 0;; ++k) {
                    const int idx = item_of(k, false);
                    if (idx >= total) break;
                    const bool dn = idx >= p.num_tiles;
                    const bool ok = dn ? mma_item(p2, 1, idx - p.num_tiles, (int)k) : mma_item(p, n_b, idx, (int)k);
                    if (!ok) break;
                    if (tr) {
                        if (dn) ++n_dn;
                        else {
                            ++n_up;
                            trace_mark(tr, TR_T_LAST_UP);
                        }
                        tr[(size_t)blockIdx.x * kTraceSlots + TR_T_UP_ITEMS] = n_up;
                        tr[(size_t)blockIdx.x * kTraceSlots + TR_T_DN_ITEMS] = n_dn;
                    }
                }
            } else {
                int local = 0;
                for (int t = unit0; t < p.num_tiles; t += unit_step, ++local)
                    if (!mma_item(p, n_b, t, local)) break;
            }
            if (*abort_flag && issued_any) {
                if constexpr (PAIR == 2) mma_commit_pair(bar_drain);
                else mma_commit(bar_drain);
                wait_drain(bar_drain, 0u, 100000000ull);
            }
        }
    } else if (warp < 2 + NEPI) {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;
        const int q = warp & 3;    // TMEM lane quadrant this warp may access
        const int half = ew >> 2;  // which of the NPART interleaved 32-column groups
        const int row = q * 32 + lane;
        const uint32_t stg0 = staging + (uint32_t)ew * 2048u;
        const uint32_t stg_alt = (uint32_t)NEPI * 2048u;  // offset of the second buffer set
        const bool dbl = p.dbl_staging != 0;
        uint32_t nstores = 0;  // this warp's stores so far: picks the buffer
        // Up projection: this CTA's rows of a stored tile are counted for the down
        // projection's producer once every epilogue warp's TMA stores of the tile have
        // completed.  The count of tile i is raised after tile i + 1's accumulator wait
        // (or after the last tile), when those stores have long completed, so that the
        // wait for their completion is off the epilogue's path.
        int pending_rows = -1;
        auto signal_ready = [&](int tm) {
            if (lane == 0) {
                bulk_wait0();
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            __syncwarp();
            epi_bar_sync<NEPI>();  // every epilogue warp's stores of the tile completed
            if (ew == 0 && lane == 0) {
                __threadfence();
                atomicAdd(p.ready + tm, 1u);
            }
        };
        // One work item of one projection: `kind` carries its epilogue (the up projection's
        // activation or EPI_DOWN), p its parameters, tmC its output store map.  Returns false
        // when the kernel aborts (uniformly across the epilogue warps).
        auto epi_item = [&](auto kind, const GemmParams& p, const CUtensorMap& tmC, const int t,
                            const int local) -> bool {
            constexpr int EPI = decltype(kind)::value;
            const int n_b = (EPI == EPI_GEGLU) ? 2 : 1;
            const int ngroups = p.BN / 32;
            const int tiles_mn = p.tiles_m * p.tiles_n;
            const size_t tile_elems = (size_t)kBM * (size_t)p.BN;
            const TileCoord c = decode_tile(t, p);
            const uint32_t buf = p.acc_bufs == 2 ? (uint32_t)(local & 1) : 0u;
            const uint32_t use = p.acc_bufs == 2 ? (uint32_t)(local >> 1) : (uint32_t)local;
            // the accumulator-empty barrier lives in the leader CTA
            const uint32_t acce = PAIR == 2 ? mapa_rank(bar_acce + 8u * buf, 0) : bar_acce + 8u * buf;
            // Stage this tile's bias slice (value and, for GEGLU, gate columns) in shared
            // memory while the MMAs run; the barrier after the accumulator wait publishes
            // it to every epilogue warp (two buffers: a warp can only reach tile + 2 after
            // every warp has finished tile).
            // Staged in fp32 (1 KB per tile: up to 256 columns, or GEGLU's 128 value
            // columns at +0 and 128 gate columns at +512 bytes).
            const uint32_t bsm = bias_smem + (uint32_t)(local & 1) * 1024u;
            if (p.bias) {
                const int per = p.BN / 8;  // 8-column chunks per operand
                const int nb0 = c.tn * p.BN;
                for (int i = ew * 32 + lane; i < n_b * per; i += NEPI * 32) {
                    const int op = i >= per ? 1 : 0;
                    const int col = nb0 + 8 * (i - op * per);
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (col < p.N)
                        v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.bias) +
                                                                 (op ? p.gate_col : 0) + col));
                    float f[8];
                    unpack8<DT>(v, f);
                    const uint32_t dst = bsm + (uint32_t)op * 512u + (uint32_t)(i - op * per) * 32u;
                    st_shared_v4(dst, __float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                                 __float_as_uint(f[3]));
                    st_shared_v4(dst + 16u, __float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                                 __float_as_uint(f[7]));
                }
            }
            const bool got = wait_phase(bar_accf + 8u * buf, use & 1u, abort_flag, p.error,
                                        DEV_TIMEOUT_EPILOGUE, p.wait_limit_ns);
            if (!epi_all<NEPI>(got)) return false;
            tc_fence_after();
            const bool tr1 = tr && local == 1 && warp == 2 && lane == 0;  // steady-state marks
            if (tr1) trace_mark(tr, TR_S_ACC);
            if (EPI != EPI_DOWN && pending_rows >= 0) {  // the previous tile's rows (see above)
                signal_ready(pending_rows);
                pending_rows = -1;
            }
            if (tr1) trace_mark(tr, TR_S_SIG);
            int gi = 0;  // this warp's column groups of the tile so far (trace marks)
            const bool tr0 = tr && local == 0 && warp == 2 && lane == 0;
            if (tr0) trace_mark(tr, TR_EPI_START);
            const int m0 = c.tm * (kBM * PAIR) + (int)rank * kBM;  // this CTA's first row
            const int y0 = m0 + q * 32;              // first row of this warp's block
            const bool rows_live = y0 < p.M;         // warp-uniform
            const int n0 = c.tn * p.BN;
            const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + buf * (uint32_t)kAccSlot;

            if (EPI != EPI_DOWN || p.split_k == 1) {
                for (int g = half; g < ngroups; g += NPART) {
                    const int col = n0 + 32 * g;
                    const bool mark = tr0 && g == half;
                    if constexpr (EPI == EPI_GEGLU) {
                        // Accumulator columns: PAIR runs of [value share | gate share], one
                        // per CTA's B share (share = BN / PAIR columns of H).  In two halves
                        // of 16 columns: value, gate and bias of one half live at a time,
                        // which leaves registers for more independent GELU chains.
                        const uint32_t share = p.geglu_share;
                        const uint32_t c32 = 32u * (uint32_t)g;
                        const uint32_t vcol = (c32 / share) * 2u * share + c32 % share;
                        if (col < p.N && rows_live) {
                            uint32_t w[16];  // the group's 32 results, rounded and packed in pairs
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t rv[16], rg[16];
                                tmem_ld16(tq + vcol + 16u * h, rv);
                                tmem_ld16(tq + vcol + share + 16u * h, rg);
                                tmem_wait_ld2(rv, rg);
                                if (mark && h == 0) trace_mark(tr, TR_EPI_LD);
                                float bv[16], bg[16];
                                if (p.bias) {
                                    const uint32_t o = 128u * (uint32_t)g + 64u * (uint32_t)h;
                                    bias_from_smem<16>(bsm + o, bv);
                                    bias_from_smem<16>(bsm + 512u + o, bg);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) bv[i] = bg[i] = 0.0f;
                                }
#pragma unroll
                                for (int i = 0; i < 16; i += 2) {
                                    float y0v, y1v;
                                    f2_split(geglu_f2<true>(f2(__uint_as_float(rv[i]), __uint_as_float(rv[i + 1])),
                                                      f2(bv[i], bv[i + 1]),
                                                      f2(__uint_as_float(rg[i]), __uint_as_float(rg[i + 1])),
                                                      f2(bg[i], bg[i + 1])),
                                             y0v, y1v);
                                    w[8 * h + i / 2] = pack2<DT>(y0v, y1v);
                                }
                            }
                            if (mark) trace_mark(tr, TR_EPI_MATH);
                            if (tr1 && gi < 2) trace_mark(tr, gi == 0 ? TR_S_G0M : TR_S_G1M);
                            stage_and_store_packed(&tmC, stg0 + (dbl && (nstores++ & 1u) ? stg_alt : 0u), lane, w, col,
                                                   y0, dbl);
                            if (mark) trace_mark(tr, TR_EPI_STORE);
                            if (tr1 && gi < 2) trace_mark(tr, gi == 0 ? TR_S_G0S : TR_S_G1S);
                            ++gi;
                        }
                    } else {
                        if (col < p.N && rows_live) {
                            uint32_t r[32];
                            tmem_ld32(tq + 32u * g, r);
                            tmem_wait_ld_only();
                            reg_fence32(r);
                            if (mark) trace_mark(tr, TR_EPI_LD);
                            uint32_t w[16];  // the group's 32 results, rounded and packed in pairs
#pragma unroll
                            for (int h = 0; h < 2; ++h) {  // in 16-column slices
                                float v[16];
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[16 * h + i]);
                                const bool has_bias = p.bias != nullptr;
                                float b[16];
                                if (has_bias) bias_from_smem<16>(bsm + 128u * (uint32_t)g + 64u * (uint32_t)h, b);
#pragma unroll
                                for (int i = 0; i < 16; i += 2) {
                                    f32x2 z = f2(v[i], v[i + 1]);
                                    if (has_bias) z = f2_add<true>(z, f2(b[i], b[i + 1]));
                                    f2_split(act_f2<EPI, true>(z), v[i], v[i + 1]);
                                }
                                if constexpr (EPI == EPI_DOWN)
                                    if (p.residual)
                                        add_residual32<DT, 16>(p.residual, y0 + lane, p.M, col + 16 * h, p.N, v);
#pragma unroll
                                for (int i = 0; i < 8; ++i) w[8 * h + i] = pack2<DT>(v[2 * i], v[2 * i + 1]);
                            }
                            if (mark) trace_mark(tr, TR_EPI_MATH);
                            if (tr1 && gi < 2) trace_mark(tr, gi == 0 ? TR_S_G0M : TR_S_G1M);
                            stage_and_store_packed(&tmC, stg0 + (dbl && (nstores++ & 1u) ? stg_alt : 0u), lane, w, col,
                                                   y0, dbl);
                            if (mark) trace_mark(tr, TR_EPI_STORE);
                            if (tr1 && gi < 2) trace_mark(tr, gi == 0 ? TR_S_G0S : TR_S_G1S);
                            ++gi;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR == 2) mbar_arrive_cluster_relaxed(acce);
                    else mbar_arrive_relaxed(acce);
                }
                if (tr1) trace_mark(tr, TR_S_ARR);
                if (EPI != EPI_DOWN && p.ready != nullptr) pending_rows = c.tm;  // counted later
            } else if constexpr (EPI == EPI_DOWN) {
              if (!TWO && p.cluster_sk) {  // (one launch for both projections: never a cluster)
                // split-K inside a cluster, reduce-scattered through L2: each 32 x 32 unit of
                // the tile (row block q, column group g, u = q * ngroups + g) is owned by CTA
                // u % SK of the cluster, and a unit is handled by the same warp in every CTA.
                // Each CTA writes its fp32 partial of every unit it does not own to global
                // scratch ([tile][unit][sender][16-byte chunk][row][4 floats]: 512 contiguous
                // bytes per warp access), the cluster's epilogue warps signal one another on
                // an mbarrier in every CTA (release / acquire at cluster scope), and each owner
                // warp sums its units' SK partials (its own from tensor memory) in split
                // order (deterministic) and stores them.
                const uint32_t crank = (uint32_t)c.split;
                float4* part = reinterpret_cast<float4*>(p.partials) + (size_t)c.mn * (size_t)(4 * ngroups) *
                                                                           (size_t)p.split_k * 256u;
                // (the partials go out as 4 KB bulk copies from the idle stage ring: the copy
                // engine stores faster than per-thread stores do)
                for (int g = half; g < ngroups; g += NPART) {
                    const int u = q * ngroups + g;
                    if ((uint32_t)(u % p.split_k) == crank) continue;
                    uint32_t r[32];
                    tmem_ld32(tq + 32u * g, r);
                    tmem_wait_ld_only();
                    reg_fence32(r);
                    const uint32_t slot = base + (uint32_t)u * 4096u;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        st_shared_v4(slot + 512u * i + 16u * (uint32_t)lane, r[4 * i], r[4 * i + 1], r[4 * i + 2],
                                     r[4 * i + 3]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) bulk_store(part + ((size_t)u * p.split_k + crank) * 256u, slot, 4096u);
                }
                __syncwarp();
                if (lane == 0) {
                    bulk_commit();
                    bulk_wait0();  // the partials are in global memory
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    asm volatile("fence.acq_rel.cluster;" ::: "memory");
                    for (int s = 0; s < p.split_k; ++s) mbar_arrive_cluster(mapa_rank(bar_pready, (uint32_t)s));
                }
                if (tr0) trace_mark(tr, TR_EPI_LD);  // (cluster split-K: partials written)
                const bool ready = wait_phase<true>(bar_pready, 0u, abort_flag, p.error, DEV_TIMEOUT_EPILOGUE,
                                                    p.wait_limit_ns);
                if (tr0) trace_mark(tr, TR_EPI_MATH);  // (cluster split-K: every partial written)
                if (ready) {
                    for (int g = half; g < ngroups; g += NPART) {
                        const int u = q * ngroups + g;
                        if ((uint32_t)(u % p.split_k) != crank) continue;
                        const int col = n0 + 32 * g;
                        if (col >= p.N || !rows_live) continue;  // warp-uniform
                        const float4* src = part + (size_t)u * p.split_k * 256u + lane;
                        uint32_t w[16];  // the unit's 32 results, rounded and packed in pairs
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // in 16-column slices
                            float v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                            for (int sp = 0; sp < p.split_k; ++sp) {  // split order: deterministic
                                if ((uint32_t)sp == crank) {
                                    float a[16];
                                    tmem_f16cols(tq + 32u * g + 16u * h, a);
#pragma unroll
                                    for (int i = 0; i < 16; ++i) v[i] += a[i];
                                    continue;
                                }
                                float4 x[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) x[i] = __ldcg(src + (size_t)sp * 256u + 32 * (4 * h + i));
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    v[4 * i] += x[i].x;
                                    v[4 * i + 1] += x[i].y;
                                    v[4 * i + 2] += x[i].z;
                                    v[4 * i + 3] += x[i].w;
                                }
                            }
                            if (p.bias) {
                                float b[16];
                                bias_from_smem<16>(bsm + 128u * (uint32_t)g + 64u * (uint32_t)h, b);
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] += b[i];
                            }
                            if (p.residual) add_residual32<DT, 16>(p.residual, y0 + lane, p.M, col + 16 * h, p.N, v);
#pragma unroll
                            for (int i = 0; i < 8; ++i) w[8 * h + i] = pack2<DT>(v[2 * i], v[2 * i + 1]);
                        }
                        stage_and_store_packed(&tmC, stg0 + (dbl && (nstores++ & 1u) ? stg_alt : 0u), lane, w, col, y0,
                                               dbl);
                    }
                }
                if (tr0) trace_mark(tr, TR_EPI_STORE);  // (cluster split-K: my units stored)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(acce);
            } else if (TWO && EPI_UP != EPI_GEGLU && p.rs_sk) {
                // (not compiled into the GEGLU kernels, whose epilogue leaves no registers for
                // it: their one-launch splits are summed by the last CTA to arrive, below)
                // split-K reduce-scatter through global memory (both projections in one launch):
                // each 32 x 32 unit of this CTA's 128-row half of the tile (row block q, column
                // group g, u = q * ngroups + g) is owned by split (g / NPART + q + half) % SK: the
                // groups one warp handles (g = half, half + NPART, ...) go to different splits, so
                // that no warp sums more units than the others (up to SK groups per warp).  Every split writes its
                // fp32 partial of each unit it does not own to global scratch ([half tile][unit]
                // [sending split][16-byte chunk][row][4 floats]: 512 contiguous bytes per warp
                // access), counts itself on the half tile's 64-bit arrival counter (release),
                // waits for all SK arrivals of its run (acquire), then sums its own units' SK
                // partials (its own still in tensor memory) in split order (deterministic) and
                // stores them.  The counter only grows, by SK per run: the value an arrival
                // returns tells its run (old / SK), so nothing resets it (a reset would put
                // atomic round trips on every CTA's path to its exit), and at 64 bits it never
                // wraps.  The splits of a tile are adjacent work items taken in increasing
                // order, so every split a CTA waits for is held by a running unit or is the
                // next item to be taken.
                const int SK = p.split_k;
                const uint32_t mine = (uint32_t)c.split;
                const size_t half_tile = (size_t)c.mn * PAIR + rank;
                auto rs_owner = [&](int g) { return (uint32_t)((g / NPART + q + half) % SK); };
                float4* part = reinterpret_cast<float4*>(p.partials) + half_tile * (size_t)(4 * ngroups) * SK * 256u;
                for (int g = half; g < ngroups; g += NPART) {
                    const int u = q * ngroups + g;
                    if (rs_owner(g) == mine || n0 + 32 * g >= p.N || !rows_live) continue;  // warp-uniform
                    uint32_t r[32];
                    tmem_ld32(tq + 32u * g, r);
                    tmem_wait_ld_only();
                    reg_fence32(r);
                    float4* dst = part + ((size_t)u * SK + mine) * 256u + lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        __stcg(dst + 32 * i, make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                         __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
                }
                if (tr1) trace_mark(tr, TR_S_G0M);  // (reduce-scatter: this warp's partials issued)
                // the barrier orders every epilogue thread's partial stores before the one
                // gpu-scope release (fences are cumulative); the arrival's return value, the
                // run's target, goes to every epilogue warp through shared memory
                unsigned long long* arrivals = reinterpret_cast<unsigned long long*>(p.counters) + half_tile;
                epi_bar_sync<NEPI>();
                if (ew == 0 && lane == 0) {
                    __threadfence();
                    const unsigned long long old = atomicAdd(arrivals, 1ull);
                    rs_target[0] = (old / (unsigned long long)SK + 1ull) * (unsigned long long)SK;
                }
                epi_bar_sync<NEPI>();
                if (tr1) trace_mark(tr, TR_S_G0S);  // (reduce-scatter: arrival counted)
                if (tr0) trace_mark(tr, TR_EPI_LD);  // (reduce-scatter: partials written)
                bool got = true;
                // one poller per CTA (the barrier below hands its outcome to every warp)
                if (ew == 0 && lane == 0) got = wait_counter64(arrivals, rs_target[0], abort_flag, p.error, p.wait_limit_ns);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!epi_all<NEPI>(got)) return false;
                if (tr && local == 1 && lane == 0) trace_max(tr, TR_S_G1M);  // (every split arrived: latest warp)
                if (tr0) trace_mark(tr, TR_EPI_MATH);  // (reduce-scatter: every split's partials written)
                for (int g = half; g < ngroups; g += NPART) {
                    const int u = q * ngroups + g;
                    const int col = n0 + 32 * g;
                    if (rs_owner(g) != mine || col >= p.N || !rows_live) continue;  // warp-uniform
                    const float4* src = part + (size_t)u * SK * 256u + lane;
                    // this split's own partial of the unit, from tensor memory, first: no
                    // tensor-memory access (an ordering point for the compiler) sits between
                    // the other splits' loads below, so they can all be in flight together
                    uint32_t own[32];
                    tmem_ld32(tq + 32u * g, own);
                    tmem_wait_ld_only();
                    reg_fence32(own);
                    uint32_t w[16];  // the unit's 32 results, rounded and packed in pairs
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // in 16-column slices
                        float v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {  // in 8-column eighths of the unit
                            // every other split's 8 columns of this row (the k-th other split
                            // is k + (k >= mine), so the array index stays a compile-time
                            // constant and x lives in registers), then the sum in split order
                            float4 x[kRsMaxSplit - 1][2];
#pragma unroll
                            for (int k = 0; k < kRsMaxSplit - 1; ++k) {
                                if (k >= SK - 1) continue;
                                const int sp = k + (k >= (int)mine ? 1 : 0);
#pragma unroll
                                for (int i = 0; i < 2; ++i)
                                    x[k][i] = __ldcg(src + (size_t)sp * 256u + 32 * (4 * h + 2 * e + i));
                            }
                            float* ve = v + 8 * e;
                            const uint32_t* oe = own + 16 * h + 8 * e;
                            auto add_own = [&]() {  // this split, at its place in split order
#pragma unroll
                                for (int i = 0; i < 8; ++i) ve[i] += __uint_as_float(oe[i]);
                            };
#pragma unroll
                            for (int k = 0; k < kRsMaxSplit - 1; ++k) {  // split order: deterministic
                                if (k >= SK - 1) continue;
                                if (k == (int)mine) add_own();  // this split comes before the k-th other one
#pragma unroll
                                for (int i = 0; i < 2; ++i) {
                                    ve[4 * i] += x[k][i].x;
                                    ve[4 * i + 1] += x[k][i].y;
                                    ve[4 * i + 2] += x[k][i].z;
                                    ve[4 * i + 3] += x[k][i].w;
                                }
                            }
                            if ((int)mine == SK - 1) add_own();  // the last split
                        }
                        if (p.bias) {
                            float b[16];
                            bias_from_smem<16>(bsm + 128u * (uint32_t)g + 64u * (uint32_t)h, b);
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] += b[i];
                        }
                        if (p.residual) add_residual32<DT, 16>(p.residual, y0 + lane, p.M, col + 16 * h, p.N, v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[8 * h + i] = pack2<DT>(v[2 * i], v[2 * i + 1]);
                    }
                    stage_and_store_packed(&tmC, stg0 + (dbl && (nstores++ & 1u) ? stg_alt : 0u), lane, w, col, y0,
                                           dbl);
                }
                if (tr0) trace_mark(tr, TR_EPI_STORE);  // (reduce-scatter: my units stored)
                // (reduce-scatter: owned units summed and their stores issued, the latest warp)
                if (tr && local == 1 && lane == 0) trace_max(tr, TR_S_G1S);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR == 2) mbar_arrive_cluster_relaxed(acce);
                    else mbar_arrive_relaxed(acce);
                }
                if (tr1) trace_mark(tr, TR_S_ARR);
                // rs_target is rewritten by the next split-K item only after every warp has
                // passed this item's barriers: the next item's first barrier orders it
            } else {
                // split-K: this split's fp32 partial in a private layout in which every
                // warp access is 512 contiguous bytes: [16-column chunk][quarter][row][4]
                const size_t half_tile = (size_t)c.mn * PAIR + rank;  // this CTA's 128-row half of the tile
                float4* part = reinterpret_cast<float4*>(
                    p.partials + (((size_t)c.split * tiles_mn) * PAIR + half_tile) * tile_elems);
                for (int g = half; g < ngroups; g += NPART) {
                    uint32_t r[32];
                    tmem_ld32(tq + 32u * g, r);
                    tmem_wait_ld_only();
                    reg_fence32(r);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float4* dst = part + (size_t)(2 * g + h) * 4 * kBM + row;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i * kBM] = make_float4(__uint_as_float(r[16 * h + 4 * i]), __uint_as_float(r[16 * h + 4 * i + 1]),
                                                 __uint_as_float(r[16 * h + 4 * i + 2]),
                                                 __uint_as_float(r[16 * h + 4 * i + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR == 2) mbar_arrive_cluster_relaxed(acce);
                    else mbar_arrive_relaxed(acce);
                }
                // the barrier orders every epilogue thread's partial stores before the
                // arrival thread's gpu-scope release (fences are cumulative)
                epi_bar_sync<NEPI>();
                if (ew == 0 && lane == 0) {
                    __threadfence();
                    const int prev = atomicAdd(p.counters + half_tile, 1);
                    const int last = (prev == p.split_k - 1);
                    if (last) {
                        atomicExch(p.counters + half_tile, 0);  // ready for the next run
                        __threadfence();                   // acquire the other splits' partials
                    }
                    *last_flag = last;
                }
                epi_bar_sync<NEPI>();
                if (*last_flag) {
                    for (int g = half; g < ngroups; g += NPART) {
                        const int col = n0 + 32 * g;
                        if (col >= p.N || !rows_live) continue;  // warp-uniform
                        uint32_t w[16];  // the group's 32 results, rounded and packed in pairs
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // 16 columns of this row from every split: up to 4 splits' loads in
                            // flight at once, summed in split order (deterministic)
                            float v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                            const size_t off = (size_t)(2 * g + h) * 4 * kBM + row;  // in float4
                            for (int s0 = 0; s0 < p.split_k; s0 += 4) {
                                float4 x[4][4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (s0 + j < p.split_k) {
                                        const float4* src = reinterpret_cast<const float4*>(
                                            p.partials + (((size_t)(s0 + j) * tiles_mn) * PAIR + half_tile) * tile_elems) + off;
#pragma unroll
                                        for (int i = 0; i < 4; ++i) x[j][i] = __ldcg(src + i * kBM);
                                    }
                                }
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (s0 + j < p.split_k) {
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            v[4 * i] += x[j][i].x;
                                            v[4 * i + 1] += x[j][i].y;
                                            v[4 * i + 2] += x[j][i].z;
                                            v[4 * i + 3] += x[j][i].w;
                                        }
                                    }
                                }
                            }
                            if (p.bias) {
                                float b[16];
                                bias_from_smem<16>(bsm + 128u * (uint32_t)g + 64u * (uint32_t)h, b);
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] += b[i];
                            }
                            if (p.residual) add_residual32<DT, 16>(p.residual, y0 + lane, p.M, col + 16 * h, p.N, v);
#pragma unroll
                            for (int i = 0; i < 8; ++i) w[8 * h + i] = pack2<DT>(v[2 * i], v[2 * i + 1]);
                        }
                        stage_and_store_packed(&tmC, stg0 + (dbl && (nstores++ & 1u) ? stg_alt : 0u), lane, w, col, y0,
                                               dbl);
                    }
                }
                epi_bar_sync<NEPI>();  // last_flag is rewritten for the next tile
              }
            }
            if (tr && warp == 2 && lane == 0) {
                if (local == 0) trace_mark(tr, TR_EPI_DONE);
                trace_mark(tr, TR_LAST_EPI);
            }
            return true;
        };
        if constexpr (TWO) {
            for (uint32_t k = 0;; ++k) {
                int idx = 0;
                if (lane == 0) idx = item_of(k, false);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                // every epilogue warp took the same item, unless the kernel is aborting
                if (!epi_all<NEPI>(idx < total)) break;
                const bool dn = idx >= p.num_tiles;
                if (dn && pending_rows >= 0) {  // before a down tile waits: its rows may be these
                    signal_ready(pending_rows);
                    pending_rows = -1;
                }
                const bool ok = dn ? epi_item(std::integral_constant<int, EPI_DOWN>{}, p2, tmC2, idx - p.num_tiles,
                                              (int)k)
                                   : epi_item(std::integral_constant<int, EPI>{}, p, tmC, idx, (int)k);
                if (!ok) break;
            }
        } else {
            int local = 0;
            for (int t = unit0; t < p.num_tiles; t += unit_step, ++local)
                if (!epi_item(std::integral_constant<int, EPI>{}, p, tmC, t, local)) break;
        }
        if (EPI != EPI_DOWN && pending_rows >= 0) signal_ready(pending_rows);  // the last up tile's rows
        // every TMA store of this warp has completed before the CTA may exit
        if (lane == 0) bulk_wait0();
        __syncwarp();
        if (tr && warp == 2 && lane == 0) trace_mark(tr, TR_EPI_DRAIN);
    }

    // ------------------------------ teardown ------------------------------
    tc_fence_before();
    __syncthreads();
    if (PAIR == 2 || p.cluster_sk) cluster_sync_all();  // no CTA leaves while a peer may still signal it
    if (threadIdx.x == 0 && tr) {
        trace_mark(tr, TR_EXIT);
        tr[(size_t)blockIdx.x * kTraceSlots + TR_SMID] = sm_id();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<PAIR>(tmem_base, kTmemCols);
    }
}

// Launch one instantiation (cluster and programmatic-dependent-launch attributes as
// the parameters ask).  TWO: both projections in one launch (tmA2 / tmB2 / tmC2 / p2: the
// down projection); otherwise the second set repeats the first and is not read.
template <int EPI, int DT, int PAIR, bool TWO>
kt_status launch_one(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC, const GemmParams& p,
                     const CUtensorMap* tmA2, const CUtensorMap* tmB2, const CUtensorMap* tmC2, const GemmParams& p2,
                     int grid, int smem, void* stream, bool pdl, const char** why) {
    auto kern = kt_gemm_kernel<EPI, DT, PAIR, TWO>;
    // opt in to the shared memory this launch needs (idempotent, cheap after the first call)
    static std::atomic<int> max_set[16];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 16 || max_set[dev].load(std::memory_order_relaxed) < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e != cudaSuccess) {
            *why = cudaGetErrorString(e);
            return KT_ERR_CUDA;
        }
        if (dev >= 0 && dev < 16) max_set[dev].store(kSmemBudget);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)((3 + epi_warps(EPI)) * 32), 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (PAIR == 2 || p.cluster_sk) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = PAIR == 2 ? 2 : (unsigned)p.split_k;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, *tmA, *tmB, *tmC, p, *tmA2, *tmB2, *tmC2, p2);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return KT_ERR_CUDA;
    }
    return KT_OK;
}

template <int EPI, int DT, int PAIR>
kt_status launch_one(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC, const GemmParams& p,
                     int grid, int smem, void* stream, bool pdl, const char** why) {
    return launch_one<EPI, DT, PAIR, false>(tmA, tmB, tmC, p, tmA, tmB, tmC, p, grid, smem, stream, pdl, why);
}

// Launch dispatch per group of epilogues (one translation unit each, compiled in parallel).
kt_status launch_gemm_act(int epi, int dtype, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                          const GemmParams& p, int grid, int smem, void* stream, bool pdl, const char** why);
kt_status launch_gemm_geglu(int dtype, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                            const GemmParams& p, int grid, int smem, void* stream, bool pdl, const char** why);
kt_status launch_gemm_down(int dtype, const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                           const GemmParams& p, int grid, int smem, void* stream, bool pdl, const char** why);
// Both projections in one launch (the up projection's epilogue `epi`; CTA pairs as up.pair);
// maps: the up projection's A, B and output maps, then the down projection's.
kt_status launch_mlp_two_act_f16(int epi, const CUtensorMap* const* maps, const GemmParams& up, const GemmParams& down,
                                 int grid, int smem, void* stream, bool pdl, const char** why);
kt_status launch_mlp_two_act_bf16(int epi, const CUtensorMap* const* maps, const GemmParams& up,
                                  const GemmParams& down, int grid, int smem, void* stream, bool pdl, const char** why);
kt_status launch_mlp_two_geglu(int dtype, const CUtensorMap* const* maps, const GemmParams& up, const GemmParams& down,
                               int grid, int smem, void* stream, bool pdl, const char** why);

}  // namespace kt
