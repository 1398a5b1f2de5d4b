// ptx.cuh -- inline-PTX wrappers used by the attention kernels (sm_103a).
//
// mbarrier (with bounded waits), TMA tensor loads, ldmatrix / movmatrix,
// warp-level mma.sync for the small-row decode kernel, and the tcgen05
// (TMEM / 5th-generation tensor core) instructions for the row-tile kernel.
// Every wait on a barrier gives up after a time limit and reports it through
// a device status word instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fmha {

// ---------------------------------------------------------------------------
// device status word (see status.cu); bit values
// ---------------------------------------------------------------------------
// The word is status[0]; status[1] holds the site code of the first failed
// index check of a checked build.
enum : unsigned {
    kStatusBarrierTimeout = 1u,   // a bounded mbarrier wait gave up
    kStatusBoundsViolation = 2u,  // checked build: an index check failed and its access was skipped
};

// ---------------------------------------------------------------------------
// checked builds
// ---------------------------------------------------------------------------
// A library compiled with -DFMHA_CHECKED tests, before the access, every
// computed shared-memory offset, tensor-memory column, global-memory index
// and TMA coordinate of the kernels against the extent of its buffer.  A
// failed check sets kStatusBoundsViolation, records its site code in
// status[1] (the first failure wins) and the access does not happen: a plain
// load or store is skipped, a warp-collective instruction (ldmatrix,
// tcgen05.ld/st) is pointed at offset 0 of its buffer instead.  A wrong index
// therefore shows up in fmha_check_device_status() and never as a fault; a
// skipped TMA load leaves its barrier short of bytes, so the consumer's
// bounded wait gives up as well.  In normal builds FMHA_IN_BOUNDS() is the
// constant true and its condition is not evaluated.
#ifdef FMHA_CHECKED
constexpr bool kCheckedBuild = true;
#else
constexpr bool kCheckedBuild = false;
#endif

// Site codes: 0x1nn row-tile kernel, 0x2nn hd-512 kernel, 0x3nn decode
// kernel, 0x4nn merge, 0x5nn shared epilogue / softmax helpers, 0x7nn
// two-row-tile kernel.
enum CheckSite : unsigned {
    kSiteTcQLoad = 0x101,   // Q box coordinates
    kSiteTcKLoad = 0x102,   // K tile: first key, stage offset
    kSiteTcVLoad = 0x103,   // V tile: first key, stage offset
    kSiteTcKDesc = 0x104,   // K stage the QK MMA reads
    kSiteTcVDesc = 0x105,   // V stage and P buffer the PV MMA reads
    kSiteTcSCol = 0x106,    // TMEM columns of the S buffer
    kSiteTcPRow = 0x107,    // row of the P buffer
    kSiteTcLse = 0x108,     // LSE / partial LSE index
    kSiteTcFp4 = 0x109,     // NVFP4 output row
    kSiteTcPTmem = 0x10a,   // TMEM columns of P (TS-form PV)
    kSiteWideItem = 0x201,  // ring slot and box coordinates of a producer item
    kSiteWideQ = 0x202,     // resident-Q box coordinates
    kSiteWideVSlots = 0x203,  // the V_ITEMS slots of a PV MMA are consecutive
    kSiteWideQKDesc = 0x204,  // Q and K slots the QK MMA reads
    kSiteWideSCol = 0x205,
    kSiteWidePRow = 0x206,
    kSiteWideLse = 0x207,
    kSiteWideRange = 0x208,  // range factor index of an fp16 partial
    kSiteWideFp4 = 0x209,    // NVFP4 output row
    kSiteDecQRow = 0x301,    // Q row loaded from global memory
    kSiteDecQSmem = 0x302,   // Q staging offset
    kSiteDecKVLoad = 0x303,  // K/V stage: first key, stage offset
    kSiteDecLdsmK = 0x304,   // ldmatrix address inside the K tile
    kSiteDecLdsmQ = 0x305,   // ldmatrix address inside the Q rows
    kSiteDecLdsmV = 0x306,   // ldmatrix address inside the V tile
    kSiteDecComb = 0x307,    // combine buffer index
    kSiteDecMl = 0x308,      // per-key-group (max, sum) index
    kSiteDecOut = 0x309,     // output / partial row (and NVFP4 output block)
    kSiteMergePart = 0x401,  // partial (split, row, column) index
    kSiteMergeRange = 0x402,
    kSiteMergeOut = 0x403,
    kSiteMergeSink = 0x404,
    kSiteMergeFp4 = 0x405,   // NVFP4 output block of the merge
    kSiteEpiRow = 0x501,     // staging row of the TMA-store epilogue
    kSiteEpiStore = 0x502,   // TMA store box coordinates
    kSiteSink = 0x503,       // sink logit head index
    kSiteSelfTest = 0x601,   // fmha_selftest_bounds_check (no access behind it)
    kSitePairQLoad = 0x701,  // Q box coordinates of either row tile
    kSitePairKLoad = 0x702,  // K tile: first key, stage offset
    kSitePairVLoad = 0x703,  // V tile: first key, stage offset
    kSitePairKDesc = 0x704,  // K stage the QK MMAs read
    kSitePairVDesc = 0x705,  // V stage the PV MMAs read
    kSitePairLse = 0x706,    // LSE / partial LSE index
    kSitePairFp4 = 0x707,    // NVFP4 output row
};

static __device__ __noinline__ bool bounds_failed(unsigned site, unsigned* status) {
    atomicOr(status, kStatusBoundsViolation);
    atomicCAS(status + 1, 0u, site);
    return false;
}

#define FMHA_IN_BOUNDS(cond, site, status) \
    (!::fmha::kCheckedBuild || (cond) || ::fmha::bounds_failed((site), (status)))

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// `limit_ns` nanoseconds: sets kStatusBarrierTimeout in *status and returns
// false.  The caller then stops its work (it must not touch the buffer the
// barrier guards).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* status,
                                          uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kStatusBarrierTimeout);
            return false;
        }
    }
}

// Exit drain of a producer thread.  `issued` loads went into a ring of `nslots`
// slots, load i into slot i % nslots, each completing one phase of full[slot].
// Waits (bounded, as mbar_wait) until the last load issued into every slot has
// landed -- slot s last received load s + ((issued - 1 - s) / nslots) * nslots,
// whose phase has that index / nslots -- so that no TMA write into this
// block's shared memory is still in flight when the block exits, whether or
// not a consumer gave up on its waits.  Nothing arms these barriers after
// the producer stops, so each waited-for phase is the barrier's latest.
__device__ __forceinline__ void drain_ring(uint64_t* full, int nslots, int issued, unsigned* status) {
    for (int s = 0; s < nslots && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / nslots) * nslots;
        mbar_wait(&full[s], (unsigned)(last / nslots) & 1u, status);
    }
}

// ---------------------------------------------------------------------------
// TMA (tensor) loads into shared memory, completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int c0, int c1, int c2,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const void* tmap, int c0, int c1, int c2,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// TMA store of one box from shared memory (bulk-group completion).  Elements
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int c0, int c1, int c2, const void* smem_src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(smem_src))
                 : "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed store has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// warp-level matrix helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Packed fp32 pairs (sm_100 and later): two lanes of fp32 arithmetic in one
// instruction, on a 64-bit register holding {lo, hi}.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The two bf16 halves of a packed pair, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t pk) { return __uint_as_float(pk << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pk) { return __uint_as_float(pk & 0xffff0000u); }

// 2^x with the hardware approximation (ex2.approx.ftz.f32: ~2 ulp, -inf -> 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// End of a row's online softmax: O = acc * inv and its natural-log LSE, from
// the running max m and the sum l relative to it (both log2 units; l = 0 for
// a row with no attended key).  sink_l2: the row's attention-sink logit in
// log2 units (-inf: none), one more term of the denominator only:
//   M = max(m, sink), l' = l 2^(m - M) + 2^(sink - M), inv = 2^(m - M) / l',
//   lse = (M + log2 l') ln 2.
// No attended key gives O = 0 and lse = sink (-inf without one).
//
// l_o: the divisor of O, when it differs from l.  A kernel that rounds P to
// bf16 before the P V product divides O by the sum of the ROUNDED values
// (the weights it actually multiplied V by), so that O is an exact convex
// combination of V rows whatever the rounding -- a dominant key's V row comes
// back unchanged -- while the LSE keeps the sum of the unrounded
// probabilities.  Both sums are relative to the same m.
__device__ __forceinline__ void finish_row(float m, float l, float l_o, float sink_l2, float& inv, float& lse) {
    constexpr float kLn2 = 0.693147180559945309f;
    if (!(l > 0.f) || !(l_o > 0.f)) {
        inv = 0.f;
        lse = sink_l2 * kLn2;
        return;
    }
    if (sink_l2 == -INFINITY) {
        inv = 1.f / l_o;
        lse = (m + log2f(l)) * kLn2;
        return;
    }
    const float M = fmaxf(m, sink_l2);
    const float c = exp2f(m - M);
    const float ls = exp2f(sink_l2 - M);
    inv = c / (l_o * c + ls);
    lse = (M + log2f(l * c + ls)) * kLn2;
}

__device__ __forceinline__ void finish_row(float m, float l, float sink_l2, float& inv, float& lse) {
    finish_row(m, l, l, sink_l2, inv, lse);
}

// Query head h's sink logit in log2 units.  The kernels take the sink as a
// compile-time option, so that without one none of this code exists.
__device__ __forceinline__ float sink_log2_of(const float* sink, int h, int n_h, unsigned* status) {
    if (!FMHA_IN_BOUNDS(h >= 0 && h < n_h, kSiteSink, status)) return -INFINITY;
    return __ldg(sink + h) * 1.4426950408889634f;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets a grid queued behind
// this one with the programmatic-serialization attribute start early; that
// grid's grid_dependency_wait returns once this grid has completed and its
// memory is visible.  Both are no-ops when no such pairing exists.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace fmha

// ---------------------------------------------------------------------------
// tcgen05: tensor memory (TMEM) and 5th-generation tensor-core MMA
// ---------------------------------------------------------------------------
namespace fmha {

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to *dst (shared memory).  Warp-collective: all 32 lanes execute it.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-collective; taddr must be the address tmem_alloc returned.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor-core operand reads, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), kind::f16 (bf16 inputs, fp32 accumulate).
// Issued by a single thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem desc), kind::f16: the "TS" form.  A is
// M x 16 bf16 held in tensor memory, row m in lane m, the 16 reduction-dim
// elements of the row packed two per 32-bit column over 8 consecutive
// columns starting at a_tmem (lane field 0).  A and B are both bf16.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05.mma this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape, x32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return __uint_as_float(r);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from raw words
// (packed bf16 pairs of P for the TS-form MMA).
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05.mma (128-byte swizzle).
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1)
//   bits 61-63 layout: 2 = 128-byte swizzle
// K-major operand: rows of 128 bytes (64 bf16 of the reduction dim), 8-row
//   atoms of 1024 bytes, SBO = distance between 8-row groups, LBO unused.
// MN-major operand: each reduction-dim row holds 64 contiguous M/N elements
//   (128 bytes); SBO = distance between groups of 8 reduction rows, LBO =
//   distance between 64-element M/N blocks.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | ((uint32_t)b_mn << 16)       // B major-ness
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

}  // namespace fmha
