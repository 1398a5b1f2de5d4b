// tc_pair_kernel.cu -- attention forward for two 128-row query tiles per
// thread block on the tcgen05 tensor cores (sm_103a), hd 64 and 128.
//
// When a KV head has more than 128 query rows (a GQA prefill: group x T >
// 128), one thread block takes two row tiles, A and B, of the same KV head and
// KV chunk.  Both use every K and V tile the block loads (128 keys each), and
// two softmax warpgroups, one per row tile, run side by side:
//   S_t(j)  = Q_t K_j^T                    per row tile t: M = 128 rows, N = 128 keys
//   O^T    += V_j^T [P_A(j); P_B(j)]^T     once for both tiles: M = hd (64 or
//                                          128), N = 256 rows, K = 128 keys
// The P V product runs transposed so that one MMA instruction covers both
// row tiles (N = 256): half the P V instructions, and so fewer operand reads
// of V and fewer points where the issuing thread must wait, in a kernel whose
// MMA operands, P writes and K/V loads keep shared memory busy.  A is V itself
// (MN-major, as it lies in memory), B is P (K-major, rows of 128 keys),
// written to shared memory by the softmax.  Tensor memory: S_A, S_B (128 columns each) and O^T (256
// columns = the two tiles' rows; head-dim index d in lane d at hd 128, and at
// hd 64, an M = 64 accumulator, in lane (d / 16) * 32 + d % 16: the first 16
// lanes of each 32-lane quarter, as measured on this GPU).
//
// The FA2 online softmax (commit e4ee9fd of the nvfp4-megamoe-kernel pages,
// multi-tile C API part), the lazy rescale and the bf16-rounded divisor are
// those of tc_kernel.cu; with O transposed, a rescale of row r scales column
// r of O^T, which all four warps of the row's tile take part in.
//
// Warp roles (10 warps):
//   warp 0      TMA producer: both Q tiles (once), then K_0 and, per KV tile
//               j, K_{j+1} and V_j through a ring of K/V tiles (three 32 KB
//               slots at hd 128, eight 16 KB slots at hd 64)
//   warp 1      TMEM owner and MMA issuer (one elected lane):
//               QK_A(0) QK_B(0) | QK_A(j+1) QK_B(j+1) PV(j) | ...
//   warps 2..5  softmax and epilogue of row tile A (one query row per thread;
//               warp w reaches TMEM lane quarter w % 4, so the four warps of a
//               tile cover quarters 2, 3, 0, 1)
//   warps 6..9  softmax and epilogue of row tile B
// A softmax warpgroup frees its S buffer as soon as it has loaded S_t(j), so
// QK_t(j+1) runs while it computes P_t(j); it writes P_t(j) once PV(j-1) has
// read the P buffer.  Both warpgroups run one copy of the softmax code (the
// row tile is a run-time value): with a copy per tile, the two interleaved
// copies of the unrolled loop ran the softmax at about half speed on this GPU
// (GQA prefill hd 128, s_k 4096: 110.7 us against 63.0 us).
//
// Measured on GB300 (GQA prefill b4 h64 kv8 T128 hd128 causal): s_k 4096 in
// 65 us (54-55 % of the bf16 peak) against 80.7 us for one row tile per block;
// s_k 32768 in 125.6 us (57 %) against 149.9 us.
#include <climits>
#include <atomic>
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fmha {
namespace {

template <int HD>
struct PCfg {
    static_assert(HD == 64 || HD == 128, "O^T is an M = hd accumulator");
    static constexpr int BM = 128;                  // query rows per row tile
    static constexpr int BN = 128;                  // keys per KV tile
    static constexpr int NB = HD / 64;              // 64-column (128-byte) boxes of Q, K, V
    static constexpr int Q_BYTES = BM * HD * 2;     // one row tile of Q
    static constexpr int P_BYTES = 2 * BM * BN * 2; // P of both tiles: BN / 64 groups of 256 rows x 128 bytes
    static constexpr int P_GROUP = 2 * BM * 128;    // one 64-key group of P
    static constexpr int KV_TILE = BN * HD * 2;     // one K or V tile
    static constexpr int NSLOT = HD == 64 ? 8 : 3;  // K/V ring slots
    static constexpr int THREADS = 320;
    static constexpr int OT_COL = 2 * BN;           // TMEM: S_A at 0, S_B at BN, O^T at 2 BN
    static constexpr int TMEM_COLS = 512;
    static constexpr int OFF_Q = 0;                 // Q_A, then Q_B
    static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_RING = OFF_P + P_BYTES;
    static constexpr int OFF_BAR = OFF_RING + NSLOT * KV_TILE;
    static constexpr int N_BARS = 1 + 2 * NSLOT + 2 + 2 + 1 + 2 + 1;
    static constexpr int OFF_ROWV = OFF_BAR + N_BARS * 8 + 16;  // after the TMEM address and abort flag
    static constexpr int SMEM = 1024 + OFF_ROWV + 2 * BM * 4;
    static_assert(OT_COL + 2 * BM <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(2 * Q_BYTES >= BM * HD * 4 && P_BYTES >= BM * HD * 4,
                  "epilogue staging: tile A in the Q tiles, tile B in the P buffer");
};

struct PairArgs {
    __nv_bfloat16* o;
    float* lse;
    float* lse_part;
    int to_partials;
    int n_h, n_kv_h, T, s_k, group, R, window, causal;
    float scale_log2;
    int kv_begin, kv_chunk;
    long long rows_total;
    unsigned* status;
    const float* sink;  // [n_h] sink logits (final output only) or NULL
};

__device__ __forceinline__ void pair_attended(int t, const PairArgs& a, int& lo, int& hi) {
    const int p = a.s_k - a.T + t;
    lo = 0;
    hi = a.s_k - 1;
    if (a.causal) hi = min(hi, p);
    if (a.window > 0) lo = max(lo, p - a.window + 1);
}

// OR of `pred` over the `nthreads` threads meeting at named barrier `id`.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Row `row` (0..255) of P (BN bf16 in packed pairs) into the K-major
// 128-byte-swizzled B-operand layout: BN / 64 groups of 256 rows x 128 bytes,
// 16-byte chunk c of row r at chunk c ^ (r % 8).
template <int BN>
__device__ __forceinline__ void write_p_row256(uint8_t* pbuf, int row, const uint32_t (&p)[BN / 2]) {
#pragma unroll
    for (int g = 0; g < BN / 64; ++g) {
        uint8_t* prow = pbuf + g * 256 * 128 + row * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const uint32_t* pv = p + g * 32 + ch * 4;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
        }
    }
}

template <int HD, int EPI>
__global__ void __launch_bounds__(PCfg<HD>::THREADS, 1)
    fwd_tc_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                       const PairArgs a) {
    using C = PCfg<HD>;
    constexpr int BM = C::BM, BN = C::BN, NSLOT = C::NSLOT;
    constexpr bool SINK = EPI == kEpiSink;
    launch_dependents();  // the merge grid may be scheduled now; it waits for this grid's results
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sq = smem + C::OFF_Q;
    uint8_t* sp = smem + C::OFF_P;
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* slot_full = bars + 1;
    uint64_t* slot_empty = slot_full + NSLOT;
    uint64_t* s_full = slot_empty + NSLOT;  // [2] by row tile: S_t(j) in TMEM
    uint64_t* s_free = s_full + 2;          // [2] by row tile: S_t(j) loaded by its softmax warps
    uint64_t* p_ready = s_free + 2;         // P_A(j) and P_B(j) in shared memory
    uint64_t* o_done = p_ready + 1;         // [2] by j & 1: PV(j) completed (O^T updated, its P buffer and V slot free)
    uint64_t* mma_drain = o_done + 2;       // every MMA the issuer launched has completed (exit drain)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::N_BARS);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    float* rowv = reinterpret_cast<float*>(smem + C::OFF_ROWV);  // [2][BM]: per-row alpha, then 1 / sum

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.y, slab = blockIdx.z;
    const int b = slab / a.n_kv_h, kvh = slab - b * a.n_kv_h;
    const long long row0 = ((long long)b * a.n_h + (long long)kvh * a.group) * a.T;  // slab's first query row
    const int rb = blockIdx.x * 2 * BM;        // first row of tile A
    const int re = min(a.R, rb + 2 * BM);      // one past the last row of tile B
    const int n_rt = (re - rb > BM) ? 2 : 1;   // row tiles with rows (tile B may lie past the slab's end)

    // KV range of this block: its chunk intersected with what its rows attend.
    const int c_lo = a.kv_begin + split * a.kv_chunk;
    const int c_hi = min(a.s_k, c_lo + a.kv_chunk);
    int u_lo, u_hi;
    {
        int t0, t1;
        if (re - rb >= a.T || (re - 1) % a.T < rb % a.T) {  // every t, or rows wrapping once past T-1
            t0 = 0;
            t1 = a.T - 1;
        } else {
            t0 = rb % a.T;
            t1 = (re - 1) % a.T;
        }
        int l0, h0, l1, h1;
        pair_attended(t0, a, l0, h0);
        pair_attended(t1, a, l1, h1);
        u_lo = l0;
        u_hi = h1;
    }
    const int k_lo = max(c_lo, u_lo), k_hi = min(c_hi, u_hi + 1);
    const int n_tiles = (k_hi > k_lo) ? (k_hi - k_lo + BN - 1) / BN : 0;

    // Ring items in the order the MMA issuer consumes them: K_0, then per KV
    // tile j: K_{j+1} (if any) and V_j.  Item i -> (is V, KV tile).
    const int n_items = 2 * n_tiles;
    uint64_t pol = 0;
    auto issue_item = [&](int i) -> bool {
        bool is_v;
        int tile;
        if (i == 0) {
            is_v = false;
            tile = 0;
        } else {
            const int r = i - 1;
            if (r / 2 < n_tiles - 1) {
                is_v = (r & 1) != 0;
                tile = is_v ? r / 2 : r / 2 + 1;
            } else {
                is_v = true;
                tile = n_tiles - 1;
            }
        }
        const int s = i % NSLOT;
        const int key = k_lo + tile * BN;
        if (!FMHA_IN_BOUNDS(key >= 0 && key < k_hi && k_hi <= a.s_k && s < NSLOT, is_v ? kSitePairVLoad : kSitePairKLoad,
                            a.status))
            return false;
        mbar_arrive_expect_tx(&slot_full[s], C::KV_TILE);
#pragma unroll
        for (int c = 0; c < C::NB; ++c)
            tma_load_3d_hint(ring + s * C::KV_TILE + c * BN * 128, is_v ? &tmv : &tmk, c * 64, key, slab, &slot_full[s],
                             pol);
        return true;
    };
    int issued = 0;  // thread 0: ring items issued (0 .. issued-1)
    bool q_issued = false;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&s_free[t], 128);
        }
        mbar_init(p_ready, 128 * n_rt);
        mbar_init(&o_done[0], 1);
        mbar_init(&o_done[1], 1);
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        // Q and the first ring-full need no free slot: thread 0, the producer,
        // starts them before the block barrier and the TMEM allocation.
        if (n_tiles > 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            pol = l2_policy_evict_first();
            grid_dependency_wait();  // the preceding kernel's writes (Q, K, V) are visible
            if (FMHA_IN_BOUNDS(rb >= 0 && rb + (n_rt - 1) * BM < a.R && slab < (int)gridDim.z, kSitePairQLoad,
                               a.status)) {
                mbar_arrive_expect_tx(q_full, n_rt * C::Q_BYTES);
                for (int t = 0; t < n_rt; ++t)
#pragma unroll
                    for (int c = 0; c < C::NB; ++c)
                        tma_load_3d(sq + t * C::Q_BYTES + c * BM * 128, &tmq, c * 64, rb + t * BM, slab, q_full);
                q_issued = true;
            }
            for (int i = 0; i < min(NSLOT, n_items); ++i) {
                if (!issue_item(i)) break;
                ++issued;
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // every global access below follows the preceding kernel

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Items 0 .. NSLOT-1 went out before the block barrier.
        if (lane == 0) {
            for (int i = NSLOT; issued == i && i < n_items; ++i) {
                const int s = i % NSLOT;
                if (!mbar_wait(&slot_empty[s], ((i / NSLOT) - 1) & 1, a.status)) break;
                if (!issue_item(i)) break;
                ++issued;
            }
            drain_ring(slot_full, NSLOT, issued, a.status);
            if (q_issued) mbar_wait(q_full, 0, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
            // O^T (M = hd) += V (MN-major A) x P (K-major B), N = the rows of the tiles present
            const uint32_t idesc_o = idesc_bf16_f32(HD, BM * n_rt, 0) | (1u << 15);
            const uint32_t q_addr = smem_u32(sq), p_addr = smem_u32(sp), ring_addr = smem_u32(ring);
            int item = 0;
            auto slot_take = [&](int& s) -> bool {
                s = item % NSLOT;
                if (!mbar_wait(&slot_full[s], (item / NSLOT) & 1, a.status)) return false;
                ++item;
                return true;
            };
            auto issue_qk = [&](int t, int s) -> bool {
                if (!FMHA_IN_BOUNDS(s >= 0 && s < NSLOT && t >= 0 && t < n_rt, kSitePairKDesc, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes into the swizzled row
                    const uint64_t ad = smem_desc_sw128(q_addr + t * C::Q_BYTES + (kk >> 2) * BM * 128 + off, 16, 1024);
                    const uint64_t bd =
                        smem_desc_sw128(ring_addr + s * C::KV_TILE + (kk >> 2) * BN * 128 + off, 16, 1024);
                    tc_mma_f16(tmem + t * BN, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[t]);
                return true;
            };
            bool ok = mbar_wait(q_full, 0, a.status);
            int sk = 0;
            if (ok) ok = slot_take(sk);
            for (int t = 0; ok && t < n_rt; ++t) ok = issue_qk(t, sk);
            if (ok) tc_commit(&slot_empty[sk]);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles) {
                    // S_t(j + 1) once the softmax warps have loaded S_t(j)
                    if (!(ok = mbar_wait(&s_free[0], j & 1, a.status))) break;
                    if (!(ok = slot_take(sk))) break;
                    if (!(ok = issue_qk(0, sk))) break;
                    if (n_rt == 2) {
                        if (!(ok = mbar_wait(&s_free[1], j & 1, a.status))) break;
                        if (!(ok = issue_qk(1, sk))) break;
                    }
                    tc_commit(&slot_empty[sk]);
                }
                // V_j's slot first: it has usually landed before P_j is written,
                // and a barrier test costs this thread ~240 cycles
                int sv = 0;
                if (!(ok = slot_take(sv))) break;
                if (!(ok = mbar_wait(p_ready, j & 1, a.status))) break;
                ok = FMHA_IN_BOUNDS(sv >= 0 && sv < NSLOT, kSitePairVDesc, a.status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // A: 16 keys of V (64-column boxes one KV tile apart); B: the same 16 keys of P
                    const uint64_t ad = smem_desc_sw128(ring_addr + sv * C::KV_TILE + kk * 16 * 128, BN * 128, 1024);
                    const uint64_t bd = smem_desc_sw128(p_addr + (kk >> 2) * C::P_GROUP + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16(tmem + C::OT_COL, ad, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&o_done[j & 1]);
                tc_commit(&slot_empty[sv]);
            }
            // Exit drain: whatever the loop issued has completed before TMEM
            // and the operand buffers are released, even if a wait gave up.
            tc_commit(mma_drain);
            mbar_wait(mma_drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue of row tile t
        const int t = (warp - 2) >> 2;  // 0: warps 2..5, 1: warps 6..9
        if (t < n_rt) {
            const int bar_id = 2 + t;
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;  // TMEM lane of S_t and row within the tile
            // head-dim index of this thread's TMEM lane of O^T (at hd 64 only the
            // first 16 lanes of each quarter hold O^T)
            const int hdi = HD == 128 ? quarter * 32 + lane : quarter * 16 + lane;
            const bool hd_lane = HD == 128 || lane < 16;
            const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
            const int r_tile = rb + t * BM;
            const int grow = r_tile + row;
            const bool valid = grow < re;
            int jlo = INT_MAX, jhi = -1;
            if (valid) {
                pair_attended(grow % a.T, a, jlo, jhi);
                jlo = max(jlo, c_lo);
                jhi = min(jhi, c_hi - 1);
            }
            float m_ref = -INFINITY, l = 0.f, l_o = 0.f;
            bool ok = true;
            // A failed (timed-out) wait must not split a warpgroup: the loop
            // holds a named barrier, which has no time limit.  So a thread whose
            // wait gave up stays in the loop with ok = false, skips every later
            // wait and all work, and still meets its warpgroup at each barrier.
            // Within a warp the result of a wait is uniform (its lanes test the
            // barrier word and the timer in the same instructions); warps of the
            // group can disagree, which the barrier then tolerates.
            for (int j = 0; j < n_tiles; ++j) {
                ok = ok && mbar_wait(&s_full[t], j & 1, a.status);
                float alpha = 1.f;
                uint32_t pk[BN / 2];
                if (ok) {
                    tc_fence_after();
                    float x[BN];
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        float v32[32];
                        tmem_ld32(t_lane + t * BN + c * 32, v32);
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[c * 32 + i] = v32[i];
                    }
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&s_free[t]);  // S_t may now be overwritten by QK_t(j + 1)
                    softmax_row_tile<BN>(x, pk, k_lo + j * BN, jlo, jhi, a.scale_log2, m_ref, l, l_o, alpha);
                    // PV(j - 1) has read the P buffer and updated O^T (each
                    // o_done barrier has at most one phase outstanding: PV(j)
                    // needs this step's P)
                    if (j > 0) ok = mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.status);
                }
                // Lazy rescale: column r of O^T (this tile's row r) times alpha_r,
                // by the four warps that own O^T's lanes.
                if (j > 0 && named_barrier_or(bar_id, 128, ok && alpha != 1.f)) {
                    ok = __all_sync(0xffffffffu, ok);  // the TMEM accesses below are warp-collective
                    rowv[t * BM + row] = ok ? alpha : 1.f;
                    named_barrier_sync(bar_id, 128);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < BM / 32; ++c) {
                            float ov[32];
                            tmem_ld32(t_lane + C::OT_COL + t * BM + c * 32, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[i] *= rowv[t * BM + c * 32 + i];
                            tmem_st32(t_lane + C::OT_COL + t * BM + c * 32, ov);
                        }
                        tmem_wait_st();
                    }
                }
                if (ok) {
                    write_p_row256<BN>(sp, t * BM + row, pk);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(p_ready);
                }
            }
            // -------------------------------------------------------- epilogue
            if (ok && n_tiles > 0)
                ok = mbar_wait(&o_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, a.status);
            ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
            if (!ok) atomicOr(abort_flag, 1);
            float inv, lse;
            // query head of this row: kvh * G + (row within the slab) / T
            finish_row(m_ref, l, l_o,
                       (SINK && valid) ? sink_log2_of(a.sink, kvh * a.group + grow / a.T, a.n_h, a.status)
                                       : -INFINITY,
                       inv, lse);
            named_barrier_sync(bar_id, 128);  // every rescale has read rowv
            rowv[t * BM + row] = inv;
            named_barrier_sync(bar_id, 128);
            tc_fence_after();
            const bool have_o = ok && n_tiles > 0;
            // O^T columns of this tile -> O rows (times 1 / sum) in the TMA box
            // layout -> TMA store.  Tile A stages in the Q tiles, tile B in the
            // P buffer: the last PV, which covers both tiles, has completed.
            uint8_t* stage = t == 0 ? sq : sp;
            if (!a.to_partials) {
                // bf16 boxes of 64 columns x 128 rows (128-byte rows, swizzled)
                uint8_t* col = stage + ((hdi >> 6) & (HD / 64 - 1)) * 16384 + (hdi & 7) * 2;
                const int chunk = (hdi & 63) >> 3;
#pragma unroll 1
                for (int c = 0; c < BM / 32; ++c) {
                    float ov[32];
                    if (have_o) {
                        tmem_ld32(t_lane + C::OT_COL + t * BM + c * 32, ov);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = 0.f;
                    }
                    if (hd_lane) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int r = c * 32 + i;
                            *reinterpret_cast<__nv_bfloat16*>(col + r * 128 + ((chunk ^ (r & 7)) << 4)) =
                                __float2bfloat16_rn(ov[i] * rowv[t * BM + r]);
                        }
                    }
                }
            } else {
                // fp32 boxes of 32 columns x 128 rows
                uint8_t* col = stage + ((hdi >> 5) & (HD / 32 - 1)) * 16384 + (hdi & 3) * 4;
                const int chunk = (hdi & 31) >> 2;
#pragma unroll 1
                for (int c = 0; c < BM / 32; ++c) {
                    float ov[32];
                    if (have_o) {
                        tmem_ld32(t_lane + C::OT_COL + t * BM + c * 32, ov);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = 0.f;
                    }
                    if (hd_lane) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int r = c * 32 + i;
                            *reinterpret_cast<float*>(col + r * 128 + ((chunk ^ (r & 7)) << 4)) =
                                ov[i] * rowv[t * BM + r];
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(bar_id, 128);
            if (threadIdx.x == 64 + 128 * t && *abort_flag == 0) {
                const int n_box = a.to_partials ? HD / 32 : HD / 64;
                const int box_cols = a.to_partials ? 32 : 64;
                const int slab_c = a.to_partials ? split * (int)(a.rows_total / a.R) + slab : slab;
                const int n_slabs = a.to_partials ? (int)(gridDim.y * gridDim.z) : (int)gridDim.z;
                for (int bx = 0; bx < n_box; ++bx) {
                    if (FMHA_IN_BOUNDS(r_tile >= 0 && r_tile < a.R && slab_c >= 0 && slab_c < n_slabs, kSiteEpiStore,
                                       a.status))
                        tma_store_3d(&tmo, bx * box_cols, r_tile, slab_c, stage + bx * 16384);
                }
                tma_store_commit();
                tma_store_wait_read();
            }
            if (valid && ok) {
                const long long gr = row0 + grow;
                if (FMHA_IN_BOUNDS(gr >= 0 && gr < a.rows_total && split < (int)gridDim.y, kSitePairLse, a.status)) {
                    if (!a.to_partials)
                        a.lse[gr] = lse;
                    else
                        a.lse_part[(long long)split * a.rows_total + gr] = lse;
                }
            }
            tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int HD, int EPI>
cudaError_t launch_pair_t(const TcLaunch& L, cudaStream_t stream) {
    using C = PCfg<HD>;
    auto kern = fwd_tc_pair_kernel<HD, EPI>;
    static std::atomic<bool> attr_set[128];  // set once per device; any host thread may set it
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 128) attr_set[dev] = true;
    }
    PairArgs a;
    a.o = static_cast<__nv_bfloat16*>(L.o);
    a.lse = L.lse;
    a.lse_part = L.lse_part;
    a.to_partials = L.to_partials ? 1 : 0;
    a.n_h = L.p.n_h;
    a.n_kv_h = L.p.n_kv_h;
    a.T = L.p.T;
    a.s_k = L.p.s_k;
    a.group = L.p.group;
    a.R = L.p.R;
    a.window = L.p.window;
    a.causal = L.p.causal;
    a.scale_log2 = (float)((double)L.p.scale * 1.4426950408889634);
    a.kv_begin = L.sp.kv_begin;
    a.kv_chunk = L.sp.kv_chunk;
    a.rows_total = (long long)L.p.batch * L.p.n_h * L.p.T;
    a.status = L.status;
    a.sink = L.sink;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((L.p.R + 2 * C::BM - 1) / (2 * C::BM), L.sp.n_splits, L.p.batch * L.p.n_kv_h);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_q, L.tmap_k, L.tmap_v, L.tmap_o, a);
}

}  // namespace

bool tc_pair_supports(int hd) { return hd == 64 || hd == 128; }
int tc_pair_kv_tile() { return PCfg<128>::BN; }

cudaError_t launch_tc_pair(const TcLaunch& L, cudaStream_t stream) {
    if (!tc_pair_supports(L.p.hd) || (L.fp4.codes && !L.to_partials)) return cudaErrorInvalidValue;
    const bool sink = L.sink && !L.to_partials;
    if (L.p.hd == 64) return sink ? launch_pair_t<64, kEpiSink>(L, stream) : launch_pair_t<64, kEpiBf16>(L, stream);
    return sink ? launch_pair_t<128, kEpiSink>(L, stream) : launch_pair_t<128, kEpiBf16>(L, stream);
}

}  // namespace fmha
