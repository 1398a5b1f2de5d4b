// tc_kernel.cu -- attention forward for 128-row query tiles on the tcgen05
// tensor cores (sm_103a).
//
// One thread block owns 128 query rows that share one KV head (a causal
// prefill slice, or the query heads of an MQA/GQA decode step) and one chunk
// of the KV range.  Both contractions are dense, so both go to the tensor
// cores:
//   S_j = Q K_j^T       tcgen05.mma M=128, N=BN, K=hd  (A = Q, B = K; both K-major)
//   O  += P_j V_j       tcgen05.mma M=128, N=hd, K=BN  (A = P K-major, B = V MN-major)
// with the accumulators S (two buffers) and O in tensor memory.
//
// Warp roles (7 warps):
//   warp 0      TMA producer for Q (once) and K_j; a K stage is released as
//               soon as QK_j has read it
//   warp 6      TMA producer for V_j; a V stage is released after PV_j
//   warp 1      TMEM owner and MMA issuer (one elected lane): QK runs two
//               tiles ahead of PV (three at hd <= 128 in the TS form, with a
//               third S buffer), P is double-buffered
//   warps 2..5  softmax: one query row per thread (its TMEM lane); reads S_j
//               with tcgen05.ld, applies scale and mask, keeps the running max
//               and sum (FA2 online softmax: commit e4ee9fd of the
//               nvfp4-megamoe-kernel pages, multi-tile C API part), writes the
//               un-normalised P_j to shared memory as bf16 and, when the
//               reference max moved, rescales its O row in TMEM (the O
//               rescale in registers of commit 593bc25, "D1.5 fix").
// The reference max only moves when a tile's max exceeds it by more than
// 2^8, so rescales are rare; P then stays <= 256, exact enough in bf16.
// Epilogue: O / running sum -> bf16 (or fp32 partials for the split-KV merge),
// LSE = (max + log2 sum) * ln 2.
//
// Every tcgen05.ld/st is executed by all 32 lanes of a warp (they are
// warp-collective: the TMEM epilogue hang on the 593bc25 page), and TMEM is
// released with the address tcgen05.alloc returned.
#include <climits>
#include <atomic>
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fmha {
namespace {

// TS = false: P goes through two shared-memory buffers and PV reads A from
// shared memory (the "SS" form).  TS = true: the softmax writes P into tensor
// memory over its own S tile (bf16 pairs in the first BN / 2 columns of the S
// buffer) and PV reads A from there (the "TS" form); the P buffers' shared
// memory holds more K / V stages instead.
template <int HD, bool TS>
struct TCfg {
    static constexpr int BM = 128;                     // query rows per CTA (MMA M)
    static constexpr int BN = (HD <= 128) ? 128 : 64;  // keys per tile
    static constexpr int KST = TS ? (HD == 64 ? 6 : 3) : (HD == 64 ? 4 : 2);  // K stages
    static constexpr int VST = TS ? (HD == 64 ? 6 : HD == 128 ? 3 : 2) : (HD == 64 ? 4 : 2);  // V stages
    static constexpr int NB = HD / 64;                 // 64-column (128-byte) boxes
    static constexpr int Q_BYTES = BM * HD * 2;
    static constexpr int KV_TILE = BN * HD * 2;        // one K or V tile
    static constexpr int P_GROUPS = (BN + 63) / 64;    // 128-byte swizzled row groups of P
    static constexpr int P_CHUNKS = (BN < 64 ? BN : 64) / 8;  // 16-byte chunks per row and group
    static constexpr int P_BYTES = TS ? 0 : BM * 128 * P_GROUPS;  // one P buffer (two are kept)
    static constexpr int THREADS = 224;
    // S buffers in TMEM (P over S in the TS form): three at hd <= 128 in the TS
    // form, so that QK runs three tiles ahead of P V, two otherwise
    static constexpr int NSB = (TS && HD <= 128) ? 3 : 2;
    static constexpr int S_COL0 = 0;                   // TMEM columns: S buffers, then O
    static constexpr int O_COL = NSB * BN;
    // TS at hd 64: P V runs with N = hd + 16, the extra columns of B a tile of
    // ones in shared memory, so O's column hd accumulates the sum of the
    // bf16-rounded P (the divisor of O) and the softmax does not
    static constexpr bool ONES = TS && HD == 64;
    static constexpr int O_N = HD + (ONES ? 16 : 0);  // O columns written by P V
    static constexpr int ONES_BYTES = ONES ? BN * 128 : 0;
    static constexpr int TMEM_COLS = 512;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + KST * KV_TILE;
    static constexpr int OFF_P = OFF_V + VST * KV_TILE;
    static constexpr int OFF_ONES = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_BAR = OFF_ONES + ONES_BYTES;
    static constexpr int N_BARS = 1 + 2 * KST + 2 * VST + 3 * NSB + 1;
    static constexpr int SMEM = 1024 + OFF_BAR + N_BARS * 8 + 16;
    static_assert(O_COL + (O_N + 31) / 32 * 32 <= TMEM_COLS, "S buffers + O must fit in TMEM");
    static_assert(TS || NSB == 2, "the SS form's P buffers pair with two S buffers");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((KST + VST) * KV_TILE >= BM * HD * 4, "the epilogue stages fp32 O in the K/V stages");
};

struct TcArgs {
    __nv_bfloat16* o;
    float* lse;
    float* o_part;
    float* lse_part;
    int to_partials;
    int n_h, n_kv_h, T, s_k, group, R, window, causal;
    float scale_log2;
    int kv_begin, kv_chunk;
    long long rows_total;
    unsigned* status;
    const float* sink;  // [n_h] sink logits (final output only) or NULL
    Fp4Out fp4;         // NVFP4 final output (EPI == kEpiNvfp4)
};

__device__ __forceinline__ void attended_rows(int t, const TcArgs& a, int& lo, int& hi) {
    const int p = a.s_k - a.T + t;
    lo = 0;
    hi = a.s_k - 1;
    if (a.causal) hi = min(hi, p);
    if (a.window > 0) lo = max(lo, p - a.window + 1);
}

template <int HD, int EPI, bool TS>
__global__ void __launch_bounds__(TCfg<HD, TS>::THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo, const TcArgs a) {
    using C = TCfg<HD, TS>;
    constexpr int BM = C::BM, BN = C::BN, KST = C::KST, VST = C::VST;
    constexpr bool SINK = EPI == kEpiSink;
    launch_dependents();  // the merge grid may be scheduled now; it waits for this grid's results
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sq = smem + C::OFF_Q;
    uint8_t* sk = smem + C::OFF_K;
    uint8_t* sv = smem + C::OFF_V;
    uint8_t* sp = smem + C::OFF_P;
    uint8_t* sones = smem + C::OFF_ONES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + KST;
    uint64_t* v_full = k_empty + KST;
    uint64_t* v_empty = v_full + VST;
    constexpr int NSB = C::NSB;
    uint64_t* s_full = v_empty + VST;    // [NSB] by S buffer
    uint64_t* p_ready = s_full + NSB;    // [NSB] by P buffer (the S buffer in the TS form)
    uint64_t* o_done = p_ready + NSB;    // [NSB] by P buffer: PV of a tile using that P buffer completed
    uint64_t* mma_drain = o_done + NSB;  // every MMA the issuer launched has completed (exit drain)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::N_BARS);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x, split = blockIdx.y, slab = blockIdx.z;
    const int b = slab / a.n_kv_h, kvh = slab - b * a.n_kv_h;
    const long long row0 = ((long long)b * a.n_h + (long long)kvh * a.group) * a.T;  // slab's first query row
    const int r_begin = rt * BM;
    const int r_end = min(a.R, r_begin + BM);

    // KV range of this CTA: its chunk intersected with what its rows attend.
    const int c_lo = a.kv_begin + split * a.kv_chunk;
    const int c_hi = min(a.s_k, c_lo + a.kv_chunk);
    int u_lo, u_hi;
    if (r_end - r_begin >= a.T) {
        int l0, h0, l1, h1;
        attended_rows(0, a, l0, h0);
        attended_rows(a.T - 1, a, l1, h1);
        u_lo = l0;
        u_hi = h1;
    } else {
        int l0, h0, l1, h1;
        attended_rows(r_begin % a.T, a, l0, h0);
        attended_rows((r_end - 1) % a.T, a, l1, h1);
        // rows r_begin..r_end-1 may wrap once past t = T-1
        if ((r_end - 1) % a.T < r_begin % a.T) {
            int lz, hz, lx, hx;
            attended_rows(0, a, lz, hz);
            attended_rows(a.T - 1, a, lx, hx);
            u_lo = lz;
            u_hi = hx;
        } else {
            u_lo = l0;
            u_hi = h1;
        }
    }
    const int k_lo = max(c_lo, u_lo), k_hi = min(c_hi, u_hi + 1);
    const int n_tiles = (k_hi > k_lo) ? (k_hi - k_lo + BN - 1) / BN : 0;

    // K tile j into stage j % KST (the caller has made sure the stage is free).
    uint64_t pol_k = 0;
    auto issue_k = [&](int j) -> bool {
        const int s = j % KST;
        const int key = k_lo + j * BN;
        if (!FMHA_IN_BOUNDS(key >= 0 && key < k_hi && k_hi <= a.s_k && s < KST, kSiteTcKLoad, a.status)) return false;
        mbar_arrive_expect_tx(&k_full[s], C::KV_TILE);
#pragma unroll
        for (int c = 0; c < C::NB; ++c)
            tma_load_3d_hint(sk + s * C::KV_TILE + c * BN * 128, &tmk, c * 64, key, slab, &k_full[s], pol_k);
        return true;
    };
    const int k_first = min(KST, n_tiles);  // K tiles issued before the block barrier
    int k_issued = 0;                        // thread 0: K tiles issued (0 .. k_issued-1)
    bool q_issued = false;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < KST; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int b2 = 0; b2 < NSB; ++b2) {
            mbar_init(&s_full[b2], 1);
            mbar_init(&p_ready[b2], 128);
            mbar_init(&o_done[b2], 1);
        }
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        // Q and the first K stages need no free slot: thread 0, the Q/K
        // producer, starts them before the block barrier and the TMEM allocation.
        if (n_tiles > 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            pol_k = l2_policy_evict_first();
            grid_dependency_wait();  // the preceding kernel's writes (Q, K, V) are visible
            if (FMHA_IN_BOUNDS(r_begin >= 0 && r_begin < a.R && slab < (int)gridDim.z, kSiteTcQLoad, a.status)) {
                mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
                for (int c = 0; c < C::NB; ++c) tma_load_3d(sq + c * BM * 128, &tmq, c * 64, r_begin, slab, q_full);
                q_issued = true;
            }
            for (int j = 0; j < k_first; ++j) {
                if (!issue_k(j)) break;
                ++k_issued;
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (C::ONES) {
        // bf16 1.0 in every element: which columns the swizzle puts where does not matter
        for (int i = threadIdx.x; i < C::ONES_BYTES / 16; i += C::THREADS)
            reinterpret_cast<uint4*>(sones)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // every global access below follows the preceding kernel

    if (warp == 0) {
        // ------------------------------------------------------------ Q / K producer
        // Q and K tiles 0 .. k_first-1 went out before the block barrier.
        if (lane == 0) {
            for (int j = k_first; k_issued == j && j < n_tiles; ++j) {
                const int s = j % KST;
                if (!mbar_wait(&k_empty[s], ((j / KST) - 1) & 1, a.status)) break;
                if (!issue_k(j)) break;
                ++k_issued;
            }
            drain_ring(k_full, KST, k_issued, a.status);
            if (q_issued) mbar_wait(q_full, 0, a.status);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ V producer
        if (lane == 0 && n_tiles > 0) {
            tma_prefetch_desc(&tmv);
            const uint64_t pol = l2_policy_evict_first();
            // V_0 is needed only after S_0 and its softmax: at hd >= 128, where Q
            // and K_0 are large, let them take the SM's load bandwidth first
            // (Q is issued just before K_0; q_full completes once per block).
            const bool q_in = HD < 128 || mbar_wait(q_full, 0, a.status);
            int v_issued = 0;
            for (int j = 0; q_in && j < n_tiles; ++j) {
                const int s = j % VST;
                if (j >= VST && !mbar_wait(&v_empty[s], ((j / VST) - 1) & 1, a.status)) break;
                const int key = k_lo + j * BN;
                if (!FMHA_IN_BOUNDS(key >= 0 && key < k_hi && k_hi <= a.s_k && s < VST, kSiteTcVLoad, a.status)) break;
                mbar_arrive_expect_tx(&v_full[s], C::KV_TILE);
#pragma unroll
                for (int c = 0; c < C::NB; ++c)
                    tma_load_3d_hint(sv + s * C::KV_TILE + c * BN * 128, &tmv, c * 64, key, slab, &v_full[s], pol);
                ++v_issued;
            }
            drain_ring(v_full, VST, v_issued, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Order: QK_0 .. QK_{NSB-1}, then per tile j: PV_j, QK_{j+NSB}.
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, C::O_N, 1);
            const uint32_t q_addr = smem_u32(sq), k_addr = smem_u32(sk), v_addr = smem_u32(sv),
                           p_addr = smem_u32(sp);
            bool ok = mbar_wait(q_full, 0, a.status);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % KST;
                if (!FMHA_IN_BOUNDS(s >= 0 && s < KST, kSiteTcKDesc, a.status)) return false;
                if (!mbar_wait(&k_full[s], (j / KST) & 1, a.status)) return false;
                tc_fence_after();
                const uint32_t d = tmem + C::S_COL0 + (j % NSB) * BN;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;  // 16 columns = 32 bytes into the swizzled row
                    const uint64_t ad = smem_desc_sw128(q_addr + (kk >> 2) * BM * 128 + off, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(k_addr + s * C::KV_TILE + (kk >> 2) * BN * 128 + off, 16, 1024);
                    tc_mma_f16(d, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[j % NSB]);
                tc_commit(&k_empty[s]);
                return true;
            };
            for (int j = 0; ok && j < NSB && j < n_tiles; ++j) ok = issue_qk(j);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int s = j % VST;
                const int pb = j % NSB;
                if (!FMHA_IN_BOUNDS(s >= 0 && s < VST && pb < NSB, kSiteTcVDesc, a.status)) break;
                // V_j has usually landed long before P_j: test it first, while the
                // softmax still works, so that no barrier test (~240 cycles for
                // this thread) stands between P_j and its MMAs
                if (!mbar_wait(&v_full[s], (j / VST) & 1, a.status)) break;
                if (!mbar_wait(&p_ready[pb], (j / NSB) & 1, a.status)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // V's 64-column boxes one tile apart, or at hd 64 the tile of ones
                    // as the second box (the leading byte offset spans the gap)
                    const uint32_t lbo = C::ONES ? smem_u32(sones) - (v_addr + s * C::KV_TILE) : BN * 128;
                    const uint64_t bd = smem_desc_sw128(v_addr + s * C::KV_TILE + kk * 16 * 128, lbo, 1024);
                    if constexpr (TS) {
                        // A = P_j in TMEM: S buffer j % NSB, 8 columns (16 bf16 keys) per MMA
                        const uint32_t a_col = C::S_COL0 + pb * BN + kk * 8;
                        if (!FMHA_IN_BOUNDS(a_col + 8 <= C::S_COL0 + NSB * BN, kSiteTcPTmem, a.status)) break;
                        tc_mma_f16_ts(tmem + C::O_COL, tmem + a_col, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                    } else {
                        const uint64_t ad = smem_desc_sw128(
                            p_addr + pb * C::P_BYTES + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                        tc_mma_f16(tmem + C::O_COL, ad, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(&o_done[pb]);
                tc_commit(&v_empty[s]);
                if (j + NSB < n_tiles && !issue_qk(j + NSB)) break;
            }
            // Exit drain: whatever the loop issued has completed before TMEM
            // and the operand buffers are released, even if a wait gave up.
            tc_commit(mma_drain);
            mbar_wait(mma_drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;              // TMEM lane and tile row
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const int grow = r_begin + row;
        const bool valid = grow < r_end;
        int jlo = INT_MAX, jhi = -1;
        if (valid) {
            attended_rows(grow % a.T, a, jlo, jhi);
            jlo = max(jlo, c_lo);
            jhi = min(jhi, c_hi - 1);
        }
        float m_ref = -INFINITY, l = 0.f, l_o = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int pb = j % NSB;
            if (!mbar_wait(&s_full[pb], (j / NSB) & 1, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[BN];
            const uint32_t s_col = FMHA_IN_BOUNDS(C::S_COL0 + pb * BN + BN <= C::O_COL, kSiteTcSCol, a.status)
                                       ? C::S_COL0 + pb * BN
                                       : 0u;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                float v32[32];
                tmem_ld32(t_lane + s_col + c * 32, v32);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[c * 32 + i] = v32[i];
            }
            tmem_wait_ld();
            // Exponentials and the row sum before waiting on the tensor core.
            float alpha;
            uint32_t pk[BN / 2];
            softmax_row_tile<BN, !C::ONES>(x, pk, k_lo + j * BN, jlo, jhi, a.scale_log2, m_ref, l, l_o, alpha);
            const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
            // SS: P buffer pb was last read by PV_{j-2}.  TS: P_j goes over S_j,
            // whose QK the MMA issuer queued after PV_{j-NSB}, so S_j being ready
            // means that PV is done.  Either way a rescale of O needs PV_{j-1} done.
            if (rescale) {
                if (!mbar_wait(&o_done[(j - 1) % NSB], ((j - 1) / NSB) & 1, a.status)) {
                    ok = false;
                    break;
                }
            } else if (!TS && j >= NSB) {
                if (!mbar_wait(&o_done[pb], ((j / NSB) - 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
            }
            if constexpr (TS) {
                // this row's P_j (BN bf16 = BN / 2 words) over the S_j columns it has read
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) tmem_st32u(t_lane + s_col + c * 32, pk + c * 32);
                tmem_wait_st();
            } else if (FMHA_IN_BOUNDS(row >= 0 && row < BM && pb < 2, kSiteTcPRow, a.status)) {
                write_p_row<BN>(sp + pb * C::P_BYTES, row, pk);
            }
            if (rescale) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < (C::O_N + 31) / 32; ++c) {  // with the column of rounded sums
                    float ov[32];
                    tmem_ld32(t_lane + C::O_COL + c * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                    tmem_st32(t_lane + C::O_COL + c * 32, ov);
                }
                tmem_wait_st();
            }
            if constexpr (!TS) fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_ready[pb]);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n_tiles > 0) ok = mbar_wait(&o_done[(n_tiles - 1) % NSB], ((n_tiles - 1) / NSB) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        if (!ok) atomicOr(abort_flag, 1);
        tc_fence_after();
        if constexpr (C::ONES) {  // the sum of the rounded P, from O's column hd (warp-collective load)
            l_o = 0.f;
            if (ok && n_tiles > 0) {
                l_o = tmem_ld1(t_lane + C::O_COL + HD);
                tmem_wait_ld();
            }
        }
        float inv, lse;
        // query head of this row: kvh * G + (row within the slab) / T
        finish_row(m_ref, l, l_o,
                   (SINK && valid) ? sink_log2_of(a.sink, kvh * a.group + grow / a.T, a.n_h, a.status) : -INFINITY,
                   inv, lse);
        // O -> shared memory (the drained K/V stages) -> TMA store; rows past
        // the slab's end fall outside the tensor map and are not written.
        uint8_t* stage = sk;
        constexpr int kStageBytes = (KST + VST) * C::KV_TILE;
        if constexpr (EPI == kEpiNvfp4) {
            // quantised in registers and stored per row; rows past the slab's
            // end and blocks that gave up store nothing
            named_barrier_sync(2, 128);
            const long long gr = row0 + grow;
            const bool row_ok = valid && *abort_flag == 0 &&
                                FMHA_IN_BOUNDS(gr >= 0 && gr < a.rows_total, kSiteTcFp4, a.status);
            epilogue_nvfp4<HD>(t_lane + C::O_COL, inv, row_ok, a.fp4.codes + (row_ok ? gr : 0) * (HD / 2),
                               a.fp4.scales + (row_ok ? gr : 0) * (HD / 16), a.fp4.g, ok && n_tiles > 0);
        } else if (!a.to_partials)
            epilogue_tma_store<HD, kOutBf16>(t_lane + C::O_COL, inv, row, stage, kStageBytes, &tmo, 0, r_begin,
                                             slab, make_int3(HD, a.R, (int)gridDim.z), ok && n_tiles > 0,
                                             threadIdx.x == 64, abort_flag, a.status);
        else
            epilogue_tma_store<HD, kOutF32>(t_lane + C::O_COL, inv, row, stage, kStageBytes, &tmo, 0, r_begin,
                                            split * (int)(a.rows_total / a.R) + slab,
                                            make_int3(HD, a.R, (int)(gridDim.y * gridDim.z)), ok && n_tiles > 0,
                                            threadIdx.x == 64, abort_flag, a.status);
        if (valid && ok) {
            const long long gr = row0 + grow;
            if (FMHA_IN_BOUNDS(gr >= 0 && gr < a.rows_total && split < (int)gridDim.y, kSiteTcLse, a.status)) {
                if (!a.to_partials)
                    a.lse[gr] = lse;
                else
                    a.lse_part[(long long)split * a.rows_total + gr] = lse;
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int HD, int EPI, bool TS>
cudaError_t launch_t(const TcLaunch& L, cudaStream_t stream) {
    using C = TCfg<HD, TS>;
    auto kern = fwd_tc_kernel<HD, EPI, TS>;
    static std::atomic<bool> attr_set[128];  // set once per device; any host thread may set it
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 128) attr_set[dev] = true;
    }
    TcArgs a;
    a.o = static_cast<__nv_bfloat16*>(L.o);
    a.lse = L.lse;
    a.o_part = static_cast<float*>(L.o_part);
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
    a.fp4 = L.fp4;
    dim3 grid((L.p.R + C::BM - 1) / C::BM, L.sp.n_splits, L.p.batch * L.p.n_kv_h);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_q, L.tmap_k, L.tmap_v, L.tmap_o, a);
}

}  // namespace

int tc_kv_tile(int hd) {
    switch (hd) {
        case 64: return TCfg<64, true>::BN;
        case 128: return TCfg<128, true>::BN;
        case 256: return TCfg<256, true>::BN;
        default: return 0;
    }
}

bool tc_supports(int hd) { return hd == 64 || hd == 128 || hd == 256; }

template <int EPI, bool TS>
cudaError_t launch_hd(const TcLaunch& L, cudaStream_t stream) {
    switch (L.p.hd) {
        case 64: return launch_t<64, EPI, TS>(L, stream);
        case 128: return launch_t<128, EPI, TS>(L, stream);
        case 256: return launch_t<256, EPI, TS>(L, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int EPI>
cudaError_t launch_form(const TcLaunch& L, cudaStream_t stream) {
    return L.ss_pv ? launch_hd<EPI, false>(L, stream) : launch_hd<EPI, true>(L, stream);
}

cudaError_t launch_tc(const TcLaunch& L, cudaStream_t stream) {
    if (L.fp4.codes && !L.to_partials) return launch_form<kEpiNvfp4>(L, stream);
    return (L.sink && !L.to_partials) ? launch_form<kEpiSink>(L, stream) : launch_form<kEpiBf16>(L, stream);
}

}  // namespace fmha
