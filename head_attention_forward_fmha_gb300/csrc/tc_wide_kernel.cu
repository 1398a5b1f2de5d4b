// tc_wide_kernel.cu -- tcgen05 attention forward for hd = 512 (128-row tiles).
//
// At hd 512 the fp32 O accumulator of a 128-row tile (128 x 512 x 4 bytes)
// fills all of tensor memory, and the bf16 Q tile alone is 128 KB of shared
// memory.  So each thread block owns 128 query rows, one KV chunk and one HALF
// of the head dim of O (256 columns; blockIdx.x = 2 * row_tile + half):
//   S_j  = sum_c Q[:, c] K_j[:, c]^T   over the 8 64-column chunks c of hd
//          (every block computes the full S; it is cheap next to the loads)
//   O_h += P_j V_j[:, 256h : 256h + 256]
// Q and K stream through one ring chunk by chunk, Q chunk c and K chunk c in
// one 32 KB item (Q chunks come from L2 after the first block reads them),
// then the four 64-column V chunks of this half in two items.  TMEM: two S
// buffers (2 x 128 columns) + O half (256).
// Softmax, lazy rescale and the epilogue are those of tc_kernel.cu; both
// halves compute identical (max, sum), and half 0 writes the LSE.
#include <algorithm>
#include <climits>
#include <atomic>
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fmha {
namespace {

// Index-check site of this kernel beside those in ptx.cuh: a block without a
// resident Q holds at most one KV tile.
constexpr unsigned kSiteWideTiles = 0x20a;

// Every ring item holds two 64-column chunks under one barrier: a barrier
// test costs the MMA-issuing thread ~240 cycles after N = 128 MMAs, so fewer
// and larger items keep the tensor pipe fed.  QRES = false: the items are
// (Q chunk c, K chunk c) pairs, then the V chunks, through a ring of six
// 32 KB items (a block with a single KV tile reads Q once either way; a
// seventh item would leave no shared memory for the merge's blocks, which
// then could not become resident before this grid ends).
// QRES = true (blocks with two or more KV tiles): the 128 KB Q tile is loaded
// once and stays resident, and only K and V chunks stream, through three
// 32 KB items; the epilogue then stages O in the Q region and the drained ring.
// With at most 32 (64) query rows per KV head, QROWS = 32 (64): only those
// rows of each Q chunk are loaded, the chunks 4 KB (8 KB) apart.  The MMA
// still reads 128 rows of A per chunk, the rows past QROWS falling on the next
// chunks (or a zeroed tail); their S rows belong to no query and are masked.
// Q then takes 44 KB (72 KB) and the ring five (four) items.  In all, P goes
// over S in tensor memory and the P V MMAs read it from there (the TS form),
// so no shared memory holds P.
template <bool QRES, int QROWS = 128>
struct WCfgT {
    static constexpr int HD = 512;
    static constexpr int HALF = 256;
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int SLOT_BYTES = 128 * 128;       // one chunk: 128 rows x 64 bf16 columns
    static constexpr int Q_CHUNKS = HD / 64;
    static constexpr int CPI = 2;                      // chunks per ring item
    static constexpr int ITEM_BYTES = CPI * SLOT_BYTES;
    static constexpr int Q_ROWS = QRES ? QROWS : 128;  // rows of each Q chunk loaded
    static constexpr int Q_STRIDE = Q_ROWS * 128;      // bytes between resident Q chunks
    // the last chunk's MMA reads a whole 128-row operand
    static constexpr int Q_REGION = QRES ? (Q_CHUNKS - 1) * Q_STRIDE + SLOT_BYTES : 0;
    static constexpr int NSLOT = QRES ? (Q_ROWS == 128 ? 3 : Q_ROWS == 64 ? 4 : 5) : 6;  // ring items
    static constexpr int QK_ITEMS = QRES ? Q_CHUNKS / CPI : Q_CHUNKS;  // (K, K) or (Q, K) chunk pairs per tile
    static constexpr int V_CHUNKS = HALF / 64;
    static constexpr int V_ITEMS = V_CHUNKS / CPI;
    static constexpr int TILE_ITEMS = QK_ITEMS + V_ITEMS;
    // P V is one MMA of N = 64 V_GROUP per group of V_GROUP chunks and 16 keys,
    // the group's chunks one SLOT_BYTES apart: one N = 256 MMA over the two V
    // items of a one-tile block (items QK_ITEMS and QK_ITEMS + 1, in
    // consecutive slots of the ring; such a block never holds a second tile);
    // two N = 128 MMAs, one per item, with the resident Q.
    static constexpr int V_GROUP = QRES ? 2 : 4;
    static constexpr int V_GROUP_ITEMS = V_GROUP / CPI;
    static_assert(QRES ? V_GROUP_ITEMS == 1 : (QK_ITEMS % NSLOT + V_ITEMS <= NSLOT && V_GROUP_ITEMS == V_ITEMS),
                  "V slot groups must be contiguous");
    static constexpr int P_BYTES = 0;  // P lives in tensor memory
    static constexpr int THREADS = 192;
    static constexpr int O_COL = 2 * BN;
    static constexpr int TMEM_COLS = 512;
    static constexpr int OFF_Q = 0;                                   // QRES: resident Q
    static constexpr int OFF_RING = OFF_Q + Q_REGION;
    static constexpr int OFF_P = OFF_RING + NSLOT * ITEM_BYTES;
    static constexpr int OFF_BAR = OFF_P + P_BYTES;
    static constexpr int OFF_STAGE = QRES ? OFF_Q : OFF_RING;         // epilogue staging
    static constexpr int STAGE_BYTES = OFF_P - OFF_STAGE;
    static constexpr int N_BARS = 2 * NSLOT + 2 + 2 + 2 + 1 + (QRES ? 1 : 0);
    static constexpr int SMEM = 1024 + OFF_BAR + N_BARS * 8 + 16;
    static_assert(O_COL + HALF <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(STAGE_BYTES >= BM * HALF * 4, "the epilogue stages fp32 O");
    static_assert(Q_ROWS == 128 || Q_ROWS == 64 || Q_ROWS == 32, "resident Q rows");
};
using WCfg = WCfgT<false>;

struct WideArgs {
    __nv_bfloat16* o;
    float* lse;
    float* lse_part;
    float* range_part;  // fp16 partials: the power-of-two factor of each (split, row, half)
    int to_partials;
    int part_f16;       // partials as fp16 (fmha_fwd's workspace) instead of fp32
    int n_h, n_kv_h, T, s_k, group, R, window, causal;
    float scale_log2;
    int kv_begin, kv_chunk;
    long long rows_total;
    unsigned* status;
    const float* sink;  // [n_h] sink logits (final output only) or NULL
    Fp4Out fp4;         // NVFP4 final output (EPI == kEpiNvfp4)
};

__device__ __forceinline__ void w_attended(int t, const WideArgs& a, int& lo, int& hi) {
    const int p = a.s_k - a.T + t;
    lo = 0;
    hi = a.s_k - 1;
    if (a.causal) hi = min(hi, p);
    if (a.window > 0) lo = max(lo, p - a.window + 1);
}

template <int EPI, bool QRES, int QROWS>
__global__ void __launch_bounds__(WCfg::THREADS, 1)
    fwd_tc_wide_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                       const WideArgs a) {
    using C = WCfgT<QRES, QROWS>;
    constexpr int BM = C::BM, BN = C::BN;
    constexpr bool SINK = EPI == kEpiSink;
    launch_dependents();  // the merge grid may be scheduled now; it waits for this grid's results
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* slot_full = bars;
    uint64_t* slot_empty = bars + C::NSLOT;
    uint64_t* s_full = slot_empty + C::NSLOT;  // [2]
    uint64_t* p_ready = s_full + 2;    // [2] by S buffer: P_j is in TMEM over S_j
    uint64_t* o_done = p_ready + 2;    // [2] by S buffer: PV_j completed
    uint64_t* mma_drain = o_done + 2;  // every MMA the issuer launched has completed (exit drain)
    uint64_t* q_full = mma_drain + 1;  // QRES only
    uint8_t* qres = smem + C::OFF_Q;
    uint8_t* stage = smem + C::OFF_STAGE;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::N_BARS);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x >> 1, half = blockIdx.x & 1;
    const int split = blockIdx.y, slab = blockIdx.z;
    const int b = slab / a.n_kv_h, kvh = slab - b * a.n_kv_h;
    const long long row0 = ((long long)b * a.n_h + (long long)kvh * a.group) * a.T;
    const int r_begin = rt * BM;
    const int r_end = min(a.R, r_begin + BM);

    const int c_lo = a.kv_begin + split * a.kv_chunk;
    const int c_hi = min(a.s_k, c_lo + a.kv_chunk);
    int u_lo, u_hi;
    {
        int t0, t1;
        if (r_end - r_begin >= a.T || (r_end - 1) % a.T < r_begin % a.T) {
            t0 = 0;
            t1 = a.T - 1;
        } else {
            t0 = r_begin % a.T;
            t1 = (r_end - 1) % a.T;
        }
        int l0, h0, l1, h1;
        w_attended(t0, a, l0, h0);
        w_attended(t1, a, l1, h1);
        u_lo = l0;
        u_hi = h1;
    }
    const int k_lo = max(c_lo, u_lo), k_hi = min(c_hi, u_hi + 1);
    const int n_tiles_all = (k_hi > k_lo) ? (k_hi - k_lo + BN - 1) / BN : 0;
    // without a resident Q a block holds one tile (the host picks the resident
    // Q for longer spans), which its ring item order relies on
    const int n_tiles =
        (QRES || FMHA_IN_BOUNDS(n_tiles_all <= 1, kSiteWideTiles, a.status)) ? n_tiles_all : 0;

    // Producer item sequence: QK(0), then for each tile j: QK(j+1) (if any)
    // and V(j) -- the order the MMA warp consumes them in.  Item i -> kind
    // (1 QK item: Q chunk c and K chunk c, or with a resident Q K chunks 2c and
    // 2c + 1; 2 V item: V chunks 2c and 2c + 1 of this half), tile and c.
    const int n_items = n_tiles * C::TILE_ITEMS;
    auto item_of = [&](int i, int& kind, int& tile, int& c) {
        if (i < C::QK_ITEMS) {
            tile = 0;
            kind = 1;
            c = i;
            return;
        }
        const int r = i - C::QK_ITEMS;
        const int j = r / C::TILE_ITEMS, o = r - j * C::TILE_ITEMS;
        if (j < n_tiles - 1 && o < C::QK_ITEMS) {
            tile = j + 1;
            kind = 1;
            c = o;
        } else {
            tile = j;
            kind = 2;
            c = (j < n_tiles - 1) ? o - C::QK_ITEMS : o;
        }
    };
    uint64_t pol_kv = 0, pol_q = 0;
    int issued = 0;  // thread 0: items issued (0 .. issued-1)
    bool q_issued = false;
    auto issue_item = [&](int i) -> bool {
        int kind, tile, c;
        item_of(i, kind, tile, c);
        const int s = i % C::NSLOT;
        const int key = k_lo + tile * BN;
        const bool key_ok = key >= 0 && key < k_hi && k_hi <= a.s_k;
        const bool in_range = kind == 1 ? (key_ok && c >= 0 && c < C::QK_ITEMS && (QRES || (r_begin >= 0 && r_begin < a.R)))
                                        : (key_ok && c >= 0 && c < C::V_ITEMS);
        if (!FMHA_IN_BOUNDS(in_range && s >= 0 && s < C::NSLOT && slab < (int)gridDim.z, kSiteWideItem, a.status))
            return false;
        mbar_arrive_expect_tx(&slot_full[s], C::ITEM_BYTES);
        uint8_t* dst = ring + s * C::ITEM_BYTES;
        if (kind == 2) {
            tma_load_3d_hint(dst, &tmv, half * C::HALF + 2 * c * 64, key, slab, &slot_full[s], pol_kv);
            tma_load_3d_hint(dst + C::SLOT_BYTES, &tmv, half * C::HALF + (2 * c + 1) * 64, key, slab, &slot_full[s],
                             pol_kv);
        } else if (QRES) {
            tma_load_3d_hint(dst, &tmk, 2 * c * 64, key, slab, &slot_full[s], pol_kv);
            tma_load_3d_hint(dst + C::SLOT_BYTES, &tmk, (2 * c + 1) * 64, key, slab, &slot_full[s], pol_kv);
        } else {
            tma_load_3d_hint(dst, &tmq, c * 64, r_begin, slab, &slot_full[s], pol_q);
            tma_load_3d_hint(dst + C::SLOT_BYTES, &tmk, c * 64, key, slab, &slot_full[s], pol_kv);
        }
        return true;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(&p_ready[b2], 128);
            mbar_init(&o_done[b2], 1);
        }
        mbar_init(mma_drain, 1);
        if (QRES) mbar_init(q_full, 1);
        *abort_flag = 0;
        mbar_fence_init();
        // The first ring-full needs no free slot: start it before the block
        // barrier and the TMEM allocation.
        if (n_tiles > 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            pol_kv = l2_policy_evict_first();
            pol_q = l2_policy_evict_last();
            grid_dependency_wait();  // the preceding kernel's writes (Q, K, V) are visible
            if (QRES && FMHA_IN_BOUNDS(r_begin >= 0 && r_begin < a.R && slab < (int)gridDim.z, kSiteWideQ, a.status)) {
                mbar_arrive_expect_tx(q_full, C::Q_CHUNKS * C::Q_STRIDE);
                for (int c = 0; c < C::Q_CHUNKS; ++c)
                    tma_load_3d_hint(qres + c * C::Q_STRIDE, &tmq, c * 64, r_begin, slab, q_full, pol_q);
                q_issued = true;
            }
            for (int i = 0; i < min(C::NSLOT, n_items); ++i) {
                if (!issue_item(i)) break;
                ++issued;
            }
        }
    }
    if constexpr (C::Q_ROWS < 128) {
        // the last chunks' A operands run past the loaded Q rows into this tail
        if (warp >= 2) {
            constexpr int TAIL = C::Q_REGION - C::Q_CHUNKS * C::Q_STRIDE;
            uint4* tail = reinterpret_cast<uint4*>(qres + C::Q_CHUNKS * C::Q_STRIDE);
            for (int i = threadIdx.x - 64; i < TAIL / 16; i += 128) tail[i] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
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
            for (int i = C::NSLOT; issued == i && i < n_items; ++i) {
                const int s = i % C::NSLOT;
                if (!mbar_wait(&slot_empty[s], ((i / C::NSLOT) - 1) & 1, a.status)) break;
                if (!issue_item(i)) break;
                ++issued;
            }
            drain_ring(slot_full, C::NSLOT, issued, a.status);
            if (q_issued) mbar_wait(q_full, 0, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, 64 * C::V_GROUP, 1);
            const uint32_t ring_addr = smem_u32(ring), q_addr = smem_u32(qres);
            int item = 0;
            bool ok = true;
            if (QRES) ok = mbar_wait(q_full, 0, a.status);
            auto slot_take = [&](int& s) -> bool {
                s = item % C::NSLOT;
                if (!mbar_wait(&slot_full[s], (item / C::NSLOT) & 1, a.status)) return false;
                ++item;
                return true;
            };
            auto issue_qk = [&](int j) -> bool {
                const uint32_t d = tmem + (j & 1) * BN;
                for (int c = 0; c < C::QK_ITEMS; ++c) {
                    int sk;
                    if (!slot_take(sk)) return false;
                    if (!FMHA_IN_BOUNDS(sk >= 0 && sk < C::NSLOT, kSiteWideQKDesc, a.status)) return false;
                    tc_fence_after();
                    const uint32_t item_addr = ring_addr + sk * C::ITEM_BYTES;
#pragma unroll
                    for (int sub = 0; sub < (QRES ? 2 : 1); ++sub) {
                        const int ch = QRES ? 2 * c + sub : c;  // 64-column chunk of hd
                        // A: Q chunk ch (resident, or the item's first half); B: its K chunk
                        const uint32_t a_base = QRES ? q_addr + ch * C::Q_STRIDE : item_addr;
                        const uint32_t b_base = QRES ? item_addr + sub * C::SLOT_BYTES : item_addr + C::SLOT_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(b_base + kk * 32, 16, 1024);
                            tc_mma_f16(d, ad, bd, idesc_s, (ch > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(&slot_empty[sk]);
                }
                tc_commit(&s_full[j & 1]);
                return true;
            };
            ok = issue_qk(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !(ok = issue_qk(j + 1))) break;
                // One-tile blocks test V_j first: it lands while the softmax still
                // works on S_j, so only the P_j test remains once P_j is written
                // (with a resident Q the other order measured faster).
                if (QRES && !(ok = mbar_wait(&p_ready[j & 1], (j >> 1) & 1, a.status))) break;
                int sv[C::V_ITEMS];
                for (int c = 0; c < C::V_ITEMS && ok; ++c) {
                    ok = slot_take(sv[c]);
                    if (ok)
                        ok = FMHA_IN_BOUNDS(sv[c] < C::NSLOT && (c % C::V_GROUP_ITEMS == 0 || sv[c] == sv[c - 1] + 1),
                                            kSiteWideVSlots, a.status);
                }
                if (!ok) break;
                if (!QRES && !(ok = mbar_wait(&p_ready[j & 1], (j >> 1) & 1, a.status))) break;
                tc_fence_after();
                // A: P_j in TMEM over S_j (8 columns = 16 keys per MMA); B: each
                // group of V_GROUP 64-column V boxes, one chunk apart (the
                // descriptor's leading byte offset), into its columns of O.
                const uint32_t p_col = (j & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
#pragma unroll
                    for (int g = 0; g < C::V_CHUNKS / C::V_GROUP; ++g) {
                        const uint64_t bd = smem_desc_sw128(
                            ring_addr + sv[g * C::V_GROUP_ITEMS] * C::ITEM_BYTES + kk * 16 * 128, C::SLOT_BYTES, 1024);
                        tc_mma_f16_ts(tmem + C::O_COL + g * 64 * C::V_GROUP, tmem + p_col + kk * 8, bd, idesc_o,
                                      (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                for (int c = 0; c < C::V_ITEMS; ++c) tc_commit(&slot_empty[sv[c]]);
                tc_commit(&o_done[j & 1]);
            }
            // Exit drain: whatever the loop issued has completed before TMEM
            // and the operand buffers are released, even if a wait gave up.
            tc_commit(mma_drain);
            mbar_wait(mma_drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const int grow = r_begin + row;
        const bool valid = grow < r_end;
        int jlo = INT_MAX, jhi = -1;
        if (valid) {
            w_attended(grow % a.T, a, jlo, jhi);
            jlo = max(jlo, c_lo);
            jhi = min(jhi, c_hi - 1);
        }
        float m_ref = -INFINITY, l = 0.f, l_o = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[BN];
            const uint32_t s_col =
                FMHA_IN_BOUNDS((j & 1) * BN + BN <= C::O_COL, kSiteWideSCol, a.status) ? (j & 1) * BN : 0u;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                float v32[32];
                tmem_ld32(t_lane + s_col + c * 32, v32);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[c * 32 + i] = v32[i];
            }
            tmem_wait_ld();
            float alpha;
            uint32_t pk[BN / 2];
            softmax_row_tile<BN>(x, pk, k_lo + j * BN, jlo, jhi, a.scale_log2, m_ref, l, l_o, alpha);
            // P_j goes over S_j, whose QK the MMA issuer queued after PV_{j-2}, so
            // S_j being ready means that PV is done; a rescale of O needs PV_{j-1}.
            const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
            if (rescale && !mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.status)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) tmem_st32u(t_lane + s_col + c * 32, pk + c * 32);
            tmem_wait_st();
            if (rescale) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < C::HALF / 32; ++c) {
                    float ov[32];
                    tmem_ld32(t_lane + C::O_COL + c * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                    tmem_st32(t_lane + C::O_COL + c * 32, ov);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&p_ready[j & 1]);
        }
        if (ok && n_tiles > 0) ok = mbar_wait(&o_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        if (!ok) atomicOr(abort_flag, 1);
        tc_fence_after();
        float inv, lse;
        // query head of this row: kvh * G + (row within the slab) / T
        finish_row(m_ref, l, l_o,
                   (SINK && valid) ? sink_log2_of(a.sink, kvh * a.group + grow / a.T, a.n_h, a.status) : -INFINITY,
                   inv, lse);
        const bool have_o = ok && n_tiles > 0;
        float range = 1.f;
        if (a.to_partials && a.part_f16) {
            // fp16 keeps 11 significant bits only between 2^-14 and 65504: store
            // O * 2^-k with k = floor(log2 max|O|) - 14, so this half-row's
            // largest |O| lands in [2^14, 2^15), and record 2^k.  inv <= 1
            // (l >= 1: the key at the running max contributes 2^0), so with
            // |k| <= 113 neither inv * 2^-k nor 2^k overflows.
            float mx = 0.f;
            if (have_o) {
#pragma unroll 1
                for (int c = 0; c < C::HALF / 32; c += 4) {  // four loads in flight per wait
                    float o0[32], o1[32], o2[32], o3[32];
                    tmem_ld32(t_lane + C::O_COL + c * 32, o0);
                    tmem_ld32(t_lane + C::O_COL + (c + 1) * 32, o1);
                    tmem_ld32(t_lane + C::O_COL + (c + 2) * 32, o2);
                    tmem_ld32(t_lane + C::O_COL + (c + 3) * 32, o3);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(o0[i]), fabsf(o1[i])), fmaxf(fabsf(o2[i]), fabsf(o3[i]))));
                }
            }
            mx *= inv;
            const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;  // floor(log2 mx) for normal mx
            if (mx > 0.f && e < 128) {  // leave zero, inf and NaN rows as they are
                const int k = min(max(e - 14, -113), 113);
                inv *= __uint_as_float((uint32_t)(127 - k) << 23);  // 2^-k
                range = __uint_as_float((uint32_t)(127 + k) << 23);
            }
        }
        // This half of O -> shared memory (the drained ring) -> TMA store.
        const int pslab = split * (int)(a.rows_total / a.R) + slab;
        constexpr int kStageBytes = C::STAGE_BYTES;
        const int3 ext = make_int3(C::HD, a.R, (int)(a.to_partials ? gridDim.y * gridDim.z : gridDim.z));
        if constexpr (EPI == kEpiNvfp4) {
            // quantised in registers and stored per row; rows past the slab's
            // end and blocks that gave up store nothing
            named_barrier_sync(2, 128);
            const long long gr = row0 + grow;
            const bool row_ok = valid && *abort_flag == 0 &&
                                FMHA_IN_BOUNDS(gr >= 0 && gr < a.rows_total && (half == 0 || half == 1),
                                               kSiteWideFp4, a.status);
            const long long r = row_ok ? gr : 0;
            epilogue_nvfp4<C::HALF>(t_lane + C::O_COL, inv, row_ok, a.fp4.codes + r * (C::HD / 2) + half * (C::HALF / 2),
                                    a.fp4.scales + r * (C::HD / 16) + half * (C::HALF / 16), a.fp4.g, have_o);
        } else if (!a.to_partials)
            epilogue_tma_store<C::HALF, kOutBf16>(t_lane + C::O_COL, inv, row, stage, kStageBytes, &tmo,
                                                  half * C::HALF, r_begin, slab, ext, have_o, threadIdx.x == 64,
                                                  abort_flag, a.status);
        else if (a.part_f16)
            epilogue_tma_store<C::HALF, kOutF16>(t_lane + C::O_COL, inv, row, stage, kStageBytes, &tmo,
                                                 half * C::HALF, r_begin, pslab, ext, have_o, threadIdx.x == 64,
                                                 abort_flag, a.status);
        else
            epilogue_tma_store<C::HALF, kOutF32>(t_lane + C::O_COL, inv, row, stage, kStageBytes, &tmo,
                                                 half * C::HALF, r_begin, pslab, ext, have_o, threadIdx.x == 64,
                                                 abort_flag, a.status);
        const long long gr = row0 + grow;
        const bool row_ok = FMHA_IN_BOUNDS(!valid || (gr >= 0 && gr < a.rows_total && split < (int)gridDim.y),
                                           kSiteWideLse, a.status);
        if (valid && ok && row_ok && half == 0) {
            if (!a.to_partials)
                a.lse[gr] = lse;
            else
                a.lse_part[(long long)split * a.rows_total + gr] = lse;
        }
        if (valid && ok && row_ok && a.to_partials && a.part_f16 &&
            FMHA_IN_BOUNDS(half == 0 || half == 1, kSiteWideRange, a.status))
            a.range_part[((long long)split * a.rows_total + gr) * 2 + half] = range;
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

int tc_wide_kv_tile() { return WCfg::BN; }

// Q stays resident when a block may see two or more 128-key tiles, and then
// only 32 or 64 rows of each chunk are loaded if no KV head has more query rows.
int tc_wide_q_box_rows(const Problem& p, const SplitPlan& sp) {
    const int span = std::min(sp.kv_chunk, p.s_k);
    if (span <= WCfg::BN) return 128;
    return p.R <= 32 ? 32 : p.R <= 64 ? 64 : 128;
}

template <int EPI, bool QRES, int QROWS>
cudaError_t launch_wide_t(const TcLaunch& L, cudaStream_t stream) {
    using C = WCfgT<QRES, QROWS>;
    static std::atomic<bool> attr_set[128];  // set once per device; any host thread may set it
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_tc_wide_kernel<EPI, QRES, QROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 128) attr_set[dev] = true;
    }
    WideArgs a;
    a.o = static_cast<__nv_bfloat16*>(L.o);
    a.lse = L.lse;
    a.lse_part = L.lse_part;
    a.range_part = L.range_part;
    a.to_partials = L.to_partials ? 1 : 0;
    a.part_f16 = L.f16_partials ? 1 : 0;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((L.p.R + C::BM - 1) / C::BM), L.sp.n_splits, L.p.batch * L.p.n_kv_h);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_tc_wide_kernel<EPI, QRES, QROWS>, L.tmap_q, L.tmap_k, L.tmap_v, L.tmap_o, a);
}

template <int EPI>
cudaError_t launch_wide_q(const TcLaunch& L, cudaStream_t stream) {
    const int rows = tc_wide_q_box_rows(L.p, L.sp);
    if (rows == 32) return launch_wide_t<EPI, true, 32>(L, stream);
    if (rows == 64) return launch_wide_t<EPI, true, 64>(L, stream);
    const int span = std::min(L.sp.kv_chunk, L.p.s_k);
    return span > WCfg::BN ? launch_wide_t<EPI, true, 128>(L, stream) : launch_wide_t<EPI, false, 128>(L, stream);
}

cudaError_t launch_tc_wide(const TcLaunch& L, cudaStream_t stream) {
    if (L.fp4.codes && !L.to_partials) return launch_wide_q<kEpiNvfp4>(L, stream);
    return (L.sink && !L.to_partials) ? launch_wide_q<kEpiSink>(L, stream) : launch_wide_q<kEpiBf16>(L, stream);
}

}  // namespace fmha
