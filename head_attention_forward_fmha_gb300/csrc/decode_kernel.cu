// decode_kernel.cu -- split-KV attention forward for few query rows per KV head.
//
// One thread block handles RT (8, 16, or 32 at hd 64) query rows that share one KV head
// (the GQA group of a decode step, or a slice of a short prefill) and one
// chunk of the KV range.  K and V stream HBM -> shared memory through a
// multi-stage TMA pipeline (128-byte swizzled boxes of 64 head-dim columns)
// fed by one producer warp; four consumer warps each take 16 keys of every
// stage tile.
//
// Per 16-key block a warp computes S^T = K Q^T with mma.sync m16n8k16 (keys
// as the M dimension, so 8 query rows fill the N = 8 tile with no padding),
// applies scale and mask, updates its running max / sum (FA2 online softmax:
// commit e4ee9fd of the nvfp4-megamoe-kernel pages, multi-tile C API part),
// transposes the bf16 P fragment in registers (movmatrix) and accumulates
// O^T += V^T P^T, again with keys as the reduction dimension.  P stays
// un-normalised; the single divide by the running sum happens in the
// epilogue, after the warps' partial states are merged through shared memory.
//
// Output: bf16 O and fp32 LSE directly, or fp32 partials (O_i, lse_i) of this
// chunk for the LSE merge (CURRENT_ISSUE.md, "Next steps" item 4).
#include <algorithm>
#include <cfloat>
#include <climits>
#include <atomic>
#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace fmha {
namespace {

template <int HD, int NB>
struct DCfg {
    static constexpr int RT = 8 * NB;                 // query rows per CTA
    static constexpr int KW = (HD <= 128) ? 4 : 2;    // key groups (16 keys each)
    static constexpr int DW = 4 / KW;                 // warps splitting head dim in PV
    static constexpr int KT = 16 * KW;                // keys per stage
    static constexpr int HDW = HD / DW;               // head-dim columns per warp in PV
    static constexpr int NCW = 4;                     // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;    // + one producer warp
    static constexpr int NBOX = HD / 64;              // 64-column (128-byte) TMA boxes per tile
    static constexpr int BOX_BYTES = KT * 128;
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile + V tile
    static constexpr int STAGES = (STAGE_BYTES <= 16384) ? 6 : 3;
    static constexpr int Q_STRIDE = HD * 2 + 16;      // padded row: conflict-free ldmatrix
    static constexpr int Q_BYTES = RT * Q_STRIDE;
    static constexpr int COMB_BYTES = KW * RT * HD * 4;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + Q_BYTES + 2 * STAGES * 8 + KW * RT * 8 + 16;
    static_assert(COMB_BYTES <= STAGES * STAGE_BYTES, "combine buffer reuses the stage ring");
    static_assert(BOX_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
};

struct DecodeArgs {
    const __nv_bfloat16* q;
    __nv_bfloat16* o;
    float* lse;
    float* o_part;
    float* lse_part;
    int to_partials;
    int n_h, n_kv_h, T, s_k, group, R, window, causal;
    float scale_log2;
    int kv_begin, kv_chunk;
    long long rows_total;  // batch * n_h * T
    unsigned* status;
    const float* sink;     // [n_h] sink logits (final output only) or NULL
};

__device__ __forceinline__ void attended(int t, const DecodeArgs& a, int& lo, int& hi) {
    const int p = a.s_k - a.T + t;
    lo = 0;
    hi = a.s_k - 1;
    if (a.causal) hi = min(hi, p);
    if (a.window > 0) lo = max(lo, p - a.window + 1);
}

// fp4: the NVFP4 output buffers, read by the kEpiNvfp4 instantiation only.  They
// are a parameter of their own: as a DecodeArgs field they changed ptxas's
// register allocation of the bf16 instantiations (hd 128 with 16 rows went from
// 147 to 128 registers and ran 11 % slower at s_k 32768).
template <int HD, int NB, int EPI>
__global__ void __launch_bounds__(DCfg<HD, NB>::THREADS)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                          const DecodeArgs a, const Fp4Out fp4) {
    using C = DCfg<HD, NB>;
    launch_dependents();  // the merge grid may be scheduled now; it waits for this grid's results
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* qs = smem + C::STAGES * C::STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(qs + C::Q_BYTES);
    uint64_t* empty = full + C::STAGES;
    float2* ml = reinterpret_cast<float2*>(empty + C::STAGES);  // [KW][RT] (max, sum) per key group
    int* abort_flag = reinterpret_cast<int*>(ml + C::KW * C::RT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x, split = blockIdx.y, slab = blockIdx.z;  // slab = b * n_kv_h + kvh
    const int b = slab / a.n_kv_h, kvh = slab - b * a.n_kv_h;
    const long long row0 = ((long long)b * a.n_h + (long long)kvh * a.group) * a.T;
    const int r_begin = rt * C::RT;
    const int r_end = min(a.R, r_begin + C::RT);

    // Keys this CTA visits: its chunk, intersected with the union of its rows' ranges.
    const int c_lo = a.kv_begin + split * a.kv_chunk;
    const int c_hi = min(a.s_k, c_lo + a.kv_chunk);
    int u_lo = INT_MAX, u_hi = -1;
    for (int r = r_begin; r < r_end; ++r) {
        int lo, hi;
        attended(r % a.T, a, lo, hi);
        u_lo = min(u_lo, lo);
        u_hi = max(u_hi, hi);
    }
    const int k_lo = max(c_lo, u_lo), k_hi = min(c_hi, u_hi + 1);
    const int n_tiles = (k_hi > k_lo) ? (k_hi - k_lo + C::KT - 1) / C::KT : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::NCW);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    grid_dependency_wait();  // every global access below follows the preceding kernel

    // ------------------------------------------------------------ producer
    if (warp == C::NCW) {
        if (lane == 0 && n_tiles > 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int it = 0; it < n_tiles; ++it) {
                const int s = it % C::STAGES;
                if (it >= C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, a.status)) break;
                const int key = k_lo + it * C::KT;
                if (!FMHA_IN_BOUNDS(key >= 0 && key < k_hi && k_hi <= a.s_k && s < C::STAGES &&
                                        slab < (int)gridDim.z,
                                    kSiteDecKVLoad, a.status))
                    break;
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                uint8_t* kst = stages + s * C::STAGE_BYTES;
                uint8_t* vst = kst + C::TILE_BYTES;
#pragma unroll
                for (int c = 0; c < C::NBOX; ++c) {
                    tma_load_3d_hint(kst + c * C::BOX_BYTES, &tmk, c * 64, key, slab, &full[s], pol);
                    tma_load_3d_hint(vst + c * C::BOX_BYTES, &tmv, c * 64, key, slab, &full[s], pol);
                }
                ++issued;
            }
            // Exit drain: the stages this warp loaded have landed before the
            // block may exit, even if the consumers gave up on their waits.
            drain_ring(full, C::STAGES, issued, a.status);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int kw = warp / C::DW, dw = warp - (warp / C::DW) * C::DW;

    // Q rows of this tile -> shared memory (zero rows past the end).
    for (int i = threadIdx.x; i < C::RT * (HD / 8); i += C::NCW * 32) {
        const int r = i / (HD / 8), c8 = i - r * (HD / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r_begin + r < r_end &&
            FMHA_IN_BOUNDS(row0 + r_begin + r >= 0 && row0 + r_begin + r < a.rows_total, kSiteDecQRow, a.status))
            val = *reinterpret_cast<const uint4*>(a.q + (row0 + r_begin + r) * HD + c8 * 8);
        if (FMHA_IN_BOUNDS(r * C::Q_STRIDE + c8 * 16 + 16 <= C::Q_BYTES, kSiteDecQSmem, a.status))
            *reinterpret_cast<uint4*>(qs + r * C::Q_STRIDE + c8 * 16) = val;
    }

    // Attended key interval of each accumulator row this thread holds
    // (rows nb*8 + 2*(lane%4) + i), clipped to the chunk.
    int jlo[NB][2], jhi[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = r_begin + nb * 8 + 2 * (lane & 3) + i;
            int lo = INT_MAX, hi = -1;
            if (r < r_end) {
                attended(r % a.T, a, lo, hi);
                lo = max(lo, c_lo);
                hi = min(hi, c_hi - 1);
            }
            jlo[nb][i] = lo;
            jhi[nb][i] = hi;
        }

    float m[NB][2], l[NB][2];
    float o[C::HDW / 16][NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        m[nb][0] = m[nb][1] = -INFINITY;
        l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
        for (int db = 0; db < C::HDW / 16; ++db) o[db][nb][0] = o[db][nb][1] = o[db][nb][2] = o[db][nb][3] = 0.f;
    }

    named_barrier_sync(1, C::NCW * 32);  // Q staged

    const uint32_t qs_addr = smem_u32(qs);
    const uint32_t q_addr = qs_addr + ((lane & 7) + (NB >= 2 ? 8 * (lane >> 4) : 0)) * C::Q_STRIDE +
                            ((lane >> 3) & 1) * 16;
    const int k_row = 16 * kw + (lane & 15);
    const int k_c8 = lane >> 4;
    const int v_row = 16 * kw + (lane & 7) + 8 * (lane >> 4);
    const int v_c8 = (lane >> 3) & 1;
    bool ok = true;

    for (int it = 0; it < n_tiles; ++it) {
        const int s = it % C::STAGES;
        if (!mbar_wait(&full[s], (it / C::STAGES) & 1, a.status)) {
            ok = false;
            break;
        }
        const uint32_t kst = smem_u32(stages + s * C::STAGE_BYTES);
        const uint32_t vst = kst + C::TILE_BYTES;

        // S^T (16 keys x RT rows) = K Q^T
        float sc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            const int d = 16 * kk + 8 * k_c8;
            uint32_t ka = kst + (d >> 6) * C::BOX_BYTES + k_row * 128 + ((((d & 63) >> 3) ^ (k_row & 7)) << 4);
            if (!FMHA_IN_BOUNDS(ka >= kst && ka + 16 <= kst + C::TILE_BYTES, kSiteDecLdsmK, a.status)) ka = kst;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(ka, a0, a1, a2, a3);
            uint32_t qa = q_addr + kk * 32;
            if (!FMHA_IN_BOUNDS(qa >= qs_addr && qa + 16 <= qs_addr + C::Q_BYTES, kSiteDecLdsmQ, a.status))
                qa = qs_addr;
            uint32_t bq[NB][2];
            if constexpr (NB == 1) {
                ldsm_x2(qa, bq[0][0], bq[0][1]);
            } else {
                ldsm_x4(qa, bq[0][0], bq[0][1], bq[1][0], bq[1][1]);
            }
            if constexpr (NB == 4) {  // rows 16..31
                uint32_t qb = qa + 16 * C::Q_STRIDE;
                if (!FMHA_IN_BOUNDS(qb + 16 <= qs_addr + C::Q_BYTES, kSiteDecLdsmQ, a.status)) qb = qs_addr;
                ldsm_x4(qb, bq[2][0], bq[2][1], bq[3][0], bq[3][1]);
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sc[nb], a0, a1, a2, a3, bq[nb][0], bq[nb][1]);
        }

        // scale + mask, online softmax (log2 domain)
        const int j0 = k_lo + it * C::KT + 16 * kw + (lane >> 2);
        const int j1 = j0 + 8;
        uint32_t pb[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float mx[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float x0 = (j0 >= jlo[nb][i] && j0 <= jhi[nb][i]) ? sc[nb][i] * a.scale_log2 : -INFINITY;
                const float x1 = (j1 >= jlo[nb][i] && j1 <= jhi[nb][i]) ? sc[nb][2 + i] * a.scale_log2 : -INFINITY;
                sc[nb][i] = x0;
                sc[nb][2 + i] = x1;
                mx[i] = fmaxf(x0, x1);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 4));
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 8));
                mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 16));
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float mn = fmaxf(m[nb][i], mx[i]);
                const float mu = (mn == -INFINITY) ? 0.f : mn;
                const float alpha = exp2f(m[nb][i] - mu);
                m[nb][i] = mn;
                const float p0 = exp2f(sc[nb][i] - mu);
                const float p1 = exp2f(sc[nb][2 + i] - mu);
                l[nb][i] = l[nb][i] * alpha + p0 + p1;
                sc[nb][i] = p0;
                sc[nb][2 + i] = p1;
#pragma unroll
                for (int db = 0; db < C::HDW / 16; ++db) {
                    o[db][nb][i] *= alpha;
                    o[db][nb][2 + i] *= alpha;
                }
            }
            pb[nb][0] = movmatrix_t(pack_bf16x2(sc[nb][0], sc[nb][1]));
            pb[nb][1] = movmatrix_t(pack_bf16x2(sc[nb][2], sc[nb][3]));
        }

        // O^T (head-dim x RT rows) += V^T P^T
#pragma unroll
        for (int db = 0; db < C::HDW / 16; ++db) {
            const int d = dw * C::HDW + 16 * db + 8 * v_c8;
            uint32_t va = vst + (d >> 6) * C::BOX_BYTES + v_row * 128 + ((((d & 63) >> 3) ^ (v_row & 7)) << 4);
            if (!FMHA_IN_BOUNDS(va >= vst && va + 16 <= vst + C::TILE_BYTES, kSiteDecLdsmV, a.status)) va = vst;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(va, a0, a1, a2, a3);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[db][nb], a0, a1, a2, a3, pb[nb][0], pb[nb][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------------------------------ epilogue
    // Row sums: reduce the per-lane partial sums of the 8 lanes sharing a row.
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            l[nb][i] += __shfl_xor_sync(0xffffffffu, l[nb][i], 4);
            l[nb][i] += __shfl_xor_sync(0xffffffffu, l[nb][i], 8);
            l[nb][i] += __shfl_xor_sync(0xffffffffu, l[nb][i], 16);
        }
    if (!ok) atomicOr(abort_flag, 1);
    named_barrier_sync(1, C::NCW * 32);  // every warp is done with the stage ring
    if (*abort_flag) return;

    if (dw == 0 && lane < 4) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int mi = kw * C::RT + nb * 8 + 2 * lane + i;
                if (FMHA_IN_BOUNDS(mi >= 0 && mi < C::KW * C::RT, kSiteDecMl, a.status))
                    ml[mi] = make_float2(m[nb][i], l[nb][i]);
            }
    }
    named_barrier_sync(1, C::NCW * 32);

    // Rescale this warp's O to the row maximum over all key groups and park it.
    float* comb = reinterpret_cast<float*>(stages);  // [KW][RT][HD]
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = nb * 8 + 2 * (lane & 3) + i;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::KW; ++w) M = fmaxf(M, ml[w * C::RT + r].x);
            const float f = exp2f(m[nb][i] - ((M == -INFINITY) ? 0.f : M));
#pragma unroll
            for (int db = 0; db < C::HDW / 16; ++db) {
                const int d = dw * C::HDW + 16 * db + (lane >> 2);
                const int ci = (kw * C::RT + r) * HD + d;
                if (!FMHA_IN_BOUNDS(ci >= 0 && ci + 8 < C::KW * C::RT * HD, kSiteDecComb, a.status)) continue;
                comb[ci] = o[db][nb][i] * f;
                comb[ci + 8] = o[db][nb][2 + i] * f;
            }
        }
    named_barrier_sync(1, C::NCW * 32);

    // Sum the key groups, divide once by the running sum (plus the sink), write out.
    if constexpr (EPI == kEpiNvfp4) {
        // NVFP4 O: one 16-column block per item, quantised in registers (nvfp4.cuh)
        for (int item = threadIdx.x; item < C::RT * (HD / 16); item += C::NCW * 32) {
            const int r = item / (HD / 16), b16 = item - r * (HD / 16);
            if (r_begin + r >= r_end) continue;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::KW; ++w) M = fmaxf(M, ml[w * C::RT + r].x);
            const float Mu = (M == -INFINITY) ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < C::KW; ++w) L += ml[w * C::RT + r].y * exp2f(ml[w * C::RT + r].x - Mu);
            const long long grow = row0 + r_begin + r;
            float inv, lse;
            finish_row(M, L, -INFINITY, inv, lse);
            float xb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) xb[e] = 0.f;
#pragma unroll
            for (int w = 0; w < C::KW; ++w) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 u = reinterpret_cast<const float4*>(comb + (w * C::RT + r) * HD + b16 * 16)[q4];
                    xb[4 * q4] += u.x;
                    xb[4 * q4 + 1] += u.y;
                    xb[4 * q4 + 2] += u.z;
                    xb[4 * q4 + 3] += u.w;
                }
            }
            if (!FMHA_IN_BOUNDS(grow >= 0 && grow < a.rows_total && split < (int)gridDim.y, kSiteDecOut, a.status))
                continue;
#pragma unroll
            for (int e = 0; e < 16; ++e) xb[e] *= inv;
            uint32_t pk[2];
            const uint32_t sc = nvfp4_block(xb, fp4.g, pk);
            *reinterpret_cast<uint2*>(fp4.codes + grow * (HD / 2) + b16 * 8) = make_uint2(pk[0], pk[1]);
            fp4.scales[grow * (HD / 16) + b16] = (uint8_t)sc;
            if (b16 == 0) a.lse[grow] = lse;
        }
        return;
    }
    for (int item = threadIdx.x; item < C::RT * (HD / 8); item += C::NCW * 32) {
        const int r = item / (HD / 8), d8 = item - r * (HD / 8);
        if (r_begin + r >= r_end) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::KW; ++w) M = fmaxf(M, ml[w * C::RT + r].x);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < C::KW; ++w) L += ml[w * C::RT + r].y * exp2f(ml[w * C::RT + r].x - Mu);
        const long long grow = row0 + r_begin + r;
        float inv, lse;
        // query head of this row: kvh * G + (row within the slab) / T
        finish_row(M, L,
                   (EPI == kEpiSink) ? sink_log2_of(a.sink, kvh * a.group + (r_begin + r) / a.T, a.n_h, a.status)
                                     : -INFINITY,
                   inv, lse);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int w = 0; w < C::KW; ++w) {
            const float4* src = reinterpret_cast<const float4*>(comb + (w * C::RT + r) * HD + d8 * 8);
            const float4 u0 = src[0], u1 = src[1];
            acc[0] += u0.x; acc[1] += u0.y; acc[2] += u0.z; acc[3] += u0.w;
            acc[4] += u1.x; acc[5] += u1.y; acc[6] += u1.z; acc[7] += u1.w;
        }
        if (!FMHA_IN_BOUNDS(grow >= 0 && grow < a.rows_total && split < (int)gridDim.y, kSiteDecOut, a.status))
            continue;
        if (!a.to_partials) {
            uint4 pk;
            pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
            pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4*>(a.o + grow * HD + d8 * 8) = pk;
            if (d8 == 0) a.lse[grow] = lse;
        } else {
            const long long prow = (long long)split * a.rows_total + grow;
            float4* dst = reinterpret_cast<float4*>(a.o_part + prow * HD + d8 * 8);
            dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
            if (d8 == 0) a.lse_part[prow] = lse;
        }
    }
}

template <int HD, int NB, int EPI>
cudaError_t launch_t(const DecodeLaunch& L, cudaStream_t stream) {
    using C = DCfg<HD, NB>;
    auto kern = decode_splitkv_kernel<HD, NB, EPI>;
    static std::atomic<bool> attr_set[128];  // set once per device; any host thread may set it
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 128) attr_set[dev] = true;
    }
    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(L.q);
    a.o = static_cast<__nv_bfloat16*>(L.o);
    a.lse = L.lse;
    a.o_part = L.o_part;
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
    const int row_tiles = (L.p.R + C::RT - 1) / C::RT;
    dim3 grid(row_tiles, L.sp.n_splits, L.p.batch * L.p.n_kv_h);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_k, L.tmap_v, a, L.fp4);
}

}  // namespace

int decode_kv_tile(int hd) { return hd <= 128 ? 64 : 32; }

// 32 rows at hd 64 when a KV head has more than 16 and its rows attend at
// least 16384 keys: each block then reads its K/V chunk for twice the rows
// (registers still allow two blocks per SM).  Measured on MHA hd 64 T 32:
// s_k 32768 121.6 -> 110.1 us, but s_k 4096 20.3 -> 23.6 us and s_k 512
// 7.4 -> 11.0 us, where half as many blocks leave the SMs short of work.
int decode_rows_per_cta(const Problem& p) {
    const long long span = p.window > 0 ? std::min<long long>(p.s_k, (long long)p.window + p.T) : p.s_k;
    if (p.hd == 64 && p.R > 16 && span >= 16384) return 32;
    return (p.R > 8 && p.hd <= 256) ? 16 : 8;
}

template <int EPI>
cudaError_t launch_hd(const DecodeLaunch& L, cudaStream_t stream) {
    const int rows = decode_rows_per_cta(L.p);
    const bool two = rows == 16;
    switch (L.p.hd) {
        case 64:
            return rows == 32 ? launch_t<64, 4, EPI>(L, stream)
                              : two ? launch_t<64, 2, EPI>(L, stream) : launch_t<64, 1, EPI>(L, stream);
        case 128: return two ? launch_t<128, 2, EPI>(L, stream) : launch_t<128, 1, EPI>(L, stream);
        case 256: return two ? launch_t<256, 2, EPI>(L, stream) : launch_t<256, 1, EPI>(L, stream);
        case 512: return launch_t<512, 1, EPI>(L, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream) {
    if (L.fp4.codes && !L.to_partials) return launch_hd<kEpiNvfp4>(L, stream);
    return (L.sink && !L.to_partials) ? launch_hd<kEpiSink>(L, stream) : launch_hd<kEpiBf16>(L, stream);
}

}  // namespace fmha
