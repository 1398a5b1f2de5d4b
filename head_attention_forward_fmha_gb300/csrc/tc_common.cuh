// tc_common.cuh -- pieces shared by the tcgen05 kernels (tc_kernel.cu and
// tc_wide_kernel.cu): the per-row online-softmax step, the write of P into the
// K-major 128-byte-swizzled operand layout, and the TMA-store epilogue.
#pragma once
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace fmha {

// One row's S tile (raw dot products, x[BN]) -> un-normalised probabilities,
// written as packed bf16 pairs to p[BN / 2] (key 2i in the low half), while
// the running reference max m_ref and two running sums are updated (FA2
// online softmax: commit e4ee9fd of the nvfp4-megamoe-kernel pages,
// multi-tile C API part): l sums the fp32 probabilities (it gives the LSE),
// l_o the bf16-rounded ones that the P V product multiplies V by (O is
// divided by it, see finish_row).  Keys outside [jlo, jhi] are masked.
// sl2 = scale * log2(e).  The reference max only moves when the tile's max
// exceeds it by more than 8 (log2 units); then alpha = 2^(m_old - m_new) and
// the caller rescales O.  Probabilities are therefore <= 2^8.  The
// scale-and-subtract and both sums run on packed fp32 pairs.
// With LO = false the rounded sum is left to the caller (l_o is not touched):
// the row-tile kernel at hd 64 gets it from the tensor core, as one more column
// of O against a column of ones.
template <int BN, bool LO = true>
__device__ __forceinline__ void softmax_row_tile(float (&x)[BN], uint32_t (&p)[BN / 2], int key0, int jlo, int jhi,
                                                 float sl2, float& m_ref, float& l, float& l_o, float& alpha) {
    const bool full = key0 >= jlo && key0 + BN - 1 <= jhi;
    float mt, mul;
    if (sl2 > 0.f) {
        // max(sl2 * x) = sl2 * max(x): scale once, fold it into the exponent's FMA
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (full) {
#pragma unroll
            for (int i = 0; i < BN; ++i) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
        } else {
#pragma unroll
            for (int i = 0; i < BN; ++i) {
                const int key = key0 + i;
                x[i] = (key >= jlo && key <= jhi) ? x[i] : -INFINITY;
                m4[i & 3] = fmaxf(m4[i & 3], x[i]);
            }
        }
        const float mr = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        mt = (mr == -INFINITY) ? -INFINITY : mr * sl2;
        mul = sl2;
    } else {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < BN; ++i) {
            const int key = key0 + i;
            x[i] = (key >= jlo && key <= jhi) ? x[i] * sl2 : -INFINITY;
            m4[i & 3] = fmaxf(m4[i & 3], x[i]);
        }
        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        mul = 1.f;
    }
    alpha = 1.f;
    float m_new = m_ref;
    if (mt > m_ref + 8.f) {
        m_new = mt;
        alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
    }
    const float mu = (m_new == -INFINITY) ? 0.f : m_new;
    const uint64_t mul2 = f32x2(mul, mul), nmu2 = f32x2(-mu, -mu);
    uint64_t s2[2] = {0ull, 0ull}, r2[2] = {0ull, 0ull};  // {even, odd} key sums, two chains each
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) {
        float y0, y1;
        f32x2_split(fma_f32x2(f32x2(x[2 * i], x[2 * i + 1]), mul2, nmu2), y0, y1);
        y0 = ex2_approx(y0);  // masked keys: 2^-inf = 0
        y1 = ex2_approx(y1);
        const uint32_t pk = pack_bf16x2(y0, y1);
        p[i] = pk;
        s2[i & 1] = add_f32x2(s2[i & 1], f32x2(y0, y1));
        if constexpr (LO) r2[i & 1] = add_f32x2(r2[i & 1], f32x2(bf16_lo(pk), bf16_hi(pk)));
    }
    float a0, a1, b0, b1;
    f32x2_split(s2[0], a0, a1);
    f32x2_split(s2[1], b0, b1);
    l = l * alpha + ((a0 + a1) + (b0 + b1));
    if constexpr (LO) {
        float c0, c1, d0, d1;
        f32x2_split(r2[0], c0, c1);
        f32x2_split(r2[1], d0, d1);
        l_o = l_o * alpha + ((c0 + c1) + (d0 + d1));
    }
    m_ref = m_new;
}

// Row `row` of P (BN bf16 values, packed in pairs) into the A-operand layout:
// groups of 64 keys, each a 128-row x 128-byte K-major tile with the 128-byte
// swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8)).
template <int BN>
__device__ __forceinline__ void write_p_row(uint8_t* pbuf, int row, const uint32_t (&p)[BN / 2]) {
    constexpr int GROUPS = (BN + 63) / 64;
    constexpr int CHUNKS = (BN < 64 ? BN : 64) / 8;
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) {
        uint8_t* prow = pbuf + g * 128 * 128 + row * 128;
#pragma unroll
        for (int ch = 0; ch < CHUNKS; ++ch) {
            const uint32_t* pv = p + g * 32 + ch * 4;
            const uint4 pk = make_uint4(pv[0], pv[1], pv[2], pv[3]);
            *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = pk;
        }
    }
}

// Output formats of the epilogue.
enum OutMode : int {
    kOutBf16 = 0,  // final O
    kOutF32 = 1,   // split-KV partials, fp32 (the public partial layout)
    kOutF16 = 2,   // split-KV partials, fp16 (fmha_fwd's workspace at hd 512)
};

// Epilogue: this thread's O row (NCOL fp32 columns in TMEM from t_col) times
// `inv`, staged in shared memory in the TMA box layout and stored by TMA.
//   bf16 / fp16: boxes of 64 columns x 128 rows (128-byte rows, swizzled);
//   fp32: boxes of 32 columns x 128 rows.
// Box b of the stage sits at stage + b * 16 KB.  All 128 threads of the four
// softmax warps call this together (they meet at named barrier `bar_id`,
// which no other thread uses meanwhile); thread `leader` issues the stores (the
// TMA store of commit e4ee9fd: bulk_group, commit_group, wait_group.read 0).
// Boxes are stored as soon as they are staged, so the TMA reads box b while
// the threads stage box b + 1; only the last read is waited for.
// have_o must be uniform within each warp (tcgen05.ld is warp-collective);
// if any thread set *abort_flag, nothing is stored.  `ext` = the tensor map's
// (columns, rows, slabs) extents and `stage_bytes` the staging space, both
// only read by the index checks of a checked build.
template <int NCOL, int MODE>
__device__ __forceinline__ void epilogue_tma_store(uint32_t t_col, float inv, int row, uint8_t* stage,
                                                   int stage_bytes, const void* tmap, int col0, int row0_coord,
                                                   int slab_coord, int3 ext, bool have_o, bool leader,
                                                   const int* abort_flag, unsigned* status, int bar_id = 2) {
    constexpr bool F32 = MODE == kOutF32;
    constexpr int BOX_COLS = F32 ? 32 : 64;
    constexpr int CHUNKS_PER_BOX = BOX_COLS / 32;
    const bool row_ok = FMHA_IN_BOUNDS(row >= 0 && row < 128 && (NCOL / BOX_COLS) * 16384 <= stage_bytes,
                                       kSiteEpiRow, status);
#pragma unroll 1
    for (int bx = 0; bx < NCOL / BOX_COLS; ++bx) {
#pragma unroll
        for (int cc = 0; cc < CHUNKS_PER_BOX; ++cc) {
            const int c = bx * CHUNKS_PER_BOX + cc;
            float ov[32];
            if (have_o) {
                tmem_ld32(t_col + c * 32, ov);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] = 0.f;
            }
            uint8_t* rowp = stage + bx * 16384 + row * 128;
            if (!row_ok) continue;
            if constexpr (F32) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = make_float4(ov[q * 4] * inv, ov[q * 4 + 1] * inv, ov[q * 4 + 2] * inv,
                                                 ov[q * 4 + 3] * inv);
                    *reinterpret_cast<float4*>(rowp + ((q ^ (row & 7)) << 4)) = v;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 pk;
                    if constexpr (MODE == kOutF16) {
                        pk.x = pack_f16x2(ov[q * 8 + 0] * inv, ov[q * 8 + 1] * inv);
                        pk.y = pack_f16x2(ov[q * 8 + 2] * inv, ov[q * 8 + 3] * inv);
                        pk.z = pack_f16x2(ov[q * 8 + 4] * inv, ov[q * 8 + 5] * inv);
                        pk.w = pack_f16x2(ov[q * 8 + 6] * inv, ov[q * 8 + 7] * inv);
                    } else {
                        pk.x = pack_bf16x2(ov[q * 8 + 0] * inv, ov[q * 8 + 1] * inv);
                        pk.y = pack_bf16x2(ov[q * 8 + 2] * inv, ov[q * 8 + 3] * inv);
                        pk.z = pack_bf16x2(ov[q * 8 + 4] * inv, ov[q * 8 + 5] * inv);
                        pk.w = pack_bf16x2(ov[q * 8 + 6] * inv, ov[q * 8 + 7] * inv);
                    }
                    const int chunk = cc * 4 + q;
                    *reinterpret_cast<uint4*>(rowp + ((chunk ^ (row & 7)) << 4)) = pk;
                }
            }
        }
        fence_proxy_async_smem();
        named_barrier_sync(bar_id, 128);
        const int c0 = col0 + bx * BOX_COLS;
        if (leader && *abort_flag == 0 &&
            FMHA_IN_BOUNDS(c0 >= 0 && c0 % BOX_COLS == 0 && c0 + BOX_COLS <= ext.x && row0_coord >= 0 &&
                               row0_coord < ext.y && slab_coord >= 0 && slab_coord < ext.z,
                           kSiteEpiStore, status)) {
            tma_store_3d(tmap, c0, row0_coord, slab_coord, stage + bx * 16384);
            tma_store_commit();
        }
    }
    if (leader) tma_store_wait_read();
}

// NVFP4 epilogue: this thread's O row (NCOL fp32 columns in TMEM from t_col)
// times `inv`, quantised in registers (see nvfp4.cuh) 32 columns at a time:
// two blocks give 16 bytes of codes and two scale bytes, stored straight to
// global memory.  codes_row / scales_row point at this row's first block in
// [rows, hd / 2] and [rows, hd / 16]; a row outside the tensor (valid false)
// stores nothing but still takes part in the warp-collective TMEM loads.
template <int NCOL>
__device__ __forceinline__ void epilogue_nvfp4(uint32_t t_col, float inv, bool valid, uint8_t* codes_row,
                                               uint8_t* scales_row, float g, bool have_o) {
#pragma unroll 1
    for (int c = 0; c < NCOL / 32; ++c) {
        float ov[32];
        if (have_o) {
            tmem_ld32(t_col + c * 32, ov);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
        if (!valid) continue;
        uint32_t pk[4], sc[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float xb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) xb[i] = ov[b * 16 + i] * inv;
            uint32_t w[2];
            sc[b] = nvfp4_block(xb, g, w);
            pk[2 * b] = w[0];
            pk[2 * b + 1] = w[1];
        }
        *reinterpret_cast<uint4*>(codes_row + c * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint16_t*>(scales_row + c * 2) = (uint16_t)(sc[0] | (sc[1] << 8));
    }
}

}  // namespace fmha
