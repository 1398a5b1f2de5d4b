// merge_kernel.cu -- LSE merge of split-KV partial results.
//
// CURRENT_ISSUE.md ("UMMA FMHA -- Full Pipeline + Production"), "Next steps"
// item 4: O = sum_i exp(lse_i) O_i / sum_i exp(lse_i).  Evaluated with the
// exponents shifted by max_i lse_i:
//     LSE = M + ln sum_i exp(lse_i - M),   O = sum_i exp(lse_i - LSE) O_i.
// One warp per (output row, slice of up to 128 columns): the lanes first
// share the chunk weights (lane i holds chunk i's weight), then stream the
// slice of every partial with coalesced 8- or 16-byte loads, several chunks
// in flight, and write one bf16 slice; with at most four chunks every load is
// issued before any arithmetic.  Partials are fp32 (the public
// layout) or fp16 (the workspace fmha_fwd uses at hd 512, where partials are a
// large share of the traffic); an fp16 partial comes with a power-of-two range
// factor per (chunk, row, 256-column half) that keeps it inside fp16's range.
// Launched as a programmatic dependent: its blocks are scheduled while the
// split kernel runs and wait in grid_dependency_wait for the partials.
#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace fmha {
namespace {

constexpr int kMergeWarps = 8;

// VEC columns per lane: 16-byte loads of fp16 partials at hd >= 256, else
// 8- or 16-byte loads of fp32 partials.
template <int HD, typename PT>
struct MCfg {
    static constexpr int VEC = (sizeof(PT) == 2 && HD >= 256) ? 8 : (HD >= 128) ? 4 : 2;
    static constexpr int SLICE = 32 * VEC;  // columns per warp
    static constexpr int NSLICE = HD / SLICE;
};

template <int VEC>
__device__ __forceinline__ void load_vec(const float* p, float (&v)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else {
        const float2 u = __ldg(reinterpret_cast<const float2*>(p));
        v[0] = u.x; v[1] = u.y;
    }
}

template <int VEC>
__device__ __forceinline__ void load_vec(const __half* p, float (&v)[VEC]) {
    if constexpr (VEC == 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
            v[2 * q] = f.x;
            v[2 * q + 1] = f.y;
        }
    } else if constexpr (VEC == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u));
        v[0] = a.x; v[1] = a.y;
    }
}

// acc * inv -> V bf16 values at dst (RNE).
template <int V>
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const float (&acc)[V], float inv) {
    if constexpr (V == 8) {
        uint4 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(dst) = pk;
    } else if constexpr (V == 4) {
        uint2 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = pk;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

template <int HD, typename PT, bool SINK>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_lse_kernel(const PT* __restrict__ o_parts, const float* __restrict__ lse_parts,
                     const float* __restrict__ range_parts, int n_splits, long long rows,
                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse, const float* __restrict__ sink, int T,
                     int n_h, unsigned* status) {
    grid_dependency_wait();  // partials of the preceding split kernel are complete and visible
    launch_dependents();     // the next kernel on the stream may start its set-up
    using C = MCfg<HD, PT>;
    constexpr int V = C::VEC;
    const int lane = threadIdx.x & 31;
    const long long task = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (task >= rows * C::NSLICE) return;
    const long long row = task / C::NSLICE;
    const int col = (int)(task - row * C::NSLICE) * C::SLICE + lane * V;
    if constexpr (kCheckedBuild) {  // the warp leaves together: shuffles follow
        const bool in = FMHA_IN_BOUNDS(row >= 0 && row < rows && col >= 0 && col + V <= HD, kSiteMergeOut, status);
        if (!__all_sync(0xffffffffu, in)) return;
    }
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr float kLn2 = 0.693147180559945309f;

    // Up to kFast chunks: every load (LSEs, range factors, the partial
    // slices) is issued before any arithmetic, so the warp waits for one
    // memory round trip instead of two.
    constexpr int kFast = 4;
    if (n_splits <= kFast) {
        const float lv = (lane < n_splits) ? __ldg(lse_parts + (long long)lane * rows + row) : -INFINITY;
        float rv = 1.f;
        if constexpr (sizeof(PT) == 2) {
            if (lane < n_splits && FMHA_IN_BOUNDS(col / 256 < 2, kSiteMergeRange, status))
                rv = __ldg(range_parts + ((long long)lane * rows + row) * 2 + col / 256);
        }
        float pv[kFast][V];
#pragma unroll
        for (int i = 0; i < kFast; ++i) {
            if (i < n_splits) {
                load_vec<V>(o_parts + ((long long)i * rows + row) * HD + col, pv[i]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) pv[i][e] = 0.f;
            }
        }
        float m = lv;
#pragma unroll
        for (int sft = 16; sft > 0; sft >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sft));
        const int head = (int)((row / T) % n_h);
        const float sg = (SINK && FMHA_IN_BOUNDS(head >= 0 && head < n_h, kSiteMergeSink, status))
                             ? __ldg(sink + head)
                             : -INFINITY;
        m = fmaxf(m, sg);
        const float w_den = (m != -INFINITY && lane < n_splits) ? exp2f((lv - m) * kLog2e) : 0.f;
        const float w_mine = w_den * rv;
        float den = w_den;
#pragma unroll
        for (int sft = 16; sft > 0; sft >>= 1) den += __shfl_xor_sync(0xffffffffu, den, sft);
        if (SINK && sg != -INFINITY) den += exp2f((sg - m) * kLog2e);
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
        for (int i = 0; i < kFast; ++i) {
            const float wi = __shfl_sync(0xffffffffu, w_mine, i);  // 0 past n_splits
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] += wi * pv[i][e];
        }
        const float inv = (den > 0.f) ? 1.f / den : 0.f;
        store_row<V>(o + row * HD + col, acc, inv);
        if (lane == 0 && col == 0) lse[row] = (den > 0.f) ? m + log2f(den) * kLn2 : -INFINITY;
        return;
    }

    float mx = -INFINITY;
    for (int i = lane; i < n_splits; i += 32) mx = fmaxf(mx, __ldg(lse_parts + (long long)i * rows + row));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    // attention sink: one more term exp(sigma) of the denominator (no value)
    const int head = (int)((row / T) % n_h);
    const float sg = (SINK && FMHA_IN_BOUNDS(head >= 0 && head < n_h, kSiteMergeSink, status)) ? __ldg(sink + head)
                                                                                               : -INFINITY;
    mx = fmaxf(mx, sg);

    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (mx != -INFINITY) {
        for (int base = 0; base < n_splits; base += 32) {
            // lane i: weight of chunk base + i (0 for an empty chunk or past the end)
            const int mine = base + lane;
            const float w_den =
                (mine < n_splits) ? exp2f((__ldg(lse_parts + (long long)mine * rows + row) - mx) * kLog2e) : 0.f;
            float w_mine = w_den;  // weight of the stored values (times the range factor for fp16)
            if constexpr (sizeof(PT) == 2) {
                if (mine < n_splits && FMHA_IN_BOUNDS(col / 256 < 2, kSiteMergeRange, status))
                    w_mine *= __ldg(range_parts + ((long long)mine * rows + row) * 2 + col / 256);
            }
            float wsum = w_den;
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
            den += wsum;
            const int cnt = min(32, n_splits - base);
            if (!FMHA_IN_BOUNDS(cnt > 0 && base + cnt <= n_splits, kSiteMergePart, status)) break;
            int i = 0;
            for (; i + 4 <= cnt; i += 4) {
                float v0[V], v1[V], v2[V], v3[V];
                load_vec<V>(o_parts + ((long long)(base + i) * rows + row) * HD + col, v0);
                load_vec<V>(o_parts + ((long long)(base + i + 1) * rows + row) * HD + col, v1);
                load_vec<V>(o_parts + ((long long)(base + i + 2) * rows + row) * HD + col, v2);
                load_vec<V>(o_parts + ((long long)(base + i + 3) * rows + row) * HD + col, v3);
                const float w0 = __shfl_sync(0xffffffffu, w_mine, i);
                const float w1 = __shfl_sync(0xffffffffu, w_mine, i + 1);
                const float w2 = __shfl_sync(0xffffffffu, w_mine, i + 2);
                const float w3 = __shfl_sync(0xffffffffu, w_mine, i + 3);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] += w0 * v0[e] + w1 * v1[e] + w2 * v2[e] + w3 * v3[e];
            }
            for (; i < cnt; ++i) {
                float v0[V];
                load_vec<V>(o_parts + ((long long)(base + i) * rows + row) * HD + col, v0);
                const float w0 = __shfl_sync(0xffffffffu, w_mine, i);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] += w0 * v0[e];
            }
        }
    }
    if (SINK && sg != -INFINITY) den += exp2f((sg - mx) * kLog2e);
    const float inv = (den > 0.f) ? 1.f / den : 0.f;
    store_row<V>(o + row * HD + col, acc, inv);
    if (lane == 0 && col == 0) lse[row] = (den > 0.f) ? mx + log2f(den) * kLn2 : -INFINITY;
}

template <int HD, typename PT>
cudaError_t launch_t(const PT* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                     long long rows, void* o, float* lse, cudaStream_t stream, const float* sink, int T, int n_h,
                     unsigned* status) {
    const long long tasks = rows * MCfg<HD, PT>::NSLICE;
    const long long blocks = (tasks + kMergeWarps - 1) / kMergeWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (sink)
        return cudaLaunchKernelEx(&cfg, merge_lse_kernel<HD, PT, true>, o_parts, lse_parts, range_parts, n_splits,
                                  rows, static_cast<__nv_bfloat16*>(o), lse, sink, T, n_h, status);
    return cudaLaunchKernelEx(&cfg, merge_lse_kernel<HD, PT, false>, o_parts, lse_parts, range_parts, n_splits, rows,
                              static_cast<__nv_bfloat16*>(o), lse, sink, T, n_h, status);
}

template <int HD>
cudaError_t launch_hd(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                      long long rows, bool f16, void* o, float* lse, cudaStream_t stream, const float* sink, int T,
                      int n_h, unsigned* status) {
    if (f16) {
        if (HD != 512 || range_parts == nullptr) return cudaErrorInvalidValue;
        return launch_t<HD>(static_cast<const __half*>(o_parts), lse_parts, range_parts, n_splits, rows, o, lse,
                            stream, sink, T, n_h, status);
    }
    return launch_t<HD>(static_cast<const float*>(o_parts), lse_parts, nullptr, n_splits, rows, o, lse, stream,
                        sink, T, n_h, status);
}

// The merge with an NVFP4 final output: one thread per (row, 16-column
// block).  The weights are the bf16 merge's, exp(lse_i - max) (times the range
// factor of fp16 partials), one divide by their sum; the 16 merged values are
// quantised in registers (nvfp4.cuh).  Consecutive threads take consecutive
// blocks of a row, so each partial's row is read in contiguous 64-byte
// (fp32) or 32-byte (fp16) pieces.
template <int HD, typename PT>
__global__ void __launch_bounds__(256)
    merge_lse_nvfp4_kernel(const PT* __restrict__ o_parts, const float* __restrict__ lse_parts,
                           const float* __restrict__ range_parts, int n_splits, long long rows, Fp4Out fp4,
                           float* __restrict__ lse, unsigned* status) {
    grid_dependency_wait();  // partials of the preceding split kernel are complete and visible
    launch_dependents();
    constexpr int NBLK = HD / 16;
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr float kLn2 = 0.693147180559945309f;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * NBLK) return;
    const long long row = t / NBLK;
    const int blk = (int)(t - row * NBLK);
    const int col = blk * 16;
    if (!FMHA_IN_BOUNDS(row >= 0 && row < rows && col + 16 <= HD, kSiteMergeFp4, status)) return;
    float m = -INFINITY;
    for (int i = 0; i < n_splits; ++i) m = fmaxf(m, __ldg(lse_parts + (long long)i * rows + row));
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (m != -INFINITY) {
        for (int i = 0; i < n_splits; ++i) {
            const float w = exp2f((__ldg(lse_parts + (long long)i * rows + row) - m) * kLog2e);
            den += w;
            float f = w;
            if constexpr (sizeof(PT) == 2) f *= __ldg(range_parts + ((long long)i * rows + row) * 2 + col / 256);
            const PT* src = o_parts + ((long long)i * rows + row) * HD + col;
#pragma unroll
            for (int q = 0; q < 16; q += 8 / (int)sizeof(PT) * 2) {
                float v[8 / sizeof(PT) * 2];
                load_vec<8 / sizeof(PT) * 2>(src + q, v);
#pragma unroll
                for (int e = 0; e < (int)(8 / sizeof(PT) * 2); ++e) acc[q + e] += f * v[e];
            }
        }
    }
    const float inv = (den > 0.f) ? 1.f / den : 0.f;
    float xb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) xb[e] = acc[e] * inv;
    uint32_t pk[2];
    const uint32_t sc = nvfp4_block(xb, fp4.g, pk);
    *reinterpret_cast<uint2*>(fp4.codes + row * (HD / 2) + blk * 8) = make_uint2(pk[0], pk[1]);
    fp4.scales[row * NBLK + blk] = (uint8_t)sc;
    if (blk == 0) lse[row] = (den > 0.f) ? m + log2f(den) * kLn2 : -INFINITY;
}

template <int HD>
cudaError_t launch_nvfp4_hd(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                            long long rows, bool f16, Fp4Out fp4, float* lse, cudaStream_t stream, unsigned* status) {
    const long long threads = rows * (HD / 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (f16) {
        if (HD != 512 || range_parts == nullptr) return cudaErrorInvalidValue;
        return cudaLaunchKernelEx(&cfg, merge_lse_nvfp4_kernel<HD, __half>, static_cast<const __half*>(o_parts),
                                  lse_parts, range_parts, n_splits, rows, fp4, lse, status);
    }
    return cudaLaunchKernelEx(&cfg, merge_lse_nvfp4_kernel<HD, float>, static_cast<const float*>(o_parts), lse_parts,
                              range_parts, n_splits, rows, fp4, lse, status);
}

}  // namespace

cudaError_t launch_merge_nvfp4(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                               long long rows, int hd, bool f16, Fp4Out fp4, float* lse, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    unsigned* status = device_status_word();
    if (!status) return cudaErrorInvalidDevicePointer;
    switch (hd) {
        case 64: return launch_nvfp4_hd<64>(o_parts, lse_parts, range_parts, n_splits, rows, f16, fp4, lse, stream, status);
        case 128: return launch_nvfp4_hd<128>(o_parts, lse_parts, range_parts, n_splits, rows, f16, fp4, lse, stream, status);
        case 256: return launch_nvfp4_hd<256>(o_parts, lse_parts, range_parts, n_splits, rows, f16, fp4, lse, stream, status);
        case 512: return launch_nvfp4_hd<512>(o_parts, lse_parts, range_parts, n_splits, rows, f16, fp4, lse, stream, status);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                         long long rows, int hd, bool f16, void* o, float* lse, cudaStream_t stream,
                         const float* sink, int T, int n_h) {
    if (rows <= 0) return cudaSuccess;
    if (sink && (T < 1 || n_h < 1)) return cudaErrorInvalidValue;
    unsigned* status = device_status_word();
    if (!status) return cudaErrorInvalidDevicePointer;
    switch (hd) {
        case 64: return launch_hd<64>(o_parts, lse_parts, range_parts, n_splits, rows, f16, o, lse, stream, sink, T, n_h, status);
        case 128: return launch_hd<128>(o_parts, lse_parts, range_parts, n_splits, rows, f16, o, lse, stream, sink, T, n_h, status);
        case 256: return launch_hd<256>(o_parts, lse_parts, range_parts, n_splits, rows, f16, o, lse, stream, sink, T, n_h, status);
        case 512: return launch_hd<512>(o_parts, lse_parts, range_parts, n_splits, rows, f16, o, lse, stream, sink, T, n_h, status);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fmha
