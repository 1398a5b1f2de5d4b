// merge_kernel.cu -- LSE merge of split-KV partial results.
//
// CURRENT_ISSUE.md ("UMMA FMHA -- Full Pipeline + Production"), "Next steps"
// item 4: O = sum_i exp(lse_i) O_i / sum_i exp(lse_i).  Evaluated with the
// exponents shifted by max_i lse_i:
//     LSE = M + ln sum_i exp(lse_i - M),   O = sum_i exp(lse_i - LSE) O_i.
// One warp per output row; each lane owns HD/32 consecutive columns, so a
// warp reads one contiguous fp32 row of every partial (coalesced 8-32 B per
// lane) and writes one bf16 row.
#include "internal.h"
#include "ptx.cuh"

namespace fmha {
namespace {

constexpr int kMergeWarps = 8;

template <int HD>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_lse_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n_splits,
                     long long rows, __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
    constexpr int V = HD / 32;  // columns per lane: 2, 4, 8 or 16
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr float kLn2 = 0.693147180559945309f;

    float mx = -INFINITY;
    for (int i = lane; i < n_splits; i += 32) mx = fmaxf(mx, lse_parts[(long long)i * rows + row]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));

    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (mx != -INFINITY) {
        for (int i = 0; i < n_splits; ++i) {
            const float li = lse_parts[(long long)i * rows + row];
            const float w = exp2f((li - mx) * kLog2e);  // 0 for an empty partial
            den += w;
            const float* src = o_parts + ((long long)i * rows + row) * HD + lane * V;
            if constexpr (V == 2) {
                const float2 u = *reinterpret_cast<const float2*>(src);
                acc[0] += w * u.x;
                acc[1] += w * u.y;
            } else {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    const float4 u = *reinterpret_cast<const float4*>(src + e);
                    acc[e] += w * u.x;
                    acc[e + 1] += w * u.y;
                    acc[e + 2] += w * u.z;
                    acc[e + 3] += w * u.w;
                }
            }
        }
    }
    const float inv = (den > 0.f) ? 1.f / den : 0.f;
    __nv_bfloat16* dst = o + row * HD + lane * V;
#pragma unroll
    for (int e = 0; e < V; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) lse[row] = (den > 0.f) ? mx + log2f(den) * kLn2 : -INFINITY;
}

template <int HD>
cudaError_t launch_t(const float* o_parts, const float* lse_parts, int n_splits, long long rows, void* o,
                     float* lse, cudaStream_t stream) {
    const long long blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    merge_lse_kernel<HD><<<(unsigned)blocks, kMergeWarps * 32, 0, stream>>>(
        o_parts, lse_parts, n_splits, rows, static_cast<__nv_bfloat16*>(o), lse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_splits, long long rows, int hd,
                         void* o, float* lse, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    switch (hd) {
        case 64: return launch_t<64>(o_parts, lse_parts, n_splits, rows, o, lse, stream);
        case 128: return launch_t<128>(o_parts, lse_parts, n_splits, rows, o, lse, stream);
        case 256: return launch_t<256>(o_parts, lse_parts, n_splits, rows, o, lse, stream);
        case 512: return launch_t<512>(o_parts, lse_parts, n_splits, rows, o, lse, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fmha
