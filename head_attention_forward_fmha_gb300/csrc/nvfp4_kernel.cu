// nvfp4_kernel.cu -- NVFP4 quantisation of fp32 rows on its own (the
// fmha_quantize_nvfp4 entry point): one thread per 16-element block, the same
// block quantiser (nvfp4.cuh) that the attention epilogues fuse, so that the
// codes they produce can be checked bit for bit against the oracle on the
// same fp32 inputs.
#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace fmha {
namespace {

__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const float* __restrict__ x, long long blocks,
                                                              float g, uint8_t* __restrict__ codes,
                                                              uint8_t* __restrict__ scales) {
    grid_dependency_wait();
    const long long blk = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= blocks) return;
    float v[16];
    const float4* src = reinterpret_cast<const float4*>(x + blk * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 u = __ldg(src + q);
        v[4 * q] = u.x;
        v[4 * q + 1] = u.y;
        v[4 * q + 2] = u.z;
        v[4 * q + 3] = u.w;
    }
    uint32_t pk[2];
    const uint32_t sc = nvfp4_block(v, g, pk);
    *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(pk[0], pk[1]);
    scales[blk] = (uint8_t)sc;
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const float* x, long long rows, int hd, float g, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream) {
    const long long blocks = rows * (hd / 16);
    if (blocks <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((blocks + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {programmatic_launch_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_nvfp4_kernel, x, blocks, g, codes, scales);
}

}  // namespace fmha
