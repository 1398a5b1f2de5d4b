// status.cu -- the per-device status word that kernels set when a bounded wait
// gives up.  Kernels receive its address as an argument; the C ABI reads and
// clears it in fmha_check_device_status().
#include <mutex>
#include "internal.h"
#include "ptx.cuh"

namespace fmha {
namespace {
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 128;
unsigned* g_addr[kMaxDevices] = {};
std::mutex g_mu;
}  // namespace

unsigned* device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_addr[dev] = static_cast<unsigned*>(p);
    }
    return g_addr[dev];
}

namespace {
// One thread waits on an mbarrier phase that nothing completes, through the
// same bounded wait the attention kernels use; it must give up after
// `limit_ns`, set the status bit and return.
__global__ void wait_timeout_selftest_kernel(unsigned* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, status, limit_ns);
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    unsigned* w = device_status_word();
    if (!w) return cudaErrorInvalidDevicePointer;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(w, limit_ns);
    return cudaGetLastError();
}

}  // namespace fmha
