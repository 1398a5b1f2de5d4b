// status.cu -- the per-device status word that kernels set when a bounded wait
// gives up.  Kernels receive its address as an argument; the C ABI reads and
// clears it in fmha_check_device_status().
#include <mutex>
#include "internal.h"

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

}  // namespace fmha
