// status.cu -- the per-device status word that kernels set when a bounded wait
// gives up (or, in a checked build, when an index check fails).  Kernels
// receive its address as an argument; the C ABI reads and clears it in
// fmha_check_device_status().
#include <mutex>
#include "internal.h"
#include "ptx.cuh"

namespace fmha {
namespace {
__device__ unsigned g_status_word[2];  // [0] status bits, [1] first failed check site (checked builds)

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

static_assert(kStatusBitTimeout == kStatusBarrierTimeout && kStatusBitBounds == kStatusBoundsViolation,
              "host and device status bits agree");

const char* check_site_name(unsigned site) {
    switch (site) {
        case kSiteTcQLoad: return "row-tile kernel: Q box coordinates";
        case kSiteTcKLoad: return "row-tile kernel: K tile key / stage";
        case kSiteTcVLoad: return "row-tile kernel: V tile key / stage";
        case kSiteTcKDesc: return "row-tile kernel: K stage of the QK MMA";
        case kSiteTcVDesc: return "row-tile kernel: V stage / P buffer of the PV MMA";
        case kSiteTcSCol: return "row-tile kernel: TMEM columns of S";
        case kSiteTcPRow: return "row-tile kernel: P row";
        case kSiteTcLse: return "row-tile kernel: LSE index";
        case kSiteTcFp4: return "row-tile kernel: NVFP4 output row";
        case kSiteTcPTmem: return "row-tile kernel: TMEM columns of P (TS-form PV)";
        case kSiteWideItem: return "hd-512 kernel: producer item slot / coordinates";
        case kSiteWideQ: return "hd-512 kernel: resident Q box coordinates";
        case kSiteWideVSlots: return "hd-512 kernel: V slots of a PV MMA not consecutive";
        case kSiteWideQKDesc: return "hd-512 kernel: Q / K slot of the QK MMA";
        case kSiteWideSCol: return "hd-512 kernel: TMEM columns of S";
        case kSiteWidePRow: return "hd-512 kernel: P row";
        case kSiteWideLse: return "hd-512 kernel: LSE index";
        case kSiteWideRange: return "hd-512 kernel: range factor index";
        case kSiteWideFp4: return "hd-512 kernel: NVFP4 output row";
        case kSiteDecQRow: return "decode kernel: Q row";
        case kSiteDecQSmem: return "decode kernel: Q staging offset";
        case kSiteDecKVLoad: return "decode kernel: K/V stage key / slot";
        case kSiteDecLdsmK: return "decode kernel: ldmatrix address in the K tile";
        case kSiteDecLdsmQ: return "decode kernel: ldmatrix address in the Q rows";
        case kSiteDecLdsmV: return "decode kernel: ldmatrix address in the V tile";
        case kSiteDecComb: return "decode kernel: combine buffer index";
        case kSiteDecMl: return "decode kernel: (max, sum) index";
        case kSiteDecOut: return "decode kernel: output row";
        case kSiteMergePart: return "merge: partial index";
        case kSiteMergeRange: return "merge: range factor index";
        case kSiteMergeOut: return "merge: output row / column";
        case kSiteMergeSink: return "merge: sink head index";
        case kSiteMergeFp4: return "merge: NVFP4 output block";
        case kSiteEpiRow: return "epilogue: staging row";
        case kSiteEpiStore: return "epilogue: TMA store coordinates";
        case kSiteSink: return "sink head index";
        case kSiteSelfTest: return "index-check self-test";
        case kSitePairQLoad: return "two-row-tile kernel: Q box coordinates";
        case kSitePairKLoad: return "two-row-tile kernel: K tile key / stage";
        case kSitePairVLoad: return "two-row-tile kernel: V tile key / stage";
        case kSitePairKDesc: return "two-row-tile kernel: K stage of the QK MMAs";
        case kSitePairVDesc: return "two-row-tile kernel: V stage of the PV MMAs";
        case kSitePairLse: return "two-row-tile kernel: LSE index";
        case kSitePairFp4: return "two-row-tile kernel: NVFP4 output row";
        default: return "unknown site";
    }
}

bool checked_build() { return kCheckedBuild; }

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
// One thread runs an index check whose condition is false; nothing is
// accessed.  `never` is 0 at run time, so the compiler cannot fold the check.
__global__ void bounds_check_selftest_kernel(unsigned* status, int never) {
    if (threadIdx.x != 0) return;
    (void)FMHA_IN_BOUNDS(never != 0, kSiteSelfTest, status);
}
}  // namespace

cudaError_t launch_bounds_check_selftest(cudaStream_t stream) {
    unsigned* w = device_status_word();
    if (!w) return cudaErrorInvalidDevicePointer;
    bounds_check_selftest_kernel<<<1, 32, 0, stream>>>(w, 0);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    unsigned* w = device_status_word();
    if (!w) return cudaErrorInvalidDevicePointer;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(w, limit_ns);
    return cudaGetLastError();
}

}  // namespace fmha
