// internal.h -- host-side interfaces between the C ABI (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fmha {

// Final-output epilogue of a kernel (a compile-time choice, so that the
// plain kernels carry none of the other code): bf16 O, bf16 O with an
// attention sink in the softmax denominator, or NVFP4 O (16-element blocks
// of E2M1 codes with E4M3 scales, see nvfp4.cuh).
enum Epilogue : int { kEpiBf16 = 0, kEpiSink = 1, kEpiNvfp4 = 2 };

// NVFP4 output buffers: codes [rows, hd / 2], scales [rows, hd / 16], global scale g.
struct Fp4Out {
    uint8_t* codes;
    uint8_t* scales;
    float g;
};

// One attention problem, validated by the API layer.
struct Problem {
    int batch, n_h, n_kv_h, T, s_k, hd;
    int window, causal;
    float scale;
    int group;  // n_h / n_kv_h
    int R;      // query rows sharing one KV head: group * T
};

// Split-KV layout: chunk i covers keys [kv_begin + i*kv_chunk, ... + kv_chunk).
struct SplitPlan {
    int kv_begin, kv_chunk, n_splits;
};

// ---- decode / small-row kernel (decode_kernel.cu) -------------------------
struct DecodeLaunch {
    const void* q;
    void* o;           // bf16 output (n_splits == 1 and !to_partials)
    float* lse;
    float* o_part;     // fp32 partial outputs (to_partials)
    float* lse_part;
    bool to_partials;
    const float* sink;  // [n_h] attention-sink logits or NULL; applied when !to_partials
    Fp4Out fp4;         // NVFP4 final output when fp4.codes != NULL (no sink, !to_partials)
    CUtensorMap tmap_k, tmap_v;
    Problem p;
    SplitPlan sp;
    unsigned* status;
};
int decode_kv_tile(int hd);                  // keys per pipeline stage (TMA box rows)
int decode_rows_per_cta(const Problem& p);   // query rows per thread block
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream);

// ---- 128-row tensor-core kernel (tc_kernel.cu) ----------------------------
struct TcLaunch {
    void* o;
    float* lse;
    void* o_part;       // fp32, or fp16 when f16_partials
    float* lse_part;
    float* range_part;  // fp16 partials only: [n_splits, rows, 2] power-of-two factor per row half
    bool to_partials;
    const float* sink;  // [n_h] attention-sink logits or NULL; applied when !to_partials
    bool f16_partials;  // hd-512 kernel only
    Fp4Out fp4;         // NVFP4 final output when fp4.codes != NULL (no sink, !to_partials)
    bool ss_pv;         // row-tile kernel: P through shared memory (SS-form PV) instead of TMEM (TS form)
    CUtensorMap tmap_q, tmap_k, tmap_v;
    // bf16 O [slabs, R, hd] (box 64 x 128), fp32 partials [n_splits*slabs, R, hd]
    // (box 32 x 128) or fp16 partials (box 64 x 128)
    CUtensorMap tmap_o;
    Problem p;
    SplitPlan sp;
    unsigned* status;
};
constexpr int kTcRows = 128;                 // query rows per thread block (MMA M)
bool tc_supports(int hd);
int tc_kv_tile(int hd);                      // keys per tile (TMA box rows of K and V)
cudaError_t launch_tc(const TcLaunch& L, cudaStream_t stream);
// hd = 512 variant (tc_wide_kernel.cu): two thread blocks per row tile, one
// per half of the head dim of O.
int tc_wide_kv_tile();
// Rows of the Q map's TMA box for the hd-512 kernel: 32 or 64 where its blocks
// keep a compact resident Q (at most that many query rows per KV head), else
// kTcRows.
int tc_wide_q_box_rows(const Problem& p, const SplitPlan& sp);
cudaError_t launch_tc_wide(const TcLaunch& L, cudaStream_t stream);
// Two 128-row tiles per thread block (tc_pair_kernel.cu), hd 64 and 128: for
// KV heads with more than 128 query rows; the same Q, O, K and V maps as
// launch_tc (K/V boxes of tc_pair_kv_tile() keys); bf16 O or fp32 partials, no
// NVFP4.
bool tc_pair_supports(int hd);
int tc_pair_kv_tile();
cudaError_t launch_tc_pair(const TcLaunch& L, cudaStream_t stream);

// Launch attribute shared by every kernel here: programmatic stream
// serialization, so a kernel may be scheduled while its predecessor on the
// stream finishes; each kernel runs its set-up (barriers, tensor memory,
// descriptor prefetch) and then executes griddepcontrol.wait before its first
// global memory access, which restores the full dependency.
inline cudaLaunchAttribute programmatic_launch_attr() {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

// ---- split-KV merge (merge_kernel.cu) -------------------------------------
// sink: [n_h] attention-sink logits added once to the merged denominator
// (NULL: none); row r belongs to head (r / T) % n_h.
cudaError_t launch_merge(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                         long long rows, int hd, bool f16_parts, void* o, float* lse, cudaStream_t stream,
                         const float* sink = nullptr, int T = 1, int n_h = 1);
// The merge writing NVFP4 O (fp4.codes / fp4.scales) instead of bf16 O; no sink.
cudaError_t launch_merge_nvfp4(const void* o_parts, const float* lse_parts, const float* range_parts, int n_splits,
                               long long rows, int hd, bool f16_parts, Fp4Out fp4, float* lse, cudaStream_t stream);

// ---- NVFP4 quantisation of fp32 rows on its own (nvfp4_kernel.cu) ---------
cudaError_t launch_quantize_nvfp4(const float* x, long long rows, int hd, float g, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream);

// ---- device status word (status.cu) ---------------------------------------
// Address of the status word on the current device (nullptr on failure).
unsigned* device_status_word();
// status[0] bits (kStatusBarrierTimeout = 1, kStatusBoundsViolation = 2) and
// the description of a site code of a checked build's index check.
constexpr unsigned kStatusBitTimeout = 1u, kStatusBitBounds = 2u;
const char* check_site_name(unsigned site);
bool checked_build();  // compiled with -DFMHA_CHECKED
// Launch a kernel whose bounded wait must time out after limit_ns.
cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream);
// Launch a kernel that runs one failing index check (a no-op unless checked).
cudaError_t launch_bounds_check_selftest(cudaStream_t stream);

}  // namespace fmha
