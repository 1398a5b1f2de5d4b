// api.cu -- the C ABI of libfmha_gb300.so (declared in include/fmha.h).
//
// Validates arguments, plans the split-KV layout, builds the TMA tensor maps
// for K and V, and launches the kernels on the caller's stream.  No call here
// synchronises the host except fmha_check_device_status() and fmha_release().
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>

#include "fmha.h"
#include "internal.h"

namespace {

using namespace fmha;

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(FMHA_ERR_LAUNCH, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool tensor_map_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// K or V [slabs, s_k, hd] bf16 viewed as a 3-D tensor (hd fastest); boxes of
// 64 head-dim columns (128 bytes, 128-byte swizzle) x box_rows keys x 1 slab.
int make_kv_map(CUtensorMap* m, const void* base, int hd, int s_k, long long slabs, int box_rows) {
    std::memset(m, 0, sizeof *m);
    if (s_k == 0) return FMHA_OK;  // nothing will be loaded
    if (!tensor_map_encoder()) return fail(FMHA_ERR_LAUNCH, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)s_k, (cuuint64_t)slabs};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)s_k * hd * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FMHA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FMHA_OK;
}

// ---------------------------------------------------------------- validation
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int batch, int n_h, int n_kv_h, int T, int s_k, int hd, float scale, int window, int causal,
                Problem* out) {
    if (hd != 64 && hd != 128 && hd != 256 && hd != 512)
        return fail(FMHA_ERR_HEADDIM, "hd=%d: supported head dims are 64, 128, 256, 512", hd);
    if (n_h < 1 || n_kv_h < 1 || n_h % n_kv_h != 0)
        return fail(FMHA_ERR_HEADS, "n_h=%d n_kv_h=%d: need n_h, n_kv_h >= 1 and n_h %% n_kv_h == 0", n_h, n_kv_h);
    if (batch < 0 || T < 0 || s_k < 0)
        return fail(FMHA_ERR_SHAPE, "negative size (batch=%d T=%d s_k=%d)", batch, T, s_k);
    if (causal != 0 && causal != 1) return fail(FMHA_ERR_SHAPE, "causal must be 0 or 1 (got %d)", causal);
    if (causal && T > s_k)
        return fail(FMHA_ERR_SHAPE, "causal with T=%d > s_k=%d leaves query rows with no key", T, s_k);
    if (window < 0) return fail(FMHA_ERR_SHAPE, "window=%d must be >= 0", window);
    if (!std::isfinite(scale)) return fail(FMHA_ERR_SHAPE, "scale must be finite");
    if ((long long)batch * n_kv_h > 65535)
        return fail(FMHA_ERR_SHAPE, "batch * n_kv_h = %lld exceeds 65535", (long long)batch * n_kv_h);
    if ((long long)n_h / n_kv_h * T > (1LL << 30)) return fail(FMHA_ERR_SHAPE, "too many query rows per KV head");
    if ((long long)batch * n_h * T > INT_MAX)  // also bounds the merge grid (one block per 8 row slices)
        return fail(FMHA_ERR_SHAPE, "batch * n_h * T = %lld query rows exceeds 2^31 - 1", (long long)batch * n_h * T);
    out->batch = batch;
    out->n_h = n_h;
    out->n_kv_h = n_kv_h;
    out->T = T;
    out->s_k = s_k;
    out->hd = hd;
    out->window = window;
    out->causal = causal;
    out->scale = scale;
    out->group = n_h / n_kv_h;
    out->R = out->group * T;
    return FMHA_OK;
}

// k and v may be NULL only when there is no key (s_k == 0).
int check_inputs(const void* q, const void* k, const void* v, int s_k) {
    if (!q || ((!k || !v) && s_k > 0)) return fail(FMHA_ERR_NULL, "q, k and v must be non-NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
        return fail(FMHA_ERR_ALIGN, "q, k and v must be 16-byte aligned");
    return FMHA_OK;
}

// Chunk count limits: the grid's y dimension, and partial slabs addressed as
// split * (batch * n_kv_h) + slab by 32-bit TMA coordinates.
int check_chunks(const Problem& p, int n_splits) {
    if (n_splits > 65535) return fail(FMHA_ERR_SHAPE, "too many KV chunks (%d)", n_splits);
    if ((long long)n_splits * p.batch * p.n_kv_h > INT_MAX)
        return fail(FMHA_ERR_SHAPE, "KV chunks x batch x n_kv_h = %lld exceeds 2^31 - 1",
                    (long long)n_splits * p.batch * p.n_kv_h);
    return FMHA_OK;
}

// First attended key of row t = 0 and the chunk count for chunks of `chunk`.
SplitPlan split_layout(int T, int s_k, int window, int chunk) {
    long long first = 0;
    if (window > 0) {
        const long long p = (long long)s_k - T;  // position of row 0
        first = p - window + 1;
        if (first < 0) first = 0;
    }
    SplitPlan sp;
    sp.kv_begin = (int)first;
    sp.kv_chunk = chunk;
    const long long span = (long long)s_k - first;
    sp.n_splits = (span <= 0) ? 1 : (int)((span + chunk - 1) / chunk);
    return sp;
}

int sm_count() {
    // Per-device cache; any host thread may fill an entry (the value it stores
    // is the same whichever thread wins).  Without a device (planning on a
    // host) the count is GB300's 152 SMs.
    static std::atomic<int> cache[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 152;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ---------------------------------------------------------------- planning
// Kernel families: the decode kernel (8 or 16 query rows per thread block,
// mma.sync) and the tensor-core kernels (128-row query tiles, tcgen05).  A KV
// head with at least tc_min_rows(hd) query rows goes to the tensor-core
// kernels: 64 rows at hd <= 128, 32 rows at hd 256 and 512, where the decode
// kernel's CUDA-core-side work per key grows with hd (measured on the MHA shape
// sweep).  At hd 64 and 128 a KV head with more than 128 rows may also take
// the two-row-tile kernel (two tiles per block sharing each K/V tile); the
// planner picks whichever of the two has the lower estimated time.
int tc_min_rows(int hd) { return hd >= 256 ? 32 : 64; }
// 0 auto, 1 decode kernel, 2 tensor-core kernels (two row tiles per block
// where the shape allows), 3 tensor-core kernels with the row-tile kernel's
// SS-form PV, 4 tensor-core kernels with one row tile per block
std::atomic<int> g_path_override{0};

enum class Path { Decode, TensorCore, TensorCorePair, TensorCoreWide };

struct KernelShape {
    int rows_per_cta, kv_tile, ctas_per_sm, blocks_per_row_tile, min_chunk;
};

KernelShape kernel_shape(const Problem& p, Path path) {
    if (path == Path::TensorCore) return {kTcRows, tc_kv_tile(p.hd), 1, 1, 256};
    if (path == Path::TensorCorePair) return {2 * kTcRows, tc_pair_kv_tile(), 1, 1, 256};
    if (path == Path::TensorCoreWide) return {kTcRows, tc_wide_kv_tile(), 1, 2, 128};
    return {decode_rows_per_cta(p), decode_kv_tile(p.hd), p.hd == 512 ? 1 : 2, 1, 256};
}

// Estimated time (us) of a tensor-core split into n chunks: waves of blocks
// (one block per SM), each moving its K/V chunk, its Q tile(s) and its output
// at its per-block rate after ~1.5 us of fixed latency, never faster than the
// bytes DRAM serves at the copy bandwidth, plus for n > 1 the merge (~2.5 us
// and its partials).  Per-block rates measured on GB300: a row-tile block
// streams ~60 GB/s unless its softmax (~1.05 us per 128 keys for 128 rows)
// is slower, as at hd 64 (256 bytes of K and V per key: ~31 GB/s); an hd-512
// block ~52 GB/s (96 KB of K/V in flight, ~1.9 us per ring-slot round trip);
// at hd <= 128 a row-tile block also needs tile_us_per_128_keys of MMAs and
// softmax per 128 keys, and a two-row-tile block pair_us_per_128_keys for its
// two tiles (GQA prefill T 128, s_k 4096: 80.7 us with one row tile per block
// and 64.9 us with two at hd 128, 71.5 and 64.3 us at hd 64).
// The two halves of an hd-512 row tile read the same K, the second from L2,
// so DRAM serves K and V once per pair of blocks.  At hd 512, s_k 32768
// (128 row-tile halves) seven chunks measured 891 us against 962 us for one.
double pair_us_per_128_keys(int) { return 1.95; }
double tile_us_per_128_keys(int hd) { return hd == 64 ? 1.1 : 1.25; }

double tc_split_cost(const Problem& p, const KernelShape& ks, Path path, long long units, long long sms,
                     long long span, long long n) {
    const bool wide = path == Path::TensorCoreWide;
    const long long ctas = units * n;
    const long long waves = (ctas + sms - 1) / sms;
    long long keys = (span + n - 1) / n;
    keys = (keys + ks.kv_tile - 1) / ks.kv_tile * ks.kv_tile;
    // bytes per key: K and V rows (the hd-512 blocks read all of K, half of V)
    const double kv = (double)keys * (wide ? 3.0 * p.hd : 4.0 * p.hd);
    const double q = (double)ks.rows_per_cta * p.hd * 2.0;
    const double part_b = n > 1 ? (wide ? 2.0 : 4.0) : 2.0;
    const double out = (double)ks.rows_per_cta * (p.hd / ks.blocks_per_row_tile) * part_b;
    const double rate = (wide || path == Path::TensorCorePair) ? (wide ? 52e3 : 60e3)
                                                               : std::min(60e3, 4.0 * p.hd / (1.05 / 128.0));
    double stream_us = (kv + q + out) / rate;
    if (path == Path::TensorCorePair) stream_us = std::max(stream_us, (double)keys / 128.0 * pair_us_per_128_keys(p.hd));
    if (path == Path::TensorCore && p.hd <= 128)
        stream_us = std::max(stream_us, (double)keys / 128.0 * tile_us_per_128_keys(p.hd));
    const double block_us = 1.5 + stream_us;
    double t = (double)waves * block_us;
    const double dram = wide ? (double)keys * 2.0 * p.hd + q / 2.0 + out : kv + q + out;
    const double floor_us = (double)ctas * dram / 6.7e6;
    if (t < floor_us) t = floor_us;
    if (n > 1) t += 2.5 + (double)p.batch * p.n_h * p.T * p.hd * part_b * (double)n / 10e6;
    return t;
}

// Best chunk count of a tensor-core kernel and its estimated time: the count
// with the least tc_split_cost; a larger count must win by 3 %.
struct TcChoice {
    long long n;
    double us;
};

TcChoice tc_best_split(const Problem& p, Path path, long long span) {
    const KernelShape ks = kernel_shape(p, path);
    const long long units = (long long)p.batch * p.n_kv_h * ((p.R + ks.rows_per_cta - 1) / ks.rows_per_cta) *
                            ks.blocks_per_row_tile;
    const long long sms = sm_count();
    TcChoice best{1, tc_split_cost(p, ks, path, units, sms, span, 1)};
    if (units <= 0 || span <= ks.min_chunk) return best;
    long long max_n = span / ks.min_chunk;
    if (max_n > 64) max_n = 64;
    for (long long c = 2; c <= max_n; ++c) {
        const double t = tc_split_cost(p, ks, path, units, sms, span, c);
        if (t < best.us * 0.97) best = TcChoice{c, t};  // a clear gain only: fewer chunks on near-ties
    }
    return best;
}

long long kv_span(const Problem& p) {
    const SplitPlan whole = split_layout(p.T, p.s_k, p.window, p.s_k > 0 ? p.s_k : 1);
    return (long long)p.s_k - whole.kv_begin;
}

Path choose_path(const Problem& p) {
    const int ov = g_path_override.load();
    const bool tc_ok = tc_supports(p.hd) || p.hd == 512;
    if (ov == 1 || !tc_ok) return Path::Decode;
    if (ov < 2 && p.R < tc_min_rows(p.hd)) return Path::Decode;
    if (p.hd == 512) return Path::TensorCoreWide;
    const bool pair_ok = tc_pair_supports(p.hd) && p.R > kTcRows;
    if (!pair_ok || ov == 3 || ov == 4) return Path::TensorCore;
    if (ov == 2) return Path::TensorCorePair;
    const long long span = kv_span(p);
    return tc_best_split(p, Path::TensorCorePair, span).us < tc_best_split(p, Path::TensorCore, span).us
               ? Path::TensorCorePair
               : Path::TensorCore;
}

// Split heuristic.  Decode kernel: as many chunks as keep every thread block
// resident in one wave (SMs x blocks per SM); a chunk scan on GB300 (MHA b4
// h16, hd 64-512, s_k 4096-32768, and the GQA window decode) found the step
// fastest there, longer chunks amortising each block's fixed latency.  Tensor-core
// kernels (one block per SM): the chunk count with the least estimated time
// (tc_best_split), which weighs wave quantisation against the Q tile each
// extra block reloads and the partials it writes.
SplitPlan choose_split(const Problem& p) {
    const Path path = choose_path(p);
    const KernelShape ks = kernel_shape(p, path);
    const long long units = (long long)p.batch * p.n_kv_h * ((p.R + ks.rows_per_cta - 1) / ks.rows_per_cta) *
                            ks.blocks_per_row_tile;
    SplitPlan whole = split_layout(p.T, p.s_k, p.window, p.s_k > 0 ? p.s_k : 1);
    const long long span = (long long)p.s_k - whole.kv_begin;
    if (units <= 0 || span <= ks.min_chunk) return whole;
    long long n = 1;
    if (path != Path::Decode) {
        n = tc_best_split(p, path, span).n;
    } else {
        const long long target = (long long)sm_count() * ks.ctas_per_sm;
        if (units >= target) return whole;
        n = target / units;
        const long long max_n = span / ks.min_chunk;
        if (n > max_n) n = max_n;
    }
    if (n <= 1) return whole;
    long long chunk = (span + n - 1) / n;
    chunk = (chunk + ks.kv_tile - 1) / ks.kv_tile * ks.kv_tile;
    return split_layout(p.T, p.s_k, p.window, (int)chunk);
}

// ---------------------------------------------------------------- workspace
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
// key: (device, stream, kind); kind 0 = split-KV partials, 1 = fmha_fwd_host's device copies
std::map<std::tuple<int, cudaStream_t, int>, Workspace> g_ws;
enum WorkspaceKind { kWsPartials = 0, kWsHostIo = 1 };

int workspace(cudaStream_t stream, size_t bytes, void** out, int kind = kWsPartials) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[std::make_tuple(dev, stream, kind)];
    if (w.bytes < bytes) {
        if (w.ptr) {
            e = cudaFreeAsync(w.ptr, stream);
            w.ptr = nullptr;
            w.bytes = 0;
            if (e != cudaSuccess) return fail(FMHA_ERR_WORKSPACE, "cudaFreeAsync: %s", cudaGetErrorString(e));
        }
        e = cudaMallocAsync(&w.ptr, bytes, stream);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return fail(FMHA_ERR_WORKSPACE, "cudaMallocAsync(%zu): %s", bytes, cudaGetErrorString(e));
        }
        w.bytes = bytes;
    }
    *out = w.ptr;
    return FMHA_OK;
}

// Partial O (fp32, or fp16 plus two fp32 range factors per row) and fp32
// partial LSE for n_splits chunks.
size_t partial_bytes(long long rows, int hd, int n_splits, bool f16 = false) {
    return (size_t)n_splits * (size_t)rows * ((size_t)hd * (f16 ? 2 : 4) + sizeof(float) * (f16 ? 3 : 1));
}

// fmha_fwd keeps hd-512 partials of the tensor-core kernel in fp16 (with a
// power-of-two range factor per row half): there the partials are a large
// share of the traffic, and fp16's 11 significant bits keep the merged error
// well under the bf16 output's rounding.
bool use_f16_partials(const Problem& p) { return p.hd == 512 && choose_path(p) == Path::TensorCoreWide; }

// Workspace carve-up: o_part | lse_part [n, rows] | range_part [n, rows, 2] (fp16 only).
struct PartialViews {
    void* o_part;
    float* lse_part;
    float* range_part;
};
PartialViews partial_views(void* ws, long long rows, int hd, int n_splits, bool f16) {
    PartialViews v;
    v.o_part = ws;
    v.lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)n_splits * rows * hd * (f16 ? 2 : 4));
    v.range_part = f16 ? v.lse_part + (size_t)n_splits * rows : nullptr;
    return v;
}

enum RowsType { kRowsBf16, kRowsF32, kRowsF16 };

// A row-tile tensor [slabs, R, hd] (Q, O, or partials) viewed as 3-D;
// boxes of 128 bytes of columns x kTcRows rows, 128-byte swizzle.
int make_rows_map(CUtensorMap* m, const void* base, int hd, int R, long long slabs, RowsType type,
                  const char* what, int box_rows = kTcRows) {
    if (!tensor_map_encoder()) return fail(FMHA_ERR_LAUNCH, "cuTensorMapEncodeTiled is unavailable");
    const int esz = type == kRowsF32 ? 4 : 2;
    const CUtensorMapDataType dt = type == kRowsF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : type == kRowsF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)R, (cuuint64_t)slabs};
    cuuint64_t strides[2] = {(cuuint64_t)hd * esz, (cuuint64_t)R * hd * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3,
                          const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FMHA_ERR_LAUNCH, "cuTensorMapEncodeTiled (%s) failed (CUresult %d)", what, (int)r);
    return FMHA_OK;
}

// Launch the kernel family the plan picks: O/LSE directly, or partials.
// o_part is fp32, or fp16 with range_part when f16_parts (hd-512 tensor-core
// kernel only).
// sink: [n_h] attention-sink logits for the final output (NULL: none; never
// applied to partials, whose merge adds it).
// fp4: when fp4.codes is set, the final output is NVFP4 (o is unused).
int run_kernel(const void* q, const void* k, const void* v, const Problem& p, const SplitPlan& sp, void* o,
               float* lse, void* o_part, float* lse_part, bool to_partials, cudaStream_t stream,
               bool f16_parts = false, float* range_part = nullptr, const float* sink = nullptr,
               Fp4Out fp4 = Fp4Out{nullptr, nullptr, 1.f}) {
    if (to_partials) {
        sink = nullptr;
        fp4.codes = nullptr;
    }
    unsigned* status = device_status_word();
    if (!status) return fail(FMHA_ERR_LAUNCH, "cannot resolve the device status word");
    const Path path = choose_path(p);
    const KernelShape ks = kernel_shape(p, path);
    const long long slabs = (long long)p.batch * p.n_kv_h;
    if (path != Path::Decode) {
        TcLaunch L;
        L.o = o;
        L.lse = lse;
        L.o_part = o_part;
        L.lse_part = lse_part;
        L.range_part = range_part;
        L.to_partials = to_partials;
        L.sink = sink;
        L.fp4 = fp4;
        L.ss_pv = g_path_override.load() == 3;
        L.f16_partials = f16_parts;
        if (f16_parts && (path != Path::TensorCoreWide || !range_part || !to_partials))
            return fail(FMHA_ERR_LAUNCH, "fp16 partials need the hd-512 kernel and a range array");
        L.p = p;
        L.sp = sp;
        L.status = status;
        int rc = make_rows_map(&L.tmap_q, q, p.hd, p.R, slabs, kRowsBf16, "Q",
                               path == Path::TensorCoreWide ? tc_wide_q_box_rows(p, sp) : kTcRows);
        if (rc) return rc;
        // An NVFP4 output is stored row by row without a tensor map; the O map
        // is then built over Q (same shape and type) and never stored through.
        rc = to_partials ? make_rows_map(&L.tmap_o, o_part, p.hd, p.R, slabs * sp.n_splits,
                                         f16_parts ? kRowsF16 : kRowsF32, "O partials")
                         : make_rows_map(&L.tmap_o, fp4.codes ? q : o, p.hd, p.R, slabs, kRowsBf16, "O");
        if (rc) return rc;
        rc = make_kv_map(&L.tmap_k, k, p.hd, p.s_k, slabs, ks.kv_tile);
        if (rc) return rc;
        rc = make_kv_map(&L.tmap_v, v, p.hd, p.s_k, slabs, ks.kv_tile);
        if (rc) return rc;
        // The two-row-tile kernel has no NVFP4 epilogue (its O is transposed in
        // tensor memory): an NVFP4 output takes the one-row-tile kernel, with
        // the same KV tiles and chunks.
        const bool pair = path == Path::TensorCorePair && !(fp4.codes && !to_partials);
        cudaError_t e = (path == Path::TensorCoreWide) ? launch_tc_wide(L, stream)
                        : pair                         ? launch_tc_pair(L, stream)
                                                       : launch_tc(L, stream);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
        return FMHA_OK;
    }
    if (f16_parts) return fail(FMHA_ERR_LAUNCH, "fp16 partials need the hd-512 kernel");
    DecodeLaunch L;
    L.q = q;
    L.o = o;
    L.lse = lse;
    L.o_part = static_cast<float*>(o_part);
    L.lse_part = lse_part;
    L.to_partials = to_partials;
    L.sink = sink;
    L.fp4 = fp4;
    L.p = p;
    L.sp = sp;
    L.status = status;
    int rc = make_kv_map(&L.tmap_k, k, p.hd, p.s_k, slabs, ks.kv_tile);
    if (rc) return rc;
    rc = make_kv_map(&L.tmap_v, v, p.hd, p.s_k, slabs, ks.kv_tile);
    if (rc) return rc;
    cudaError_t e = launch_decode(L, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return FMHA_OK;
}

}  // namespace

extern "C" {

int fmha_fwd_sink(const void* q, const void* k, const void* v, void* o, float* lse, const float* sink, int batch,
                  int n_h, int n_kv_h, int T, int s_k, int hd, float scale, int window, int causal,
                  fmha_stream_t stream) {
    try {
        Problem p;
        int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, &p);
        if (rc) return rc;
        rc = check_inputs(q, k, v, s_k);
        if (rc) return rc;
        if (!o || !lse) return fail(FMHA_ERR_NULL, "o and lse must be non-NULL");
        if (!aligned(o, 16) || !aligned(lse, 4)) return fail(FMHA_ERR_ALIGN, "o must be 16-byte, lse 4-byte aligned");
        if (sink && !aligned(sink, 4)) return fail(FMHA_ERR_ALIGN, "sink must be 4-byte aligned");
        const long long rows = (long long)batch * n_h * T;
        if (rows == 0) return FMHA_OK;
        const SplitPlan sp = choose_split(p);
        rc = check_chunks(p, sp.n_splits);
        if (rc) return rc;
        if (sp.n_splits == 1)
            return run_kernel(q, k, v, p, sp, o, lse, nullptr, nullptr, false, stream, false, nullptr, sink);
        void* ws = nullptr;
        const bool f16 = use_f16_partials(p);
        rc = workspace(stream, partial_bytes(rows, hd, sp.n_splits, f16), &ws);
        if (rc) return rc;
        const PartialViews pv = partial_views(ws, rows, hd, sp.n_splits, f16);
        rc = run_kernel(q, k, v, p, sp, nullptr, nullptr, pv.o_part, pv.lse_part, true, stream, f16, pv.range_part);
        if (rc) return rc;
        cudaError_t e = launch_merge(pv.o_part, pv.lse_part, pv.range_part, sp.n_splits, rows, hd, f16, o, lse, stream,
                                     sink, T, n_h);
        if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
        return FMHA_OK;
    } catch (...) {
        return fail(FMHA_ERR_LAUNCH, "unexpected host exception in fmha_fwd");
    }
}

int fmha_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int n_h, int n_kv_h,
             int T, int s_k, int hd, float scale, int window, int causal, fmha_stream_t stream) {
    return fmha_fwd_sink(q, k, v, o, lse, nullptr, batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, stream);
}

int fmha_fwd_nvfp4(const void* q, const void* k, const void* v, void* o_codes, void* o_scales, float* lse,
                   float o_global_scale, int batch, int n_h, int n_kv_h, int T, int s_k, int hd, float scale,
                   int window, int causal, fmha_stream_t stream) {
    try {
        Problem p;
        int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, &p);
        if (rc) return rc;
        rc = check_inputs(q, k, v, s_k);
        if (rc) return rc;
        if (!o_codes || !o_scales || !lse) return fail(FMHA_ERR_NULL, "o_codes, o_scales and lse must be non-NULL");
        if (!aligned(o_codes, 16) || !aligned(o_scales, 4) || !aligned(lse, 4))
            return fail(FMHA_ERR_ALIGN, "o_codes must be 16-byte, o_scales and lse 4-byte aligned");
        if (!(o_global_scale > 0.f) || !std::isfinite(o_global_scale))
            return fail(FMHA_ERR_SHAPE, "o_global_scale must be finite and > 0");
        const long long rows = (long long)batch * n_h * T;
        if (rows == 0) return FMHA_OK;
        const Fp4Out fp4{static_cast<uint8_t*>(o_codes), static_cast<uint8_t*>(o_scales), o_global_scale};
        const SplitPlan sp = choose_split(p);
        rc = check_chunks(p, sp.n_splits);
        if (rc) return rc;
        if (sp.n_splits == 1)
            return run_kernel(q, k, v, p, sp, nullptr, lse, nullptr, nullptr, false, stream, false, nullptr, nullptr,
                              fp4);
        void* ws = nullptr;
        const bool f16 = use_f16_partials(p);
        rc = workspace(stream, partial_bytes(rows, hd, sp.n_splits, f16), &ws);
        if (rc) return rc;
        const PartialViews pv = partial_views(ws, rows, hd, sp.n_splits, f16);
        rc = run_kernel(q, k, v, p, sp, nullptr, nullptr, pv.o_part, pv.lse_part, true, stream, f16, pv.range_part);
        if (rc) return rc;
        cudaError_t e = launch_merge_nvfp4(pv.o_part, pv.lse_part, pv.range_part, sp.n_splits, rows, hd, f16, fp4, lse,
                                           stream);
        if (e != cudaSuccess) return cuda_fail(e, "NVFP4 merge kernel launch");
        return FMHA_OK;
    } catch (...) {
        return fail(FMHA_ERR_LAUNCH, "unexpected host exception in fmha_fwd_nvfp4");
    }
}

int fmha_quantize_nvfp4(const float* x, long long rows, int hd, float global_scale, void* codes, void* scales,
                        fmha_stream_t stream) {
    if (rows < 0 || hd < 16 || hd % 16 != 0)
        return fail(FMHA_ERR_SHAPE, "fmha_quantize_nvfp4: need rows >= 0 and hd a positive multiple of 16");
    if (!(global_scale > 0.f) || !std::isfinite(global_scale))
        return fail(FMHA_ERR_SHAPE, "fmha_quantize_nvfp4: global_scale must be finite and > 0");
    if (rows == 0) return FMHA_OK;
    if (!x || !codes || !scales) return fail(FMHA_ERR_NULL, "fmha_quantize_nvfp4: NULL buffer");
    if (!aligned(x, 16) || !aligned(codes, 8))
        return fail(FMHA_ERR_ALIGN, "fmha_quantize_nvfp4: x must be 16-byte, codes 8-byte aligned");
    if (rows > (1LL << 40) / hd) return fail(FMHA_ERR_SHAPE, "fmha_quantize_nvfp4: too many elements");
    cudaError_t e = launch_quantize_nvfp4(x, rows, hd, global_scale, static_cast<uint8_t*>(codes),
                                          static_cast<uint8_t*>(scales), stream);
    if (e != cudaSuccess) return cuda_fail(e, "NVFP4 quantisation kernel launch");
    return FMHA_OK;
}

int fmha_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  int batch, int n_h, int n_kv_h, int T, int s_k, int hd, float scale, int window, int causal,
                  fmha_stream_t stream) {
    try {
        Problem p;
        int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, &p);
        if (rc) return rc;
        if (!q_host || ((!k_host || !v_host) && s_k > 0) || !o_host || !lse_host)
            return fail(FMHA_ERR_NULL, "q, k, v, o and lse must be non-NULL");
        const long long rows = (long long)batch * n_h * T;
        if (rows == 0) return FMHA_OK;
        // device copies, each 256-byte aligned: q | k | v | o | lse
        auto up = [](size_t b) { return (b + 255) / 256 * 256; };
        const size_t q_b = (size_t)rows * hd * 2;
        const size_t kv_b = (size_t)batch * n_kv_h * s_k * hd * 2;
        const size_t lse_b = (size_t)rows * sizeof(float);
        const size_t off_k = up(q_b), off_v = off_k + up(kv_b), off_o = off_v + up(kv_b), off_l = off_o + up(q_b);
        void* ws = nullptr;
        rc = workspace(stream, off_l + up(lse_b), &ws, kWsHostIo);
        if (rc) return rc;
        char* base = static_cast<char*>(ws);
        cudaError_t e = cudaMemcpyAsync(base, q_host, q_b, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess && kv_b) e = cudaMemcpyAsync(base + off_k, k_host, kv_b, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess && kv_b) e = cudaMemcpyAsync(base + off_v, v_host, kv_b, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        rc = fmha_fwd(base, base + off_k, base + off_v, base + off_o, reinterpret_cast<float*>(base + off_l), batch,
                      n_h, n_kv_h, T, s_k, hd, scale, window, causal, stream);
        if (rc) return rc;
        e = cudaMemcpyAsync(o_host, base + off_o, q_b, cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(lse_host, base + off_l, lse_b, cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
        return FMHA_OK;
    } catch (...) {
        return fail(FMHA_ERR_LAUNCH, "unexpected host exception in fmha_fwd_host");
    }
}

int fmha_fwd_plan(int batch, int n_h, int n_kv_h, int T, int s_k, int hd, int window, int causal, int* kv_chunk,
                  int* kernel) {
    Problem p;
    int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, 1.0f, window, causal, &p);
    if (rc) return rc;
    const SplitPlan sp = choose_split(p);
    if (kv_chunk) *kv_chunk = sp.kv_chunk;
    if (kernel) {
        const Path path = choose_path(p);
        *kernel = path == Path::Decode ? 1 : path == Path::TensorCore ? 2 : path == Path::TensorCoreWide ? 3 : 4;
    }
    return sp.n_splits;
}

int fmha_split_layout(int T, int s_k, int window, int kv_chunk, int* first_key) {
    if (T < 0 || s_k < 0 || window < 0 || kv_chunk < 1)
        return fail(FMHA_ERR_SHAPE, "fmha_split_layout: need T, s_k, window >= 0 and kv_chunk >= 1");
    const SplitPlan sp = split_layout(T, s_k, window, kv_chunk);
    if (first_key) *first_key = sp.kv_begin;
    return sp.n_splits;
}

int fmha_fwd_splitkv_ex(const void* q, const void* k, const void* v, void* o_parts, float* lse_parts,
                        float* range_parts, int parts_format, int kv_chunk, int batch, int n_h, int n_kv_h, int T,
                        int s_k, int hd, float scale, int window, int causal, fmha_stream_t stream) {
    try {
        Problem p;
        int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, &p);
        if (rc) return rc;
        if (parts_format != FMHA_PARTS_F32 && parts_format != FMHA_PARTS_F16)
            return fail(FMHA_ERR_SHAPE, "parts_format=%d is not a partial format", parts_format);
        const bool f16 = parts_format == FMHA_PARTS_F16;
        if (f16 && !use_f16_partials(p))
            return fail(FMHA_ERR_UNSUPPORTED, "fp16 partials are written by the hd-512 tensor-core kernel only "
                                              "(hd=%d, %d query rows per KV head)", hd, p.R);
        rc = check_inputs(q, k, v, s_k);
        if (rc) return rc;
        if (kv_chunk < 1) return fail(FMHA_ERR_SHAPE, "kv_chunk=%d must be >= 1", kv_chunk);
        if (!o_parts || !lse_parts || (f16 && !range_parts))
            return fail(FMHA_ERR_NULL, "o_parts, lse_parts (and range_parts for fp16) must be non-NULL");
        if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || (f16 && !aligned(range_parts, 4)))
            return fail(FMHA_ERR_ALIGN, "o_parts must be 16-byte, lse_parts and range_parts 4-byte aligned");
        const long long rows = (long long)batch * n_h * T;
        if (rows == 0) return FMHA_OK;
        const SplitPlan sp = split_layout(T, s_k, window, kv_chunk);
        rc = check_chunks(p, sp.n_splits);
        if (rc) return rc;
        return run_kernel(q, k, v, p, sp, nullptr, nullptr, o_parts, lse_parts, true, stream, f16,
                          f16 ? range_parts : nullptr);
    } catch (...) {
        return fail(FMHA_ERR_LAUNCH, "unexpected host exception in fmha_fwd_splitkv");
    }
}

int fmha_fwd_splitkv(const void* q, const void* k, const void* v, float* o_parts, float* lse_parts, int kv_chunk,
                     int batch, int n_h, int n_kv_h, int T, int s_k, int hd, float scale, int window, int causal,
                     fmha_stream_t stream) {
    return fmha_fwd_splitkv_ex(q, k, v, o_parts, lse_parts, nullptr, FMHA_PARTS_F32, kv_chunk, batch, n_h, n_kv_h,
                               T, s_k, hd, scale, window, causal, stream);
}

int fmha_merge_ex(const void* o_parts, const float* lse_parts, const float* range_parts, int parts_format,
                  int n_splits, const float* sink, void* o, float* lse, int batch, int n_h, int T, int hd,
                  fmha_stream_t stream) {
    if (hd != 64 && hd != 128 && hd != 256 && hd != 512)
        return fail(FMHA_ERR_HEADDIM, "hd=%d: supported head dims are 64, 128, 256, 512", hd);
    if (batch < 0 || n_h < 0 || T < 0 || n_splits < 1)
        return fail(FMHA_ERR_SHAPE, "fmha_merge: need batch, n_h, T >= 0 and n_splits >= 1");
    if (parts_format != FMHA_PARTS_F32 && parts_format != FMHA_PARTS_F16)
        return fail(FMHA_ERR_SHAPE, "parts_format=%d is not a partial format", parts_format);
    const bool f16 = parts_format == FMHA_PARTS_F16;
    if (f16 && hd != 512) return fail(FMHA_ERR_UNSUPPORTED, "fp16 partials exist for hd = 512 only");
    const long long rows = (long long)batch * n_h * T;
    if (rows == 0) return FMHA_OK;
    if (!o_parts || !lse_parts || !o || !lse || (f16 && !range_parts))
        return fail(FMHA_ERR_NULL, "fmha_merge: NULL buffer");
    if (!aligned(o_parts, 16) || !aligned(o, 16) || !aligned(lse_parts, 4) || !aligned(lse, 4) ||
        (f16 && !aligned(range_parts, 4)) || (sink && !aligned(sink, 4)))
        return fail(FMHA_ERR_ALIGN, "fmha_merge: o_parts and o 16-byte, lse, range and sink buffers 4-byte aligned");
    if (rows > (1LL << 32)) return fail(FMHA_ERR_SHAPE, "fmha_merge: too many rows");
    cudaError_t e = launch_merge(o_parts, lse_parts, f16 ? range_parts : nullptr, n_splits, rows, hd, f16, o, lse,
                                 stream, sink, T, n_h);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
    return FMHA_OK;
}

int fmha_merge(const float* o_parts, const float* lse_parts, int n_splits, void* o, float* lse, int batch, int n_h,
               int T, int hd, fmha_stream_t stream) {
    return fmha_merge_ex(o_parts, lse_parts, nullptr, FMHA_PARTS_F32, n_splits, nullptr, o, lse, batch, n_h, T, hd,
                         stream);
}

size_t fmha_splitkv_workspace_bytes(int batch, int n_h, int T, int hd, int n_splits) {
    if (batch < 0 || n_h < 0 || T < 0 || hd < 0 || n_splits < 0) return 0;
    return partial_bytes((long long)batch * n_h * T, hd, n_splits);
}

size_t fmha_workspace_bytes(int batch, int n_h, int T, int hd, int n_splits) {
    return fmha_splitkv_workspace_bytes(batch, n_h, T, hd, n_splits);
}

int fmha_check_device_status(fmha_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned* w = device_status_word();
    if (!w) return fail(FMHA_ERR_LAUNCH, "cannot resolve the device status word");
    unsigned h[2] = {0u, 0u};
    e = cudaMemcpy(h, w, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (h[0] || h[1]) {
        e = cudaMemset(w, 0, sizeof h);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
        if (h[0] & fmha::kStatusBitBounds)
            return fail(FMHA_ERR_DEVICE_BOUNDS, "an index check failed at site 0x%x (%s); status 0x%x", h[1],
                        fmha::check_site_name(h[1]), h[0]);
        return fail(FMHA_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait gave up (status 0x%x)", h[0]);
    }
    return FMHA_OK;
}

int fmha_build_flags(void) { return fmha::checked_build() ? FMHA_BUILD_CHECKED : 0; }

const char* fmha_get_last_error(void) { return g_last_error.c_str(); }

void fmha_release(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(std::get<0>(kv.first));
        cudaDeviceSynchronize();
        cudaFree(kv.second.ptr);
    }
    g_ws.clear();
    cudaSetDevice(cur);
}

int fmha_version(void) { return 100; }

int fmha_selftest_wait_timeout(unsigned timeout_us, fmha_stream_t stream) {
    if (timeout_us < 1 || timeout_us > 10000000u)
        return fail(FMHA_ERR_SHAPE, "timeout_us must be in [1, 10^7] (got %u)", timeout_us);
    cudaError_t e = launch_wait_timeout_selftest((unsigned long long)timeout_us * 1000ull, stream);
    if (e != cudaSuccess) return cuda_fail(e, "wait-timeout self-test launch");
    return FMHA_OK;
}

int fmha_selftest_bounds_check(fmha_stream_t stream) {
    cudaError_t e = launch_bounds_check_selftest(stream);
    if (e != cudaSuccess) return cuda_fail(e, "index-check self-test launch");
    return FMHA_OK;
}

int fmha_set_kernel_path(int path) {
    if (path < 0 || path > 4)
        return fail(FMHA_ERR_SHAPE, "fmha_set_kernel_path: 0 to 4 expected (got %d)", path);
    g_path_override.store(path);
    return FMHA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation entry point
// fmha_fwd_noalloc: the same computation as fmha_fwd for callers that cannot
// allocate device memory.  Its split-KV partials live in the file-scope array
// below instead of a workspace from cudaMallocAsync.  In host code the array's
// name is only a host-side stand-in, so the device address is looked up once
// per device with cudaGetSymbolAddress (with that device current) and passed
// to the kernels.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FMHA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxNoallocDevices = 128;
void* g_noalloc_addr[kMaxNoallocDevices] = {};
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxNoallocDevices) return fail(FMHA_ERR_LAUNCH, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the no-allocation scratch");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return FMHA_OK;
}

}  // namespace

extern "C" int fmha_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int n_h,
                                int n_kv_h, int T, int s_k, int hd, float scale, int window, int causal,
                                fmha_stream_t stream) {
    try {
        Problem p;
        int rc = check_shape(batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, &p);
        if (rc) return rc;
        rc = check_inputs(q, k, v, s_k);
        if (rc) return rc;
        if (!o || !lse) return fail(FMHA_ERR_NULL, "o and lse must be non-NULL");
        if (!aligned(o, 16) || !aligned(lse, 4)) return fail(FMHA_ERR_ALIGN, "o must be 16-byte, lse 4-byte aligned");
        const long long rows = (long long)batch * n_h * T;
        if (rows == 0) return FMHA_OK;
        const SplitPlan sp = choose_split(p);
        rc = check_chunks(p, sp.n_splits);
        if (rc) return rc;
        if (sp.n_splits == 1) return run_kernel(q, k, v, p, sp, o, lse, nullptr, nullptr, false, stream);
        // The partial format is fmha_fwd's: fp16 with range factors on the
        // hd-512 tensor-core kernel, fp32 elsewhere.
        const bool f16 = use_f16_partials(p);
        const size_t need = partial_bytes(rows, hd, sp.n_splits, f16);
        if (need > (size_t)FMHA_NOALLOC_SCRATCH_BYTES)
            return fail(FMHA_ERR_WORKSPACE,
                        "fmha_fwd_noalloc: this shape needs %zu bytes of split-KV scratch (%d chunks x %lld rows); "
                        "the fixed scratch holds %zu bytes",
                        need, sp.n_splits, rows, (size_t)FMHA_NOALLOC_SCRATCH_BYTES);
        void* scratch = nullptr;
        rc = noalloc_scratch(&scratch);
        if (rc) return rc;
        const PartialViews pv = partial_views(scratch, rows, hd, sp.n_splits, f16);
        rc = run_kernel(q, k, v, p, sp, nullptr, nullptr, pv.o_part, pv.lse_part, true, stream, f16, pv.range_part);
        if (rc) return rc;
        cudaError_t e =
            launch_merge(pv.o_part, pv.lse_part, pv.range_part, sp.n_splits, rows, hd, f16, o, lse, stream);
        if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
        return FMHA_OK;
    } catch (...) {
        return fail(FMHA_ERR_LAUNCH, "unexpected host exception in fmha_fwd_noalloc");
    }
}
