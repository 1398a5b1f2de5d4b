/*
 * fmha.h -- C ABI of libfmha_gb300.so, the GB300 (sm_103a) fused attention
 * forward.
 *
 * What is computed (per batch b, query head h, query row t):
 *
 *     O[b,h,t,:] = softmax_j( scale * <Q[b,h,t,:], K[b,kvh,j,:]> + mask ) V[b,kvh,j,:]
 *     LSE[b,h,t] = ln sum_{j attended} exp(scale * <Q[b,h,t,:], K[b,kvh,j,:]>)
 *
 * with kvh = h / (n_h / n_kv_h).  Sources: the commit pages of the
 * nvfp4-megamoe-kernel repository (dsv4 directory) and its CURRENT_ISSUE.md
 * "UMMA FMHA -- Full Pipeline + Production":
 *   - FA2 online softmax over KV tiles with a running max and sum, P kept
 *     un-normalised, one final divide by the running sum: commit e4ee9fd,
 *     multi-tile C API part.
 *   - scores are the unscaled dot product, the scale is applied in the
 *     softmax: CURRENT_ISSUE.md, "Key lessons from this session".
 *   - split-KV partials merged as O = sum_i exp(lse_i) O_i / sum_i exp(lse_i):
 *     CURRENT_ISSUE.md, "Next steps" item 4.
 *   - MQA as a K/V head shared by every query head (head stride 0): commit
 *     e4ee9fd, "Architecture".
 *   - sliding-window ("D3") and causal ("D4") masks: commit 593bc25, scalar
 *     reference kernel part.
 *   - a pure C ABI with no framework types and no host synchronisation on the
 *     hot path: commit e4ee9fd, multihead C API and "Architecture" parts.
 *
 * Readings of points the pages leave open:
 *   - query row t sits at absolute key position p = s_k - T + t (the T new
 *     queries follow the s_k - T cached keys: bottom-right alignment);
 *   - causal: key j is attended iff j <= p;
 *   - window w > 0: key j is attended iff j > p - w (the last w positions up to
 *     and including p); w = 0 disables the window;
 *   - LSE is the natural log of the sum over attended keys of exp(scaled
 *     score); a row that attends no key gets O = 0 and LSE = -inf.
 *
 * Layouts (all contiguous, row-major, device memory owned by the caller):
 *   Q, O        [batch, n_h,    T,   hd]  bf16 (raw bits, round-to-nearest-even on output)
 *   K, V        [batch, n_kv_h, s_k, hd]  bf16
 *   LSE         [batch, n_h,    T]        fp32
 *   o_parts     [n_splits, batch, n_h, T, hd] fp32   (split-KV partial outputs)
 *   lse_parts   [n_splits, batch, n_h, T]     fp32
 *
 * Accepted shapes: hd in {64, 128, 256, 512}; n_h % n_kv_h == 0;
 * batch * n_kv_h <= 65535; batch >= 0, T >= 0 (zero means nothing to do);
 * s_k >= 0; with causal, T <= s_k; window >= 0.  q, k, v, o, o_parts must be
 * 16-byte aligned, lse and lse_parts 4-byte aligned.
 *
 * Errors: every call returns FMHA_OK (0) or a negative FMHA_ERR_* code and
 * never aborts.  On an argument error nothing is launched.  The message of the
 * last failure on the calling thread is available from fmha_get_last_error().
 *
 * Asynchrony: every compute call is ordered on `stream` (NULL = the legacy
 * default stream) and returns without synchronising the host.  Kernels bound
 * every internal wait; a wait that gives up sets a device status word that
 * fmha_check_device_status() reports.
 */
#ifndef FMHA_GB300_H
#define FMHA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fmha_stream_t;

enum fmha_status {
    FMHA_OK = 0,
    FMHA_ERR_NULL = -1,           /* a required pointer is NULL */
    FMHA_ERR_ALIGN = -2,          /* a pointer is not aligned as required */
    FMHA_ERR_HEADDIM = -3,        /* hd not in {64, 128, 256, 512} */
    FMHA_ERR_HEADS = -4,          /* n_h, n_kv_h < 1 or n_h % n_kv_h != 0 */
    FMHA_ERR_SHAPE = -5,          /* negative size, causal with T > s_k, grid limits, bad window/chunk/scale */
    FMHA_ERR_WORKSPACE = -6,      /* the internal split-KV workspace could not be allocated */
    FMHA_ERR_LAUNCH = -7,         /* a CUDA call failed; the message names it */
    FMHA_ERR_DEVICE_TIMEOUT = -8, /* a kernel's bounded wait gave up (from fmha_check_device_status) */
    FMHA_ERR_UNSUPPORTED = -9,    /* a partial format this shape's kernel does not write */
    FMHA_ERR_DEVICE_BOUNDS = -10  /* checked build: a kernel's index check failed (from fmha_check_device_status) */
};

/*
 * Fused attention forward.  Writes O (bf16) and LSE (fp32).
 *
 * scale: multiplies the raw dot products (usually 1/sqrt(hd)).
 * window: sliding-window length in keys, 0 = none.  causal: 0 or 1.
 *
 * The library chooses whether to split the KV range over several thread
 * blocks.  When it splits, the partials live in a workspace the library
 * allocates on `stream` with cudaMallocAsync the first time a (device,
 * stream) pair needs more than it holds, and keeps until fmha_release().
 * They are fp32, except on the hd-512 tensor-core kernel, where they are fp16
 * scaled by a power of two per row half (so any finite value keeps 11
 * significant bits), which halves their traffic.
 * Callers that must not allocate use fmha_fwd_splitkv + fmha_merge with their
 * own buffers.
 */
int fmha_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
             float scale, int window, int causal, fmha_stream_t stream);

/*
 * The plan fmha_fwd uses for this shape: returns the number of KV chunks
 * (1 = no split: one kernel writes O and LSE directly; > 1 = a split pass
 * into the workspace followed by the merge), stores the chunk length in
 * *kv_chunk and the kernel family in *kernel (1 = decode kernel, 2 =
 * tensor-core kernel, one 128-row tile per thread block, 3 = tensor-core
 * kernel for hd 512, 4 = tensor-core kernel with two 128-row tiles per thread
 * block, hd 64 and 128; fmha_fwd_nvfp4 runs kernel 2 there, with the same
 * chunks);
 * either pointer may be NULL.  Pure host arithmetic apart from reading the current device's SM
 * count; negative FMHA_ERR_* code on invalid shapes.
 */
int fmha_fwd_plan(int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                  int window, int causal, int* kv_chunk, int* kernel);

/*
 * Split-KV layout for chunks of kv_chunk keys (kv_chunk >= 1): returns the
 * number of chunks n_splits (>= 1) and stores in *first_key the first key of
 * chunk 0, which is the first key that query row t = 0 attends (0 without a
 * window).  Chunk i covers keys [first_key + i*kv_chunk, first_key +
 * (i+1)*kv_chunk) clipped to s_k.  Pure host arithmetic; returns a negative
 * FMHA_ERR_* code for invalid arguments.  first_key may be NULL.
 */
int fmha_split_layout(int T, int s_k, int window, int kv_chunk, int* first_key);

/*
 * Split-KV partial pass (the "D5" split of CURRENT_ISSUE.md, "Next steps"
 * item 4).  For every chunk i of fmha_split_layout(T, s_k, window, kv_chunk)
 * writes the normalised partial output O_i and its log-sum-exp lse_i over the
 * keys of that chunk (O_i = 0, lse_i = -inf where the chunk holds no attended
 * key).  o_parts / lse_parts are caller buffers in the layouts above.
 */
int fmha_fwd_splitkv(const void* q, const void* k, const void* v,
                     float* o_parts, float* lse_parts, int kv_chunk,
                     int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                     float scale, int window, int causal, fmha_stream_t stream);

/*
 * Merge split-KV partials (CURRENT_ISSUE.md, "Next steps" item 4):
 *     LSE = ln sum_i exp(lse_i),   O = sum_i exp(lse_i - LSE) O_i
 * Partials with lse_i = -inf carry no weight; if all do, O = 0, LSE = -inf.
 * Writes bf16 O [batch, n_h, T, hd] and fp32 LSE [batch, n_h, T].
 */
int fmha_merge(const float* o_parts, const float* lse_parts, int n_splits,
               void* o, float* lse, int batch, int n_h, int T, int hd,
               fmha_stream_t stream);

/*
 * Partial formats for fmha_fwd_splitkv_ex / fmha_merge_ex.  The merge formula
 * is the one above; only the storage of O_i differs.
 *   FMHA_PARTS_F32: o_parts fp32 [n_splits, batch, n_h, T, hd] (what
 *     fmha_fwd_splitkv writes); range_parts unused, may be NULL.
 *   FMHA_PARTS_F16: o_parts fp16 [n_splits, batch, n_h, T, hd] holding
 *     O_i * 2^-k, and range_parts fp32 [n_splits, batch, n_h, T, 2] holding
 *     2^k for each 256-column half of each row; k is chosen per half row so
 *     that its largest |O_i| * 2^-k lies in [2^14, 2^15) before rounding (so
 *     in [2^14, 2^15] stored), so every finite partial keeps fp16's 11
 *     significant bits and none overflows.  Half the bytes of
 *     FMHA_PARTS_F32 (for callers that move partials elsewhere before merging;
 *     fmha_fwd uses this format internally at hd 512).  Written only by the
 *     hd-512 tensor-core kernel: hd = 512 and fmha_fwd_plan reporting kernel 3,
 *     else FMHA_ERR_UNSUPPORTED.  range_parts must be 4-byte aligned.
 * This extension has no counterpart on the pages; it is a storage format of
 * the partials whose merge they define.
 */
enum fmha_parts_format { FMHA_PARTS_F32 = 0, FMHA_PARTS_F16 = 1 };

/* fmha_fwd_splitkv writing partials in `parts_format`. */
int fmha_fwd_splitkv_ex(const void* q, const void* k, const void* v,
                        void* o_parts, float* lse_parts, float* range_parts, int parts_format,
                        int kv_chunk, int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                        float scale, int window, int causal, fmha_stream_t stream);

/* fmha_merge of partials in `parts_format` (range_parts as written by
 * fmha_fwd_splitkv_ex; FMHA_PARTS_F16 needs hd = 512), with an optional
 * attention sink (see fmha_fwd_sink): sink is NULL or a device array of n_h
 * fp32 logits, added once to each row's denominator. */
int fmha_merge_ex(const void* o_parts, const float* lse_parts, const float* range_parts, int parts_format,
                  int n_splits, const float* sink, void* o, float* lse, int batch, int n_h, int T, int hd,
                  fmha_stream_t stream);

/*
 * fmha_fwd with an attention sink.  The pages list "D5c sink" as a TODO and
 * define nothing; the reading taken here: query head h has a logit sigma_h
 * (natural-log units, the same units as scale * q.k) that joins the softmax
 * denominator only, as one more key whose value row is zero:
 *     O   = sum_j exp(s_j) v_j / (sum_j exp(s_j) + exp(sigma_h))
 *     LSE = ln(sum_j exp(s_j) + exp(sigma_h))
 * A row with no attended key gets O = 0, LSE = sigma_h; sigma_h = -inf is no
 * sink.  sink: device array of n_h fp32 logits, 4-byte aligned, caller-owned;
 * NULL makes this call fmha_fwd.  Everything else as fmha_fwd.
 */
int fmha_fwd_sink(const void* q, const void* k, const void* v, void* o, float* lse, const float* sink,
                  int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                  float scale, int window, int causal, fmha_stream_t stream);

/*
 * fmha_fwd with the output O quantised to NVFP4 in the epilogue, from the fp32
 * values that would otherwise be rounded to bf16 (commit 593bc25 of the
 * pages, TMEM-epilogue part: "register slot for FP4 pack"; its quantiser part
 * names an E2M1 element nibble, an E4M3 scale and round-to-nearest-even, and
 * gives no block size).  Format taken:
 *   - each O row [hd] is cut into hd / 16 blocks of 16 consecutive elements;
 *   - block scale s = E4M3(amax / (6 g)), amax the block's largest |O|, g =
 *     o_global_scale (finite, > 0); E4M3: 4 exponent bits (bias 7), 3
 *     mantissa bits, subnormals, largest finite value 448;
 *   - element code e = E2M1(O / (g s)): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
 *     for codes 0..7, sign in bit 3 (never set on a zero magnitude);
 *   - both roundings go to the nearest representable value, a tie to the even
 *     code, and saturate at the largest finite value; s = 0 gives codes 0;
 *   - amax / (6 g) and O / (g s) are IEEE fp32 divisions;
 *   - O is recovered as g * s * e.
 * o_codes:  [batch, n_h, T, hd / 2] bytes, element 2i in the low nibble of
 *           byte i of its row; 16-byte aligned.
 * o_scales: [batch, n_h, T, hd / 16] E4M3 bytes; 4-byte aligned.
 * lse as fmha_fwd.  No attention sink.  Plan, kernels, workspace, errors and
 * asynchrony are fmha_fwd's; when the plan splits, the merge quantises.
 */
int fmha_fwd_nvfp4(const void* q, const void* k, const void* v, void* o_codes, void* o_scales, float* lse,
                   float o_global_scale, int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                   float scale, int window, int causal, fmha_stream_t stream);

/*
 * The NVFP4 quantisation of fmha_fwd_nvfp4 applied to fp32 rows on their own:
 * x [rows, hd] fp32 (hd a multiple of 16, x 16-byte aligned) -> codes
 * [rows, hd / 2] (8-byte aligned) and scales [rows, hd / 16], with the same
 * block quantiser the fused epilogues run, so its codes can be checked bit
 * for bit.  Stream-ordered; FMHA_ERR_SHAPE for a bad hd, rows or global scale.
 */
int fmha_quantize_nvfp4(const float* x, long long rows, int hd, float global_scale, void* codes, void* scales,
                        fmha_stream_t stream);

/* Bytes of fp32 partial output (o_parts + lse_parts) that fmha_fwd_splitkv
 * writes for n_splits chunks: n_splits * batch * n_h * T * (hd + 1) * 4.
 * Negative arguments give 0. */
size_t fmha_splitkv_workspace_bytes(int batch, int n_h, int T, int hd, int n_splits);

/* The same number under the name the split-KV workspace query is usually
 * given: the caller buffers fmha_fwd_splitkv + fmha_merge need for n_splits
 * chunks (the count fmha_fwd_plan or fmha_split_layout returns). */
size_t fmha_workspace_bytes(int batch, int n_h, int T, int hd, int n_splits);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns FMHA_ERR_DEVICE_BOUNDS if, in a checked build, a kernel's
 * index check failed since the last check (the message names the check's
 * site), else FMHA_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up,
 * FMHA_ERR_LAUNCH if the synchronisation failed, else FMHA_OK. */
int fmha_check_device_status(fmha_stream_t stream);

/*
 * Checked build (no counterpart on the pages; the pages debugged an illegal
 * memory access by hand, CURRENT_ISSUE.md "Key lessons from this session").
 * The same sources compiled with -DFMHA_CHECKED give
 * libfmha_gb300_checked.so, with the same entry points.  Its kernels test
 * every computed shared-memory offset, tensor-memory column, global-memory
 * index and TMA coordinate against the extent of its buffer before the
 * access; a failed check skips the access (a warp-collective instruction is
 * pointed at offset 0 of its buffer instead), and the next
 * fmha_check_device_status() returns FMHA_ERR_DEVICE_BOUNDS naming the site.
 * It is a debugging aid and slower; results are otherwise identical.
 * fmha_build_flags() returns FMHA_BUILD_CHECKED in that library, 0 in the
 * normal one.
 */
#define FMHA_BUILD_CHECKED 1
int fmha_build_flags(void);

/* Message for the last non-zero return on the calling thread ("" if none). */
const char* fmha_get_last_error(void);

/* Frees every workspace fmha_fwd allocated (synchronises each device that
 * holds one first).  Safe to call at any time no fmha call is in flight. */
void fmha_release(void);

/*
 * Failure-detection self-test: launches one thread that waits, through the
 * same bounded mbarrier wait the attention kernels use, on a barrier phase
 * that nothing completes.  After timeout_us microseconds (1 .. 10^7) the wait
 * gives up, sets the device status word and the kernel returns normally, so
 * the next fmha_check_device_status() on this device returns
 * FMHA_ERR_DEVICE_TIMEOUT and the context stays usable.  No fault, trap or
 * hang is involved.
 */
int fmha_selftest_wait_timeout(unsigned timeout_us, fmha_stream_t stream);

/*
 * (This entry point has no counterpart on the pages the method comes from;
 * the computation is fmha_fwd's.)
 * fmha_fwd from host memory: copies Q, K and V (layouts of fmha_fwd) from
 * host memory into device buffers the library owns, runs fmha_fwd on them and
 * copies O (bf16) and LSE (fp32) back into host memory.  Everything is
 * stream-ordered on `stream` (one cudaMemcpyAsync per tensor, no host
 * synchronisation), so the host buffers must stay valid and unmodified until
 * `stream` has passed this call; page-locked host memory gives asynchronous
 * copies.  The device buffers (Q + K + V + O + LSE bytes) are cached per
 * device and stream like fmha_fwd's workspace, grown with cudaMallocAsync and
 * freed by fmha_release(); calls on one stream reuse them in stream order.
 * Calls on two streams use two sets, so the host-to-device copies of one can
 * overlap the kernels and the device-to-host copies of the other.
 * Errors: those of fmha_fwd (host pointers need no alignment), and
 * FMHA_ERR_WORKSPACE if the device buffers cannot be allocated.
 */
int fmha_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                  float scale, int window, int causal, fmha_stream_t stream);

/*
 * Index-check self-test: launches one thread that runs an index check whose
 * condition is false, with no memory access behind it.  In the checked build
 * the next fmha_check_device_status() on this device returns
 * FMHA_ERR_DEVICE_BOUNDS and names the self-test site; in the normal build
 * the check is compiled out and nothing is recorded.  Returns FMHA_OK, or
 * FMHA_ERR_LAUNCH if the launch failed.
 */
int fmha_selftest_bounds_check(fmha_stream_t stream);

/*
 * Kernel-family selection for every later call in the process: 0 = automatic
 * (default: the 128-row tensor-core kernels when a KV head has at least 64
 * query rows at hd <= 128, or 32 at hd 256 and 512, else the decode kernel;
 * at hd 64 and 128 with more than 128 rows per KV head, one or two row tiles
 * per thread block, whichever the planner estimates faster), 1 = always the
 * decode kernel, 2 = always the tensor-core kernels, with two row tiles per
 * thread block wherever that kernel applies (hd 64 and 128, more than 128 rows
 * per KV head), 3 = always the tensor-core kernels, one row tile per thread
 * block, and the row-tile kernel (hd <= 256) with its P V product in the "SS"
 * form (P staged in shared memory) instead of the default "TS" form (P
 * written over S in tensor memory and read from there as the MMA's A operand;
 * CURRENT_ISSUE.md "Next steps", TS MMA for PV), 4 = always the tensor-core
 * kernels, one row tile per thread block, TS form.  Meant for tests and
 * measurements that compare kernels on one shape; results agree within the
 * documented tolerance.  Returns FMHA_ERR_SHAPE for other values.
 */
int fmha_set_kernel_path(int path);

/*
 * fmha_fwd_noalloc -- fmha_fwd for callers that cannot allocate device memory.
 * (This entry point has no counterpart on the pages the method comes from.)
 *
 * Some callers must not allocate: an inference runtime that reserves all of
 * its device memory up front and accounts for every byte, code that runs on a
 * strict memory budget, or a hot loop that must not risk the synchronisation
 * and latency that cudaMalloc/cudaFree (or a pool growing) can bring.  For
 * them this call computes what fmha_fwd computes, with the same plan, the
 * same kernels and the same partial format (fp32, or fp16 with range factors
 * on the hd-512 tensor-core kernel; see fmha_fwd), so its results are
 * fmha_fwd's bit for bit, and it calls no allocating routine: when the plan
 * splits the KV range, the partials go to one fixed scratch array of
 * FMHA_NOALLOC_SCRATCH_BYTES (32 MiB) that is part of the library's device
 * image, so every GPU that loads the library holds it until the process exits.
 *
 * - A shape whose partials (fmha_fwd_plan's chunk count times the rows, in
 *   that format) exceed the scratch is rejected with FMHA_ERR_WORKSPACE and a
 *   message naming both sizes; nothing is launched.  Shapes that fmha_fwd_plan
 *   does not split need no scratch at all.
 * - The first call on each device looks up the scratch's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it for the
 *   life of the process; make that first call before any stream capture.  The
 *   library (this call, and the status word every call uses) must not be used
 *   on a device after cudaDeviceReset: the addresses it kept belong to the
 *   context that the reset destroyed.
 * - Every call on a device shares the one scratch array, which keeps the last
 *   call's contents.  Nothing in it needs to start at zero: each call writes
 *   every partial before its merge reads it.  Calls whose work overlaps on the
 *   GPU (for example on two streams without ordering between them) race on the
 *   scratch and may return wrong results; order them on one stream or with
 *   events.
 * Arguments, layouts and errors are those of fmha_fwd.
 */
#define FMHA_NOALLOC_SCRATCH_BYTES (32u << 20)
int fmha_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                     int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                     float scale, int window, int causal, fmha_stream_t stream);

/* ABI version: major * 10000 + minor * 100 + patch. */
int fmha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FMHA_GB300_H */
