/*
 * moe_w4.h -- C ABI of the routed W4A16 mixture-of-experts FFN layer (GB300, sm_103a).
 *
 * The layer, stage by stage:
 *   1. top-k expert selection from router logits               moe_route_topk
 *   2. token -> expert permutation (histogram, scan, gather)    moe_permute
 *   3. grouped gate_up / down expert GEMMs on int4 weights     moe_expert_ffn_w4a16
 *      (group 128, fp16 scale and zero), SiLU(gate) * up fused
 *   4. router-weighted combine back to token order              moe_combine
 *   whole layer                                                  moe_layer_forward
 *
 * Sources for what each call computes:
 *   - "Performance and verification" (bloomery docs/performance.md), section
 *     "Why it is fast": grouping a batch by expert means one fetch of each
 *     expert's weights per batch; a prompt's expert products are batched into
 *     grouped tensor-core GEMMs; the host computes on the packed 4-bit codes
 *     without expanding them.  Section "How it is verified": expert ids are
 *     integers held to exact equality.
 *   - "Measured results" (vllm-omni docs/edge/results.md), sections Speed and
 *     Fidelity: W4A16 with groups of 128, 4.25 bits per weight; the prefill
 *     path dequantises to 16-bit and runs a dense GEMM.
 *
 * Conventions (every entry point):
 *   - Pointers named *_dev or documented "device" are CUDA device pointers on the
 *     current device; the caller allocates and owns every buffer.  The library
 *     never allocates, frees or synchronises (except moe_get_device_error).
 *   - Every call is asynchronous on `stream` (0 = legacy default stream).
 *   - bf16 tensors are raw 16-bit bfloat16 patterns; fp16 tensors raw IEEE half
 *     patterns.  All arrays are dense, row-major, no padding.
 *   - Device pointers must be 16-byte aligned (MOE_ERR_MISALIGNED otherwise).
 *   - Argument checks run on the host before any launch; a failed check returns
 *     a status and launches nothing.  A launch failure returns MOE_ERR_CUDA.
 *     Data errors seen on the device (an expert id out of range, a bounded wait
 *     that timed out) are recorded in the workspace error word and read back
 *     with moe_get_device_error; the kernels never trap.
 *   - Workspaces: the first 256 bytes of every workspace hold the device error
 *     word.  They must be zero before the workspace's first use (allocate it
 *     zeroed); kernels only OR error bits into them and moe_get_device_error
 *     reads and clears them.  The rest is scratch, rewritten by each call.
 *     Calls that share a workspace must not overlap on the GPU.
 *   - Limits: 1 <= k <= E <= 1024; d_model and d_ff multiples of 256 and at
 *     most 16384 (MOE_ERR_UNSUPPORTED otherwise); group = 128; T >= 0 (T = 0
 *     is a valid no-op); T * k < 2^31.
 */
#ifndef MOE_W4_H
#define MOE_W4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a size, count or null pointer is out of contract */
    MOE_ERR_MISALIGNED = 2,    /* a device pointer is not 16-byte aligned */
    MOE_ERR_UNSUPPORTED = 3,   /* shape outside the supported set (e.g. group != 128) */
    MOE_ERR_WORKSPACE = 4,     /* workspace null or smaller than the *_workspace_size */
    MOE_ERR_CUDA = 5,          /* a CUDA launch or runtime call failed */
    MOE_ERR_DEVICE_RANGE = 6,  /* device side: an expert id was outside [0, E) */
    MOE_ERR_TIMEOUT = 7,       /* device side: a bounded pipeline wait gave up */
    MOE_ERR_F16_RANGE = 8,     /* device side: a value left fp16's range in the tensor-core regime */
    MOE_ERR_SCRATCH_LIMIT = 9, /* moe_permute_noalloc: T*k larger than its fixed scratch allows */
    MOE_ERR_CAPTURE = 10       /* moe_permute_noalloc: first call on a device made while its stream captures */
} moe_status_t;

/*
 * One layer's quantised expert weights (device pointers, caller-owned).
 * Weight format: "Measured results", section Fidelity (W4A16, 4.25 bits per
 * weight) and section Memory (4-bit codes packed eight per 32-bit word).
 *
 *   w13_q [E][2*d_ff][d_model/8]   uint32: int4 codes along d_model, 8 per word,
 *                                  code k in bits 4*(k%8)..+3 of word k/8.
 *                                  Rows 0..d_ff-1 = gate, d_ff..2*d_ff-1 = up.
 *   w13_s, w13_z [E][2*d_ff][d_model/128]  fp16 scale and zero of each group
 *   w2_q  [E][d_model][d_ff/8]     uint32: down projection, packed along d_ff
 *   w2_s, w2_z  [E][d_model][d_ff/128]     fp16
 *
 * Dequantised weight: w = (code - zero) * scale, zero in code units.
 */
typedef struct {
    int32_t E;        /* number of experts, 1..1024 */
    int32_t d_model;  /* hidden size, multiple of 256 */
    int32_t d_ff;     /* expert intermediate size, multiple of 256 */
    int32_t group;    /* must be 128 */
    const uint32_t* w13_q;
    const uint16_t* w13_s;
    const uint16_t* w13_z;
    const uint32_t* w2_q;
    const uint16_t* w2_s;
    const uint16_t* w2_z;
} moe_w4_layer;

/*
 * Stage 1 -- top-k routing.  "Performance and verification", section
 * "How it is verified": the chosen expert ids are integers, checked for
 * exact equality.
 *
 * For each token t: the k experts with the largest logits, slot 0 the largest,
 * equal logits ordered by ascending expert id; the comparison is exact on the
 * fp32 values.  topk_w[t][j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the
 * k selected logits (softmax over the selection), computed in fp32.
 *
 *   logits   device fp32 [T][E], finite values
 *   topk_ids device int32 [T][k] (out)
 *   topk_w   device fp32  [T][k] (out)
 */
moe_status_t moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                            int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/*
 * Stage 2 -- token -> expert permutation.  "Performance and verification",
 * section "Why it is fast": an expert's weights are fetched a single time per
 * batch, so assignments are grouped by expert first.
 *
 * Assignment a = t*k + j goes to expert topk_ids[a].  Outputs:
 *   counts  [E]    assignments per expert
 *   offsets [E+1]  exclusive prefix sum of counts (offsets[E] = T*k)
 *   sorted  [T*k]  sorted[i] = assignment at permuted position i; segment e is
 *                  offsets[e]..offsets[e+1]-1, ascending a inside a segment
 *   inv     [T*k]  inv[a] = permuted position of assignment a
 *   x_perm  [T*k][d] bf16 (optional, NULL to skip): x_perm[i] = x[sorted[i] / k]
 * All int32 / bf16 device arrays.  x may be NULL when x_perm is NULL.
 * Ids outside [0, E) are skipped and reported as MOE_ERR_DEVICE_RANGE through
 * the workspace error word (the outputs are then unspecified).
 * Workspace: >= moe_permute_workspace_size(T, k, E) bytes of device memory.
 */
moe_status_t moe_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                         const void* x_bf16, int32_t d, int32_t* counts, int32_t* offsets,
                         int32_t* sorted, int32_t* inv, void* x_perm_bf16,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t moe_permute_workspace_size(int32_t T, int32_t k, int32_t E);

/*
 * moe_permute without a workspace, for callers that cannot allocate device
 * memory.  (No counterpart in the method; this is an interface for callers.)
 *
 * Who needs it: a host runtime that reserves all of its device memory at
 * start-up and refuses allocations afterwards (a fixed-pool serving engine),
 * code that runs where allocating CUDA calls are not allowed (a host function
 * enqueued with cudaLaunchHostFunc), or a C program that owns only its input
 * and output buffers.  Such a caller passes inputs and outputs exactly as for
 * moe_permute; the scratch lives in a fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes of device global memory that belongs to the
 * library image, held by every GPU that loads the library until the process
 * exits.  Nothing is allocated or freed by this call.
 *
 *   - T * k above MOE_NOALLOC_MAX_ROWS returns MOE_ERR_SCRATCH_LIMIT and
 *     launches nothing.  Other argument errors as for moe_permute.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address and caches it; make that first call before any
 *     stream capture.  A first call made while `stream` is capturing returns
 *     MOE_ERR_CAPTURE, launches nothing and leaves the capture intact (the
 *     lookup could load device code, which a capture does not allow).
 *   - All calls share the one array and it keeps the last call's contents
 *     (the call rewrites every part it reads, so no clearing is needed).
 *     Calls that overlap on the GPU -- on different streams or from different
 *     host threads on one device -- race on it and must be serialised.
 *   - There is no error word to read back: ids outside [0, E) are skipped,
 *     so the sum of counts falls short of T * k.
 */
#define MOE_NOALLOC_MAX_ROWS 32768
#define MOE_NOALLOC_SCRATCH_BYTES (160 * 1024)
moe_status_t moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                 const void* x_bf16, int32_t d, int32_t* counts, int32_t* offsets,
                                 int32_t* sorted, int32_t* inv, void* x_perm_bf16, cudaStream_t stream);

/*
 * Stage 3 -- grouped expert FFN on the permuted rows.  "Performance and
 * verification", section "Why it is fast" (grouped tensor-core GEMMs for the
 * routed experts of a prompt; arithmetic directly on the packed codes) and
 * "Measured results", section Speed (W4A16 g128; prefill dequantises to
 * 16-bit for a dense GEMM).
 *
 * For every expert e and every permuted row i in offsets[e]..offsets[e+1]-1:
 *   g = x_perm[i] . Wg[e]^T,  u = x_perm[i] . Wu[e]^T      (fp32 accumulation)
 *   h = SiLU(g) * u,   SiLU(g) = g / (1 + exp(-g))   (intermediate: fp32 in the
 *                      GEMV regime, rounded to fp16 in the tensor-core regime)
 *   y_perm[i] = (row_w ? row_w[i] : 1) * (h . Wd[e]^T)      the output, rounded to bf16
 * Experts with no rows are not read.  Two regimes, chosen from R on the host:
 * a CUDA-core GEMV for few rows and a tcgen05 tensor-core grouped GEMM for
 * many (override with the environment variable MOE_W4_REGIME=decode|prefill).
 * Intermediate precision: the GEMV keeps h in fp32; the tensor-core regime
 * runs fp16 x fp16 -> fp32 MMAs (activations converted exactly from bf16,
 * weights (q - z) * s rounded once to fp16, h in fp16), so |x|, |h| and, inside
 * moe_layer_forward, |y| must stay below 65504 there; a value outside fp16's
 * range is reported as MOE_ERR_F16_RANGE by moe_get_device_error.
 *
 *   x_perm   device bf16 [R][d_model]
 *   offsets  device int32 [E+1], offsets[0] = 0, offsets[E] = R, non-decreasing
 *   row_w    device fp32 [R] or NULL
 *   y_perm   device bf16 [R][d_model] (out)
 * Workspace: >= moe_expert_ffn_workspace_size(L, R) bytes.
 */
moe_status_t moe_expert_ffn_w4a16(const moe_w4_layer* L, const void* x_perm_bf16,
                                  const int32_t* offsets, int32_t R, const float* row_w,
                                  void* y_perm_bf16, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);
size_t moe_expert_ffn_workspace_size(const moe_w4_layer* L, int32_t R);

/*
 * Stage 4 -- combine.  out[t] = sum over j = 0..k-1 of
 * topk_w[t][j] * y_perm[inv[t*k + j]], accumulated in fp32 in slot order and
 * rounded to bf16 (nearest even).
 *
 *   y_perm device bf16 [T*k][d], inv device int32 [T*k], topk_w device fp32 [T][k]
 *   out    device bf16 [T][d] (out)
 * inv must be a permutation of 0..T*k-1; an entry outside that range is
 * skipped (its term contributes nothing) rather than read out of bounds.
 */
moe_status_t moe_combine(const void* y_perm_bf16, const int32_t* inv, const float* topk_w,
                         int32_t T, int32_t k, int32_t d, void* out_bf16, cudaStream_t stream);

/*
 * The whole layer: stages 1-4 on one stream, nothing allocated, no host sync.
 * With T <= 8 and T*k <= 64 the layer runs as ONE kernel (routing repeated in
 * every CTA, gate_up, one grid barrier, down with the combine fused; one CTA
 * per SM, cooperative launch).  Consecutive calls on a stream may be launched
 * as programmatic dependents of the previous kernel: a call's CTAs start their
 * shared-memory setup early but read and write no global memory (inputs,
 * outputs, workspace) before the previous kernel on the stream has completed,
 * so stream order is unchanged; early on they only hint L2 to fetch x and
 * logits, a prefetch that returns no value.  Its intermediate precision: activations and h
 * in fp16 (|x|, |h| < 65504, else MOE_ERR_F16_RANGE), products of the exact
 * int4 codes with fp32 accumulation, zero and scale applied per group of 128
 * in fp32.  MOE_W4_DECODE_KERNEL=split runs the stage chain instead.
 *
 *   x        device bf16 [T][d_model]
 *   logits   device fp32 [T][E]
 *   out      device bf16 [T][d_model] (out)
 *   topk_ids_out  device int32 [T][k] or NULL: the routing actually used
 * Workspace: >= moe_layer_workspace_size(L, T, k) bytes; it also holds the
 * device error word that moe_get_device_error reads.
 */
moe_status_t moe_layer_forward(const moe_w4_layer* L, const void* x_bf16, const float* logits,
                               int32_t T, int32_t k, void* out_bf16, int32_t* topk_ids_out,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t moe_layer_workspace_size(const moe_w4_layer* L, int32_t T, int32_t k);

/*
 * Reads and clears the device error word kept at the start of a workspace
 * used by moe_permute, moe_expert_ffn_w4a16 or moe_layer_forward.  Waits for
 * `stream` to finish.  When it reports an error it clears the whole 256-byte
 * header, which also holds the grid-barrier counter of the one-kernel decode
 * layer (a call that gave up can leave that counter inconsistent).  Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_RANGE
 * or MOE_ERR_F16_RANGE, in that order of precedence (or MOE_ERR_CUDA if the
 * copy fails).
 */
moe_status_t moe_get_device_error(void* workspace, cudaStream_t stream);

/*
 * Diagnostics (no counterpart in the method; used by the benchmark).
 *
 * moe_profile_stages: while `events` is non-NULL, every moe_layer_forward
 * call made from this host thread records six caller-created CUDA events on
 * its stream, at events[*cursor + 0..5], and advances *cursor by 6:
 *   0 start, 1 after routing, 2 after the permutation, 3 after gate_up,
 *   4 after down (the decode regime's down kernel also combines), 5 end.
 * Nothing is recorded once fewer than 6 slots remain.  Pass NULL to stop.
 * The events are recorded as external events, so a call captured into a CUDA
 * graph records them on every replay of the graph.
 * `events` and `cursor` are host memory owned by the caller.
 *
 * moe_kernel_launches: number of CUDA kernels this library has launched in
 * this process (all threads, all devices).
 */
moe_status_t moe_profile_stages(cudaEvent_t* events, int32_t capacity, int32_t* cursor);
uint64_t moe_kernel_launches(void);

/* Human-readable name of a status code (static storage). */
const char* moe_status_str(moe_status_t status);

/* Library version string, e.g. "moe_w4 1.0 sm_103a". */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4_H */
