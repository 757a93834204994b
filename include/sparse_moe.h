/*
 * sparse_moe.h -- C ABI of the GB300 (sm_103a) sparse mixture-of-experts layer.
 *
 * The layer is the one described in "Optimizing On-Device Inference for Apple
 * Silicon" (Perplexity):
 *   - section "Qwen creates three distinct workload shapes": a router scores E
 *     experts and selects k per token; one shared expert processes every token;
 *   - section "Keep expert routing on the GPU": histogram, prefix scan,
 *     scatter and block map, all enqueued with no host synchronisation;
 *   - section "Dequantize weights during matrix multiplication": grouped expert
 *     GEMM with fp32 accumulation, bf16 output, optional 4-bit weights expanded
 *     one tile at a time in on-chip memory;
 *   - section "Match tile size to expert load": tile shapes follow each
 *     expert's row count;
 *   - section "Optimize the one-row weight path" and "Reduce intermediate and
 *     state traffic": batch-1 decode as a row-parallel GEMV with the gate/up
 *     projections fused with the gated activation and the output projection
 *     fused with the routing score and the shared-expert result;
 *   - section "Bound temporary memory with prompt chunking": long prompts run
 *     in bounded chunks with unchanged output.
 *
 * For each token t (x[t] in bf16):
 *   l[t,e]   = sum_h x[t,h] * Wr[e,h] (+ b[e])              fp32 accumulate
 *   idx[t,:] = the k largest l[t,:], descending; equal logits -> lower e first
 *   w[t,j]   = exp(l[t,idx_j]) / sum_j' exp(l[t,idx_j'])       (= softmax over
 *              all experts, renormalised over the selected ones)
 *   h_e(x)   = silu(Wg_e x) * (Wu_e x),   silu(z) = z / (1 + exp(-z))
 *   y[t]     = sum_j w[t,j] * Wd_{idx_j} h_{idx_j}(x[t])
 *              + sigmoid(x[t] . w_sg) * Sd h_shared(x[t])       bf16 output
 *
 * Layouts (row-major; every weight is K-major, i.e. each output row is
 * contiguous along the reduction dimension):
 *   x, y          bf16  [T, H]
 *   router_w      bf16  [E, H]            router_b  fp32 [E] or NULL
 *   gate_up       bf16  [E, 2I, H]        rows 0..I-1 gate, I..2I-1 up
 *   down          bf16  [E, H, I]
 *   sh_gate_up    bf16  [2Is, H]          rows 0..Is-1 gate, Is..2Is-1 up
 *   sh_down       bf16  [H, Is]
 *   sh_gate_w     bf16  [H]
 * int4 symmetric group-64 format (wfmt = MOE_W_INT4_SYM_G64), for gate_up,
 * down, sh_gate_up and sh_down:
 *   <w>           uint8 [rows, K/2]  element 2m in the low nibble of byte m,
 *                                    element 2m+1 in the high nibble, each a
 *                                    two's-complement code q in [-8, 7]
 *   <w>_scale     bf16  [rows, K/64] weight = scale[r, k/64] * q[r, k]
 * int4 affine group-64 format (wfmt = MOE_W_INT4_AFFINE_G64), the checkpoint
 * format of "Dequantize weights during matrix multiplication" (a bf16 scale
 * and a bf16 bias per group of 64 weights), same tensors plus:
 *   <w>           uint8 [rows, K/2]  as above, but each code an unsigned q in
 *                                    [0, 15]
 *   <w>_bias      bf16  [rows, K/64] weight = scale[r, k/64] * q[r, k]
 *                                             + bias[r, k/64]
 * The router and sh_gate_w stay bf16 in every format.
 *
 * Routing outputs (moe_route), per chunk of T tokens, assignment a = t*k + j:
 *   counts[e]          number of assignments to expert e             int32 [E]
 *   offsets[e]         exclusive prefix sum of counts, offsets[E]=T*k int32 [E+1]
 *   sorted_rows[p]     token of grouped row p; inside an expert's segment
 *                      [offsets[e], offsets[e+1]) tokens ascend      int32 [T*k]
 *   pos_of_assign[a]   grouped row of assignment a                  int32 [T*k]
 *
 * Ownership: all device memory (weights, activations, workspace) belongs to
 * the caller.  The context borrows weight pointers from moe_load_weights until
 * the slot is reloaded or the context is destroyed, and carves its workspace
 * out of the caller's buffer.  Pointers marked "device" must be device memory
 * of the context's device; every device pointer must be 16-byte aligned.
 *
 * Streams: every compute call is asynchronous on `stream` (a cudaStream_t
 * passed as void*, NULL = legacy default stream) and never synchronises the
 * host.  Calls on one context must not overlap in time (they share the
 * workspace); a context is not thread-safe.
 *
 * Errors: every entry returns a moe_status.  Arguments are checked before any
 * launch; on failure nothing is enqueued and moe_last_error() explains why.
 * Launch errors are returned as MOE_ERR_CUDA.  Kernels never spin without a
 * bound: a wait that runs out records a code in a device status word, the
 * kernel returns, and moe_check_device() reports MOE_ERR_DEVICE_TIMEOUT.
 */
#ifndef SPARSE_MOE_H
#define SPARSE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* NULL, misaligned or out-of-range argument      */
  MOE_ERR_UNSUPPORTED = 2,     /* shape or format the library does not implement */
  MOE_ERR_WORKSPACE = 3,       /* workspace missing, too small or misaligned     */
  MOE_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed              */
  MOE_ERR_NOT_LOADED = 5,      /* weights of the requested layer slot not loaded */
  MOE_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait ran out             */
  MOE_ERR_RANGE = 7            /* a prefill intermediate left the fp16 range     */
} moe_status;

typedef enum {
  MOE_W_BF16 = 0,              /* all weights bf16                                */
  MOE_W_INT4_SYM_G64 = 1,      /* expert + shared-expert weights int4, group 64   */
  MOE_W_INT4_AFFINE_G64 = 2    /* the same, unsigned codes with a scale and bias  */
} moe_wfmt;

typedef struct {
  int hidden;          /* H: multiple of 64, 64..16384                         */
  int n_experts;       /* E: 1..1024                                           */
  int top_k;           /* k: 1..min(E, 32)                                     */
  int inter;           /* I: expert intermediate size, multiple of 64          */
  int shared_inter;    /* Is: shared-expert intermediate size, multiple of 64  */
  int n_layers;        /* number of weight slots (layers) the context holds    */
  int max_chunk_rows;  /* prefill rows per chunk (1..65536); longer prompts run
                          chunk by chunk with identical per-token results      */
  int wfmt;            /* moe_wfmt                                             */
} moe_config;

typedef struct {       /* device pointers, borrowed (see Ownership above)      */
  const void  *router_w;          /* bf16 [E, H]                               */
  const float *router_b;          /* fp32 [E] or NULL                          */
  const void  *gate_up;           /* bf16 [E, 2I, H] | uint8 [E, 2I, H/2]      */
  const void  *gate_up_scale;     /* NULL (bf16)     | bf16  [E, 2I, H/64]     */
  const void  *down;              /* bf16 [E, H, I]  | uint8 [E, H, I/2]       */
  const void  *down_scale;        /* NULL (bf16)     | bf16  [E, H, I/64]      */
  const void  *sh_gate_up;        /* bf16 [2Is, H]   | uint8 [2Is, H/2]        */
  const void  *sh_gate_up_scale;  /* NULL (bf16)     | bf16  [2Is, H/64]       */
  const void  *sh_down;           /* bf16 [H, Is]    | uint8 [H, Is/2]         */
  const void  *sh_down_scale;     /* NULL (bf16)     | bf16  [H, Is/64]        */
  const void  *sh_gate_w;         /* bf16 [H]                                  */
  /* Optional (bf16 format only; both or neither, else NULL): fp16 copies of
   * down and sh_down, same shapes, each value the round-to-nearest fp16 of
   * the bf16 one (moe_convert_bf16_to_f16 writes them).  The prefill down
   * projection runs on fp16 operands (h is stored in fp16 for its 11
   * significant bits); given these copies its weight tiles go from TMA
   * straight to the tensor cores instead of being converted in shared memory
   * first, with bit-identical results.  Decode never reads them. */
  const void  *down_f16;          /* fp16 [E, H, I] or NULL                    */
  const void  *sh_down_f16;       /* fp16 [H, Is]   or NULL                    */
  /* Affine int4 only (else NULL): the per-group biases, bf16 [rows, K/64] of
   * gate_up, down, sh_gate_up, sh_down. */
  const void  *gate_up_bias;
  const void  *down_bias;
  const void  *sh_gate_up_bias;
  const void  *sh_down_bias;
} moe_weights;

/* Bytes of device workspace a context with this config needs (host only). */
moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes);

/* Validates cfg, binds to `device`, carves `workspace` (device memory,
 * 256-byte aligned, >= moe_workspace_size bytes, owned by the caller and kept
 * alive until moe_ctx_destroy) and returns a context in *out.  Host-side set-up
 * only: it enqueues one zero-fill of the workspace's status words on the legacy
 * default stream and waits for it. */
moe_status moe_ctx_create(const moe_config *cfg, int device, void *workspace,
                          size_t ws_bytes, moe_ctx **out);

/* Frees the host-side context (the workspace and weights stay the caller's). */
moe_status moe_ctx_destroy(moe_ctx *ctx);

/* Records the device pointers of one layer slot (0 <= layer < n_layers) and
 * encodes the TMA tensor maps for them.  Host-side only; no device work. */
moe_status moe_load_weights(moe_ctx *ctx, int layer, const moe_weights *w);

/* Routing only ("Keep expert routing on the GPU"): router logits, top-k,
 * renormalised weights, histogram, exclusive scan and the stable scatter for
 * T tokens, 1 <= T <= max_chunk_rows (T = 0 is a no-op).  x is device bf16
 * [T, H]; outputs are device arrays of the sizes in the header comment:
 * logits fp32 [T, E] (may be NULL), topk_idx int32 [T, k], topk_w fp32 [T, k],
 * counts int32 [E], offsets int32 [E+1], sorted_rows int32 [T*k],
 * pos_of_assign int32 [T*k].  The same kernels run inside
 * moe_forward_prefill, so its routing is bitwise the one returned here. */
moe_status moe_route(moe_ctx *ctx, int layer, const void *x, int T,
                     float *logits, int32_t *topk_idx, float *topk_w,
                     int32_t *counts, int32_t *offsets,
                     int32_t *sorted_rows, int32_t *pos_of_assign, void *stream);

/* Prefill: y[T, H] = MoE(x[T, H]) for T >= 0 tokens (device bf16 in and out,
 * x and y must not overlap).  T > max_chunk_rows runs chunk by chunk
 * ("Bound temporary memory with prompt chunking").  With int4 weights the
 * grouped GEMMs dequantise each weight tile in shared memory right before its
 * MMA ("Dequantize weights during matrix multiplication"): no expanded copy
 * of the weights is ever written.
 *   Range: the prefill path keeps the two per-row intermediates in fp16 (11
 *   significant bits, finite up to 65504): h = silu(gate) * up of every
 *   routed and shared expert, and o, each expert's output row.  The kernels
 *   check both as they store them; if one is not finite or beyond 65504 in
 *   magnitude (activations about 70 times larger than unit-variance inputs
 *   through N(0, 0.02) weights), y is not valid and moe_check_device()
 *   reports MOE_ERR_RANGE.  The decode and few-rows paths keep these values
 *   in fp32 and have no such limit.  Down-projection weights below 2^-17 in
 *   magnitude keep fewer than 8 significant bits in the fp16 operands. */
moe_status moe_forward_prefill(moe_ctx *ctx, int layer, const void *x, int T,
                               void *y, void *stream);

/* Batch-1 decode: y[1, H] = MoE(x[1, H]) with the GEMV path (device bf16). */
moe_status moe_forward_decode(moe_ctx *ctx, int layer, const void *x, void *y,
                              void *stream);

/* Batch-1 decode of layer slots first_layer .. first_layer + n_layers - 1 in
 * order, for a caller that has their inputs at hand (or chains them), in one
 * persistent launch per up to 48 layers instead of one per layer: layer l
 * reads x + l * x_stride and writes y + l * y_stride (device bf16 rows of H;
 * strides in elements, multiples of 8, 0 allowed for x).  It computes exactly
 * what moe_forward_decode computes for each layer, with the same arithmetic.
 * Layer l + 1 starts only after every CTA has written layer l's output (a
 * grid barrier), so its input may be layer l's output (x + (l + 1) *
 * x_stride == y + l * y_stride): a layer's output is written after its last
 * read of its input.  Only the next layer's weights (its router, shared gate
 * and shared expert, which do not depend on the routing) are fetched ahead,
 * during the current layer's output projection.  Layers must be loaded;
 * n_layers = 0 is a no-op.  Afterwards moe_decode_routing reports the last
 * layer's routing. */
moe_status moe_forward_decode_layers(moe_ctx *ctx, int first_layer, int n_layers,
                                     const void *x, size_t x_stride, void *y,
                                     size_t y_stride, void *stream);

/* Routing of the most recent moe_forward_decode on this context, copied
 * (asynchronously, on `stream`) to device buffers: logits fp32 [E] (may be
 * NULL), idx int32 [k], w fp32 [k] (either may be NULL). */
moe_status moe_decode_routing(moe_ctx *ctx, float *logits, int32_t *idx, float *w,
                              void *stream);

/* A few rows through the decode-style path: y[T, H] = MoE(x[T, H]) for
 * 1 <= T <= 16 (and T <= the context's max_chunk_rows), device bf16, 16-byte
 * aligned, in one cooperative launch of the decode grid.  Section "Limits of
 * further optimization": verifying drafted tokens processes groups of two to
 * five rows that often select different experts, so the weights read grow
 * with the union of the rows' experts.  Here every weight row in that union
 * (and of the router and the shared expert) is read from HBM once for all
 * the rows that need it; the prefill path would instead run its routing and
 * grouped GEMMs for a handful of rows.  int4 weights, and bf16 weights
 * with T < 5: the arithmetic of moe_forward_decode, operation for
 * operation.  bf16 weights with T >= 5: the gate/up dot products run on the
 * tensor cores (fp32 accumulation, every weight byte loaded once for all
 * rows), the rest as in moe_forward_decode; the tolerances are the
 * decode's.  Row t's result does not depend on the values of the other
 * rows.  Uses the workspace's prefill regions: do not overlap
 * with a prefill call on the same context.  Errors: MOE_ERR_INVALID_ARG for
 * T out of range or misaligned buffers. */
moe_status moe_forward_rows(moe_ctx *ctx, int layer, const void *x, int T, void *y,
                            void *stream);

/* Routing of the most recent moe_forward_rows (T rows) on this context,
 * copied asynchronously on `stream` to device buffers: logits fp32 [T, E],
 * idx int32 [T, k], w fp32 [T, k] (any may be NULL).  Valid until the next
 * prefill or rows call; MOE_ERR_INVALID_ARG before the first rows call. */
moe_status moe_rows_routing(moe_ctx *ctx, float *logits, int32_t *idx, float *w, void *stream);

/* End-to-end prefill from HOST memory: copies x_host [T, H] bf16 to the
 * device chunk by chunk, runs the prefill path and copies y back into y_host
 * [T, H].  Pinned host buffers make the copies asynchronous; the call returns
 * once the work is enqueued (synchronise `stream` before reading y_host).
 * The input copies run on the context's own copy stream through two staging
 * slots, so that a chunk's input copy overlaps the previous chunk's (or the
 * previous call's) compute.  A page-locked y_host is written directly by the
 * combine kernel (it is addressable from the device); a pageable one through
 * a staging slot and an output copy on a second copy stream, which overlaps
 * the next chunk's compute.  The layer's kernels are ordered after earlier
 * work on `stream`, but the input copy is not: x_host must hold the input
 * when the call is made. */
moe_status moe_forward_prefill_host(moe_ctx *ctx, int layer, const void *x_host,
                                    int T, void *y_host, void *stream);

/* Same for one decode token (x_host, y_host: bf16 [H] in host memory); a
 * page-locked y_host is written by the decode kernel directly. */
moe_status moe_forward_decode_host(moe_ctx *ctx, int layer, const void *x_host,
                                   void *y_host, void *stream);

/* Batch-1 decode that allocates nothing (the page has no counterpart: this is
 * an interface for callers that cannot allocate device memory, such as code
 * inside a host framework that forbids allocation on this path or owns a
 * fixed device-memory budget, and therefore cannot provide the workspace a
 * context needs).  It computes exactly what moe_forward_decode computes,
 * with the same kernel, for x[1, H] -> y[1, H] (device bf16, 16-byte
 * aligned) and the weights in `w` (device pointers, as for moe_load_weights);
 * `cfg` supplies the shape and weight format (n_layers and max_chunk_rows
 * are ignored).
 *   Scratch: the per-token intermediates live in one fixed device array
 *   inside the library, 64 KiB, held by every device that loads the library
 *   until the process exits.  Shapes whose intermediates need more (E + 2k +
 *   (k + 1) * max(I, Is) floats plus alignment) are rejected with
 *   MOE_ERR_WORKSPACE; nothing is launched then.
 *   Set-up: the first call on each device looks up the array's device
 *   address (with that device current) and raises the decode kernel's
 *   shared-memory limit; make that first call before any stream capture.
 *   The cached set-up belongs to the device's primary context: it assumes
 *   one primary context per device for the life of the process (no
 *   cudaDeviceReset between calls).
 *   Sharing: every call uses the same array, which keeps the previous call's
 *   contents; calls that overlap on the GPU (different streams, or several
 *   host threads) race on it, so serialise them.
 *   Launch: programmatic dependent launch is on unless the environment
 *   variable MOE_DECODE_PDL is 0 when the first call on a device is made, the
 *   same switch as a context's decode launches.
 *   Device waits: the call returns before its kernel runs, so a bounded wait
 *   that runs out cannot change its return value; the kernel records the
 *   site in a status word inside the array, which moe_check_device(NULL,
 *   &code) reads and clears.
 * Returns MOE_ERR_INVALID_ARG for bad arguments, MOE_ERR_UNSUPPORTED for
 * shapes the decode kernels do not take, MOE_ERR_CUDA if a CUDA call fails. */
moe_status moe_forward_decode_noalloc(const moe_config *cfg, const moe_weights *w,
                                      const void *x, void *y, void *stream);

/* dst[i] = fp16(src[i]) for 0 <= i < n: bf16 -> fp16 with round-to-nearest-
 * even (values beyond the fp16 range become +-inf, bf16 NaN stays NaN), on
 * the current device, asynchronously on `stream`.  src and dst are device
 * arrays of n 2-byte elements, 16-byte aligned, not overlapping.  Meant for
 * the optional down_f16 / sh_down_f16 weight copies.  Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned pointer with n > 0 (nothing
 * is launched), MOE_ERR_CUDA if the launch fails; n = 0 is a no-op. */
moe_status moe_convert_bf16_to_f16(const void *src, void *dst, size_t n, void *stream);

/* Expands int4 weights (wfmt MOE_W_INT4_SYM_G64 or MOE_W_INT4_AFFINE_G64;
 * codes uint8 [rows, K/2], scale bf16 [rows, K/64], bias bf16 [rows, K/64]
 * for the affine format, else ignored) into dst [rows, K], bf16 (out_f16 = 0)
 * or fp16 (out_f16 = 1), on the current device, asynchronously on `stream`.
 * Each value is rounded exactly as the grouped GEMMs round it when they expand
 * a weight tile in shared memory, so a bf16/fp16 layer on the expanded arrays
 * computes what the int4 layer computes.  This is the separate dequantisation
 * that "Dequantize weights during matrix multiplication" measures its fused
 * expansion against.  codes and dst 16-byte aligned; K a multiple of 64.
 * Returns MOE_ERR_INVALID_ARG for bad arguments (nothing launched),
 * MOE_ERR_CUDA if the launch fails; rows = 0 is a no-op. */
moe_status moe_dequant_int4(const void *codes, const void *scale, const void *bias, void *dst,
                            size_t rows, int K, int wfmt, int out_f16, void *stream);

/* Synchronises the device, reads and clears the device status word: MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT (a bounded wait ran out; *code, if non-NULL,
 * receives the site code), MOE_ERR_RANGE (a prefill intermediate left the
 * fp16 range since the last check; *code receives 0x201 for h, 0x202 for o),
 * or MOE_ERR_CUDA.  With ctx = NULL it does the
 * same for the status word of moe_forward_decode_noalloc on the current
 * device. */
moe_status moe_check_device(moe_ctx *ctx, int32_t *code);

/* Per-kernel timing with CUDA events recorded on the launching stream. */
typedef struct {
  char   name[32];     /* kernel family                                       */
  int64_t launches;    /* launches recorded since profiling was enabled       */
  double total_ms;     /* sum of event-measured durations                     */
} moe_kernel_stat;

/* While profiling is on, every launch also records CUDA events around it,
 * and decode launches stamp their phase B (moe_decode_phase_read).
 * Enabling clears the counts and the stamps. */
moe_status moe_profile_enable(moe_ctx *ctx, int on);
/* Synchronises the recorded events and returns up to `max` entries. */
moe_status moe_profile_read(moe_ctx *ctx, moe_kernel_stat *stats, int max, int *n);

/* Phase B of the most recent moe_forward_decode launched while profiling was
 * enabled (the k routed experts' gate/up rows streamed by every CTA, the
 * output-projection rows bulk-copied alongside): each CTA stamps the global
 * timer when its phase B starts (after the top-k) and ends.  Synchronises
 * the device; *window_us = latest end - earliest start over the CTAs,
 * *median_us = the median CTA's duration.  MOE_ERR_INVALID_ARG if no
 * profiled decode launch has stamped every CTA since profiling was enabled
 * on this context. */
moe_status moe_decode_phase_read(moe_ctx *ctx, double *window_us, double *median_us);

/* Number of kernels this context has launched since creation. */
int64_t moe_launch_count(const moe_ctx *ctx);

/* Human-readable description of the last failure on this context ("" if none). */
const char *moe_last_error(const moe_ctx *ctx);
const char *moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* SPARSE_MOE_H */
