// Internal declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// Rows per grouped-GEMM block (and the largest MMA N).  An expert with c rows
// becomes ceil(c / kBlockRowsMax) blocks; each block's MMA N is its row count
// rounded up to 16.
constexpr int kBlockRowsMax = 256;
// Smallest block of the grouped GEMMs' block list (a measurement option;
// the MMA N of such a block is still at least 32).
constexpr int kBlockRowsMin = 16;
// Tokens per routing block (one 32-bit mask word per expert per block).
constexpr int kRouteBlockTokens = 32;

// Device status codes of a prefill intermediate (h, o) outside the fp16
// range (the bounded-wait timeout codes are 0x1xx).
constexpr int kDevRangeH = 0x201;
constexpr int kDevRangeO = 0x202;

enum GemmMode : int { MODE_ROUTER = 0, MODE_GATEUP = 1, MODE_DOWN = 2 };
// In-shared-memory conversion of the weight (A) tile before the MMA: none,
// bf16 -> fp16 in place, or int4 codes -> bf16 / fp16, symmetric (one bf16
// scale per 64 along K) or affine (a bf16 scale and bias per 64).
enum GemmConv : int {
  CONV_NONE = 0,
  CONV_BF16_TO_F16 = 1,
  CONV_INT4_TO_BF16 = 2,
  CONV_INT4_TO_F16 = 3,
  CONV_INT4A_TO_BF16 = 4,
  CONV_INT4A_TO_F16 = 5
};
__host__ __device__ constexpr bool conv_int4(int c) { return c >= CONV_INT4_TO_BF16; }
__host__ __device__ constexpr bool conv_affine(int c) { return c >= CONV_INT4A_TO_BF16; }
__host__ __device__ constexpr bool conv_to_f16(int c) {
  return c == CONV_BF16_TO_F16 || c == CONV_INT4_TO_F16 || c == CONV_INT4A_TO_F16;
}

struct GemmParams {
  int mode;
  const void *a_routed;      // weights (A, K-major bf16): router / gate_up / down
  const void *a_shared;      // shared-expert weights for the same role (or = a_routed)
  int lda_routed;            // elements per A row
  int lda_shared;
  int a_rows_routed;         // rows of the A tensors (rows past them read as zeros)
  int a_rows_shared;
  const int4 *blocks;        // grouped modes: {expert (E = shared), row_start, n_rows, 0}
  const int *n_blocks_dev;   // grouped modes: block count in device memory
  int n_blocks_host;         // router: token blocks
  int block_rows;            // router: tokens per block
  int T;                     // tokens of the chunk
  int m_tiles;               // weight-row tiles per block
  int n_experts;             // E
  int hidden;                // H
  int inter_routed;          // I
  int inter_shared;          // Is
  int k_routed;              // reduction length (router, gate/up: H)
  int shared_row0;           // first grouped row of the shared expert (T*k)
  void *out;                 // router: fp32 [T,E]; gate/up: fp16 h [R,ld]; down: fp16 o [R,H]
  int out_ld;                // elements per output row
  const float *bias;         // router bias or null
  int *status;               // device status word
  const void *a_scale_routed;   // int4 weights: bf16 scales [rows, K/64] (else null)
  const void *a_scale_shared;
  const void *a_bias_routed;    // affine int4 weights: bf16 biases [rows, K/64] (else null)
  const void *a_bias_shared;
  int ab_f16;                // CONV_NONE only: A and B are fp16 (else bf16)
  int fixed_n;               // grouped modes: MMA N = kBlockRowsMax for every block (measurement)
  int k_split;               // router: split-K parts (>= 1); part s writes out + s * out_split_stride
  size_t out_split_stride;   // router: floats between split-K parts of `out`
};

cudaError_t gemm_configure();
// Weight rows one GEMM tile covers (a CTA pair, 128 rows per CTA).
int gemm_pair_rows();
// Largest persistent grid (CTAs, whole pairs) whose clusters are co-resident.
int gemm_max_grid(int num_sms);
// `pdl` (here and below): programmatic dependent launch on the previous
// kernel of the stream (the kernel waits for it before reading its inputs).
// a_routed, a_shared: the weight maps (router: 2-D {K, E}, box {64, 128};
// gate/up: 3-D {K, I, 2 E} (2 for the shared expert), box {64, 64, 2}; down:
// 2-D {K, rows}, box {64, 128}; int4: 2-D code maps, box {32 bytes, 64 or
// 128}).  b, b2: token-row maps of one matrix each, boxes of 64 elements x
// (16 << i) rows for i = 0..3 (b: x for the router, x in grouped order for
// gate/up, h for down; b2: x, for the shared expert's gate/up tiles).
cudaError_t launch_tc_gemm(const CUtensorMap &a_routed, const CUtensorMap &a_shared,
                           const CUtensorMap (&b)[4], const CUtensorMap (&b2)[4],
                           const GemmParams &p, int conv, int grid, bool pdl, cudaStream_t stream);

// Routing: top-k + masks, then the placement (counts, offsets, block map,
// stable scatter, shared gate, grouped copy of x).
// Top-k over logits = sum of nsplit parts (part s at partial + s * split_stride,
// summed in order s = 0, 1, ...); writes the sums to logits_out if non-null.
cudaError_t launch_topk(const float *partial, int nsplit, size_t split_stride, float *logits_out,
                        int T, int E, int k, int32_t *idx, float *w, uint32_t *blk_mask, bool pdl,
                        cudaStream_t stream);
// After the top-k kernel: the per-expert counts and segment offsets
// (offsets[E] = T * k), each assignment's grouped row (pos_of_assign) and
// its inverse (sorted_rows), and the block map of the grouped GEMMs
// (block_rows in kBlockRowsMin..kBlockRowsMax rows per block).  With xg
// non-null, also writes xg[pos(t, j)] = x[t] (x [T, H] bf16, xg [T * k, H]
// bf16: the token rows in grouped order, the routed gate/up GEMM's B
// operand); with gate non-null, gate[t] = sigmoid(x[t] . wsg) (wsg [H] bf16).
cudaError_t launch_place(const int32_t *idx, const uint32_t *blk_mask, int T, int E, int k,
                         int32_t *counts, int32_t *offsets, int4 *blocks, int32_t *n_blocks,
                         int block_rows, int32_t *sorted_rows, int32_t *pos_of_assign,
                         const void *x, void *xg, const void *wsg, float *gate, int H, bool pdl,
                         cudaStream_t stream);

// y[t] = sum_j w[t,j] o[pos(t,j)] + g[t] o[T*k + t]
cudaError_t launch_combine(const float *gate, const void *o, const int32_t *pos, const float *w,
                           int T, int H, int k, void *y, bool pdl, cudaStream_t stream);

// int4 codes [rows, K/2] (+ bf16 scales, and biases if affine, [rows, K/64])
// -> bf16 or fp16 weights [rows, K], rounded as the grouped GEMMs round them.
cudaError_t launch_dequant_int4(const void *codes, const void *scale, const void *bias, void *dst,
                                size_t rows, int K, bool affine, bool out_f16,
                                cudaStream_t stream);
// dst[i] = fp16(src[i]) (round to nearest even), n elements, 16-byte aligned.
cudaError_t launch_convert_bf16_to_f16(const void *src, void *dst, size_t n, cudaStream_t stream);

// Batch-1 decode.
struct DecodeParams {
  const void *x;             // bf16 [H]
  void *y;                   // bf16 [H]
  int H, E, k, I, Is, wfmt;
  const void *router_w;
  const float *router_b;
  const void *gate_up, *gate_up_scale, *down, *down_scale;
  const void *sh_gate_up, *sh_gate_up_scale, *sh_down, *sh_down_scale;
  const void *sh_gate_w;
  // affine int4 (wfmt 2): bf16 biases [rows, K/64] beside the scales (else null)
  const void *gate_up_bias, *down_bias, *sh_gate_up_bias, *sh_down_bias;
  float *logits;             // [E]
  int32_t *idx;              // [k]
  float *w;                  // [k]
  float *g;                  // [1]
  float *h;                  // [(k+1) h_ld] fp32: h of the k experts, then of the shared expert
  int h_ld;                  // max(I, Is)
  unsigned long long *bar;   // grid-barrier arrival counter (16-byte slot, zeroed once)
  unsigned long long *phase_ts;   // null, or [gridDim.x][2]: global-timer ns at the start and
                                  // the end of phase B in each CTA (profiling only)
  int *status;               // device status word
  int p3_rows, p3_stage;     // set by launch_decode_layer
  int p3_scales;             // set by launch_decode_layer: int4 scales (biases) staged too
  int T;                     // launch_rows: rows of x and y (x, y [T, H]; logits [T, E];
                             // idx, w [T, k]; g [T]; h [T][k + 1][h_ld]); 1 otherwise
};
// Up to kMaxDecodeLayers layers (same shapes) for one multi-layer decode launch.
constexpr int kMaxDecodeLayers = 48;
struct DecodeLayersParams {
  DecodeParams layer[kMaxDecodeLayers];
  int n;
};
// CTAs whose phase-B stamps the workspace holds (profiling).
constexpr int kMaxPhaseCtas = 1024;
// Floats of the h region a decode needs.
inline size_t decode_h_floats(int k, int h_ld) { return (static_cast<size_t>(k) + 1) * h_ld; }
// Raises the decode kernel's dynamic shared-memory limit on the current
// device to the device maximum and returns it in *smem_limit.
cudaError_t decode_configure(int *smem_limit);
// Co-resident grid of the decode layer kernel.
int decode_layer_grid(int num_sms);
// One decode layer (see decode.cu): a cooperative launch of decode_layer_grid
// CTAs, with at most smem_limit bytes of dynamic shared memory; `pdl` lets it
// start while the previous kernel in the stream finishes.
cudaError_t launch_decode_layer(const DecodeParams &p, int grid, int smem_limit, bool pdl,
                                cudaStream_t stream);
// n consecutive layers (1 <= n <= kMaxDecodeLayers) in one launch of the
// same grid: layer l + 1 starts after a grid barrier behind layer l's outputs.
cudaError_t launch_decode_layers(const DecodeParams *layers, int n, int grid, int smem_limit,
                                 bool pdl, cudaStream_t stream);
// A few rows (1 <= p.T <= kSmallMaxRows) of one layer in one cooperative
// launch of the decode grid: every weight row the rows need is streamed once
// for all of them (see decode.cu).
constexpr int kSmallMaxRows = 16;
cudaError_t launch_rows(const DecodeParams &p, int grid, int smem_limit, bool pdl,
                        cudaStream_t stream);

// Reads and clears the device status word of moe_forward_decode_noalloc on
// the current device, after waiting for the device (decode_noalloc.cu).
// Returns false if a CUDA call fails.
bool noalloc_status_read_clear(int32_t *code);

}  // namespace moe
