// Batch-1 decode path (sections "Optimize the one-row weight path" and
// "Reduce intermediate and state traffic" of "Optimizing On-Device Inference
// for Apple Silicon"): with one activation row there is no weight reuse, so
// every kernel is a row-parallel GEMV on the vector ALUs that streams each
// weight row once with coalesced 128-bit loads.  One persistent cooperative
// launch per layer runs three phases separated by grid barriers:
//
//   1. router logits (+bias), the shared-expert gate sigmoid(x . w_sg) and the
//      shared expert's gate/up projections with SwiGLU (all only need x);
//   2. top-k selection (redone by every CTA from the logits in L2), then the
//      k routed experts' gate and up dot products;
//   3. the output projections of the k experts and of the shared expert,
//      fused with SwiGLU, the routing weights and the shared gate:
//      y[n] = sum_j w_j (Wd_j h_j)[n] + g (Sd h_s)[n], in fixed j order.
//
// Every warp issues all of its weight loads (and its slice of x, read
// straight from global memory) before any arithmetic, so each SM keeps a
// large number of 16-byte requests in flight; staying resident across the
// phases removes per-launch ramp-up and tails, which dominate a layer that
// moves 58 MB in a few microseconds.  int4 weights are read packed (32 codes per
// 128-bit load) and expanded in registers; each 16-byte chunk lies inside one
// 64-wide scale group.
#include "moe_internal.h"
#include "warp_topk.cuh"

namespace moe {

constexpr int kDecLayerThreads = 512;

// Optional phase timestamps (compiled only with -DMOE_TRACE): per CTA, clock64
// at each phase boundary of the last decode launch, read back with
// moe_debug_read_decode_trace().
#ifdef MOE_TRACE
__device__ long long g_dec_trace[1024][8];
#define DEC_MARK(i) \
  if (threadIdx.x == 0) g_dec_trace[blockIdx.x & 1023][i] = clock64()
#else
#define DEC_MARK(i)
#endif

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// 8 bf16 weights . 8 bf16 activations (one 16-byte chunk each)
__device__ __forceinline__ float dot8_bf16_bf16(const uint4 wv, const uint4 xv) {
  float a = bf16_lo(wv.x) * bf16_lo(xv.x);
  a = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), a);
  a = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), a);
  a = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), a);
  a = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), a);
  a = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), a);
  a = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), a);
  a = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), a);
  return a;
}

// 8 bf16 weights . 8 fp32 activations
__device__ __forceinline__ float dot8_bf16_f32(const uint4 wv, const float *xs) {
  const float4 x0 = *reinterpret_cast<const float4 *>(xs);
  const float4 x1 = *reinterpret_cast<const float4 *>(xs + 4);
  float a = bf16_lo(wv.x) * x0.x;
  a = fmaf(bf16_hi(wv.x), x0.y, a);
  a = fmaf(bf16_lo(wv.y), x0.z, a);
  a = fmaf(bf16_hi(wv.y), x0.w, a);
  a = fmaf(bf16_lo(wv.z), x1.x, a);
  a = fmaf(bf16_hi(wv.z), x1.y, a);
  a = fmaf(bf16_lo(wv.w), x1.z, a);
  a = fmaf(bf16_hi(wv.w), x1.w, a);
  return a;
}

// Signed code of nibble n (0..7) of a 32-bit word.
__device__ __forceinline__ float nib(uint32_t word, int n) {
  return static_cast<float>(static_cast<int>(word << (28 - 4 * n)) >> 28);
}

// 32 int4 codes (one 16-byte chunk; element n of word w is nibble n) . 32
// bf16 activations (four 16-byte chunks).  Returns sum q * x without the
// group scale.
__device__ __forceinline__ float dot32_int4_bf16(const uint4 wv, const uint4 (&xv)[4]) {
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
  float a = 0.0f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t xs[4] = {xv[w].x, xv[w].y, xv[w].z, xv[w].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      a = fmaf(nib(words[w], 2 * m), bf16_lo(xs[m]), a);
      a = fmaf(nib(words[w], 2 * m + 1), bf16_hi(xs[m]), a);
    }
  }
  return a;
}

// Same with 32 fp32 activations.
__device__ __forceinline__ float dot32_int4_f32(const uint4 wv, const float *xs) {
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
  float a = 0.0f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 x0 = *reinterpret_cast<const float4 *>(xs + 8 * w);
    const float4 x1 = *reinterpret_cast<const float4 *>(xs + 8 * w + 4);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int n = 0; n < 8; ++n) a = fmaf(nib(words[w], n), xv[n], a);
  }
  return a;
}

// Chunking of one weight row for a warp: 16-byte chunks of EPC elements;
// lane l takes chunks l + 32 u.  A segment is U chunks per lane (2048
// elements for both formats), whose x slice is U * XPC 16-byte bf16 chunks.
template <int WF> struct Fmt;
template <> struct Fmt<0> { static constexpr int EPC = 8, XPC = 1, U = 8; };
template <> struct Fmt<1> { static constexpr int EPC = 32, XPC = 4, U = 2; };

// Dot products of NR weight rows of length K with the bf16 vector x (global
// memory), by one warp.  All loads of a segment (weights first, then x) are
// issued before any arithmetic.
template <int WF, int NR>
__device__ __forceinline__ void warp_dots_x(const void *const (&rows)[NR],
                                            const __nv_bfloat16 *const (&srows)[NR], int K,
                                            const __nv_bfloat16 *x, float (&out)[NR]) {
  using F = Fmt<WF>;
  const int lane = threadIdx.x & 31;
  const int nchunk = K / F::EPC;
  const uint4 *xg = reinterpret_cast<const uint4 *>(x);
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
  for (int c0 = 0; c0 < nchunk; c0 += 32 * F::U) {
    uint4 wv[NR][F::U];
    uint4 xv[F::U][F::XPC];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < F::U; ++u) {
        const int c = c0 + lane + 32 * u;
        wv[r][u] = (c < nchunk) ? ld_stream(reinterpret_cast<const uint4 *>(rows[r]) + c)
                                : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int u = 0; u < F::U; ++u)
#pragma unroll
      for (int q = 0; q < F::XPC; ++q) {
        const int c = c0 + lane + 32 * u;
        xv[u][q] = (c < nchunk) ? __ldg(xg + c * F::XPC + q) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < F::U; ++u) {
        const int c = c0 + lane + 32 * u;
        if (c < nchunk) {
          if constexpr (WF == 0) {
            acc[r] += dot8_bf16_bf16(wv[r][u], xv[u][0]);
          } else {
            const float s = __bfloat162float(srows[r][c >> 1]);
            acc[r] = fmaf(s, dot32_int4_bf16(wv[r][u], xv[u]), acc[r]);
          }
        }
      }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

// Row r of a K-major matrix with K columns, bf16 or packed int4.
template <int WF>
__device__ __forceinline__ const void *row_ptr(const void *base, size_t r, int K) {
  return (WF == 0) ? static_cast<const void *>(reinterpret_cast<const __nv_bfloat16 *>(base) + r * K)
                   : static_cast<const void *>(reinterpret_cast<const uint8_t *>(base) + r * (K / 2));
}
__device__ __forceinline__ const __nv_bfloat16 *scale_row(const void *base, size_t r, int K) {
  return base ? reinterpret_cast<const __nv_bfloat16 *>(base) + r * (K / 64) : nullptr;
}

// ------------------------------------------------------ grid barrier --
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier across all CTAs of a cooperative launch (all co-resident).  The
// counter resets itself; the generation word only grows.  A CTA that waits
// longer than kWaitLimitCycles records DEV_TIMEOUT_GRID and carries on.
__device__ __forceinline__ void grid_barrier(unsigned int *count, unsigned int *gen, int *status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int g0 = ld_acquire_gpu(gen);   // read before arriving
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      const long long t0 = clock64();
      while (ld_acquire_gpu(gen) == g0) {
        if (clock64() - t0 > kWaitLimitCycles) {
          atomicExch(status, DEV_TIMEOUT_GRID);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// ------------------------------------------------- one decode layer --
// Persistent cooperative kernel, one CTA per SM, three phases:
//   1. router logits, shared gate sigmoid(x . w_sg), shared-expert SwiGLU h;
//   2. (every CTA) top-k of the logits, then the k routed experts' gate and
//      up dot products gu[j][r] = W_{e_j}[r] . x, one weight row per warp
//      item, two items in flight per warp;
//   3. y[n] = sum_j w_j (Wd_j h_j)[n] + g (Sd h_s)[n], one warp per n, with
//      h_j = silu(gu[j][:I]) * gu[j][I:] staged in shared memory.
// Each warp issues its first phase-3 weight loads before the last grid
// barrier, so they overlap the barrier and the staging of h.
template <int WF, int R, int KMAX>
__global__ void __launch_bounds__(kDecLayerThreads, 1) decode_layer_kernel(const DecodeParams p) {
  using F = Fmt<WF>;
  extern __shared__ float hs[];   // (k+1) rows of h_ld floats
  __shared__ int idx_s[32];
  __shared__ float w_s[33];
  const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kDecLayerThreads / 32;
  const int gw = blockIdx.x * nwarps + warp;
  const int nw = gridDim.x * nwarps;
  float *gu = p.h;                                            // [k][2 I]
  float *h_sh = p.h + static_cast<size_t>(p.k) * 2 * p.h_ld;  // [Is]
  unsigned int *bar_count = p.counter;
  unsigned int *bar_gen = p.counter + 1;

  DEC_MARK(0);
  // ---- phase 1: router rows, shared gate, shared-expert row pairs
  const int n1 = p.E + 1 + p.Is;
  for (int it = gw; it < n1; it += nw) {
    if (it < p.E) {
      const void *rows[1] = {row_ptr<0>(p.router_w, it, p.H)};
      const __nv_bfloat16 *sr[1] = {nullptr};
      float d[1];
      warp_dots_x<0, 1>(rows, sr, p.H, x, d);
      if (lane == 0) p.logits[it] = d[0] + (p.router_b ? p.router_b[it] : 0.0f);
    } else if (it == p.E) {
      const void *rows[1] = {p.sh_gate_w};
      const __nv_bfloat16 *sr[1] = {nullptr};
      float d[1];
      warp_dots_x<0, 1>(rows, sr, p.H, x, d);
      if (lane == 0) *p.g = sigmoid_f(d[0]);
    } else {
      const int i = it - p.E - 1;
      const void *rows[2] = {row_ptr<WF>(p.sh_gate_up, i, p.H),
                             row_ptr<WF>(p.sh_gate_up, p.Is + i, p.H)};
      const __nv_bfloat16 *sr[2] = {scale_row(p.sh_gate_up_scale, i, p.H),
                                    scale_row(p.sh_gate_up_scale, p.Is + i, p.H)};
      float d[2];
      warp_dots_x<WF, 2>(rows, sr, p.H, x, d);
      if (lane == 0) h_sh[i] = silu_f(d[0]) * d[1];
    }
  }
  DEC_MARK(1);
  grid_barrier(bar_count, bar_gen, p.status);
  DEC_MARK(2);

  // ---- top-k in every CTA (logits are in L2)
  if (warp == 0) {
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = lane + 32 * r;
      v[r] = (e < p.E) ? __ldcg(p.logits + e) : -INFINITY;
    }
    float sv, sw;
    int se;
    warp_topk<R>(v, p.E, p.k, sv, se, sw);
    if (lane < p.k) {
      idx_s[lane] = min(max(se, 0), p.E - 1);
      w_s[lane] = sw;
      if (blockIdx.x == 0) {
        p.idx[lane] = se;
        p.w[lane] = sw;
      }
    }
    if (lane == 0) w_s[32] = __ldcg(p.g);
  }
  __syncthreads();
  DEC_MARK(3);

  // ---- phase 2: routed gate/up rows, two per warp iteration
  const int I2 = 2 * p.I;
  const int n2 = p.k * I2;
  for (int base = gw; base < n2; base += 2 * nw) {
    const int r0 = base;
    const int r1 = (base + nw < n2) ? base + nw : base;
    const int j0 = r0 / I2, rr0 = r0 - j0 * I2;
    const int j1 = r1 / I2, rr1 = r1 - j1 * I2;
    const size_t w0 = static_cast<size_t>(idx_s[j0]) * I2 + rr0;
    const size_t w1 = static_cast<size_t>(idx_s[j1]) * I2 + rr1;
    const void *rows[2] = {row_ptr<WF>(p.gate_up, w0, p.H), row_ptr<WF>(p.gate_up, w1, p.H)};
    const __nv_bfloat16 *sr[2] = {scale_row(p.gate_up_scale, w0, p.H),
                                  scale_row(p.gate_up_scale, w1, p.H)};
    float d[2];
    warp_dots_x<WF, 2>(rows, sr, p.H, x, d);
    if (lane == 0) {
      gu[static_cast<size_t>(j0) * I2 + rr0] = d[0];
      if (r1 != r0) gu[static_cast<size_t>(j1) * I2 + rr1] = d[1];
    }
  }

  // ---- phase 3 weight loads for this warp's first output, ahead of the barrier
  const int n_first = gw;
  uint4 wv[KMAX + 1][2];
  const uint4 *rowp[KMAX + 1];
  const __nv_bfloat16 *srow[KMAX + 1];
  int nchunk[KMAX + 1];
  auto load_rows = [&](int n) {
#pragma unroll
    for (int j = 0; j <= KMAX; ++j) {
      wv[j][0] = wv[j][1] = make_uint4(0, 0, 0, 0);
      rowp[j] = nullptr;
      srow[j] = nullptr;
      nchunk[j] = 0;
      if (j > p.k) continue;
      const bool shared = (j == p.k);
      const int K = shared ? p.Is : p.I;
      const size_t r = shared ? static_cast<size_t>(n) : static_cast<size_t>(idx_s[j]) * p.H + n;
      nchunk[j] = K / F::EPC;
      rowp[j] = reinterpret_cast<const uint4 *>(row_ptr<WF>(shared ? p.sh_down : p.down, r, K));
      srow[j] = scale_row(shared ? p.sh_down_scale : p.down_scale, r, K);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        if (c < nchunk[j]) wv[j][u] = ld_stream(rowp[j] + c);
      }
    }
  };
  DEC_MARK(4);
  if (n_first < p.H) load_rows(n_first);
  grid_barrier(bar_count, bar_gen, p.status);
  DEC_MARK(5);

  // ---- stage h: routed SwiGLU from the gate/up dots, then the shared row
  const int nh = p.k * p.I;
  for (int e = threadIdx.x; e < nh; e += blockDim.x) {
    const int j = e / p.I, i = e - j * p.I;
    const float g = __ldcg(gu + static_cast<size_t>(j) * I2 + i);
    const float u = __ldcg(gu + static_cast<size_t>(j) * I2 + p.I + i);
    hs[static_cast<size_t>(j) * p.h_ld + i] = silu_f(g) * u;
  }
  for (int i = threadIdx.x; i < p.Is; i += blockDim.x)
    hs[static_cast<size_t>(p.k) * p.h_ld + i] = __ldcg(h_sh + i);
  __syncthreads();
  DEC_MARK(6);

  // ---- phase 3: outputs
  for (int n = n_first; n < p.H; n += nw) {
    if (n != n_first) load_rows(n);
    float y = 0.0f;
#pragma unroll
    for (int j = 0; j <= KMAX; ++j) {
      if (j > p.k) continue;
      const float *hj = hs + static_cast<size_t>(j) * p.h_ld;
      float d = 0.0f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        if (c < nchunk[j]) {
          if constexpr (WF == 0) d += dot8_bf16_f32(wv[j][u], hj + c * 8);
          else d = fmaf(__bfloat162float(srow[j][c >> 1]), dot32_int4_f32(wv[j][u], hj + c * 32), d);
        }
      }
      // chunks beyond the first 64 per row (I > 512 for bf16, > 2048 for int4)
      for (int c = lane + 64; c < nchunk[j]; c += 32) {
        const uint4 wc = ld_stream(rowp[j] + c);
        if constexpr (WF == 0) d += dot8_bf16_f32(wc, hj + c * 8);
        else d = fmaf(__bfloat162float(srow[j][c >> 1]), dot32_int4_f32(wc, hj + c * 32), d);
      }
      d = warp_sum(d);
      y = fmaf(j == p.k ? w_s[32] : w_s[j], d, y);
    }
    if (lane == 0) reinterpret_cast<__nv_bfloat16 *>(p.y)[n] = __float2bfloat16_rn(y);
  }
  __syncthreads();
  DEC_MARK(7);
}

template <int WF, int R, int KMAX>
static cudaError_t launch_layer(const DecodeParams &p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kDecLayerThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.k + 1) * p.h_ld * sizeof(float);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<WF, R, KMAX>, p);
}

template <int WF>
static cudaError_t launch_layer_wf(const DecodeParams &p, int grid, cudaStream_t stream) {
  if (p.E <= 256) {
    if (p.k <= 2) return launch_layer<WF, 8, 2>(p, grid, stream);
    if (p.k <= 8) return launch_layer<WF, 8, 8>(p, grid, stream);
    return launch_layer<WF, 8, 32>(p, grid, stream);
  }
  if (p.k <= 8) return launch_layer<WF, 32, 8>(p, grid, stream);
  return launch_layer<WF, 32, 32>(p, grid, stream);
}

cudaError_t launch_decode_layer(const DecodeParams &p, int grid, cudaStream_t stream) {
  return p.wfmt == 0 ? launch_layer_wf<0>(p, grid, stream) : launch_layer_wf<1>(p, grid, stream);
}

template <int WF, int R, int KMAX>
static cudaError_t configure_one(int bytes) {
  return cudaFuncSetAttribute(decode_layer_kernel<WF, R, KMAX>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t decode_configure(int max_smem_floats) {
  // Allow more than 48 KB of dynamic shared memory for large (k+1)*Imax.
  const int bytes = max_smem_floats * static_cast<int>(sizeof(float));
  cudaError_t e;
  if ((e = configure_one<0, 8, 2>(bytes)) || (e = configure_one<0, 8, 8>(bytes)) ||
      (e = configure_one<0, 8, 32>(bytes)) || (e = configure_one<0, 32, 8>(bytes)) ||
      (e = configure_one<0, 32, 32>(bytes)) || (e = configure_one<1, 8, 2>(bytes)) ||
      (e = configure_one<1, 8, 8>(bytes)) || (e = configure_one<1, 8, 32>(bytes)) ||
      (e = configure_one<1, 32, 8>(bytes)) || (e = configure_one<1, 32, 32>(bytes)))
    return e;
  return cudaSuccess;
}

int decode_layer_grid(int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel<0, 8, 8>,
                                                    kDecLayerThreads, 20 * 1024) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  cudaGetLastError();
  return num_sms;   // one CTA per SM: every CTA must be co-resident
}

}  // namespace moe

#ifdef MOE_TRACE
extern "C" int moe_debug_read_decode_trace(void *dst, size_t bytes) {
  size_t n = bytes < sizeof(moe::g_dec_trace) ? bytes : sizeof(moe::g_dec_trace);
  return cudaMemcpyFromSymbol(dst, moe::g_dec_trace, n) == cudaSuccess ? 0 : 1;
}
#endif
