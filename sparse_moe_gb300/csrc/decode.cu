// Batch-1 decode path (sections "Optimize the one-row weight path" and
// "Reduce intermediate and state traffic" of "Optimizing On-Device Inference
// for Apple Silicon"): with one activation row there is no weight reuse, so
// every kernel is a row-parallel GEMV on the vector ALUs that streams each
// weight row once with coalesced 128-bit loads.  Three launches per layer:
//
//   1. router logits (+bias), the shared-expert gate sigmoid(x . w_sg) and the
//      shared expert's gate/up projections with SwiGLU; the last CTA to finish
//      selects the top-k and writes the renormalised weights.  The router and
//      the shared expert only need x, so they share one launch and overlap.
//   2. the k routed experts' gate/up projections fused with SwiGLU
//      (h[j, i] = silu(Wg x) * (Wu x)), one warp per (expert, row pair);
//   3. the output projections of the k experts and of the shared expert,
//      fused with the routing weights and the shared gate:
//      y[n] = sum_j w_j (Wd_j h_j)[n] + g (Sd h_s)[n], in fixed j order.
//
// int4 weights are read packed (32 codes per 128-bit load) and expanded in
// registers; each 16-byte chunk lies inside one 64-wide scale group.
#include "moe_internal.h"
#include "warp_topk.cuh"

namespace moe {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// 8 bf16 weights . 8 fp32 activations
__device__ __forceinline__ float dot8_bf16(const uint4 wv, const float *xs) {
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

// 32 int4 codes (one 16-byte chunk; element n of word w is nibble n) . 32
// fp32 activations.  Returns sum q * x without the group scale.
__device__ __forceinline__ float dot32_int4(const uint4 wv, const float *xs) {
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
  float a = 0.0f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 x0 = *reinterpret_cast<const float4 *>(xs + 8 * w);
    const float4 x1 = *reinterpret_cast<const float4 *>(xs + 8 * w + 4);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int q = static_cast<int>(words[w] << (28 - 4 * n)) >> 28;   // sign-extended nibble
      a = fmaf(static_cast<float>(q), xv[n], a);
    }
  }
  return a;
}

// Dot products of NR weight rows (same K, same activation xs in shared
// memory) computed by one warp.  Rows are given by pointers; for int4 the
// matching scale rows are given too.  All loads of a round are issued before
// any arithmetic so each lane keeps NR * 4 128-bit loads in flight.
template <int WF, int NR>
__device__ __forceinline__ void warp_dots(const void *const (&rows)[NR],
                                          const __nv_bfloat16 *const (&srows)[NR], int K,
                                          const float *xs, float (&out)[NR]) {
  const int lane = threadIdx.x & 31;
  constexpr int EPC = (WF == 0) ? 8 : 32;        // elements per 16-byte chunk
  constexpr int U = 4;                            // chunks per lane per round
  const int nchunk = K / EPC;
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
  for (int c0 = 0; c0 < nchunk; c0 += 32 * U) {
    uint4 wv[NR][U];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + lane + 32 * u;
        wv[r][u] = (c < nchunk) ? ld_stream(reinterpret_cast<const uint4 *>(rows[r]) + c)
                                : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + lane + 32 * u;
        if (c < nchunk) {
          if (WF == 0) {
            acc[r] += dot8_bf16(wv[r][u], xs + c * 8);
          } else {
            const float s = __bfloat162float(srows[r][c >> 1]);
            acc[r] = fmaf(s, dot32_int4(wv[r][u], xs + c * 32), acc[r]);
          }
        }
      }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

__device__ __forceinline__ void stage_x(const __nv_bfloat16 *x, float *xs, int H) {
  for (int i = threadIdx.x; i < H; i += blockDim.x) xs[i] = __bfloat162float(x[i]);
  __syncthreads();
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

// ------------------------------------------- 1: router + shared expert --
template <int WF, int R>
__global__ void __launch_bounds__(kDecThreads) decode_router_shared_kernel(const DecodeParams p) {
  extern __shared__ float xs[];
  __shared__ int last_s;
  const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x);
  stage_x(x, xs, p.H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nitems = p.E + 1 + p.Is;
  for (int it = blockIdx.x * kDecWarps + warp; it < nitems; it += gridDim.x * kDecWarps) {
    if (it < p.E) {
      const void *rows[1] = {row_ptr<0>(p.router_w, it, p.H)};
      const __nv_bfloat16 *sr[1] = {nullptr};
      float d[1];
      warp_dots<0, 1>(rows, sr, p.H, xs, d);
      if (lane == 0) p.logits[it] = d[0] + (p.router_b ? p.router_b[it] : 0.0f);
    } else if (it == p.E) {
      const void *rows[1] = {p.sh_gate_w};
      const __nv_bfloat16 *sr[1] = {nullptr};
      float d[1];
      warp_dots<0, 1>(rows, sr, p.H, xs, d);
      if (lane == 0) *p.g = sigmoid_f(d[0]);
    } else {
      const int i = it - p.E - 1;
      const void *rows[2] = {row_ptr<WF>(p.sh_gate_up, i, p.H),
                             row_ptr<WF>(p.sh_gate_up, p.Is + i, p.H)};
      const __nv_bfloat16 *sr[2] = {scale_row(p.sh_gate_up_scale, i, p.H),
                                    scale_row(p.sh_gate_up_scale, p.Is + i, p.H)};
      float d[2];
      warp_dots<WF, 2>(rows, sr, p.H, xs, d);
      if (lane == 0) p.h[static_cast<size_t>(p.k) * p.h_ld + i] = silu_f(d[0]) * d[1];
    }
  }
  // The last CTA to finish selects the top-k over all logits.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = (atomicAdd(p.counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
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
      p.idx[lane] = se;
      p.w[lane] = sw;
    }
    if (lane == 0) *p.counter = 0u;
  }
}

// ---------------------------------------------- 2: routed gate/up+SwiGLU --
template <int WF>
__global__ void __launch_bounds__(kDecThreads) decode_gateup_kernel(const DecodeParams p) {
  extern __shared__ float xs[];
  stage_x(reinterpret_cast<const __nv_bfloat16 *>(p.x), xs, p.H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nitems = p.k * p.I;
  for (int it = blockIdx.x * kDecWarps + warp; it < nitems; it += gridDim.x * kDecWarps) {
    const int j = it / p.I;
    const int i = it - j * p.I;
    const int e = min(max(__ldcg(p.idx + j), 0), p.E - 1);
    const size_t rg = static_cast<size_t>(e) * 2 * p.I + i;
    const void *rows[2] = {row_ptr<WF>(p.gate_up, rg, p.H), row_ptr<WF>(p.gate_up, rg + p.I, p.H)};
    const __nv_bfloat16 *sr[2] = {scale_row(p.gate_up_scale, rg, p.H),
                                  scale_row(p.gate_up_scale, rg + p.I, p.H)};
    float d[2];
    warp_dots<WF, 2>(rows, sr, p.H, xs, d);
    if (lane == 0) p.h[static_cast<size_t>(j) * p.h_ld + i] = silu_f(d[0]) * d[1];
  }
}

// --------------------------------- 3: down projections + weighted combine --
template <int WF>
__global__ void __launch_bounds__(kDecThreads) decode_down_kernel(const DecodeParams p) {
  extern __shared__ float hs[];   // (k+1) rows of h_ld floats
  __shared__ int e_s[33];
  __shared__ float w_s[33];
  const int nrows_h = p.k + 1;
  for (int i = threadIdx.x; i < nrows_h * p.h_ld; i += blockDim.x) hs[i] = __ldcg(p.h + i);
  if (threadIdx.x < p.k) {
    e_s[threadIdx.x] = min(max(__ldcg(p.idx + threadIdx.x), 0), p.E - 1);
    w_s[threadIdx.x] = __ldcg(p.w + threadIdx.x);
  }
  if (threadIdx.x == 0) w_s[32] = __ldcg(p.g);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int n = blockIdx.x * kDecWarps + warp; n < p.H; n += gridDim.x * kDecWarps) {
    float y = 0.0f;
    for (int j = 0; j < p.k; ++j) {
      const size_t r = static_cast<size_t>(e_s[j]) * p.H + n;
      const void *rows[1] = {row_ptr<WF>(p.down, r, p.I)};
      const __nv_bfloat16 *sr[1] = {scale_row(p.down_scale, r, p.I)};
      float d[1];
      warp_dots<WF, 1>(rows, sr, p.I, hs + static_cast<size_t>(j) * p.h_ld, d);
      y = fmaf(w_s[j], d[0], y);
    }
    {
      const void *rows[1] = {row_ptr<WF>(p.sh_down, n, p.Is)};
      const __nv_bfloat16 *sr[1] = {scale_row(p.sh_down_scale, n, p.Is)};
      float d[1];
      warp_dots<WF, 1>(rows, sr, p.Is, hs + static_cast<size_t>(p.k) * p.h_ld, d);
      y = fmaf(w_s[32], d[0], y);
    }
    if (lane == 0) reinterpret_cast<__nv_bfloat16 *>(p.y)[n] = __float2bfloat16_rn(y);
  }
}

cudaError_t launch_decode_router_shared(const DecodeParams &p, cudaStream_t stream) {
  const size_t xs_bytes = static_cast<size_t>(p.H) * sizeof(float);
  const int n1 = p.E + 1 + p.Is;
  const int g1 = (n1 + kDecWarps - 1) / kDecWarps;
  const bool small = p.E <= 256;
  if (p.wfmt == 0) {
    if (small) decode_router_shared_kernel<0, 8><<<g1, kDecThreads, xs_bytes, stream>>>(p);
    else decode_router_shared_kernel<0, 32><<<g1, kDecThreads, xs_bytes, stream>>>(p);
  } else {
    if (small) decode_router_shared_kernel<1, 8><<<g1, kDecThreads, xs_bytes, stream>>>(p);
    else decode_router_shared_kernel<1, 32><<<g1, kDecThreads, xs_bytes, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_gateup(const DecodeParams &p, cudaStream_t stream) {
  const size_t xs_bytes = static_cast<size_t>(p.H) * sizeof(float);
  const int g2 = (p.k * p.I + kDecWarps - 1) / kDecWarps;
  if (p.wfmt == 0) decode_gateup_kernel<0><<<g2, kDecThreads, xs_bytes, stream>>>(p);
  else decode_gateup_kernel<1><<<g2, kDecThreads, xs_bytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_down(const DecodeParams &p, cudaStream_t stream) {
  const size_t hs_bytes = static_cast<size_t>(p.k + 1) * p.h_ld * sizeof(float);
  const int g3 = (p.H + kDecWarps - 1) / kDecWarps;
  if (p.wfmt == 0) decode_down_kernel<0><<<g3, kDecThreads, hs_bytes, stream>>>(p);
  else decode_down_kernel<1><<<g3, kDecThreads, hs_bytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t decode_configure(int max_smem_floats) {
  // Allow more than 48 KB of dynamic shared memory for large (k+1)*Imax or H.
  const int bytes = max_smem_floats * static_cast<int>(sizeof(float));
  cudaError_t e = cudaSuccess;
  e = cudaFuncSetAttribute(decode_down_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_down_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (auto fn : {decode_gateup_kernel<0>, decode_gateup_kernel<1>}) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  for (auto fn : {decode_router_shared_kernel<0, 8>, decode_router_shared_kernel<0, 32>,
                  decode_router_shared_kernel<1, 8>, decode_router_shared_kernel<1, 32>}) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
