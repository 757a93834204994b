// Device-resident routing for the prefill path (section "Keep expert routing
// on the GPU" of "Optimizing On-Device Inference for Apple Silicon"): top-k
// selection, a histogram of assignments per expert, an exclusive prefix scan
// into segment offsets, a stable scatter of rows into their expert segments,
// and the block map the grouped GEMMs walk.  No host synchronisation; every
// result is independent of thread timing (integer counts and bit masks only).
//
// Tokens are processed in routing blocks of 32.  For each block and expert a
// 32-bit mask records which of the block's tokens chose the expert; the rank
// of a token inside its expert segment is then
//     offsets[e] + (rows of e in earlier blocks) + popc(mask & lower bits),
// i.e. segments are ordered by ascending token index.
#include "moe_internal.h"

#include <algorithm>
#include "warp_topk.cuh"

namespace moe {

// ----------------------------------------------------------------- top-k --
// One routing block of 32 tokens per CTA, one token per warp: the token's
// logits (the sum of the router GEMM's split-K parts, in part order), its
// top-k and weights, and its bit in the block's per-expert masks.
constexpr int kTopkThreads = 32 * kRouteBlockTokens;

template <int R, int SP>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float *__restrict__ partial, int nsplit, size_t split_stride, float *__restrict__ logits_out,
    int T, int E, int k, int32_t *__restrict__ idx, float *__restrict__ w,
    uint32_t *__restrict__ blk_mask) {
  __shared__ uint32_t mask_s[1024];
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask_s[e] = 0;
  __syncthreads();
  pdl_wait();
  const int tl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteBlockTokens + tl;
  if (t < T) {
    float v[R];
    const float *row = partial + static_cast<size_t>(t) * E;
    if constexpr (SP > 0) {
      // up to SP parts' loads in flight together, then the sums in part order
      float pv[SP][R];
#pragma unroll
      for (int sp = 0; sp < SP; ++sp)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int e = lane + 32 * r;
          pv[sp][r] = (e < E && sp < nsplit) ? __ldcs(row + sp * split_stride + e) : 0.0f;
        }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        v[r] = pv[0][r];
#pragma unroll
        for (int sp = 1; sp < SP; ++sp)
          if (sp < nsplit) v[r] += pv[sp][r];
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = lane + 32 * r;
        v[r] = (e < E) ? __ldcs(row + e) : 0.0f;
      }
      for (int sp = 1; sp < nsplit; ++sp) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int e = lane + 32 * r;
          if (e < E) v[r] += __ldcs(row + sp * split_stride + e);
        }
      }
    }
    if (logits_out != nullptr) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = lane + 32 * r;
        if (e < E) logits_out[static_cast<size_t>(t) * E + e] = v[r];
      }
    }
    int se;
    float sw;
    warp_topk_redux<R>(v, E, k, se, sw);
    if (lane < k) {
      idx[static_cast<size_t>(t) * k + lane] = se;
      w[static_cast<size_t>(t) * k + lane] = sw;
      atomicOr(&mask_s[se], 1u << tl);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blk_mask[static_cast<size_t>(blockIdx.x) * E + e] = mask_s[e];
}

cudaError_t launch_topk(const float *partial, int nsplit, size_t split_stride, float *logits_out,
                        int T, int E, int k, int32_t *idx, float *w, uint32_t *blk_mask, bool pdl,
                        cudaStream_t stream) {
  const int nblk = (T + kRouteBlockTokens - 1) / kRouteBlockTokens;
  const int R = (E + 31) / 32;
  // SP: parts loaded together (up to 4 parts for E <= 256), 0: part by part
  cudaError_t e = cudaSuccess;
#define MOE_TOPK(RR, SS)                                                                        \
  e = launch_kernel(topk_kernel<RR, SS>, dim3(nblk), dim3(kTopkThreads), 0, stream, pdl, partial, \
                    nsplit, split_stride, logits_out, T, E, k, idx, w, blk_mask)
#define MOE_TOPK_R(RR)                        \
  if (nsplit == 1) MOE_TOPK(RR, 1);           \
  else if (nsplit <= 4) MOE_TOPK(RR, 4);      \
  else MOE_TOPK(RR, 0)
  if (R <= 1) { MOE_TOPK_R(1); }
  else if (R <= 2) { MOE_TOPK_R(2); }
  else if (R <= 4) { MOE_TOPK_R(4); }
  else if (R <= 8) { MOE_TOPK_R(8); }
  else if (R <= 16) { MOE_TOPK(16, 0); }
  else { MOE_TOPK(32, 0); }
#undef MOE_TOPK_R
#undef MOE_TOPK
  return e;
}

// ------------------------------------------------------------- placement --
// One routing block of 32 tokens per CTA (1024 threads), after the top-k
// kernel has written every block's per-expert masks:
//  1. every CTA counts, for each expert e, its rows in all blocks (total[e])
//     and in the blocks before its own (before[e]): 128 KB of masks at
//     T = 4096, read by each CTA from L2 (parts of the block range per
//     thread, summed in a fixed order);
//  2. the exclusive scan of the totals gives the segment offsets (identical
//     in every CTA: integer sums);
//  3. one thread per assignment (t, j) of the block: pos(t, j) = offsets[e] +
//     before[e] + (lower tokens of this block that chose e), sorted_rows[pos]
//     = t;
//  4. the block map the grouped GEMMs walk: ceil(total[e] / block_rows)
//     blocks per expert in expert order, then the shared expert's T rows at
//     grouped row T * k; each CTA writes the blocks of the experts e with
//     e % gridDim.x == blockIdx.x, CTA 0 the counts, offsets, shared blocks and
//     block count;
//  5. one warp per token reads the token's x row once, into registers: with
//     gate, the shared-expert gate g[t] = sigmoid(x[t] . w_sg) for the
//     combine; with xg, the row is written to the token's k positions of xg,
//     so that the grouped gate/up GEMM reads its token rows as consecutive
//     rows.
// Every result is an integer function of the masks and indices: independent
// of thread timing and of which CTA computes it.
constexpr int kPlaceThreads = 1024;
constexpr int kScatterChunks = 8;   // 16-byte chunks of a row per lane and pass

// Exclusive scan of one int per thread over a 1024-thread block.
__device__ __forceinline__ int block_excl_scan_1024(int v, int *warp_tot, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wv = warp_tot[lane];
    int wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += n;
    }
    warp_tot[lane] = wi - wv;   // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const int excl = incl - v + warp_tot[warp];
  total = warp_tot[32];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kPlaceThreads) place_kernel(
    const int32_t *__restrict__ idx, const uint32_t *__restrict__ blk_mask, int nblk, int T, int E,
    int k, int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int4 *__restrict__ blocks,
    int32_t *__restrict__ n_blocks, int block_rows, int32_t *__restrict__ sorted_rows,
    int32_t *__restrict__ pos_of_assign, const uint4 *__restrict__ x, uint4 *__restrict__ xg,
    const uint4 *__restrict__ wsg, float *__restrict__ gate, int H) {
  __shared__ int tot_s[kPlaceThreads];    // per (part, expert), then per expert
  __shared__ int bef_s[kPlaceThreads];
  __shared__ int off_s[kPlaceThreads];
  __shared__ int warp_tot[33];
  __shared__ int pos_s[kRouteBlockTokens * 32];   // [token][slot], k <= 32
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  // 1. counts: P parts of the block range per expert (Ep = E rounded up to a
  //    power of two, P = 1024 / Ep)
  int Ep = 1;
  while (Ep < E) Ep <<= 1;
  const int P = kPlaceThreads / Ep;
  {
    const int e = tid & (Ep - 1), part = tid / Ep;
    const int b0 = static_cast<int>((static_cast<long long>(nblk) * part) / P);
    const int b1 = static_cast<int>((static_cast<long long>(nblk) * (part + 1)) / P);
    int tot = 0, bef = 0;
    if (e < E) {
      const uint32_t *col = blk_mask + e;
      int bb = b0;
      for (; bb + 8 <= b1; bb += 8) {
        uint32_t m[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = __ldcg(col + static_cast<size_t>(bb + i) * E);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = __popc(m[i]);
          tot += c;
          bef += (bb + i < b) ? c : 0;
        }
      }
      for (; bb < b1; ++bb) {
        const int c = __popc(__ldcg(col + static_cast<size_t>(bb) * E));
        tot += c;
        bef += (bb < b) ? c : 0;
      }
    }
    tot_s[tid] = tot;
    bef_s[tid] = bef;
  }
  __syncthreads();
  int total_e = 0, before_e = 0;
  if (tid < E) {
    for (int part = 0; part < P; ++part) {
      total_e += tot_s[part * Ep + tid];
      before_e += bef_s[part * Ep + tid];
    }
  }
  // 2. segment offsets
  int all = 0;
  const int off = block_excl_scan_1024(total_e, warp_tot, all);   // all = T * k
  if (tid < E) {
    off_s[tid] = off;
    bef_s[tid] = before_e;   // (read only after the barrier below)
  }
  // 4a. block counts and starts (every CTA computes them; the scan's
  //     barriers order the writes above)
  const int nb = (tid < E) ? (total_e + block_rows - 1) / block_rows : 0;
  int nb_total = 0;
  const int bstart = block_excl_scan_1024(nb, warp_tot, nb_total);
  // 3. positions of this block's assignments
  const int tl = tid / k;
  const int j = tid - tl * k;
  const int t = b * kRouteBlockTokens + tl;
  if (tl < kRouteBlockTokens && t < T) {
    const int a = t * k + j;
    const int e = idx[a];
    const uint32_t m = __ldcg(blk_mask + static_cast<size_t>(b) * E + e);
    const int rank = __popc(m & ((1u << tl) - 1u));
    const int p = off_s[e] + bef_s[e] + rank;
    pos_of_assign[a] = p;
    sorted_rows[p] = t;
    pos_s[tl * k + j] = p;
  }
  // 4b. this CTA's share of the block map
  if (tid < E && (tid % gridDim.x) == b) {
    for (int i = 0; i < nb; ++i) {
      const int r0 = i * block_rows;
      blocks[bstart + i] = make_int4(tid, off + r0, min(block_rows, total_e - r0), 0);
    }
  }
  if (b == 0) {
    if (tid < E) {
      counts[tid] = total_e;
      offsets[tid] = off;
    }
    if (tid == 0) offsets[E] = all;
    const int nb_sh = (T + block_rows - 1) / block_rows;
    for (int i = tid; i < nb_sh; i += blockDim.x) {
      const int r0 = i * block_rows;
      blocks[nb_total + i] = make_int4(E, T * k + r0, min(block_rows, T - r0), 0);
    }
    if (tid == 0) *n_blocks = nb_total + nb_sh;
  }
  if (xg == nullptr && gate == nullptr) return;
  __syncthreads();
  // 5. the shared gate and the token rows in grouped order
  const int warp = tid >> 5, lane = tid & 31;
  const int nwarps = blockDim.x >> 5;
  const int nch = H / 8;   // 16-byte chunks per row
  for (int u = warp; u < kRouteBlockTokens; u += nwarps) {
    const int tt = b * kRouteBlockTokens + u;
    if (tt >= T) break;
    const uint4 *src = x + static_cast<size_t>(tt) * nch;
    float d = 0.0f;   // this lane's part of x[tt] . w_sg (chunks lane + 32 i, in order)
    for (int c0 = 0; c0 < nch; c0 += 32 * kScatterChunks) {
      uint4 v[kScatterChunks];
#pragma unroll
      for (int i = 0; i < kScatterChunks; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < nch) v[i] = __ldg(src + c);
      }
      if (gate != nullptr) {
#pragma unroll
        for (int i = 0; i < kScatterChunks; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < nch) {
            const uint4 gv = __ldg(wsg + c);
            const uint32_t xa[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            const uint32_t ga[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              d = fmaf(bf16_lo(xa[q]), bf16_lo(ga[q]), d);
              d = fmaf(bf16_hi(xa[q]), bf16_hi(ga[q]), d);
            }
          }
        }
      }
      if (xg == nullptr) continue;
      for (int jj = 0; jj < k; ++jj) {
        uint4 *dst = xg + static_cast<size_t>(pos_s[u * k + jj]) * nch;
#pragma unroll
        for (int i = 0; i < kScatterChunks; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < nch) dst[c] = v[i];
        }
      }
    }
    if (gate != nullptr) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0) gate[tt] = sigmoid_f(d);
    }
  }
}

cudaError_t launch_place(const int32_t *idx, const uint32_t *blk_mask, int T, int E, int k,
                         int32_t *counts, int32_t *offsets, int4 *blocks, int32_t *n_blocks,
                         int block_rows, int32_t *sorted_rows, int32_t *pos_of_assign,
                         const void *x, void *xg, const void *wsg, float *gate, int H, bool pdl,
                         cudaStream_t stream) {
  const int nblk = (T + kRouteBlockTokens - 1) / kRouteBlockTokens;
  return launch_kernel(place_kernel, dim3(nblk), dim3(kPlaceThreads), 0, stream, pdl, idx,
                       blk_mask, nblk, T, E, k, counts, offsets, blocks, n_blocks, block_rows,
                       sorted_rows, pos_of_assign, static_cast<const uint4 *>(x),
                       static_cast<uint4 *>(xg), static_cast<const uint4 *>(wsg), gate, H);
}

// --------------------------------------------------------------- combine --
// y[t] = sum_j w[t,j] * o[pos(t,j)] + g[t] * o[T*k + t], fp32 accumulation in
// fixed slot order (o holds the per-expert outputs in fp16; g[t] comes from
// the top-k kernel) (section "Reduce intermediate and state traffic": the
// output projection combined with its routing score and the shared-expert
// result).  No atomics: each output element is written once.  For k <= KF
// all of a chunk's loads are issued before its arithmetic.
template <int KF>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ gate,
                                                      const __half *__restrict__ o,
                                                      const int32_t *__restrict__ pos,
                                                      const float *__restrict__ w, int T, int H,
                                                      int k, __nv_bfloat16 *__restrict__ y) {
  // rows and weights of the CTA's current token (buffer it & 1) and of its
  // next one (k <= 32)
  __shared__ int pos_s[2][32];
  __shared__ float w_s[2][32];
  pdl_trigger();
  pdl_wait();
  const int nchunk = H / 8;
  const int tid = threadIdx.x;
  int t = blockIdx.x;
  if (t < T && tid < k) {
    pos_s[0][tid] = pos[static_cast<size_t>(t) * k + tid];
    w_s[0][tid] = w[static_cast<size_t>(t) * k + tid];
  }
  __syncthreads();
  // tokens t = blockIdx.x, + gridDim.x, ...: one resident wave of CTAs; the
  // next token's rows are read while this token's outputs stream
  for (int it = 0; t < T; t += gridDim.x, ++it) {
    const int buf = it & 1;
    const int tn = t + gridDim.x;
    const bool pre = tn < T && tid < k;
    int pos_n = 0;
    float w_n = 0.0f;
    if (pre) {
      pos_n = __ldg(pos + static_cast<size_t>(tn) * k + tid);
      w_n = __ldg(w + static_cast<size_t>(tn) * k + tid);
    }
    const float g = __ldg(gate + t);
    const size_t shared_row = static_cast<size_t>(T) * k + t;
    for (int c = tid; c < nchunk; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      uint4 ov[KF > 0 ? KF : 1];
      if constexpr (KF > 0) {
#pragma unroll
        for (int j = 0; j < KF; ++j)
          ov[j] = j < k ? __ldcs(reinterpret_cast<const uint4 *>(o + static_cast<size_t>(pos_s[buf][j]) * H + c * 8))
                        : make_uint4(0, 0, 0, 0);
      }
      const uint4 sv = __ldcs(reinterpret_cast<const uint4 *>(o + shared_row * H + c * 8));
      auto add = [&](const uint4 oj, float wj) {
        const uint32_t oa[4] = {oj.x, oj.y, oj.z, oj.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = half2_to_float2(oa[i]);
          acc[2 * i] = fmaf(wj, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(wj, f.y, acc[2 * i + 1]);
        }
      };
      if constexpr (KF > 0) {
#pragma unroll
        for (int j = 0; j < KF; ++j)
          if (j < k) add(ov[j], w_s[buf][j]);
      } else {
        for (int j = 0; j < k; ++j)
          add(*reinterpret_cast<const uint4 *>(o + static_cast<size_t>(pos_s[buf][j]) * H + c * 8),
              w_s[buf][j]);
      }
      const uint32_t sa[4] = {sv.x, sv.y, sv.z, sv.w};
      uint4 out;
      uint32_t *oo = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = half2_to_float2(sa[i]);
        const float lo = fmaf(g, f.x, acc[2 * i]);
        const float hi = fmaf(g, f.y, acc[2 * i + 1]);
        oo[i] = pack_bf16x2(lo, hi);
      }
      *reinterpret_cast<uint4 *>(y + static_cast<size_t>(t) * H + c * 8) = out;
    }
    // buffer buf ^ 1 was last read before the previous iteration's barrier
    if (pre) {
      pos_s[buf ^ 1][tid] = pos_n;
      w_s[buf ^ 1][tid] = w_n;
    }
    __syncthreads();
  }
}

cudaError_t launch_combine(const float *gate, const void *o, const int32_t *pos, const float *w,
                           int T, int H, int k, void *y, bool pdl, cudaStream_t stream) {
  const __half *oh = reinterpret_cast<const __half *>(o);
  __nv_bfloat16 *yb = reinterpret_cast<__nv_bfloat16 *>(y);
  // one resident wave: SMs x CTAs of the kernel per SM (the latter depends
  // only on the kernel and the architecture; computed once, thread-safely)
  static const int per_sm8 = [] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel<8>, 256, 0) == cudaSuccess ? n : 1;
  }();
  static const int per_sm0 = [] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel<0>, 256, 0) == cudaSuccess ? n : 1;
  }();
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int wave = std::max(1, sms * std::max(1, k <= 8 ? per_sm8 : per_sm0));
  const int grid = std::max(1, std::min(T, wave));
  if (k <= 8)
    return launch_kernel(combine_kernel<8>, dim3(grid), dim3(256), 0, stream, pdl, gate, oh, pos, w,
                         T, H, k, yb);
  return launch_kernel(combine_kernel<0>, dim3(grid), dim3(256), 0, stream, pdl, gate, oh, pos, w, T,
                       H, k, yb);
}

// bf16 -> fp16 copy of a weight array, 8 elements (16 bytes) per thread and
// step; the last n % 8 elements one by one.  Each pair is widened to fp32
// exactly and narrowed with cvt.rn.f16x2.f32, the conversion the down GEMM
// applies to weight tiles in shared memory when no copy is supplied.
__global__ void __launch_bounds__(256) convert_bf16_to_f16_kernel(const uint4 *__restrict__ src,
                                                                  uint4 *__restrict__ dst,
                                                                  size_t nvec, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const uint4 v = __ldg(src + i);
    const uint32_t wi[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm("cvt.rn.f16x2.f32 %0, %1, %2;"
          : "=r"(o[j])
          : "f"(__uint_as_float(wi[j] & 0xffff0000u)), "f"(__uint_as_float(wi[j] << 16)));
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (blockIdx.x == 0 && threadIdx.x < n - nvec * 8) {
    const size_t e = nvec * 8 + threadIdx.x;
    const uint16_t b = reinterpret_cast<const uint16_t *>(src)[e];
    reinterpret_cast<__half *>(dst)[e] = __float2half_rn(__uint_as_float(static_cast<uint32_t>(b) << 16));
  }
}

cudaError_t launch_convert_bf16_to_f16(const void *src, void *dst, size_t n, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
    return e;
  const size_t nvec = n / 8;
  const size_t want = (nvec + 255) / 256;
  const int grid = static_cast<int>(std::max<size_t>(1, std::min<size_t>(want, static_cast<size_t>(sms) * 8)));
  convert_bf16_to_f16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(src),
                                                       static_cast<uint4 *>(dst), nvec, n);
  return cudaGetLastError();
}

}  // namespace moe
