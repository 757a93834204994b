// Batch-1 decode path (sections "Optimize the one-row weight path" and
// "Reduce intermediate and state traffic" of "Optimizing On-Device Inference
// for Apple Silicon"): with one activation row there is no weight reuse, so
// the layer is a chain of row-parallel GEMVs on the vector ALUs that stream
// every weight row once.  One persistent cooperative launch per layer runs it
// as three phases separated by two grid barriers:
//
//   A. router logits (+bias), the shared-expert gate sigmoid(x . w_sg) and
//      the shared expert's gate and up dot products (all need only x);
//   B. top-k selection (redone by one warp of every CTA from the logits in
//      L2), then the k routed experts' gate and up dot products;
//   C. y[n] = sum_j w_j (Wd_j h_j)[n] + g (Sd h_s)[n] in fixed j order, with
//      h = silu(gate) * up formed from the phase-A/B dot products.
//
// The first barrier waits for the router rows alone: the shared expert's
// rows, whose h only C needs, run beside it on the other warps and are
// announced on a second counter.
//
// Phase C's weights are known early: the shared expert's output rows at the
// start, the routed experts' right after top-k.  Each CTA owns a contiguous
// range of output rows n and bulk-copies (cp.async.bulk, completing on an
// mbarrier) exactly those rows of the k + 1 output projections into its
// shared memory while the gate/up rows stream through registers.  The HBM
// traffic of phases B and C therefore overlaps, and after the last barrier
// only the h exchange (through L2) and shared-memory arithmetic remain.
//
// Gate/up rows are read with 128-bit loads, every load of a segment issued
// before any arithmetic.  int4 weights are read packed (32 codes per 128-bit
// load) and expanded in registers; each 16-byte chunk lies inside one 64-wide
// scale group.
#include "moe_common.cuh"
#include "moe_internal.h"
#include "warp_topk.cuh"

namespace moe {

constexpr int kDecLayerThreads = 512;
constexpr int kDecWarps = kDecLayerThreads / 32;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// `bytes` (a multiple of 16) from global `src` to this CTA's shared memory at
// `dst` (both 16-byte aligned); completes on the mbarrier at `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_l2_line(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Start of the 128-byte line holding p.
__device__ __forceinline__ const char *line_of(const char *p) {
  return reinterpret_cast<const char *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127));
}

// This warp's L2 prefetch of `bytes` of one weight row.
__device__ __forceinline__ void prefetch_row_l2(const void *row, size_t bytes) {
  const char *b = static_cast<const char *>(row);
  for (size_t off = (threadIdx.x & 31) * 128; off < bytes; off += 32 * 128) prefetch_l2_line(b + off);
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

// 8 bf16 weights . 8 fp32 activations held in registers
__device__ __forceinline__ float dot8_bf16_f32(const uint4 wv, const float (&xs)[8]) {
  float a = bf16_lo(wv.x) * xs[0];
  a = fmaf(bf16_hi(wv.x), xs[1], a);
  a = fmaf(bf16_lo(wv.y), xs[2], a);
  a = fmaf(bf16_hi(wv.y), xs[3], a);
  a = fmaf(bf16_lo(wv.z), xs[4], a);
  a = fmaf(bf16_hi(wv.z), xs[5], a);
  a = fmaf(bf16_lo(wv.w), xs[6], a);
  a = fmaf(bf16_hi(wv.w), xs[7], a);
  return a;
}

// int4 dot products on packed fp16 pairs.  For a 32-bit word of eight codes
// (element n in nibble n), ((word >> 4 k) & 0x000F000F) | 0x6400_6400 is the
// fp16 pair (1024 + u_k, 1024 + u_{k+4}) exactly (fp16 has unit spacing on
// [1024, 2048)), so one packed subtract gives the codes (u - 8 for the
// signed format, whose nibbles are first flipped to u = q + 8; u for the
// affine one) and one packed fma multiplies them by the activation pair
// (x_k, x_{k+4}).  Per 32-code chunk the products are summed in fp16 (eight
// per half), then in fp32: about three instructions per weight instead of
// five for a convert-and-fma per code.

// fp16 pair (lo, hi), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The activation pairs of one code word from 8 bf16 values (one 16-byte
// chunk): pair k = (x_k, x_{k+4}).
__device__ __forceinline__ void xpairs_bf16(const uint4 xv, uint32_t (&h)[4]) {
  h[0] = pack_f16x2(bf16_lo(xv.x), bf16_lo(xv.z));
  h[1] = pack_f16x2(bf16_hi(xv.x), bf16_hi(xv.z));
  h[2] = pack_f16x2(bf16_lo(xv.y), bf16_lo(xv.w));
  h[3] = pack_f16x2(bf16_hi(xv.y), bf16_hi(xv.w));
}

// Same from 8 fp32 values.
__device__ __forceinline__ void xpairs_f32(const float *x8, uint32_t (&h)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = pack_f16x2(x8[k], x8[k + 4]);
}

// acc + (q_k x_k, q_{k+4} x_{k+4}) summed over k, packed fp16.
template <bool SIGNED>
__device__ __forceinline__ uint32_t hdot8(uint32_t word, const uint32_t (&h)[4], uint32_t acc) {
  if (SIGNED) word ^= 0x88888888u;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t v = ((word >> (4 * k)) & 0x000F000Fu) | 0x64006400u;
    asm("{\n .reg .b32 t;\n sub.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %0;\n}"
        : "+r"(acc)
        : "r"(v), "r"(SIGNED ? 0x64086408u : 0x64006400u), "r"(h[k]));
  }
  return acc;
}

// fp32 sum of the four halves of two fp16 pairs.
__device__ __forceinline__ float hsum4(uint32_t a, uint32_t b) {
  const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&a));
  const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&b));
  return (fa.x + fa.y) + (fb.x + fb.y);
}

// 32 codes (one 16-byte chunk; word w holds elements 8 w .. 8 w + 7) . the
// activation pairs of their four words: sum q * x without the group scale.
template <bool SIGNED>
__device__ __forceinline__ float dot32_int4(const uint4 wv, const uint32_t (&h)[4][4]) {
  uint32_t a0 = 0u, a1 = 0u;
  a0 = hdot8<SIGNED>(wv.x, h[0], a0);
  a1 = hdot8<SIGNED>(wv.y, h[1], a1);
  a0 = hdot8<SIGNED>(wv.z, h[2], a0);
  a1 = hdot8<SIGNED>(wv.w, h[3], a1);
  return hsum4(a0, a1);
}

// Chunking of one weight row for a warp: 16-byte chunks of EPC elements;
// lane l takes chunks l + 32 u.  A segment is U chunks per lane (2048
// elements for both formats), whose x slice is U * XPC 16-byte bf16 chunks.
template <int WF> struct Fmt;
template <> struct Fmt<0> { static constexpr int EPC = 8, XPC = 1, U = 8; };
template <> struct Fmt<1> { static constexpr int EPC = 32, XPC = 4, U = 2; };
template <> struct Fmt<2> : Fmt<1> {};   // affine int4: the same packing

// Bytes of one weight row of K elements.
template <int WF> __host__ __device__ __forceinline__ size_t row_bytes(int K) {
  return WF == 0 ? static_cast<size_t>(K) * 2 : static_cast<size_t>(K) / 2;
}

// One segment of a warp's dot products: lane l takes 16-byte chunks
// c0 + l + 32 u (u < U) of NR weight rows (seg_load_w) and the matching
// chunks of x (seg_load_x, from shared memory); seg_dots adds the chunks'
// dot products to acc.  Chunks past the row end load as zeros and add
// nothing: no branches, so the NR * U dot chains interleave.
template <int WF, int NR, bool L1>
__device__ __forceinline__ void seg_load_w(const void *const (&rows)[NR],
                                           const __nv_bfloat16 *const (&srows)[NR],
                                           const __nv_bfloat16 *const (&brows)[NR], int nchunk,
                                           int c0, int lane, uint4 (&wv)[NR][Fmt<WF>::U],
                                           float (&sv)[NR][Fmt<WF>::U],
                                           float (&bv)[NR][Fmt<WF>::U]) {
  using F = Fmt<WF>;
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int u = 0; u < F::U; ++u) {
      const int c = c0 + lane + 32 * u;
      const uint4 *wp = reinterpret_cast<const uint4 *>(rows[r]) + c;
      wv[r][u] = (c < nchunk) ? (L1 ? __ldg(wp) : ld_stream(wp)) : make_uint4(0, 0, 0, 0);
      if constexpr (WF != 0) sv[r][u] = (c < nchunk) ? __bfloat162float(__ldg(srows[r] + (c >> 1))) : 0.0f;
      if constexpr (WF == 2) bv[r][u] = (c < nchunk) ? __bfloat162float(__ldg(brows[r] + (c >> 1))) : 0.0f;
    }
}

template <int WF>
__device__ __forceinline__ void seg_load_x(const uint4 *xs, int nchunk, int c0, int lane,
                                           uint4 (&xv)[Fmt<WF>::U][Fmt<WF>::XPC]) {
  using F = Fmt<WF>;
#pragma unroll
  for (int u = 0; u < F::U; ++u)
#pragma unroll
    for (int q = 0; q < F::XPC; ++q) {
      const int c = c0 + lane + 32 * u;
      xv[u][q] = (c < nchunk) ? xs[c * F::XPC + q] : make_uint4(0, 0, 0, 0);
    }
}

template <int WF, int NR>
__device__ __forceinline__ void seg_dots(const uint4 (&wv)[NR][Fmt<WF>::U],
                                         const float (&sv)[NR][Fmt<WF>::U],
                                         const float (&bv)[NR][Fmt<WF>::U],
                                         const uint4 (&xv)[Fmt<WF>::U][Fmt<WF>::XPC],
                                         float (&acc)[NR]) {
  using F = Fmt<WF>;
  if constexpr (WF == 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < F::U; ++u) acc[r] += dot8_bf16_bf16(wv[r][u], xv[u][0]);
  } else {
    // the activation pairs (and, affine, the sum) of each chunk, once for
    // all NR rows
    uint32_t xh[F::U][4][4];
    float xs[F::U];
#pragma unroll
    for (int u = 0; u < F::U; ++u) {
      xs[u] = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xpairs_bf16(xv[u][q], xh[u][q]);
        if constexpr (WF == 2)
          xs[u] += (bf16_lo(xv[u][q].x) + bf16_hi(xv[u][q].x)) +
                   (bf16_lo(xv[u][q].y) + bf16_hi(xv[u][q].y)) +
                   (bf16_lo(xv[u][q].z) + bf16_hi(xv[u][q].z)) +
                   (bf16_lo(xv[u][q].w) + bf16_hi(xv[u][q].w));
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < F::U; ++u) {
        const float qx = dot32_int4<WF == 1>(wv[r][u], xh[u]);
        if constexpr (WF == 1) acc[r] = fmaf(sv[r][u], qx, acc[r]);
        else acc[r] = fmaf(sv[r][u], qx, fmaf(bv[r][u], xs[u], acc[r]));   // s * sum q x + b * sum x
      }
  }
}

// Dot products of NR weight rows of length K with the bf16 vector x, by one
// warp.  x is in shared memory (xs), filled by a bulk copy that completes
// phase `par` of the mbarrier mb_x: the weight loads of a segment are issued
// first, then the wait, then the x loads and the arithmetic.  (Every warp
// reading x from L2 instead moved more bytes into the SMs than the weights
// themselves for int4 rows.)  L1: weights through L1, for rows that the
// caller reads again soon.
template <int WF, int NR, bool L1 = false>
__device__ __forceinline__ void warp_dots_x(const void *const (&rows)[NR],
                                            const __nv_bfloat16 *const (&srows)[NR],
                                            const __nv_bfloat16 *const (&brows)[NR], int K,
                                            const uint4 *xs, uint32_t mb_x, uint32_t par,
                                            int *status, float (&out)[NR]) {
  using F = Fmt<WF>;
  const int lane = threadIdx.x & 31;
  const int nchunk = K / F::EPC;
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
  for (int c0 = 0; c0 < nchunk; c0 += 32 * F::U) {
    uint4 wv[NR][F::U];
    uint4 xv[F::U][F::XPC];
    float sv[NR][F::U], bv[NR][F::U];
    seg_load_w<WF, NR, L1>(rows, srows, brows, nchunk, c0, lane, wv, sv, bv);
    {
      volatile int no_abort = 0;
      mbar_wait_bounded(mb_x, par, &no_abort, status, DEV_TIMEOUT_STAGE);
    }
    seg_load_x<WF>(xs, nchunk, c0, lane, xv);
    seg_dots<WF, NR>(wv, sv, bv, xv, acc);
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

// int4 rows: the activation pairs (and, affine, the sums) of this lane's
// chunks of x, formed once per warp for every row it dots in a phase;
// warp_dots_x forms them again for each call.  The same values in the same
// order, so the dot products are bit-identical.  Only for a single segment
// (K <= 32 * U * EPC elements: K <= 2048).
template <int WF> struct XPairs {
  uint32_t h[Fmt<WF>::U][4][4];
  float s[Fmt<WF>::U];
};
template <int WF>
__device__ __forceinline__ bool xpairs_fit(int K) {
  return K / Fmt<WF>::EPC <= 32 * Fmt<WF>::U;
}
template <int WF>
__device__ __forceinline__ void make_xpairs(const uint4 *xs, int K, uint32_t mb_x, uint32_t par,
                                            int *status, XPairs<WF> &xp) {
  using F = Fmt<WF>;
  const int lane = threadIdx.x & 31;
  const int nchunk = K / F::EPC;
  {
    volatile int no_abort = 0;
    mbar_wait_bounded(mb_x, par, &no_abort, status, DEV_TIMEOUT_STAGE);
  }
  uint4 xv[F::U][F::XPC];
  seg_load_x<WF>(xs, nchunk, 0, lane, xv);
#pragma unroll
  for (int u = 0; u < F::U; ++u) {
    xp.s[u] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xpairs_bf16(xv[u][q], xp.h[u][q]);
      if constexpr (WF == 2)
        xp.s[u] += (bf16_lo(xv[u][q].x) + bf16_hi(xv[u][q].x)) +
                   (bf16_lo(xv[u][q].y) + bf16_hi(xv[u][q].y)) +
                   (bf16_lo(xv[u][q].z) + bf16_hi(xv[u][q].z)) +
                   (bf16_lo(xv[u][q].w) + bf16_hi(xv[u][q].w));
    }
  }
}
// warp_dots_x for int4 rows with the activation pairs already formed.
template <int WF, int NR>
__device__ __forceinline__ void warp_dots_xp(const void *const (&rows)[NR],
                                             const __nv_bfloat16 *const (&srows)[NR],
                                             const __nv_bfloat16 *const (&brows)[NR], int K,
                                             const XPairs<WF> &xp, float (&out)[NR]) {
  using F = Fmt<WF>;
  const int lane = threadIdx.x & 31;
  const int nchunk = K / F::EPC;
  uint4 wv[NR][F::U];
  float sv[NR][F::U], bv[NR][F::U];
  seg_load_w<WF, NR, false>(rows, srows, brows, nchunk, 0, lane, wv, sv, bv);
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    acc[r] = 0.0f;
#pragma unroll
    for (int u = 0; u < F::U; ++u) {
      const float qx = dot32_int4<WF == 1>(wv[r][u], xp.h[u]);
      if constexpr (WF == 1) acc[r] = fmaf(sv[r][u], qx, acc[r]);
      else acc[r] = fmaf(sv[r][u], qx, fmaf(bv[r][u], xp.s[u], acc[r]));
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

// The same for several activation rows: row t (bit t of `users`) is at
// xs + t * xq, and out(t, d) receives its NR sums (in every lane).  One
// warp_dots_x per user, the weights through L1, so that a row comes from HBM
// once.  (Keeping the weights in registers across the users instead measured
// slower: the kernel then spills.)
template <int WF, int NR, class Out>
__device__ __forceinline__ void warp_dots_users(const void *const (&rows)[NR],
                                                const __nv_bfloat16 *const (&srows)[NR],
                                                const __nv_bfloat16 *const (&brows)[NR], int K,
                                                const uint4 *xs, int xq, unsigned int users,
                                                uint32_t mb_x, int *status, Out out) {
  for (unsigned int m = users; m != 0u; m &= m - 1u) {
    const int t = __ffs(m) - 1;
    float d[NR];
    warp_dots_x<WF, NR, true>(rows, srows, brows, K, xs + t * xq, mb_x, 0u, status, d);
    out(t, d);
  }
}

// D += A . B on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32
// accumulators).  Lane l = 4 g + t holds A (16 x 16, row-major) rows g and
// g + 8 at columns 2t, 2t+1 (a0, a1) and 2t+8, 2t+9 (a2, a3); B (16 x 8,
// column-major) rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1) of column g; D rows
// g (d0, d1) and g + 8 (d2, d3) at columns 2t, 2t + 1.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The same for tf32 operands (mma.sync m16n8k8, fp32 accumulators): lane
// l = 4 g + t holds A (16 x 8) rows g, g + 8 at columns t (a0, a1) and t + 4
// (a2, a3), B (8 x 8) rows t (b0) and t + 4 (b1) of column g; D as above.
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t tf32_rn(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float f4_at(const float4 &lo, const float4 &hi, int e) {
  const float4 &v = e < 4 ? lo : hi;
  const int w = e & 3;
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Sixteen bf16 output-projection rows of K elements (K a multiple of 32;
// this lane's rows g and g + 8 at rg, rg8) dotted with up to 8 NH users' h
// (fp32 in global memory: hp[h] for user 8 h + g, null for none) on the
// tensor cores in tf32 (the weights exactly, h rounded to 10 fraction bits).
// In 32-wide chunk c, lane t's k slots t and t + 4 of step s are elements
// 32 c + 8 t + 2 s and 32 c + 8 t + 2 s + 1.  Two chunks of loads in flight.
// d[h] as for warp_mma_rows_users.
template <int NH>
__device__ __forceinline__ void warp_mma_tf32_rows_users(const __nv_bfloat16 *rg,
                                                         const __nv_bfloat16 *rg8, int K,
                                                         const float *const (&hp)[NH],
                                                         float (&d)[NH][4]) {
  const int lane = threadIdx.x & 31, t = lane & 3;
#pragma unroll
  for (int h = 0; h < NH; ++h) d[h][0] = d[h][1] = d[h][2] = d[h][3] = 0.0f;
  const int nch = K / 32;
  const uint4 *pa = reinterpret_cast<const uint4 *>(rg) + t;   // chunk c: pa[4 c]
  const uint4 *pb = reinterpret_cast<const uint4 *>(rg8) + t;
  uint4 w[2][2];
  float4 hv[2][NH][2];
  auto load = [&](int b, int c) {
    w[b][0] = __ldcg(pa + 4 * c);
    w[b][1] = __ldcg(pb + 4 * c);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (hp[h] != nullptr) {
        const float4 *q = reinterpret_cast<const float4 *>(hp[h] + 32 * c + 8 * t);
        hv[b][h][0] = __ldcg(q);
        hv[b][h][1] = __ldcg(q + 1);
      } else {
        hv[b][h][0] = hv[b][h][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
  };
#pragma unroll
  for (int b = 0; b < 2; ++b)
    if (b < nch) load(b, b);
  for (int c = 0; c < nch; c += 2) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int cc = c + b;
      if (cc < nch) {
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const uint32_t wg = st == 0 ? w[b][0].x : st == 1 ? w[b][0].y : st == 2 ? w[b][0].z : w[b][0].w;
          const uint32_t wg8 = st == 0 ? w[b][1].x : st == 1 ? w[b][1].y : st == 2 ? w[b][1].z : w[b][1].w;
          const uint32_t a0 = wg << 16, a2 = wg & 0xffff0000u;
          const uint32_t a1 = wg8 << 16, a3 = wg8 & 0xffff0000u;
#pragma unroll
          for (int h = 0; h < NH; ++h)
            mma_tf32_1688(d[h], a0, a1, a2, a3, tf32_rn(f4_at(hv[b][h][0], hv[b][h][1], 2 * st)),
                          tf32_rn(f4_at(hv[b][h][0], hv[b][h][1], 2 * st + 1)));
        }
        if (cc + 2 < nch) load(b, cc + 2);
      }
    }
  }
}

constexpr int kRowsMmaDepth = 2;
constexpr int kRowsMmaPrefetch = 6;   // chunks further ahead prefetched into L2
// Word m (0..7) of the 32 bytes lo, hi.
__device__ __forceinline__ uint32_t word8(const uint4 &lo, const uint4 &hi, int m) {
  const uint4 &v = m < 4 ? lo : hi;
  const int w = m & 3;
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Sixteen bf16 weight rows of K elements (K a multiple of 64; this lane's
// rows g and g + 8 start at rg and rg8) dotted with the rows of up to 8 NH
// users in shared memory (xs: [T][K] bf16), on the tensor cores: every
// weight byte is loaded once for all users.  Inside each 16-wide MMA step
// the k order is permuted so that each lane's operands are whole 16-byte
// loads: in 64-wide chunk c, the k slots 2t, 2t+1, 2t+8, 2t+9 of step s are
// elements 64 c + 16 t + 4 s + 0..3, for A and B alike (the products summed
// are the same).  kRowsMmaDepth chunks of loads are kept in flight, and the
// next kRowsMmaPrefetch chunks are prefetched into L2.  On return d[h]
// holds rows g, g + 8 (d0, d1 and d2, d3) of users 8 h + 2 t, 8 h + 2 t + 1.
template <int NH>
__device__ __forceinline__ void warp_mma_rows_users(const __nv_bfloat16 *rg,
                                                    const __nv_bfloat16 *rg8, int K,
                                                    const __nv_bfloat16 *xs, int T,
                                                    uint32_t mb_x, int *status,
                                                    float (&d)[NH][4]) {
  constexpr int DEPTH = kRowsMmaDepth;   // chunks of loads in flight
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int h = 0; h < NH; ++h) d[h][0] = d[h][1] = d[h][2] = d[h][3] = 0.0f;
  const int nch = K / 64;
  const uint4 *pa = reinterpret_cast<const uint4 *>(rg) + 2 * t;   // chunk c: pa[8 c], pa[8 c + 1]
  const uint4 *pb = reinterpret_cast<const uint4 *>(rg8) + 2 * t;
  uint4 w[DEPTH][4];
#pragma unroll
  for (int b = 0; b < DEPTH; ++b)
    if (b < nch) {
      w[b][0] = ld_stream(pa + 8 * b);
      w[b][1] = ld_stream(pa + 8 * b + 1);
      w[b][2] = ld_stream(pb + 8 * b);
      w[b][3] = ld_stream(pb + 8 * b + 1);
    }
  if (t == 0)
    for (int c = DEPTH; c < DEPTH + kRowsMmaPrefetch && c < nch; ++c) {
      prefetch_l2_line(rg + 64 * c);
      prefetch_l2_line(rg8 + 64 * c);
    }
  {
    volatile int no_abort = 0;   // the users' rows have landed in shared memory
    mbar_wait_bounded(mb_x, 0u, &no_abort, status, DEV_TIMEOUT_STAGE);
  }
  for (int c = 0; c < nch; c += DEPTH) {
#pragma unroll
    for (int b = 0; b < DEPTH; ++b) {
      const int cc = c + b;
      if (cc < nch) {
        uint4 xv[NH][2];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int user = 8 * h + g;
          if (user < T) {
            const uint4 *px = reinterpret_cast<const uint4 *>(xs + static_cast<size_t>(user) * K) +
                              8 * cc + 2 * t;
            xv[h][0] = px[0];
            xv[h][1] = px[1];
          } else {
            xv[h][0] = xv[h][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          const uint32_t a0 = word8(w[b][0], w[b][1], 2 * st);
          const uint32_t a2 = word8(w[b][0], w[b][1], 2 * st + 1);
          const uint32_t a1 = word8(w[b][2], w[b][3], 2 * st);
          const uint32_t a3 = word8(w[b][2], w[b][3], 2 * st + 1);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            mma_bf16_16816(d[h], a0, a1, a2, a3, word8(xv[h][0], xv[h][1], 2 * st),
                           word8(xv[h][0], xv[h][1], 2 * st + 1));
        }
        if (t == 0 && cc + DEPTH + kRowsMmaPrefetch < nch) {
          // one 128-byte line per row and chunk
          prefetch_l2_line(rg + 64 * (cc + DEPTH + kRowsMmaPrefetch));
          prefetch_l2_line(rg8 + 64 * (cc + DEPTH + kRowsMmaPrefetch));
        }
        if (cc + DEPTH < nch) {
          w[b][0] = ld_stream(pa + 8 * (cc + DEPTH));
          w[b][1] = ld_stream(pa + 8 * (cc + DEPTH) + 1);
          w[b][2] = ld_stream(pb + 8 * (cc + DEPTH));
          w[b][3] = ld_stream(pb + 8 * (cc + DEPTH) + 1);
        }
      }
    }
  }
}

// Row r of a K-major matrix with K columns, bf16 or packed int4.
template <int WF>
__device__ __forceinline__ const void *row_ptr(const void *base, size_t r, int K) {
  return static_cast<const uint8_t *>(base) + r * row_bytes<WF>(K);
}
__device__ __forceinline__ const __nv_bfloat16 *scale_row(const void *base, size_t r, int K) {
  return base ? reinterpret_cast<const __nv_bfloat16 *>(base) + r * (K / 64) : nullptr;
}

// ------------------------------------------------------ grid barrier --
// A 64-bit arrival counter that only grows: barrier b of a launch completes
// when the counter reaches base + b * gridDim.x, where base is the counter's
// value at launch (a multiple of gridDim.x: every completed launch adds
// exactly two grid-widths).  A CTA reads base before its first arrival; no
// barrier of this launch can complete before that arrival, so the value it
// reads lies in [base, base + gridDim.x).
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait (one thread) until the counter holds `target` arrivals; the writes
// those arrivals released are visible afterwards.  A thread that waits longer
// than kWaitLimitCycles records DEV_TIMEOUT_GRID and carries on.
__device__ __forceinline__ void grid_wait(const unsigned long long *bar, unsigned long long target,
                                          int *status) {
  if (ld_acquire_u64(bar) < target) {
    const long long t0 = clock64();
    while (ld_acquire_u64(bar) < target) {
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicExch(status, DEV_TIMEOUT_GRID);
        break;
      }
    }
  }
}

// Arrive and wait until `target` arrivals; the CTA's earlier writes are
// released with the arrival.
__device__ __forceinline__ void grid_sync(unsigned long long *bar, unsigned long long target,
                                          int *status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    red_release_add_u64(bar, 1ull);
    grid_wait(bar, target, status);
  }
  __syncthreads();
}

// ------------------------------------------------- one decode layer --
// Dynamic shared memory of one CTA, in this order:
//   x     [H] bf16               the layer's input (one bulk copy per layer)
//   part  [(k+1) p3_rows] fp32   per-slot dot products of the CTA's output rows
//   w3    the CTA's output-projection rows (p3_stage only): k slots of p3_rows
//         rows of I for the routed experts, then one of p3_rows rows of Is
//   ws    int4 (p3_scales only): the bf16 group scales of those rows, then
//         (affine) their biases, in the same order
struct DecSmem {
  size_t part, w3, w3_sh, unstaged, staged;
  size_t ws, ws_sh, wb, wb_sh, scaled;
};
template <int WF>
__host__ __device__ __forceinline__ DecSmem dec_smem(int k, int I, int Is, int rows, int H) {
  DecSmem L{};
  L.part = (static_cast<size_t>(H) * 2 + 127) / 128 * 128;   // x (bf16) first
  L.w3 = L.part + (static_cast<size_t>(k + 1) * rows * sizeof(float) + 127) / 128 * 128;
  L.unstaged = L.w3;
  L.w3_sh = L.w3 + static_cast<size_t>(k) * rows * row_bytes<WF>(I);
  L.staged = L.w3_sh + static_cast<size_t>(rows) * row_bytes<WF>(Is);
  const size_t sI = static_cast<size_t>(rows) * (I / 64) * 2, sIs = static_cast<size_t>(rows) * (Is / 64) * 2;
  L.ws = (L.staged + 127) / 128 * 128;
  L.ws_sh = L.ws + k * sI;
  L.wb = L.ws_sh + sIs;
  L.wb_sh = L.wb + (WF == 2 ? k * sI : 0);
  L.scaled = L.wb_sh + (WF == 2 ? sIs : 0);
  return L;
}

// Per-CTA state shared by every layer of a launch: the shared-memory carve-up
// (part, staged output-projection rows), the CTA's output rows and its two
// mbarriers (shared-expert rows, routed rows; one phase per layer).
struct DecCta {
  float *part;
  unsigned char *w3, *w3_sh;
  unsigned char *ws, *ws_sh, *wb, *wb_sh;   // staged int4 scales / biases (p3_scales)
  const uint4 *x_s;   // the layer input in shared memory
  int n0, n1, nrows, ngroups;
  uint32_t mb_sh, mb_rt, mb_x;
};

// One phase-C task: part[j][t0 + r] = (output-projection row n0 + t0 + r of
// slot j) . h_j for r < 8, slot j < k a routed expert and j = k the shared
// one; h_j = hbase + j h_ld.  The rows come from shared memory (STAGED) or global memory; h_j comes
// from global memory (L2).  Lane l takes 16-byte chunks l + 32 m and keeps
// the matching h elements in registers across the eight rows.
template <int WF, bool STAGED>
__device__ __forceinline__ void slot_task(const DecodeParams &p, const float *hbase, int j, int t0,
                                          int n0, int nrows, int expert, float *part,
                                          const unsigned char *w3, const unsigned char *w3_sh,
                                          const DecCta *cs = nullptr) {
  using F = Fmt<WF>;
  const int lane = threadIdx.x & 31;
  const bool sh = (j == p.k);
  const int K = sh ? p.Is : p.I;
  const int nch = K / F::EPC, ng = K / 64;
  const size_t rb = row_bytes<WF>(K);
  const float *hj = hbase + static_cast<size_t>(j) * p.h_ld;
  const size_t r0 = (sh ? 0 : static_cast<size_t>(expert) * p.H) + n0 + t0;   // global row
  const unsigned char *wrow;   // row t0 of the group
  if constexpr (STAGED)
    wrow = sh ? w3_sh + static_cast<size_t>(t0) * rb
              : w3 + (static_cast<size_t>(j) * p.p3_rows + t0) * rb;
  else
    wrow = static_cast<const unsigned char *>(sh ? p.sh_down : p.down) + r0 * rb;
  const __nv_bfloat16 *srow =
      WF != 0 ? static_cast<const __nv_bfloat16 *>(sh ? p.sh_down_scale : p.down_scale) + r0 * ng
              : nullptr;
  const __nv_bfloat16 *brow =
      WF == 2 ? static_cast<const __nv_bfloat16 *>(sh ? p.sh_down_bias : p.down_bias) + r0 * ng
              : nullptr;
  if (STAGED && WF != 0 && cs != nullptr && p.p3_scales) {
    // the scales (and biases) staged in shared memory beside the rows
    const size_t so = (sh ? static_cast<size_t>(t0) : static_cast<size_t>(j) * p.p3_rows + t0) * ng * 2;
    srow = reinterpret_cast<const __nv_bfloat16 *>((sh ? cs->ws_sh : cs->ws) + so);
    if (WF == 2) brow = reinterpret_cast<const __nv_bfloat16 *>((sh ? cs->wb_sh : cs->wb) + so);
  }
  // bf16 rows: two chunks per lane per pass, so that both h loads (from L2)
  // are in flight together
  constexpr int CU = WF == 0 ? 2 : 1;
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
  if constexpr (WF != 0) {
    if (nch <= 16) {
      // int4 rows of at most 16 chunks (K <= 512): two lanes per chunk, 16
      // codes (two words) each, so that every lane works
      const int hc = lane;                       // half chunk: codes 16 hc .. 16 hc + 15
      const bool act = hc < 2 * nch;
      float hv[16];
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const float4 h4 = act ? __ldcg(reinterpret_cast<const float4 *>(hj + hc * 16 + e))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        hv[e] = h4.x;
        hv[e + 1] = h4.y;
        hv[e + 2] = h4.z;
        hv[e + 3] = h4.w;
      }
      float hs = 0.0f;
      if constexpr (WF == 2)
#pragma unroll
        for (int e = 0; e < 16; ++e) hs += hv[e];
      uint32_t hh[2][4];
      xpairs_f32(&hv[0], hh[0]);
      xpairs_f32(&hv[8], hh[1]);
      const int hcc = act ? hc : 0;   // inactive lanes read a valid word and add 0 (h = 0)
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int rr = min(r, nrows - 1 - t0);
        const uint2 wv = reinterpret_cast<const uint2 *>(wrow + rr * rb)[hcc];
        uint32_t a0 = hdot8<WF == 1>(wv.x, hh[0], 0u);
        uint32_t a1 = hdot8<WF == 1>(wv.y, hh[1], 0u);
        const float qx = hsum4(a0, a1);
        const float sc = __bfloat162float(srow[rr * ng + (hcc >> 2)]);
        if constexpr (WF == 1) {
          acc[r] = fmaf(sc, qx, acc[r]);
        } else {
          const float bc = __bfloat162float(brow[rr * ng + (hcc >> 2)]);
          acc[r] = fmaf(sc, qx, fmaf(bc, hs, acc[r]));
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) acc[r] = warp_sum(acc[r]);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (t0 + r < nrows) part[j * p.p3_rows + t0 + r] = acc[r];
      }
      return;
    }
  }
  for (int c0 = lane; c0 < nch; c0 += 32 * CU) {
    float hv[CU][F::EPC];
#pragma unroll
    for (int u = 0; u < CU; ++u) {
      const int c = c0 + 32 * u;
#pragma unroll
      for (int e = 0; e < F::EPC; e += 4) {
        const float4 h4 = c < nch ? __ldcg(reinterpret_cast<const float4 *>(hj + c * F::EPC + e))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        hv[u][e] = h4.x;
        hv[u][e + 1] = h4.y;
        hv[u][e + 2] = h4.z;
        hv[u][e + 3] = h4.w;
      }
    }
    // rows past the CTA's last repeat that row (their sums are dropped) and
    // chunks past the row end hold zero h: no branches, so the chains of the
    // eight rows interleave
    float hs[CU];   // affine: the sum of each chunk's h values (for the group bias)
#pragma unroll
    for (int u = 0; u < CU; ++u) {
      hs[u] = 0.0f;
      if constexpr (WF == 2)
#pragma unroll
        for (int e = 0; e < F::EPC; ++e) hs[u] += hv[u][e];
    }
#pragma unroll
    for (int u = 0; u < CU; ++u) {
      const int c = min(c0 + 32 * u, nch - 1);
      uint32_t hh[4][4];   // int4: h as the fp16 pairs of the chunk's four code words
      if constexpr (WF != 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) xpairs_f32(&hv[u][8 * q], hh[q]);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int rr = min(r, nrows - 1 - t0);
        const uint4 wv = reinterpret_cast<const uint4 *>(wrow + rr * rb)[c];
        if constexpr (WF == 0) {
          acc[r] += dot8_bf16_f32(wv, hv[u]);
        } else if constexpr (WF == 1) {
          const float sc = __bfloat162float(srow[rr * ng + (c >> 1)]);
          acc[r] = fmaf(sc, dot32_int4<true>(wv, hh), acc[r]);
        } else {
          const float sc = __bfloat162float(srow[rr * ng + (c >> 1)]);
          const float bc = __bfloat162float(brow[rr * ng + (c >> 1)]);
          acc[r] = fmaf(sc, dot32_int4<false>(wv, hh), fmaf(bc, hs[u], acc[r]));
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = warp_sum(acc[r]);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (t0 + r < nrows) part[j * p.p3_rows + t0 + r] = acc[r];
  }
}

// slot_task for several activation rows: users (bit t) of one output
// projection (the shared one if sh), row t's h at h0 + t * hrow + j(t) h_ld
// and its parts at part0 + t * pstride; one slot_task per user, whose weight
// rows come from L1 after the first.
template <int WF, class SlotOf>
__device__ __forceinline__ void slot_task_users(const DecodeParams &p, const float *h0, size_t hrow,
                                                unsigned int users, SlotOf slot_of_t, int t0,
                                                int n0, int nrows, int expert, float *part0,
                                                size_t pstride) {
  for (unsigned int m = users; m != 0u; m &= m - 1u) {
    const int t = __ffs(m) - 1;
    slot_task<WF, false>(p, h0 + t * hrow, slot_of_t(t), t0, n0, nrows, expert, part0 + t * pstride,
                         nullptr, nullptr);
  }
}

template <int WF>
__device__ __forceinline__ void run_slot_task(const DecodeParams &p, int j, int t0, int n0,
                                              int nrows, int expert, float *part,
                                              const unsigned char *w3,
                                              const unsigned char *w3_sh, const DecCta *cs) {
  if (p.p3_stage) slot_task<WF, true>(p, p.h, j, t0, n0, nrows, expert, part, w3, w3_sh, cs);
  else slot_task<WF, false>(p, p.h, j, t0, n0, nrows, expert, part, w3, w3_sh);
}

template <int WF>
__device__ __forceinline__ DecCta make_dec_cta(const DecodeParams &p, unsigned char *dsm,
                                               uint64_t *mbar) {
  const DecSmem S = dec_smem<WF>(p.k, p.I, p.Is, p.p3_rows, p.H);
  DecCta c;
  c.x_s = reinterpret_cast<const uint4 *>(dsm);
  c.part = reinterpret_cast<float *>(dsm + S.part);
  c.w3 = dsm + S.w3;
  c.w3_sh = dsm + S.w3_sh;
  c.ws = dsm + S.ws;
  c.ws_sh = dsm + S.ws_sh;
  c.wb = dsm + S.wb;
  c.wb_sh = dsm + S.wb_sh;
  c.n0 = static_cast<int>((static_cast<long long>(blockIdx.x) * p.H) / gridDim.x);
  c.n1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.H) / gridDim.x);
  c.nrows = c.n1 - c.n0;
  c.ngroups = (c.nrows + 7) / 8;
  c.mb_sh = smem_u32(&mbar[0]);
  c.mb_rt = smem_u32(&mbar[1]);
  c.mb_x = smem_u32(&mbar[2]);
  return c;
}

// Routing-independent weight traffic of layer p, which may start before the
// layer's input is ready: thread 0 bulk-copies the CTA's rows of the shared
// expert's output projection into shared memory (one phase of mb_sh), and
// warp gw (numbered across CTAs) prefetches phase-A row gw into L2.
template <int WF>
__device__ __forceinline__ void layer_prefetch(const DecodeParams &p, const DecCta &c, int gw) {
  if (threadIdx.x == 0 && p.p3_stage) {
    const uint32_t bytes = static_cast<uint32_t>(c.nrows * row_bytes<WF>(p.Is));
    const uint32_t sbytes = p.p3_scales ? static_cast<uint32_t>(c.nrows * (p.Is / 64) * 2) : 0u;
    mbar_arrive_expect_tx(c.mb_sh, bytes + (WF == 2 ? 2 : 1) * sbytes);
    if (bytes) bulk_copy_g2s(smem_u32(c.w3_sh), row_ptr<WF>(p.sh_down, c.n0, p.Is), bytes, c.mb_sh);
    if (sbytes) {
      bulk_copy_g2s(smem_u32(c.ws_sh), scale_row(p.sh_down_scale, c.n0, p.Is), sbytes, c.mb_sh);
      if (WF == 2)
        bulk_copy_g2s(smem_u32(c.wb_sh), scale_row(p.sh_down_bias, c.n0, p.Is), sbytes, c.mb_sh);
    }
  }
  const int nA = p.E + 1 + p.Is;
  if (gw < nA) {
    if (gw < p.E) prefetch_row_l2(row_ptr<0>(p.router_w, gw, p.H), row_bytes<0>(p.H));
    else if (gw == p.E) prefetch_row_l2(p.sh_gate_w, row_bytes<0>(p.H));
    else {
      prefetch_row_l2(row_ptr<WF>(p.sh_gate_up, gw - p.E - 1, p.H), row_bytes<WF>(p.H));
      prefetch_row_l2(row_ptr<WF>(p.sh_gate_up, p.Is + gw - p.E - 1, p.H), row_bytes<WF>(p.H));
    }
  }
}

// One decode layer, phases A to C (see the top of this file), after
// layer_prefetch(p) has been issued and the layer's input is ready.  `par`
// is the parity of this layer's mbarrier phases, bar_base the value of the
// barrier counter p.bar[0] its two grid barriers count from (thread 0 only),
// sh_base that of p.bar[1], on which every CTA announces its share of the
// shared expert's h (all threads); `next`, if not null, is the following
// layer, whose layer_prefetch is issued after this layer's second grid
// barrier.
template <int WF, int R>
__device__ __forceinline__ void decode_layer(const DecodeParams &p, const DecCta &c, uint32_t par,
                                             unsigned long long bar_base,
                                             unsigned long long sh_base, const DecodeParams *next,
                                             int *idx_s, float *w_s) {
  float *part = c.part;
  unsigned char *w3 = c.w3;
  unsigned char *w3_sh = c.w3_sh;
  const int n0 = c.n0, n1 = c.n1, nrows = c.nrows, ngroups = c.ngroups;
  const uint32_t mb_sh = c.mb_sh, mb_rt = c.mb_rt, mb_x = c.mb_x;
  const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  // warps numbered across CTAs first, so that a partly filled phase spreads
  // over every SM
  const int gw = warp * G + blockIdx.x;
  const int nw = G * kDecWarps;
  float *hg = p.h;   // [k+1][h_ld]: h of the k experts, then of the shared expert
  const size_t rbI = row_bytes<WF>(p.I);
  // int4: this warp's activation pairs, formed once for phases A and B
  const bool use_xp = WF != 0 && xpairs_fit<WF>(p.H);
  XPairs<WF == 0 ? 1 : WF> xp;
  bool have_xp = false;
  (void)n1;
  (void)lane;
  (void)x;
  if (threadIdx.x == 0) {
    // the layer input into shared memory (x was written by generic stores of
    // the previous kernel or layer, acquired before this point)
    const uint32_t xbytes = static_cast<uint32_t>(p.H) * 2;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    fence_proxy_async_smem();   // the previous layer's reads of x_s come first
    mbar_arrive_expect_tx(mb_x, xbytes);
    bulk_copy_g2s(smem_u32(c.x_s), p.x, xbytes, mb_x);
  }
  // ---- phase A: router rows and the shared gate row on the first RW warps
  // of every CTA, which arrive on the grid barrier as soon as they are done;
  // the shared expert's row pairs on the other warps meanwhile (their h is
  // needed only by the output projection: every CTA announces its share on
  // the second counter, p.bar[1]).  Top-k then waits for the router alone.
  const int nR = p.E + 1;
  const int RW = min(kDecWarps - 1, (nR + G - 1) / G);
  if (warp < RW) {
    for (int it = warp * G + blockIdx.x; it < nR; it += RW * G) {
      const void *rows[1] = {it < p.E ? row_ptr<0>(p.router_w, it, p.H) : p.sh_gate_w};
      const __nv_bfloat16 *sr[1] = {nullptr};
      float d[1];
      warp_dots_x<0, 1>(rows, sr, sr, p.H, c.x_s, c.mb_x, par, p.status, d);
      if (lane == 0) {
        if (it < p.E) p.logits[it] = d[0] + (p.router_b ? p.router_b[it] : 0.0f);
        else *p.g = sigmoid_f(d[0]);
      }
    }
    named_bar_sync(1, RW * 32);
    if (threadIdx.x == 0) {
      red_release_add_u64(p.bar, 1ull);
      grid_wait(p.bar, bar_base + G, p.status);
    }
  } else {
    for (int i = (warp - RW) * G + blockIdx.x; i < p.Is; i += (kDecWarps - RW) * G) {
      const void *rows[2] = {row_ptr<WF>(p.sh_gate_up, i, p.H),
                             row_ptr<WF>(p.sh_gate_up, p.Is + i, p.H)};
      const __nv_bfloat16 *sr[2] = {scale_row(p.sh_gate_up_scale, i, p.H),
                                    scale_row(p.sh_gate_up_scale, p.Is + i, p.H)};
      const __nv_bfloat16 *br[2] = {scale_row(p.sh_gate_up_bias, i, p.H),
                                    scale_row(p.sh_gate_up_bias, p.Is + i, p.H)};
      float d[2];
      if constexpr (WF != 0) {
        if (use_xp) {
          if (!have_xp) {
            make_xpairs<WF>(c.x_s, p.H, c.mb_x, par, p.status, xp);
            have_xp = true;
          }
          warp_dots_xp<WF, 2>(rows, sr, br, p.H, xp, d);
        } else {
          warp_dots_x<WF, 2>(rows, sr, br, p.H, c.x_s, c.mb_x, par, p.status, d);
        }
      } else {
        warp_dots_x<WF, 2>(rows, sr, br, p.H, c.x_s, c.mb_x, par, p.status, d);
      }
      if (lane == 0) hg[static_cast<size_t>(p.k) * p.h_ld + i] = silu_f(d[0]) * d[1];
    }
    named_bar_sync(2, (kDecWarps - RW) * 32);
    if (threadIdx.x == RW * 32) red_release_add_u64(p.bar + 1, 1ull);
  }

  // ---- top-k (one warp per CTA, after the first grid barrier; the logits
  // are in L2)
  if (warp == 0) {
    __syncwarp();
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = lane + 32 * r;
      v[r] = (e < p.E) ? __ldcg(p.logits + e) : 0.0f;
    }
    const float g = __ldcg(p.g);
    int sel_e;
    float sel_w;
    warp_topk_redux<R>(v, p.E, p.k, sel_e, sel_w);
    sel_e = min(max(sel_e, 0), p.E - 1);
    if (lane < p.k) {
      idx_s[lane] = sel_e;
      w_s[lane] = sel_w;
      if (blockIdx.x == 0) {
        p.idx[lane] = sel_e;
        p.w[lane] = sel_w;
      }
    }
    if (lane == 0) w_s[32] = g;
  }
  __syncthreads();
  if (p.phase_ts != nullptr && threadIdx.x == 0) p.phase_ts[2 * blockIdx.x] = global_ns();
  // The last warps have the fewest phase-B rows: they issue the copies.
  if (warp == kDecWarps - 1 && p.p3_stage) {
    // the k routed experts' output rows n0..n1, one bulk copy per expert
    const uint32_t bytes = static_cast<uint32_t>(nrows * rbI);
    const uint32_t sbytes = p.p3_scales ? static_cast<uint32_t>(nrows * (p.I / 64) * 2) : 0u;
    if (lane == 0) {
      mbar_arrive_expect_tx(mb_rt, (bytes + (WF == 2 ? 2 : 1) * sbytes) * p.k);
      if (bytes)
        for (int j = 0; j < p.k; ++j) {
          const size_t r0 = static_cast<size_t>(idx_s[j]) * p.H + n0;
          bulk_copy_g2s(smem_u32(w3 + static_cast<size_t>(j) * p.p3_rows * rbI),
                        row_ptr<WF>(p.down, r0, p.I), bytes, mb_rt);
          if (sbytes) {
            const size_t so = static_cast<size_t>(j) * p.p3_rows * (p.I / 64) * 2;
            bulk_copy_g2s(smem_u32(c.ws + so), scale_row(p.down_scale, r0, p.I), sbytes, mb_rt);
            if (WF == 2)
              bulk_copy_g2s(smem_u32(c.wb + so), scale_row(p.down_bias, r0, p.I), sbytes, mb_rt);
          }
        }
    }
  }
  if (WF != 0 && !p.p3_scales && warp == kDecWarps - 2 && nrows > 0) {
    // int4 group scales (and affine biases) of those rows, into L2 for phase C
    for (int j = 0; j <= p.k; ++j) {
      const bool sh = (j == p.k);
      const size_t r0 = sh ? 0 : static_cast<size_t>(idx_s[j]) * p.H;
      const int K = sh ? p.Is : p.I;
      for (int t = 0; t < (WF == 2 ? 2 : 1); ++t) {
        const void *sb = t == 0 ? (sh ? p.sh_down_scale : p.down_scale)
                                : (sh ? p.sh_down_bias : p.down_bias);
        const char *s0 = reinterpret_cast<const char *>(scale_row(sb, r0 + n0, K));
        const char *s1 = reinterpret_cast<const char *>(scale_row(sb, r0 + n1, K));
        for (const char *a = line_of(s0) + lane * 128; a < s1; a += 32 * 128) prefetch_l2_line(a);
      }
    }
  }

  // ---- phase B: routed gate/up row pairs -> h
  const int nB = p.k * p.I;
  for (int q = gw; q < nB; q += nw) {
    const int j = q / p.I, i = q - j * p.I;
    const size_t rg = static_cast<size_t>(idx_s[j]) * 2 * p.I + i;
    const void *rows[2] = {row_ptr<WF>(p.gate_up, rg, p.H), row_ptr<WF>(p.gate_up, rg + p.I, p.H)};
    const __nv_bfloat16 *sr[2] = {scale_row(p.gate_up_scale, rg, p.H),
                                  scale_row(p.gate_up_scale, rg + p.I, p.H)};
    const __nv_bfloat16 *br[2] = {scale_row(p.gate_up_bias, rg, p.H),
                                  scale_row(p.gate_up_bias, rg + p.I, p.H)};
    float d[2];
    if constexpr (WF != 0) {
      if (use_xp) {
        if (!have_xp) {
          make_xpairs<WF>(c.x_s, p.H, c.mb_x, par, p.status, xp);
          have_xp = true;
        }
        warp_dots_xp<WF, 2>(rows, sr, br, p.H, xp, d);
      } else {
        warp_dots_x<WF, 2>(rows, sr, br, p.H, c.x_s, c.mb_x, par, p.status, d);
      }
    } else {
      warp_dots_x<WF, 2>(rows, sr, br, p.H, c.x_s, c.mb_x, par, p.status, d);
    }
    if (lane == 0) hg[static_cast<size_t>(j) * p.h_ld + i] = silu_f(d[0]) * d[1];
  }
  // The shared expert's slot needs only h_s (announced on p.bar[1] long
  // before): the last warps, which have the fewest phase-B rows, do it now.
  if (kDecWarps - 1 - warp < ngroups) {
    if (lane == 0) grid_wait(p.bar + 1, sh_base + G, p.status);
    __syncwarp();
  }
  for (int s = kDecWarps - 1 - warp; s < ngroups; s += kDecWarps) {
    if (p.p3_stage) {
      volatile int no_abort = 0;
      mbar_wait_bounded(mb_sh, par, &no_abort, p.status, DEV_TIMEOUT_STAGE);
    }
    run_slot_task<WF>(p, p.k, 8 * s, n0, nrows, 0, part, w3, w3_sh, &c);
  }
  if (p.phase_ts != nullptr) {   // profiling: the end of this CTA's phase B
    __syncthreads();
    if (threadIdx.x == 0) p.phase_ts[2 * blockIdx.x + 1] = global_ns();
  }
  grid_sync(p.bar, bar_base + 2 * static_cast<unsigned long long>(G), p.status);
  // The next layer's routing-independent weight traffic can start now: this
  // layer's shared-expert rows are consumed (phase B) and DRAM is idle from
  // here on.
  if (next != nullptr) {
    if (threadIdx.x == 0 && p.p3_stage) {
      volatile int no_abort = 0;   // this layer's phase of mb_sh is complete
      mbar_wait_bounded(mb_sh, par, &no_abort, p.status, DEV_TIMEOUT_STAGE);
    }
    layer_prefetch<WF>(*next, c, gw);
  }

  // ---- phase C: the routed slots, one (slot j, group of 8 rows) per warp
  if (p.p3_stage) {
    // the staged rows must have landed before this thread reads them
    volatile int no_abort = 0;
    mbar_wait_bounded(mb_rt, par, &no_abort, p.status, DEV_TIMEOUT_STAGE);
  }
  for (int task = warp; task < p.k * ngroups; task += kDecWarps) {
    const int j = task / ngroups, t0 = (task - j * ngroups) * 8;
    run_slot_task<WF>(p, j, t0, n0, nrows, idx_s[j], part, w3, w3_sh, &c);
  }
  __syncthreads();
  // y[n] = sum_j w_j part[j] + g part[k], in that order
  for (int t = threadIdx.x; t < nrows; t += kDecLayerThreads) {
    float y = 0.0f;
    for (int j0 = 0; j0 <= p.k; j0 += 8) {
      // eight slots per pass, loads first; slots past k add 0 * (a valid part)
      float pw[8], pv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = min(j0 + u, p.k);
        pv[u] = part[j * p.p3_rows + t];
        pw[u] = j0 + u > p.k ? 0.0f : w_s[j == p.k ? 32 : j];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) y = fmaf(pw[u], pv[u], y);
    }
    reinterpret_cast<__nv_bfloat16 *>(p.y)[n0 + t] = __float2bfloat16_rn(y);
  }
}

// Persistent cooperative kernel, one CTA per SM (see the top of this file):
// one layer.
template <int WF, int R>
__global__ void __launch_bounds__(kDecLayerThreads, 1) decode_layer_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) uint64_t mbar[3];   // shared expert rows, routed rows, x
  __shared__ int idx_s[32];
  __shared__ float w_s[33];                   // routing weights, then the shared gate
  const DecCta c = make_dec_cta<WF>(p, dsm, mbar);
  const int G = gridDim.x;
  const int gw = (threadIdx.x >> 5) * G + blockIdx.x;

  __shared__ unsigned long long sh_base_s;
  unsigned long long base = 0;   // barrier counter at launch (used by thread 0)
  if (threadIdx.x == 0) {
    // With a programmatic launch this CTA can start while the previous
    // layer's CTAs finish, but only after the one on this SM exited, i.e.
    // after that layer's last barrier completed: both counters are final.
    const unsigned long long v = ld_acquire_u64(p.bar);
    base = v - v % static_cast<unsigned long long>(G);
    const unsigned long long v1 = ld_acquire_u64(p.bar + 1);
    sh_base_s = v1 - v1 % static_cast<unsigned long long>(G);
    if (p.p3_stage) {
      mbar_init(c.mb_sh, 1);
      mbar_init(c.mb_rt, 1);
    }
    mbar_init(c.mb_x, 1);
    fence_mbarrier_init();
  }
  __syncthreads();   // the barriers exist before any thread waits on mb_x
  // Only weights are read before the wait below: x, and every buffer this
  // kernel writes, may still be in use by the previous layer.
  layer_prefetch<WF>(p, c, gw);
  pdl_trigger();
  pdl_wait();
  decode_layer<WF, R>(p, c, 0u, base, sh_base_s, nullptr, idx_s, w_s);
}

// The same for n consecutive layers in one launch (P.layer[0..n-1], same
// shapes): layer l + 1 starts after a grid barrier that follows layer l's
// last write (so its input may be layer l's output), and its
// routing-independent weight traffic starts during layer l's output
// projection.  The barrier counter advances by 3 n - 1 grid widths.
template <int WF, int R>
__global__ void __launch_bounds__(kDecLayerThreads, 1)
    decode_layers_kernel(const __grid_constant__ DecodeLayersParams P) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) uint64_t mbar[3];
  __shared__ int idx_s[32];
  __shared__ float w_s[33];
  const DecodeParams &p0 = P.layer[0];
  const DecCta c = make_dec_cta<WF>(p0, dsm, mbar);
  const int G = gridDim.x;
  const int gw = (threadIdx.x >> 5) * G + blockIdx.x;
  __shared__ unsigned long long sh_base_s;
  unsigned long long base = 0;
  if (threadIdx.x == 0) {
    const unsigned long long v = ld_acquire_u64(p0.bar);
    base = v - v % static_cast<unsigned long long>(G);
    const unsigned long long v1 = ld_acquire_u64(p0.bar + 1);
    sh_base_s = v1 - v1 % static_cast<unsigned long long>(G);
    if (p0.p3_stage) {
      mbar_init(c.mb_sh, 1);
      mbar_init(c.mb_rt, 1);
    }
    mbar_init(c.mb_x, 1);
    fence_mbarrier_init();
  }
  __syncthreads();   // the barriers exist before any thread waits on mb_x
  layer_prefetch<WF>(p0, c, gw);
  pdl_trigger();
  pdl_wait();
  for (int l = 0; l < P.n; ++l) {
    const DecodeParams &p = P.layer[l];
    const unsigned long long lb = base + 3ull * static_cast<unsigned long long>(l) * G;
    decode_layer<WF, R>(p, c, static_cast<uint32_t>(l & 1), lb,
                        sh_base_s + static_cast<unsigned long long>(l) * G,
                        l + 1 < P.n ? &P.layer[l + 1] : nullptr, idx_s, w_s);
    // layer l's outputs are complete before layer l + 1 reads its input
    if (l + 1 < P.n) grid_sync(p.bar, lb + 3ull * G, p.status);
  }
}

// ------------------------------------------------------------ a few rows --
// T = 1 .. kSmallMaxRows rows of one layer ("Limits of further optimization":
// verifying drafted tokens processes groups of two to five rows, which often
// select different experts).  The decode layer's structure, with every weight
// row streamed once for all the rows that use it:
//   A. router rows, the shared gate row and the shared expert's row pairs,
//      each dotted with all T inputs (x [T, H] staged in shared memory);
//   B. per-row top-k (warp t of every CTA for row t), the union of the
//      selected experts in ascending expert order, then items (u, i): the
//      gate/up row pair i of union expert u with every row that selected u
//      (bf16 weights: items of eight row pairs on the tensor cores, with all
//      T rows as the MMA's N columns, one or two blocks of eight);
//   C. each CTA's output rows n0..n1 of every union expert and of the shared
//      expert (tasks of 8 rows) with the h of each user row, then
//      y[t][n] = sum_j w[t][j] part[t][j][n] + g[t] part[t][k][n] in fixed j
//      order.
// A row read for several users comes from HBM once and from L1 after that.
// Phase C reads its rows from global memory (no staging: the union holds up
// to T k experts).
//
// Dynamic shared memory: x [T][H] bf16, then part [T][k + 1][p3_rows] fp32.
struct RowsSmem {
  size_t part, total;
};
__host__ __device__ __forceinline__ RowsSmem rows_smem(int T, int k, int H, int rows) {
  RowsSmem L{};
  L.part = (static_cast<size_t>(T) * H * 2 + 127) / 128 * 128;
  L.total = L.part + static_cast<size_t>(T) * (k + 1) * rows * sizeof(float);
  return L;
}
constexpr int kRowsMaxUnion = kSmallMaxRows * 32;   // T k with k <= 32
// From this many rows up, bf16 gate/up items run on the tensor cores: with
// fewer rows the per-user passes keep more loads in flight per SM.
constexpr int kRowsMmaMinRows = 5;

template <int WF, int R>
__global__ void __launch_bounds__(kDecLayerThreads, 1) rows_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) uint64_t mb_x_store;
  __shared__ int idx_s[kSmallMaxRows * 32];
  __shared__ float w_s[kSmallMaxRows * 32];
  __shared__ float g_s[kSmallMaxRows];
  __shared__ short umap[1024];                      // expert -> union index
  __shared__ short ue[kRowsMaxUnion];               // union index -> expert
  __shared__ unsigned int users[kRowsMaxUnion];     // bit t: row t selected the expert
  __shared__ signed char slot_of[kRowsMaxUnion][kSmallMaxRows];
  __shared__ int n_union;
  const int T = p.T, H = p.H, E = p.E, k = p.k;
  const RowsSmem S = rows_smem(T, k, H, p.p3_rows);
  const uint4 *x_s = reinterpret_cast<const uint4 *>(dsm);
  float *part = reinterpret_cast<float *>(dsm + S.part);
  const uint32_t mb_x = smem_u32(&mb_x_store);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int gw = warp * G + blockIdx.x;
  const int nw = G * kDecWarps;
  const int n0 = static_cast<int>((static_cast<long long>(blockIdx.x) * H) / G);
  const int n1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * H) / G);
  const int nrows = n1 - n0, ngroups = (nrows + 7) / 8;
  const size_t hrow = static_cast<size_t>(k + 1) * p.h_ld;   // h floats per row t
  const uint32_t all_rows = T >= 32 ? 0xffffffffu : (1u << T) - 1u;

  unsigned long long base = 0;
  if (threadIdx.x == 0) {
    const unsigned long long v = ld_acquire_u64(p.bar);
    base = v - v % static_cast<unsigned long long>(G);
    mbar_init(mb_x, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  // only weights before the wait: x and the scratch may still be in use
  layer_prefetch<WF>(p, DecCta{}, gw);
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    const uint32_t xbytes = static_cast<uint32_t>(T) * H * 2;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_arrive_expect_tx(mb_x, xbytes);
    bulk_copy_g2s(smem_u32(x_s), p.x, xbytes, mb_x);
  }
  const int xq = H / 8;   // uint4 per x row

  // ---- A: router rows, the gate row, shared pairs; all T rows
  const int nA = E + 1 + p.Is;
  for (int it = gw; it < nA; it += nw) {
    if (it <= E) {
      const void *rows[1] = {it < E ? row_ptr<0>(p.router_w, it, H) : p.sh_gate_w};
      const __nv_bfloat16 *sr[1] = {nullptr};
      warp_dots_users<0, 1>(rows, sr, sr, H, x_s, xq, all_rows, mb_x, p.status,
                            [&](int t, const float (&d)[1]) {
                              if (lane == 0) {
                                if (it < E)
                                  p.logits[static_cast<size_t>(t) * E + it] =
                                      d[0] + (p.router_b ? p.router_b[it] : 0.0f);
                                else
                                  p.g[t] = sigmoid_f(d[0]);
                              }
                            });
    } else {
      const int i = it - E - 1;
      const void *rows[2] = {row_ptr<WF>(p.sh_gate_up, i, H), row_ptr<WF>(p.sh_gate_up, p.Is + i, H)};
      const __nv_bfloat16 *sr[2] = {scale_row(p.sh_gate_up_scale, i, H),
                                    scale_row(p.sh_gate_up_scale, p.Is + i, H)};
      const __nv_bfloat16 *br[2] = {scale_row(p.sh_gate_up_bias, i, H),
                                    scale_row(p.sh_gate_up_bias, p.Is + i, H)};
      warp_dots_users<WF, 2>(rows, sr, br, H, x_s, xq, all_rows, mb_x, p.status,
                             [&](int t, const float (&d)[2]) {
                               if (lane == 0)
                                 p.h[t * hrow + static_cast<size_t>(k) * p.h_ld + i] = silu_f(d[0]) * d[1];
                             });
    }
  }
  grid_sync(p.bar, base + G, p.status);

  // ---- top-k per row (warps 0..T-1 of every CTA), then the union
  if (warp < T) {
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = lane + 32 * r;
      v[r] = (e < E) ? __ldcg(p.logits + static_cast<size_t>(warp) * E + e) : 0.0f;
    }
    int sel_e;
    float sel_w;
    warp_topk_redux<R>(v, E, k, sel_e, sel_w);
    sel_e = min(max(sel_e, 0), E - 1);
    if (lane < k) {
      idx_s[warp * 32 + lane] = sel_e;
      w_s[warp * 32 + lane] = sel_w;
      if (blockIdx.x == 0) {
        p.idx[warp * k + lane] = sel_e;
        p.w[warp * k + lane] = sel_w;
      }
    }
    if (lane == 0) g_s[warp] = __ldcg(p.g + warp);
  }
  for (int e = threadIdx.x; e < E; e += kDecLayerThreads) umap[e] = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < T * k; q += kDecLayerThreads) umap[idx_s[(q / k) * 32 + q % k]] = 1;
  __syncthreads();
  if (warp == 0) {
    // union in ascending expert order: rank = number of marked experts below
    int nu = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool f = e < E && umap[e] != 0;
      const unsigned int b = __ballot_sync(0xffffffffu, f);
      const int rank = nu + __popc(b & ((1u << lane) - 1u));
      __syncwarp();
      if (f) {
        umap[e] = static_cast<short>(rank);
        ue[rank] = static_cast<short>(e);
      }
      nu += __popc(b);
    }
    if (lane == 0) n_union = nu;
  }
  for (int u = threadIdx.x; u < kRowsMaxUnion; u += kDecLayerThreads) users[u] = 0u;
  __syncthreads();
  const int U = n_union;
  for (int q = threadIdx.x; q < T * k; q += kDecLayerThreads) {
    const int t = q / k, j = q - (q / k) * k;
    const int u = umap[idx_s[t * 32 + j]];
    atomicOr(&users[u], 1u << t);
    slot_of[u][t] = static_cast<signed char>(j);
  }
  __syncthreads();
  if (warp == kDecWarps - 1 && nrows > 0) {
    // this CTA's output rows of the union experts (and their int4 scales and
    // biases) into L2 while phase B streams the gate/up rows
    const size_t rbI = row_bytes<WF>(p.I);
    for (int u = 0; u < U; ++u) {
      const size_t r0 = static_cast<size_t>(ue[u]) * H + n0;
      prefetch_row_l2(row_ptr<WF>(p.down, r0, p.I), nrows * rbI);
      if (WF != 0) prefetch_row_l2(scale_row(p.down_scale, r0, p.I), nrows * (p.I / 64) * 2);
      if (WF == 2) prefetch_row_l2(scale_row(p.down_bias, r0, p.I), nrows * (p.I / 64) * 2);
    }
  }

  // ---- B: union gate/up row pairs with their user rows -> h
  bool b_done = false;
  if constexpr (WF == 0) {
    if (T >= kRowsMmaMinRows && p.I % 8 == 0 && H % 64 == 0) {
      // bf16 rows on the tensor cores: items of 8 row pairs (gate rows
      // i0..i0+7 as A rows 0..7, the matching up rows as A rows 8..15) with
      // all T rows at once; lane (g, t) ends with gate and up of row pair
      // i0 + g for users 2t, 2t + 1 (and 8 + 2t, 9 + 2t)
      const int I8 = p.I / 8;
      const int nB8 = U * I8;
      const int g = lane >> 2, t2 = 2 * (lane & 3);
      const __nv_bfloat16 *xsb = reinterpret_cast<const __nv_bfloat16 *>(x_s);
      const __nv_bfloat16 *gu = static_cast<const __nv_bfloat16 *>(p.gate_up);
      for (int q = gw; q < nB8; q += nw) {
        const int u = q / I8, i = (q - u * I8) * 8 + g;
        const size_t rg = static_cast<size_t>(ue[u]) * 2 * p.I + i;
        const unsigned int us = users[u];
        auto put = [&](const float (&dd)[4], int tb) {
          if ((us >> tb) & 1u)
            p.h[tb * hrow + static_cast<size_t>(slot_of[u][tb]) * p.h_ld + i] = silu_f(dd[0]) * dd[2];
          if ((us >> (tb + 1)) & 1u)
            p.h[(tb + 1) * hrow + static_cast<size_t>(slot_of[u][tb + 1]) * p.h_ld + i] =
                silu_f(dd[1]) * dd[3];
        };
        if (T > 8) {
          float d[2][4];
          warp_mma_rows_users<2>(gu + rg * H, gu + (rg + p.I) * H, H, xsb, T, mb_x, p.status, d);
          put(d[0], t2);
          put(d[1], 8 + t2);
        } else {
          float d[1][4];
          warp_mma_rows_users<1>(gu + rg * H, gu + (rg + p.I) * H, H, xsb, T, mb_x, p.status, d);
          put(d[0], t2);
        }
      }
      b_done = true;
    }
  }
  // int4 rows (and bf16 rows of other shapes): one CUDA-core pass per user
  const int nB = b_done ? 0 : U * p.I;
  for (int q = gw; q < nB; q += nw) {
    const int u = q / p.I, i = q - u * p.I;
    const size_t rg = static_cast<size_t>(ue[u]) * 2 * p.I + i;
    const void *rows[2] = {row_ptr<WF>(p.gate_up, rg, H), row_ptr<WF>(p.gate_up, rg + p.I, H)};
    const __nv_bfloat16 *sr[2] = {scale_row(p.gate_up_scale, rg, H),
                                  scale_row(p.gate_up_scale, rg + p.I, H)};
    const __nv_bfloat16 *br[2] = {scale_row(p.gate_up_bias, rg, H),
                                  scale_row(p.gate_up_bias, rg + p.I, H)};
    warp_dots_users<WF, 2>(rows, sr, br, H, x_s, xq, users[u], mb_x, p.status,
                           [&](int t, const float (&d)[2]) {
                             if (lane == 0)
                               p.h[t * hrow + static_cast<size_t>(slot_of[u][t]) * p.h_ld + i] =
                                   silu_f(d[0]) * d[1];
                           });
  }
  grid_sync(p.bar, base + 2 * static_cast<unsigned long long>(G), p.status);

  // ---- C: output rows n0..n1 of the union experts (u < U) and the shared
  // expert (u = U), 8 rows per task, for each user row
  const size_t pstride = static_cast<size_t>(k + 1) * p.p3_rows;   // part floats per row t
  bool c_done = false;
  if constexpr (WF == 0) {
    if (b_done && p.I % 32 == 0 && p.Is % 32 == 0) {
      // bf16 rows on the tensor cores (tf32): tasks of 16 output rows with
      // all T rows at once; lane (g, t) ends with rows r0 + g, r0 + 8 + g
      // for users 2t, 2t + 1 (and 8 + 2t, 9 + 2t)
      const int g = lane >> 2, t2 = 2 * (lane & 3);
      const int ng16 = (nrows + 15) / 16;
      for (int task = warp; task < (U + 1) * ng16; task += kDecWarps) {
        const int u = task / ng16, r0 = (task - u * ng16) * 16;
        const bool sh = (u == U);
        const int K = sh ? p.Is : p.I;
        const unsigned int us = sh ? all_rows : users[u];
        const __nv_bfloat16 *base = static_cast<const __nv_bfloat16 *>(sh ? p.sh_down : p.down);
        const size_t row0 = (sh ? 0 : static_cast<size_t>(ue[u]) * H) + n0;
        const int ra = min(r0 + g, nrows - 1), rb8 = min(r0 + 8 + g, nrows - 1);
        auto slot = [&](int tt) { return sh ? k : static_cast<int>(slot_of[u][tt]); };
        auto hptr = [&](int tt) -> const float * {
          return (tt < T && ((us >> tt) & 1u)) ? p.h + tt * hrow + static_cast<size_t>(slot(tt)) * p.h_ld
                                               : nullptr;
        };
        auto put = [&](const float (&dd)[4], int tb) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tt = tb + e;
            if (tt < T && ((us >> tt) & 1u)) {
              float *pt = part + tt * pstride + static_cast<size_t>(slot(tt)) * p.p3_rows;
              if (r0 + g < nrows) pt[r0 + g] = dd[e];
              if (r0 + 8 + g < nrows) pt[r0 + 8 + g] = dd[2 + e];
            }
          }
        };
        if (T > 8) {
          const float *hp[2] = {hptr(g), hptr(8 + g)};
          float d[2][4];
          warp_mma_tf32_rows_users<2>(base + (row0 + ra) * K, base + (row0 + rb8) * K, K, hp, d);
          put(d[0], t2);
          put(d[1], 8 + t2);
        } else {
          const float *hp[1] = {hptr(g)};
          float d[1][4];
          warp_mma_tf32_rows_users<1>(base + (row0 + ra) * K, base + (row0 + rb8) * K, K, hp, d);
          put(d[0], t2);
        }
      }
      c_done = true;
    }
  }
  for (int task = warp; task < (c_done ? 0 : (U + 1) * ngroups); task += kDecWarps) {
    const int u = task / ngroups, t0 = (task - u * ngroups) * 8;
    const bool sh = (u == U);
    slot_task_users<WF>(p, p.h, hrow, sh ? all_rows : users[u],
                        [&](int t) { return sh ? k : static_cast<int>(slot_of[u][t]); }, t0, n0,
                        nrows, sh ? 0 : ue[u], part, pstride);
  }
  __syncthreads();
  // y[t][n] = sum_j w[t][j] part[t][j][n] + g[t] part[t][k][n], in that order
  for (int q = threadIdx.x; q < T * nrows; q += kDecLayerThreads) {
    const int t = q / nrows, n = q - t * nrows;
    const float *pt = part + t * pstride;
    float y = 0.0f;
    for (int j = 0; j < k; ++j) y = fmaf(w_s[t * 32 + j], pt[j * p.p3_rows + n], y);
    y = fmaf(g_s[t], pt[k * p.p3_rows + n], y);
    reinterpret_cast<__nv_bfloat16 *>(p.y)[static_cast<size_t>(t) * H + n0 + n] = __float2bfloat16_rn(y);
  }
}

template <int WF>
static void set_p3(DecodeParams &p, int grid, int smem_limit, size_t *smem) {
  p.p3_rows = (p.H + grid - 1) / grid;
  const DecSmem S = dec_smem<WF>(p.k, p.I, p.Is, p.p3_rows, p.H);
  p.p3_stage = S.staged <= static_cast<size_t>(smem_limit) ? 1 : 0;
  // int4: stage the rows' scales (and biases) too when their row slices are
  // whole 16-byte bulk copies (I and Is multiples of 512, 16-byte aligned
  // bases) and they fit
  auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  const bool aligned = a16(p.down_scale) && a16(p.sh_down_scale) &&
                       (WF != 2 || (a16(p.down_bias) && a16(p.sh_down_bias)));
  p.p3_scales = WF != 0 && p.p3_stage && p.I % 512 == 0 && p.Is % 512 == 0 && aligned &&
                        S.scaled <= static_cast<size_t>(smem_limit)
                    ? 1
                    : 0;
  *smem = p.p3_scales ? S.scaled : p.p3_stage ? S.staged : S.unstaged;
}

static cudaLaunchConfig_t dec_config(int grid, size_t smem, bool pdl, cudaStream_t stream,
                                     cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kDecLayerThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

template <int WF, int R>
static cudaError_t launch_layer(DecodeParams p, int grid, int smem_limit, bool pdl,
                                cudaStream_t stream) {
  size_t smem = 0;
  set_p3<WF>(p, grid, smem_limit, &smem);
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = dec_config(grid, smem, pdl, stream, attr);
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<WF, R>, p);
}

template <int WF, int R>
static cudaError_t launch_layers(const DecodeParams *layers, int n, int grid, int smem_limit,
                                 bool pdl, cudaStream_t stream) {
  DecodeLayersParams P;
  size_t smem = 0;
  P.n = n;
  for (int l = 0; l < n; ++l) {
    P.layer[l] = layers[l];
    set_p3<WF>(P.layer[l], grid, smem_limit, &smem);
  }
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = dec_config(grid, smem, pdl, stream, attr);
  return cudaLaunchKernelEx(&cfg, decode_layers_kernel<WF, R>, P);
}

cudaError_t launch_decode_layer(const DecodeParams &p, int grid, int smem_limit, bool pdl,
                                cudaStream_t stream) {
  if (p.wfmt == 0)
    return p.E <= 256 ? launch_layer<0, 8>(p, grid, smem_limit, pdl, stream)
                      : launch_layer<0, 32>(p, grid, smem_limit, pdl, stream);
  if (p.wfmt == 2)
    return p.E <= 256 ? launch_layer<2, 8>(p, grid, smem_limit, pdl, stream)
                      : launch_layer<2, 32>(p, grid, smem_limit, pdl, stream);
  return p.E <= 256 ? launch_layer<1, 8>(p, grid, smem_limit, pdl, stream)
                    : launch_layer<1, 32>(p, grid, smem_limit, pdl, stream);
}

cudaError_t launch_decode_layers(const DecodeParams *layers, int n, int grid, int smem_limit,
                                 bool pdl, cudaStream_t stream) {
  if (n < 1 || n > kMaxDecodeLayers) return cudaErrorInvalidValue;
  const DecodeParams &p = layers[0];
  if (p.wfmt == 0)
    return p.E <= 256 ? launch_layers<0, 8>(layers, n, grid, smem_limit, pdl, stream)
                      : launch_layers<0, 32>(layers, n, grid, smem_limit, pdl, stream);
  if (p.wfmt == 2)
    return p.E <= 256 ? launch_layers<2, 8>(layers, n, grid, smem_limit, pdl, stream)
                      : launch_layers<2, 32>(layers, n, grid, smem_limit, pdl, stream);
  return p.E <= 256 ? launch_layers<1, 8>(layers, n, grid, smem_limit, pdl, stream)
                    : launch_layers<1, 32>(layers, n, grid, smem_limit, pdl, stream);
}

// Largest dynamic shared memory of the rows kernels (the device's opt-in
// limit less their static shared memory), set by decode_configure.
static int g_rows_smem_limit = 0;

template <int WF, int R>
static cudaError_t launch_rows_t(DecodeParams p, int grid, int smem_limit, bool pdl,
                                 cudaStream_t stream) {
  p.p3_rows = (p.H + grid - 1) / grid;
  p.p3_stage = 0;
  p.p3_scales = 0;
  const RowsSmem S = rows_smem(p.T, p.k, p.H, p.p3_rows);
  (void)smem_limit;
  if (S.total > static_cast<size_t>(g_rows_smem_limit)) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = dec_config(grid, S.total, pdl, stream, attr);
  return cudaLaunchKernelEx(&cfg, rows_kernel<WF, R>, p);
}

cudaError_t launch_rows(const DecodeParams &p, int grid, int smem_limit, bool pdl,
                        cudaStream_t stream) {
  if (p.T < 1 || p.T > kSmallMaxRows || p.k > 32 || p.E > 1024) return cudaErrorInvalidValue;
  if (p.wfmt == 0)
    return p.E <= 256 ? launch_rows_t<0, 8>(p, grid, smem_limit, pdl, stream)
                      : launch_rows_t<0, 32>(p, grid, smem_limit, pdl, stream);
  if (p.wfmt == 2)
    return p.E <= 256 ? launch_rows_t<2, 8>(p, grid, smem_limit, pdl, stream)
                      : launch_rows_t<2, 32>(p, grid, smem_limit, pdl, stream);
  return p.E <= 256 ? launch_rows_t<1, 8>(p, grid, smem_limit, pdl, stream)
                    : launch_rows_t<1, 32>(p, grid, smem_limit, pdl, stream);
}

cudaError_t decode_configure(int *smem_limit) {
  // Opt every instantiation into the device's largest dynamic shared memory;
  // each launch then asks for what its shape needs.
  int dev = 0, optin = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return e;
  const int bytes = optin - 1024;   // room for the kernel's static shared memory
  const void *kernels[] = {
      reinterpret_cast<const void *>(decode_layer_kernel<0, 8>),
      reinterpret_cast<const void *>(decode_layer_kernel<0, 32>),
      reinterpret_cast<const void *>(decode_layer_kernel<1, 8>),
      reinterpret_cast<const void *>(decode_layer_kernel<1, 32>),
      reinterpret_cast<const void *>(decode_layer_kernel<2, 8>),
      reinterpret_cast<const void *>(decode_layer_kernel<2, 32>),
      reinterpret_cast<const void *>(decode_layers_kernel<0, 8>),
      reinterpret_cast<const void *>(decode_layers_kernel<0, 32>),
      reinterpret_cast<const void *>(decode_layers_kernel<1, 8>),
      reinterpret_cast<const void *>(decode_layers_kernel<1, 32>),
      reinterpret_cast<const void *>(decode_layers_kernel<2, 8>),
      reinterpret_cast<const void *>(decode_layers_kernel<2, 32>)};
  for (const void *k : kernels)
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) !=
        cudaSuccess)
      return e;
  // the rows kernels hold about 17 KB of static shared memory (the union
  // tables): each may ask for the opt-in limit less that
  const void *rows_kernels[] = {
      reinterpret_cast<const void *>(rows_kernel<0, 8>),
      reinterpret_cast<const void *>(rows_kernel<0, 32>),
      reinterpret_cast<const void *>(rows_kernel<1, 8>),
      reinterpret_cast<const void *>(rows_kernel<1, 32>),
      reinterpret_cast<const void *>(rows_kernel<2, 8>),
      reinterpret_cast<const void *>(rows_kernel<2, 32>)};
  int rows_limit = bytes;
  for (const void *k : rows_kernels) {
    cudaFuncAttributes a{};
    if ((e = cudaFuncGetAttributes(&a, k)) != cudaSuccess) return e;
    const int dyn = optin - static_cast<int>(a.sharedSizeBytes) - 1024;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) !=
        cudaSuccess)
      return e;
    rows_limit = dyn < rows_limit ? dyn : rows_limit;
  }
  g_rows_smem_limit = rows_limit;
  *smem_limit = bytes;
  return cudaSuccess;
}

int decode_layer_grid(int num_sms) {
  return num_sms;   // one CTA per SM: every CTA must be co-resident
}

}  // namespace moe

