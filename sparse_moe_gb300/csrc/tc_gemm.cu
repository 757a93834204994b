// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for the prefill path:
//
//   router:  l[t, e]  = sum_h x[t,h] Wr[e,h] (+ b[e])              -> fp32
//   gate/up: h[p, i]  = silu(sum_h x[tok(p),h] Wg[e,i,h]) *
//                       sum_h x[tok(p),h] Wu[e,i,h]                 -> bf16
//   down:    o[p, n]  = sum_i h[p,i] Wd[e,n,i]                      -> bf16
//
// (sections "Dequantize weights during matrix multiplication", "Keep expert
// routing on the GPU" and "Match tile size to expert load" of "Optimizing
// On-Device Inference for Apple Silicon": grouped GEMM over the rows routed
// to each expert, fp32 accumulation, bf16 output, tile shape from the
// expert's row count.)
//
// Design (GB300-first, not the page's Metal design):
//  * weights sit on the MMA M side (128 rows per tile) and the routed token
//    rows on the N side (N = row count rounded up to 16, at most 256), so an
//    expert with 5 rows runs a 128x16 MMA rather than padding to 128 rows;
//  * the gate/up tile stacks 64 gate rows over the 64 matching up rows, so one
//    MMA produces both halves of 64 SwiGLU outputs; the epilogue pairs them
//    through a small shared-memory exchange;
//  * token rows of the gate/up GEMM are gathered straight from x by TMA
//    gather4 using the device-built permutation (no permuted copy of x);
//  * one persistent CTA per SM walks the device-built tile list; warp 0 is
//    the TMA producer, one thread of warp 1 issues tcgen05.mma, warps 2..5
//    drain the double-buffered TMEM accumulator while the next tile computes.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int BM = 128;                 // MMA M
constexpr int BK = 64;                  // K per pipeline stage (128-byte rows)
constexpr int BN_MAX = kBlockRowsMax;   // max MMA N (tokens per tile)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN_MAX * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int ACC_COLS = 256;                   // one accumulator buffer
constexpr int TMEM_COLS = 512;                  // two buffers
constexpr int NUM_THREADS = 192;                // producer, MMA, 4 epilogue warps
constexpr int XCH_FLOATS = 2 * 2 * 2 * 8 * 32;  // [buf][pair][dir][8 cols][32 lanes]

struct SmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vote[4];
};

constexpr size_t kGemmSmemBytes =
    1024 /*align slack*/ + STAGES * STAGE_BYTES + XCH_FLOATS * sizeof(float) + sizeof(SmemTail);

struct Tile {
  int valid;
  int row0, nrows, nmma;
  int nk;
  int a_row, a_row2;   // A rows (a_row2: up rows for gate/up)
  int m;
  int shared;
};

__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int tile) {
  Tile t;
  const int b = tile / p.m_tiles;
  t.m = tile - b * p.m_tiles;
  int e = 0;
  if (p.mode == MODE_ROUTER) {
    t.row0 = b * p.block_rows;
    t.nrows = min(p.block_rows, p.T - t.row0);
    t.shared = 0;
  } else {
    const int4 blk = p.blocks[b];
    e = blk.x;
    t.row0 = blk.y;
    t.nrows = blk.z;
    t.shared = (e == p.n_experts);
  }
  t.nmma = max(16, (t.nrows + 15) & ~15);
  t.valid = t.nrows > 0;
  if (p.mode == MODE_ROUTER) {
    t.nk = p.k_routed / BK;
    t.a_row = t.m * BM;
    t.a_row2 = 0;
  } else if (p.mode == MODE_GATEUP) {
    const int inter = t.shared ? p.inter_shared : p.inter_routed;
    t.nk = p.k_routed / BK;
    t.valid = t.valid && (t.m * 64 < inter);
    const int base = t.shared ? 0 : e * 2 * p.inter_routed;
    t.a_row = base + t.m * 64;
    t.a_row2 = base + inter + t.m * 64;
  } else {  // MODE_DOWN
    t.nk = (t.shared ? p.inter_shared : p.inter_routed) / BK;
    t.a_row = (t.shared ? 0 : e * p.hidden) + t.m * BM;
    t.a_row2 = 0;
  }
  return t;
}

__device__ __forceinline__ int num_tiles(const GemmParams &p) {
  const int nb = (p.mode == MODE_ROUTER) ? p.n_blocks_host : *p.n_blocks_dev;
  return nb * p.m_tiles;
}

// Token (row of x) feeding row r of a gate/up tile.
__device__ __forceinline__ int gather_row(const GemmParams &p, const Tile &t, int r) {
  const int pr = t.row0 + min(r, t.nrows - 1);
  return t.shared ? pr - p.shared_row0 : __ldg(p.sorted_rows + pr);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a_routed,
                   const __grid_constant__ CUtensorMap map_a_shared,
                   const __grid_constant__ CUtensorMap map_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float *xch = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
  SmemTail *tail = reinterpret_cast<SmemTail *>(xch + XCH_FLOATS);
  volatile int *abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tail->tmem_full[a]), 1);
      mbar_init(smem_u32(&tail->tmem_empty[a]), 4);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&map_a_routed);
    prefetch_tensormap(&map_a_shared);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tail->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  const int ntiles = num_tiles(p);

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile);
      if (!t.valid) continue;
      const CUtensorMap *amap = t.shared ? &map_a_shared : &map_a_routed;
      // Gather indices for this tile (gate/up): lane handles 4-row groups
      // g = lane and lane + 32.
      int rows[8];
      if (p.mode == MODE_GATEUP) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int r = 0; r < 4; ++r) rows[h * 4 + r] = gather_row(p, t, (lane + 32 * h) * 4 + r);
      }
      const uint32_t b_bytes = static_cast<uint32_t>(t.nmma) * BK * 2;
      for (int ks = 0; ks < t.nk; ++ks) {
        int got = 1;
        if (lane == 0)
          got = mbar_wait_bounded(smem_u32(&tail->empty[stage]), phase ^ 1, abort_flag, p.status,
                                  DEV_TIMEOUT_PRODUCER);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t full_bar = smem_u32(&tail->full[stage]);
        const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
        const uint32_t b_dst = a_dst + A_BYTES;
        const int k0 = ks * BK;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar, A_BYTES + b_bytes);
          if (p.mode == MODE_GATEUP) {
            tma_load_2d(a_dst, amap, k0, t.a_row, full_bar);
            tma_load_2d(a_dst + A_BYTES / 2, amap, k0, t.a_row2, full_bar);
          } else {
            tma_load_2d(a_dst, amap, k0, t.a_row, full_bar);
          }
        }
        __syncwarp();
        if (p.mode == MODE_GATEUP) {
          const int ngroups = t.nmma >> 2;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int g = lane + 32 * h;
            if (g < ngroups)
              tma_gather4(b_dst + g * 512, &map_b, k0, rows[h * 4 + 0], rows[h * 4 + 1],
                          rows[h * 4 + 2], rows[h * 4 + 3], full_bar);
          }
        } else {
          const int nbox = t.nmma >> 4;   // 16-row boxes
          if (lane < nbox) tma_load_2d(b_dst + lane * 2048, &map_b, k0, t.row0 + lane * 16, full_bar);
        }
        issued_parity[stage] = static_cast<int>(phase);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // Wait (bounded) for copies still in flight before the CTA exits.
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) {
          const unsigned long long t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&tail->full[s]), static_cast<uint32_t>(issued_parity[s])) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const Tile t = decode_tile(p, tile);
        if (!t.valid) continue;
        if (!mbar_wait_bounded(smem_u32(&tail->tmem_empty[acc]), aphase ^ 1, abort_flag, p.status,
                               DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const uint32_t idesc = idesc_bf16_f32(BM, t.nmma);
        for (int ks = 0; ks < t.nk; ++ks) {
          if (!mbar_wait_bounded(smem_u32(&tail->full[stage]), phase, abort_flag, p.status,
                                 DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + stage * STAGE_BYTES;
          const uint64_t a_desc = smem_desc_sw128(a_addr);
          const uint64_t b_desc = smem_desc_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (ks | kk) != 0);
          tc_commit(smem_u32(&tail->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tail->tmem_full[acc]));
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1;
        }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      tc_commit(smem_u32(&tail->drain));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&tail->drain), 0)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicExch(p.status, DEV_TIMEOUT_DRAIN);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int ew = warp - 2;              // 0..3
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile);
      if (!t.valid) continue;
      int got = 1;
      if (lane == 0)
        got = mbar_wait_bounded(smem_u32(&tail->tmem_full[acc]), aphase, abort_flag, p.status,
                                DEV_TIMEOUT_EPILOGUE);
      got = __shfl_sync(0xffffffffu, got, 0);
      // Agree across the four epilogue warps before any named barrier.
      if (lane == 0) tail->vote[ew] = got;
      named_bar_sync(1, 128);
      const int all_ok = tail->vote[0] & tail->vote[1] & tail->vote[2] & tail->vote[3];
      named_bar_sync(1, 128);
      if (!all_ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);

      if (p.mode == MODE_GATEUP) {
        // Lanes 0..63 of the accumulator hold gate rows, 64..127 the matching
        // up rows.  Warp quarter q<2 (gate) pairs with quarter q+2 (up).
        const bool is_gate = q < 2;
        const int pair = q & 1;
        const int i_col = t.m * 64 + pair * 32 + lane;
        __nv_bfloat16 *hout = reinterpret_cast<__nv_bfloat16 *>(p.out);
        int buf = 0;
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          float *mine_to = xch + ((buf * 2 + pair) * 2 + (is_gate ? 0 : 1)) * 256;
          const float *from = xch + ((buf * 2 + pair) * 2 + (is_gate ? 1 : 0)) * 256;
          // gate warp sends columns 8..15, up warp sends columns 0..7
#pragma unroll
          for (int c = 0; c < 8; ++c)
            mine_to[c * 32 + lane] = __uint_as_float(r[is_gate ? 8 + c : c]);
          named_bar_sync(1, 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int col = c0 + (is_gate ? c : 8 + c);
            const float g = is_gate ? __uint_as_float(r[c]) : from[c * 32 + lane];
            const float u = is_gate ? from[c * 32 + lane] : __uint_as_float(r[8 + c]);
            if (col < t.nrows) {
              const float hv = silu_f(g) * u;
              hout[static_cast<size_t>(t.row0 + col) * p.out_ld + i_col] = __float2bfloat16_rn(hv);
            }
          }
          buf ^= 1;
        }
      } else if (p.mode == MODE_DOWN) {
        const int n = t.m * BM + q * 32 + lane;
        __nv_bfloat16 *oout = reinterpret_cast<__nv_bfloat16 *>(p.out);
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (n < p.hidden) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c0 + c < t.nrows)
                oout[static_cast<size_t>(t.row0 + c0 + c) * p.out_ld + n] =
                    __float2bfloat16_rn(__uint_as_float(r[c]));
          }
        }
      } else {  // MODE_ROUTER
        const int e = t.m * BM + q * 32 + lane;
        float *lout = reinterpret_cast<float *>(p.out);
        const float bias = (p.bias != nullptr && e < p.n_experts) ? __ldg(p.bias + e) : 0.0f;
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (e < p.n_experts) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c0 + c < t.nrows)
                lout[static_cast<size_t>(t.row0 + c0 + c) * p.out_ld + e] =
                    __uint_as_float(r[c]) + bias;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tail->tmem_empty[acc]));
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

cudaError_t gemm_configure() {
  return cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kGemmSmemBytes));
}

cudaError_t launch_tc_gemm(const CUtensorMap &a_routed, const CUtensorMap &a_shared,
                           const CUtensorMap &b, const GemmParams &p, int grid,
                           cudaStream_t stream) {
  tc_gemm_kernel<<<grid, NUM_THREADS, kGemmSmemBytes, stream>>>(a_routed, a_shared, b, p);
  return cudaGetLastError();
}

}  // namespace moe
