// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM)
// for the prefill path:
//
//   router:  l[t, e]  = sum_h x[t,h] Wr[e,h] (+ b[e])              -> fp32
//   gate/up: h[p, i]  = silu(sum_h x[tok(p),h] Wg[e,i,h]) *
//                       sum_h x[tok(p),h] Wu[e,i,h]                 -> fp16
//   down:    o[p, n]  = sum_i h[p,i] Wd[e,n,i]                      -> fp16
//
// (sections "Dequantize weights during matrix multiplication", "Keep expert
// routing on the GPU" and "Match tile size to expert load" of "Optimizing
// On-Device Inference for Apple Silicon": grouped GEMM over the rows routed
// to each expert, fp32 accumulation, tile shape from the expert's row count.)
//
// Design (GB300-first, not the page's Metal design):
//  * weights sit on the MMA M side (128 rows per tile) and the routed token
//    rows on the N side (N = row count rounded up to 16, at most 256), so an
//    expert with 5 rows runs a 128x16 MMA rather than padding to 128 rows;
//  * the gate/up tile stacks 64 gate rows over the 64 matching up rows, so one
//    MMA produces both halves of 64 SwiGLU outputs; the epilogue pairs them
//    through a small shared-memory exchange;
//  * the weight tile (A) of each k-step is one or two TMA boxes (128-byte
//    swizzle) prefetched into L2 a tile ahead; the token rows (B) are
//    gathered by a group of warps per pipeline stage with 16-byte cp.async
//    copies written straight into the same 128-byte-swizzled K-major layout,
//    so no permuted copy of x is ever written.  (Measured on GB300: TMA
//    gather4 moves 512 bytes per request and tops out near 7-18 bytes/clock
//    per SM; the load/store path scales with the number of issuing warps.)
//  * one persistent CTA per SM walks the device-built tile list; one thread
//    of the MMA warp issues tcgen05.mma, four epilogue warps drain the
//    double-buffered TMEM accumulator while the next tile computes, and
//    transpose each 32x16 piece through shared memory so global stores are
//    16-byte vectors;
//  * the down projection runs with fp16 operands: the gate/up epilogue stores
//    h in fp16 (11 significant bits instead of bf16's 8), and four converter
//    warps turn each bf16 weight tile into fp16 in place in shared memory
//    before the MMA reads it (exact for |w| >= 2^-17; the swizzled layout is
//    unchanged since both types are 2 bytes).  o is stored in fp16.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// Optional wait-time tracing (compiled only with -DMOE_TRACE): per CTA, clock
// cycles each role spends waiting on each barrier, read back with
// moe_debug_read_trace().
#ifdef MOE_TRACE
__device__ unsigned long long g_moe_trace[3][1024][16];
#define MOE_T0() const long long _t0 = clock64()
#define MOE_TADD(slot)                                        \
  atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][slot], \
            static_cast<unsigned long long>(clock64() - _t0))
#else
#define MOE_T0()
#define MOE_TADD(slot)
#endif

constexpr int BM = 128;                 // MMA M
constexpr int BK = 64;                  // K per pipeline stage (128-byte rows)
constexpr int BN_MAX = kBlockRowsMax;   // max MMA N (tokens per tile)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN_MAX * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int ACC_COLS = 256;                   // one accumulator buffer
constexpr int TMEM_COLS = 512;                  // two buffers
// Warp roles.  The weight tile (A, contiguous rows) is loaded by TMA, issued
// by one thread; the token rows (B, gathered) by 16-byte cp.async from a
// group of warps per pipeline stage.  Measured on GB300: one warp sustains
// only about 7 bytes/clock of cp.async traffic, TMA about 30 bytes/clock per
// SM, and an M128 x N256 tile needs 32 (A) + 64 (B) bytes/clock.
constexpr int B_WARPS_PER_STAGE = 4;
constexpr int TMA_WARP = 0;                                  // warp 0
constexpr int B_WARP0 = 1;                                   // warps 1..16
constexpr int B_WARPS = STAGES * B_WARPS_PER_STAGE;
constexpr int MMA_WARP = B_WARP0 + B_WARPS;                  // warp 17
constexpr int EPI_WARP0 = MMA_WARP + 1;                      // warps 18..21
constexpr int CONV_WARP0 = EPI_WARP0 + 4;                    // warps 22..25 (converting modes)
constexpr int BASE_THREADS = CONV_WARP0 * 32;
constexpr int CONV_THREADS = 128;
constexpr int XCH_FLOATS = 2 * 2 * 2 * 8 * 32;  // [buf][pair][dir][8 cols][32 lanes]
constexpr int EPI_STAGE_BYTES = 4 * 16 * 64;    // per epilogue warp: 16 rows x 64 bytes
// Per B producer warp: offsets of the token rows it copies (every
// B_WARPS_PER_STAGE-th group of four rows of up to 256).
constexpr int kRowTab = 4 * ((BN_MAX / 4 + B_WARPS_PER_STAGE - 1) / B_WARPS_PER_STAGE);

struct SmemTail {
  uint64_t full[STAGES];
  uint64_t conv[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vote[4];
};

constexpr size_t kGemmSmemBytes = 1024 /*align slack*/ + STAGES * STAGE_BYTES +
                                  XCH_FLOATS * sizeof(float) + EPI_STAGE_BYTES +
                                  B_WARPS * kRowTab * sizeof(int) + sizeof(SmemTail);

struct Tile {
  int valid;
  int row0, nrows, nmma;
  int nk;
  int m;
  int shared;
  int a_row, a_row2;   // first A row (a_row2: first up row for gate/up)
  int a_valid_rows;    // A rows at or beyond this (tile-relative) read as zero
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
    t.a_valid_rows = p.n_experts - t.m * BM;
  } else if (p.mode == MODE_GATEUP) {
    const int inter = t.shared ? p.inter_shared : p.inter_routed;
    t.nk = p.k_routed / BK;
    t.valid = t.valid && (t.m * 64 < inter);
    const int base = t.shared ? 0 : e * 2 * p.inter_routed;
    t.a_row = base + t.m * 64;
    t.a_row2 = base + inter + t.m * 64;
    t.a_valid_rows = BM;
  } else {  // MODE_DOWN
    t.nk = (t.shared ? p.inter_shared : p.inter_routed) / BK;
    t.a_row = (t.shared ? 0 : e * p.hidden) + t.m * BM;
    t.a_row2 = 0;
    t.a_valid_rows = p.hidden - t.m * BM;
  }
  return t;
}

__device__ __forceinline__ int num_tiles(const GemmParams &p) {
  const int nb = (p.mode == MODE_ROUTER) ? p.n_blocks_host : *p.n_blocks_dev;
  return nb * p.m_tiles;
}

// Row of the B operand (x for router and gate/up, h for down) feeding row r
// of a tile; rows past the tile's end repeat its last row.
__device__ __forceinline__ int b_row(const GemmParams &p, const Tile &t, int r) {
  const int pr = t.row0 + min(r, t.nrows - 1);
  if (p.mode != MODE_GATEUP) return pr;
  return t.shared ? pr - p.shared_row0 : __ldg(p.sorted_rows + pr);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// In-place bf16 -> fp16 conversion of one 128x64 A tile (1024 16-byte
// chunks) by the 128 converter threads.
__device__ __forceinline__ void convert_tile_bf16_to_f16(uint32_t tile_addr, int ctid) {
#pragma unroll
  for (int i = 0; i < (A_BYTES / 16) / CONV_THREADS; ++i) {
    const uint32_t addr = tile_addr + (ctid + i * CONV_THREADS) * 16;
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(addr));
    uint32_t o[4];
    const uint32_t wi[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(wi[j] << 16);
      const float hi = __uint_as_float(wi[j] & 0xffff0000u);
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(hi), "f"(lo));
    }
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3])
                 : "memory");
  }
}

// One warp stores a [rows x 32] block of fp16 values (row-major, 64 bytes per
// row, staged in shared memory at `stage`) to global memory with 16-byte
// stores: lane l writes row (l / 4) + 8 * pass, columns 8 * (l % 4) .. +7.
__device__ __forceinline__ void warp_store_rows_f16(const uint8_t *stage, int rows, int valid_rows,
                                                    __half *dst, size_t ld, int lane) {
  for (int r0 = 0; r0 < rows; r0 += 8) {
    const int r = r0 + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * 64 + (lane & 3) * 16);
    if (r < valid_rows) *reinterpret_cast<uint4 *>(dst + r * ld + (lane & 3) * 8) = v;
  }
}

template <int CONV>
__global__ void __launch_bounds__(BASE_THREADS + (CONV != CONV_NONE ? CONV_THREADS : 0), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a_routed,
                   const __grid_constant__ CUtensorMap map_a_shared, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float *xch = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
  uint8_t *epi_stage = reinterpret_cast<uint8_t *>(xch + XCH_FLOATS);
  int *row_tab = reinterpret_cast<int *>(epi_stage + EPI_STAGE_BYTES);
  SmemTail *tail = reinterpret_cast<SmemTail *>(row_tab + B_WARPS * kRowTab);
  volatile int *abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&tail->full[s]), 1 + B_WARPS_PER_STAGE);
      mbar_init(smem_u32(&tail->conv[s]), CONV_THREADS / 32);
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
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&tail->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  const int ntiles = num_tiles(p);
#ifdef MOE_TRACE
  const long long t_kernel0 = clock64();
#endif

  if (warp == TMA_WARP) {
    // ------------------------------------------------ weight tiles (TMA) --
    // Lane 0 loads each k-step's 128 weight rows with TMA into the stage's A
    // region (complete_tx on the stage's full barrier); all lanes prefetch the
    // next tile's weight rows (all of K) into L2 first, since they stream from
    // DRAM and one SM cannot keep enough requests in flight to cover its
    // latency.
    const __nv_bfloat16 *a_routed = reinterpret_cast<const __nv_bfloat16 *>(p.a_routed);
    const __nv_bfloat16 *a_shared = reinterpret_cast<const __nv_bfloat16 *>(p.a_shared);
    auto prefetch_a = [&](int tile_id) {
      if (tile_id >= ntiles) return;
      const Tile u = decode_tile(p, tile_id);
      if (!u.valid) return;
      const __nv_bfloat16 *ab = u.shared ? a_shared : a_routed;
      const int ld = u.shared ? p.lda_shared : p.lda_routed;
      const uint32_t kbytes = static_cast<uint32_t>(u.nk * BK * 2);
      for (int r = lane; r < BM && r < u.a_valid_rows; r += 32) {
        const int row = (p.mode == MODE_GATEUP) ? ((r < 64) ? u.a_row + r : u.a_row2 + (r - 64))
                                                : u.a_row + r;
        prefetch_l2_bulk(ab + static_cast<size_t>(row) * ld, kbytes);
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s2 = 0; s2 < STAGES; ++s2) issued_parity[s2] = -1;
    int ok = 1;
    if (blockIdx.x < ntiles) prefetch_a(blockIdx.x);
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile);
      prefetch_a(tile + gridDim.x);
      if (!t.valid) continue;
      if (lane == 0) {
        const CUtensorMap *amap = t.shared ? &map_a_shared : &map_a_routed;
        for (int ks = 0; ks < t.nk; ++ks) {
          MOE_T0();
          if (!mbar_wait_bounded(smem_u32(&tail->empty[stage]), phase ^ 1, abort_flag, p.status,
                                 DEV_TIMEOUT_PRODUCER)) {
            ok = 0;
            break;
          }
          MOE_TADD(0);
          const uint32_t full_bar = smem_u32(&tail->full[stage]);
          const uint32_t a_dst = smem_base + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full_bar, A_BYTES);
          if (p.mode == MODE_GATEUP) {
            tma_load_2d(a_dst, amap, ks * BK, t.a_row, full_bar);
            tma_load_2d(a_dst + A_BYTES / 2, amap, ks * BK, t.a_row2, full_bar);
          } else {
            tma_load_2d(a_dst, amap, ks * BK, t.a_row, full_bar);
          }
          issued_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0) {
      // Wait (bounded) for copies still in flight before the CTA exits.
      for (int s2 = 0; s2 < STAGES; ++s2)
        if (issued_parity[s2] >= 0) {
          const long long t0 = cycles_now();
          while (!mbar_try_wait(smem_u32(&tail->full[s2]), static_cast<uint32_t>(issued_parity[s2])) &&
                 cycles_now() - t0 < kWaitLimitCycles) {
          }
        }
    }
    __syncwarp();
  } else if (warp >= B_WARP0 && warp < B_WARP0 + B_WARPS) {
    // ------------------------------------------------- token rows (cp.async) --
    // Warp group g owns pipeline stage g: for every k-step that lands in its
    // stage it copies the B slice (nmma rows of 128 bytes), each warp of the
    // group every B_WARPS_PER_STAGE-th group of four rows, waits for its own
    // copies, fences them for the tensor core and arrives on the stage's full
    // barrier.  Lane l copies 16-byte chunk l % 8 of rows 4 j + l / 8.
    const int bw = warp - B_WARP0;
    const int g = bw / B_WARPS_PER_STAGE;
    const int gq = bw - g * B_WARPS_PER_STAGE;
    int *rows_tab = row_tab + bw * kRowTab;          // my rows' element offsets
    const int c = lane & 7;
    const int rsub = lane >> 3;
    const __nv_bfloat16 *bsrc = reinterpret_cast<const __nv_bfloat16 *>(p.b);
    const uint32_t stage_b = smem_base + g * STAGE_BYTES + A_BYTES;
    const uint32_t full_bar = smem_u32(&tail->full[g]);
    const uint32_t empty_bar = smem_u32(&tail->empty[g]);
    const int btid = bw * 32 + lane;
    auto prefetch_b = [&](int tile_id) {
      if (tile_id >= ntiles) return;
      const Tile u = decode_tile(p, tile_id);
      if (!u.valid) return;
      const uint32_t kbytes = static_cast<uint32_t>(u.nk * BK * 2);
      for (int rb = btid; rb < u.nrows; rb += B_WARPS * 32)
        prefetch_l2_bulk(bsrc + static_cast<size_t>(b_row(p, u, rb)) * p.ldb, kbytes);
    };
    if (blockIdx.x < ntiles) prefetch_b(blockIdx.x);
    int it = 0;   // k-step counter over all tiles of this CTA
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile);
      prefetch_b(tile + gridDim.x);
      if (!t.valid) continue;
      bool table_ready = false;
      const int nquads = t.nmma / 4;
      for (int ks = 0; ks < t.nk; ++ks, ++it) {
        if ((it % STAGES) != g) continue;
        if (!table_ready) {
          __syncwarp();   // previous tile's table no longer read
          for (int e = lane; e < kRowTab; e += 32) {
            const int r = 4 * (gq + B_WARPS_PER_STAGE * (e >> 2)) + (e & 3);
            rows_tab[e] = (r < t.nmma) ? b_row(p, t, r) * p.ldb : 0;
          }
          __syncwarp();
          table_ready = true;
        }
        const uint32_t phase = static_cast<uint32_t>(it / STAGES) & 1u;
        int got = 1;
#ifdef MOE_TRACE
        const long long tb0 = clock64();
#endif
        if (lane == 0)
          got = mbar_wait_bounded(empty_bar, phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_PRODUCER);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
#ifdef MOE_TRACE
        const long long tb1 = clock64();
#endif
        const int kc = ks * BK + c * 8;
        for (int j = gq, e = rsub; j < nquads; j += B_WARPS_PER_STAGE, e += 4) {
          const int r = 4 * j + rsub;
          const uint32_t dst = stage_b + r * 128 + static_cast<uint32_t>((c ^ (r & 7)) << 4);
          cp_async16(dst, bsrc + rows_tab[e] + kc, 16u);
        }
        cp_async_commit();
#ifdef MOE_TRACE
        const long long tb2 = clock64();
#endif
        cp_async_wait<0>();
#ifdef MOE_TRACE
        if (lane == 0) {
          const long long tb3 = clock64();
          atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][8], static_cast<unsigned long long>(tb1 - tb0));
          atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][9], static_cast<unsigned long long>(tb2 - tb1));
          atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][10], static_cast<unsigned long long>(tb3 - tb2));
          atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][11], 1ull);
        }
#endif
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full_bar);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
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
        {
          MOE_T0();
          const bool w_ok = mbar_wait_bounded(smem_u32(&tail->tmem_empty[acc]), aphase ^ 1,
                                              abort_flag, p.status, DEV_TIMEOUT_MMA);
          MOE_TADD(3);
          if (!w_ok) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const uint32_t idesc =
            (CONV == CONV_BF16_TO_F16) ? idesc_f16_f32(BM, t.nmma) : idesc_bf16_f32(BM, t.nmma);
        for (int ks = 0; ks < t.nk; ++ks) {
          const uint32_t ready_bar =
              (CONV != CONV_NONE) ? smem_u32(&tail->conv[stage]) : smem_u32(&tail->full[stage]);
          MOE_T0();
          const bool r_ok = mbar_wait_bounded(ready_bar, phase, abort_flag, p.status, DEV_TIMEOUT_MMA);
          MOE_TADD(2);
          if (!r_ok) {
            ok = false;
            break;
          }
          tc_fence_after();
#ifdef MOE_TRACE
          const long long _ti = clock64();
#endif
          const uint32_t a_addr = smem_base + stage * STAGE_BYTES;
          const uint64_t a_desc = smem_desc_sw128(a_addr);
          const uint64_t b_desc = smem_desc_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (ks | kk) != 0);
          tc_commit(smem_u32(&tail->empty[stage]));
#ifdef MOE_TRACE
          atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][1],
                    static_cast<unsigned long long>(clock64() - _ti));
#endif
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
      const long long t0 = cycles_now();
      while (!mbar_try_wait(smem_u32(&tail->drain), 0)) {
        if (cycles_now() - t0 > kWaitLimitCycles) {
          atomicExch(p.status, DEV_TIMEOUT_DRAIN);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp >= CONV_WARP0) {
    // ---------------------------------------------------------- converter --
    if (CONV != CONV_NONE) {
      const int ctid = threadIdx.x - CONV_WARP0 * 32;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const Tile t = decode_tile(p, tile);
        if (!t.valid) continue;
        for (int ks = 0; ks < t.nk; ++ks) {
          int got = 1;
          if (lane == 0)
            got = mbar_wait_bounded(smem_u32(&tail->full[stage]), phase, abort_flag, p.status,
                                    DEV_TIMEOUT_CONVERTER);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          convert_tile_bf16_to_f16(smem_base + stage * STAGE_BYTES, ctid);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tail->conv[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int ew = warp - EPI_WARP0;      // 0..3
    uint8_t *my_stage = epi_stage + ew * (16 * 64);
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = decode_tile(p, tile);
      if (!t.valid) continue;
      int got = 1;
      if (lane == 0) {
        MOE_T0();
        got = mbar_wait_bounded(smem_u32(&tail->tmem_full[acc]), aphase, abort_flag, p.status,
                                DEV_TIMEOUT_EPILOGUE);
        if (ew == 0) MOE_TADD(4);
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      // Agree across the four epilogue warps before any named barrier.
      if (lane == 0) tail->vote[ew] = got;
      named_bar_sync(1, 128);
      const int all_ok = tail->vote[0] & tail->vote[1] & tail->vote[2] & tail->vote[3];
      named_bar_sync(1, 128);
      if (!all_ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
#ifdef MOE_TRACE
      const long long _te = clock64();
#endif

      if (p.mode == MODE_GATEUP) {
        // Lanes 0..63 of the accumulator hold gate rows, 64..127 the matching
        // up rows.  Warp quarter q<2 (gate) pairs with quarter q+2 (up); the
        // gate warp finishes columns 0..7 of each 16-column chunk, the up warp
        // columns 8..15.
        const bool is_gate = q < 2;
        const int pair = q & 1;
        __half *hout = reinterpret_cast<__half *>(p.out) + t.m * 64 + pair * 32;
        __half *sh = reinterpret_cast<__half *>(my_stage);
        int buf = 0;
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          float *mine_to = xch + ((buf * 2 + pair) * 2 + (is_gate ? 0 : 1)) * 256;
          const float *from = xch + ((buf * 2 + pair) * 2 + (is_gate ? 1 : 0)) * 256;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            mine_to[cc * 32 + lane] = __uint_as_float(r[is_gate ? 8 + cc : cc]);
          named_bar_sync(1, 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const float g = is_gate ? __uint_as_float(r[cc]) : from[cc * 32 + lane];
            const float u = is_gate ? from[cc * 32 + lane] : __uint_as_float(r[8 + cc]);
            sh[cc * 32 + lane] = __float2half_rn(silu_f(g) * u);
          }
          __syncwarp();
          const int col0 = c0 + (is_gate ? 0 : 8);
          warp_store_rows_f16(my_stage, 8, t.nrows - col0,
                              hout + static_cast<size_t>(t.row0 + col0) * p.out_ld, p.out_ld, lane);
          __syncwarp();
          buf ^= 1;
        }
      } else if (p.mode == MODE_DOWN) {
        const int n0 = t.m * BM + q * 32;
        __half *oout = reinterpret_cast<__half *>(p.out) + n0;
        __half *sh = reinterpret_cast<__half *>(my_stage);
        const bool full_rows = n0 + 32 <= p.hidden;
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (full_rows) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) sh[cc * 32 + lane] = __float2half_rn(__uint_as_float(r[cc]));
            __syncwarp();
            warp_store_rows_f16(my_stage, 16, t.nrows - c0,
                                oout + static_cast<size_t>(t.row0 + c0) * p.out_ld, p.out_ld, lane);
            __syncwarp();
          } else if (n0 + lane < p.hidden) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if (c0 + cc < t.nrows)
                oout[static_cast<size_t>(t.row0 + c0 + cc) * p.out_ld + lane] =
                    __float2half_rn(__uint_as_float(r[cc]));
          }
        }
      } else {  // MODE_ROUTER: fp32 logits, 128 contiguous bytes per column
        const int e = t.m * BM + q * 32 + lane;
        float *lout = reinterpret_cast<float *>(p.out);
        const float bias = (p.bias != nullptr && e < p.n_experts) ? __ldg(p.bias + e) : 0.0f;
        for (int c0 = 0; c0 < t.nmma; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (e < p.n_experts) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if (c0 + cc < t.nrows)
                lout[static_cast<size_t>(t.row0 + c0 + cc) * p.out_ld + e] =
                    __uint_as_float(r[cc]) + bias;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
#ifdef MOE_TRACE
      if (lane == 0 && ew == 0)
        atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][5],
                  static_cast<unsigned long long>(clock64() - _te));
#endif
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
#ifdef MOE_TRACE
  if (threadIdx.x == 0) {
    atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][6],
              static_cast<unsigned long long>(clock64() - t_kernel0));
    atomicAdd(&g_moe_trace[p.mode][blockIdx.x & 1023][7], 1ull);
  }
#endif
  if (warp == MMA_WARP) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int CONV>
static constexpr int gemm_threads() {
  return BASE_THREADS + (CONV != CONV_NONE ? CONV_THREADS : 0);
}

cudaError_t gemm_configure() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<CONV_NONE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kGemmSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_gemm_kernel<CONV_BF16_TO_F16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kGemmSmemBytes));
}

cudaError_t launch_tc_gemm(const CUtensorMap &a_routed, const CUtensorMap &a_shared,
                           const GemmParams &p, int conv, int grid, cudaStream_t stream) {
  if (conv == CONV_BF16_TO_F16)
    tc_gemm_kernel<CONV_BF16_TO_F16>
        <<<grid, gemm_threads<CONV_BF16_TO_F16>(), kGemmSmemBytes, stream>>>(a_routed, a_shared, p);
  else
    tc_gemm_kernel<CONV_NONE>
        <<<grid, gemm_threads<CONV_NONE>(), kGemmSmemBytes, stream>>>(a_routed, a_shared, p);
  return cudaGetLastError();
}

}  // namespace moe

#ifdef MOE_TRACE
extern "C" int moe_debug_read_trace(void *dst, size_t bytes, int clear) {
  size_t n = bytes < sizeof(moe::g_moe_trace) ? bytes : sizeof(moe::g_moe_trace);
  if (cudaMemcpyFromSymbol(dst, moe::g_moe_trace, n) != cudaSuccess) return 1;
  if (clear) {
    static unsigned long long zeros[3][1024][16];
    if (cudaMemcpyToSymbol(moe::g_moe_trace, zeros, sizeof(zeros)) != cudaSuccess) return 2;
  }
  return 0;
}
#endif
