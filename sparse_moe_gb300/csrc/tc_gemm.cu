// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM)
// for the prefill path:
//
//   router:  l[t, e]  = sum_h x[t,h] Wr[e,h] (+ b[e])              -> fp32
//   gate/up: h[p, i]  = silu(sum_h xg[p,h] Wg[e,i,h]) *
//                       sum_h xg[p,h] Wu[e,i,h]                     -> fp16
//   down:    o[p, n]  = sum_i h[p,i] Wd[e,n,i]                      -> fp16
//
// where p runs over the rows routed to expert e in grouped order and xg is x
// in that order (written by the routing's placement kernel).
// (Sections "Dequantize weights during matrix multiplication", "Keep expert
// routing on the GPU" and "Match tile size to expert load" of "Optimizing
// On-Device Inference for Apple Silicon": grouped GEMM over the rows routed
// to each expert, fp32 accumulation, tile shape from the expert's row count.)
//
// Design (GB300-first, not the page's Metal design):
//  * a pair of CTAs on two SMs (a cluster of 2) runs one 256 x N tile with
//    tcgen05.mma.cta_group::2: weights on the MMA M side (each CTA stages its
//    own 128 rows) and the routed token rows on the N side (each CTA stages
//    half of them), so every SM takes in up to 32 KB per 64-deep k-step for
//    2 x 128 x N x 64 multiply-adds.  N is the block's row count rounded up
//    to 32 (at most 256): an expert with 5 rows runs a 256x32 MMA, not a
//    padded 256-row token tile;
//  * both operands come by TMA with 128-byte swizzle.  Each CTA's share of a
//    stage is one weight box (the gate/up tile as a 3-D box that stacks 64
//    gate rows over the matching 64 up rows, so one MMA yields both halves of
//    64 SwiGLU outputs) and one or two token-row boxes of 16..128 rows chosen
//    from the block's size, all consecutive rows: x for the router and the
//    shared expert, x in grouped order for the routed gate/up tiles, h (in
//    grouped order) for the down projection;
//  * two producer threads fill alternate stages.  (Measured on GB300 with
//    every SM streaming from L2: one thread issuing one 16 KB box per stage
//    moves about 23-28 bytes/clock per SM whatever the pipeline depth; two
//    threads issuing 32 KB stages move about 78.  The tiles need about 64 at
//    the tensor cores' full rate.  cp.async gathers of scattered rows reach
//    about 28 and TMA gather4 about 3, which is why the gate/up token rows
//    are read from a grouped copy of x rather than gathered.  A version
//    whose own gather warps copied the rows from x with cp.async measured
//    slower: gate/up 217 against 167 us at T=4096.)
//  * the pair's CTAs walk the device-built tile list persistently; one thread
//    of the leader issues the MMAs once both CTAs' stage is ready.  Without a
//    conversion (router, bf16 gate/up, down on fp16 weights) both CTAs' boxes
//    complete on the leader's full barrier (cta_group::2 loads), so readiness
//    needs no relay; when the weight tile must be converted first (int4
//    codes, or bf16 down weights without fp16 copies), a team of four
//    converter warps per k-step arrives on the leader's ready barrier;
//    epilogue warps (two groups of four without a conversion) drain the
//    double-buffered TMEM accumulator while the next tile computes, and
//    transpose each 32x16 piece through shared memory so global stores are
//    16-byte vectors;
//  * the down projection runs with fp16 operands: the gate/up epilogue stores
//    h in fp16 (11 significant bits instead of bf16's 8), and bf16 weight
//    tiles are turned into fp16 in place in shared memory before the MMA
//    reads them (exact for |w| >= 2^-17; the swizzled layout is unchanged
//    since both types are 2 bytes) unless the caller supplies fp16 copies.
//    o is stored in fp16.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <algorithm>

namespace moe {

constexpr int BM = 128;                 // A rows per CTA (MMA M = 256 per pair)
constexpr int PAIR_M = 2 * BM;
constexpr int BK = 64;                  // K per k-step (128-byte rows): one half of a stage
constexpr int HALVES = 2;               // k-steps per pipeline stage
constexpr int BN_MAX = kBlockRowsMax;   // max MMA N (tokens per tile)
constexpr int BN_HALF = BN_MAX / 2;     // token rows staged per CTA
constexpr int STAGES = 3;               // pipeline stages of HALVES k-steps each
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN_HALF * BK * 2;       // 16 KB
constexpr int SLOT_BYTES = A_BYTES + B_BYTES;   // 32 KB: one k-step (A, then B)
constexpr int STAGE_BYTES = HALVES * SLOT_BYTES;
// int4 weights: a k-step's packed codes (BM rows x BK/2 bytes) land in a ring
// of their own, from which the converter warps expand them into the stage.
constexpr int A_CODE_BYTES = BM * BK / 2;       // 4 KB: one k-step's int4 codes
constexpr int kCodeSlots = 4;                   // int4 code ring (ahead of the stages)
constexpr int ACC_COLS = 256;                   // one accumulator buffer
constexpr int TMEM_COLS = 512;                  // two buffers
// Warp roles (identical in both CTAs of a pair).
constexpr int kProducers = 2;                   // warps 0, 1: stage producers (lane 0)
constexpr int CODE_WARP = 2;                    // int4 code ring producer (lane 0)
constexpr int MMA_WARP = 3;
constexpr int EPI_WARP0 = 4;                    // epilogue groups of four warps from warp 4
constexpr int FIN_WARPS = 8;                    // converters (after the epilogue warps)
constexpr int XCH_FLOATS = 2 * 2 * 2 * 8 * 32;  // per group: [buf][pair][dir][8 cols][32 lanes]
constexpr int EPI_WARP_STAGE_BYTES = 16 * 64;   // per epilogue warp: 16 rows x 64 bytes
static_assert(EPI_WARP0 % 4 == 0, "epilogue warp q reads TMEM lanes 32 q .. 32 q + 31");

// Epilogue groups: four warps (one per TMEM lane quarter) each; group g
// drains the 16-column chunks g, g + G, g + 2G, ... of a tile.  Without a
// conversion the converter warps are not needed and a second group takes
// their place (the epilogue of a 256-column gate/up tile otherwise takes
// longer than the tile's MMAs).
template <int CONV> __host__ __device__ constexpr int epi_groups() { return CONV == CONV_NONE ? 2 : 1; }
template <int CONV> __host__ __device__ constexpr int fin_warp0() {
  return EPI_WARP0 + 4 * epi_groups<CONV>();
}
template <int CONV> __host__ __device__ constexpr int num_threads() {
  return (fin_warp0<CONV>() + (CONV == CONV_NONE ? 0 : FIN_WARPS)) * 32;
}

// Warps that convert one stage's weight tiles, per CTA: kInt4Warps converter
// warps per k-step, each handling kInt4Batches batches of 32 weight rows (int4:
// expanding codes from the ring; bf16 -> fp16: converting the landed tile in
// place).  The converters form kInt4Groups = HALVES teams: team h takes half
// h of every stage.  Measured at T=4096 (int4): four warps of 32 rows per
// k-step beat two of 64 rows by 20 %.
//
// A team's next k-step is in the next stage; its parity waits on the stage
// and code-ring barriers stay unambiguous only if no team can reach a barrier
// phase two ahead of the completed one: every ring slot belongs to one team
// (kCodeSlots a multiple of HALVES, ring slot = half-slot counter % kCodeSlots)
// and a team waits for a stage's release before each use.
constexpr int kInt4Warps = 4;
constexpr int kInt4Batches = (BM / 32) / kInt4Warps;
constexpr int kInt4Groups = FIN_WARPS / kInt4Warps;
static_assert(kInt4Warps * kInt4Batches * 32 == BM && kInt4Groups * kInt4Warps == FIN_WARPS,
              "converter teams");
static_assert(kInt4Groups == HALVES && kCodeSlots % HALVES == 0,
              "converter teams must not alias barrier phases");
template <int CONV> __host__ __device__ constexpr int conv_team() {
  return CONV == CONV_NONE ? 1 : HALVES * kInt4Warps;
}

struct SmemTail {
  uint64_t full[STAGES];        // unconverted: leader's, both CTAs' boxes; else local (A + B or B)
  uint64_t cfull[kCodeSlots];   // local, int4: a k-step's weight codes landed in the ring (TMA)
  uint64_t cempty[kCodeSlots];  // local, int4: the k-step's converters hold their codes
  uint64_t ready[STAGES];       // leader: both CTAs' converter teams (both halves)
  uint64_t empty[STAGES];       // local: arrives from the leader's commit
  uint64_t tmem_full[2];        // local: arrives from the leader's commit
  uint64_t tmem_empty[2];       // leader: every epilogue warp of both CTAs
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vote[8];
};

// Shared memory: the stages, the epilogue groups' exchange buffers and
// staging rows, the barriers, and (int4) the code ring.
template <int CONV> __host__ __device__ constexpr size_t gemm_smem_bytes() {
  return 1024 /*align slack*/ + STAGES * STAGE_BYTES +
         epi_groups<CONV>() * (XCH_FLOATS * sizeof(float) + 4 * EPI_WARP_STAGE_BYTES) +
         sizeof(SmemTail) + (conv_int4(CONV) ? 128 /*ring alignment*/ + kCodeSlots * A_CODE_BYTES : 0);
}
static_assert(gemm_smem_bytes<CONV_NONE>() <= 227 * 1024 &&
                  gemm_smem_bytes<CONV_INT4_TO_BF16>() <= 227 * 1024 &&
                  gemm_smem_bytes<CONV_BF16_TO_F16>() <= 227 * 1024,
              "shared memory per CTA");

struct Tile {
  int valid;
  int row0, nrows, nmma;
  int nk;              // k-steps (of BK)
  int ns;              // pipeline stages (HALVES k-steps each; the last may hold one)
  int k0;              // first k-step (router split-K: split * nk)
  int split;           // router split-K part of this tile
  int m;
  int e;               // expert (E: the shared expert; router: 0)
  int shared;
  int a_row, a_row2;   // this CTA's first A row (a_row2: first up row for gate/up)
  int a_valid_rows;    // this CTA's A rows at or beyond this index are not outputs
  int out_base;        // first output row (gate/up: i, down: n, router: e) of this CTA
  int out_limit;       // number of valid output rows of the operator (I/Is, H, E)
};

// The block-list entry of a grouped tile (zeros for the router, whose tiles
// need none, and past the last tile).  Each role loads the entry of its next
// tile while it works on the current one, so that decoding a tile never waits
// for a global load (about 800 cycles at the top of every tile in the
// MMA-issuing thread otherwise).
__device__ __forceinline__ int4 load_tile_block(const GemmParams &p, int tile, int ntiles) {
  if (p.mode == MODE_ROUTER || tile >= ntiles) return make_int4(0, 0, 0, 0);
  return p.blocks[tile / p.m_tiles];
}

__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int tile, int rank, int4 blk) {
  Tile t;
  t.k0 = 0;
  t.split = 0;
  if (p.mode == MODE_ROUTER) {   // router tiles: (block, m, split), split fastest
    t.split = tile % p.k_split;
    tile /= p.k_split;
  }
  const int b = tile / p.m_tiles;
  t.m = tile - b * p.m_tiles;
  int e = 0;
  if (p.mode == MODE_ROUTER) {
    t.row0 = b * p.block_rows;
    t.nrows = min(p.block_rows, p.T - t.row0);
    t.shared = 0;
  } else {
    e = blk.x;
    t.row0 = blk.y;
    t.nrows = blk.z;
    t.shared = (e == p.n_experts);
  }
  t.e = e;
  t.nmma = p.fixed_n && p.mode != MODE_ROUTER ? BN_MAX : max(32, (t.nrows + 31) & ~31);
  t.valid = t.nrows > 0;
  if (p.mode == MODE_ROUTER) {
    t.nk = p.k_routed / BK / p.k_split;
    t.k0 = t.split * t.nk;
    t.out_base = t.m * PAIR_M + rank * BM;
    t.out_limit = p.n_experts;
    t.a_row = t.out_base;
    t.a_row2 = 0;
  } else if (p.mode == MODE_GATEUP) {
    const int inter = t.shared ? p.inter_shared : p.inter_routed;
    t.nk = p.k_routed / BK;
    t.valid = t.valid && (t.m * 128 < inter);
    t.out_base = t.m * 128 + rank * 64;     // 64 SwiGLU outputs per CTA
    t.out_limit = inter;
    const int base = t.shared ? 0 : e * 2 * p.inter_routed;
    t.a_row = base + t.out_base;
    t.a_row2 = base + inter + t.out_base;
  } else {  // MODE_DOWN
    t.nk = (t.shared ? p.inter_shared : p.inter_routed) / BK;
    t.out_base = t.m * PAIR_M + rank * BM;
    t.out_limit = p.hidden;
    t.a_row = (t.shared ? 0 : e * p.hidden) + t.out_base;
    t.a_row2 = 0;
  }
  t.a_valid_rows = t.out_limit - t.out_base;
  t.ns = (t.nk + HALVES - 1) / HALVES;
  return t;
}

__device__ __forceinline__ int num_tiles(const GemmParams &p) {
  if (p.mode == MODE_ROUTER) return p.n_blocks_host * p.m_tiles * p.k_split;
  return *p.n_blocks_dev * p.m_tiles;
}

// The token-row boxes of one CTA's share of a stage: `rows` (a multiple of
// 16, at most BN_HALF) rows as at most two boxes of 16 << i rows (map i of
// the GemmMaps row-box sets), covering them with at most 16 rows to spare.
struct BBoxes {
  int n;
  int map[2];
  int rows[2];
};
__device__ __forceinline__ BBoxes b_boxes(int rows) {
  BBoxes b;
  const int u = rows >> 4;   // 1 .. 8
  if (u >= 7) {
    b.n = 1; b.map[0] = 3; b.rows[0] = 128;
  } else if (u == 5 || u == 6) {
    b.n = 2; b.map[0] = 2; b.rows[0] = 64; b.map[1] = u - 5; b.rows[1] = 16 << (u - 5);
  } else if (u == 4) {
    b.n = 1; b.map[0] = 2; b.rows[0] = 64;
  } else if (u == 3) {
    b.n = 2; b.map[0] = 1; b.rows[0] = 32; b.map[1] = 0; b.rows[1] = 16;
  } else {
    b.n = 1; b.map[0] = u - 1; b.rows[0] = 16 * u;
  }
  b.map[1] = b.n > 1 ? b.map[1] : 0;
  b.rows[1] = b.n > 1 ? b.rows[1] : 0;
  return b;
}

// Conversion, two values per 32-bit word: with u = q + 8 in [0, 15], the
// 16-bit pattern M | u is the number M + u exactly (M = 1024.0 for fp16,
// 128.0 for bf16, both with unit spacing there), so one packed subtract of
// M + 8 gives q exactly and one packed multiply by the scale rounds q * s
// once -- the same value as rounding the exact product (exact in fp16: q * s
// has at most 11 significant bits).
template <bool F16>
__device__ __forceinline__ uint32_t dq_pair(uint32_t lo_nib, uint32_t hi_nib, int h,
                                            uint32_t s2) {
  // result byte 0 <- byte h of lo_nib, byte 2 <- byte h of hi_nib (selector
  // nibbles 0 and 2; bytes 1 and 3 are masked off)
  const uint32_t sel = static_cast<uint32_t>(h) | (static_cast<uint32_t>(h + 4) << 8);
  const uint32_t b = __byte_perm(lo_nib, hi_nib, sel) & 0x00FF00FFu;
  const uint32_t v = b | (F16 ? 0x64006400u : 0x43004300u);
  uint32_t r;
  if constexpr (F16) {
    asm("{\n .reg .b32 t;\n sub.f16x2 t, %1, %2;\n mul.f16x2 %0, t, %3;\n}"
        : "=r"(r)
        : "r"(v), "r"(0x64086408u), "r"(s2));
  } else {
    asm("{\n .reg .b32 t;\n sub.rn.bf16x2 t, %1, %2;\n mul.rn.bf16x2 %0, t, %3;\n}"
        : "=r"(r)
        : "r"(v), "r"(0x43084308u), "r"(s2));
  }
  return r;
}

// Affine codes, two values per 32-bit word: with u in [0, 15] the pattern
// M | u is M + u exactly, so one packed subtract of M gives u and one packed
// fma u * s + b rounds the weight once.
template <bool F16>
__device__ __forceinline__ uint32_t dq_pair_affine(uint32_t lo_nib, uint32_t hi_nib, int h,
                                                   uint32_t s2, uint32_t b2) {
  const uint32_t sel = static_cast<uint32_t>(h) | (static_cast<uint32_t>(h + 4) << 8);
  const uint32_t b = __byte_perm(lo_nib, hi_nib, sel) & 0x00FF00FFu;
  const uint32_t v = b | (F16 ? 0x64006400u : 0x43004300u);
  uint32_t r;
  if constexpr (F16) {
    asm("{\n .reg .b32 t;\n sub.f16x2 t, %1, %2;\n fma.rn.f16x2 %0, t, %3, %4;\n}"
        : "=r"(r)
        : "r"(v), "r"(0x64006400u), "r"(s2), "r"(b2));
  } else {
    asm("{\n .reg .b32 t;\n sub.rn.bf16x2 t, %1, %2;\n fma.rn.bf16x2 %0, t, %3, %4;\n}"
        : "=r"(r)
        : "r"(v), "r"(0x43004300u), "r"(s2), "r"(b2));
  }
  return r;
}

// Dequantisation of rows 32 j .. 32 j + 31 of one stage's A tile by one
// warp.  Row r's int4 codes (32 bytes = 64 K values, element 2m in the low
// nibble of byte m) sit at codes + 32 r in a slot of the code ring; they
// become q * s_r (+ b_r) in bf16 (or fp16) in the 128-byte-swizzled K-major
// layout the MMA reads.  Lane l handles 16-byte chunk l % 8 (K values
// 8 (l % 8) .. +7) of rows 32 j + 4 m + l / 8, m = 0..7: load_codes_int4
// reads its 8 code words, expand_rows_int4 writes the outputs, bytes
// [4096 j, 4096 j + 4096) of the tile.
__device__ __forceinline__ void load_codes_int4(uint32_t codes, int j, int lane,
                                                uint32_t (&w)[8]) {
  const uint32_t code0 = codes + 1024 * j + (lane >> 3) * 32 + (lane & 7) * 4;
#pragma unroll
  for (int m = 0; m < 8; ++m)
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[m]) : "r"(code0 + 128 * m));
}

// s_lane, b_lane: the scale (and affine bias) of row 32 j + lane.
template <bool F16, bool AFF>
__device__ __forceinline__ void expand_rows_int4(uint32_t tile, const uint32_t (&w)[8], int j,
                                                 float s_lane, float b_lane, int lane) {
  const int c = lane & 7, rs = lane >> 3;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int r = 32 * j + 4 * m + rs;
    // the row's scale (held by lane 4 m + l / 8) as a packed pair
    const float sv = __shfl_sync(0xffffffffu, s_lane, 4 * m + rs);
    uint32_t s2;
    if constexpr (F16) asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(s2) : "f"(sv));
    else asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(s2) : "f"(sv));
    uint32_t o[4];
    if constexpr (AFF) {
      const float bv = __shfl_sync(0xffffffffu, b_lane, 4 * m + rs);
      uint32_t b2;
      if constexpr (F16) asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(b2) : "f"(bv));
      else asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(b2) : "f"(bv));
      const uint32_t lo = w[m] & 0x0F0F0F0Fu;           // elements 0, 2, 4, 6
      const uint32_t hi = (w[m] >> 4) & 0x0F0F0F0Fu;    // elements 1, 3, 5, 7
#pragma unroll
      for (int h = 0; h < 4; ++h) o[h] = dq_pair_affine<F16>(lo, hi, h, s2, b2);
    } else {
      const uint32_t lo = (w[m] & 0x0F0F0F0Fu) ^ 0x08080808u;          // elements 0, 2, 4, 6
      const uint32_t hi = ((w[m] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // elements 1, 3, 5, 7
#pragma unroll
      for (int h = 0; h < 4; ++h) o[h] = dq_pair<F16>(lo, hi, h, s2);
    }
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(tile + r * 128 + ((c ^ (r & 7)) << 4)),
                 "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                 : "memory");
  }
}

// Converter q's share of the in-place bf16 -> fp16 conversion of one stage's
// A tile: rows 32 q .. 32 q + 31 (4 KB, 16-byte chunks q * 256 + lane + 32 m).
__device__ __forceinline__ void convert_rows_bf16_to_f16(uint32_t tile, int q, int lane) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint32_t addr = tile + (q * 256 + lane + 32 * m) * 16;
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

// Scale rows (int4) of A rows 32 j + lane of a tile; rows past the
// operator's end get -1 (scale 0).
__device__ __forceinline__ void tile_scale_rows(const GemmParams &p, const Tile &t, int lane,
                                                int (&srow)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 32 * j + lane;
    if (p.mode == MODE_GATEUP) {
      const int rr = r & 63;
      srow[j] = rr < t.a_valid_rows ? ((r < 64) ? t.a_row : t.a_row2) + rr : -1;
    } else {
      srow[j] = r < t.a_valid_rows ? t.a_row + r : -1;
    }
  }
}

// int4: the scale (and affine bias) of this k-step for A row 32 j + lane (0
// past the operator's end).
template <bool AFF>
__device__ __forceinline__ void load_row_scale(const GemmParams &p, const Tile &t, int ks, int j,
                                               int lane, float &sv, float &bv) {
  int srow[4];
  tile_scale_rows(p, t, lane, srow);
  int row = srow[0];
#pragma unroll
  for (int q = 1; q < 4; ++q)
    if (j == q) row = srow[q];
  const __nv_bfloat16 *sbase =
      static_cast<const __nv_bfloat16 *>(t.shared ? p.a_scale_shared : p.a_scale_routed);
  const __nv_bfloat16 *bbase =
      static_cast<const __nv_bfloat16 *>(t.shared ? p.a_bias_shared : p.a_bias_routed);
  const size_t off = static_cast<size_t>(row) * t.nk + ks;
  sv = row >= 0 ? __bfloat162float(__ldg(sbase + off)) : 0.0f;
  bv = 0.0f;
  if constexpr (AFF) bv = row >= 0 ? __bfloat162float(__ldg(bbase + off)) : 0.0f;
}

// Arrival of one converting warp on the pair leader's ready barrier of
// `stage` (after its writes are fenced for the tensor core).
__device__ __forceinline__ void arrive_ready(SmemTail *tail, int stage, int rank) {
  const uint32_t ready = smem_u32(&tail->ready[stage]);
  if (rank == 0) mbar_arrive(ready);
  else mbar_arrive_cluster(mapa_shared(ready, 0));
}

// Where converter work sits in the pipeline: stage counter st (stage st %
// STAGES, phase (st / STAGES) & 1), half h of the stage (k-step slot
// (st % STAGES) * HALVES + h of the shared memory), and the half-slot counter
// hs = HALVES * st + h (int4 code ring slot hs % kCodeSlots, phase
// (hs / kCodeSlots) & 1).  `real`: the tile has a k-step in this half (the
// second half of a tile's last stage is empty when its k-step count is odd;
// the converters still take part in its barriers, so that every phase sees
// the same arrivals).
struct ConvPos {
  int st, h, hs;
  bool real;
};

// bf16 -> fp16 converter q of one half-stage: a bounded wait for the stage's
// boxes (weights and token rows) to land in this CTA, its 32 rows converted
// in place, and its arrival on the pair leader's ready barrier.  Returns false
// on a timeout or abort.
__device__ __forceinline__ bool convert_stage_bf16(const GemmParams &p, int q, const ConvPos &c,
                                                   int rank, uint32_t smem_base, SmemTail *tail,
                                                   volatile int *abort_flag, int lane) {
  const int stage = c.st % STAGES;
  const uint32_t phase = static_cast<uint32_t>(c.st / STAGES) & 1u;
  int got = 1;
  if (lane == 0)
    got = mbar_wait_bounded(smem_u32(&tail->full[stage]), phase, abort_flag, p.status,
                            DEV_TIMEOUT_CONVERTER);
  if (!__shfl_sync(0xffffffffu, got, 0)) return false;
  if (c.real) {
    convert_rows_bf16_to_f16(smem_base + (stage * HALVES + c.h) * SLOT_BYTES, q, lane);
    fence_proxy_async_smem();
  }
  __syncwarp();
  if (lane == 0) arrive_ready(tail, stage, rank);
  return true;
}

// int4 converter q (0 .. kInt4Warps - 1) of one half-stage: takes its codes
// (batches q * kInt4Batches + b) from the ring as soon as they land and frees
// its share of the slot, waits until the MMA has released the stage, expands
// its weight rows into the half's A region, and arrives on the pair leader's
// ready barrier (the last converter only after the stage's token rows have
// landed).  sv, bv: this lane's row scales and biases, one per batch, loaded
// by the caller before the waits.  Returns false on a timeout or abort.
template <int CONV>
__device__ __forceinline__ bool convert_stage_int4(const GemmParams &p, int q,
                                                   const float (&sv)[kInt4Batches],
                                                   const float (&bv)[kInt4Batches],
                                                   const ConvPos &c, int rank, uint32_t smem_base,
                                                   uint32_t code_ring, SmemTail *tail,
                                                   volatile int *abort_flag, int lane) {
  const int stage = c.st % STAGES, slot = c.hs % kCodeSlots;
  const uint32_t sph = static_cast<uint32_t>(c.st / STAGES) & 1u;
  const uint32_t cph = static_cast<uint32_t>(c.hs / kCodeSlots) & 1u;
  const uint32_t tile = smem_base + (stage * HALVES + c.h) * SLOT_BYTES;
  int got = 1;
  if (lane == 0)
    got = mbar_wait_bounded(smem_u32(&tail->cfull[slot]), cph, abort_flag, p.status,
                            DEV_TIMEOUT_CONVERTER);
  if (!__shfl_sync(0xffffffffu, got, 0)) return false;
  uint32_t w[kInt4Batches][8];
  if (c.real) {
#pragma unroll
    for (int b = 0; b < kInt4Batches; ++b)
      load_codes_int4(code_ring + slot * A_CODE_BYTES, q * kInt4Batches + b, lane, w[b]);
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(smem_u32(&tail->cempty[slot]));
    got = mbar_wait_bounded(smem_u32(&tail->empty[stage]), sph ^ 1, abort_flag, p.status,
                            DEV_TIMEOUT_CONVERTER);
  }
  if (!__shfl_sync(0xffffffffu, got, 0)) return false;
  if (c.real) {
#pragma unroll
    for (int b = 0; b < kInt4Batches; ++b)
      expand_rows_int4<conv_to_f16(CONV), conv_affine(CONV)>(tile, w[b], q * kInt4Batches + b,
                                                             sv[b], bv[b], lane);
    fence_proxy_async_smem();
  }
  __syncwarp();
  if (lane == 0) {
    // one converter per CTA and half checks the token rows: the leader's
    // ready phase needs every converter's arrival
    if (q == kInt4Warps - 1)
      got = mbar_wait_bounded(smem_u32(&tail->full[stage]), sph, abort_flag, p.status,
                              DEV_TIMEOUT_CONVERTER);
    if (got) arrive_ready(tail, stage, rank);
  }
  return __shfl_sync(0xffffffffu, got, 0) != 0;
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

// TMA descriptors of one grouped-GEMM launch: the weight tiles (routed
// experts, shared expert) and two sets of token-row maps whose boxes are
// 16, 32, 64 and 128 rows of 64 elements: b for the router (x), the routed
// gate/up tiles (x in grouped order) and the down projection (h); b2 for the
// shared expert's gate/up tiles (x).
struct GemmMaps {
  CUtensorMap a_routed, a_shared;
  CUtensorMap b[4], b2[4];
};

template <int CONV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(num_threads<CONV>(), 1)
    tc_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  constexpr int G = epi_groups<CONV>();
  constexpr int FIN_WARP0 = fin_warp0<CONV>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float *xch_all = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);   // [G][XCH_FLOATS]
  uint8_t *epi_stage = reinterpret_cast<uint8_t *>(xch_all + G * XCH_FLOATS);
  SmemTail *tail = reinterpret_cast<SmemTail *>(epi_stage + 4 * G * EPI_WARP_STAGE_BYTES);
  const uint32_t code_ring = (smem_u32(tail + 1) + 127u) & ~127u;   // int4: kCodeSlots x 4 KB
  volatile int *abort_flag = &tail->abort_flag;
  pdl_trigger();   // the next kernel may start its set-up as SMs free up

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  const uint32_t smem_base = smem_u32(smem);
  const int rank = static_cast<int>(cluster_ctarank());   // 0: leader, 1: peer
  const int pair_id = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // one arrival per phase: the stage producer's arrive.expect_tx (the
      // leader's, covering both CTAs' bytes, in the unconverted modes)
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->ready[s]), 2 * conv_team<CONV>());
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    for (int s = 0; s < kCodeSlots; ++s) {
      mbar_init(smem_u32(&tail->cfull[s]), 1);
      mbar_init(smem_u32(&tail->cempty[s]), kInt4Warps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tail->tmem_full[a]), 1);
      mbar_init(smem_u32(&tail->tmem_empty[a]), 2 * 4 * G);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp < kProducers && lane == 0) {
    prefetch_tensormap(&maps.a_routed);
    prefetch_tensormap(&maps.a_shared);
    for (int i = 0; i < 4; ++i) prefetch_tensormap(&maps.b[i]);
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(smem_u32(&tail->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  pdl_wait();   // inputs (block list, token rows) written by earlier kernels
  const uint32_t tmem_base = tail->tmem_base;
  const int ntiles = num_tiles(p);

  if (warp < kProducers) {
    // ------------------------------------------------- stage producers --
    // Lane 0 of producer warp pp fills the stages st with st % kProducers ==
    // pp (st counts this CTA's stages over all its tiles): it waits until the
    // MMA has released the stage, then issues this CTA's boxes for each of the
    // stage's k-steps: the weight box (unless the weights are int4 codes,
    // which come through the code ring) and the token-row boxes.  Unconverted
    // modes: both CTAs' boxes complete on the leader's full barrier, which
    // expects the pair's bytes (cta_group::2 loads).
    constexpr bool INT4 = conv_int4(CONV);
    const int pp = warp;
    int issued_parity[STAGES];
#pragma unroll
    for (int s2 = 0; s2 < STAGES; ++s2) issued_parity[s2] = -1;
    bool ok = true;
    if (lane == 0) {
      int st = 0;
      int4 blk = load_tile_block(p, pair_id, ntiles);
      for (int tile = pair_id; tile < ntiles && ok; tile += num_pairs) {
        const Tile t = decode_tile(p, tile, rank, blk);
        blk = load_tile_block(p, tile + num_pairs, ntiles);
        if (!t.valid) continue;
        const CUtensorMap *amap = t.shared ? &maps.a_shared : &maps.a_routed;
        const bool b_from_x = p.mode == MODE_GATEUP && t.shared;   // shared expert: x rows
        const CUtensorMap *bmaps = b_from_x ? maps.b2 : maps.b;
        const int half = t.nmma / 2;
        const BBoxes bb = b_boxes(half);
        const int b_row0 = (b_from_x ? t.row0 - p.shared_row0 : t.row0) + rank * half;
        const uint32_t b_bytes = static_cast<uint32_t>((bb.rows[0] + bb.rows[1]) * BK * 2);
        for (int j = 0; j < t.ns; ++j, ++st) {
          if (st % kProducers != pp) continue;
          const int stage = st % STAGES;
          const uint32_t phase = static_cast<uint32_t>(st / STAGES) & 1u;
          if (!mbar_wait_bounded(smem_u32(&tail->empty[stage]), phase ^ 1, abort_flag, p.status,
                                 DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const int nh = min(HALVES, t.nk - j * HALVES);   // k-steps in this stage
          const uint32_t full_bar = smem_u32(&tail->full[stage]);
          if constexpr (CONV == CONV_NONE) {
            const uint32_t lead_full = mapa_shared(full_bar, 0);
            if (rank == 0) mbar_arrive_expect_tx(full_bar, 2 * nh * (A_BYTES + b_bytes));
            for (int h = 0; h < nh; ++h) {
              const uint32_t a_dst = smem_base + (stage * HALVES + h) * SLOT_BYTES;
              const uint32_t b_dst = a_dst + A_BYTES;
              const int kx = (t.k0 + j * HALVES + h) * BK;
              if (p.mode == MODE_GATEUP)
                tma_load_3d_pair(a_dst, amap, kx, t.out_base, t.shared ? 0 : 2 * t.e, lead_full);
              else
                tma_load_2d_pair(a_dst, amap, kx, t.a_row, lead_full);
              tma_load_2d_pair(b_dst, &bmaps[bb.map[0]], kx, b_row0, lead_full);
              if (bb.n > 1)
                tma_load_2d_pair(b_dst + bb.rows[0] * 128, &bmaps[bb.map[1]], kx,
                                 b_row0 + bb.rows[0], lead_full);
            }
            // (the peer's boxes complete on the leader's barrier: the leader's
            // producers wait for them on abort)
            if (rank == 0) issued_parity[stage] = static_cast<int>(phase);
          } else {
            mbar_arrive_expect_tx(full_bar,
                                  nh * ((INT4 ? 0u : static_cast<uint32_t>(A_BYTES)) + b_bytes));
            for (int h = 0; h < nh; ++h) {
              const uint32_t a_dst = smem_base + (stage * HALVES + h) * SLOT_BYTES;
              const uint32_t b_dst = a_dst + A_BYTES;
              const int kx = (t.k0 + j * HALVES + h) * BK;
              if constexpr (!INT4) {
                if (p.mode == MODE_GATEUP)
                  tma_load_3d(a_dst, amap, kx, t.out_base, t.shared ? 0 : 2 * t.e, full_bar);
                else
                  tma_load_2d(a_dst, amap, kx, t.a_row, full_bar);
              }
              tma_load_2d(b_dst, &bmaps[bb.map[0]], kx, b_row0, full_bar);
              if (bb.n > 1)
                tma_load_2d(b_dst + bb.rows[0] * 128, &bmaps[bb.map[1]], kx, b_row0 + bb.rows[0],
                            full_bar);
            }
            issued_parity[stage] = static_cast<int>(phase);
          }
        }
      }
      if (!ok) {
        // Wait (bounded) for this thread's copies still in flight before the CTA exits.
        for (int s2 = 0; s2 < STAGES; ++s2)
          if (issued_parity[s2] >= 0) {
            const uint32_t bar = smem_u32(&tail->full[s2]);
            const long long t0 = cycles_now();
            while (!mbar_try_wait(bar, static_cast<uint32_t>(issued_parity[s2])) &&
                   cycles_now() - t0 < kWaitLimitCycles) {
            }
          }
      }
    }
    __syncwarp();
  } else if (warp == CODE_WARP) {
    // ------------------------------------------- int4 codes (code ring) --
    // Lane 0 loads each k-step's packed codes (128 rows x 32 bytes) into ring
    // slot hs % kCodeSlots (complete_tx on cfull; hs counts half-stages,
    // including the empty second half of a tile's last stage, whose slot phase
    // completes with a plain arrival), paced by the converters freeing slots,
    // not by the MMA.
    if (conv_int4(CONV) && lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      int issued_parity[kCodeSlots];
#pragma unroll
      for (int s2 = 0; s2 < kCodeSlots; ++s2) issued_parity[s2] = -1;
      bool ok = true;
      int4 blk = load_tile_block(p, pair_id, ntiles);
      for (int tile = pair_id; tile < ntiles && ok; tile += num_pairs) {
        const Tile t = decode_tile(p, tile, rank, blk);
        blk = load_tile_block(p, tile + num_pairs, ntiles);
        if (!t.valid) continue;
        const CUtensorMap *amap = t.shared ? &maps.a_shared : &maps.a_routed;
        for (int ks = 0; ks < t.ns * HALVES; ++ks) {
          if (!mbar_wait_bounded(smem_u32(&tail->cempty[slot]), phase ^ 1, abort_flag, p.status,
                                 DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t cfull_bar = smem_u32(&tail->cfull[slot]);
          if (ks < t.nk) {
            const uint32_t c_dst = code_ring + slot * A_CODE_BYTES;
            const int kx = (t.k0 + ks) * (BK / 2);
            mbar_arrive_expect_tx(cfull_bar, A_CODE_BYTES);
            if (p.mode == MODE_GATEUP) {
              tma_load_2d(c_dst, amap, kx, t.a_row, cfull_bar);
              tma_load_2d(c_dst + A_CODE_BYTES / 2, amap, kx, t.a_row2, cfull_bar);
            } else {
              tma_load_2d(c_dst, amap, kx, t.a_row, cfull_bar);
            }
            issued_parity[slot] = static_cast<int>(phase);
          } else {
            mbar_arrive(cfull_bar);   // an empty half: no codes
            issued_parity[slot] = -1;
          }
          if (++slot == kCodeSlots) {
            slot = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s2 = 0; s2 < kCodeSlots; ++s2)
          if (issued_parity[s2] >= 0) {
            const uint32_t bar = smem_u32(&tail->cfull[s2]);
            const long long t0 = cycles_now();
            while (!mbar_try_wait(bar, static_cast<uint32_t>(issued_parity[s2])) &&
                   cycles_now() - t0 < kWaitLimitCycles) {
            }
          }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (rank == 0) {
      // ----------------------------------------------- MMA issuer (leader) --
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t aphase = 0;
        bool ok = true;
        // descriptors of k-step slot 0 (A and B); slot s adds s * SLOT_BYTES
        // to the start-address field (addresses >> 4, 14 bits: no carry below
        // 256 KB)
        const uint64_t a_desc0 = smem_desc_sw128(smem_base);
        const uint64_t b_desc0 = smem_desc_sw128(smem_base + A_BYTES);
        int4 blk = load_tile_block(p, pair_id, ntiles);
        for (int tile = pair_id; tile < ntiles && ok; tile += num_pairs) {
          const Tile t = decode_tile(p, tile, 0, blk);
          blk = load_tile_block(p, tile + num_pairs, ntiles);
          if (!t.valid) continue;
          if (!mbar_wait_bounded_cluster(smem_u32(&tail->tmem_empty[acc]), aphase ^ 1, abort_flag,
                                         p.status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
          const bool f16 = conv_to_f16(CONV) || (CONV == CONV_NONE && p.ab_f16);
          const uint32_t idesc = f16 ? idesc_f16_f32(PAIR_M, t.nmma) : idesc_bf16_f32(PAIR_M, t.nmma);
          for (int j = 0; j < t.ns; ++j) {
            // unconverted modes: both CTAs' boxes complete on this CTA's full
            // barrier; otherwise the converter teams' ready barrier (CTA-scope
            // acquire, as the converters' arrivals are CTA-scope releases:
            // measured 2-3 % faster than a cluster-scope acquire).  One wait
            // per stage of HALVES k-steps: a barrier wait in the issuing thread
            // costs about as long as four MMAs of N = 256 (measured), so
            // waiting once per k-step held small tiles to a fraction of the
            // tensor cores' rate.
            const uint32_t stage_bar = CONV == CONV_NONE ? smem_u32(&tail->full[stage])
                                                         : smem_u32(&tail->ready[stage]);
            if (!mbar_wait_spin_bounded(stage_bar, phase, abort_flag, p.status, DEV_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int nh = min(HALVES, t.nk - j * HALVES);
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
              if (h < nh) {
                const uint64_t off = static_cast<uint64_t>((stage * HALVES + h) * (SLOT_BYTES >> 4));
                const uint64_t a_desc = a_desc0 + off, b_desc = b_desc0 + off;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                  tc_mma_pair(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                              (j | h | kk) != 0);
              }
            }
            tc_commit_pair_mc(smem_u32(&tail->empty[stage]), 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit_pair_mc(smem_u32(&tail->tmem_full[acc]), 0x3);
          if (++acc == 2) {
            acc = 0;
            aphase ^= 1;
          }
        }
        // All pair MMAs complete before TMEM is released or the peer exits.
        tc_commit_pair_mc(smem_u32(&tail->drain), 0x1);
        const long long t0 = cycles_now();
        while (!mbar_try_wait(smem_u32(&tail->drain), 0)) {
          if (cycles_now() - t0 > kWaitLimitCycles) {
            atomicExch(p.status, DEV_TIMEOUT_DRAIN);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= FIN_WARP0) {
    // ------------------------------------------------------- converters --
    // Team h (converters kInt4Warps h ..) takes half h of every stage.  int4:
    // each warp expands its share of the weight rows as soon as the codes land
    // and the stage is free, overlapping the token-row copies; the codes run
    // up to kCodeSlots k-steps ahead in their own ring.  bf16 -> fp16: each
    // warp converts its 32 rows once the stage's boxes have landed.  An empty
    // half (odd k-step count) only takes part in the barriers.  Unconverted
    // modes have no converter warps.
    const int f = warp - FIN_WARP0;
    const int h = f / kInt4Warps;
    const int q = f % kInt4Warps;
    int st = 0;
    bool ok = true;
    // int4: the row scales of the team's next k-step in the tile (ks +
    // HALVES) are loaded while this one converts (a global load's latency
    // would otherwise sit inside every expansion).
    float sv_next[kInt4Batches] = {}, bv_next[kInt4Batches] = {};
    bool have_next = false;
    int4 blk = load_tile_block(p, pair_id, ntiles);
    for (int tile = pair_id; tile < ntiles && ok; tile += num_pairs) {
      const Tile t = decode_tile(p, tile, rank, blk);
      blk = load_tile_block(p, tile + num_pairs, ntiles);
      if (!t.valid) continue;
      for (int jj = 0; jj < t.ns; ++jj, ++st) {
        const int ks = jj * HALVES + h;
        const ConvPos pos{st, h, HALVES * st + h, ks < t.nk};
        if constexpr (conv_int4(CONV)) {
          float sv[kInt4Batches], bv[kInt4Batches];
#pragma unroll
          for (int b = 0; b < kInt4Batches; ++b) {
            sv[b] = sv_next[b];
            bv[b] = bv_next[b];
            if (!have_next && pos.real)
              load_row_scale<conv_affine(CONV)>(p, t, ks, q * kInt4Batches + b, lane, sv[b], bv[b]);
          }
          have_next = ks + HALVES < t.nk;
          if (have_next) {
#pragma unroll
            for (int b = 0; b < kInt4Batches; ++b)
              load_row_scale<conv_affine(CONV)>(p, t, ks + HALVES, q * kInt4Batches + b, lane,
                                                sv_next[b], bv_next[b]);
          }
          ok = convert_stage_int4<CONV>(p, q, sv, bv, pos, rank, smem_base, code_ring, tail,
                                        abort_flag, lane);
        } else {
          ok = convert_stage_bf16(p, q, pos, rank, smem_base, tail, abort_flag, lane);
        }
        if (!ok) break;
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int ew = warp - EPI_WARP0;      // 0 .. 4 G - 1
    const int grp = ew >> 2;              // epilogue group: column chunks grp, grp + G, ...
    const int bar_id = 1 + grp;           // the group's named barrier (128 threads)
    float *xch = xch_all + grp * XCH_FLOATS;
    uint8_t *my_stage = epi_stage + ew * EPI_WARP_STAGE_BYTES;
    const uint32_t tmem_empty0 = mapa_shared(smem_u32(&tail->tmem_empty[0]), 0);
    int acc = 0;
    uint32_t aphase = 0;
    bool range_bad = false;   // a stored h or o value outside the fp16 range
    int4 blk = load_tile_block(p, pair_id, ntiles);
    for (int tile = pair_id; tile < ntiles; tile += num_pairs) {
      const Tile t = decode_tile(p, tile, rank, blk);
      blk = load_tile_block(p, tile + num_pairs, ntiles);
      if (!t.valid) continue;
      int got = 1;
      if (lane == 0) {
        got = mbar_wait_bounded(smem_u32(&tail->tmem_full[acc]), aphase, abort_flag, p.status,
                                DEV_TIMEOUT_EPILOGUE);
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      // Agree across the group's four warps before any named barrier.
      if (lane == 0) tail->vote[ew] = got;
      named_bar_sync(bar_id, 128);
      const int v0 = grp * 4;
      const int all_ok = tail->vote[v0] & tail->vote[v0 + 1] & tail->vote[v0 + 2] & tail->vote[v0 + 3];
      named_bar_sync(bar_id, 128);
      if (!all_ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);

      if (p.mode == MODE_GATEUP) {
        // Lanes 0..63 of this CTA's accumulator hold gate rows, 64..127 the
        // matching up rows.  Warp quarter q<2 (gate) pairs with quarter q+2
        // (up); the gate warp finishes columns 0..7 of each 16-column chunk,
        // the up warp columns 8..15.
        const bool is_gate = q < 2;
        const int pair = q & 1;
        const int i0 = t.out_base + pair * 32;
        const bool live = i0 < t.out_limit;        // whole 32-row group inside I
        __half *hout = reinterpret_cast<__half *>(p.out) + i0;
        __half *sh = reinterpret_cast<__half *>(my_stage);
        int buf = 0;
        for (int c0 = 16 * grp; c0 < t.nmma; c0 += 16 * G) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          float *mine_to = xch + ((buf * 2 + pair) * 2 + (is_gate ? 0 : 1)) * 256;
          const float *from = xch + ((buf * 2 + pair) * 2 + (is_gate ? 1 : 0)) * 256;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            mine_to[cc * 32 + lane] = __uint_as_float(r[is_gate ? 8 + cc : cc]);
          named_bar_sync(bar_id, 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const float g = is_gate ? __uint_as_float(r[cc]) : from[cc * 32 + lane];
            const float u = is_gate ? from[cc * 32 + lane] : __uint_as_float(r[8 + cc]);
            const float hv = silu_f(g) * u;
            // fp16 range check of the stored values (token columns that exist)
            range_bad |= live && (c0 + (is_gate ? 0 : 8) + cc < t.nrows) && !(fabsf(hv) <= 65504.0f);
            sh[cc * 32 + lane] = __float2half_rn(hv);
          }
          __syncwarp();
          const int col0 = c0 + (is_gate ? 0 : 8);
          if (live)
            warp_store_rows_f16(my_stage, 8, t.nrows - col0,
                                hout + static_cast<size_t>(t.row0 + col0) * p.out_ld, p.out_ld, lane);
          __syncwarp();
          buf ^= 1;
        }
      } else if (p.mode == MODE_DOWN) {
        const int n0 = t.out_base + q * 32;
        __half *oout = reinterpret_cast<__half *>(p.out) + n0;
        __half *sh = reinterpret_cast<__half *>(my_stage);
        const bool full_rows = n0 + 32 <= p.hidden;
        for (int c0 = 16 * grp; c0 < t.nmma; c0 += 16 * G) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (full_rows) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const float ov = __uint_as_float(r[cc]);
              range_bad |= (c0 + cc < t.nrows) && !(fabsf(ov) <= 65504.0f);
              sh[cc * 32 + lane] = __float2half_rn(ov);
            }
            __syncwarp();
            warp_store_rows_f16(my_stage, 16, t.nrows - c0,
                                oout + static_cast<size_t>(t.row0 + c0) * p.out_ld, p.out_ld, lane);
            __syncwarp();
          } else if (n0 + lane < p.hidden) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if (c0 + cc < t.nrows) {
                const float ov = __uint_as_float(r[cc]);
                range_bad |= !(fabsf(ov) <= 65504.0f);
                oout[static_cast<size_t>(t.row0 + c0 + cc) * p.out_ld + lane] = __float2half_rn(ov);
              }
          }
        }
      } else {  // MODE_ROUTER: fp32 logits (split-K part t.split), 128 contiguous bytes per column
        const int e0 = t.out_base + q * 32;   // the warp's 32 experts, one per lane
        const int e = e0 + lane;
        float *lout = reinterpret_cast<float *>(p.out) + t.split * p.out_split_stride;
        const float bias =
            (p.bias != nullptr && e < p.n_experts && t.split == 0) ? __ldg(p.bias + e) : 0.0f;
        // 8 tokens x 32 experts at a time through the warp's staging area,
        // then 16-byte stores: a quarter of the store instructions of one
        // 4-byte store per lane and token
        const bool vec = e0 + 32 <= p.n_experts && (p.out_ld & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(lout) & 15) == 0;
        float *sf = reinterpret_cast<float *>(my_stage);   // [8 tokens][32 experts]
        for (int c0 = 16 * grp; c0 < t.nmma; c0 += 16 * G) {
          uint32_t r[16];
          tmem_ld16(tacc + c0, r);
          tmem_ld_wait();
          if (vec) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) sf[cc * 32 + lane] = __uint_as_float(r[h * 8 + cc]) + bias;
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int f = i * 32 + lane;            // float4 f of the 8 x 32 tile
                const int row = f >> 3, col = (f & 7) * 4;
                const int tok = c0 + h * 8 + row;
                if (tok < t.nrows)
                  *reinterpret_cast<float4 *>(lout + static_cast<size_t>(t.row0 + tok) * p.out_ld + e0 + col) =
                      *reinterpret_cast<const float4 *>(sf + row * 32 + col);
              }
              __syncwarp();
            }
          } else if (e < p.n_experts) {
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
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(&tail->tmem_empty[acc]));
        else mbar_arrive_cluster(tmem_empty0 + acc * 8);
      }
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1;
      }
    }
    // h or o outside the fp16 range: recorded once per warp (a timeout code
    // already there is kept)
    if (__any_sync(0xffffffffu, range_bad) && lane == 0 && p.mode != MODE_ROUTER)
      atomicCAS(p.status, 0, p.mode == MODE_GATEUP ? DEV_RANGE_H : DEV_RANGE_O);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the pair's MMAs and epilogues are done in both CTAs
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// Stand-alone dequantisation of int4 weights into a bf16 (or fp16) array,
// with the same per-pair arithmetic as the GEMMs' in-shared-memory expansion
// (so a GEMM on the expanded array sees the same operands).  One thread turns
// 4 code bytes (8 weights of one group) into one 16-byte output chunk.
template <bool F16, bool AFF>
__global__ void __launch_bounds__(256) dequant_int4_kernel(const uint32_t *__restrict__ codes,
                                                           const __nv_bfloat16 *__restrict__ scale,
                                                           const __nv_bfloat16 *__restrict__ bias,
                                                           uint4 *__restrict__ dst, size_t rows,
                                                           int K) {
  const size_t per_row = static_cast<size_t>(K) / 8;   // chunks of 8 weights
  const size_t total = rows * per_row;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t r = i / per_row, c = i - r * per_row;
    const size_t g = r * (K / 64) + c / 8;
    const uint32_t w = __ldg(codes + i);
    uint32_t s2, b2 = 0;
    const float sf = __bfloat162float(scale[g]);
    if constexpr (F16) asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(s2) : "f"(sf));
    else asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(s2) : "f"(sf));
    uint32_t o[4];
    if constexpr (AFF) {
      const float bf = __bfloat162float(bias[g]);
      if constexpr (F16) asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(b2) : "f"(bf));
      else asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(b2) : "f"(bf));
      const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int h = 0; h < 4; ++h) o[h] = dq_pair_affine<F16>(lo, hi, h, s2, b2);
    } else {
      const uint32_t lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u;
      const uint32_t hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
#pragma unroll
      for (int h = 0; h < 4; ++h) o[h] = dq_pair<F16>(lo, hi, h, s2);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_dequant_int4(const void *codes, const void *scale, const void *bias, void *dst,
                                size_t rows, int K, bool affine, bool out_f16,
                                cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
    return e;
  const size_t total = rows * static_cast<size_t>(K) / 8;
  const int grid = static_cast<int>(std::max<size_t>(1, std::min<size_t>((total + 255) / 256,
                                                                          static_cast<size_t>(sms) * 8)));
  const auto *cw = static_cast<const uint32_t *>(codes);
  const auto *sc = static_cast<const __nv_bfloat16 *>(scale);
  const auto *bi = static_cast<const __nv_bfloat16 *>(bias);
  auto *d = static_cast<uint4 *>(dst);
  if (affine) {
    if (out_f16) dequant_int4_kernel<true, true><<<grid, 256, 0, stream>>>(cw, sc, bi, d, rows, K);
    else dequant_int4_kernel<false, true><<<grid, 256, 0, stream>>>(cw, sc, bi, d, rows, K);
  } else {
    if (out_f16) dequant_int4_kernel<true, false><<<grid, 256, 0, stream>>>(cw, sc, bi, d, rows, K);
    else dequant_int4_kernel<false, false><<<grid, 256, 0, stream>>>(cw, sc, bi, d, rows, K);
  }
  return cudaGetLastError();
}

template <int CONV> cudaError_t gemm_configure_one() {
  return cudaFuncSetAttribute(tc_gemm_kernel<CONV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(gemm_smem_bytes<CONV>()));
}

cudaError_t gemm_configure() {
  cudaError_t e;
  if ((e = gemm_configure_one<CONV_NONE>()) || (e = gemm_configure_one<CONV_BF16_TO_F16>()) ||
      (e = gemm_configure_one<CONV_INT4_TO_BF16>()) || (e = gemm_configure_one<CONV_INT4_TO_F16>()) ||
      (e = gemm_configure_one<CONV_INT4A_TO_BF16>()) || (e = gemm_configure_one<CONV_INT4A_TO_F16>()))
    return e;
  return cudaSuccess;
}

int gemm_pair_rows() { return PAIR_M; }

// Co-resident pairs of one kernel instance (both instances used here take
// one CTA per SM).
template <int CONV> int max_clusters(int grid) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(num_threads<CONV>(), 1, 1);
  cfg.dynamicSmemBytes = gemm_smem_bytes<CONV>();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tc_gemm_kernel<CONV>, &cfg) != cudaSuccess)
    clusters = 0;
  cudaGetLastError();
  return clusters;
}

int gemm_max_grid(int num_sms) {
  int grid = num_sms & ~1;
  const int c0 = max_clusters<CONV_NONE>(grid), c1 = max_clusters<CONV_INT4_TO_BF16>(grid);
  const int clusters = std::min(c0 > 0 ? c0 : grid / 2, c1 > 0 ? c1 : grid / 2);
  grid = std::min(grid, 2 * clusters);
  return grid > 2 ? grid : 2;
}

template <int CONV>
cudaError_t launch_one(dim3 g, const GemmMaps &maps, const GemmParams &p, bool pdl,
                       cudaStream_t stream) {
  return launch_kernel(tc_gemm_kernel<CONV>, g, dim3(num_threads<CONV>()), gemm_smem_bytes<CONV>(),
                       stream, pdl, maps, p);
}

cudaError_t launch_tc_gemm(const CUtensorMap &a_routed, const CUtensorMap &a_shared,
                           const CUtensorMap (&b)[4], const CUtensorMap (&b2)[4],
                           const GemmParams &p, int conv, int grid, bool pdl, cudaStream_t stream) {
  grid &= ~1;   // whole CTA pairs
  if (grid < 2) grid = 2;
  GemmMaps maps;
  maps.a_routed = a_routed;
  maps.a_shared = a_shared;
  for (int i = 0; i < 4; ++i) {
    maps.b[i] = b[i];
    maps.b2[i] = b2[i];
  }
  const dim3 g(grid);
  switch (conv) {
    case CONV_BF16_TO_F16: return launch_one<CONV_BF16_TO_F16>(g, maps, p, pdl, stream);
    case CONV_INT4_TO_BF16: return launch_one<CONV_INT4_TO_BF16>(g, maps, p, pdl, stream);
    case CONV_INT4_TO_F16: return launch_one<CONV_INT4_TO_F16>(g, maps, p, pdl, stream);
    case CONV_INT4A_TO_BF16: return launch_one<CONV_INT4A_TO_BF16>(g, maps, p, pdl, stream);
    case CONV_INT4A_TO_F16: return launch_one<CONV_INT4A_TO_F16>(g, maps, p, pdl, stream);
    default: return launch_one<CONV_NONE>(g, maps, p, pdl, stream);
  }
}

}  // namespace moe
