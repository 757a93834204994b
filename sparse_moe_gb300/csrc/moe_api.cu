// Host side of the C ABI declared in include/sparse_moe.h: argument checks,
// workspace carving, TMA tensor-map encoding, and the enqueue order of the
// prefill and decode kernels.  Nothing here synchronises the host except
// moe_ctx_create, moe_check_device and moe_profile_read.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/sparse_moe.h"
#include "moe_internal.h"

namespace {

using namespace moe;

constexpr size_t kAlign = 256;
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
  int Tc, nblk, R, Imax, max_blocks;
  size_t status, logits, idx, w, gate, mask, counts, offsets, sorted, pos, blocks, nblocks, xg, h,
      o;
  size_t dec_logits, dec_idx, dec_w, dec_g, dec_h, dec_counter, dec_phase, x_stage, y_stage,
      dec_x_stage, dec_y_stage, total;
};

WsLayout make_layout(const moe_config &c) {
  WsLayout L{};
  L.Tc = c.max_chunk_rows;
  L.nblk = (L.Tc + kRouteBlockTokens - 1) / kRouteBlockTokens;
  L.R = L.Tc * c.top_k + L.Tc;
  L.Imax = std::max(c.inter, c.shared_inter);
  L.max_blocks = (L.Tc * c.top_k) / kBlockRowsMin + c.n_experts +
                 (L.Tc + kBlockRowsMin - 1) / kBlockRowsMin + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  const size_t E = c.n_experts, k = c.top_k, H = c.hidden, Tc = L.Tc;
  L.status = take(256);
  L.logits = take(Tc * E * 4);
  L.idx = take(Tc * k * 4);
  L.w = take(Tc * k * 4);
  L.gate = take(Tc * 4);
  L.mask = take(static_cast<size_t>(L.nblk) * E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.sorted = take(Tc * k * 4);
  L.pos = take(Tc * k * 4);
  L.blocks = take(static_cast<size_t>(L.max_blocks) * 16);
  L.nblocks = take(16);
  L.xg = take(Tc * k * H * 2);
  L.h = take(static_cast<size_t>(L.R) * L.Imax * 2);
  L.o = take(static_cast<size_t>(L.R) * H * 2);
  L.dec_logits = take(E * 4);
  L.dec_idx = take(k * 4);
  L.dec_w = take(k * 4);
  L.dec_g = take(4);
  L.dec_h = take(decode_h_floats(c.top_k, L.Imax) * 4);
  L.dec_counter = take(16);
  L.dec_phase = take(static_cast<size_t>(kMaxPhaseCtas) * 2 * 8);
  L.x_stage = take(2 * Tc * H * 2);   // two slots: see moe_forward_prefill_host
  L.y_stage = take(2 * Tc * H * 2);
  L.dec_x_stage = take(H * 2);   // moe_forward_decode_host (apart from the prefill slots,
  L.dec_y_stage = take(H * 2);   // whose input copies do not wait for the caller's stream)
  L.total = off;
  return L;
}

// ---------------------------------------------------------- tensor maps --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 (or fp16) matrix [outer, inner] (inner contiguous), 128-byte
// swizzled boxes of {64, box_rows} elements: the K-major weight tiles of the
// grouped GEMMs.
bool encode_weight_map(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
                       uint32_t box_rows, bool f16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four token-row maps of a 2-D bf16 (or fp16) matrix [rows, inner]:
// boxes of {64, 16 << i} elements, 128-byte swizzled (the grouped GEMMs' B
// operand, one or two boxes per stage chosen from the block's size).
bool encode_row_maps(CUtensorMap (&m)[4], const void *ptr, uint64_t inner, uint64_t rows,
                     bool f16 = false) {
  for (int i = 0; i < 4; ++i)
    if (!encode_weight_map(&m[i], ptr, inner, rows, 16u << i, f16)) return false;
  return true;
}

// The gate/up weights [experts, 2 inter, K] as a 3-D bf16 tensor {K, inter,
// 2 experts}: a box {64, 64, 2} holds 64 gate rows followed by the matching
// 64 up rows of one expert, 128-byte swizzled (one TMA box per CTA and
// k-step).
bool encode_gateup_map(CUtensorMap *m, const void *ptr, uint64_t K, uint64_t inter,
                       uint64_t experts) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {K, inter, 2 * experts};
  const cuuint64_t strides[2] = {K * 2, inter * K * 2};
  const cuuint32_t box[3] = {64, 64, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D matrix of packed int4 codes [outer rows, inner bytes] (two codes per
// byte along K), unswizzled boxes of {32 bytes (64 codes), box_rows}: the
// int4 weight tiles, dequantised in shared memory by the GEMM.
bool encode_code_map(CUtensorMap *m, const void *ptr, uint64_t inner_bytes, uint64_t outer,
                     uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner_bytes, outer};
  const cuuint64_t strides[1] = {inner_bytes};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

enum KernelId : int {
  K_ROUTER_GEMM = 0, K_TOPK, K_PLACE, K_GATEUP_GEMM, K_DOWN_GEMM, K_COMBINE,
  K_DEC_LAYER, K_H2D, K_D2H, K_DEC_LAYERS, K_ROWS, K_COUNT
};
const char *kKernelNames[K_COUNT] = {
    "router_gemm", "topk", "route_place", "gateup_swiglu_gemm", "down_gemm",
    "combine", "decode_layer", "h2d_copy", "d2h_copy", "decode_layers", "rows"};

}  // namespace

struct LayerSlot {
  bool loaded = false;
  bool down_f16 = false;   // caller-supplied fp16 copies of down / sh_down
  moe_weights w{};
  // TMA descriptors of the weight (A) operands, encoded at load time
  CUtensorMap map_router, map_gu, map_gu_sh, map_dn, map_dn_sh;
};

struct moe_ctx {
  moe_config cfg{};
  int device = 0;
  int num_sms = 0;
  int gemm_grid = 0;   // CTAs of the persistent grouped-GEMM grid (whole pairs)
  int router_split = 1;    // router GEMM split-K parts (router_split())
  CUtensorMap map_h[4];    // h [R, Imax] fp16 in the workspace: the down GEMM's token rows
  CUtensorMap map_xg[4];   // x in grouped order [Tc k, H] bf16: the routed gate/up token rows
  bool prefill_pdl = true; // programmatic dependent launch between prefill kernels (MOE_PREFILL_PDL)
  // Measurement options (environment, read at creation; off by default), each
  // undoing one mechanism of the page to measure what it is worth here:
  //   MOE_ABLATE_HOST_ROUTING=1  the host waits for the routing and reads the
  //                              block count before the grouped GEMMs launch;
  //   MOE_ABLATE_TILE=fixed256   every block runs the full 256-row MMA N;
  //   MOE_ABLATE_TILE=rows<n>    blocks of at most n rows (16 <= n <= 256).
  bool ablate_host_routing = false;
  int ablate_fixed_n = 0;
  int block_rows = kBlockRowsMax;
  int32_t host_nblocks = 0;
  int decode_grid = 0;     // CTAs of the cooperative decode launch
  int last_rows = 0;       // rows of the last moe_forward_rows (its routing is in the prefill regions)
  // moe_forward_prefill_host: copy streams and the events of the two staging
  // slots (created on first use)
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t ev_x[2] = {}, ev_y[2] = {}, ev_out[2] = {};
  int host_slot = 0;
  int decode_smem = 0;     // dynamic shared-memory limit of the decode kernel
  bool decode_pdl = true;  // decode launches overlap the previous kernel's tail
  char *ws = nullptr;
  size_t ws_bytes = 0;
  WsLayout L{};
  std::vector<LayerSlot> layers;
  std::string last_error;
  int64_t launches = 0;
  // profiling
  bool profiling = false;
  struct Rec { int id; cudaEvent_t a, b; };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> event_pool;
  int64_t prof_launches[K_COUNT] = {};
  double prof_ms[K_COUNT] = {};

  template <class T> T *at(size_t off) const { return reinterpret_cast<T *>(ws + off); }
  int *status() const { return at<int>(L.status); }
};

namespace {

moe_status fail(moe_ctx *ctx, moe_status s, const char *fmt, ...) {
  if (ctx) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    ctx->last_error = buf;
  }
  return s;
}

moe_status cuda_fail(moe_ctx *ctx, cudaError_t e, const char *what) {
  return fail(ctx, MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

moe_status check_config(const moe_config *c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->hidden < 64 || c->hidden > 16384 || c->hidden % 64) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->n_experts > 1024) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > std::min(c->n_experts, 32)) return MOE_ERR_INVALID_ARG;
  if (c->inter < 64 || c->inter % 64 || c->shared_inter < 64 || c->shared_inter % 64)
    return MOE_ERR_INVALID_ARG;
  if (c->inter > 16384 || c->shared_inter > 16384) return MOE_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->n_layers > 4096) return MOE_ERR_INVALID_ARG;
  if (c->max_chunk_rows < 1 || c->max_chunk_rows > 65536) return MOE_ERR_INVALID_ARG;
  if (c->wfmt != MOE_W_BF16 && c->wfmt != MOE_W_INT4_SYM_G64 && c->wfmt != MOE_W_INT4_AFFINE_G64)
    return MOE_ERR_INVALID_ARG;
  const size_t imax = std::max(c->inter, c->shared_inter);
  // the GEMM producers address operand rows with 32-bit element offsets
  const size_t lim = size_t(1) << 31;
  const size_t R = static_cast<size_t>(c->max_chunk_rows) * (c->top_k + 1);
  if (static_cast<size_t>(c->n_experts) * 2 * c->inter * c->hidden >= lim ||
      static_cast<size_t>(c->n_experts) * c->hidden * c->inter >= lim ||
      R * imax >= lim || static_cast<size_t>(c->max_chunk_rows) * c->hidden >= lim)
    return MOE_ERR_UNSUPPORTED;
  if ((c->top_k + 1) * imax * 4 > 200 * 1024 || c->hidden * 4 > 200 * 1024)
    return MOE_ERR_UNSUPPORTED;   // decode staging must fit in shared memory
  return MOE_OK;
}

struct ProfScope {
  moe_ctx *ctx;
  int id;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  ProfScope(moe_ctx *c, int kid, cudaStream_t st) : ctx(c), id(kid), s(st) {
    if (!ctx->profiling) return;
    if (ctx->event_pool.size() < 2) {
      for (int i = 0; i < 64; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) break;
        ctx->event_pool.push_back(e);
      }
      if (ctx->event_pool.size() < 2) return;
    }
    a = ctx->event_pool.back();
    ctx->event_pool.pop_back();
    b = ctx->event_pool.back();
    ctx->event_pool.pop_back();
    cudaEventRecord(a, s);
  }
  ~ProfScope() {
    if (!a) return;
    cudaEventRecord(b, s);
    ctx->pending.push_back({id, a, b});
  }
};

moe_status ensure_device(moe_ctx *ctx) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
  if (cur != ctx->device) {
    e = cudaSetDevice(ctx->device);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaSetDevice");
  }
  return MOE_OK;
}

moe_status launched(moe_ctx *ctx, cudaError_t e, const char *what) {
  ++ctx->launches;
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  return MOE_OK;
}

// Router GEMM split-K parts S (4, 2 or 1: the largest dividing H / 64 whose
// parts fit the scratch).  S depends on the configuration only, so every
// token's logits are summed in the same order whatever the chunk length
// ("Bound temporary memory with prompt chunking": chunking leaves the output
// bit for bit unchanged).  With S > 1 the parts go to scratch space of
// S * T * E floats (the o buffer, which a chunk does not use until its down
// projection) and the top-k kernel adds them in part order.
int router_split(const moe_config &c, const WsLayout &L) {
  const int nk = c.hidden / 64;
  const size_t scratch_floats = static_cast<size_t>(L.R) * c.hidden / 2;
  for (int S = 4; S > 1; S /= 2)
    if (nk % S == 0 && static_cast<size_t>(S) * L.Tc * c.n_experts <= scratch_floats) return S;
  return 1;
}

// Token rows per router tile: enough tiles (with the split-K parts) for every
// CTA pair, 32..256 rows.
int router_block_rows(const moe_ctx *ctx, int T) {
  const long long mt = (ctx->cfg.n_experts + gemm_pair_rows() - 1) / gemm_pair_rows();
  const long long pairs = std::max(1, ctx->num_sms / 2);
  long long br = (static_cast<long long>(T) * mt * ctx->router_split + pairs - 1) / pairs;
  br = (br + 31) & ~31LL;
  return static_cast<int>(std::min<long long>(kBlockRowsMax, std::max<long long>(32, br)));
}

// Router GEMM, top-k, then the placement kernel (histogram, scan, block map,
// scatter, shared gate) for T <= Tc tokens; the summed logits go to `logits`
// when it is non-null.  map_x: the token-row maps of x (T rows); with_xg: the
// placement also writes x in grouped order into the workspace (the routed
// gate/up GEMM's token rows).
moe_status enqueue_route(moe_ctx *ctx, const LayerSlot &ls, const void *x, int T, float *logits,
                         int32_t *idx, float *w, int32_t *counts, int32_t *offsets,
                         int32_t *sorted_rows, int32_t *pos, const CUtensorMap (&map_x)[4],
                         bool with_xg, cudaStream_t s) {
  const moe_config &c = ctx->cfg;
  const WsLayout &L = ctx->L;
  GemmParams gp{};
  gp.mode = MODE_ROUTER;
  gp.a_routed = gp.a_shared = ls.w.router_w;
  gp.lda_routed = gp.lda_shared = c.hidden;
  gp.a_rows_routed = gp.a_rows_shared = c.n_experts;
  gp.block_rows = router_block_rows(ctx, T);
  gp.k_split = ctx->router_split;
  gp.n_blocks_host = (T + gp.block_rows - 1) / gp.block_rows;
  gp.T = T;
  gp.m_tiles = (c.n_experts + gemm_pair_rows() - 1) / gemm_pair_rows();
  gp.n_experts = c.n_experts;
  gp.hidden = c.hidden;
  gp.inter_routed = c.inter;
  gp.inter_shared = c.shared_inter;
  gp.k_routed = c.hidden;
  // one part: logits straight into the caller's buffer (or the workspace's);
  // several: parts in the o scratch, summed by the top-k kernel
  float *part = gp.k_split > 1 ? ctx->at<float>(L.o) : (logits ? logits : ctx->at<float>(L.logits));
  gp.out = part;
  gp.out_split_stride = static_cast<size_t>(T) * c.n_experts;
  gp.out_ld = c.n_experts;
  gp.bias = ls.w.router_b;
  gp.status = ctx->status();
  const int tiles = gp.n_blocks_host * gp.m_tiles * gp.k_split;
  moe_status st;
  {
    ProfScope ps(ctx, K_ROUTER_GEMM, s);
    st = launched(ctx, launch_tc_gemm(ls.map_router, ls.map_router, map_x, map_x, gp, CONV_NONE,
                                      std::min(ctx->gemm_grid, 2 * tiles), ctx->prefill_pdl, s),
                  "router gemm launch");
  }
  if (st) return st;
  uint32_t *mask = ctx->at<uint32_t>(L.mask);
  {
    ProfScope ps(ctx, K_TOPK, s);
    st = launched(ctx,
                  launch_topk(part, gp.k_split, gp.out_split_stride,
                              gp.k_split > 1 ? logits : nullptr, T, c.n_experts, c.top_k, idx,
                              w, mask, ctx->prefill_pdl, s),
                  "topk launch");
  }
  if (st) return st;
  {
    ProfScope ps(ctx, K_PLACE, s);
    st = launched(ctx,
                  launch_place(idx, mask, T, c.n_experts, c.top_k, counts, offsets,
                               ctx->at<int4>(L.blocks), ctx->at<int32_t>(L.nblocks),
                               ctx->block_rows, sorted_rows, pos, x,
                               with_xg ? ctx->at<void>(L.xg) : nullptr, ls.w.sh_gate_w,
                               ctx->at<float>(L.gate), c.hidden, ctx->prefill_pdl, s),
                  "placement launch");
  }
  return st;
}

moe_status enqueue_prefill_chunk(moe_ctx *ctx, const LayerSlot &ls, const void *x, int T, void *y,
                                 cudaStream_t s) {
  const moe_config &c = ctx->cfg;
  const WsLayout &L = ctx->L;
  int32_t *idx = ctx->at<int32_t>(L.idx);
  float *w = ctx->at<float>(L.w);
  int32_t *sorted = ctx->at<int32_t>(L.sorted);
  int32_t *pos = ctx->at<int32_t>(L.pos);
  // token-row maps of this call's x (the router's, and the shared expert's
  // gate/up token rows)
  CUtensorMap map_x[4];
  if (!encode_row_maps(map_x, x, c.hidden, static_cast<uint64_t>(T)))
    return fail(ctx, MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for x");
  moe_status st = enqueue_route(ctx, ls, x, T, nullptr, idx, w,
                                ctx->at<int32_t>(L.counts), ctx->at<int32_t>(L.offsets), sorted,
                                pos, map_x, true, s);
  if (st) return st;
  if (ctx->ablate_host_routing) {
    // measurement option: the CPU waits for the routing and inspects it
    // before it submits the grouped GEMMs
    cudaError_t e = cudaMemcpyAsync(&ctx->host_nblocks, ctx->at<int32_t>(L.nblocks), 4,
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "host routing read-back");
  }
  GemmParams gp{};
  gp.fixed_n = ctx->ablate_fixed_n;
  gp.blocks = ctx->at<int4>(L.blocks);
  gp.n_blocks_dev = ctx->at<int32_t>(L.nblocks);
  gp.T = T;
  gp.n_experts = c.n_experts;
  gp.hidden = c.hidden;
  gp.inter_routed = c.inter;
  gp.inter_shared = c.shared_inter;
  gp.k_routed = c.hidden;
  gp.shared_row0 = T * c.top_k;
  gp.status = ctx->status();
  const bool int4 = c.wfmt != MOE_W_BF16;
  const bool aff = c.wfmt == MOE_W_INT4_AFFINE_G64;
  // gate/up + SwiGLU -> h
  gp.mode = MODE_GATEUP;
  gp.m_tiles = (L.Imax + gemm_pair_rows() / 2 - 1) / (gemm_pair_rows() / 2);   // 128 SwiGLU outputs per pair
  gp.a_routed = ls.w.gate_up;
  gp.a_shared = ls.w.sh_gate_up;
  gp.lda_routed = gp.lda_shared = c.hidden;
  gp.a_rows_routed = c.n_experts * 2 * c.inter;
  gp.a_rows_shared = 2 * c.shared_inter;
  gp.out = ctx->at<void>(L.h);
  gp.out_ld = L.Imax;
  gp.a_scale_routed = int4 ? ls.w.gate_up_scale : nullptr;
  gp.a_scale_shared = int4 ? ls.w.sh_gate_up_scale : nullptr;
  gp.a_bias_routed = aff ? ls.w.gate_up_bias : nullptr;
  gp.a_bias_shared = aff ? ls.w.sh_gate_up_bias : nullptr;
  {
    ProfScope ps(ctx, K_GATEUP_GEMM, s);
    st = launched(ctx,
                  launch_tc_gemm(ls.map_gu, ls.map_gu_sh, ctx->map_xg, map_x, gp,
                                 aff ? CONV_INT4A_TO_BF16 : int4 ? CONV_INT4_TO_BF16 : CONV_NONE,
                                 ctx->gemm_grid, ctx->prefill_pdl, s),
                  "gate/up gemm launch");
  }
  if (st) return st;
  // down -> o
  gp.mode = MODE_DOWN;
  gp.a_routed = ls.down_f16 ? ls.w.down_f16 : ls.w.down;
  gp.a_shared = ls.down_f16 ? ls.w.sh_down_f16 : ls.w.sh_down;
  gp.ab_f16 = ls.down_f16 ? 1 : 0;
  gp.lda_routed = c.inter;
  gp.lda_shared = c.shared_inter;
  gp.a_rows_routed = c.n_experts * c.hidden;
  gp.a_rows_shared = c.hidden;
  gp.m_tiles = (c.hidden + gemm_pair_rows() - 1) / gemm_pair_rows();
  gp.out = ctx->at<void>(L.o);
  gp.out_ld = c.hidden;
  gp.a_scale_routed = int4 ? ls.w.down_scale : nullptr;
  gp.a_scale_shared = int4 ? ls.w.sh_down_scale : nullptr;
  gp.a_bias_routed = aff ? ls.w.down_bias : nullptr;
  gp.a_bias_shared = aff ? ls.w.sh_down_bias : nullptr;
  {
    ProfScope ps(ctx, K_DOWN_GEMM, s);
    st = launched(ctx,
                  launch_tc_gemm(ls.map_dn, ls.map_dn_sh, ctx->map_h, ctx->map_h, gp,
                                 aff ? CONV_INT4A_TO_F16 : int4 ? CONV_INT4_TO_F16
                                      : (ls.down_f16 ? CONV_NONE : CONV_BF16_TO_F16),
                                 ctx->gemm_grid, ctx->prefill_pdl, s),
                  "down gemm launch");
  }
  if (st) return st;
  {
    ProfScope ps(ctx, K_COMBINE, s);
    st = launched(ctx,
                  launch_combine(ctx->at<float>(L.gate), ctx->at<void>(L.o), pos, w, T, c.hidden,
                                 c.top_k, y, ctx->prefill_pdl, s),
                  "combine launch");
  }
  return st;
}

moe_status check_layer(moe_ctx *ctx, int layer) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.n_layers)
    return fail(ctx, MOE_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, ctx->cfg.n_layers);
  if (!ctx->layers[layer].loaded) return fail(ctx, MOE_ERR_NOT_LOADED, "layer %d not loaded", layer);
  return MOE_OK;
}

DecodeParams decode_params(const moe_ctx *ctx, const LayerSlot &ls, const void *x, void *y) {
  const moe_config &c = ctx->cfg;
  const WsLayout &L = ctx->L;
  DecodeParams p{};
  p.x = x;
  p.y = y;
  p.H = c.hidden;
  p.E = c.n_experts;
  p.k = c.top_k;
  p.I = c.inter;
  p.Is = c.shared_inter;
  p.wfmt = c.wfmt;
  p.router_w = ls.w.router_w;
  p.router_b = ls.w.router_b;
  p.gate_up = ls.w.gate_up;
  p.gate_up_scale = ls.w.gate_up_scale;
  p.down = ls.w.down;
  p.down_scale = ls.w.down_scale;
  p.sh_gate_up = ls.w.sh_gate_up;
  p.sh_gate_up_scale = ls.w.sh_gate_up_scale;
  p.sh_down = ls.w.sh_down;
  p.sh_down_scale = ls.w.sh_down_scale;
  p.sh_gate_w = ls.w.sh_gate_w;
  p.gate_up_bias = ls.w.gate_up_bias;
  p.down_bias = ls.w.down_bias;
  p.sh_gate_up_bias = ls.w.sh_gate_up_bias;
  p.sh_down_bias = ls.w.sh_down_bias;
  p.logits = ctx->at<float>(L.dec_logits);
  p.idx = ctx->at<int32_t>(L.dec_idx);
  p.w = ctx->at<float>(L.dec_w);
  p.g = ctx->at<float>(L.dec_g);
  p.h = ctx->at<float>(L.dec_h);
  p.h_ld = L.Imax;
  p.bar = ctx->at<unsigned long long>(L.dec_counter);
  p.phase_ts = ctx->profiling && ctx->decode_grid <= kMaxPhaseCtas
                   ? ctx->at<unsigned long long>(L.dec_phase)
                   : nullptr;
  p.status = ctx->status();
  return p;
}

moe_status enqueue_decode(moe_ctx *ctx, const LayerSlot &ls, const void *x, void *y,
                          cudaStream_t s) {
  const DecodeParams p = decode_params(ctx, ls, x, y);
  ProfScope ps(ctx, K_DEC_LAYER, s);
  return launched(ctx, launch_decode_layer(p, ctx->decode_grid, ctx->decode_smem, ctx->decode_pdl, s),
                  "decode layer launch");
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_NOT_LOADED: return "layer weights not loaded";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_RANGE: return "prefill intermediate outside the fp16 range";
  }
  return "unknown status";
}

moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const moe_status st = check_config(cfg);
  if (st) return st;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_ctx_create(const moe_config *cfg, int device, void *workspace, size_t ws_bytes,
                          moe_ctx **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status st = check_config(cfg);
  if (st) return st;
  const WsLayout L = make_layout(*cfg);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 || ws_bytes < L.total)
    return MOE_ERR_WORKSPACE;
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;   // built for sm_103a only
  if (!encode_fn()) return MOE_ERR_CUDA;
  moe_ctx *ctx = new moe_ctx();
  ctx->cfg = *cfg;
  ctx->device = device;
  ctx->num_sms = sms;
  ctx->ws = static_cast<char *>(workspace);
  ctx->ws_bytes = ws_bytes;
  ctx->L = L;
  ctx->layers.resize(cfg->n_layers);
  if ((e = gemm_configure()) != cudaSuccess) {
    delete ctx;
    return MOE_ERR_CUDA;
  }
  ctx->gemm_grid = gemm_max_grid(sms);
  ctx->router_split = router_split(ctx->cfg, ctx->L);
  if (!encode_row_maps(ctx->map_h, ctx->ws + L.h, L.Imax, static_cast<uint64_t>(L.R), true) ||
      !encode_row_maps(ctx->map_xg, ctx->ws + L.xg, cfg->hidden,
                       static_cast<uint64_t>(L.Tc) * cfg->top_k)) {
    delete ctx;
    return MOE_ERR_CUDA;
  }
  ctx->decode_grid = decode_layer_grid(sms);
  if (const char *env = std::getenv("MOE_DECODE_PDL")) ctx->decode_pdl = std::atoi(env) != 0;
  if (const char *env = std::getenv("MOE_PREFILL_PDL")) ctx->prefill_pdl = std::atoi(env) != 0;
  if (const char *env = std::getenv("MOE_ABLATE_HOST_ROUTING"))
    ctx->ablate_host_routing = std::atoi(env) != 0;
  if (const char *env = std::getenv("MOE_ABLATE_TILE")) {
    if (std::strcmp(env, "fixed256") == 0) ctx->ablate_fixed_n = 1;
    if (std::strncmp(env, "rows", 4) == 0)
      ctx->block_rows = std::min(kBlockRowsMax, std::max(kBlockRowsMin, std::atoi(env + 4)));
  }
  if (
      (e = decode_configure(&ctx->decode_smem)) != cudaSuccess ||
      (e = cudaMemset(ctx->ws + L.status, 0, 256)) != cudaSuccess ||
      (e = cudaMemset(ctx->ws + L.dec_counter, 0, 16)) != cudaSuccess ||
      (e = cudaDeviceSynchronize()) != cudaSuccess) {
    delete ctx;
    return MOE_ERR_CUDA;
  }
  *out = ctx;
  return MOE_OK;
}

moe_status moe_ctx_destroy(moe_ctx *ctx) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  for (auto &r : ctx->pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : ctx->event_pool) cudaEventDestroy(e);
  for (int i = 0; i < 2; ++i) {
    if (ctx->ev_x[i]) cudaEventDestroy(ctx->ev_x[i]);
    if (ctx->ev_y[i]) cudaEventDestroy(ctx->ev_y[i]);
    if (ctx->ev_out[i]) cudaEventDestroy(ctx->ev_out[i]);
  }
  if (ctx->copy_in) cudaStreamDestroy(ctx->copy_in);
  if (ctx->copy_out) cudaStreamDestroy(ctx->copy_out);
  delete ctx;
  return MOE_OK;
}

moe_status moe_load_weights(moe_ctx *ctx, int layer, const moe_weights *w) {
  if (!ctx || !w) return fail(ctx, MOE_ERR_INVALID_ARG, "null context or weights");
  if (layer < 0 || layer >= ctx->cfg.n_layers)
    return fail(ctx, MOE_ERR_INVALID_ARG, "layer %d out of range", layer);
  const moe_config &c = ctx->cfg;
  const bool int4 = c.wfmt != MOE_W_BF16;
  const bool aff = c.wfmt == MOE_W_INT4_AFFINE_G64;
  const void *req[] = {w->router_w, w->gate_up, w->down, w->sh_gate_up, w->sh_down, w->sh_gate_w};
  for (const void *p : req)
    if (!p || !aligned16(p)) return fail(ctx, MOE_ERR_INVALID_ARG, "weight pointer null or not 16-byte aligned");
  if (w->router_b && (reinterpret_cast<uintptr_t>(w->router_b) & 3))
    return fail(ctx, MOE_ERR_INVALID_ARG, "router_b misaligned");
  if (int4) {
    const void *sc[] = {w->gate_up_scale, w->down_scale, w->sh_gate_up_scale, w->sh_down_scale};
    for (const void *p : sc)
      if (!p || (reinterpret_cast<uintptr_t>(p) & 1))
        return fail(ctx, MOE_ERR_INVALID_ARG, "int4 format needs all four scale pointers");
  }
  const void *bi[] = {w->gate_up_bias, w->down_bias, w->sh_gate_up_bias, w->sh_down_bias};
  for (const void *p : bi) {
    if (aff && (!p || (reinterpret_cast<uintptr_t>(p) & 1)))
      return fail(ctx, MOE_ERR_INVALID_ARG, "affine int4 format needs all four bias pointers");
    if (!aff && p) return fail(ctx, MOE_ERR_INVALID_ARG, "bias pointers apply to affine int4 only");
  }
  const bool f16_down = w->down_f16 != nullptr || w->sh_down_f16 != nullptr;
  if (f16_down) {
    if (int4) return fail(ctx, MOE_ERR_INVALID_ARG, "fp16 down copies apply to bf16 weights only");
    if (!w->down_f16 || !w->sh_down_f16)
      return fail(ctx, MOE_ERR_INVALID_ARG, "down_f16 and sh_down_f16 go together");
    if (!aligned16(w->down_f16) || !aligned16(w->sh_down_f16))
      return fail(ctx, MOE_ERR_INVALID_ARG, "fp16 down copies not 16-byte aligned");
  }
  LayerSlot &ls = ctx->layers[layer];
  ls.loaded = false;
  ls.w = *w;
  ls.down_f16 = f16_down;
  bool ok = encode_weight_map(&ls.map_router, w->router_w, c.hidden, c.n_experts, 128);
  if (!int4) {
    ok = ok && encode_gateup_map(&ls.map_gu, w->gate_up, c.hidden, c.inter, c.n_experts);
    ok = ok && encode_gateup_map(&ls.map_gu_sh, w->sh_gate_up, c.hidden, c.shared_inter, 1);
    ok = ok && encode_weight_map(&ls.map_dn, f16_down ? w->down_f16 : w->down, c.inter,
                                 static_cast<uint64_t>(c.n_experts) * c.hidden, 128, f16_down);
    ok = ok && encode_weight_map(&ls.map_dn_sh, f16_down ? w->sh_down_f16 : w->sh_down,
                                 c.shared_inter, c.hidden, 128, f16_down);
  } else {
    ok = ok && encode_code_map(&ls.map_gu, w->gate_up, c.hidden / 2,
                               static_cast<uint64_t>(c.n_experts) * 2 * c.inter, 64);
    ok = ok && encode_code_map(&ls.map_gu_sh, w->sh_gate_up, c.hidden / 2, 2 * c.shared_inter, 64);
    ok = ok && encode_code_map(&ls.map_dn, w->down, c.inter / 2,
                               static_cast<uint64_t>(c.n_experts) * c.hidden, 128);
    ok = ok && encode_code_map(&ls.map_dn_sh, w->sh_down, c.shared_inter / 2, c.hidden, 128);
  }
  if (!ok) return fail(ctx, MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for layer %d", layer);
  ls.loaded = true;
  return MOE_OK;
}

moe_status moe_route(moe_ctx *ctx, int layer, const void *x, int T, float *logits,
                     int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets,
                     int32_t *sorted_rows, int32_t *pos_of_assign, void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  if (T < 0 || T > ctx->cfg.max_chunk_rows)
    return fail(ctx, MOE_ERR_INVALID_ARG, "T=%d outside [0, max_chunk_rows=%d]", T,
                ctx->cfg.max_chunk_rows);
  if (T == 0) return MOE_OK;
  if (!x || !aligned16(x) || !topk_idx || !topk_w || !counts || !offsets || !sorted_rows ||
      !pos_of_assign)
    return fail(ctx, MOE_ERR_INVALID_ARG, "null or misaligned routing buffer");
  if ((st = ensure_device(ctx))) return st;
  CUtensorMap map_x[4];
  if (!encode_row_maps(map_x, x, ctx->cfg.hidden, static_cast<uint64_t>(T)))
    return fail(ctx, MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for x");
  return enqueue_route(ctx, ctx->layers[layer], x, T, logits, topk_idx, topk_w, counts, offsets,
                       sorted_rows, pos_of_assign, map_x, false, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_prefill(moe_ctx *ctx, int layer, const void *x, int T, void *y,
                               void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  if (T < 0) return fail(ctx, MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (T == 0) return MOE_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y))
    return fail(ctx, MOE_ERR_INVALID_ARG, "x/y null or not 16-byte aligned");
  const size_t row_bytes = static_cast<size_t>(ctx->cfg.hidden) * 2;
  const char *xb = static_cast<const char *>(x);
  char *yb = static_cast<char *>(y);
  if (xb < yb + T * row_bytes && yb < xb + T * row_bytes)
    return fail(ctx, MOE_ERR_INVALID_ARG, "x and y overlap");
  if ((st = ensure_device(ctx))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const LayerSlot &ls = ctx->layers[layer];
  for (int c0 = 0; c0 < T; c0 += ctx->cfg.max_chunk_rows) {
    const int n = std::min(ctx->cfg.max_chunk_rows, T - c0);
    st = enqueue_prefill_chunk(ctx, ls, xb + c0 * row_bytes, n, yb + c0 * row_bytes, s);
    if (st) return st;
  }
  return MOE_OK;
}

moe_status moe_forward_decode(moe_ctx *ctx, int layer, const void *x, void *y, void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  if (!x || !y || !aligned16(x) || !aligned16(y))
    return fail(ctx, MOE_ERR_INVALID_ARG, "x/y null or not 16-byte aligned");
  if ((st = ensure_device(ctx))) return st;
  return enqueue_decode(ctx, ctx->layers[layer], x, y, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_decode_layers(moe_ctx *ctx, int first_layer, int n_layers, const void *x,
                                     size_t x_stride, void *y, size_t y_stride, void *stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (n_layers < 0 || first_layer < 0 || first_layer + n_layers > ctx->cfg.n_layers)
    return fail(ctx, MOE_ERR_INVALID_ARG, "layers [%d, %d) outside the context's %d slots",
                first_layer, first_layer + n_layers, ctx->cfg.n_layers);
  if (n_layers == 0) return MOE_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y) || (x_stride & 7) || (y_stride & 7))
    return fail(ctx, MOE_ERR_INVALID_ARG, "x/y null or rows not 16-byte aligned");
  for (int l = first_layer; l < first_layer + n_layers; ++l) {
    moe_status st = check_layer(ctx, l);
    if (st) return st;
  }
  moe_status st = ensure_device(ctx);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char *xb = static_cast<const char *>(x);
  char *yb = static_cast<char *>(y);
  DecodeParams ps[kMaxDecodeLayers];
  for (int l0 = 0; l0 < n_layers; l0 += kMaxDecodeLayers) {
    const int n = std::min(kMaxDecodeLayers, n_layers - l0);
    for (int i = 0; i < n; ++i) {
      const size_t l = static_cast<size_t>(l0 + i);
      ps[i] = decode_params(ctx, ctx->layers[first_layer + l0 + i], xb + l * x_stride * 2,
                            yb + l * y_stride * 2);
    }
    ProfScope pr(ctx, K_DEC_LAYERS, s);
    st = launched(ctx,
                  launch_decode_layers(ps, n, ctx->decode_grid, ctx->decode_smem, ctx->decode_pdl,
                                       s),
                  "multi-layer decode launch");
    if (st) return st;
  }
  return MOE_OK;
}

moe_status moe_forward_rows(moe_ctx *ctx, int layer, const void *x, int T, void *y,
                            void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  const moe_config &c = ctx->cfg;
  const WsLayout &L = ctx->L;
  if (T < 1 || T > kSmallMaxRows || T > L.Tc)
    return fail(ctx, MOE_ERR_INVALID_ARG, "T = %d outside 1..%d (and the context's max_chunk_rows %d)",
                T, kSmallMaxRows, L.Tc);
  if (!x || !y || !aligned16(x) || !aligned16(y))
    return fail(ctx, MOE_ERR_INVALID_ARG, "x/y null or not 16-byte aligned");
  // h [T][k + 1][Imax] fp32 lives in the o region ([R, H] fp16)
  if (static_cast<size_t>(T) * (c.top_k + 1) * L.Imax * 4 > static_cast<size_t>(L.R) * c.hidden * 2)
    return fail(ctx, MOE_ERR_UNSUPPORTED, "rows scratch does not fit the workspace");
  if ((st = ensure_device(ctx))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DecodeParams p = decode_params(ctx, ctx->layers[layer], x, y);
  p.T = T;
  p.logits = ctx->at<float>(L.logits);
  p.idx = ctx->at<int32_t>(L.idx);
  p.w = ctx->at<float>(L.w);
  p.g = ctx->at<float>(L.gate);
  p.h = ctx->at<float>(L.o);
  ProfScope ps(ctx, K_ROWS, s);
  st = launched(ctx, launch_rows(p, ctx->decode_grid, ctx->decode_smem, ctx->decode_pdl, s),
                "rows launch");
  if (st == MOE_OK) ctx->last_rows = T;
  return st;
}

moe_status moe_rows_routing(moe_ctx *ctx, float *logits, int32_t *idx, float *w, void *stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (ctx->last_rows < 1) return fail(ctx, MOE_ERR_INVALID_ARG, "no moe_forward_rows call yet");
  moe_status st = ensure_device(ctx);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe_config &c = ctx->cfg;
  const size_t T = static_cast<size_t>(ctx->last_rows);
  cudaError_t e = cudaSuccess;
  if (logits)
    e = cudaMemcpyAsync(logits, ctx->ws + ctx->L.logits, T * c.n_experts * 4,
                        cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && idx)
    e = cudaMemcpyAsync(idx, ctx->ws + ctx->L.idx, T * c.top_k * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && w)
    e = cudaMemcpyAsync(w, ctx->ws + ctx->L.w, T * c.top_k * 4, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(ctx, e, "rows routing copy");
}

moe_status moe_decode_routing(moe_ctx *ctx, float *logits, int32_t *idx, float *w, void *stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  moe_status st = ensure_device(ctx);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe_config &c = ctx->cfg;
  cudaError_t e = cudaSuccess;
  if (logits)
    e = cudaMemcpyAsync(logits, ctx->ws + ctx->L.dec_logits, c.n_experts * 4,
                        cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && idx)
    e = cudaMemcpyAsync(idx, ctx->ws + ctx->L.dec_idx, c.top_k * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && w)
    e = cudaMemcpyAsync(w, ctx->ws + ctx->L.dec_w, c.top_k * 4, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(ctx, e, "decode routing copy");
}

moe_status moe_forward_prefill_host(moe_ctx *ctx, int layer, const void *x_host, int T,
                                    void *y_host, void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  if (T < 0 || (T > 0 && (!x_host || !y_host)))
    return fail(ctx, MOE_ERR_INVALID_ARG, "bad host buffers or T");
  if (T == 0) return MOE_OK;
  if ((st = ensure_device(ctx))) return st;
  cudaError_t e = cudaSuccess;
  if (!ctx->copy_in) {
    if ((e = cudaStreamCreateWithFlags(&ctx->copy_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&ctx->copy_out, cudaStreamNonBlocking)) != cudaSuccess)
      return cuda_fail(ctx, e, "copy stream creation");
    for (int i = 0; i < 2; ++i)
      if ((e = cudaEventCreateWithFlags(&ctx->ev_x[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&ctx->ev_y[i], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&ctx->ev_out[i], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(ctx, e, "copy event creation");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t row_bytes = static_cast<size_t>(ctx->cfg.hidden) * 2;
  const size_t slot_bytes = static_cast<size_t>(ctx->L.Tc) * row_bytes;
  const LayerSlot &ls = ctx->layers[layer];
  // Page-locked y_host is directly addressable by the device: the combine
  // kernel then writes y into it (over the CPU-GPU link) and no output copy
  // or staging is needed.
  char *y_direct = nullptr;
  {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer != nullptr && aligned16(pa.devicePointer))
      y_direct = static_cast<char *>(pa.devicePointer);
    else
      cudaGetLastError();   // pageable memory: not an error here
  }
  // Chunk c uses staging slot c % 2 (alternating across calls too): its
  // input copy runs on copy_in once the slot's previous use is over, so it
  // overlaps the previous chunk's (or call's) compute; its output copy, if
  // any, runs on copy_out and overlaps the next chunk's compute.  `stream`
  // waits for the last output copies at the end, so synchronising it covers
  // y_host.
  bool used[2] = {false, false};
  for (int c0 = 0; c0 < T; c0 += ctx->cfg.max_chunk_rows) {
    const int n = std::min(ctx->cfg.max_chunk_rows, T - c0);
    const int slot = ctx->host_slot;
    ctx->host_slot ^= 1;
    used[slot] = true;
    void *xs = ctx->ws + ctx->L.x_stage + slot * slot_bytes;
    void *ys = ctx->ws + ctx->L.y_stage + slot * slot_bytes;
    if ((e = cudaStreamWaitEvent(ctx->copy_in, ctx->ev_out[slot], 0)) == cudaSuccess) {
      ProfScope ps(ctx, K_H2D, ctx->copy_in);
      e = cudaMemcpyAsync(xs, static_cast<const char *>(x_host) + c0 * row_bytes, n * row_bytes,
                          cudaMemcpyHostToDevice, ctx->copy_in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_x[slot], ctx->copy_in);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
    if ((e = cudaStreamWaitEvent(s, ctx->ev_x[slot], 0)) != cudaSuccess)
      return cuda_fail(ctx, e, "stream wait");
    st = enqueue_prefill_chunk(ctx, ls, xs, n, y_direct ? y_direct + c0 * row_bytes : ys, s);
    if (st) return st;
    // the slot's input is free once this chunk's kernels are done
    if ((e = cudaEventRecord(y_direct ? ctx->ev_out[slot] : ctx->ev_y[slot], s)) != cudaSuccess)
      return cuda_fail(ctx, e, "event record");
    if (y_direct) continue;
    if ((e = cudaStreamWaitEvent(ctx->copy_out, ctx->ev_y[slot], 0)) == cudaSuccess) {
      ProfScope ps(ctx, K_D2H, ctx->copy_out);
      e = cudaMemcpyAsync(static_cast<char *>(y_host) + c0 * row_bytes, ys, n * row_bytes,
                          cudaMemcpyDeviceToHost, ctx->copy_out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_out[slot], ctx->copy_out);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "device-to-host copy");
  }
  for (int i = 0; i < 2; ++i)
    if (used[i] && (e = cudaStreamWaitEvent(s, ctx->ev_out[i], 0)) != cudaSuccess)
      return cuda_fail(ctx, e, "stream wait");
  return MOE_OK;
}

moe_status moe_forward_decode_host(moe_ctx *ctx, int layer, const void *x_host, void *y_host,
                                   void *stream) {
  moe_status st = check_layer(ctx, layer);
  if (st) return st;
  if (!x_host || !y_host) return fail(ctx, MOE_ERR_INVALID_ARG, "null host buffer");
  if ((st = ensure_device(ctx))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(ctx->cfg.hidden) * 2;
  void *xs = ctx->ws + ctx->L.dec_x_stage;
  void *ys = ctx->ws + ctx->L.dec_y_stage;
  // a page-locked y_host is written by the kernel directly (as in
  // moe_forward_prefill_host)
  void *y_direct = nullptr;
  {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer != nullptr && aligned16(pa.devicePointer))
      y_direct = pa.devicePointer;
    else
      cudaGetLastError();
  }
  cudaError_t e = cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "host-to-device copy");
  st = enqueue_decode(ctx, ctx->layers[layer], xs, y_direct ? y_direct : ys, s);
  if (st || y_direct) return st;
  e = cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(ctx, e, "device-to-host copy");
}

moe_status moe_convert_bf16_to_f16(const void *src, void *dst, size_t n, void *stream) {
  if (n == 0) return MOE_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
  const char *a = static_cast<const char *>(src);
  const char *b = static_cast<const char *>(dst);
  if (a < b + 2 * n && b < a + 2 * n) return MOE_ERR_INVALID_ARG;   // overlap
  return launch_convert_bf16_to_f16(src, dst, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_dequant_int4(const void *codes, const void *scale, const void *bias, void *dst,
                            size_t rows, int K, int wfmt, int out_f16, void *stream) {
  if (rows == 0) return MOE_OK;
  if (wfmt != MOE_W_INT4_SYM_G64 && wfmt != MOE_W_INT4_AFFINE_G64) return MOE_ERR_INVALID_ARG;
  if (K < 64 || K % 64 || !codes || !scale || !dst || !aligned16(codes) || !aligned16(dst) ||
      (reinterpret_cast<uintptr_t>(scale) & 1))
    return MOE_ERR_INVALID_ARG;
  const bool aff = wfmt == MOE_W_INT4_AFFINE_G64;
  if (aff && (!bias || (reinterpret_cast<uintptr_t>(bias) & 1))) return MOE_ERR_INVALID_ARG;
  return launch_dequant_int4(codes, scale, aff ? bias : nullptr, dst, rows, K, aff, out_f16 != 0,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_check_device(moe_ctx *ctx, int32_t *code) {
  if (!ctx) {
    // no context: the status word of moe_forward_decode_noalloc on the
    // current device
    int32_t v = 0;
    if (!noalloc_status_read_clear(&v)) return MOE_ERR_CUDA;
    if (code) *code = v;
    return v != 0 ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
  }
  moe_status st = ensure_device(ctx);
  if (st) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device synchronize");
  int32_t v = 0;
  e = cudaMemcpy(&v, ctx->status(), 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
  if (code) *code = v;
  if (v != 0) {
    cudaMemset(ctx->status(), 0, 4);
    cudaMemset(ctx->ws + ctx->L.dec_counter, 0, 16);   // a timed-out grid barrier
    cudaDeviceSynchronize();
    if (v == kDevRangeH || v == kDevRangeO)
      return fail(ctx, MOE_ERR_RANGE, "prefill %s outside the fp16 range", v == kDevRangeH ? "h" : "o");
    return fail(ctx, MOE_ERR_DEVICE_TIMEOUT, "device wait timed out (site 0x%x)", v);
  }
  return MOE_OK;
}

moe_status moe_profile_enable(moe_ctx *ctx, int on) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (on && !ctx->profiling) {
    const moe_status st = ensure_device(ctx);
    if (st) return st;
    for (int i = 0; i < K_COUNT; ++i) {
      ctx->prof_ms[i] = 0.0;
      ctx->prof_launches[i] = 0;
    }
    // no decode phase stamps from before this point
    const cudaError_t e = cudaMemset(ctx->ws + ctx->L.dec_phase, 0,
                                     static_cast<size_t>(kMaxPhaseCtas) * 2 * 8);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "phase stamp reset");
  }
  ctx->profiling = on != 0;
  return MOE_OK;
}

moe_status moe_profile_read(moe_ctx *ctx, moe_kernel_stat *stats, int max, int *n) {
  if (!ctx || !n || (max > 0 && !stats)) return MOE_ERR_INVALID_ARG;
  moe_status st = ensure_device(ctx);
  if (st) return st;
  for (auto &r : ctx->pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      ctx->prof_ms[r.id] += ms;
      ctx->prof_launches[r.id] += 1;
    }
    ctx->event_pool.push_back(r.a);
    ctx->event_pool.push_back(r.b);
  }
  ctx->pending.clear();
  int cnt = 0;
  for (int i = 0; i < K_COUNT; ++i) {
    if (ctx->prof_launches[i] == 0) continue;
    if (cnt < max) {
      std::memset(&stats[cnt], 0, sizeof(moe_kernel_stat));
      std::snprintf(stats[cnt].name, sizeof(stats[cnt].name), "%s", kKernelNames[i]);
      stats[cnt].launches = ctx->prof_launches[i];
      stats[cnt].total_ms = ctx->prof_ms[i];
    }
    ++cnt;
  }
  *n = cnt;
  return MOE_OK;
}

moe_status moe_decode_phase_read(moe_ctx *ctx, double *window_us, double *median_us) {
  if (!ctx || !window_us || !median_us) return MOE_ERR_INVALID_ARG;
  moe_status st = ensure_device(ctx);
  if (st) return st;
  const int G = ctx->decode_grid;
  if (G <= 0 || G > kMaxPhaseCtas) return fail(ctx, MOE_ERR_UNSUPPORTED, "no phase stamps for this grid");
  std::vector<unsigned long long> ts(static_cast<size_t>(G) * 2);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(ts.data(), ctx->ws + ctx->L.dec_phase, ts.size() * 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "phase stamp read");
  unsigned long long lo = ~0ull, hi = 0;
  std::vector<double> d(static_cast<size_t>(G));
  for (int b = 0; b < G; ++b) {
    const unsigned long long s0 = ts[2 * b], s1 = ts[2 * b + 1];
    if (s0 == 0 || s1 < s0)
      return fail(ctx, MOE_ERR_INVALID_ARG, "no profiled decode launch since profiling was enabled");
    lo = std::min(lo, s0);
    hi = std::max(hi, s1);
    d[b] = static_cast<double>(s1 - s0) * 1e-3;
  }
  std::sort(d.begin(), d.end());
  *window_us = static_cast<double>(hi - lo) * 1e-3;
  *median_us = d[static_cast<size_t>(G) / 2];
  return MOE_OK;
}

int64_t moe_launch_count(const moe_ctx *ctx) { return ctx ? ctx->launches : 0; }

const char *moe_last_error(const moe_ctx *ctx) { return ctx ? ctx->last_error.c_str() : ""; }

}  // extern "C"
