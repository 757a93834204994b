// Batch-1 decode without a context or workspace, for callers that cannot
// allocate device memory: for example code running inside a host framework
// whose allocator forbids allocations on this path (a captured or
// latency-critical section, a plugin that only receives the caller's
// buffers), or a process whose device-memory budget is fixed up front.
//
// The per-token intermediates of the decode kernel (router logits, the
// selected experts and their weights, the shared-expert gate, the experts'
// gate/up dot products, the shared expert's activations, and the grid-barrier
// words) live in one file-scope device array instead of a workspace.  The
// array is part of the loaded library: every device that loads it holds
// kNoAllocScratchBytes until the process exits.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sparse_moe.h"
#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64 * 1024;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char *g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device
int g_grid[kMaxDevices] = {};                       // cooperative decode grid, per device
int g_smem_limit[kMaxDevices] = {};                 // decode kernel's shared-memory limit, per device
int g_pdl[kMaxDevices] = {};                        // 1 + programmatic dependent launch flag, per device

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct ScratchLayout {
  size_t logits, idx, w, g, h, counter, status, total;
};

// The status word sits at a fixed offset (the start of the array), whatever
// the shape of the call that wrote it, so that it can be read without one.
constexpr size_t kStatusOffset = 0;

ScratchLayout scratch_layout(const moe_config &c) {
  ScratchLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t imax = static_cast<size_t>(c.inter > c.shared_inter ? c.inter : c.shared_inter);
  L.status = take(16);
  L.logits = take(static_cast<size_t>(c.n_experts) * 4);
  L.idx = take(static_cast<size_t>(c.top_k) * 4);
  L.w = take(static_cast<size_t>(c.top_k) * 4);
  L.g = take(4);
  L.h = take(moe::decode_h_floats(c.top_k, static_cast<int>(imax)) * 4);
  L.counter = take(16);
  L.total = off;
  return L;
}

bool config_ok(const moe_config *c) {
  if (!c) return false;
  if (c->hidden < 64 || c->hidden > 16384 || c->hidden % 64) return false;
  if (c->n_experts < 1 || c->n_experts > 1024) return false;
  if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > 32) return false;
  if (c->inter < 64 || c->inter % 64 || c->shared_inter < 64 || c->shared_inter % 64) return false;
  if (c->inter > 16384 || c->shared_inter > 16384) return false;
  if (c->wfmt != MOE_W_BF16 && c->wfmt != MOE_W_INT4_SYM_G64 && c->wfmt != MOE_W_INT4_AFFINE_G64)
    return false;
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_forward_decode_noalloc(const moe_config *cfg, const moe_weights *w,
                                                 const void *x, void *y, void *stream) {
  if (!config_ok(cfg) || !w || !x || !y || !aligned16(x) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const void *req[] = {w->router_w, w->gate_up, w->down, w->sh_gate_up, w->sh_down, w->sh_gate_w};
  for (const void *p : req)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->wfmt != MOE_W_BF16 &&
      (!w->gate_up_scale || !w->down_scale || !w->sh_gate_up_scale || !w->sh_down_scale))
    return MOE_ERR_INVALID_ARG;
  if (cfg->wfmt == MOE_W_INT4_AFFINE_G64 &&
      (!w->gate_up_bias || !w->down_bias || !w->sh_gate_up_bias || !w->sh_down_bias))
    return MOE_ERR_INVALID_ARG;
  const ScratchLayout L = scratch_layout(*cfg);
  if (L.total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;   // beyond the fixed scratch
  const int imax = cfg->inter > cfg->shared_inter ? cfg->inter : cfg->shared_inter;
  if ((cfg->top_k + 1) * imax * 4 > 200 * 1024) return MOE_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  unsigned char *base = nullptr;
  int grid = 0, smem_limit = 0;
  bool pdl = true;
  {
    // Set-up, once per device and with that device current: the host-side
    // name of the array is not a device address, so ask the runtime for it.
    // What is cached here (the address, the grid, the shared-memory opt-in)
    // belongs to the device's primary context: it stays valid as long as the
    // process keeps that context (no cudaDeviceReset in between).
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
      g_scratch_addr[dev] = static_cast<unsigned char *>(ptr);
    }
    if (!g_grid[dev]) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return MOE_ERR_CUDA;
      g_grid[dev] = moe::decode_layer_grid(sms);
    }
    if (!g_smem_limit[dev]) {
      int limit = 0;
      if (moe::decode_configure(&limit) != cudaSuccess) return MOE_ERR_CUDA;
      g_smem_limit[dev] = limit;
    }
    if (!g_pdl[dev]) {
      // the same switch as a context's decode launches (MOE_DECODE_PDL=0
      // turns programmatic dependent launch off), read once per device
      const char *env = std::getenv("MOE_DECODE_PDL");
      g_pdl[dev] = 1 + ((env && std::atoi(env) == 0) ? 0 : 1);
    }
    base = g_scratch_addr[dev];
    grid = g_grid[dev];
    smem_limit = g_smem_limit[dev];
    pdl = g_pdl[dev] == 2;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The grid-barrier counter must start at a multiple of the grid (zero);
  // everything else is written before it is read within the call.
  if (cudaMemsetAsync(base + L.counter, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;

  moe::DecodeParams p{};
  p.x = x;
  p.y = y;
  p.H = cfg->hidden;
  p.E = cfg->n_experts;
  p.k = cfg->top_k;
  p.I = cfg->inter;
  p.Is = cfg->shared_inter;
  p.wfmt = cfg->wfmt;
  p.router_w = w->router_w;
  p.router_b = w->router_b;
  p.gate_up = w->gate_up;
  p.gate_up_scale = w->gate_up_scale;
  p.down = w->down;
  p.down_scale = w->down_scale;
  p.sh_gate_up = w->sh_gate_up;
  p.sh_gate_up_scale = w->sh_gate_up_scale;
  p.sh_down = w->sh_down;
  p.sh_down_scale = w->sh_down_scale;
  p.sh_gate_w = w->sh_gate_w;
  p.gate_up_bias = w->gate_up_bias;
  p.down_bias = w->down_bias;
  p.sh_gate_up_bias = w->sh_gate_up_bias;
  p.sh_down_bias = w->sh_down_bias;
  p.logits = reinterpret_cast<float *>(base + L.logits);
  p.idx = reinterpret_cast<int32_t *>(base + L.idx);
  p.w = reinterpret_cast<float *>(base + L.w);
  p.g = reinterpret_cast<float *>(base + L.g);
  p.h = reinterpret_cast<float *>(base + L.h);
  p.h_ld = imax;
  p.bar = reinterpret_cast<unsigned long long *>(base + L.counter);
  p.status = reinterpret_cast<int *>(base + L.status);
  if (moe::launch_decode_layer(p, grid, smem_limit, pdl, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

namespace moe {

// Status word of the allocation-free decode on the current device (see
// moe_check_device with a null context): waits for the device, then reads
// the word and clears it.  (The grid-barrier counter needs no clearing: every
// call zeroes it before its launch.)  Returns false if a CUDA call fails.
bool noalloc_status_read_clear(int32_t *code) {
  *code = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return false;
  int32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_scratch, sizeof(v), kStatusOffset) != cudaSuccess)
    return false;
  if (v != 0) {
    const int32_t zero = 0;
    if (cudaMemcpyToSymbol(g_decode_scratch, &zero, sizeof(zero), kStatusOffset) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return false;
  }
  *code = v;
  return true;
}

}  // namespace moe
