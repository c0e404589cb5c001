// musemoe_route_static: the router GEMV + routing rule for callers that
// cannot allocate device memory. Its scratch (the fp32 logits) is a fixed
// file-scope device array, so the call needs no handle and makes no
// allocation. Nothing in it has to start at zero: the router writes every
// logit the routing kernel reads.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "kernels.h"
#include "musemoe.h"

using namespace musemoe;

namespace {

constexpr size_t kLogitsBytes = 64 * 1024;  // rows * E * 4 <= 64 * 256 * 4
static_assert(kLogitsBytes <= MUSEMOE_STATIC_SCRATCH_BYTES, "scratch too small");
constexpr int kMaxDevices = 64;
constexpr int kStaticMaxHidden = 8192;  // the router GEMV's row held in registers

// The scratch. In host code this name is only a stand-in for the device
// array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_route_scratch[MUSEMOE_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

musemoe_status fail(musemoe_status st, const std::string& m) {
  set_thread_error(m);  // read back with musemoe_last_error(NULL)
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" musemoe_status musemoe_route_static(int32_t hidden, int32_t experts, int32_t top_k,
                                               const musemoe_config* config,
                                               const float* w_router, const float* expert_bias,
                                               const uint16_t* x, int32_t rows,
                                               int32_t* ids_out, float* weights_out,
                                               musemoe_stream_t stream) {
  if (!config) return fail(MUSEMOE_EINVAL, "config is NULL");
  if (rows < 1 || rows > MUSEMOE_STATIC_MAX_ROWS)
    return fail(MUSEMOE_EINVAL, "rows " + std::to_string(rows) + " outside 1.." +
                                    std::to_string(MUSEMOE_STATIC_MAX_ROWS) +
                                    " (the static scratch holds at most that many rows)");
  if (experts < 1 || experts > 256)
    return fail(MUSEMOE_EUNSUPPORTED, "experts " + std::to_string(experts) + " outside 1..256");
  if (top_k < 1 || top_k > experts)
    return fail(MUSEMOE_EINVAL, "top_k " + std::to_string(top_k) + " outside 1..experts");
  if (hidden < 64 || hidden % 64)
    return fail(MUSEMOE_EUNSUPPORTED, "hidden " + std::to_string(hidden) + " is not a multiple of 64");
  if (hidden > kStaticMaxHidden)
    return fail(MUSEMOE_EUNSUPPORTED, "hidden " + std::to_string(hidden) + " above " +
                                          std::to_string(kStaticMaxHidden) +
                                          " (a router thread holds at most 32 weights of a row)");
  if (config->score != 0 && config->score != 1)
    return fail(MUSEMOE_EINVAL, "score is not sigmoid (0) or softmax (1)");
  const void* ptrs[] = {w_router, expert_bias, x, ids_out, weights_out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return fail(MUSEMOE_EINVAL, "tensors must be non-NULL and 16-byte aligned");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MUSEMOE_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MUSEMOE_EUNSUPPORTED, "device index out of range");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (st) {
    // the kernels run on the stream's device but write the scratch of the
    // current device: the two must be the same
    int sdev = -1;
    e = cudaStreamGetDevice(st, &sdev);
    if (e != cudaSuccess)
      return fail(MUSEMOE_EINVAL, std::string("cudaStreamGetDevice: ") + cudaGetErrorString(e));
    if (sdev != dev)
      return fail(MUSEMOE_EINVAL, "stream belongs to device " + std::to_string(sdev) +
                                      ", not the current device " + std::to_string(dev));
  }
  void* base = nullptr;
  {
    // first call on this device: look up the array's device address (with
    // the device current); later calls reuse it
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_dev[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_route_scratch);
      if (e != cudaSuccess)
        return fail(MUSEMOE_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      g_scratch_dev[dev] = ptr;
    }
    base = g_scratch_dev[dev];
  }
  float* logits = static_cast<float*>(base);  // [rows, experts]
  FrontParams fp{};
  fp.x = x;
  fp.rows = rows;
  fp.w_router = w_router;
  fp.logits = logits;
  fp.E = experts;
  fp.router_ctas = experts * ((rows + 7) / 8);
  fp.K = hidden;
  e = launch_router(fp, st, false);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MUSEMOE_ECUDA, std::string("launch of router: ") + cudaGetErrorString(e));
  RouteParams rp{};
  rp.logits = logits;
  rp.expert_bias = expert_bias;
  rp.ids = ids_out;
  rp.weights = weights_out;
  rp.rows = rows;
  rp.E = experts;
  rp.k = top_k;
  rp.score = config->score;
  rp.has_multiplier = config->has_multiplier;
  rp.multiplier = config->multiplier;
  rp.has_division_eps = config->has_division_eps;
  rp.division_eps = config->division_eps;
  rp.route_scale = config->route_scale;
  rp.central = rows <= 32;
  e = launch_route(rp, st, true);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MUSEMOE_ECUDA, std::string("launch of route: ") + cudaGetErrorString(e));
  return MUSEMOE_OK;
}
