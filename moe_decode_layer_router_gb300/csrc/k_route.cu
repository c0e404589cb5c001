// The route kernel: routing and the token -> expert permute after the
// router's launch (routing rule, top-k and permute: route_dev.cuh). The
// forward chain routes in the router kernel's tail instead; this launch
// serves the routing-only entry points.
#include "route_dev.cuh"

namespace musemoe {

// Grid: with p.central one CTA routes every row (one warp per row) and
// builds the permute from shared memory. Otherwise one CTA per 8 rows, one
// warp per row; the CTA that finishes last (atomic ticket, no waiting)
// builds the permute.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads) k_route(RouteParams p) {
  pdl_launch_dependents();
  // the selection bias is a weight: loaded before the wait for the router
  __shared__ float bias_s[256];
  for (int i = threadIdx.x; i < p.E; i += kRouteThreads) bias_s[i] = __ldg(p.expert_bias + i);
  __syncthreads();
  pdl_wait();
  __shared__ float s_w[kRouteThreads / 32][256];
  __shared__ int top[kRouteThreads / 32][256];
  __shared__ int flag;
  extern __shared__ __align__(16) unsigned char dyn[];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int rt = p.rows * p.k;
  int16_t* ids_s = reinterpret_cast<int16_t*>(dyn);
  unsigned char* work = dyn + (((size_t)rt * 2 + 15) & ~(size_t)15);

  if (p.central) {
    const bool perm = p.route_list != nullptr;
    for (int t = wid; t < p.rows; t += kRouteThreads / 32)
      route_row_warp<EPL>(p, t, lane, s_w[wid], top[wid], perm ? ids_s : nullptr, bias_s);
    if (!perm) return;
    __syncthreads();
    if (rt <= kRouteThreads && p.E <= kRouteThreads) permute_small(p, ids_s);
    else permute(p, ids_s, work);
    return;
  }

  const int t = blockIdx.x * (kRouteThreads / 32) + wid;
  if (t < p.rows) route_row_warp<EPL>(p, t, lane, s_w[wid], top[wid], nullptr, bias_s);
  if (p.route_list == nullptr) return;
  // ---- last CTA: permute --------------------------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(p.counters + kTicket, 1);
    flag = (prev == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!flag) return;
  __threadfence();
  for (int i = tid; i < rt; i += kRouteThreads) ids_s[i] = (int16_t)__ldcg(p.ids + i);
  __syncthreads();
  permute(p, ids_s, work);
}

static size_t route_dyn_smem(const RouteParams& p) {
  if (p.route_list == nullptr) return 16;
  const size_t rt = (size_t)p.rows * p.k;
  const size_t nch = (rt + 31) / 32;
  return ((((rt * 2 + 15) & ~(size_t)15) + ((rt + 15) & ~(size_t)15) + nch * p.E * 2) + 15) &
         ~(size_t)15;
}

template <int EPL>
static cudaError_t launch_route_t(const RouteParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = route_dyn_smem(p);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_route<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.central ? 1 : (p.rows + kRouteThreads / 32 - 1) / (kRouteThreads / 32));
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_route<EPL>, p);
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t s, bool pdl) {
  if (p.E <= 32) return launch_route_t<1>(p, s, pdl);
  if (p.E <= 64) return launch_route_t<2>(p, s, pdl);
  if (p.E <= 128) return launch_route_t<4>(p, s, pdl);
  return launch_route_t<8>(p, s, pdl);
}

}  // namespace musemoe
