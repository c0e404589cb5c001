// Routing of one row per warp and the token -> expert permute, shared by the
// route kernel and the router kernel's tail.
//
// Routing rule (page "vllm.models.muse_spark.amd.muse_moe_runner", class
// MuseSpark1xRouter, docstring and _compute_routing_native): optional output
// multiplier -> sigmoid or softmax -> expert bias added for SELECTION only ->
// top-k -> gather the UNBIASED scores -> divide by (sum + division_eps) ->
// multiply by route_scale. All in fp32, as the recipe's torch ops are.
// Top-k: one warp per row takes k rounds of a warp-wide argmax over the E
// (<= 256) selection keys (largest score first, the lower id on equal
// scores).
//
// Permute: the routes per expert, written grouped by expert in route order
// (a stable counting sort), then the token groups the expert kernels walk.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace musemoe {

constexpr int kRouteThreads = 256;

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one int per thread (blockDim.x == kRouteThreads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < kRouteThreads / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kRouteThreads / 32) scratch[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before = wid ? scratch[wid - 1] : 0;
  *total = scratch[kRouteThreads / 32 - 1];
  return before + x - v;
}

// One warp routes row t: scores from the fp32 logits, selection keys, the
// top-k as k rounds of a warp argmax, then the weights from the UNBIASED scores of the selected
// ids. `s_w` (E floats) and `top` (k ints) are the warp's shared scratch.
template <int EPL>
__device__ void route_row_warp(const RouteParams& p, int t, int lane, float* s_w, int* top,
                               int16_t* ids_smem, const float* bias_s) {
  const int E = p.E, k = p.k;
  float g[EPL], bias[EPL];
#pragma unroll
  for (int r = 0; r < EPL; ++r) {
    const int i = lane * EPL + r;
    g[r] = (i < E) ? __ldcg(p.logits + (size_t)t * E + i) : -INFINITY;
    bias[r] = (i < E) ? bias_s[i] : 0.f;
  }
  float gmax = -INFINITY;
#pragma unroll
  for (int r = 0; r < EPL; ++r) {
    const int i = lane * EPL + r;
    if (p.has_multiplier && i < E) g[r] = g[r] * p.multiplier;
    gmax = fmaxf(gmax, g[r]);
  }
  float sc[EPL];
  if (p.score == 1) {  // softmax over the experts
    gmax = warp_max(gmax);
    float part = 0.f;
#pragma unroll
    for (int r = 0; r < EPL; ++r) {
      sc[r] = (lane * EPL + r < E) ? expf(g[r] - gmax) : 0.f;
      part += sc[r];
    }
    const float tot = warp_sum(part);
#pragma unroll
    for (int r = 0; r < EPL; ++r) sc[r] = sc[r] / tot;
  } else {
#pragma unroll
    for (int r = 0; r < EPL; ++r) sc[r] = 1.0f / (1.0f + expf(-g[r]));
  }
  // selection keys; 0 marks padding and experts already taken (a real key
  // is at least 1)
  uint32_t key[EPL];
#pragma unroll
  for (int r = 0; r < EPL; ++r) {
    const int i = lane * EPL + r;
    if (i < E) {
      s_w[i] = sc[r];
      const float sel = sc[r] + bias[r];  // selection only
      key[r] = max(orderable(sel), 1u);
    } else {
      key[r] = 0u;
    }
  }
  // top-k: k rounds of a warp argmax, the largest key and, among equal
  // keys, the lowest id (the order a descending sort by (key, -id) gives)
  for (int j = 0; j < k; ++j) {
    uint32_t lm = 0u;
#pragma unroll
    for (int r = 0; r < EPL; ++r) lm = max(lm, key[r]);
    const uint32_t m = __reduce_max_sync(0xffffffffu, lm);
    uint32_t cand = 0xffffffffu;
#pragma unroll
    for (int r = EPL - 1; r >= 0; --r)
      if (key[r] == m) cand = (uint32_t)(lane * EPL + r);
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
#pragma unroll
    for (int r = 0; r < EPL; ++r)
      if ((uint32_t)(lane * EPL + r) == win) key[r] = 0u;
    if (lane == 0) top[j] = (int)win;
  }
  __syncwarp();
  float part = 0.f;
  for (int i = lane; i < k; i += 32) part += s_w[top[i]];
  float denom = warp_sum(part);
  if (p.has_division_eps) denom += p.division_eps;
  for (int i = lane; i < k; i += 32) {
    const int e = top[i];
    p.ids[(size_t)t * k + i] = e;
    p.weights[(size_t)t * k + i] = s_w[e] / denom * p.route_scale;
    if (ids_smem) ids_smem[(size_t)t * k + i] = (int16_t)e;
  }
  __syncwarp();
}

// Token -> expert permute from the ids in ids_s (shared): counts per expert,
// routes grouped by expert in route order (a stable counting sort), then the
// token groups the expert kernels walk.
static __device__ void permute(const RouteParams& p, int16_t* ids_s, unsigned char* work) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int E = p.E, rt = p.rows * p.k;
  const int nch = (rt + 31) / 32;
  uint8_t* rank_s = work;
  uint16_t* hist = reinterpret_cast<uint16_t*>(rank_s + ((rt + 15) & ~15));
  __shared__ int cnt_s[256], off_s[257], goff_s[257];
  __shared__ int scan_scratch[32];

  for (int i = tid; i < nch * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();
  // per 32-route chunk: rank of each route among equal experts, chunk counts
  for (int c = wid; c < nch; c += kRouteThreads / 32) {
    const int r = c * 32 + lane;
    const int e = r < rt ? (int)ids_s[r] : E + lane;  // pads never match
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (r < rt) {
      rank_s[r] = (uint8_t)rank;
      if (rank == 0) hist[c * E + e] = (uint16_t)__popc(peers);
    }
  }
  __syncthreads();
  // per expert: exclusive prefix over chunks
  for (int e = tid; e < E; e += kRouteThreads) {
    int run = 0;
    for (int c = 0; c < nch; ++c) {
      const int t = hist[c * E + e];
      hist[c * E + e] = (uint16_t)run;
      run += t;
    }
    cnt_s[e] = run;
  }
  __syncthreads();
  // offsets of experts, and of their token groups
  const int ep_lo = p.ep_count > 0 ? p.ep_first : 0;
  const int ep_hi = p.ep_count > 0 ? p.ep_first + p.ep_count : E;
  {
    const int e = tid;
    const int c = e < E ? cnt_s[e] : 0;
    // token groups of this rank's experts only
    const int ng = (e >= ep_lo && e < ep_hi) ? (c + p.token_group - 1) / p.token_group : 0;
    int tot;
    const int off = block_exclusive_scan(c, scan_scratch, &tot);
    if (e < E) off_s[e] = off;
    if (e == 0) off_s[E] = tot;
    int gtot;
    const int goff = block_exclusive_scan(ng, scan_scratch, &gtot);
    if (e < E) goff_s[e] = goff;
    if (e == 0) goff_s[E] = gtot;
  }
  __syncthreads();
  for (int r = tid; r < rt; r += kRouteThreads) {
    const int e = ids_s[r];
    p.route_list[off_s[e] + hist[(r >> 5) * E + e] + rank_s[r]] = r;
  }
  for (int e = tid; e < E; e += kRouteThreads) {
    if (e < ep_lo || e >= ep_hi) continue;
    const int c = cnt_s[e];
    for (int gi = 0, s = 0; s < c; ++gi, s += p.token_group) {
      int4 gd = make_int4(e - ep_lo, off_s[e] + s, min(p.token_group, c - s), 0);
      reinterpret_cast<int4*>(p.groups)[goff_s[e] + gi] = gd;
    }
  }
  if (tid == 0) {
    p.counters[kNumGroups] = goff_s[E];
    p.counters[kTicket] = 0;
  }
}

// The permute for at most kRouteThreads routes (and experts): one pass over
// the ids in shared memory gives each route its slot (routes of lower
// experts, then earlier routes of its own expert) and each expert its count
// and first slot; the same stable counting sort as permute().
static __device__ void permute_small(const RouteParams& p, const int16_t* ids_s) {
  const int tid = threadIdx.x;
  const int E = p.E, rt = p.rows * p.k;
  __shared__ int scan_scratch[32];
  const int my_e = tid < rt ? (int)ids_s[tid] : -1;
  int rank = 0, cnt = 0, first = 0;
  for (int r = 0; r < rt; ++r) {
    const int e2 = ids_s[r];
    rank += (e2 < my_e) | ((e2 == my_e) & (r < tid));
    cnt += (e2 == tid);
    first += (e2 < tid);
  }
  if (tid < rt) p.route_list[rank] = tid;
  const int ep_lo = p.ep_count > 0 ? p.ep_first : 0;
  const int ep_hi = p.ep_count > 0 ? p.ep_first + p.ep_count : E;
  const bool local = tid < E && tid >= ep_lo && tid < ep_hi;  // token groups of this rank's experts
  const int ng = local ? (cnt + p.token_group - 1) / p.token_group : 0;
  int gtot;
  const int goff = block_exclusive_scan(ng, scan_scratch, &gtot);
  for (int gi = 0, s = 0; s < cnt && local; ++gi, s += p.token_group)
    reinterpret_cast<int4*>(p.groups)[goff + gi] =
        make_int4(tid - ep_lo, first + s, min(p.token_group, cnt - s), 0);
  if (tid == 0) {
    p.counters[kNumGroups] = gtot;
    p.counters[kTicket] = 0;
  }
}

}  // namespace musemoe
