// C ABI of the musemoe library: validation, workspace and the launch chain.
// See include/musemoe.h for the contract of every entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <new>
#include <string>
#include <vector>

#include "kernels.h"
#include "musemoe.h"

using namespace musemoe;

namespace {

thread_local std::string g_thread_err;

std::string fmt(const char* f, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, f);
  vsnprintf(buf, sizeof buf, f, ap);
  va_end(ap);
  return buf;
}

constexpr int kMaxRoutes = 4096;  // rows * top_k served by the permute
constexpr size_t kAlign = 256;
constexpr int kExpertCtasPerSm = 2;  // expert kernels: resident CTAs per SM, at most
constexpr size_t kPackTmpBytes = 64ull << 20;  // in-place pack: tiles per pass

int nt_front(int rows) { return rows <= 8 ? 1 : rows <= 16 ? 2 : 4; }
// Token tile of the expert kernels (8 * NT routes per group). Up to 32 rows
// an expert rarely gets more than 8 routes, and one that does becomes two
// groups (its weights stream twice), cheaper than wider, mostly empty tiles.
int nt_expert(int rows) { return rows <= 32 ? 1 : rows <= 64 ? 4 : 8; }
int nt_index(int nt) { return nt == 1 ? 0 : nt == 2 ? 1 : nt == 4 ? 2 : 3; }
// Above this many rows an expert's token group is a dense contraction
// (dozens of tokens per hot expert): the tensor-core (tcgen05) expert kernels
// take MXFP4, NVFP4, FP8 and the W4A4 forms there.
constexpr int kTcMinRows = 33;

// Router CTAs: one per (expert, block of 8 tokens).
int router_ctas(int E, int rows) { return E * ((rows + 7) / 8); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

void musemoe::set_thread_error(const std::string& m) { g_thread_err = m; }

struct musemoe_handle {
  musemoe_dims d{};
  int quant = 0;  // the weight format (Quant)
  int expert_path = 0;  // MUSEMOE_PATH_AUTO / _MMA / _TCGEN05
  int act4 = 0;   // W4A4: expert inputs rounded to MXFP4 (1) or NVFP4 (2)
  musemoe_config cfg{};
  int device = -1, sms = 0;
  int max_routes = 0, max_groups = 0;
  int expert_grid[2][4] = {};
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // workspace views
  float *logits = nullptr, *weights = nullptr, *h_scale = nullptr, *act_scale = nullptr;
  float *h_raw = nullptr, *u = nullptr;
  float *y = nullptr, *stream_stage = nullptr, *expert_part = nullptr;
  int32_t* expert_tickets[2] = {nullptr, nullptr};
  size_t expert_ticket_bytes[2] = {0, 0};
  size_t block_ticket_bytes = 0;  // norm_ticket and route_ticket, each
  int32_t* norm_ticket = nullptr;
  int32_t *route_ticket = nullptr, *route_done = nullptr;
  int32_t* never_set = nullptr;  // zero for good: the health self-test's flag
  int32_t *ids = nullptr, *route_list = nullptr, *groups = nullptr, *counters = nullptr;
  int32_t* health = nullptr;
  uint16_t *h = nullptr, *moe_out = nullptr, *x_stage = nullptr, *out_stage = nullptr;
  uint8_t *h_op = nullptr, *act = nullptr, *act_q = nullptr;
  uint8_t *h_sf = nullptr, *act_sf = nullptr;  // W4A4: block scales of h_op / act_q
  std::string err;
};

namespace {

// public quant code -> the weights' format and the W4A4 activation rounding
constexpr int kMXFP4_A4 = 4, kNVFP4_A4 = 5;
int weight_format(int q) { return q == kMXFP4_A4 ? kMXFP4 : q == kNVFP4_A4 ? kNVFP4 : q; }
int act4_of(int q) { return q == kMXFP4_A4 ? 1 : q == kNVFP4_A4 ? 2 : 0; }

struct Layout {
  size_t off = 0;
  std::vector<std::pair<void**, size_t>> items;
  template <typename T>
  void add(T** p, size_t bytes) {
    items.push_back({reinterpret_cast<void**>(p), off});
    off += (bytes + kAlign - 1) / kAlign * kAlign;
  }
};

void plan(musemoe_handle* h, Layout& L) {
  const musemoe_dims& d = h->d;
  const size_t R = d.max_rows, E = d.experts, H = d.hidden, P = d.pooled, I = d.inter;
  const size_t RT = R * d.top_k;
  const bool fp8 = h->quant == kFP8;
  L.add(&h->logits, R * E * 4);
  L.add(&h->h_raw, R * P * 4);
  L.add(&h->u, R * H * 4);
  L.add(&h->ids, RT * 4);
  L.add(&h->weights, RT * 4);
  L.add(&h->h, R * P * 2);
  if (h->act4) {
    L.add(&h->h_op, R * P / 2);   // W4A4: h's e2m1 codes
    L.add(&h->h_sf, R * P / 16);  // and its block scales (one per 16 at most)
  } else {
    L.add(&h->h_op, R * P * (fp8 ? 1 : 2));
  }
  L.add(&h->h_scale, R * 4);
  L.add(&h->route_list, RT * 4);
  L.add(&h->groups, (size_t)h->max_groups * 16);
  L.add(&h->counters, kNumCounters * 4);
  h->block_ticket_bytes = (R + 7) / 8 * 4;
  L.add(&h->norm_ticket, h->block_ticket_bytes);   // one per pooler token block
  L.add(&h->route_ticket, h->block_ticket_bytes);  // one per router token block
  L.add(&h->route_done, 4);
  L.add(&h->never_set, 4);
  L.add(&h->health, 16);
  L.add(&h->act, RT * I * 2);
  if (fp8) {
    L.add(&h->act_q, RT * I);
    L.add(&h->act_scale, RT * 4);
  } else if (h->act4) {
    L.add(&h->act_q, RT * I / 2);    // w2's e2m1 codes
    L.add(&h->act_sf, RT * I / 16);  // and block scales
  }
  L.add(&h->y, RT * P * 4);
  // Stream-K partial sums (shared by w13 and w2, which run one after the
  // other) for the widest token tile, and one ticket array per matrix; at
  // most kExpertCtasPerSm CTAs per SM
  const int nt_max = nt_expert(d.max_rows);
  L.add(&h->expert_part, std::max(expert_part_bytes(kExpertCtasPerSm * h->sms, nt_max),
                                  expert_tc_part_bytes(h->sms)));
  h->expert_ticket_bytes[0] = expert_tickets(h->max_groups, h->quant, 0, d.pooled, 2 * d.inter) * 4;
  h->expert_ticket_bytes[1] = expert_tickets(h->max_groups, h->quant, 1, d.inter, d.pooled) * 4;
  L.add(&h->expert_tickets[0], h->expert_ticket_bytes[0]);
  L.add(&h->expert_tickets[1], h->expert_ticket_bytes[1]);
  L.add(&h->moe_out, R * P * 2);
  L.add(&h->x_stage, R * H * 2);
  L.add(&h->stream_stage, R * H * 4);
  L.add(&h->out_stage, R * H * 2);
}

std::vector<std::string> refusals(const musemoe_dims* d, int32_t quant, const musemoe_config* c) {
  std::vector<std::string> r;
  if (d->max_rows < 1) r.push_back(fmt("max_rows %d < 1", d->max_rows));
  if (d->hidden < 64 || d->hidden % 64) r.push_back(fmt("hidden %d is not a multiple of 64", d->hidden));
  if (d->pooled < 128 || d->pooled % 128)
    r.push_back(fmt("pooled %d is not a multiple of 128", d->pooled));
  if (d->inter < 128 || d->inter % 128) r.push_back(fmt("inter %d is not a multiple of 128", d->inter));
  if (d->experts < 1 || d->experts > 256)
    r.push_back(fmt("experts %d outside 1..256 (the register top-k)", d->experts));
  if (d->top_k < 1 || d->top_k > d->experts)
    r.push_back(fmt("top_k %d outside 1..experts (%d)", d->top_k, d->experts));
  if ((long long)d->max_rows * d->top_k > kMaxRoutes)
    r.push_back(fmt("max_rows * top_k = %lld exceeds %d routes", (long long)d->max_rows * d->top_k,
                    kMaxRoutes));
  if ((size_t)d->pooled * 4 > 200 * 1024) r.push_back(fmt("pooled %d too large for one CTA row", d->pooled));
  if (d->hidden > front_max_k())
    r.push_back(fmt("hidden %d above %d (a pooler row tile held in shared memory)", d->hidden, front_max_k()));
  if (d->pooled > front_max_k())
    r.push_back(fmt("pooled %d above %d (an unpooler row tile held in shared memory)", d->pooled, front_max_k()));
  if (quant < 0 || quant > 5)
    r.push_back(fmt("quant %d is not MXFP4 (0), NVFP4 (1), FP8_W8A8 (2), BF16 (3), "
                    "MXFP4_A4 (4) or NVFP4_A4 (5)", quant));
  if (c->score != 0 && c->score != 1) r.push_back(fmt("score %d is not sigmoid (0) or softmax (1)", c->score));
  if (!std::isfinite(c->route_scale)) r.push_back("route_scale is not finite");
  if (c->has_multiplier && !std::isfinite(c->multiplier)) r.push_back("multiplier is not finite");
  if (c->has_division_eps && !(c->division_eps >= 0.f)) r.push_back("division_eps < 0");
  if (!(c->norm_eps >= 0.f)) r.push_back("norm_eps < 0");
  return r;
}

std::string join(const std::vector<std::string>& v) {
  std::string s;
  for (size_t i = 0; i < v.size(); ++i) s += (i ? "; " : "") + v[i];
  return s;
}

musemoe_status set_err(musemoe_handle* h, musemoe_status st, const std::string& m) {
  if (h) h->err = m;
  else g_thread_err = m;
  return st;
}

musemoe_status cuda_err(musemoe_handle* h, cudaError_t e, const char* what) {
  return set_err(h, MUSEMOE_ECUDA, fmt("%s: %s", what, cudaGetErrorString(e)));
}

// Returns an error text, or empty when the weights are usable.
std::string check_weights(const musemoe_handle* h, const musemoe_weights* w, bool route_only) {
  if (!w) return "weights is NULL";
  std::vector<std::string> bad;
  auto need = [&](const void* p, const char* name) {
    if (!p) bad.push_back(fmt("%s is NULL", name));
    else if (!aligned16(p)) bad.push_back(fmt("%s is not 16-byte aligned", name));
  };
  need(w->w_router, "w_router");
  need(w->expert_bias, "expert_bias");
  if (!route_only) {
    need(w->w_pool, "w_pool");
    need(w->w_pre_norm, "w_pre_norm");
    need(w->w13, "w13");
    if (h->quant != kBF16) need(w->w13_scale, "w13_scale");
    need(w->w2, "w2");
    if (h->quant != kBF16) need(w->w2_scale, "w2_scale");
    if (h->quant == kNVFP4) {
      need(w->w13_gscale, "w13_gscale");
      need(w->w2_gscale, "w2_gscale");
    }
    need(w->w_post_norm, "w_post_norm");
    need(w->w_unpool, "w_unpool");
    need(w->w_ffn_norm, "w_ffn_norm");
    need(w->w_next_norm, "w_next_norm");
    need(w->gate, "gate");
  }
  return join(bad);
}

// Whether a forward of `rows` runs the pooler and unpooler as dense
// tensor-core GEMMs (the same rows as the expert kernels' dense buckets).
bool use_dense_tc(int rows) { return rows >= kTcMinRows; }

// W4A4: h (bf16, written by the pooler's norm) rounded per token to the
// weights' FP4 format, e2m1 codes into h_op and block scales into h_sf (the
// per-route rounding kernel, one warp per 256 elements of a row).
cudaError_t launch_h_fp4(const musemoe_handle* h, int rows, cudaStream_t s, bool pdl) {
  ActQuantParams q{};
  q.act = h->h;
  q.q = h->h_op;
  q.sf = h->h_sf;
  q.routes = rows;
  q.I = h->d.pooled;
  q.mode = h->act4;
  q.health = h->health;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? launch_act_quant(q, s, pdl) : e;
}

// Whether a forward of `rows` runs its experts on the tensor-core kernels.
bool use_tc(const musemoe_handle* h, int rows) {
  if (h->act4) return true;  // W4A4: the FP4 tensor cores at every size
  if (h->quant == kBF16 || h->expert_path == MUSEMOE_PATH_MMA) return false;
  return h->expert_path == MUSEMOE_PATH_TCGEN05 || rows >= kTcMinRows;
}

// Expert parallelism: the forward runs this rank's experts [first, first +
// count) only and stops after the finalize, which writes the fp32 partial.
struct EpArgs {
  int first, count;
  float* part;
};

musemoe_status launch_back(musemoe_handle* h, const musemoe_weights* w, float* stream,
                           uint16_t* out, int rows, cudaStream_t s, bool pdl,
                           const std::function<void()>& before,
                           const std::function<bool(cudaError_t, const char*)>& after);

musemoe_status launch_chain(musemoe_handle* h, const musemoe_weights* w, const uint16_t* x,
                            float* stream, uint16_t* out, int rows, cudaStream_t s,
                            const musemoe_taps* taps, const EpArgs* epa = nullptr) {
  const musemoe_dims& d = h->d;
  musemoe_event_t* ev = taps ? taps->events : nullptr;
  const bool pdl = (ev == nullptr);
  int ki = 0;
  cudaError_t e = cudaSuccess;
  bool bad_event = false;
  auto before = [&]() {
    if (ev && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[2 * ki]), s) != cudaSuccess)
      bad_event = true;
  };
  auto after = [&](cudaError_t r, const char* name) -> bool {
    if (r == cudaSuccess) r = cudaGetLastError();
    if (r != cudaSuccess) {
      e = r;
      h->err = fmt("launch of %s failed: %s", name, cudaGetErrorString(r));
      return false;
    }
    if (ev && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[2 * ki + 1]), s) != cudaSuccess)
      bad_event = true;
    ++ki;
    return true;
  };

  // 1. router GEMV; its tail routes each 8-token block and builds the
  // permute (the last CTA of a block, then the last block: no waiting)
  const int ntf = nt_front(rows);
  const int nte = nt_expert(rows);
  const bool tc = use_tc(h, rows);
  FrontParams fp{};
  fp.x = x;
  fp.rows = rows;
  fp.w_router = w->w_router;
  fp.logits = h->logits;
  fp.E = d.experts;
  fp.router_ctas = router_ctas(d.experts, rows);
  fp.w = w->w_pool;
  fp.y = h->h_raw;
  fp.health = h->health;
  fp.M = d.pooled;
  fp.K = d.hidden;
  fp.gemv_ctas = front_gemv_ctas(d.pooled, rows, ntf);
  fp.w_pre_norm = w->w_pre_norm;
  fp.pre_norm = h->cfg.pre_expert_norm;
  fp.quant = h->quant;
  fp.act4 = h->act4;
  fp.norm_eps = h->cfg.norm_eps;
  fp.h = h->h;
  fp.h_op = h->h_op;
  fp.h_sf = h->h_sf;
  fp.h_scale = h->h_scale;
  fp.norm_ticket = h->norm_ticket;
  // one CTA normalizes a token block in the GEMV's tail only for 8 rows;
  // wider blocks (16 or 32 rows) take the norm launch, eight rows per CTA
  fp.norm_in_tail = ntf == 1;
  fp.route_tail = 1;
  fp.route_ticket = h->route_ticket;
  fp.route_done = h->route_done;
  RouteParams& rp = fp.route;
  rp.logits = h->logits;
  rp.expert_bias = w->expert_bias;
  rp.ids = h->ids;
  rp.weights = h->weights;
  rp.rows = rows;
  rp.E = d.experts;
  rp.k = d.top_k;
  rp.score = h->cfg.score;
  rp.has_multiplier = h->cfg.has_multiplier;
  rp.multiplier = h->cfg.multiplier;
  rp.has_division_eps = h->cfg.has_division_eps;
  rp.division_eps = h->cfg.division_eps;
  rp.route_scale = h->cfg.route_scale;
  rp.route_list = h->route_list;
  rp.groups = h->groups;
  rp.counters = h->counters;
  rp.health = h->health;
  rp.token_group = tc ? expert_tc_group_tokens() : 8 * nte;
  rp.central = 0;
  rp.ep_first = epa ? epa->first : 0;
  rp.ep_count = epa ? epa->count : 0;
  before();
  if (!after(launch_router(fp, s, pdl), "router")) return MUSEMOE_ECUDA;

  // 2. pooler GEMV (its weight copies overlap the router); for 8 rows the
  // last CTA applies the pre-expert norm to them, for 16 or 32 rows the norm
  // is its own launch. Above 32 rows: a dense tensor-core GEMM, then the
  // norm launch
  const bool dense = use_dense_tc(rows);
  if (dense) {
    DenseParams dp{};
    dp.x = x;
    dp.w = w->w_pool;
    dp.y = h->h_raw;
    dp.rows = rows;
    dp.M = d.pooled;
    dp.K = d.hidden;
    dp.x_ready = 1;  // x is the router's input, final before the router's launch
    dp.health = h->health;
    dp.grid = h->sms;
    // one "pool" stage of the taps' events: the GEMM and the norm launch
    // (W4A4: and the FP4 rounding of h)
    before();
    cudaError_t r = launch_dense_tc(dp, s, pdl);
    if (r == cudaSuccess) r = cudaGetLastError();
    if (r == cudaSuccess) r = launch_pool_norm(fp, s, pdl);
    if (r == cudaSuccess && h->act4) r = launch_h_fp4(h, rows, s, pdl);
    if (!after(r, "pool")) return MUSEMOE_ECUDA;
  } else {
    before();
    cudaError_t r = launch_front(fp, ntf, s, pdl);
    if (r == cudaSuccess && !fp.norm_in_tail) r = launch_pool_norm(fp, s, pdl);
    if (r == cudaSuccess && h->act4) r = launch_h_fp4(h, rows, s, pdl);
    if (!after(r, "pool")) return MUSEMOE_ECUDA;
  }

  // 3. w13 + SiLU * up
  ExpertParams ep{};
  ep.quant = h->quant;
  ep.role = 0;
  ep.E = d.experts;
  ep.N = 2 * d.inter;
  ep.K = d.pooled;
  ep.I = d.inter;
  ep.P = d.pooled;
  ep.k = d.top_k;
  ep.w = w->w13;
  ep.scale = w->w13_scale;
  ep.gscale = w->w13_gscale;
  ep.b = h->quant == kBF16 ? reinterpret_cast<const uint8_t*>(h->h) : h->h_op;  // BF16: h itself
  ep.b_scale = h->h_scale;
  ep.act4 = h->act4;
  ep.b_sf = h->h_sf;
  ep.b_by_token = 1;
  ep.route_list = h->route_list;
  ep.groups = h->groups;
  ep.counters = h->counters;
  ep.out = h->act;
  ep.act_bf16 = h->act4 != 0;
  ep.health = h->health;
  ep.part = h->expert_part;
  ep.tickets = h->expert_tickets[0];
  ep.grid = tc ? h->sms : h->expert_grid[0][nt_index(nte)];
  before();
  if (!after(tc ? launch_expert_tc(ep, s, pdl) : launch_expert(ep, nte, s, pdl), "w13"))
    return MUSEMOE_ECUDA;

  // 3b. FP8 and W4A4: quantize the activation per route
  if (h->quant == kFP8 || h->act4) {
    ActQuantParams aq{};
    aq.act = reinterpret_cast<const uint16_t*>(h->act);
    aq.q = h->act_q;
    aq.scale = h->act_scale;
    aq.sf = h->act_sf;
    aq.routes = rows * d.top_k;
    aq.I = d.inter;
    aq.mode = h->act4;
    aq.health = h->health;
    before();
    if (!after(launch_act_quant(aq, s, pdl), "act_quant")) return MUSEMOE_ECUDA;
  }

  // 4. w2
  ep.role = 1;
  ep.N = d.pooled;
  ep.K = d.inter;
  ep.w = w->w2;
  ep.scale = w->w2_scale;
  ep.gscale = w->w2_gscale;
  ep.b = (h->quant == kFP8 || h->act4) ? h->act_q : h->act;
  ep.b_scale = h->act_scale;
  ep.b_sf = h->act_sf;
  ep.b_by_token = 0;
  ep.out = h->y;
  ep.tickets = h->expert_tickets[1];
  ep.grid = tc ? h->sms : h->expert_grid[1][nt_index(nte)];
  before();
  if (!after(tc ? launch_expert_tc(ep, s, pdl) : launch_expert(ep, nte, s, pdl), "w2"))
    return MUSEMOE_ECUDA;

  // 5. post-expert norm, weight, reduce
  FinalizeParams fz{};
  fz.y = h->y;
  fz.weights = h->weights;
  fz.w_post_norm = w->w_post_norm;
  fz.moe_out = h->moe_out;
  fz.rows = rows;
  fz.k = d.top_k;
  fz.P = d.pooled;
  fz.eps = h->cfg.norm_eps;
  if (epa) {
    fz.ids = h->ids;
    fz.part = epa->part;
    fz.ep_first = epa->first;
    fz.ep_count = epa->count;
  }
  before();
  if (!after(launch_finalize(fz, s, pdl), "finalize")) return MUSEMOE_ECUDA;
  if (epa) return MUSEMOE_OK;  // the partial moe_out is the rank's output
  const musemoe_status bs = launch_back(h, w, stream, out, rows, s, pdl, before, after);
  if (bs != MUSEMOE_OK) return bs;

  if (taps) {
    struct Cp {
      void* dst;
      const void* src;
      size_t bytes;
    } cps[] = {
        {taps->logits, h->logits, (size_t)rows * d.experts * 4},
        {taps->ids, h->ids, (size_t)rows * d.top_k * 4},
        {taps->weights, h->weights, (size_t)rows * d.top_k * 4},
        {taps->h, h->h, (size_t)rows * d.pooled * 2},
        {taps->act, h->act, (size_t)rows * d.top_k * d.inter * 2},
        {taps->y, h->y, (size_t)rows * d.top_k * d.pooled * 4},
        {taps->moe_out, h->moe_out, (size_t)rows * d.pooled * 2},
        {taps->u, h->u, (size_t)rows * d.hidden * 4},
    };
    for (const Cp& c : cps)
      if (c.dst) {
        const cudaError_t r = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, s);
        if (r != cudaSuccess) return cuda_err(h, r, "tap copy");
      }
  }
  (void)e;
  if (bad_event) {
    cudaGetLastError();  // clear the failed record
    return set_err(h, MUSEMOE_EINVAL, "taps->events holds an event that could not be recorded");
  }
  return MUSEMOE_OK;
}

musemoe_status launch_back(musemoe_handle* h, const musemoe_weights* w, float* stream,
                           uint16_t* out, int rows, cudaStream_t s, bool pdl,
                           const std::function<void()>& before,
                           const std::function<bool(cudaError_t, const char*)>& after) {
  const musemoe_dims& d = h->d;
  const int ntf = nt_front(rows);
  const bool dense = use_dense_tc(rows);
  // 6. unpooler GEMV
  FrontParams up{};
  up.x = h->moe_out;
  up.rows = rows;
  up.router_ctas = 0;
  up.w = w->w_unpool;
  up.y = h->u;
  up.health = h->health;
  up.M = d.hidden;
  up.K = d.pooled;
  up.gemv_ctas = front_gemv_ctas(d.hidden, rows, ntf);
  if (dense) {
    DenseParams dp{};
    dp.x = h->moe_out;
    dp.w = w->w_unpool;
    dp.y = h->u;
    dp.rows = rows;
    dp.M = d.hidden;
    dp.K = d.pooled;
    dp.health = h->health;
    dp.grid = h->sms;
    before();
    if (!after(launch_dense_tc(dp, s, pdl), "unpool")) return MUSEMOE_ECUDA;
  } else {
    before();
    if (!after(launch_front(up, ntf, s, pdl), "unpool")) return MUSEMOE_ECUDA;
  }

  // 7. FFN boundary
  BoundaryParams bp{};
  bp.u = h->u;
  bp.stream = stream;
  bp.out = out;
  bp.w_ffn_norm = w->w_ffn_norm;
  bp.w_next_norm = w->w_next_norm;
  bp.gate = w->gate;
  bp.rows = rows;
  bp.H = d.hidden;
  bp.eps = h->cfg.norm_eps;
  before();
  if (!after(launch_boundary(bp, s, pdl), "boundary")) return MUSEMOE_ECUDA;

  return MUSEMOE_OK;
}

musemoe_status check_call(musemoe_handle* h, const musemoe_weights* w, const void* x,
                          const void* stream, const void* out, int32_t rows, bool route_only) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  if (rows < 1 || rows > h->d.max_rows)
    return set_err(h, MUSEMOE_EINVAL, fmt("rows %d outside 1..max_rows (%d)", rows, h->d.max_rows));
  std::vector<std::string> bad;
  if (!x) bad.push_back("x is NULL");
  else if (!aligned16(x)) bad.push_back("x is not 16-byte aligned");
  if (!route_only) {
    if (!stream) bad.push_back("stream is NULL");
    else if (!aligned16(stream)) bad.push_back("stream is not 16-byte aligned");
    if (!out) bad.push_back("out is NULL");
    else if (!aligned16(out)) bad.push_back("out is not 16-byte aligned");
  }
  const std::string wb = check_weights(h, w, route_only);
  if (!wb.empty()) bad.push_back(wb);
  if (!bad.empty()) return set_err(h, MUSEMOE_EINVAL, join(bad));
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != h->device)
    return set_err(h, MUSEMOE_EINVAL,
                   fmt("current device %d is not the handle's device %d", dev, h->device));
  return MUSEMOE_OK;
}

}  // namespace

extern "C" {

musemoe_status musemoe_create(const musemoe_dims* dims, int32_t quant, const musemoe_config* config,
                              musemoe_handle** out) {
  if (out) *out = nullptr;
  if (!dims || !config || !out) return set_err(nullptr, MUSEMOE_EINVAL, "dims, config and out must not be NULL");
  const std::vector<std::string> r = refusals(dims, quant, config);
  if (!r.empty()) return set_err(nullptr, MUSEMOE_EUNSUPPORTED, join(r));
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_err(nullptr, MUSEMOE_ECUDA, fmt("no CUDA device: %s", cudaGetErrorString(e)));
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return set_err(nullptr, MUSEMOE_ECUDA, fmt("cudaGetDeviceProperties: %s", cudaGetErrorString(e)));
  if (!(prop.major == 10 && prop.minor == 3))
    return set_err(nullptr, MUSEMOE_EUNSUPPORTED,
                   fmt("device %d is sm_%d%d; the kernels are built for sm_103a", dev, prop.major,
                       prop.minor));
  musemoe_handle* h = new (std::nothrow) musemoe_handle();
  if (!h) return set_err(nullptr, MUSEMOE_ENOMEM, "host allocation failed");
  h->d = *dims;
  h->quant = weight_format(quant);
  h->act4 = act4_of(quant);
  h->cfg = *config;
  h->device = dev;
  h->sms = prop.multiProcessorCount;
  h->max_routes = dims->max_rows * dims->top_k;
  h->max_groups = std::min(dims->experts, h->max_routes) + (h->max_routes + 7) / 8 + 1;
  for (int role = 0; role < 2; ++role)
    for (int i = 0; i < 4; ++i)
      h->expert_grid[role][i] =
          h->sms * std::min(kExpertCtasPerSm,
                            expert_ctas_per_sm(h->quant, role, 1 << i,
                                                  role == 0 ? dims->pooled : dims->inter,
                                                  role == 0 ? 2 * dims->inter : dims->pooled));
  Layout L;
  plan(h, L);
  h->ws_bytes = L.off;
  e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) {
    delete h;
    return set_err(nullptr, MUSEMOE_ENOMEM,
                   fmt("workspace of %zu bytes: %s", L.off, cudaGetErrorString(e)));
  }
  for (auto& it : L.items) *it.first = static_cast<char*>(h->ws) + it.second;
  e = cudaMemset(h->ws, 0, h->ws_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return set_err(nullptr, MUSEMOE_ECUDA, fmt("workspace init: %s", cudaGetErrorString(e)));
  }
  *out = h;
  return MUSEMOE_OK;
}

void musemoe_destroy(musemoe_handle* h) {
  if (!h) return;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->ws);
  if (cur >= 0) cudaSetDevice(cur);
  delete h;
}

const char* musemoe_last_error(const musemoe_handle* h) {
  return h ? h->err.c_str() : g_thread_err.c_str();
}

size_t musemoe_workspace_bytes(const musemoe_dims* dims, int32_t quant) {
  if (!dims) return 0;
  musemoe_config c{};
  c.route_scale = 1.f;
  if (!refusals(dims, quant, &c).empty()) return 0;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  musemoe_handle h;
  h.d = *dims;
  h.quant = weight_format(quant);
  h.act4 = act4_of(quant);
  h.sms = sms;
  h.max_routes = dims->max_rows * dims->top_k;
  h.max_groups = std::min(dims->experts, h.max_routes) + (h.max_routes + 7) / 8 + 1;
  Layout L;
  plan(&h, L);
  return L.off;
}

int32_t musemoe_num_kernels(int32_t quant) { return (quant == kFP8 || act4_of(quant)) ? 8 : 7; }

const char* musemoe_kernel_name(int32_t quant, int32_t i) {
  static const char* fp4[] = {"router", "pool", "w13", "w2", "finalize", "unpool", "boundary"};
  static const char* fp8[] = {"router", "pool", "w13", "act_quant", "w2", "finalize", "unpool",
                              "boundary"};
  if (quant == kFP8 || act4_of(quant)) return (i >= 0 && i < 8) ? fp8[i] : "";
  return (i >= 0 && i < 7) ? fp4[i] : "";
}

musemoe_status musemoe_pack_experts(const musemoe_dims* d, int32_t quant, const uint8_t* w13_src,
                                    const void* w13_scale_src, uint8_t* w13_dst,
                                    void* w13_scale_dst, const uint8_t* w2_src,
                                    const void* w2_scale_src, uint8_t* w2_dst, void* w2_scale_dst,
                                    musemoe_stream_t stream) {
  if (!d) return set_err(nullptr, MUSEMOE_EINVAL, "dims is NULL");
  musemoe_config c{};
  c.route_scale = 1.f;
  const std::vector<std::string> r = refusals(d, quant, &c);
  if (!r.empty()) return set_err(nullptr, MUSEMOE_EUNSUPPORTED, join(r));
  const int a4 = act4_of(quant);     // W4A4: the FP4 tensor cores' layouts
  quant = weight_format(quant);      // W4A4 weights are MXFP4 / NVFP4
  const bool bf16 = quant == kBF16;  // no scales
  const void* ptrs[8] = {w13_src, w13_scale_src, w13_dst, w13_scale_dst,
                         w2_src,  w2_scale_src,  w2_dst,  w2_scale_dst};
  for (int i = 0; i < 8; ++i) {
    const void* q = ptrs[i];
    if (bf16 && (i % 2)) continue;
    if (!q) return set_err(nullptr, MUSEMOE_EINVAL, "expert tensor pointers must not be NULL");
    if (!aligned16(q)) return set_err(nullptr, MUSEMOE_EINVAL, "expert tensors must be 16-byte aligned");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t E = d->experts, P = d->pooled, I = d->inter;
  const bool fp8 = quant == kFP8;
  // bytes per row of K values: FP4 K / 2, FP8 K, BF16 2 K
  auto row_bytes = [&](size_t K) { return fp8 ? K : bf16 ? 2 * K : K / 2; };
  const int sper = quant == kMXFP4 ? 4 : 8;  // scale bytes per 64-byte code chunk
  struct M {
    const uint8_t* src;
    uint8_t* dst;
    const void* ssrc;
    void* sdst;
    size_t rows;
    size_t K;
  } ms[2] = {{w13_src, w13_dst, w13_scale_src, w13_scale_dst, E * 2 * I, P},
             {w2_src, w2_dst, w2_scale_src, w2_scale_dst, E * P, I}};
  cudaError_t e = cudaSuccess;
  if (quant == kMXFP4) {
    // the kernels decode UE8M0 as a bare exponent: 0x00 (2^-127) and 0xFF
    // (NaN) are refused here, before anything is re-laid
    int* bad = nullptr;
    int bad_h = 0;
    e = cudaMalloc(&bad, sizeof(int));
    if (e == cudaSuccess) e = cudaMemsetAsync(bad, 0, sizeof(int), s);
    for (const M& m : ms)
      if (e == cudaSuccess)
        e = check_ue8m0(reinterpret_cast<const uint8_t*>(m.ssrc), m.rows * (m.K / 32), bad, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&bad_h, bad, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (bad) cudaFree(bad);
    if (e != cudaSuccess) return set_err(nullptr, MUSEMOE_ECUDA, fmt("pack: %s", cudaGetErrorString(e)));
    if (bad_h)
      return set_err(nullptr, MUSEMOE_EUNSUPPORTED,
                     "an MXFP4 scale is UE8M0 0x00 (2^-127) or 0xFF (NaN); the kernels take 0x01..0xFE");
  }
  // in-place re-layouts pass through a temporary buffer of whole row tiles
  size_t tmp_bytes = 0;
  for (const M& m : ms) {
    const size_t rowbytes = row_bytes(m.K);
    const size_t total = m.rows * rowbytes, tile = 64 * rowbytes;
    if (m.src == m.dst) tmp_bytes = std::max(tmp_bytes, std::max(tile, std::min(total, kPackTmpBytes)));
    if (!fp8 && !bf16 && m.ssrc == m.sdst) tmp_bytes = std::max(tmp_bytes, 64 * (rowbytes / 64) * sper);
    // W4A4 scale atoms mix the gate and up halves of an expert: one expert's
    // scales pass through the temporary
    if (a4 && m.ssrc == m.sdst) tmp_bytes = std::max(tmp_bytes, m.rows / E * (m.K / (a4 == 2 ? 16 : 32)));
  }
  uint8_t* tmp = nullptr;
  if (tmp_bytes) {
    e = cudaMalloc(&tmp, tmp_bytes);
    if (e != cudaSuccess)
      return set_err(nullptr, MUSEMOE_ENOMEM, fmt("pack: temporary of %zu bytes: %s", tmp_bytes,
                                                  cudaGetErrorString(e)));
  }
  for (int mi = 0; mi < 2; ++mi) {
    const M& m = ms[mi];
    const int rowbytes = (int)row_bytes(m.K);
    // codes: FP8 and W4A4 in natural order with the 64-byte swizzle (the
    // tensor cores read them as they land), the other forms in mma fragment order
    const int permute = (fp8 || a4) ? 3 : bf16 ? 2 : 1;
    if (e == cudaSuccess) e = launch_pack_tiles(m.src, m.dst, m.rows, rowbytes, 64, permute, tmp, tmp_bytes, s);
    if (e != cudaSuccess) break;
    if (bf16) continue;  // no scales
    if (a4) {
      e = launch_pack_sf_atoms(reinterpret_cast<const uint8_t*>(m.ssrc), reinterpret_cast<uint8_t*>(m.sdst),
                               (int)E, (int)(m.rows / E), (int)I, (int)m.K, mi, a4 == 2, tmp, tmp_bytes, s);
      continue;
    }
    if (fp8) {  // per-row fp32 scales stay as they are
      if (m.ssrc != m.sdst)
        e = cudaMemcpyAsync(m.sdst, m.ssrc, m.rows * 4, cudaMemcpyDeviceToDevice, s);
    } else {
      const int srow = (int)(rowbytes / 64) * sper;
      e = launch_pack_tiles(reinterpret_cast<const uint8_t*>(m.ssrc), reinterpret_cast<uint8_t*>(m.sdst),
                            m.rows, srow, sper, 0, tmp, tmp_bytes, s);
    }
  }
  if (tmp) {
    const cudaError_t e2 = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = e2;
    cudaFree(tmp);
  }
  if (e != cudaSuccess) return set_err(nullptr, MUSEMOE_ECUDA, fmt("pack: %s", cudaGetErrorString(e)));
  return MUSEMOE_OK;
}

musemoe_status musemoe_route(musemoe_handle* h, const musemoe_weights* w, const uint16_t* x,
                             int32_t rows, int32_t* ids_out, float* weights_out,
                             musemoe_stream_t stream) {
  musemoe_status st = check_call(h, w, x, nullptr, nullptr, rows, true);
  if (st != MUSEMOE_OK) return st;
  if (!ids_out || !weights_out || !aligned16(ids_out) || !aligned16(weights_out))
    return set_err(h, MUSEMOE_EINVAL, "ids_out and weights_out must be non-NULL and 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const musemoe_dims& d = h->d;
  FrontParams fp{};
  fp.x = x;
  fp.rows = rows;
  fp.w_router = w->w_router;
  fp.logits = h->logits;
  fp.E = d.experts;
  fp.health = h->health;
  fp.router_ctas = router_ctas(d.experts, rows);
  fp.M = 0;
  fp.K = d.hidden;
  cudaError_t e = launch_router(fp, s, true);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_err(h, e, "launch of router");
  RouteParams rp{};
  rp.logits = h->logits;
  rp.expert_bias = w->expert_bias;
  rp.ids = ids_out;
  rp.weights = weights_out;
  rp.rows = rows;
  rp.E = d.experts;
  rp.k = d.top_k;
  rp.score = h->cfg.score;
  rp.has_multiplier = h->cfg.has_multiplier;
  rp.multiplier = h->cfg.multiplier;
  rp.has_division_eps = h->cfg.has_division_eps;
  rp.division_eps = h->cfg.division_eps;
  rp.route_scale = h->cfg.route_scale;
  rp.central = rows <= 32;
  e = launch_route(rp, s, true);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_err(h, e, "launch of route");
  return MUSEMOE_OK;
}

musemoe_status musemoe_forward(musemoe_handle* h, const musemoe_weights* w, const uint16_t* x,
                               float* stream, uint16_t* out, int32_t rows, musemoe_stream_t s) {
  musemoe_status st = check_call(h, w, x, stream, out, rows, false);
  if (st != MUSEMOE_OK) return st;
  return launch_chain(h, w, x, stream, out, rows, reinterpret_cast<cudaStream_t>(s), nullptr);
}

musemoe_status musemoe_forward_debug(musemoe_handle* h, const musemoe_weights* w, const uint16_t* x,
                                     float* stream, uint16_t* out, int32_t rows, musemoe_stream_t s,
                                     const musemoe_taps* taps) {
  musemoe_status st = check_call(h, w, x, stream, out, rows, false);
  if (st != MUSEMOE_OK) return st;
  return launch_chain(h, w, x, stream, out, rows, reinterpret_cast<cudaStream_t>(s), taps);
}

musemoe_status musemoe_forward_ep_partial(musemoe_handle* h, const musemoe_weights* w,
                                         const uint16_t* x, float* moe_partial, int32_t rows,
                                         int32_t expert_first, int32_t expert_count,
                                         musemoe_stream_t stream) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  if (rows < 1 || rows > h->d.max_rows)
    return set_err(h, MUSEMOE_EINVAL, fmt("rows %d outside 1..max_rows (%d)", rows, h->d.max_rows));
  std::vector<std::string> bad;
  if (expert_count < 1 || expert_first < 0 || expert_first + expert_count > h->d.experts)
    bad.push_back(fmt("expert range [%d, %d) is not a non-empty range of the %d experts",
                      expert_first, expert_first + expert_count, h->d.experts));
  auto need = [&](const void* q, const char* name) {
    if (!q) bad.push_back(fmt("%s is NULL", name));
    else if (!aligned16(q)) bad.push_back(fmt("%s is not 16-byte aligned", name));
  };
  need(x, "x");
  need(moe_partial, "moe_partial");
  if (!w) {
    bad.push_back("weights is NULL");
  } else {
    need(w->w_router, "w_router");
    need(w->expert_bias, "expert_bias");
    need(w->w_pool, "w_pool");
    need(w->w_pre_norm, "w_pre_norm");
    need(w->w13, "w13");
    need(w->w2, "w2");
    if (h->quant != kBF16) {
      need(w->w13_scale, "w13_scale");
      need(w->w2_scale, "w2_scale");
    }
    if (h->quant == kNVFP4) {
      need(w->w13_gscale, "w13_gscale");
      need(w->w2_gscale, "w2_gscale");
    }
    need(w->w_post_norm, "w_post_norm");
  }
  if (!bad.empty()) return set_err(h, MUSEMOE_EINVAL, join(bad));
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != h->device)
    return set_err(h, MUSEMOE_EINVAL, fmt("current device %d is not the handle's device %d", dev, h->device));
  const EpArgs ep{expert_first, expert_count, moe_partial};
  return launch_chain(h, w, x, nullptr, nullptr, rows, reinterpret_cast<cudaStream_t>(stream),
                      nullptr, &ep);
}

musemoe_status musemoe_forward_ep_combine(musemoe_handle* h, const musemoe_weights* w,
                                         const float* moe_sum, float* stream_io, uint16_t* out,
                                         int32_t rows, musemoe_stream_t stream) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  if (rows < 1 || rows > h->d.max_rows)
    return set_err(h, MUSEMOE_EINVAL, fmt("rows %d outside 1..max_rows (%d)", rows, h->d.max_rows));
  std::vector<std::string> bad;
  auto need = [&](const void* q, const char* name) {
    if (!q) bad.push_back(fmt("%s is NULL", name));
    else if (!aligned16(q)) bad.push_back(fmt("%s is not 16-byte aligned", name));
  };
  need(moe_sum, "moe_sum");
  need(stream_io, "stream_io");
  need(out, "out");
  if (!w) {
    bad.push_back("weights is NULL");
  } else {
    need(w->w_unpool, "w_unpool");
    need(w->w_ffn_norm, "w_ffn_norm");
    need(w->w_next_norm, "w_next_norm");
    need(w->gate, "gate");
  }
  if (!bad.empty()) return set_err(h, MUSEMOE_EINVAL, join(bad));
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != h->device)
    return set_err(h, MUSEMOE_EINVAL, fmt("current device %d is not the handle's device %d", dev, h->device));
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // moe_out = bf16(sum of the ranks' partials): the rounding the single-GPU
  // finalize applies to the same fp32 sum; launched without programmatic
  // dependency on the caller's previous kernel (the all-reduce)
  cudaError_t e = launch_round_bf16(moe_sum, h->moe_out, (long long)rows * h->d.pooled, s);
  if (e != cudaSuccess) return cuda_err(h, e, "launch of the moe_out rounding");
  auto before = []() {};
  auto after = [&](cudaError_t r, const char* name) -> bool {
    if (r == cudaSuccess) r = cudaGetLastError();
    if (r != cudaSuccess) {
      h->err = fmt("launch of %s failed: %s", name, cudaGetErrorString(r));
      return false;
    }
    return true;
  };
  return launch_back(h, w, stream_io, out, rows, s, true, before, after);
}

musemoe_status musemoe_forward_host(musemoe_handle* h, const musemoe_weights* w,
                                    const uint16_t* x_host, float* stream_host, uint16_t* out_host,
                                    int32_t rows, musemoe_stream_t stream) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  if (!x_host || !stream_host || !out_host)
    return set_err(h, MUSEMOE_EINVAL, "host buffers must not be NULL");
  if (rows < 1 || rows > h->d.max_rows)
    return set_err(h, MUSEMOE_EINVAL, fmt("rows %d outside 1..max_rows (%d)", rows, h->d.max_rows));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t nh = (size_t)rows * h->d.hidden;
  cudaError_t e = cudaMemcpyAsync(h->x_stage, x_host, nh * 2, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->stream_stage, stream_host, nh * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_err(h, e, "copy to device");
  musemoe_status st = check_call(h, w, h->x_stage, h->stream_stage, h->out_stage, rows, false);
  if (st != MUSEMOE_OK) return st;
  st = launch_chain(h, w, h->x_stage, h->stream_stage, h->out_stage, rows, s, nullptr);
  if (st != MUSEMOE_OK) return st;
  e = cudaMemcpyAsync(stream_host, h->stream_stage, nh * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, h->out_stage, nh * 2, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(h, e, "copy to host");
  return MUSEMOE_OK;
}

musemoe_status musemoe_attention_boundary(const uint16_t* partial, float* stream_io, uint16_t* out,
                                          const uint16_t* w_pre_ffn_norm, const float* gate,
                                          int32_t rows, int32_t hidden, float eps,
                                          musemoe_stream_t stream) {
  std::vector<std::string> bad;
  if (rows < 1) bad.push_back(fmt("rows %d < 1", rows));
  if (hidden < 4 || hidden % 4 || hidden > kBoundaryMaxH)
    bad.push_back(fmt("hidden %d is not a multiple of 4 in 4..%d", hidden, kBoundaryMaxH));
  if (!(eps >= 0.f)) bad.push_back("eps < 0");
  auto need = [&](const void* q, const char* name) {
    if (!q) bad.push_back(fmt("%s is NULL", name));
    else if (!aligned16(q)) bad.push_back(fmt("%s is not 16-byte aligned", name));
  };
  need(partial, "partial");
  need(stream_io, "stream_io");
  need(out, "out");
  need(w_pre_ffn_norm, "w_pre_ffn_norm");
  if (!gate) bad.push_back("gate is NULL");
  if (!bad.empty()) return set_err(nullptr, MUSEMOE_EINVAL, join(bad));
  BoundaryParams bp{};
  bp.u_bf16 = partial;
  bp.stream = stream_io;
  bp.out = out;
  bp.w_ffn_norm = nullptr;  // post_attn_norm is weightless
  bp.w_next_norm = w_pre_ffn_norm;
  bp.gate = gate;
  bp.rows = rows;
  bp.H = hidden;
  bp.eps = eps;
  cudaError_t e = launch_boundary(bp, reinterpret_cast<cudaStream_t>(stream), false);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_err(nullptr, e, "launch of the attention boundary");
  return MUSEMOE_OK;
}

musemoe_status musemoe_quantize_mxfp4(const uint16_t* w_bf16, uint8_t* codes, uint8_t* scales,
                                      int64_t rows, int32_t cols, musemoe_stream_t stream) {
  std::vector<std::string> bad;
  if (rows < 1) bad.push_back(fmt("rows %lld < 1", (long long)rows));
  if (cols < 32 || cols % 32) bad.push_back(fmt("cols %d is not a positive multiple of 32", cols));
  if (!w_bf16) bad.push_back("w_bf16 is NULL");
  else if (!aligned16(w_bf16)) bad.push_back("w_bf16 is not 16-byte aligned");
  if (!codes) bad.push_back("codes is NULL");
  else if (!aligned16(codes)) bad.push_back("codes is not 16-byte aligned");
  if (!scales) bad.push_back("scales is NULL");
  if (!bad.empty()) return set_err(nullptr, MUSEMOE_EINVAL, join(bad));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = launch_quant_mxfp4(w_bf16, codes, scales, (long long)rows * cols, sms,
                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(nullptr, e, "launch of the MXFP4 rounding");
  return MUSEMOE_OK;
}

musemoe_status musemoe_quantize_act_nvfp4(const uint16_t* x_bf16, uint8_t* codes, uint8_t* scales,
                                          int64_t rows, int32_t cols, musemoe_stream_t stream) {
  std::vector<std::string> bad;
  if (rows < 1) bad.push_back(fmt("rows %lld < 1", (long long)rows));
  if (cols < 16 || cols % 16) bad.push_back(fmt("cols %d is not a positive multiple of 16", cols));
  if (!x_bf16) bad.push_back("x_bf16 is NULL");
  else if (!aligned16(x_bf16)) bad.push_back("x_bf16 is not 16-byte aligned");
  if (!codes) bad.push_back("codes is NULL");
  else if (!aligned16(codes)) bad.push_back("codes is not 16-byte aligned");
  if (!scales) bad.push_back("scales is NULL");
  if (!bad.empty()) return set_err(nullptr, MUSEMOE_EINVAL, join(bad));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = launch_quant_act_nvfp4(x_bf16, codes, scales, (long long)rows * cols, sms,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(nullptr, e, "launch of the NVFP4 expert input");
  return MUSEMOE_OK;
}

musemoe_status musemoe_health_selftest(musemoe_handle* h, musemoe_stream_t stream) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != h->device)
    return set_err(h, MUSEMOE_EINVAL, fmt("current device %d is not the handle's device %d", dev, h->device));
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the split-tile tickets as contributors arriving after their owner gave
  // up would leave them (raised), for the poll that reports the timeout to
  // clear
  cudaError_t e = cudaSuccess;
  for (int r = 0; r < 2 && e == cudaSuccess; ++r)
    e = cudaMemsetAsync(h->expert_tickets[r], 0x01, h->expert_ticket_bytes[r], s);
  if (e == cudaSuccess) e = launch_wait_selftest(h->health, h->never_set, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(h, e, "health self-test");
  return MUSEMOE_OK;
}

musemoe_status musemoe_set_expert_path(musemoe_handle* h, int32_t path) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  if (path != MUSEMOE_PATH_AUTO && path != MUSEMOE_PATH_MMA && path != MUSEMOE_PATH_TCGEN05)
    return set_err(h, MUSEMOE_EINVAL, fmt("expert path %d is not AUTO (0), MMA (1) or TCGEN05 (2)", path));
  if (path == MUSEMOE_PATH_TCGEN05 && h->quant == kBF16)
    return set_err(h, MUSEMOE_EUNSUPPORTED, "BF16 experts have no tensor-core (tcgen05) expert kernel");
  if (path == MUSEMOE_PATH_MMA && h->act4)
    return set_err(h, MUSEMOE_EUNSUPPORTED,
                   "the W4A4 forms run on the FP4 tensor cores only (their weights are packed for them)");
  h->expert_path = path;
  return MUSEMOE_OK;
}

musemoe_status musemoe_poll_health(musemoe_handle* h) {
  if (!h) return set_err(nullptr, MUSEMOE_EINVAL, "handle is NULL");
  int32_t word = 0;
  cudaError_t e = cudaMemcpy(&word, h->health, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->health, 0, 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_err(h, e, "health read");
  if (word & kHealthTimeout) {
    // A CTA that gave up left its tile tickets in an unknown state (a late
    // contributor may still have added to one): the next forward must start
    // from zeroed tickets. The device is idle here (synchronized above).
    for (int r = 0; r < 2 && e == cudaSuccess; ++r)
      e = cudaMemset(h->expert_tickets[r], 0, h->expert_ticket_bytes[r]);
    if (e == cudaSuccess) e = cudaMemset(h->norm_ticket, 0, h->block_ticket_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->route_ticket, 0, h->block_ticket_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->route_done, 0, 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_err(h, e, "ticket reset");
  }
  if (word) {
    std::string m;
    if (word & kHealthTimeout) m += "an expert kernel's bounded wait on its weight copies ran out; ";
    if (word & kHealthHRange) m += "h beyond the fp16 operand range (W4A4: not finite); ";
    if (word & kHealthActRange)
      m += "SiLU(gate)*up beyond the fp16 operand range (W4A4: not finite); ";
    if (word & kHealthWRange)
      m += "an MXFP4 block scale outside 2^-23..2^13, beyond the fp16 operand range of the "
           "tensor-core expert kernels; ";
    return set_err(h, (word & kHealthTimeout) ? MUSEMOE_ETIMEOUT : MUSEMOE_ERANGE, m);
  }
  return MUSEMOE_OK;
}

}  // extern "C"
