// Internal launch interface of the musemoe kernels (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace musemoe {

enum Quant : int { kMXFP4 = 0, kNVFP4 = 1, kFP8 = 2, kBF16 = 3 };

// The calling thread's error text that musemoe_last_error(NULL) returns.
void set_thread_error(const std::string& m);

// counters[] slots in the workspace
enum Counter : int { kNumGroups = 0, kTicket = 1, kNumCounters = 8 };
// health bits
enum Health : int { kHealthHRange = 1, kHealthActRange = 2, kHealthTimeout = 4, kHealthWRange = 8 };

// ---- route: routing rule + token->expert permute ---------------------------
struct RouteParams {
  const float* logits;      // [rows, E]
  const float* expert_bias;
  int32_t* ids;             // [rows, k]
  float* weights;           // [rows, k]
  int rows, E, k;
  int score;  // 0 sigmoid, 1 softmax
  int has_multiplier;
  float multiplier;
  int has_division_eps;
  float division_eps;
  float route_scale;
  // permute (skipped when route_list == nullptr)
  int32_t* route_list;  // [rows*k]
  int32_t* groups;      // [max_groups, 4]: expert, first route slot, ntok, 0
  int32_t* counters;
  int32_t* health;
  int token_group;  // routes per group (8 * NT of the expert kernels)
  int central;      // 1: one CTA routes every row and permutes (rows <= 32)
  // expert parallelism: token groups only for the experts [ep_first,
  // ep_first + ep_count), whose group expert index is local (e - ep_first);
  // ep_count 0 = every expert
  int ep_first, ep_count;
};
// ---- router GEMV (fp32 FFMA) and pooler / unpooler GEMV ------------------
// The router runs router_ctas = E * ceil(rows / 8) (expert, 8-token block)
// tasks, each over the whole reduction: one task per CTA, or above 8 rows
// four experts' tasks per CTA. The bf16 GEMV Y = X W^T
// (W [M, K] row-major, K a multiple of 64 and at most front_max_k()) runs on
// front_gemv_ctas(M, rows, nt) CTAs, one per 16-row tile and token block.
struct FrontParams {
  const uint16_t* x;  // bf16 [rows, K]
  int rows;
  // router (skipped when router_ctas == 0)
  const float* w_router;  // fp32 [E, K]
  float* logits;          // [rows, E]
  int E, router_ctas;
  // bf16 GEMV (skipped when gemv_ctas == 0)
  const uint16_t* w;  // bf16 [M, K]
  float* y;           // fp32 [rows, M]
  int32_t* health;
  int M, K;
  int gemv_ctas;
  // pooler only (skipped when h == nullptr): with norm_in_tail the last CTA
  // of each token block applies the pre-expert RMSNorm to the block's rows
  // of y; without, launch_pool_norm follows (eight rows per CTA)
  int norm_in_tail;
  const uint16_t* w_pre_norm;  // bf16 [M]
  int pre_norm, quant;
  int act4;             // W4A4 (1 MXFP4, 2 NVFP4): the norm writes h only (no operand);
                        // the forward rounds h into h_op / h_sf next
  float norm_eps;
  uint16_t* h;          // bf16 [rows, M]
  uint8_t* h_op;        // f16 [rows, M] (FP4), e4m3 [rows, M] (FP8), W4A4: e2m1 codes [rows, M / 2]
  float* h_scale;       // [rows] (FP8)
  uint8_t* h_sf;        // W4A4: block scales [rows, M / 32] (UE8M0) or [rows, M / 16] (e4m3)
  int32_t* norm_ticket; // [token blocks], zero between launches (norm_in_tail)
  // router only (route_tail != 0): the last router CTA of each 8-token block
  // routes the block's rows, and the last block to finish builds the permute
  int route_tail;
  RouteParams route;
  int32_t* route_ticket;  // [8-token blocks], zero between launches
  int32_t* route_done;    // [1], zero between launches
};
cudaError_t launch_front(const FrontParams& p, int nt, cudaStream_t s, bool pdl);   // GEMV
// The pooler's pre-expert norm as its own launch (after launch_dense_tc):
// rows of p.y -> p.h / p.h_op / p.h_scale, eight rows per CTA. Waits for its
// predecessor before it lets its dependents launch.
cudaError_t launch_pool_norm(const FrontParams& p, cudaStream_t s, bool pdl);

// ---- dense bf16 GEMM on the tensor cores (pooler / unpooler, larger buckets)
// y[rows, M] = x[rows, K] w[M, K]^T, fp32; K a multiple of 64; split K over
// thread-block clusters of at most `grid` CTAs in all, the partial sums
// exchanged in distributed shared memory (no global workspace).
struct DenseParams {
  const uint16_t* x;  // bf16 [rows, K]
  const uint16_t* w;  // bf16 [M, K]
  float* y;           // fp32 [rows, M]
  int rows, M, K;
  int x_ready;  // x is final when the launch starts (the pooler's input, which
                // the router before it only reads): its copies do not wait
  int32_t* health;
  int grid;  // CTAs the launch may use (the SMs)
};
cudaError_t launch_dense_tc(const DenseParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_router(const FrontParams& p, cudaStream_t s, bool pdl);          // router
int front_gemv_ctas(int M, int rows, int nt);
int front_max_k();

cudaError_t launch_route(const RouteParams& p, cudaStream_t s, bool pdl);

// ---- routed experts --------------------------------------------------------
struct ExpertParams {
  int quant;
  int role;      // 0: w13 + SiLU*up -> act; 1: w2 -> y
  int E, N, K;   // rows N and reduction K of the weight matrix
  int I, P, k;
  const uint8_t* w;        // codes, kernel layout (launch_pack_tiles, cb = 64)
  const void* scale;       // MX/NV: kernel layout (cb = 4 / 8); FP8: fp32 [E, N]
  const float* gscale;     // NVFP4 [E]
  const uint8_t* b;        // activation operand: f16 [*, K], e4m3 [*, K] or (BF16 experts) bf16 [*, K];
                           // W4A4: e2m1 codes [*, K / 2] (two per byte, the lower element in the low nibble)
  const float* b_scale;    // FP8: per B row
  int act4;                // W4A4 on the FP4 tensor cores: 1 MXFP4, 2 NVFP4 (launch_expert_tc only;
                           // w and scale then in the layouts of launch_pack_tiles permute 3 and
                           // launch_pack_sf_atoms)
  const uint8_t* b_sf;     // W4A4: block scales of the B rows [*, K / 32] (UE8M0) or [*, K / 16] (e4m3)
  int b_by_token;          // 1: B row = route / k (w13 reads h); 0: B row = route
  const int32_t* route_list;
  const int32_t* groups;
  const int32_t* counters;
  void* out;               // role 0: act f16/bf16 [rows*k, I]; role 1: y fp32 [rows*k, P]
  int act_bf16;            // role 0, FP4 weights: store act as bf16 (W4A4 rounds it next)
  int32_t* health;
  float* part;             // partial sums of tiles split across CTAs (expert_part_bytes)
  int32_t* tickets;        // tile tickets (expert_tickets), zero between launches
  int grid;
  int stages;  // set by the launcher
};
cudaError_t launch_expert(const ExpertParams& p, int nt, cudaStream_t s, bool pdl);
// The same work on the fifth-generation tensor cores (tcgen05; MXFP4, NVFP4
// and FP8 weights): token groups of up to expert_tc_group_tokens() routes,
// p.grid CTAs (one per SM), partial sums in expert_tc_part_bytes(p.grid).
cudaError_t launch_expert_tc(const ExpertParams& p, cudaStream_t s, bool pdl);
size_t expert_tc_part_bytes(int grid);
int expert_tc_group_tokens();
int expert_ctas_per_sm(int quant, int role, int nt, int K, int N);
size_t expert_part_bytes(int grid, int nt);
size_t expert_tickets(int max_groups, int quant, int role, int K, int N);

// FP8 only: per-route dynamic e4m3 quantization of the bf16 activation.
// W4A4 (mode 1 MXFP4, 2 NVFP4): per-row FP4 rounding of a bf16 operand,
// w2's activation per route (and w13's h per token), into e2m1 codes and
// block scales.
struct ActQuantParams {
  const uint16_t* act;  // bf16 [routes, I]
  uint8_t* q;           // mode 0: e4m3 [routes, I]; modes 1, 2: e2m1 codes [routes, I / 2]
  float* scale;         // mode 0: [routes]
  uint8_t* sf;          // modes 1, 2: block scales [routes, I / 32] (UE8M0) or [routes, I / 16] (e4m3)
  int routes, I;
  int mode;             // 0 FP8, 1 MXFP4, 2 NVFP4
  int32_t* health;      // modes 1, 2: kHealthActRange for a value that is not finite
};
cudaError_t launch_act_quant(const ActQuantParams& p, cudaStream_t s, bool pdl);

// ---- tail: per-route post-expert norm, router weight, sum over k --------
struct FinalizeParams {
  const float* y;  // [rows*k, P]
  const float* weights;
  const uint16_t* w_post_norm;
  uint16_t* moe_out;  // bf16 [rows, P]
  int rows, k, P;
  float eps;
  int stash;  // set by launch_finalize: route rows kept in shared memory
  // expert parallelism (part != nullptr): only the routes whose expert id is
  // in [ep_first, ep_first + ep_count) contribute, and the fp32 sum goes to
  // part [rows, P] (no bf16 rounding: the ranks' parts are summed first)
  const int32_t* ids;  // [rows, k]
  float* part;
  int ep_first, ep_count;
};
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s, bool pdl);
// fp32 [n] -> bf16 [n] (round to nearest even), n a multiple of 4; no
// programmatic dependency on the previous kernel.
cudaError_t launch_round_bf16(const float* src, uint16_t* dst, long long n, cudaStream_t s);

// ---- FFN boundary ------------------------------------------------------------
struct BoundaryParams {
  const float* u;          // unpooler output fp32 [rows, H] (FFN boundary), or
  const uint16_t* u_bf16;  // the o_proj output bf16 [rows, H] (attention boundary)
  float* stream;           // fp32 [rows, H], in place
  uint16_t* out;           // bf16 [rows, H]
  const uint16_t* w_ffn_norm;   // weight of the first norm; nullptr: weightless
  const uint16_t* w_next_norm;  // weight of the second norm
  const float* gate;
  int rows, H;
  float eps;
};
constexpr int kBoundaryMaxH = 8192;  // the row held in registers
cudaError_t launch_boundary(const BoundaryParams& p, cudaStream_t s, bool pdl);

// ---- health self-test: the bounded waits time out into the health word -----
cudaError_t launch_wait_selftest(int32_t* health, const int32_t* never, cudaStream_t s);

// ---- online rounding of bf16 weights to MXFP4 ------------------------------
// elements = rows * cols with cols a multiple of 32: codes [rows, cols/2],
// scales [rows, cols/32]; w 16-byte aligned, codes 4-byte aligned.
cudaError_t launch_quant_mxfp4(const uint16_t* w, uint8_t* codes, uint8_t* scales,
                               long long elements, int sms, cudaStream_t s);
// The NVFP4 expert input: bf16 [*, 16 m] -> e2m1 codes + e4m3 scales per 16.
cudaError_t launch_quant_act_nvfp4(const uint16_t* x, uint8_t* codes, uint8_t* scales,
                                   long long elements, int sms, cudaStream_t s);

// ---- weight re-layout ----------------------------------------------------
// Kernel layout of a [rows, row_bytes] expert tensor cut into cb-byte chunks
// (cb = 64 for codes, the scale bytes of one code chunk for scales): tiles of
// 64 rows, each stored K-slice by K-slice (kSliceChunks chunks, the last
// slice the remainder), each slice by 8-row group, chunk, row:
// [rows / 64][slice][8][chunks of the slice][8][cb]. permute 1 (FP4) or 2
// (BF16) also reorders the bytes of each 64-byte code chunk for the mma
// fragments; 3 (FP8) swizzles the 16-byte units of each [8][64 B] block
// (unit u of row r at u ^ ((r >> 1) & 3), the tensor cores' 64-byte
// swizzle); 0 keeps them.
// src may equal dst: the tiles then pass through `tmp` (at least one tile).
// Sets *bad_dev to 1 if any of the n UE8M0 bytes is 0x00 or 0xFF.
constexpr int kSliceChunks = 4;
cudaError_t check_ue8m0(const uint8_t* p, size_t n, int* bad_dev, cudaStream_t s);
cudaError_t launch_pack_tiles(const uint8_t* src, uint8_t* dst, size_t rows, int row_bytes, int cb,
                              int permute, uint8_t* tmp, size_t tmp_bytes, cudaStream_t s);
// Block scales of one FP4 expert matrix (plain [E, N, K / blk] bytes, blk 32
// MXFP4 or 16 NVFP4) -> the tensor cores' scale atoms for W4A4: per expert,
// A tile of 128 rows (w13, role 0: gate rows t*64.. and up rows I + t*64..
// interleaved by 8-row groups, row m of the tile in group m / 8; w2: rows
// t*128..), K-slice of kSliceChunks 128-element chunks, atom of 4 blocks
// (MXFP4: one chunk; NVFP4: half a chunk), 512 bytes with the scale of tile
// row m and block j at byte (m % 32) * 16 + (m / 32) * 4 + j:
// [E][tiles][slice][atoms of the slice][512]. src may equal dst (each
// expert's scales then pass through `tmp`, at least N * K / blk bytes).
cudaError_t launch_pack_sf_atoms(const uint8_t* src, uint8_t* dst, int E, int N, int I, int K,
                                 int role, int nv, uint8_t* tmp, size_t tmp_bytes, cudaStream_t s);

}  // namespace musemoe
