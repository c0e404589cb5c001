/*
 * musemoe -- the MuseSpark1x MoE decode block on one GB300 (sm_103a).
 *
 * One call runs, for `rows` input rows (a small-batch decode / speculative
 * verify step):
 *   router GEMV (fp32 weight [E, H] x bf16 input [rows, H] -> fp32 logits)
 *   routing rule: optional output multiplier -> sigmoid or softmax -> expert
 *     bias added for SELECTION only -> top-k -> gather the UNBIASED scores ->
 *     divide by (sum + division_eps) -> multiply by route_scale
 *     (page "vllm.models.muse_spark.amd.muse_moe_runner", class
 *     MuseSpark1xRouter, docstring and _compute_routing_native);
 *   pooler GEMM H -> P and the pre-expert RMSNorm -> bf16 h
 *     (page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
 *     MoEProvider docstring);
 *   routed experts on MXFP4 / NVFP4 / FP8 / BF16 weights (and the W4A4
 *     forms, FP4 activations): fused w13 (gate rows
 *     first), SiLU(gate) * up -> bf16, w2; one UNWEIGHTED output per route
 *     (muse_moe_runner page, MuseSparkAiterExperts: unit router weights);
 *   per-route post-expert RMSNorm, then the router weight, summed over the
 *     k routes -> bf16 moe_out (muse_moe_runner page,
 *     MuseSparkTopKWeightAndReduce.apply);
 *   unpooler GEMM P -> H;
 *   FFN boundary: post_ffn_norm, gated add into the fp32 residual stream in
 *     place, next pre-norm -> bf16 out (providers page, BoundaryProvider).
 *
 * Conventions (providers page, Provider: build once, then a run that
 * allocates nothing and is CUDA-graph capturable):
 *   - musemoe_create validates the configuration and allocates the handle's
 *     device workspace (sized for dims.max_rows) on the current device. It
 *     is the only call that allocates device memory.
 *   - musemoe_route / musemoe_forward / musemoe_forward_debug allocate
 *     nothing, never synchronize, launch only on the given stream and can be
 *     captured in a CUDA graph. All tensors are caller-owned device memory
 *     (e.g. PyTorch tensors); the library keeps no pointer after a call.
 *   - Arguments are validated before anything is launched; on failure the
 *     call returns MUSEMOE_EINVAL / MUSEMOE_EUNSUPPORTED, launches nothing and
 *     musemoe_last_error(handle) says why. A failed launch returns
 *     MUSEMOE_ECUDA.
 *   - One handle serves one stream at a time (its workspace is shared by
 *     consecutive calls). Use one handle per concurrent stream.
 *   - bf16 tensors are passed as uint16_t bit patterns; all tensors are
 *     row-major and contiguous, 16-byte aligned.
 */
#ifndef MUSEMOE_H
#define MUSEMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *musemoe_stream_t; /* a cudaStream_t */
typedef struct CUevent_st *musemoe_event_t;   /* a cudaEvent_t */
typedef struct musemoe_handle musemoe_handle;

typedef enum {
  MUSEMOE_OK = 0,
  MUSEMOE_EINVAL = 1,       /* bad argument: null, misaligned, out of range */
  MUSEMOE_EUNSUPPORTED = 2, /* a configuration or device the kernels do not serve */
  MUSEMOE_ECUDA = 3,        /* a CUDA runtime call or launch failed */
  MUSEMOE_ENOMEM = 4,       /* workspace allocation failed (create only) */
  MUSEMOE_ERANGE = 5,       /* health: an expert operand left the fp16 range */
  MUSEMOE_ETIMEOUT = 6,     /* health: a kernel's bounded wait ran out */
} musemoe_status;

typedef enum {
  /* e2m1 codes + UE8M0 scale per 32 along K (page
   * "vllm.models.muse_spark.amd.mono.decoder", MonoDims.expert_shapes) */
  MUSEMOE_MXFP4 = 0,
  /* e2m1 codes + e4m3 scale per 16 along K + fp32 global scale per expert */
  MUSEMOE_NVFP4 = 1,
  /* e4m3 codes + fp32 scale per output row; expert inputs quantized to e4m3
   * per row with a dynamic fp32 scale (amax / 448) */
  MUSEMOE_FP8_W8A8 = 2,
  /* unquantized bf16 experts, the form the first and last decoder layers
   * keep (page "vllm.models.muse_spark.amd.muse_moe_runner",
   * MuseSparkUnquantizedFusedMoE and _online_mxfp4_applies); no scales */
  MUSEMOE_BF16 = 3,
  /* W4A4: MXFP4 weights (as MUSEMOE_MXFP4) and both expert inputs, h per
   * token and SiLU(gate)*up per route, rounded dynamically to MXFP4 (OCP
   * rule: scale 2^(floor(log2 amax) - 2) per 32, nearest e2m1, ties to
   * even); page "vllm.models.muse_spark.amd.muse_moe_runner", the Quark
   * w_mxfp4_a_mxfp4 scheme. One extra launch (act_quant) per forward. The
   * W4A4 forms multiply e2m1 by e2m1 on the block-scaled FP4 tensor cores
   * (tcgen05.mma kind::mxf4nvf4) at every batch size; musemoe_pack_experts
   * lays their weights out for that kernel only. */
  MUSEMOE_MXFP4_A4 = 4,
  /* W4A4: NVFP4 weights (as MUSEMOE_NVFP4) and both expert inputs rounded
   * to NVFP4 (e4m3 scale nearest amax / 6 per 16, no global scale;
   * providers page, ExpertsInput); the FP4 tensor cores as above. */
  MUSEMOE_NVFP4_A4 = 5,
} musemoe_quant;

typedef enum { MUSEMOE_SIGMOID = 0, MUSEMOE_SOFTMAX = 1 } musemoe_score;

/* Which kernels run the routed experts (musemoe_set_expert_path). */
typedef enum {
  /* the tensor-core (tcgen05) kernels above 32 rows, where a hot expert's
   * token group is a dense contraction; the warp-level kernels below (the
   * W4A4 forms: the FP4 tensor cores at every size) */
  MUSEMOE_PATH_AUTO = 0,
  MUSEMOE_PATH_MMA = 1,     /* always the warp-level (mma.sync) kernels (not W4A4) */
  MUSEMOE_PATH_TCGEN05 = 2, /* always the tensor-core kernels (not BF16) */
} musemoe_expert_path;

/* Block sizes. hidden H, pooled P, inter I (per expert), experts E. */
typedef struct {
  int32_t max_rows; /* largest `rows` any call of this handle will pass */
  int32_t hidden;   /* H: multiple of 32 */
  int32_t pooled;   /* P: multiple of 128 */
  int32_t inter;    /* I: multiple of 128 */
  int32_t experts;  /* E: 1..256 */
  int32_t top_k;    /* k: 1..E */
} musemoe_dims;

/* Routing rule and norm parameters (MuseSpark1xRouter constructor). */
typedef struct {
  int32_t score;            /* musemoe_score */
  float route_scale;
  int32_t has_multiplier;   /* 0: router_output_multiplier is None */
  float multiplier;
  int32_t has_division_eps; /* 0: router_score_division_eps is None */
  float division_eps;
  float norm_eps;           /* epsilon of all four RMSNorms */
  int32_t pre_expert_norm;  /* 1: apply the pre-expert RMSNorm (default) */
} musemoe_config;

/* One layer's weights: caller-owned device pointers, read in place.
 * Expert codes and scales must be in the kernel layout musemoe_pack_experts
 * writes. */
typedef struct {
  const float *w_router;      /* fp32 [E, H] */
  const float *expert_bias;   /* fp32 [E], selection only */
  const uint16_t *w_pool;     /* bf16 [P, H] */
  const uint16_t *w_pre_norm; /* bf16 [P] (effective weight) */
  const uint8_t *w13;         /* kernel layout of [E, 2I, P/2] (FP4) / [E, 2I, P] (FP8) / bf16 [E, 2I, P] */
  const void *w13_scale;      /* kernel layout: MX u8, NV e4m3; FP8 fp32 [E, 2I]; BF16 unused */
  const float *w13_gscale;    /* NVFP4 only: fp32 [E] */
  const uint8_t *w2;          /* kernel layout of [E, P, I/2] (FP4) / [E, P, I] (FP8) / bf16 [E, P, I] */
  const void *w2_scale;       /* kernel layout: MX u8, NV e4m3; FP8 fp32 [E, P]; BF16 unused */
  const float *w2_gscale;     /* NVFP4 only: fp32 [E] */
  const uint16_t *w_post_norm; /* bf16 [P] */
  const uint16_t *w_unpool;    /* bf16 [H, P] */
  const uint16_t *w_ffn_norm;  /* bf16 [H] (post_ffn_norm) */
  const uint16_t *w_next_norm; /* bf16 [H] (the next layer's pre-norm) */
  const float *gate;           /* fp32 [1]: the gated add's per-layer gate */
} musemoe_weights;

/* Optional device buffers that musemoe_forward_debug fills (each may be
 * NULL) and optional events recorded around every kernel. */
typedef struct {
  float *logits;          /* fp32 [rows, E] router logits */
  int32_t *ids;           /* int32 [rows, k] selected experts, best first */
  float *weights;         /* fp32 [rows, k] routing weights */
  uint16_t *h;            /* bf16 [rows, P] pre-expert-normed pooled input */
  uint16_t *act;          /* [rows * k, I] SiLU(gate) * up per route: f16 bits for
                             MXFP4/NVFP4, bf16 bits for FP8 W8A8 */
  float *y;               /* fp32 [rows * k, P] unweighted route outputs */
  uint16_t *moe_out;      /* bf16 [rows, P] */
  float *u;               /* fp32 [rows, H] unpooler output */
  musemoe_event_t *events; /* 2 * musemoe_num_kernels(quant) existing events:
                              start and end of kernel i at [2i] and [2i+1];
                              an event that cannot be recorded gives EINVAL.
                              With events the kernels run without programmatic
                              dependent launch, so each is timed alone. */
} musemoe_taps;

/* Validates dims/quant/config against the kernels (every reason is listed
 * in the error text) and allocates the workspace on the current device.
 * Returns EUNSUPPORTED for dims the kernels do not serve or a device that is
 * not sm_103, EINVAL for null/invalid arguments, ENOMEM/ECUDA on allocation
 * failure. On failure *out is NULL and musemoe_last_error(NULL) says why. */
musemoe_status musemoe_create(const musemoe_dims *dims, int32_t quant,
                              const musemoe_config *config, musemoe_handle **out);

/* Frees the workspace (synchronizes the device first). NULL is a no-op. */
void musemoe_destroy(musemoe_handle *handle);

/* The last error text of this handle; with NULL, the calling thread's last
 * musemoe_create / musemoe_pack_experts error. Never NULL. */
const char *musemoe_last_error(const musemoe_handle *handle);

/* Device workspace bytes musemoe_create allocates for these dims. */
size_t musemoe_workspace_bytes(const musemoe_dims *dims, int32_t quant);

/* Stages one musemoe_forward runs for this quant (for taps->events): one
 * kernel each, except that above 8 rows the "pool" stage is two launches
 * (the pooler GEMV, or above 32 rows the dense tensor-core GEMM, then the
 * pre-expert norm), and for W4A4 one more (h rounded to FP4), timed
 * together. */
int32_t musemoe_num_kernels(int32_t quant);
/* Name of stage i of the forward ("router", "pool", "w13", ...). */
const char *musemoe_kernel_name(int32_t quant, int32_t i);

/* Re-lays the expert tensors from their plain layout into the kernel layout
 * the forward reads (done once, e.g. after loading weights).
 * Plain layout: codes row-major [E, N, K/2] for MXFP4/NVFP4 (two e2m1 codes
 * per byte, element 2j in the low nibble of byte j), [E, N, K] e4m3 for FP8 or
 * [E, N, K] bf16 for BF16; scales [E, N, K/32] UE8M0 (MXFP4), [E, N, K/16]
 * e4m3 (NVFP4), fp32 [E, N] (FP8), none for BF16 (the scale pointers may be
 * NULL). w13: N = 2I (gate rows first), K = P; w2: N = P, K = I.
 * Kernel layout: every row is cut into 64-byte code chunks (128 FP4, 64 FP8 or
 * 32 BF16 elements); rows are taken in tiles of 64, each tile is stored K-slice by
 * K-slice (4 chunks; the last slice holds the remaining 1..4), each slice by
 * group of 8 rows, then chunk, then row: codes
 * [E][N/64][slice][8 groups][chunks of the slice][8 rows][64 B]; scales the
 * same with the 4 (MXFP4) or 8 (NVFP4) scale bytes of a row's chunk in place
 * of its 64 code bytes; FP8 scales keep their layout. For FP4 the 64 bytes of
 * a chunk are also reordered: byte 8j + 2q + b moves to 16q + 2j + b (q < 4,
 * j < 8, b < 2); for BF16 its 4-byte words are transposed as a 4 x 4 block:
 * byte 16j + 4q + b moves to 16q + 4j + b (q, j, b < 4). FP8 and the W4A4
 * forms keep the bytes of a chunk in order but swizzle its 16-byte units
 * within each [8 rows][64 B] block (unit u of row r stored at unit
 * u ^ ((r >> 1) & 3), the tensor cores' 64-byte swizzle). W4A4 scales are
 * laid out as the tensor cores' scale atoms instead: per expert, tile of 128
 * rows (w13: gate rows 64t.. and up rows I + 64t.. interleaved by groups of
 * 8 rows, row m of the tile in group m / 8, even groups gate; w2: rows
 * 128t..), K-slice of 4 chunks and atom of 4 scale blocks (MXFP4: one chunk,
 * NVFP4: half a chunk), 512 bytes holding the scale of tile row m and block
 * j at byte (m % 32) * 16 + (m / 32) * 4 + j:
 * [E][tiles][slice][atoms of the slice][512 B]. Each src may be its
 * dst (in place): the tensors then pass
 * through a temporary device buffer of at most 64 MB, allocated and freed by
 * this call, which synchronizes the stream before it returns. The NVFP4
 * global scales need no re-layout. MXFP4 scales must be UE8M0 codes
 * 0x01..0xFE (0x00 = 2^-127 and 0xFF = NaN give EUNSUPPORTED, nothing is
 * re-laid); with MXFP4 the call synchronizes the stream to read that check. */
musemoe_status musemoe_pack_experts(const musemoe_dims *dims, int32_t quant,
                                    const uint8_t *w13_src, const void *w13_scale_src,
                                    uint8_t *w13_dst, void *w13_scale_dst,
                                    const uint8_t *w2_src, const void *w2_scale_src,
                                    uint8_t *w2_dst, void *w2_scale_dst,
                                    musemoe_stream_t stream);

/* Router GEMV + routing rule only: ids_out int32 [rows, k] (descending
 * selection score, equal scores to the lower expert id), weights_out fp32
 * [rows, k]. Needs w->w_router and w->expert_bias. */
musemoe_status musemoe_route(musemoe_handle *handle, const musemoe_weights *w,
                             const uint16_t *x, int32_t rows, int32_t *ids_out,
                             float *weights_out, musemoe_stream_t stream);

/* The whole block: x bf16 [rows, H] in; stream fp32 [rows, H] updated in
 * place; out bf16 [rows, H] (the next layer's input). 1 <= rows <= max_rows. */
musemoe_status musemoe_forward(musemoe_handle *handle, const musemoe_weights *w,
                               const uint16_t *x, float *stream, uint16_t *out,
                               int32_t rows, musemoe_stream_t stream_);

/* musemoe_forward plus the taps (any may be NULL). */
musemoe_status musemoe_forward_debug(musemoe_handle *handle, const musemoe_weights *w,
                                     const uint16_t *x, float *stream, uint16_t *out,
                                     int32_t rows, musemoe_stream_t stream_,
                                     const musemoe_taps *taps);

/* Expert parallelism, the rank's half of the block (page
 * "vllm.models.muse_spark.amd.mono.decoder", deployment_refusals and
 * MonoDims: expert parallel ranks each hold experts [r E/g, (r+1) E/g); page
 * "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
 * MoEProvider: the tail's EP combine). Runs the replicated front (router,
 * routing rule, pooler + pre-expert norm) on all rows, the routed experts
 * for the routes whose expert lies in [expert_first, expert_first +
 * expert_count) only, and the post-expert norm and router weight of those
 * routes, and writes their sum per row to moe_partial, fp32 [rows, pooled]
 * (no bf16 rounding: the ranks' partials are summed first, by the caller's
 * all-reduce). w->w_router and w->expert_bias hold all experts; w13, w2 and
 * their scales (NVFP4: global scales) hold the rank's expert_count experts,
 * packed by musemoe_pack_experts with dims->experts = expert_count. Device
 * pointers, 16-byte aligned; asynchronous; allocates nothing. EINVAL for an
 * empty or out-of-range expert range or missing tensors. */
musemoe_status musemoe_forward_ep_partial(musemoe_handle *handle, const musemoe_weights *w,
                                         const uint16_t *x, float *moe_partial, int32_t rows,
                                         int32_t expert_first, int32_t expert_count,
                                         musemoe_stream_t stream_);

/* The replicated back of an expert-parallel block: moe_out = bf16(moe_sum)
 * (moe_sum fp32 [rows, pooled], the all-reduced sum of every rank's
 * moe_partial), then the unpooler and the FFN boundary into stream_io (fp32,
 * in place) and out (bf16), as musemoe_forward ends. Uses w->w_unpool,
 * w_ffn_norm, w_next_norm and gate. With one rank holding every expert,
 * partial + combine equals musemoe_forward bit for bit. */
musemoe_status musemoe_forward_ep_combine(musemoe_handle *handle, const musemoe_weights *w,
                                         const float *moe_sum, float *stream_io, uint16_t *out,
                                         int32_t rows, musemoe_stream_t stream_);

/* musemoe_forward on HOST buffers (pinned memory recommended): copies x and
 * stream to the workspace, runs the block, copies stream and out back and
 * synchronizes the stream. Not graph-capturable. */
musemoe_status musemoe_forward_host(musemoe_handle *handle, const musemoe_weights *w,
                                    const uint16_t *x_host, float *stream_host,
                                    uint16_t *out_host, int32_t rows,
                                    musemoe_stream_t stream_);

/* No allocation: the router GEMV + routing rule of musemoe_route without a
 * handle, for callers that cannot allocate device memory (their memory
 * belongs to another allocator, such as a serving engine's pooled one, or a
 * new allocation is not allowed where they run). The source pages have no
 * counterpart: it is a calling convention of this library. Inputs and
 * outputs as musemoe_route (w_router fp32 [experts, hidden], expert_bias
 * fp32 [experts], x bf16 [rows, hidden] -> ids_out int32 [rows, top_k],
 * weights_out fp32 [rows, top_k]); hidden a multiple of 64 up to 8192
 * (larger gives EUNSUPPORTED), experts 1..256, rows
 * 1..MUSEMOE_STATIC_MAX_ROWS (larger gives EINVAL with the reason in
 * musemoe_last_error(NULL)). A non-NULL stream must belong to the current
 * device (else EINVAL): the scratch used is the current device's.
 * The scratch (the fp32 logits) is one fixed device array of
 * MUSEMOE_STATIC_SCRATCH_BYTES inside the library, held on every device
 * that loads the library until the process exits; the call makes no
 * cudaMalloc/cudaFree or other allocation. The first call on a device looks
 * up that array's device address (cudaGetSymbolAddress, with the device
 * current): make it before any stream capture. Every call shares the array
 * and the array keeps the last call's contents; nothing in it has to start
 * at zero (the router writes every logit the routing reads). Calls that
 * overlap on the GPU (e.g. on two streams) race on the array: serialize
 * them. */
#define MUSEMOE_STATIC_MAX_ROWS 64
#define MUSEMOE_STATIC_SCRATCH_BYTES (64 * 1024)
musemoe_status musemoe_route_static(int32_t hidden, int32_t experts, int32_t top_k,
                                    const musemoe_config *config, const float *w_router,
                                    const float *expert_bias, const uint16_t *x, int32_t rows,
                                    int32_t *ids_out, float *weights_out,
                                    musemoe_stream_t stream);

/* Attention boundary, the step before the block (page
 * "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
 * AttentionBoundaryProvider docstring; post_attn_norm has no weight: page
 * "vllm.models.muse_spark.amd.mono.decoder", the weight check of each
 * layer): stream += gate * RMSNorm(partial) (weightless) into the fp32
 * residual stream in place, then out = bf16(RMSNorm(stream) * w_pre_ffn_norm),
 * the block's input x. partial bf16 [rows, hidden] is the o_proj output
 * already summed over ranks (this library has no all-reduce). gate: one fp32
 * on the device; w_pre_ffn_norm: the effective bf16 weight [hidden]. Every
 * pointer is device memory, 16-byte aligned; the caller owns all of them.
 * hidden a multiple of 4, at most 8192; rows >= 1; eps >= 0. No handle and
 * no allocation; asynchronous on stream. EINVAL with the reason in
 * musemoe_last_error(NULL) on bad arguments (nothing launched), ECUDA if the
 * launch fails. */
musemoe_status musemoe_attention_boundary(const uint16_t *partial, float *stream_io,
                                          uint16_t *out, const uint16_t *w_pre_ffn_norm,
                                          const float *gate, int32_t rows, int32_t hidden,
                                          float eps, musemoe_stream_t stream);

/* Online rounding of BF16 expert weights to MXFP4 (page
 * "vllm.models.muse_spark.amd.muse_moe_runner", _quantize_experts_to_mxfp4,
 * which rounds the experts of every decoder layer but the first and the
 * last on load). w_bf16 [rows, cols] bf16 (finite values), cols a multiple
 * of 32 -> codes [rows, cols/2] (two e2m1 codes per byte, element 2j in the
 * low nibble) and scales [rows, cols/32] (UE8M0), the plain layout that
 * musemoe_pack_experts takes as its source. Per block of 32 elements: scale
 * 2^(floor(log2(amax)) - 2) with the exponent clamped to [-126, 127] (2^0
 * for an all-zero block); each element the e2m1 value nearest v / scale,
 * ties to the even code, saturating at +-6, sign kept. Device pointers:
 * w_bf16 and codes 16-byte aligned; the caller owns them. No handle and no
 * allocation; asynchronous on stream. EINVAL with the reason in
 * musemoe_last_error(NULL) on bad arguments, ECUDA if the launch fails. */
musemoe_status musemoe_quantize_mxfp4(const uint16_t *w_bf16, uint8_t *codes, uint8_t *scales,
                                      int64_t rows, int32_t cols, musemoe_stream_t stream);

/* The NVFP4 expert input (page
 * "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
 * ExpertsInput): bf16 activations [rows, cols] -> e2m1 codes [rows, cols/2]
 * (element 2j in the low nibble of byte j) and e4m3 block scales
 * [rows, cols/16]. Per 16 elements the scale is the e4m3 value nearest
 * fp32(amax / 6) (ties to even, saturating at 448); each element takes the
 * e2m1 magnitude nearest fp32(|v| / scale), ties to the even code,
 * saturating at 6, sign kept; a block whose scale is 0 gets magnitude 0.
 * The same rounding as the MUSEMOE_NVFP4_A4 forward. Device pointers:
 * x_bf16 and codes 16-byte aligned; cols a multiple of 16; the caller owns
 * them. No handle and no allocation; asynchronous on stream. EINVAL with the
 * reason in musemoe_last_error(NULL) on bad arguments, ECUDA if the launch
 * fails. (The MXFP4 expert input of MUSEMOE_MXFP4_A4 is
 * musemoe_quantize_mxfp4 applied to the activations.) */
musemoe_status musemoe_quantize_act_nvfp4(const uint16_t *x_bf16, uint8_t *codes, uint8_t *scales,
                                          int64_t rows, int32_t cols, musemoe_stream_t stream);

/* Health self-test: runs the library's two bounded waits once on the
 * handle's device, each on something nothing ever completes (an mbarrier
 * phase, as a stage whose weight copies never land; a flag, as a split
 * tile's owner waiting for a partial that never comes). Each gives up after
 * its limit (200 ms) and records the timeout in the health word exactly as a
 * forward would, so the next musemoe_poll_health returns MUSEMOE_ETIMEOUT
 * and the context stays usable. It also leaves the expert kernels' split-tile
 * tickets raised, as contributors arriving after their owner gave up
 * would. For checking the failure path of a deployment; synchronizes the
 * stream; not concurrent with forwards on the same handle. */
musemoe_status musemoe_health_selftest(musemoe_handle *handle, musemoe_stream_t stream);

/* Reads (synchronously) and clears the handle's device health word. Returns
 * MUSEMOE_ETIMEOUT if an expert kernel's bounded wait for its weight copies
 * ran out since the last poll (that forward's outputs are invalid; the poll
 * then zeroes every inter-CTA ticket of the handle, so the next forward
 * starts clean),
 * MUSEMOE_ERANGE if a forward produced an expert operand (h or the
 * SiLU(gate)*up activation) beyond the fp16 range (|v| > 65504; W4A4: a
 * value that is not finite) or, on the tensor-core
 * expert kernels, met an MXFP4 block scale outside 2^-23..2^13 (its products
 * with e2m1 are exact f16 operands only inside), MUSEMOE_OK otherwise. */
musemoe_status musemoe_poll_health(musemoe_handle *handle);

/* Selects the routed-expert kernels of the handle's later forwards
 * (musemoe_expert_path; AUTO after create). Both paths compute the same
 * block (page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.
 * providers", RoutedExpertsOps: the routed experts of the MoE provider) with
 * the same operands and fp32 accumulation; they differ in summation order.
 * The tensor-core path (tcgen05.mma: kind::f8f6f4 for FP8, kind::f16 on
 * dequantized FP4, kind::mxf4nvf4 block-scaled for the W4A4 forms) serves
 * MXFP4, NVFP4, FP8 and W4A4; TCGEN05 on a BF16 handle and MMA on a W4A4
 * handle are EUNSUPPORTED. EINVAL for an unknown path. Host only; not
 * concurrent with a forward on the handle. */
musemoe_status musemoe_set_expert_path(musemoe_handle *handle, int32_t path);

#ifdef __cplusplus
}
#endif
#endif /* MUSEMOE_H */
