/*
 * flint_moe.h — C ABI of the Flint small-batch decode MoE layer for GB300 (sm_103a).
 *
 * The layer: hidden 2048, 256 routed experts scored by a sigmoid and selected
 * top-6, plus one always-on shared expert; every expert is a SwiGLU FFN
 * (gate/up projection, SiLU-and-mul, down projection).
 *   - "256 routed experts with top-6 sigmoid routing plus one shared expert",
 *     "Qwen3-MoE-style decoder": [Flint on Intel Arc Pro B70, "Setup"].
 *   - "hidden size of 2048", "256 experts, sigmoid top-6 selection plus a
 *     shared expert": [vLLM Day-0 Support for Recursive's Flint,
 *     "Flint Model Architecture"].
 *   - "router and expert GEMVs ... read only the selected experts' weights":
 *     [vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies",
 *     "Small-batch MoE Kernels"].
 *   - SiLU written as g / (1 + exp(-g)): [Flint on Intel Arc Pro B70,
 *     "norm.py: Triton kernels that assumed CUDA"].
 *   - NVFP4 weights run weight-only (W4A16) with BF16 activations:
 *     [vLLM Day-0 Support for Recursive's Flint, "Flint Model Overview and
 *     Capabilities"]; [RecursiveSI/flint — vLLM serving recipe, "Guide",
 *     "Overview"].
 * The intermediate (expert FFN) size is not given by the pages; this library
 * is specialised to 512.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer, owned by the caller.  Weight,
 *    activation and workspace pointers must be 16-byte aligned; the small
 *    fp32 / int32 vectors (logit offsets, tensor scales, routing outputs,
 *    bucket outputs) need only 4-byte alignment.  Tensors are dense and
 *    row-major in the shapes written beside each argument.  bf16 tensors are
 *    passed as `const void*` holding IEEE bfloat16 bit patterns.
 *  - The library allocates no device or host memory.  Scratch lives in a
 *    caller-provided workspace (see flint_moe_workspace_bytes /
 *    flint_moe_workspace_init), which also keeps a count of the calls made on
 *    it (the batch <= 8 kernels tell this call's data from older data by it).
 *    Two calls may run concurrently only with distinct workspaces.  The one
 *    exception to all of this is flint_moe_decode_bf16_noalloc (below), which
 *    uses a static device array of the library instead of a workspace.
 *  - Calls validate their arguments on the host and return an error status
 *    BEFORE any launch if anything is wrong; nothing is then written.  On
 *    FLINT_OK, the work has been enqueued on `stream` and nothing has been
 *    synchronised (except in the first flint_moe_decode_bf16_noalloc call on
 *    a device): results are visible after the caller's next sync on that
 *    stream.  Launch failures reported by the runtime map to FLINT_ERR_CUDA.
 *  - BF16 decode calls of batch <= 8 and NVFP4 decode calls of batch <= 2
 *    run one persistent kernel whose CTAs, one per SM, exchange data while
 *    they run.  It is launched as a cooperative
 *    grid, which the runtime starts only when every CTA can be resident at
 *    once and otherwise refuses (FLINT_ERR_CUDA, e.g. in a context limited to
 *    fewer SMs).  While it runs it occupies every SM: kernels of other streams
 *    wait for it, and it waits for them to leave the SMs before it starts.
 *  - Every wait inside a kernel is bounded by a time limit stored in the
 *    workspace.  A kernel that runs out of time records
 *    FLINT_ERR_DEVICE_TIMEOUT in the workspace's error word, waits (bounded)
 *    for its own asynchronous copies and returns; read the word with
 *    flint_moe_get_device_status.  The outputs of such a call are undefined,
 *    and the workspace must be re-initialised before the next call.
 *  - Routing: router scores are computed in fp32 from bf16 inputs and the
 *    logit offsets (if any) are added to them in fp32.  Experts are ranked by
 *    (score + offset descending, expert index ascending), the first top_k are
 *    kept, and each kept expert's weight is sigmoid(score + offset) -- or
 *    sigmoid(score) with FLINT_OFFSET_SELECT -- divided by the sum over the
 *    kept experts (so the weights sum to 1).  topk_idx rows list the experts
 *    in that rank order.
 */
#ifndef FLINT_MOE_H_
#define FLINT_MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLINT_OK = 0,
  FLINT_ERR_INVALID_ARG = 1,    /* NULL / misaligned pointer, bad batch, aliasing, bad input */
  FLINT_ERR_UNSUPPORTED = 2,    /* dims other than the specialised shape */
  FLINT_ERR_WORKSPACE = 3,      /* workspace NULL or smaller than required */
  FLINT_ERR_CUDA = 4,           /* the CUDA runtime reported an error */
  FLINT_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait ran out */
} flint_status;

/* What per-expert logit offsets (logit_bias) change.  The pages give only
 * "sigmoid top-6 selection" ([vLLM Day-0 Support for Recursive's Flint,
 * "Flint Model Architecture"]) and no offsets; both common conventions are
 * offered:
 *   FLINT_OFFSET_LOGIT  (0, default): the offset is added to the router score
 *     before ranking and before the sigmoid, so it moves both the selection
 *     and the weights;
 *   FLINT_OFFSET_SELECT (1): experts are ranked by score + offset, but each
 *     kept expert's weight is the sigmoid of its score without the offset
 *     (renormalised over the kept experts), so the offset steers the
 *     selection only. */
#define FLINT_OFFSET_LOGIT 0
#define FLINT_OFFSET_SELECT 1

/* Layer shape and routing convention.  Supported: hidden 2048, n_experts 256,
 * top_k 6, inter 512, n_shared 1, offset_mode FLINT_OFFSET_LOGIT or
 * FLINT_OFFSET_SELECT.  Any other value returns FLINT_ERR_UNSUPPORTED.  A
 * zero-initialised offset_mode is the default convention. */
typedef struct {
  int32_t hidden;       /* H */
  int32_t n_experts;    /* E, routed experts */
  int32_t top_k;        /* k, experts selected per token */
  int32_t inter;        /* I, expert intermediate size */
  int32_t n_shared;     /* S, always-on shared experts (added with weight 1) */
  int32_t offset_mode;  /* FLINT_OFFSET_LOGIT or FLINT_OFFSET_SELECT */
} flint_moe_dims;

/* Largest batch (tokens per call) any entry point accepts. */
#define FLINT_MOE_MAX_BATCH 256

/* Human-readable name of a status code.  Never NULL. */
const char* flint_status_string(flint_status status);

/* Bytes of workspace a call with `max_batch` tokens needs (0 if the dims are
 * unsupported or max_batch is outside [1, FLINT_MOE_MAX_BATCH]).  One
 * workspace sized for max_batch serves every call with batch <= max_batch. */
size_t flint_moe_workspace_bytes(const flint_moe_dims* dims, int32_t max_batch);

/* Prepares a workspace for use: zero-fills it (cudaMemsetAsync on `stream`)
 * and stores the device-side wait limit.  wait_limit_ns = 0 selects the
 * default limit of one second.  Must be called once before the first call
 * that uses the workspace, and again after any call whose device status was
 * not FLINT_OK.  Every successful call leaves the workspace ready for the
 * next one. */
flint_status flint_moe_workspace_init(void* workspace, size_t ws_bytes,
                                      uint64_t wait_limit_ns, cudaStream_t stream);

/* Synchronises `stream`, then reads and returns the workspace's device error
 * word: FLINT_OK, FLINT_ERR_DEVICE_TIMEOUT, or FLINT_ERR_INVALID_ARG when
 * flint_moe_bucket was given a routing row that is not k distinct experts or
 * an NVFP4 call met an activation (x, or h above 2 tokens) beyond the range
 * its f16 operands hold. */
flint_status flint_moe_get_device_status(const void* workspace, cudaStream_t stream);

/* Router only: logits, sigmoid top-k, renormalised weights.
 *   x_bf16        [batch, H]   token activations (already normalised)
 *   w_router_bf16 [E, H]       router matrix
 *   logit_bias    [E] fp32 or NULL; per-expert logit offsets, applied as
 *                 dims->offset_mode says (by default added to the logit
 *                 before ranking and before the sigmoid)
 *   topk_idx      [batch, k]   int32 out, expert ids in rank order
 *   topk_w        [batch, k]   fp32 out, renormalised weights
 * Also leaves the token-to-expert buckets in the workspace for the stage
 * calls below (flint_moe_gateup_bf16 / flint_moe_down_bf16).
 * Router matrix and logits follow "sigmoid top-6" routing:
 * [vLLM Day-0 Support for Recursive's Flint, "Flint Model Architecture"]. */
flint_status flint_moe_route(const flint_moe_dims* dims, int32_t batch,
                             const void* x_bf16, const void* w_router_bf16,
                             const float* logit_bias,
                             int32_t* topk_idx, float* topk_w,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Token-to-expert bucketing alone: the dedup pass the decode calls run after
 * routing, so that each selected expert's weights are read once per batch
 * ("router and expert GEMVs ... read only the selected experts' weights":
 * [vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies"]).
 *   topk_idx [batch, k] int32   device routing; every row must hold k distinct
 *                               experts in [0, E) (otherwise the device error
 *                               word becomes FLINT_ERR_INVALID_ARG and the
 *                               outputs are undefined)
 *   uniq     [E]   int32 out    distinct experts, ascending (first n_uniq valid)
 *   offsets  [E+1] int32 out    first pair of each distinct expert; entry n_uniq
 *                               holds batch*k
 *   pairs    [batch*k] int32 out  token*8 + slot, ordered by (expert, token)
 *   n_uniq   [1]   int32 out
 * Uses (and leaves ready) the workspace like the other calls. */
flint_status flint_moe_bucket(const flint_moe_dims* dims, int32_t batch,
                              const int32_t* topk_idx, int32_t* uniq, int32_t* offsets,
                              int32_t* pairs, int32_t* n_uniq,
                              void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The whole BF16 decode MoE layer:
 *   out[t] = residual[t] + sum_s FFN_shared_s(x[t])
 *                        + sum_{j<k} topk_w[t,j] * FFN_{topk_idx[t,j]}(x[t])
 *   FFN_e(v) = Wd_e ( silu(Wg_e v) * (Wu_e v) ),  silu(g) = g / (1 + exp(-g))
 * Only the selected experts' weights, the shared expert and the router are
 * read ("read only the selected experts' weights":
 * [vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies"]).
 *   x_bf16, residual_bf16 [batch, H]
 *   w_router_bf16 [E, H]; logit_bias [E] fp32 or NULL (as flint_moe_route)
 *   w13_bf16  [E, 2I, H]   rows 0..I-1 are Wg, rows I..2I-1 are Wu
 *   w2_bf16   [E, H, I]    Wd
 *   ws13_bf16 [S, 2I, H], ws2_bf16 [S, H, I]  shared expert(s), same layout
 *   out_bf16  [batch, H]   out; may alias residual_bf16 exactly (in-place
 *                          residual add); no other overlap is allowed
 *   topk_idx_out [batch, k] int32, topk_w_out [batch, k] fp32: optional
 *                          copies of the routing (NULL to skip)
  * Accumulation is fp32 and `out` is rounded to bf16 once.  The SiLU-and-mul
 * output h is kept in fp32 for batches of <= 8 tokens and as a bf16 pair
 * hi + lo (about 16 significant bits, the range of fp32) above that. */
flint_status flint_moe_decode_bf16(const flint_moe_dims* dims, int32_t batch,
                                   const void* x_bf16, const void* residual_bf16,
                                   const void* w_router_bf16, const float* logit_bias,
                                   const void* w13_bf16, const void* w2_bf16,
                                   const void* ws13_bf16, const void* ws2_bf16,
                                   void* out_bf16,
                                   int32_t* topk_idx_out, float* topk_w_out,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The two expert stages of flint_moe_decode_bf16, callable on their own.
 * They use the routing and buckets that the last flint_moe_route or decode
 * call left in `workspace` (same batch, earlier on the same stream), so
 *   flint_moe_route; flint_moe_gateup_bf16; flint_moe_down_bf16
 * computes exactly what flint_moe_decode_bf16 computes (with the routing
 * copies written by flint_moe_route).
 * flint_moe_gateup_bf16: for every selected (token, expert) pair and for the
 *   shared expert(s), h = silu(Wg x) * (Wu x), kept in the workspace (each
 *   fp32 value as a bf16 pair hi + lo, ~16 significant bits).
 * flint_moe_down_bf16: out = residual + sum of the routing-weighted
 *   Wd h terms + the shared expert's Wd h ("expert combine" fused into the
 *   down GEMV: [vLLM Day-0 Support for Recursive's Flint, "Optimization
 *   Strategies", "Low-Latency Decode Path"]).  out may alias residual exactly.
 * Arguments as in flint_moe_decode_bf16. */
flint_status flint_moe_gateup_bf16(const flint_moe_dims* dims, int32_t batch,
                                   const void* x_bf16, const void* w13_bf16,
                                   const void* ws13_bf16,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream);
flint_status flint_moe_down_bf16(const flint_moe_dims* dims, int32_t batch,
                                 const void* residual_bf16, const void* w2_bf16,
                                 const void* ws2_bf16, void* out_bf16,
                                 void* workspace, size_t ws_bytes, cudaStream_t stream);

/* NVFP4 weight-only (W4A16) variant of flint_moe_decode_bf16.  The router,
 * activations and output stay bf16.  Each expert projection is stored as
 *   q   uint8 [rows, K/2]   e2m1 codes; byte j holds k = 2j in its low nibble
 *                           and k = 2j+1 in its high nibble
 *   sf  uint8 [rows, K/16]  OCP E4M3FN scale of each block of 16 consecutive k
 *   ts  fp32                one tensor scale per (expert, projection)
 * and dequantises to W[r,k] = e2m1(q) * e4m3(sf[r, k/16]) * ts.
 * The products e2m1 * e4m3 are exact in f16 and multiply f16 activations on
 * the tensor cores, so every activation must satisfy |x| < 65504 (an
 * RMS-normalised x is below sqrt(H) = 45.3): a larger one sets the device
 * status to FLINT_ERR_INVALID_ARG, and the outputs are undefined.  h is kept
 * as h / 256 in an f16 pair hi + lo (about 22 significant bits), which holds
 * |h| < 65520 * 256 (~1.7e7): a larger h also sets FLINT_ERR_INVALID_ARG.
 *   w13_q [E, 2I, H/2], w13_sf [E, 2I, H/16], w13_ts [E, 2] (gate, up)
 *   w2_q  [E, H, I/2],  w2_sf  [E, H, I/16],  w2_ts  [E]
 *   ws13_q/ws13_sf/ws13_ts and ws2_q/ws2_sf/ws2_ts: the shared expert(s),
 *   same layouts with S in place of E.
 * NVFP4 with BF16 activations: [vLLM Day-0 Support for Recursive's Flint,
 * "Flint Model Overview and Capabilities"]. */
flint_status flint_moe_decode_nvfp4_w4a16(
    const flint_moe_dims* dims, int32_t batch,
    const void* x_bf16, const void* residual_bf16,
    const void* w_router_bf16, const float* logit_bias,
    const uint8_t* w13_q, const uint8_t* w13_sf, const float* w13_ts,
    const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_ts,
    const uint8_t* ws13_q, const uint8_t* ws13_sf, const float* ws13_ts,
    const uint8_t* ws2_q, const uint8_t* ws2_sf, const float* ws2_ts,
    void* out_bf16, int32_t* topk_idx_out, float* topk_w_out,
    void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Pre-norm between stacked layers: out[t] = bf16( in[t] / sqrt(mean(in[t]^2) + eps) )
 * (unit gain).  in_bf16 and out_bf16 are [batch, H] and must not overlap.
 * Pre-norm decoder: [vLLM Day-0 Support for Recursive's Flint, "Flint Model
 * Architecture"]. */
flint_status flint_moe_rmsnorm_bf16(const flint_moe_dims* dims, int32_t batch,
                                    const void* in_bf16, void* out_bf16, float eps,
                                    cudaStream_t stream);

/* flint_moe_decode_bf16 with the layer's input RMSNorm folded in: the layer
 * input is x = bf16( residual / sqrt(mean(residual^2) + norm_eps) ) (unit
 * gain, exactly as flint_moe_rmsnorm_bf16 computes it), so a pre-norm stack
 * calls this once per layer on the previous layer's output (pre-norm
 * decoder: [vLLM Day-0 Support for Recursive's Flint, "Flint Model
 * Architecture"]; the low-latency decode path folds the small ops around the
 * MoE GEMVs into them: same page, "Optimization Strategies").  For batches of
 * <= 4 tokens the persistent kernel normalises the rows itself (no extra
 * launch; measured faster there); above that the norm runs first, into the
 * workspace.
 *   residual_bf16 [batch, H]  the pre-norm activations (the residual stream)
 *   norm_eps      >= 0 (a NaN or negative value is FLINT_ERR_INVALID_ARG)
 *   out_bf16      [batch, H]  may alias residual_bf16 exactly; no other
 *                             overlap; residual_bf16 must not overlap the
 *                             workspace
 *   the rest as flint_moe_decode_bf16.
 * Results are bit for bit those of flint_moe_rmsnorm_bf16 into a separate x
 * followed by flint_moe_decode_bf16. */
flint_status flint_moe_decode_bf16_prenorm(const flint_moe_dims* dims, int32_t batch,
                                           const void* residual_bf16, float norm_eps,
                                           const void* w_router_bf16, const float* logit_bias,
                                           const void* w13_bf16, const void* w2_bf16,
                                           const void* ws13_bf16, const void* ws2_bf16,
                                           void* out_bf16,
                                           int32_t* topk_idx_out, float* topk_w_out,
                                           void* workspace, size_t ws_bytes,
                                           cudaStream_t stream);

/* Shape of the attention side of a decode step: query heads, KV heads, head
 * size.  Supported: 32, 4, 128 ("Grouped Query Attention (GQA) with 32 query
 * and 4 KV heads": [vLLM Day-0 Support for Recursive's Flint, "Flint Model
 * Architecture"]; 128 from the same section's 28 KiB of KV per token over its
 * 14 full-attention layers: K and V of 4 heads x 128 bf16 values per layer). */
typedef struct {
  int32_t n_q_heads, n_kv_heads, head_dim;
} flint_attn_dims;

/* The attention side of a decode step fused in one kernel: per-head Q/K
 * RMSNorm, rotary position embedding and the bf16 KV-cache write ("The fusion
 * of Q/K norm, RoPE, and KV-cache write into a single kernel": [vLLM Day-0
 * Support for Recursive's Flint, "Optimization Strategies", "Fused Kernels"]).
 * For each token t (D = head_dim, nq = n_q_heads, nkv = n_kv_heads):
 *   qkv_bf16      [batch, (nq + 2 nkv) * D]: the token's projection row,
 *                 query heads, then key heads, then value heads;
 *   q_norm_bf16, k_norm_bf16 [D]: the learned per-element gains of the
 *                 query and key head norms ("per-head Q/K RMSNorm");
 *   positions     [batch] int32 (device): the token's position;
 *   slot_mapping  [batch] int32 (device): the cache row the token's K and V go
 *                 to; a slot outside [0, cache_slots) writes nothing (a
 *                 negative slot marks a padding token);
 *   q and k heads: n[i] = x[i] / sqrt(mean_i x^2 + eps) * g[i]; then, if
 *                 rope_theta > 0, elements i and i + D/2 turn by the angle
 *                 positions[t] * rope_theta^(-2i/D) (rotate-half pairing;
 *                 rope_theta = 0 for the layers without positional encoding);
 *   q_out_bf16    [batch, nq, D] <- the query heads;
 *   k_cache_bf16, v_cache_bf16 [cache_slots, nkv, D]: row slot_mapping[t]
 *                 <- the key heads, and the value heads unchanged (bit for
 *                 bit); every other row is left as it was.
 * fp32 arithmetic (the angles in fp64), one bf16 rounding per output.  The
 * rotate-half pairing and rope_theta as an argument are this library's
 * readings: the pages name RoPE only.  Errors (before any launch):
 * FLINT_ERR_UNSUPPORTED for other dims; FLINT_ERR_INVALID_ARG for a NULL or
 * misaligned pointer (16 bytes; 4 for positions and slot_mapping), batch
 * outside [1, FLINT_MOE_MAX_BATCH], cache_slots < 1, a negative or
 * non-finite rope_theta or eps, or overlapping outputs / inputs.  Needs no
 * workspace. */
flint_status flint_qk_norm_rope_kv_bf16(const flint_attn_dims* dims, int32_t batch,
                                        const void* qkv_bf16, const void* q_norm_bf16,
                                        const void* k_norm_bf16, const int32_t* positions,
                                        const int32_t* slot_mapping, float rope_theta, float eps,
                                        void* q_out_bf16, void* k_cache_bf16, void* v_cache_bf16,
                                        int64_t cache_slots, cudaStream_t stream);

/* Fault-injection hook for tests: arms a one-shot device-side wait, in the
 * next routing launch on this workspace, on a workspace flag that nothing ever
 * sets.  That wait runs out after the workspace's wait limit and records
 * FLINT_ERR_DEVICE_TIMEOUT, exactly as a stuck pipeline wait would; the
 * kernels then finish without hanging the GPU.  Re-initialise the workspace
 * afterwards. */
flint_status flint_moe_debug_arm_stall(void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Largest batch flint_moe_decode_bf16_noalloc accepts. */
#define FLINT_MOE_NOALLOC_MAX_BATCH 8

/* flint_moe_decode_bf16 for callers that cannot allocate device memory.
 * The pages describe no such entry point: it exists for hosts that own all
 * device memory themselves -- a serving engine that splits the GPU into fixed
 * pools and forbids its plugins to call cudaMalloc, a runtime with a memory
 * budget fixed at build time, a step loop that may never take the allocator's
 * locks -- and so cannot provide the workspace the other entry points take.
 *
 * Instead of a workspace it uses one static device array of this library
 * (about 860 KiB, sized for FLINT_MOE_NOALLOC_MAX_BATCH tokens), which every
 * GPU that loads the library holds until the process exits.  It calls no
 * allocating routine.  Inputs, outputs and their layouts are those of
 * flint_moe_decode_bf16, and so are the results.
 *  - batch must be in [1, FLINT_MOE_NOALLOC_MAX_BATCH]; a larger batch returns
 *    FLINT_ERR_INVALID_ARG before anything is enqueued.
 *  - device_status_out: optional device pointer (4-byte aligned).  After the
 *    layer, the call's device-side status is copied there, in stream order, as
 *    a flint_status code (FLINT_OK, FLINT_ERR_INVALID_ARG for bad routing,
 *    FLINT_ERR_DEVICE_TIMEOUT); it takes the place of
 *    flint_moe_get_device_status, which needs a workspace.
 *  - The first call on a device (the current device) looks up the array's
 *    address, initialises its header and synchronises `stream` once.  Make
 *    that first call before any stream capture: during a capture it returns
 *    FLINT_ERR_CUDA instead.
 *  - Each call clears the header's error word and counters; the array keeps
 *    the rest of the previous call's contents, which the layer overwrites
 *    before reading.
 *  - All calls on a device share the one array: calls whose GPU work overlaps
 *    (other streams, other host threads) race and corrupt each other's
 *    results.  Order them, or use flint_moe_decode_bf16 with one workspace per
 *    stream. */
flint_status flint_moe_decode_bf16_noalloc(const flint_moe_dims* dims, int32_t batch,
                                           const void* x_bf16, const void* residual_bf16,
                                           const void* w_router_bf16, const float* logit_bias,
                                           const void* w13_bf16, const void* w2_bf16,
                                           const void* ws13_bf16, const void* ws2_bf16,
                                           void* out_bf16,
                                           int32_t* topk_idx_out, float* topk_w_out,
                                           int32_t* device_status_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H_ */
