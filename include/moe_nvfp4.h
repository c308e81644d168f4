/*
 * moe_nvfp4.h -- C ABI of a GB300 (sm_103a) decode-step library for one
 * sigmoid-top-k Mixture-of-Experts layer whose experts are NVFP4 weights run
 * weight-only (W4A16: BF16 activations, 4-bit weights, FP32 accumulation).
 *
 * What the layer computes, per token t (sources are cited by page title and
 * section):
 *   a1  FP32 router GEMV      z[e] = sum_h x[t,h] * Wr[e,h] (+ b[e])
 *         "Inkling 2 Small on vLLM: Day-0 Support", "Accuracy evaluation"
 *         (FP32 router); "Day 0 support for Mistral Large 4 on vLLM",
 *         "Breakable CUDA graphs and fusions" (FP32 routing GEMM).
 *   a2  sigmoid top-k         s = sigmoid(z); the k largest s (lowest expert
 *                             index first on ties); w = s_sel / sum(s_sel)
 *         "vLLM Day-0 support for Recursive's Flint", "Flint model
 *         architecture" (256 experts, sigmoid top-6 + one shared expert).
 *   a3  gate/up + SwiGLU      h = bf16(silu(Wg x) * (Wu x)) for each selected
 *                             expert and each shared expert
 *   a4  down                  y = Wd h
 *         Inkling 2 Small page, "vLLM integration and optimisation" (SwiGLU
 *         between the gate/up and down projections); Flint page, "Optimisation
 *         strategy" (the expert GEMVs read only the selected experts' weights).
 *   a5  combine               out[t] = bf16(sum_j w_j y_j + sum_shared y_s)
 *         Flint page, "Optimisation strategy" (routing and the expert combine
 *         fused into the neighbouring GEMVs).
 * Expert weights are NVFP4: E2M1 codes, one E4M3 (fn) scale per 16 elements
 * along K (Inkling 2 Small page, "Mixed-precision MoE and Four-Over-Six
 * NVFP4": 16-element blocks), one FP32 tensor scale per (expert, matrix).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless the name ends in _host.
 *   - Integers are int32; BF16 tensors are arrays of uint16 bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - All work is enqueued asynchronously on `stream`; nothing here blocks the
 *     host unless documented (moe_init, moe_check, moe_debug_dequant).
 *   - Argument errors are detected on the host before anything is enqueued and
 *     return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED; moe_last_error() then
 *     names every reason.  The library never aborts, traps or prints.
 *   - A handle may be used from one host thread at a time; different handles
 *     are independent.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer;   /* opaque handle */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, T out of range ... */
    MOE_ERR_UNSUPPORTED = -2,   /* configuration outside what the kernels cover */
    MOE_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
    MOE_ERR_OOM = -4,           /* device allocation failed in moe_init */
    MOE_ERR_TIMEOUT = -5,       /* a bounded in-kernel wait gave up */
    MOE_ERR_DEVICE = -6         /* the sticky device error word was set */
} moe_status;

/* Expert weight formats (moe_config.expert_format / shared_format).  The
 * codes and scales of a [rows, cols] matrix (cols = K, the input size):
 *   MOE_FMT_NVFP4      codes uint8 [rows, cols/2] E2M1, element 2j in the low
 *                      nibble of byte j; scales uint8 [rows, cols/16] E4M3
 *                      (fn), one per 16 elements; one FP32 tensor scale per
 *                      matrix (gate and up separately).  W = e2m1*e4m3*gs.
 *   MOE_FMT_MXFP4      codes as NVFP4; scales uint8 [rows, cols/32] E8M0, one
 *                      per 32 elements; no tensor scale.  W = e2m1*2^(s-127).
 *                      "Day 0 support for Mistral Large 4 on vLLM", "MXFP4
 *                      experts at load, one layer at a time".  Repacked
 *                      exactly into the NVFP4 layout: the E8M0 codes of one
 *                      matrix (of the gate or the up half) must span at most
 *                      17 octaves, else moe_init returns MOE_ERR_UNSUPPORTED.
 *   MOE_FMT_FP8_BLOCK  codes uint8 [rows, cols] E4M3 (fn); scales FP32
 *                      [ceil(rows/128), ceil(cols/128)], one per 128 x 128
 *                      block of the stored matrix, passed through the uint8
 *                      scale pointer (16-byte aligned).  W = e4m3*scale.  The
 *                      Mistral Large 4 page, "Highlights": its NVFP4
 *                      checkpoint keeps the shared experts in block-scaled FP8
 *                      (the page gives no block size; 128 x 128 is read).
 *   MOE_FMT_MXFP8      codes as FP8_BLOCK; scales uint8 [rows, cols/32] E8M0.
 *                      W = e4m3*2^(s-127).  "Inkling 2 Small on vLLM: Day-0
 *                      Support", "Mixed-precision MoE and Four-Over-Six NVFP4"
 *                      (its last eight layers' experts).
 * The tensor-scale pointers (w13_gs, w2_gs, ...) are read for NVFP4 only and
 * may be NULL otherwise.  Experts in an FP8 format run on the GEMV kernels
 * and the single launch, never on the grouped tensor-core kernels. */
#define MOE_FMT_NVFP4 0
#define MOE_FMT_MXFP4 1
#define MOE_FMT_FP8_BLOCK 2
#define MOE_FMT_MXFP8 3

/* Layer configuration (host struct).
 * Supported (anything else -> MOE_ERR_UNSUPPORTED with every reason listed;
 * default-deny, as the Mistral Large 4 page's "Fail-stop" section describes
 * for its specialised decode kernel):
 *   hidden % 64 == 0, 64 <= hidden <= 16384
 *   inter % 64 == 0 and shared_inter % 64 == 0 (when num_shared > 0), <= 16384
 *   1 <= top_k <= 8, top_k <= num_experts <= 512
 *   0 <= num_shared <= 2
 *   1 <= max_tokens <= 64
 *   normalize_topk in {0, 1}, score_func in {0, 1}, routed_scale finite
 *   expert_format, shared_format in MOE_FMT_*, w4a4 in {0, 1}                */
typedef struct {
    int hidden;             /* H */
    int num_experts;        /* E routed experts */
    int top_k;              /* k */
    int inter;              /* I, routed expert intermediate size */
    int num_shared;         /* S shared (always-on, weight 1) experts */
    int shared_inter;       /* I of the shared experts */
    int max_tokens;         /* largest T a call may pass; sizes the workspace */
    int normalize_topk;     /* 1: routing weights normalised to sum to 1 */
    float routed_scale;     /* multiplies every routed weight (1.0) */
    int grouped_min_tokens; /* experts with at least this many tokens use the
                               grouped tensor-core path when T > 8;
                               0 = library default (8), < 0 = never.  For a
                               routed expert the library may raise the
                               threshold per step, up to 16, so that the
                               grouped kernels get at most one item per SM
                               (the GEMV kernels take the rest); results do
                               not depend on the split beyond FP32 rounding */
    int fused;              /* 0: moe_decode_forward runs the whole step as
                               one launch when the shape allows it (T <= 8,
                               H <= 8192, E <= 256 and <= 4 x SM count, the
                               activations and the weight rings fit in shared
                               memory); 1: the same, launched as a
                               cooperative grid (the driver starts it only
                               when every block can be resident, so kernels
                               on other streams cannot keep a block waiting
                               on the others); < 0: always the three-kernel
                               chain of the moe_stage_* entry points */
    int score_func;         /* routing score: 0 = sigmoid of each logit (Flint
                               page, "Flint model architecture"); 1 = softmax
                               over all experts' logits (Mistral Large 4 page,
                               "Specialized decode": its softmax top-4 router).
                               The top-k is the same for both (both scores
                               increase with the logit); the weights are the
                               chosen experts' scores, normalised to sum to 1
                               when normalize_topk = 1 (for softmax:
                               exp(z_j - z_max) / sum over the chosen of
                               exp(z_i - z_max)), times routed_scale. */
    int expert_format;      /* MOE_FMT_* of the routed experts (0 = NVFP4) */
    int shared_format;      /* MOE_FMT_* of the shared experts (0 = NVFP4) */
    int w4a4;               /* 1: W4A4 -- the tokens (before gate/up) and the
                               SwiGLU output (before down) are quantised to
                               NVFP4 with "Four Over Six" block scales
                               ("Inkling 2 Small on vLLM: Day-0 Support",
                               "Mixed-precision MoE and Four-Over-Six NVFP4"):
                               a per-row global scale a / 1792 (a the row's
                               max |v|), and per 16-element block the block
                               maximum scaled to 6 and to 4, keeping the lower
                               sum of absolute reconstruction errors (ties: 6),
                               every step in FP32.  The router reads the
                               unquantised x.  Such layers run the chain (no
                               single launch); the GEMMs see the dequantised
                               values, exact in f16, on the same kernels. */
} moe_config;

/* Weights in the canonical layout (device pointers, only read during
 * moe_init; the caller may free them afterwards).  Shapes below are those of
 * NVFP4; the other formats' codes and scales follow MOE_FMT_* above.
 *   router_w  FP32 [E, H] row-major
 *   router_b  FP32 [E] or NULL (added to the logit)
 *   w13       uint8 [E, 2I, H/2]   E2M1 codes, row-major over K; element 2j in
 *                                  the low nibble of byte j.  Rows 0..I-1 are
 *                                  the gate projection, rows I..2I-1 the up one.
 *   w13_sf    uint8 [E, 2I, H/16]  E4M3 (fn) block scales, one per 16 elements
 *   w13_gs    FP32  [E, 2]         tensor scales (gate, up)
 *   w2        uint8 [E, H, I/2]    down projection codes
 *   w2_sf     uint8 [E, H, I/16]
 *   w2_gs     FP32  [E]
 *   sw13 ... sw2_gs: the same seven tensors for the shared experts, with E ->
 *   num_shared and I -> shared_inter (NULL when num_shared == 0).
 * Every pointer must be 16-byte aligned. */
typedef struct {
    const float *router_w;
    const float *router_b;
    const uint8_t *w13;
    const uint8_t *w13_sf;
    const float *w13_gs;
    const uint8_t *w2;
    const uint8_t *w2_sf;
    const float *w2_gs;
    const uint8_t *sw13;
    const uint8_t *sw13_sf;
    const float *sw13_gs;
    const uint8_t *sw2;
    const uint8_t *sw2_sf;
    const float *sw2_gs;
} moe_weights;

/* Sizes a handle holds (for accounting). */
typedef struct {
    size_t weight_bytes;     /* repacked expert weights + router, device */
    size_t workspace_bytes;  /* per-call scratch, device */
    size_t expert_bytes;     /* bytes one routed expert's repacked weights occupy */
    size_t shared_bytes;     /* the same for one shared expert */
    int max_slots;           /* worst-case number of distinct experts per call */
    int sm_count;            /* SMs of the device the handle lives on */
    int single_launch_max_tokens; /* largest T run as one launch (0: none) */
} moe_layer_info;

/* Create a handle on the current device: validate `cfg` (default-deny), copy
 * the router, repack every expert LOSSLESSLY into the kernels' streaming layout
 * (the load-time repack of the Flint page, "Flint model overview": the NVFP4
 * checkpoint is repacked without loss when it is loaded) and allocate the
 * workspace for `max_tokens`.  Blocks until the repack has finished on
 * `stream`.  On success *out owns all of it; release with moe_destroy. */
moe_status moe_init(const moe_config *cfg, const moe_weights *w, void *stream,
                    moe_layer **out);

/* Release a handle (synchronises its device first).  NULL is a no-op. */
void moe_destroy(moe_layer *layer);

/* One decode step, rows a1..a5 above, for T tokens (1 <= T <= max_tokens).
 * Small steps run as ONE launch of one block per SM.  It has no grid
 * barrier: blocks hand the router logits and the SwiGLU output to each other
 * as words tagged with the call number, and a reader polls the words it
 * needs.  Every block must therefore get an SM while the others poll.  A
 * kernel on another stream that holds SMs delays the blocks that wait for
 * them; a wait that exceeds about a second gives up, the call's outputs are
 * then invalid and moe_check reports MOE_ERR_TIMEOUT.  Otherwise the step
 * runs as the chain moe_stage_route, moe_stage_gate_up, moe_stage_down.
 * The call tags of one handle are 32-bit: the library restarts them (with
 * the tagged words) after 2^31 single-launch calls made through this entry
 * point; a CUDA graph that replays such a call needs moe_check (which
 * restarts them too) at least every 2^31 replays.
 *   x         BF16 [T, H], 16-byte aligned, read only
 *   out       BF16 [T, H], 16-byte aligned, written; must not alias x
 *   topk_ids  int32 [T, k] or NULL: selected experts, descending score
 *   topk_w    FP32  [T, k] or NULL: their routing weights (routed scale
 *             applied)
 * No host synchronisation; the launches form a chain of kernels that each
 * start early (programmatic dependent launch) and wait for their inputs, so
 * the call can be captured into a CUDA graph.  The handle's workspace is
 * reused by every call: calls on one handle must be ordered on one stream. */
moe_status moe_decode_forward(moe_layer *layer, const void *x, int T, void *out,
                              int *topk_ids, float *topk_w, void *stream);

/* The same step with HOST buffers (pinned memory for asynchronous copies):
 * copies x_host to the device and runs moe_decode_forward; when out_host is
 * pinned (page-locked and mapped, as cudaHostAlloc gives) and 16-byte
 * aligned the kernels store the output straight into it through its device
 * alias, otherwise it is copied back; the routing result (optional) is copied
 * back.  When the step takes the single launch with one or two tokens and
 * x_host is pinned, mapped, 16-byte aligned and apart from out_host, the
 * kernel reads x_host in place through its device alias instead of a copy
 * (no copy then stands between two layers' kernels); x_host must then stay
 * unchanged until the stream reaches the call.  Returns after enqueueing;
 * the host buffers may be read after the stream has been synchronised. */
moe_status moe_decode_forward_host(moe_layer *layer, const void *x_host, int T,
                                   void *out_host, int *topk_ids_host,
                                   float *topk_w_host, void *stream);

/* The step split into its kernels, for measurement.  moe_decode_forward is
 * exactly moe_stage_route; moe_stage_gate_up; moe_stage_down on one stream
 * with the same T.  Each of the last two consumes the state that the calls
 * before it in this order left in the handle's workspace (the routing, its
 * work counters, h): call the three in order, once each per step.  With
 * moe_config.w4a4 set, moe_stage_gate_up must follow moe_stage_route on the
 * stream with no other work between them and with the same, unchanged x:
 * its token quantiser reads x while the router still runs.
 *   moe_stage_route     a1+a2: logits, sigmoid, top-k, weights (also written
 *                       to topk_ids / topk_w when not NULL), and the list of
 *                       distinct selected experts with their tokens
 *   moe_stage_gate_up   a3: gate/up GEMV + SwiGLU over the selected and the
 *                       shared experts (BF16 intermediate in the workspace)
 *   moe_stage_down      a4+a5: down GEMV, then the routing-weighted combine
 *                       with the shared experts into BF16 `out` */
moe_status moe_stage_route(moe_layer *layer, const void *x, int T, int *topk_ids,
                           float *topk_w, void *stream);
moe_status moe_stage_gate_up(moe_layer *layer, const void *x, int T, void *stream);
moe_status moe_stage_down(moe_layer *layer, int T, void *out, void *stream);

/* Synchronise `stream`, then read and clear the handle's sticky device error
 * word: MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (reason in
 * moe_last_error()).  It also restarts the single launch's call tags (see
 * moe_decode_forward), so no work of this handle may be in flight on another
 * stream. */
moe_status moe_check(moe_layer *layer, void *stream);

/* Decode one repacked matrix back to the canonical row-major FP32 layout with
 * the kernels' own decoder: value = fl32(e2m1 * e4m3 * gs), which must equal
 * the canonical weights' exact dequantisation rounded once to FP32.
 *   which   0 routed w13 [2I, H], 1 routed w2 [H, I],
 *           2 shared w13 [2Is, H], 3 shared w2 [H, Is]
 *   expert  routed expert id (which 0, 1) or shared index (which 2, 3)
 *   dst     FP32 device buffer of rows*cols elements
 * Synchronises `stream`. */
moe_status moe_debug_dequant(moe_layer *layer, int which, int expert, float *dst,
                             void *stream);

/* Test hook for the fail-stop path (the pages' "Fail-stop" requirement of the
 * persistent decode kernel: in-kernel waits give up after a bound and report
 * instead of hanging).  what = MOE_INJECT_WAIT_STALL: the NEXT
 * moe_decode_forward call on this handle that runs as one launch makes its
 * first grid-wide wait (every block polls the other blocks' router logits,
 * which carry the call's tag) expect a tag `value` (>= 1) calls ahead --
 * words nothing writes.  That wait gives up after about one second, sets the
 * sticky error word and lets the call finish (its outputs are then invalid);
 * moe_check reports MOE_ERR_TIMEOUT and restores the handle, and the call
 * after that is correct again.  Nothing faults or traps.  The hook is
 * consumed by that one call; value 0 clears it.
 * Errors: MOE_ERR_INVALID_ARG for a NULL handle, an unknown `what` or a
 * negative value. */
#define MOE_INJECT_WAIT_STALL 1
moe_status moe_debug_inject(moe_layer *layer, int what, int value);

/* Diagnostics: install a device buffer of 5 * blocks_per_kernel * 16 uint64
 * that the traced build of the library (compiled with MOE_TRACE) fills with
 * %globaltimer stamps at numbered phase points of its kernels (kernel 0
 * router or the single launch, 1 gate/up GEMV (the single launch: SM cycle
 * counts), 2 down GEMV, 3 grouped gate/up, 4 grouped down; index
 * [kernel][block][point]).  NULL detaches.  The regular build returns
 * MOE_ERR_UNSUPPORTED. */
moe_status moe_trace_attach(moe_layer *layer, unsigned long long *buf, int blocks_per_kernel);

/* Fill *info (host struct). */
moe_status moe_get_info(const moe_layer *layer, moe_layer_info *info);

/* Routing only (rows a1 + a2) WITHOUT any device allocation, for callers that
 * cannot call cudaMalloc where they route: an engine whose free device memory
 * is already handed to its KV cache, code under an allocator that forbids raw
 * cudaMalloc/cudaFree after start-up, or code that must avoid the implicit
 * synchronisation an allocation may cause.  The pages have no counterpart to
 * this entry point; it exists for such embedders.
 *   router_w  FP32 [E, H] device, 16-byte aligned;  router_b FP32 [E] or NULL
 *   x         BF16 [T, H] device, 16-byte aligned
 *   topk_ids  int32 [T, k] device (written): selected experts, descending score
 *   topk_w    FP32  [T, k] device (written): weights (normalised when
 *             normalize_topk = 1, then times routed_scale)
 * The score is always the sigmoid of the logit (there is no softmax option
 * here); the choice and its order follow moe_stage_route's rule (FP32 logits,
 * lowest index on ties).  Its logits are summed in another order than the
 * handle path's, so the weights agree with that path to FP32 rounding (about
 * 1e-6 relative), not bit for bit.  No handle is needed.
 * Limits: 1 <= T <= 64, 1 <= E <= 512, 1 <= k <= min(8, E), hidden a multiple
 * of 64 in [64, 16384]; anything else returns MOE_ERR_UNSUPPORTED naming the
 * limit.  Scratch: a 128 KiB + 256 B static device array inside the library
 * (every GPU that loads the library holds it until exit), shared by all calls
 * on a device; calls whose kernels may overlap on the GPU (different streams or
 * host threads on one device) race on it, so order them on one stream.  The
 * first call on each device looks up that array's device address; make it
 * before any stream capture.  Asynchronous on `stream`. */
moe_status moe_route_topk_static(const float *router_w, const float *router_b,
                                 int num_experts, int hidden, int top_k,
                                 int normalize_topk, float routed_scale,
                                 const void *x, int T, int *topk_ids,
                                 float *topk_w, void *stream);

/* The W4A4 activation quantiser on its own (moe_config.w4a4 applies it to
 * the tokens and to the SwiGLU output): "Four Over Six" NVFP4 quantisation of
 * `rows` rows of n BF16 values ("Inkling 2 Small on vLLM: Day-0 Support",
 * "Mixed-precision MoE and Four-Over-Six NVFP4"), as described at
 * moe_config.w4a4.
 *   x    BF16 [rows, n] device, 8-byte aligned, read
 *   deq  BF16 [rows, n] device, 8-byte aligned, written (may equal x): the dequantised values
 *        without the global scale, e2m1 * e4m3 (exact in BF16)
 *   gs   FP32 [rows] device, written: the rows' global scales (value =
 *        deq * gs)
 * n must be a positive multiple of 16, rows >= 0; a NULL or misaligned
 * pointer returns MOE_ERR_INVALID_ARG.  A row is split over a cluster of up
 * to 8 CTAs.  Asynchronous on `stream`; no handle is needed. */
moe_status moe_quant_fos(const void *x, int rows, int n, void *deq, float *gs, void *stream);

/* Reasons for the last failure on this host thread ("" if none). */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
