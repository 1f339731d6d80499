/*
 * ft_moe.h -- C ABI of the GB300 MoE expert-cache layer step.
 *
 * The operation is one MoE layer of FreeToken-style edge-native serving
 * ("FreeToken: Efficient Edge-Native MoE Serving with Bandwidth-Adaptive
 * Execution", summarised on theainews.cc, 2026-08-22-freetoken-edge-moe):
 * the full expert pool lives in pinned host memory and is the source of
 * truth; one device-resident cache of expert slots is shared by every MoE
 * layer (section "设计：三大机制", intro).  Per layer step:
 *
 *   routes     top-k of E routed experts per token (section "为什么个人跑 MoE
 *              这么难"; routing stays exact, section "与相关工作").
 *   control    dedup, classify hits/misses against a device residency table,
 *              split the m misses by q* ~ m*BP/BH between GPU fill and an
 *              external (CPU) partial sum, pick K least-recently-used victim
 *              slots in one scan, rewrite logical expert ids to slot ids --
 *              one kernel with fixed-shape buffers and device-resident counts
 *              so the step can be captured in a CUDA graph (section "实现要点",
 *              first bullet; "设计 1" Decode bullet).
 *   fill       copy the q fetched experts from the host pool into their slots
 *              on a side stream (Decode bullet).
 *   prefill    full-layer double buffer: while layer l computes, a transfer
 *              stream uploads all experts of layer l+1 (Prefill bullet).
 *   experts    routed SwiGLU FFNs, weighted and summed per token, plus an exact
 *              merge of a caller-supplied partial sum (Decode bullet: CPU and
 *              GPU partial sums merge exactly).
 *
 * Conventions
 *  - Every call returns FT_OK (0) or a negative FT_E_* code; ft_last_error()
 *    returns the calling thread's last message.  Argument errors are found on
 *    the host before anything is launched.  Faults found on the device (a
 *    route id outside [0, E), a NaN logit, the step clock about to wrap) set
 *    bits in a device status word read by ft_get_status(); the step still
 *    completes with the offending route treated as absent.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *    Calls enqueue work and never synchronise unless stated.
 *  - Device pointers (suffix _dev) are owned by the caller unless stated.
 *    Pointers returned in ft_step_out are owned by the context.
 *  - bf16 values are passed as their 16-bit patterns (uint16_t).
 *
 * Canonical host pool layout (the layout the experts are served from, written
 * once by the loader before the memory is pinned; section "设计 3", fast
 * start):
 *  expert (l, e) starts at byte (l*E + e) * B_x;
 *  bf16   expert: [W_gate f x d | W_up f x d | W_down d x f], row-major,
 *         B_x = 6*d*f;
 *  mxfp4  expert: [codes gate f*d/2 | codes up | codes down d*f/2 |
 *         scales gate f*d/32 | scales up | scales down d*f/32];
 *         two e2m1 codes per byte, element 2i in the low nibble; one e8m0
 *         scale byte per 32 consecutive elements of a row (OCP MX v1.0).
 *         B_x = 3*d*f/2 + 3*d*f/32.
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define FT_OK 0
#define FT_E_ARG -1         /* bad argument (checked on the host) */
#define FT_E_PIN -2         /* the host pool could not be pinned/mapped */
#define FT_E_NOMEM -3       /* device allocation failed */
#define FT_E_CUDA -4        /* a CUDA runtime call failed */
#define FT_E_STATE -5       /* call not allowed now (e.g. during stream capture) */
#define FT_E_UNSUPPORTED -6 /* shape or mode not built into this library */

/* device status bits (ft_get_status) */
#define FT_ST_ROUTE_RANGE 1u /* a route id was outside [0, E) */
#define FT_ST_NAN 2u         /* a router logit was NaN */
#define FT_ST_CLOCK_WRAP 4u  /* the LRU step clock reached 2^32 - 1 */
#define FT_ST_BAD_SLOT 8u    /* a slot id outside [0, S) reached a kernel */
#define FT_ST_TIMEOUT 16u    /* a bounded wait for an asynchronous copy ran out; the kernel exited early */

#define FT_DTYPE_BF16 0
#define FT_DTYPE_MXFP4 1

#define FT_DECODE_CACHED 0 /* experts from the shared cache, after ft_cache_step */
#define FT_PREFILL_LAYER 1 /* experts from the full-layer buffers */

/* When only q < m misses can be filled (q* < m, K_max or free slots), which
 * ones: the first q in ascending expert id (the plain reading of the article,
 * section "设计：三大机制" 1, Decode bullet), or the q with the most routes in
 * the step, ties to the lower id (a variant: the experts that serve the most
 * routes run on the GPU).  Either way the fetch and CPU lists are in ascending
 * id and fetch i goes to victim i. */
#define FT_FILL_ORDER_ID 0
#define FT_FILL_ORDER_MOST_ROUTED 1

#define FT_FILL_KERNEL 0      /* SM copy from the mapped pool; graph capturable */
#define FT_FILL_COPY_ENGINE 1 /* cudaMemcpyAsync per expert; reads the fetch list back (host sync) */

/* How a decode step's fill and experts are launched (FT_FILL_KERNEL, bf16
 * experts or MXFP4 experts with hidden a multiple of 512; other
 * configurations always take the split path):
 *  FUSED  one cooperative kernel per layer, one CTA per SM: fill_ctas CTAs copy
 *         the fetched experts from the host pool, the others run the experts
 *         resident before the step and then each installed expert as soon as
 *         its bytes are in its slot;
 *  SPLIT  a fill kernel on the context's transfer stream beside an expert
 *         launch for the resident experts, then a second expert launch for the
 *         installed ones after the fill. */
#define FT_DECODE_FUSED 0
#define FT_DECODE_SPLIT 1

typedef struct ft_config {
  int32_t num_layers;    /* L: MoE layers sharing the cache */
  int32_t num_experts;   /* E: routed experts per layer (<= 1024) */
  int32_t top_k;         /* k: experts per token (<= 32, <= E) */
  int32_t hidden;        /* d (multiple of 256) */
  int32_t inter;         /* f: expert intermediate size (multiple of 128) */
  int32_t dtype;         /* FT_DTYPE_BF16 or FT_DTYPE_MXFP4 */
  int32_t num_slots;     /* S: cache slots (<= 32768) */
  int32_t k_max;         /* K_max: fixed victim-buffer size (1..1024) */
  int32_t t_max;         /* tokens per decode/control step (1..1024) */
  int32_t r_num, r_den;  /* r = BP/BH as a rational, r_num >= 0, r_den >= 1 */
  int32_t prefill_buffers; /* 0: no prefill; 1: one layer buffer (no overlap); 2: double buffer
                              (MXFP4 experts: hidden and inter multiples of 512, else FT_E_UNSUPPORTED) */
  int32_t prefill_t_max; /* tokens per prefill chunk (0 if no prefill) */
  int32_t fill_mode;     /* FT_FILL_KERNEL or FT_FILL_COPY_ENGINE */
  int32_t fill_order;    /* FT_FILL_ORDER_ID or FT_FILL_ORDER_MOST_ROUTED: which q of the m misses are filled */
  int32_t decode_path;   /* FT_DECODE_FUSED (default) or FT_DECODE_SPLIT */
  int32_t fill_ctas;     /* CTAs that fill, on either decode path (0 = the library's choice: fused path
                            3/8 of the SMs for bf16 experts, 1/4 for MXFP4) */
  int32_t reserved[1];   /* must be zero */
} ft_config;

/* Per-layer results of ft_cache_step / ft_cache_control.  All pointers are
 * device memory owned by the context and stay valid (and unchanged) until the
 * next step of the same layer or ft_cache_rebuild.  Sizes are fixed
 * capacities; the valid lengths are in counts. */
typedef struct ft_step_out {
  int32_t* ids;       /* [T, k] local expert ids, logit-descending per token */
  float* weights;     /* [T, k] routing weights (softmax renormalised over the k) */
  int32_t* slot_ids;  /* [T, k] cache slot of each route, -1 = CPU route */
  int32_t* uniq;      /* [E] unique global expert ids (layer*E + e), ascending */
  int32_t* hit_list;  /* [E] unique ids that hit, ascending */
  int32_t* fetch;     /* [K_max] filled global expert ids, ascending */
  int32_t* victims;   /* [K_max] slot receiving fetch[i] */
  int32_t* evicted;   /* [K_max] expert that victims[i] held before, -1 if empty */
  int32_t* cpu_list;  /* [E] misses left to the CPU, ascending */
  int32_t* counts;    /* [8] n, hits, m, q, cpu, n_groups, now, 0 */
} ft_step_out;

typedef struct ft_ctx ft_ctx;

/* Create a context on the current device.  host_pool holds num_layers *
 * num_experts experts in the canonical layout, already written by the caller
 * (pool_bytes >= L*E*B_x); the library registers it as mapped pinned memory
 * (pin after write) and unregisters it in ft_moe_destroy -- the caller keeps
 * ownership and must keep it alive.  If the range is already pinned it is
 * used as is.  Allocates the slot arena (S*B_x bytes), the residency table,
 * fixed-shape work buffers and, if prefill_buffers > 0, the layer buffers.
 * The cache starts cold: every slot empty, clock 0.
 * Errors: FT_E_ARG, FT_E_PIN (no fallback), FT_E_NOMEM, FT_E_CUDA. */
int ft_moe_init(const ft_config* cfg, void* host_pool, size_t pool_bytes, ft_ctx** out);

/* Free everything the context allocated and unregister the pool.  Waits for
 * the context's streams.  NULL is accepted. */
int ft_moe_destroy(ft_ctx* ctx);

/* Pinned, device-mapped host memory for a pool (cudaHostAlloc, mapped and
 * portable), for callers that write the pool into memory that is already
 * pinned instead of pinning it after the write.  The pages are mapped in the
 * GPU's own page tables when the call returns, so the host link streams them
 * at full rate from the first read; registered pageable memory can read
 * slowly the first time each page is touched.  The cost moves to start-up:
 * the whole range is faulted in here.  *out receives the host address (the
 * device view is the one ft_moe_init takes by itself).  The caller owns the
 * memory and frees it with ft_host_free after destroying every context that
 * uses it.  Errors: FT_E_ARG (bytes == 0 or out == NULL), FT_E_PIN. */
int ft_host_alloc(size_t bytes, void** out);

/* Free memory from ft_host_alloc.  NULL is accepted.  Errors: FT_E_CUDA. */
int ft_host_free(void* p);

/* Routing + cache control for one decode step of `layer`: logits_dev is
 * [T, E] float32 row-major, 1 <= T <= t_max.  Enqueues one kernel on `stream`
 * that routes the T tokens and then runs the control step; no host
 * synchronisation, so the call can be
 * captured in a CUDA graph (shapes are fixed by T).  The step clock advances
 * by one per call.  `out` (may be NULL) receives the context's buffers. */
int ft_cache_step(ft_ctx* ctx, int layer, const float* logits_dev, int T, ft_step_out* out, void* stream);

/* The control kernel alone, on routes the caller supplies: ids_dev is [T, k]
 * local expert ids (each token's ids distinct), read in place -- keep it
 * unchanged until the step's kernels have run (out->ids points to it).
 * Weights are left untouched. */
int ft_cache_control(ft_ctx* ctx, int layer, const int32_t* ids_dev, int T, ft_step_out* out, void* stream);

/* Expert FFNs of one layer.
 *  mode FT_DECODE_CACHED: uses the last ft_cache_step of `layer` (same T);
 *    fills the q fetched experts into their slots on the context's transfer
 *    stream; meanwhile runs on `stream` the routed SwiGLU experts that were
 *    resident before the step, then (after joining the fill into `stream`)
 *    the experts the step installed, and merges:
 *      out[t] = partial[t] + sum_j w[t,j] * y_{ids[t,j]}(hidden[t])   (slot >= 0)
 *    logits_dev is ignored.
 *  mode FT_PREFILL_LAYER: routes logits_dev itself (no cache access; the
 *    residency table is untouched), waits for layer `layer` in its layer
 *    buffer (uploading it first if it is not there), runs all routes, and --
 *    with prefill_buffers == 2 -- starts the upload of layer+1 into the other
 *    buffer before returning.  T <= prefill_t_max.  MXFP4 experts are
 *    dequantised exactly to bf16 on the way into the tensor cores; the
 *    activations stay bf16.
 *  hidden_dev [T, d] bf16; partial_dev [T, d] float32 or NULL (= 0);
 *  out_dev [T, d] float32, written (not accumulated).
 * Never synchronises (except FT_FILL_COPY_ENGINE, which reads the fetch list
 * back and so cannot be captured). */
int ft_moe_forward(ft_ctx* ctx, int layer, int mode, const float* logits_dev, const uint16_t* hidden_dev,
                   int T, const float* partial_dev, float* out_dev, void* stream);

/* Rebuild the cache with new_slots slots under a revised memory budget
 * ("设计 3" runtime cache rebuild): only at a safe point -- the caller's
 * streams idle, no capture in progress (FT_E_STATE otherwise).  Frees and
 * reallocates the slot arena and resets the residency table to cold; the
 * host pool stays pinned.  CUDA graphs captured earlier must be recaptured:
 * the epoch (ft_get_epoch) increases by one.  Synchronises the device. */
int ft_cache_rebuild(ft_ctx* ctx, int new_slots);

/* Read (and clear, if clear != 0) the device status word; synchronises the
 * context's streams. */
int ft_get_status(ft_ctx* ctx, uint32_t* status, int clear);

/* Per-layer counters since init/rebuild, summed over steps, copied to the
 * host array counters[L][6] = {hits, misses, fills, cpu routes, evictions,
 * steps}.  Synchronises. */
int ft_get_counters(ft_ctx* ctx, uint64_t* counters);

/* Copy the residency table to host arrays (any may be NULL): slot_of[L*E],
 * expert_of[S], last_use[S], now[1].  Synchronises.  For tests and tools. */
int ft_get_table(ft_ctx* ctx, int32_t* slot_of, int32_t* expert_of, uint32_t* last_use, uint32_t* now);

/* Device pointer of slot s's bytes in the arena (for tests), or NULL. */
void* ft_slot_ptr(ft_ctx* ctx, int slot);

/* As ft_cache_rebuild, but the most recently used residents stay: residents
 * ordered by last use (most recent first, ties to the lower slot) fill the new
 * slots 0, 1, ... with their last use; the clock and counters are unchanged
 * (FreeToken article, section "设计：三大机制" 3, runtime cache rebuild: GPU
 * memory changes only performance, so which residents survive is a choice;
 * this one keeps the recency the LRU would act on).  The old and the new
 * arenas exist together during the call; if the new one does not fit,
 * FT_E_NOMEM is returned and the cache is left as it was.  Epoch +1 on
 * success; graphs captured before must be re-captured.  Synchronises.
 * Errors: FT_E_ARG, FT_E_STATE (during a capture), FT_E_NOMEM, FT_E_CUDA. */
int ft_cache_rebuild_retain(ft_ctx* ctx, int new_slots);

/* Change r = BP/BH (FreeToken article, section "设计：三大机制" 1, Decode
 * bullet: the fill-vs-CPU split of the misses follows the measured link and
 * host bandwidths, which vary at run time) for the steps enqueued on `stream`
 * after this call.  r lives in device memory and the control kernel reads it
 * at every step, so CUDA graphs captured earlier pick up the new value
 * without re-capture; the call itself enqueues one tiny kernel and can be
 * captured too (the captured values are then fixed).  The caller measures
 * the two bandwidths (its CPU expert executor's, and the fill rate reported
 * by ft_profile_read or its own timing) and chooses r.
 * Errors: FT_E_ARG (r_num < 0 or r_den < 1), FT_E_CUDA. */
int ft_set_ratio(ft_ctx* ctx, int32_t r_num, int32_t r_den, void* stream);

/* ---- Run-time adaptation of r = BP/BH ----
 * FreeToken article, section "设计：三大机制" 1, Decode bullet: the split of
 * the misses between GPU fills and CPU execution follows the two bandwidths
 * as measured while the system runs.  The context measures both itself:
 *   BP  the decode fill kernel's link rate: bytes it copied from the host
 *       pool over the summed spans of its launches (first CTA start to last
 *       CTA end, device clock), launches that copied nothing excluded;
 *   BH  the host expert rate: expert bytes the CPU executor read (B_x per
 *       CPU route) over the time its host functions spent computing, plus
 *       whatever the caller reports with ft_report_host_rate.
 * The adapter below turns successive measurements into r; it is plain host
 * state owned by the caller. */
typedef struct ft_ratio_adapter {
  double alpha;      /* weight of a new sample in the running estimates, in (0, 1] */
  int32_t r_den;     /* r = r_num / r_den: the grid r is quantised to (>= 1) */
  int32_t r_num_max; /* upper bound of r_num (>= 0) */
  double bp_gbs;     /* running estimate of BP in GB/s, 0 = no sample yet */
  double bh_gbs;     /* running estimate of BH in GB/s, 0 = no sample yet */
  int32_t r_num;     /* r in effect is r_num / r_den; -1 until both estimates exist */
  int32_t updates;   /* how many times r_num has been computed */
} ft_ratio_adapter;

/* Initialise an adapter: no estimates, r_num = -1.  Pure host code.
 * Errors: FT_E_ARG (alpha outside (0, 1], r_den < 1 or r_num_max < 0). */
int ft_ratio_adapter_init(ft_ratio_adapter* a, double alpha, int32_t r_den, int32_t r_num_max);

/* Feed one measurement window.  A sample <= 0 means the window had none and
 * leaves that estimate as it is; otherwise the estimate becomes the sample
 * (the first one) or alpha*sample + (1 - alpha)*estimate.  Once both
 * estimates exist, r_num = min(r_num_max, floor(r_den * bp/bh + 1/2)).
 * Pure host code (no context, no GPU).  Returns 1 if r_num changed, 0 if not,
 * FT_E_ARG for an adapter that was not initialised. */
int ft_ratio_adapter_update(ft_ratio_adapter* a, double bp_sample_gbs, double bh_sample_gbs);

/* Report host expert work done outside the context's CPU executor (a
 * caller's own CPU engine): `bytes` of expert weights read in `seconds`.
 * It counts toward BH until the next reset.  Errors: FT_E_ARG. */
int ft_report_host_rate(ft_ctx* ctx, double bytes, double seconds);

/* BP and BH (GB/s) measured since the last reset; 0 where the window had no
 * sample (no fill copied anything, e.g. all hits or FT_FILL_COPY_ENGINE, which
 * is not measured; no CPU route and nothing reported).  reset != 0 starts a
 * new window.  Synchronises the device (reads device counters). */
int ft_measured_bandwidths(ft_ctx* ctx, double* bp_gbs, double* bh_gbs, int reset);

/* Device-side meters of the decode step since the last reset, as
 * out[6] = {fill bytes, fill seconds, fill launches, resident-expert bytes,
 * resident-expert seconds, fused launches with resident experts}.  The fill
 * figures are those of BP above (first fill CTA start to last fill CTA end per
 * launch that copied something).  The resident-expert figures come from the
 * fused path only: per launch, the bytes of the experts resident before the
 * step and the span from the first compute CTA start to the end of the last
 * resident work item -- the experts' HBM-bound phase, which shares no SM with
 * the fill.  reset != 0 clears them.  Synchronises.  Errors: FT_E_ARG,
 * FT_E_CUDA. */
int ft_decode_meters(ft_ctx* ctx, double* out, int reset);

/* The decode path the context runs: FT_DECODE_FUSED, or FT_DECODE_SPLIT when
 * that was asked for or the configuration has no fused kernel (MXFP4 experts,
 * FT_FILL_COPY_ENGINE, a hidden size whose ring does not fit one CTA per SM). */
int ft_decode_path(ft_ctx* ctx);

/* One adaptation step, for use between decode steps: ft_measured_bandwidths
 * with reset, ft_ratio_adapter_update, and -- if r_num changed --
 * ft_set_ratio(ctx, a->r_num, a->r_den, stream), which graphs captured
 * earlier see.  *changed (may be NULL) receives 1 or 0.  Synchronises; not
 * allowed while `stream` is capturing (FT_E_STATE).  Errors: FT_E_ARG,
 * FT_E_STATE, FT_E_CUDA. */
int ft_adapt_ratio(ft_ctx* ctx, ft_ratio_adapter* a, void* stream, int* changed);

/* Cache epoch: starts at 0, +1 per ft_cache_rebuild. */
int ft_get_epoch(ft_ctx* ctx);

/* Current slot count S. */
int ft_num_slots(ft_ctx* ctx);

/* Standalone routing kernel (no context): logits_dev [T, E] float32 ->
 * ids_dev [T, k] int32 and w_dev [T, k] float32; status_dev (may be NULL) is
 * a device uint32 that receives FT_ST_NAN bits.  E <= 1024, k <= 32. */
int ft_route(const float* logits_dev, int T, int E, int k, int32_t* ids_dev, float* w_dev, uint32_t* status_dev,
             void* stream);

/* Kernel classes of ft_profile_read. */
#define FT_K_ROUTE 0   /* routing kernel (ft_route, prefill); decode routing runs inside the control kernel */
#define FT_K_CONTROL 1 /* cache-control kernel */
#define FT_K_FILL 2    /* decode fill (kernel or copy-engine copies), transfer stream */
#define FT_K_EXPERTS 3 /* decode expert kernel */
#define FT_K_MERGE 4   /* merge kernel */
#define FT_K_UPLOAD 5  /* prefill full-layer upload, transfer stream */
#define FT_K_PREFILL 6 /* prefill routing, dispatch, gather and combine */
#define FT_K_GEMM 7    /* prefill grouped GEMMs (gate/up + down) */
#define FT_K_CPU 8     /* CPU expert executor: route copies, host function, partial copy (its own stream) */
#define FT_K_COUNT 9

/* Per-kernel timing for measurement.  While on, every kernel or copy the
 * context enqueues outside a stream capture is bracketed by CUDA events
 * recorded on the stream it is launched on (nothing is recorded during a
 * capture).  Costs two event records per launch. */
int ft_profile_enable(ft_ctx* ctx, int on);

/* Synchronise, then return per class (arrays of FT_K_COUNT) the summed
 * elapsed milliseconds and the number of launches recorded since the last
 * reset; reset != 0 clears the records. */
int ft_profile_read(ft_ctx* ctx, double* total_ms, uint64_t* launches, int reset);

/* Decode experts + merge without any allocation, for callers that cannot
 * allocate device memory when they run the step (a runtime that fixes its
 * memory budget at start-up and forbids allocation afterwards, a framework
 * that owns every device buffer through its own pool, or code inside a
 * stream capture in global mode, where cudaMalloc is not permitted).  The
 * paper has no counterpart: this is an interface for such callers.
 *
 * Computes, for T tokens and bf16 experts in the canonical layout held in
 * `arena_dev` (num_slots slots of 6*hidden*inter bytes, 16-byte aligned):
 *   out[t] = partial[t] + sum_j [slot_ids[t,j] >= 0] weights[t,j] *
 *            SwiGLU expert in slot slot_ids[t,j] applied to hidden[t]
 * -- the same arithmetic as ft_moe_forward(FT_DECODE_CACHED) after the fills,
 * with every route its own group.  slot_ids_dev [T, top_k] int32,
 * weights_dev [T, top_k] float32, hidden_dev [T, hidden] bf16, partial_dev
 * [T, hidden] float32 or NULL, out_dev [T, hidden] float32 (written);
 * status_dev: a device uint32 that receives FT_ST_* bits, or NULL.
 * Scratch lives in a fixed 8 MiB device array inside the library (held by
 * every GPU that loads it until exit); T*top_k*(inter/32)*hidden*4 bytes of
 * partial sums plus small route lists must fit, else FT_E_ARG.  The first call
 * on a device looks the array up (cudaGetSymbolAddress) and should come before
 * any stream capture.  All calls share the array, which keeps the last call's
 * contents; calls that overlap on the GPU race on it.  Enqueues on `stream`,
 * never synchronises, calls no allocating routine. */
int ft_decode_experts_noalloc(const void* arena_dev, int num_slots, int hidden, int inter, int top_k, int T,
                              const int32_t* slot_ids_dev, const float* weights_dev, const uint16_t* hidden_dev,
                              const float* partial_dev, float* out_dev, uint32_t* status_dev, void* stream);

/* CPU expert executor: the host side of the decode split (FreeToken article,
 * section "设计 1", Decode bullet: the m - q* misses that are not filled run
 * on the CPU from the host pool, and their partial sum is merged exactly with
 * the GPU's).  threads >= 1 enables it with that many host threads (the
 * calling CUDA callback thread counts as one); threads == 0 disables it (the
 * default).  While enabled, ft_moe_forward(FT_DECODE_CACHED) computes
 *   partial[t] = sum over the routes of token t with slot id < 0 of
 *                w[t,j] * SwiGLU expert ids[t,j] (host pool bytes) of hidden[t]
 * in fp32 on the host and merges it in place of partial_dev, which must then
 * be NULL (FT_E_ARG otherwise).  Stream order: after the step's control kernel
 * the route ids, weights, slot ids and hidden rows are copied to pinned host
 * memory and a host function (cudaLaunchHostFunc, capturable in a CUDA graph)
 * computes the sum into mapped pinned memory, which the merge reads; this
 * runs on a stream of the context beside the fill and the GPU experts.  One
 * set of staging buffers serves all layers, so the decode calls of a context
 * go to one stream (as for the rest of the step).  For ft_cache_control steps
 * the weights are those the caller wrote to out->weights.  Not during a
 * stream capture; synchronises the device.  Errors: FT_E_ARG, FT_E_STATE,
 * FT_E_NOMEM. */
int ft_cpu_executor(ft_ctx* ctx, int threads);

/* The executor's arithmetic on host arrays, without a context or a GPU:
 * pool_host holds the experts in the canonical layout (expert (layer, e) at
 * (layer*num_experts + e) * B_x); ids, weights, slot_ids are [T, top_k];
 * hidden_rows [T, hidden] bf16; partial [T, hidden] float32 is written with
 * the sum over the routes with slot_ids < 0 (ids outside [0, num_experts)
 * are skipped).  hidden and inter: positive multiples of 32.  Runs on the
 * calling thread plus threads - 1 helpers; returns when done.  The result does
 * not depend on threads.  Errors: FT_E_ARG. */
int ft_cpu_experts(const void* pool_host, int num_experts, int top_k, int hidden, int inter, int dtype, int layer,
                   int T, const int32_t* ids, const float* weights, const int32_t* slot_ids,
                   const uint16_t* hidden_rows, float* partial, int threads);

/* Message of the calling thread's last error ("" if none). */
const char* ft_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* FT_MOE_H */
