/*
 * moecache — a routed Mixture-of-Experts layer served from one GPU-resident
 * expert cache shared by all layers, backed by a pinned host expert pool.
 *
 * Method (FreeToken, "Efficient Edge-Native MoE Serving with Bandwidth-
 * Adaptive Execution", as summarised on discuss.pytorch.kr "FreeToken:
 * 프론티어급 MoE 모델을 게이밍 데스크톱 수준에서 서빙하기 위한 Edge-Serving에
 * 대한 연구" and read on qqtang-code.github.io):
 *  - "FreeToken's design": a host expert pool is the source of truth; the
 *    free GPU memory is one elastic expert cache shared by every MoE layer,
 *    each slot holding every tensor of one (layer, expert) pair.
 *  - "Router-following LRU cache": hits refresh recency, fills admit the
 *    newly selected expert, eviction removes the expert not requested for
 *    the longest time.
 *  - "CUDA Graph-compatible LRU cache": per layer one GPU kernel deduplicates
 *    the routed experts, classifies them against the residency table, picks
 *    K victims in one pass and rewrites logical ids to slot ids.
 *  - "Measured bandwidths decide the split": the GPU evaluates G = H ∪ F as
 *    one grouped FFN after the batched copy of the fills; partial sums merge
 *    exactly.
 *  - "Full-layer double buffering" (prefill): two full-layer buffers from
 *    the global slot pool; a transfer stream loads layer l+1 while layer l
 *    computes.
 *  - "Elastic memory management": at a scheduler safe point the cache is
 *    rebuilt to a new budget without reloading the host pool.
 *
 * Conventions for every entry point:
 *  - Returns a moe_status; nothing throws or aborts across this boundary.
 *    On failure moe_last_error() returns a message (thread-local).
 *  - "device" pointers are CUDA device addresses on the device that was
 *    current at moe_cache_create; "host" pointers are ordinary process
 *    memory.  Streams are cudaStream_t values passed as void* (NULL = the
 *    legacy default stream).
 *  - One cache is driven by one host thread at a time.
 *  - Expert key of (layer l, expert e) is l*E + e.
 *
 * Expert record (one host-pool row, one cache slot), row-major [out][in]:
 *  MOE_FP32, MOE_BF16: W_gate[I][H] | W_up[I][H] | W_down[H][I]
 *  MOE_FP4: gate codes[I][H/2] | up codes[I][H/2] | gate scales[I][H/16] |
 *           up scales[I][H/16] | down codes[H][I/2] | down scales[H][I/16]
 *  In every format the first part (everything the gate/up projections read)
 *  and the second part (W_down) are each contiguous.
 *    (e2m1 codes, element 2c in the low nibble of byte c; one e4m3 scale per
 *     16 consecutive elements of a row; no per-tensor scale)
 *  Expert FFN: h = SiLU(x W_gate^T) * (x W_up^T), o = h W_down^T.
 */
#ifndef MOECACHE_H
#define MOECACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, shape or state */
  MOE_ERR_OOM = 2,         /* device or pinned memory could not be obtained */
  MOE_ERR_CAPACITY = 3,    /* a call routes more distinct experts than there are slots */
  MOE_ERR_BUSY = 4,        /* resize while work of this cache is still in flight */
  MOE_ERR_CUDA = 5,        /* a CUDA call failed; see moe_last_error() */
  MOE_ERR_TIMEOUT = 6      /* a bounded wait gave up */
};

/* weight formats */
enum { MOE_FP32 = 0, MOE_BF16 = 1, MOE_FP4 = 2 };

/* event kinds in the cache trace */
enum { MOE_EV_HIT = 0, MOE_EV_MISS = 1, MOE_EV_RESIZE_EVICT = 2, MOE_EV_PREFILL_EVICT = 3 };

typedef struct {
  int32_t L;          /* MoE layers */
  int32_t E;          /* routed experts per layer (1 .. 1024) */
  int32_t k;          /* experts per token (1 .. 16, <= E) */
  int32_t H;          /* hidden size */
  int32_t I;          /* per-expert SwiGLU intermediate size */
  int32_t wdtype;     /* MOE_FP32 | MOE_BF16 | MOE_FP4 */
  int32_t has_shared; /* 1: every layer also runs one always-resident, ungated shared expert */
  int32_t max_tokens; /* largest B passed to moe_layer_forward (1 .. 16) */
} moe_model_desc;
/* Shape rules: MOE_FP32/MOE_BF16 need H and I multiples of 64; MOE_FP4 needs
 * multiples of 256 and H <= 16384.  Activations x and outputs y are float32 for MOE_FP32
 * models and bf16 otherwise. */

typedef struct {
  int64_t calls;             /* moe_layer_forward calls that completed */
  int64_t tokens;            /* tokens over those calls */
  int64_t hits, misses;      /* distinct (call, expert) accesses */
  int64_t evictions;         /* misses that displaced a resident expert */
  int64_t routed_pairs;      /* (token, rank) pairs */
  int64_t routed_pair_hits;  /* pairs whose expert was resident before the call */
  int64_t bytes_filled;      /* host -> device bytes copied by fills */
  int64_t layer_launches;    /* layer-kernel launches (one per call) */
  int64_t records_streamed;  /* expert records read by the completed calls (incl. shared) */
  double layer_ms;           /* summed device time of timed launches (profiling on) */
  int64_t layer_timed;       /* launches included in layer_ms */
  double hit_only_ms;        /* ... of those, launches of calls without fills */
  int64_t hit_only_timed;
  int64_t hit_only_records;  /* records those calls read */
  double host_wait_us;       /* host time from launch to seeing the call's miss list */
  double host_issue_us;      /* host time spent issuing fills */
  int64_t resize_calls, resize_moves, resize_evictions;
  int64_t prefill_layers;
  int64_t prefill_tokens;    /* tokens x layers processed by moe_prefill_stream */
  double prefill_ms;         /* device time of whole moe_prefill_stream calls (profiling on) */
  double prefill_copy_ms;    /* summed duration of the per-layer host -> device expert streams */
  double prefill_compute_ms; /* summed per-layer compute time after each layer's experts landed */
  double prefill_gemm_ms;    /* summed time of the grouped GEMM launches */
  double prefill_gemm_flop;  /* useful flops of those launches (2 * rows * N * K) */
  int64_t deferred_calls;    /* copy-fill calls finished by the completion kernel (fills landed late) */
  int64_t finish_launches;   /* completion-kernel launches (one per copy-fill call with misses) */
  int64_t pdl_launches;      /* layer-kernel launches made as programmatic dependents of the previous launch */
  int64_t prefill_records_streamed;  /* expert records moe_prefill_stream copied into its buffers */
  int64_t prefill_records_in_place;  /* expert records it read where they were already resident */
  int64_t qstar_fills;       /* sum over calls of q*, the fill count of the bandwidth split */
  int64_t summaries_lost;    /* graph mode: calls whose summary a later call overwrote before moe_cache_sync
                                read it (more than 256 calls in between); not counted in the other fields */
} moe_stats;

typedef struct {
  int64_t call;        /* index of the moe_layer_forward call (resize: calls so far) */
  int32_t layer;
  int32_t expert;
  int32_t kind;        /* MOE_EV_* */
  int32_t slot;
  int32_t evicted_key; /* key displaced by a miss or resize eviction, -1 if none */
  int32_t pad;
} moe_event;

/* Optional device outputs of one forward call, for inspection.  Every field
 * may be NULL.  Sizes are for B tokens. */
typedef struct {
  int32_t* ids;      /* [B][k] selected experts, descending logit, ties -> lower id */
  float* weights;    /* [B][k] routing weights (softmax over the k selected logits) */
  int32_t* slots;    /* [B][k] cache slot of each selected expert after the call */
  int32_t* perm;     /* [B*k] flat pair indices t*k+j grouped by expert (stable) */
  int32_t* offsets;  /* [E+1] start of each expert's group in perm */
  float* logits;     /* [B][E] router logits actually used (float32) */
  int32_t* qstar;    /* [1] q*: how many of the call's misses the bandwidth split fills */
} moe_layer_aux;

typedef struct moe_cache* moe_cache_t;

/* Bytes of one expert record for desc (0 if desc is invalid). */
size_t moe_record_bytes(const moe_model_desc* desc);

/* Create a cache.
 * host_pool: host memory holding L*E records back to back (row l*E+e).  It
 *   must be page-locked (cudaHostAlloc or cudaHostRegister), stay valid and
 *   unchanged until moe_cache_destroy, and is never written by the library.
 * shared_dev: device memory with L records (shared expert of layer l at row
 *   l), required iff desc->has_shared; owned by the caller.
 * n_slots: initial capacity C (>= 0).  max_slots: upper bound for resizes
 *   (0 means L*E); device virtual address space for max_slots records is
 *   reserved up front and physical memory is mapped for the first C only.
 * copy_stream: stream for fills (NULL: the library creates one).  The
 *   library also creates one internal copy stream; copy-mode fill records
 *   alternate between the two, both ordered after the work that precedes
 *   each layer call on the compute stream.
 * Errors: MOE_ERR_INVALID_ARG (shapes, pointers, unpinned pool),
 *   MOE_ERR_OOM, MOE_ERR_CUDA.  On error *out is NULL. */
moe_status moe_cache_create(const moe_model_desc* desc, const void* host_pool, const void* shared_dev,
                            int64_t n_slots, int64_t max_slots, void* copy_stream, moe_cache_t* out);

/* Rebuild the cache with n_slots slots at a safe point ("elastic memory
 * management").  Shrinking keeps the n_slots most recently used experts,
 * evicts the rest (logged as MOE_EV_RESIZE_EVICT in ascending slot order)
 * and moves survivors sitting in slots >= n_slots into the vacant low slots
 * (ascending old slot -> ascending vacant slot), then unmaps the tail.
 * Growing maps more slots, empty.  Recency and the host pool are untouched.
 * stream: where the device copies run; the call returns after they finish.
 * Errors: MOE_ERR_BUSY if a forward of this cache has not finished on the
 * GPU, MOE_ERR_INVALID_ARG if n_slots > max_slots, MOE_ERR_OOM, MOE_ERR_CUDA. */
moe_status moe_cache_resize(moe_cache_t cache, int64_t n_slots, void* stream);

/* One decode-size MoE layer call (1 <= B <= desc->max_tokens).
 * x: device [B][H] (bf16, or float32 for MOE_FP32).  y: device [B][H], same
 *   type, written.
 * logits: device float32 [B][E], or NULL to compute logits = x W_r^T from
 *   router_w: device float32 [E][H] (then router_w must not be NULL).
 * The call routes (top-k softmax), updates the LRU cache (inside the layer
 * kernel), copies each miss's record from the host pool into its victim slot
 * with cudaMemcpyAsync on the copy streams while the resident experts already
 * run, evaluates every selected expert (and the shared expert) straight from
 * the cache slots, and writes y_t = sum_j w_tj * o_tj (+ shared) in rank order.
 * Arithmetic: products exact, sums in float32; for MOE_FP4 models x is read as
 * f16 (exact for 2^-14 <= |x| <= 65504 and 0) and the SwiGLU intermediate is
 * rounded to f16 before the down projection (float32 otherwise).  Every dot
 * product has a fixed summation order, so y is bitwise the same whatever the
 * residency, fill mode or cache size.
 * Copy-fill mode (default): the host waits once per call for the layer
 * kernel's miss list (it issues the copies), then enqueues a small completion
 * kernel on `stream` after the call's copies; the layer kernel consumes each
 * fill as it lands, and if a fill is late (see moe_cache_set_wait_limit_ns)
 * it hands the remaining work to the completion kernel, so y is always this
 * call's result once `stream` reaches the end of the call.  Device-fill mode:
 * the call does not wait for the GPU at all when B*k <= n_slots.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CAPACITY (more distinct experts than
 *   slots; cache unchanged, y unspecified), MOE_ERR_CUDA (a fill could not be
 *   issued: the completion kernel rolls recency back and leaves this call's
 *   victim slots empty; y unspecified), MOE_ERR_TIMEOUT (a bounded wait inside
 *   an earlier kernel of this cache gave up: the outputs of that call are NaN;
 *   the state has been recovered and this call did nothing).  Errors that the
 *   GPU finds after the call returned (a bounded wait that gave up, or, in
 *   device-fill mode, an inconsistent victim list) are reported by
 *   moe_cache_sync and by the next call. */
moe_status moe_layer_forward(moe_cache_t cache, int32_t layer, const void* x, const float* logits,
                             const float* router_w, int32_t B, void* y, void* stream);

/* moe_layer_forward with optional inspection outputs (aux may be NULL). */
moe_status moe_layer_forward_ex(moe_cache_t cache, int32_t layer, const void* x, const float* logits,
                                const float* router_w, int32_t B, void* y, void* stream,
                                const moe_layer_aux* aux);

/* Prefill of T tokens through layers [layer_begin, layer_end) with full-layer
 * double buffering ("전층 이중 버퍼링" in the FreeToken write-up): two buffers
 * of E slots each are carved from the slot pool (the last 2*E slots; their
 * entries are evicted, logged as MOE_EV_PREFILL_EVICT in ascending slot
 * order); while layer l runs on one, layer l+1's experts stream into the
 * other on the copy stream.  An expert already resident elsewhere in the
 * cache is read where it is, not streamed.  Every expert of a prefilled layer
 * counts as used by it (stamps g + e per layer, in layer order), and the
 * buffers' contents stay cached afterwards: what survives prefill seeds
 * decode.  Prompts longer than 8192 tokens run as consecutive 8192-token
 * chunks, each a full pass over the layers.
 * x: device [n_layers][T][H] bf16 (each layer's input), logits: device float32
 * [n_layers][T][E], y: device [n_layers][T][H] bf16.  Only MOE_BF16 / MOE_FP4
 * models; prefill also needs I % 128 == 0 and H % 256 == 0.  The expert GEMMs
 * accumulate in float32; their operands are bf16 for MOE_BF16 models and f16
 * for MOE_FP4 models (an activation converts exactly when 2^-14 <= |x| <=
 * 65504 or x = 0; smaller magnitudes round to the f16 subnormal grid, an
 * absolute error of at most 2^-25; the FP4 weights expand exactly; the SwiGLU
 * intermediate is rounded to f16), or,
 * after moe_cache_set_prefill_precision(MOE_PREFILL_W4A4), FP4 x FP4.
 * The host waits once at the start for the cache's earlier work (it plans the
 * copies from the residency table); the rest is asynchronous on `stream`.
 * When the pool has fewer than 2*E slots the experts are loaded on demand
 * instead (the pages' fallback, without oversubscribing GPU memory): per
 * layer the host reads which experts the tokens route to (one wait per
 * layer), and accesses them in ascending order in chunks of at most n_slots,
 * each chunk like one decode call (hits refresh recency, misses take victims
 * and are copied in, logged as MOE_EV_HIT / MOE_EV_MISS), then evaluates the
 * chunk before the next one may evict it.
 * Errors: MOE_ERR_CAPACITY (no slots at all), MOE_ERR_INVALID_ARG,
 * MOE_ERR_OOM, MOE_ERR_CUDA. */
moe_status moe_prefill_stream(moe_cache_t cache, int32_t layer_begin, int32_t layer_end, const void* x,
                              const float* logits, int32_t T, void* y, void* stream);

/* Optional device outputs of moe_prefill_stream_ex; every field may be NULL.
 * perm, offsets and slots need T <= 8192 (one chunk). */
typedef struct {
  int32_t* ids;      /* [n_layers][T][k] selected experts, descending logit, ties -> lower id */
  float* weights;    /* [n_layers][T][k] routing weights */
  int32_t* perm;     /* [n_layers][T*k] flat pairs t*k+j grouped by expert (stable) */
  int32_t* offsets;  /* [n_layers][E+1] start of each expert's group in perm */
  int32_t* slots;    /* [n_layers][E] cache slot each expert of the layer was read from (on demand: -1 when
                        no token routes to it) */
} moe_prefill_aux;

/* moe_prefill_stream with optional inspection outputs (aux may be NULL). */
moe_status moe_prefill_stream_ex(moe_cache_t cache, int32_t layer_begin, int32_t layer_end, const void* x,
                                 const float* logits, int32_t T, void* y, void* stream, const moe_prefill_aux* aux);

/* Wait for every call of this cache enqueued so far (on `stream` and on the
 * cache's copy streams), read their summaries, and return the first error
 * the GPU found after the calls returned: MOE_ERR_TIMEOUT when a bounded
 * wait inside a kernel gave up (the rows of that call are NaN; the state is
 * recovered), MOE_ERR_CUDA for an inconsistent victim list in device-fill
 * mode.  MOE_OK otherwise.  The error is cleared once returned. */
moe_status moe_cache_sync(moe_cache_t cache, void* stream);

/* How long the layer kernel waits for a fill's gate/up half (gate_up_ns) and
 * for its W_down half (down_ns) in copy-fill mode before it hands the rest of
 * the call to the completion kernel (default 2 ms each; 0 hands over at once
 * whenever a half has not landed yet).  Either way the result is the same,
 * bit for bit; the limits only trade SM time spent waiting against a second
 * pass over the fills.  Errors: MOE_ERR_INVALID_ARG (negative or above 60 s). */
moe_status moe_cache_set_wait_limit_ns(moe_cache_t cache, int64_t gate_up_ns, int64_t down_ns);

/* Bandwidths of the fill / host-execution split ("measured bandwidths decide
 * the split" in the FreeToken write-up): with m misses in a call, the layer
 * kernel derives q* = m * b_p / b_h rounded to the nearest integer (halves
 * up), clamped to [1, m], q* = m when b_h <= b_p, 0 when m = 0; b_p is the
 * measured host-to-device expert-transfer bandwidth, b_h the host's expert
 * execution bandwidth, any unit.  This library has no host execution branch:
 * every miss is still filled, and q* is reported (moe_layer_aux.qstar,
 * moe_stats.qstar_fills) for the split a hybrid engine would take.  Both 0
 * (the default) means q* = m.  Errors: MOE_ERR_INVALID_ARG (negative). */
moe_status moe_cache_set_split_bandwidths(moe_cache_t cache, double b_p, double b_h);

/* Counters since creation (or the last reset).  Synchronises the events of
 * profiled launches and reads the summaries of calls in flight. */
moe_status moe_cache_stats(moe_cache_t cache, moe_stats* out);
moe_status moe_cache_reset_stats(moe_cache_t cache);

/* on >= 1: time every layer-kernel and prefill launch with CUDA events.
 * on >= 2: also record GPU timestamps at the phases of every layer call
 * (see moe_phase_times). */
moe_status moe_cache_set_profiling(moe_cache_t cache, int32_t on);

/* Mean time, in microseconds after the layer kernel starts, at which a call
 * reaches each phase, over the calls profiled at level 2 (split by whether
 * the call had fills), as seen by CTA 1 unless noted.  Stamps: 0 start, 1
 * routing and lookup done, 2 gate/up rows of the resident experts streamed, 3
 * W_down rows started (after the grid barrier), 4 W_down rows of the resident experts
 * done, 5 first fill's first half landed, 6 gate/up rows of the fills done, 7
 * plan of the fills read, 8 last fill's second half landed, 9 end, 10 control
 * CTA: victims and plan written, 11 control CTA: recency committed, 12 router
 * done, 13 the router starts loading the first token's logits, 14 lookups and grouping done,
 * 15 the first token's router logits loaded; over all CTAs: 16 the first and
 * 17 the last to finish the gate/up rows of the resident experts, 18 the last
 * to finish routing and lookup, 19 the last to end.  A call that never
 * reaches a stamp does not count towards it. */
typedef struct {
  int64_t calls_hit_only, calls_with_fills;
  double hit_only_us[20];
  double with_fills_us[20];
} moe_phase_times;
moe_status moe_cache_phase_times(moe_cache_t cache, moe_phase_times* out);

/* on != 0: record one moe_event per distinct expert access and per resize
 * eviction.  moe_cache_trace copies up to cap recorded events to buf (host)
 * and sets *n to the number recorded in total. */
moe_status moe_cache_set_trace(moe_cache_t cache, int32_t on);
moe_status moe_cache_trace(moe_cache_t cache, moe_event* buf, int64_t cap, int64_t* n);

/* Copy of the cache state to host buffers (each may be NULL): owner key of
 * every slot (-1 empty) and its recency stamp (cap entries at most), the
 * current slot count and the global recency counter.  Synchronises. */
moe_status moe_cache_state(moe_cache_t cache, int32_t* owner, uint64_t* stamp, int64_t cap, int64_t* n_slots,
                           uint64_t* counter);

/* Device address of slot s (for inspection); NULL if s is out of range. */
const void* moe_cache_slot_ptr(moe_cache_t cache, int64_t s);

/* How misses are filled.
 * MOE_FILL_COPY (default): the host issues cudaMemcpyAsync of each missed
 *   record from the pinned pool into its victim slot on the copy stream, and
 *   the layer kernel consumes each half as its stream-written flag arrives.
 * MOE_FILL_DEVICE: the layer kernel reads each missed record from the pinned
 *   pool itself (the pool must be mapped at the same device address, as on
 *   unified-addressing systems), uses it for the call and stores it in its
 *   victim slot: the fused, fixed-shape, device-driven transfer of the
 *   "CUDA Graph-compatible LRU cache" section, with no host step on the fill
 *   path.  Results are identical in both modes.
 * Errors: MOE_ERR_INVALID_ARG (unknown mode, pool not mapped). */
enum { MOE_FILL_COPY = 0, MOE_FILL_DEVICE = 1 };
moe_status moe_cache_set_fill_mode(moe_cache_t cache, int32_t mode);

/* Arithmetic of moe_prefill_stream for MOE_FP4 models.
 * MOE_PREFILL_W4A16 (default): the FP4 weights expand exactly to f16 and the
 *   GEMMs run on f16 activations (see moe_prefill_stream).
 * MOE_PREFILL_W4A4: the activations are quantised to the weights' own format
 *   (the pages deploy MXFP4 / NVFP4 experts, FreeToken write-up, experimental
 *   setup; they do not say how activations are treated, this is the reading
 *   that lets both GEMM operands use the block-scaled FP4 tensor-core path):
 *   the layer input x before the gate/up GEMM and the SwiGLU output h, rounded
 *   to float32, before the down GEMM, each with moe_quantize_fp4's rule; the
 *   GEMMs then run as block-scaled FP4 x FP4 products accumulating in float32.
 *   Needs H and I multiples of 256 (the MOE_FP4 rule).
 * The setting applies to later moe_prefill_stream calls; decode is unaffected.
 * Errors: MOE_ERR_INVALID_ARG (unknown mode, or W4A4 for a model that is not
 * MOE_FP4). */
enum { MOE_PREFILL_W4A16 = 0, MOE_PREFILL_W4A4 = 1 };
moe_status moe_cache_set_prefill_precision(moe_cache_t cache, int32_t mode);

/* The FP4 quantiser of the W4A4 prefill, for rows of activations.
 * Each block of 16 consecutive elements of a row gets one e4m3 scale
 * s = e4m3(amax / 6) and each element the e2m1 code of v / s; both are
 * rounded to nearest with ties to the even code and saturated to the largest
 * finite value (448 and 6); amax / 6 and v / s are IEEE float32 divisions.
 * A block whose scale rounds to 0 gets codes 0, and a value that rounds to
 * magnitude 0 gets code 0 (never the negative zero 0x8).
 * x: device [rows][K], bf16 (x_dtype MOE_BF16) or float32 (MOE_FP32), aligned
 * to its element size; codes: device [rows][K/2], element 2c of a row in the
 * low nibble of byte c, 8-byte aligned; scales: device [rows][K/16].  K a
 * positive multiple of 16.  Asynchronous on `stream`; all buffers owned by
 * the caller.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA (launch failure). */
moe_status moe_quantize_fp4(const void* x, int32_t x_dtype, int64_t rows, int32_t K, uint8_t* codes,
                            uint8_t* scales, void* stream);

/* Graph mode (on = 1): decode calls may be captured into CUDA graphs and
 * replayed ("CUDA Graph와 공존하는 LRU 캐시" in the FreeToken write-up: the
 * control step runs on the device so the whole decode step can be a graph).
 * Needs MOE_FILL_DEVICE (a copy-mode call waits on the host).  In graph mode
 * moe_layer_forward only enqueues the layer kernel (no host wait, event or
 * allocation); the kernel numbers the call from a device counter, so every
 * replay of a captured call is a new call with its own recency, fills and
 * evictions, exactly as if it had been launched.  The host reads the calls'
 * summaries (statistics, trace) at moe_cache_sync, or when graph mode is
 * turned off; call moe_cache_sync at least every 256 calls or the oldest
 * summaries are overwritten (counted in summaries_lost; the cache state
 * itself is never affected).  Calls need B * k <= n_slots.  Profiling
 * timestamps and per-launch events are not recorded in graph mode.
 * Turning it on or off synchronises the device.
 * Errors: MOE_ERR_INVALID_ARG (copy-fill mode). */
moe_status moe_cache_set_graph_mode(moe_cache_t cache, int32_t on);

/* Test hook: the next fill copies of this cache fail after `after` successful
 * copies (-1 disables).  Used to check the rollback path without a GPU fault. */
moe_status moe_cache_inject_fill_failure(moe_cache_t cache, int32_t after);

/* Routed MoE layer for callers that cannot allocate device memory (their
 * device memory is owned by another allocator or a fixed budget, or a
 * synchronising cudaMalloc/cudaFree is not acceptable on their path).  The
 * pages have no counterpart: it is the same layer as moe_layer_forward with
 * every expert resident, without a cache.
 * desc: E, k, H, I, wdtype, has_shared are used (L, max_tokens ignored).
 * bank: device, the E expert records of the layer back to back (record
 *   layout as above); shared_rec: device record of the shared expert, required
 *   iff desc->has_shared.  x: device [B][H], logits: device float32 [B][E],
 *   y: device [B][H] written; 1 <= B <= 16.  All owned by the caller.
 * Scratch: a 4 MiB + 16 KiB array inside the library, held by every GPU that
 *   loads it until the process exits; (B*k + B) * I * 4 bytes must fit in
 *   4 MiB, otherwise MOE_ERR_INVALID_ARG.  The first call on a device looks the
 *   array's device address up (cudaGetSymbolAddress) and should come before
 *   any stream capture.  Nothing in the scratch needs to start at zero; every
 *   call overwrites it, so calls that overlap on the GPU (different streams,
 *   different threads) race and must be serialised by the caller.
 * Never calls cudaMalloc, cudaFree or any allocating routine.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA (launch failure). */
moe_status moe_layer_forward_resident_noalloc(const moe_model_desc* desc, const void* bank, const void* shared_rec,
                                              const void* x, const float* logits, int32_t B, void* y, void* stream);

/* Free everything the library allocated.  Synchronises. */
moe_status moe_cache_destroy(moe_cache_t cache);

/* Bounds checks of the debug build (the library compiled with
 * -DMOE_DEBUG_BOUNDS, a stand-in for a device memory checker): every index
 * the kernels derive from the cache state or the routing (slots, keys, pair
 * positions, h rows, output rows) is checked before use; a bad one is
 * counted and its access skipped.  moe_debug_bounds_enabled: 1 when this
 * library has the checks, 0 otherwise. */
int32_t moe_debug_bounds_enabled(void);

/* Violations the checks counted in this process so far and the site of the
 * first (0 if none).  Synchronises the device.  A release build reports 0.
 * Errors: MOE_ERR_INVALID_ARG (NULL argument), MOE_ERR_CUDA. */
moe_status moe_debug_violations(int64_t* count, int32_t* first_site);

/* Measurement aid (no counterpart on the pages): the HBM read rate, in GB/s,
 * of a kernel that does nothing but read `bytes` per launch with the decode
 * layer kernel's weight loads (16-byte, L2 evict-first, every SM).  bufs:
 * device memory of n_bufs * bytes, caller-owned; launch r reads buffer
 * r % n_bufs, so with n_bufs * bytes well above the 129 MB L2 no launch finds
 * its bytes in L2.  One untimed pass over every buffer, then reps launches
 * back to back timed with events on `stream`; blocks until they end.  It is
 * the practical ceiling for a layer call that streams the same bytes (a
 * launch's ramp-up and drain included).  Errors: MOE_ERR_INVALID_ARG (NULL,
 * bytes not a positive multiple of 16, bufs not 16-byte aligned, n_bufs or
 * reps < 1), MOE_ERR_CUDA. */
moe_status moe_measure_read_rate(const void* bufs, int64_t bytes, int32_t n_bufs, int32_t reps, void* stream,
                                 double* gbps);

/* Message of the last error on this thread ("" if none). */
const char* moe_last_error(void);

/* Library ABI version. */
int32_t moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOECACHE_H */
