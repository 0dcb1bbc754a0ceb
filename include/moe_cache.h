/*
 * moe_cache.h -- C ABI of the GB300 offloaded-MoE expert slot cache.
 *
 * One MoE decode layer whose expert weights live in pinned host memory: the
 * GPU keeps the hot experts in a fixed pool of device "slots".  The library
 * runs, all on one GPU (sm_103a) and without a host synchronisation:
 *   1. admission (moe_admit): dedup the step's top-k ids, look them up in the
 *      expert->slot map, refresh recency on hits, pick least-recently-used
 *      victims for misses, write a device-side miss plan, rewrite ids to slot
 *      ids (-1 for routes that get no slot);
 *   2. the miss gather (moe_gather_missing): copy the planned experts' bytes
 *      from pinned host memory into their slots;
 *   3. the routed expert FFNs over the slots, the sigmoid-gated shared expert
 *      and the weighted combine (moe_routed_experts, moe_decode_layer).
 * Look-ahead prefetch with an LFRU eviction guard (moe_prefetch) fills slots
 * for the next layer.
 *
 * Sources (page title, section):
 *  [P1] FreeToken PR #491 "refactor(moe): extract hybrid decode orchestration"
 *  [P2] FreeToken issue #753 "[Perf] Offloaded decode: overlap the expert-miss
 *       gather with the same layer's shared expert, event-ordered inside the
 *       CUDA graph"
 *  [P3] FreeToken PR #680 "fix(moe): admit a wide offloaded decode step's
 *       experts 128 at a time"
 *  [P4] llama.cpp fork PR #126 "cuda : MoE look-ahead expert prefetch (PR-A
 *       consumer) + LFRU eviction guard"
 *
 * ---------------------------------------------------------------- conventions
 * Pointers named d_* are device pointers (or device-accessible), h_* host
 * pointers.  Streams are cudaStream_t passed as void* (NULL = legacy default
 * stream).  Expert ids, slot ids and route indices are int32; routing weights
 * float32; hidden states and outputs bfloat16 (uint16 bit patterns).
 *
 * Ownership: the caller owns every tensor it passes (inputs, outputs, the slot
 * storage, the pinned host blobs, the streams); pinned host blobs and slot
 * storage must outlive the cache.  The cache owns its state (maps, stamps,
 * frequencies, plans, statistics, scratch) and two CUDA events, all created in
 * moe_cache_create, i.e. before any stream capture.
 *
 * Errors: every call returns MOE_OK (0) or a negative MOE_ERR_* code and never
 * aborts or throws.  Argument errors are detected on the host before any work
 * is enqueued.  Data-dependent anomalies never stop the stream: an id outside
 * [0, n_experts) becomes route -1 and sets MOE_STATUS_INVALID_ID in the
 * layer's statistics; a pool with too few evictable slots admits what it can
 * (lowest expert ids first), the rest overflow (-1) and MOE_STATUS_CAPACITY is
 * set.  Only moe_read_stats, moe_cache_prefill and moe_cache_destroy
 * synchronise with the device; every other call only enqueues work and may be
 * captured into a CUDA graph (fixed n_routes / n_rows / n_pred per capture).
 *
 * Single writer [P2 What we changed]: moe_admit, moe_prefetch and the layer's
 * routed compute must be ordered on one (compute) stream; the gather only
 * reads the plan and writes slot bytes.
 *
 * ---------------------------------------------------------------- layouts
 * Keys: key = layer * n_experts + expert.  Pools: MOE_POOL_SHARED has one pool
 * of n_slots used by every layer; MOE_POOL_PER_LAYER has n_layers pools of
 * n_slots each.  A slot id is the index within its pool.  Slot s of pool p
 * lives at slot_storage + (p * n_slots + s) * slot_stride.
 *
 * Expert blob (the copy unit, one contiguous block per expert, identical in
 * host memory and in a slot) [P2 What we changed "fused copy layout",
 * Correctness "six-bank NVFP4 row sizes"]:
 *   MOE_W_BF16:  gate [I][H], up [I][H], down [H][I], bf16 row-major;
 *                6*H*I bytes.
 *   MOE_W_NVFP4: six banks then the global scales:
 *                gate codes [I][H/2], up codes [I][H/2], down codes [H][I/2]
 *                  (FP4 E2M1, two per byte, even element in the low nibble),
 *                gate scales [I][H/16], up scales [I][H/16], down scales
 *                  [H][I/16] (FP8 E4M3, one per 16 consecutive row elements),
 *                float32 global scale of gate, up, down, 4 bytes of padding;
 *                3*H*I/2 + 3*H*I/16 + 16 bytes.
 *                element (n,k) = e2m1(code) * e4m3(scale[n][k/16]) * global.
 *   MOE_W_MXFP4: the same three code banks, then gate scales [I][H/32], up
 *                scales [I][H/32], down scales [H][I/32] (E8M0: 2^(s - 127),
 *                0xFF = NaN, one per 32 consecutive row elements), no global
 *                scale; 3*H*I/2 + 3*H*I/32 bytes [P1 section 7 lists MXFP4
 *                among the expert formats; layout of the OCP Microscaling
 *                MXFP4 blocks].  element (n,k) = e2m1(code) * 2^(scale[n][k/32] - 127).
 *                Every path but the tensor-core one: the decode-sized streaming
 *                kernels (H a multiple of 2048, I of 512), the wide steps'
 *                grouped kernels on the CUDA cores, the per-route kernels
 *                beyond both, and the hybrid CPU executor.
 *   MOE_W_Q4_0:  the arithmetic of Q4_0 (blocks of 32 weights, weight =
 *                d * (q - 8) with q an unsigned 4-bit code and d an fp16
 *                scale) in the same banked layout: the three code banks (q,
 *                two per byte, even element in the low nibble), then gate
 *                scales [I][H/32], up scales [I][H/32], down scales [H][I/32]
 *                as fp16 d; 3*H*I/2 + 3*H*I/16 bytes [P1 section 7 lists
 *                Q4_0].  Not the interleaved block bytes of other libraries.
 *                Same shapes and paths as MOE_W_MXFP4.
 *   H, I and shared_inter must be multiples of 32 (checked at create).
 * Shared expert: a blob of the same format with I = shared_inter, plus a gate
 *   vector w_g bf16 [H]: shared(x) = sigmoid(x . w_g) * FFN_shared(x).
 * Expert FFN: g = W_g x, u = W_u x, h = silu(g) * u, y = W_d h.
 * Layer output: out[b] = bf16( sum_j w[b,j] * y(slot[b,j], x[b])  +  shared(x[b]) )
 *   routes with slot -1 contribute nothing; the sum runs over j ascending, then
 *   adds the shared term; fp32 accumulation throughout.
 *
 * Miss plan (device, int32): [count, (slot, layer, expert) * count], entries
 *   in ascending expert id; a plan holds at most max_routes (demand) or
 *   max_pred (prefetch) entries.  There is one demand plan and two prefetch
 *   plans: a prefetch for layer l writes plan l & 1, so the side-stream gather
 *   of layer l's prefetch may still read its plan while layer l+1's prefetch
 *   (for l+2) is admitted; moe_gather_missing / moe_rollback_plan with
 *   MOE_PLAN_PREFETCH use the plan of the most recent prefetch call.
 * Route groups (device, int32, written by moe_routed_experts on the grouped
 * path, i.e. for steps wider than the streaming kernel takes: more than 16
 * rows or 64 routes):
 *   [G, slot[max_routes], start[max_routes + 1], route[max_routes]]: group g
 *   is the g-th distinct resident expert in ascending id, its slot, and its
 *   routes route[start[g] .. start[g+1]) in ascending route index.
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_CACHE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

enum moe_err {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* a NULL, a size out of range, a bad enum */
  MOE_ERR_CONFIG = -2,        /* inconsistent moe_cache_desc */
  MOE_ERR_CUDA = -3,          /* a CUDA runtime call failed (see moe_last_cuda_error) */
  MOE_ERR_CAPACITY = -4,      /* more routes / rows / predictions than the cache was sized for */
  MOE_ERR_UNSUPPORTED = -5,   /* shape or format this build does not handle */
  MOE_ERR_STATE = -6,         /* call not valid in the cache's current state */
  MOE_ERR_INJECTED = -7,      /* a test-requested failure (moe_cache_fail_next_gather) */
  MOE_ERR_SCRATCH = -8        /* request larger than MOE_NOALLOC_SCRATCH_BYTES allows */
};

typedef enum { MOE_W_BF16 = 0, MOE_W_NVFP4 = 1, MOE_W_MXFP4 = 2, MOE_W_Q4_0 = 3 } moe_wfmt;
typedef enum { MOE_POOL_SHARED = 0, MOE_POOL_PER_LAYER = 1 } moe_pool_mode;
typedef enum { MOE_PLAN_DEMAND = 0, MOE_PLAN_PREFETCH = 1 } moe_plan_kind;

/* moe_decode_layer flags */
#define MOE_OVERLAP 1u        /* gather on the side stream, joined by events [P2] */
#define MOE_FUSED 2u          /* one launch per layer: the admission, the gathers, the shared
                                 expert and the routed experts (decode-sized steps) */
#define MOE_HYBRID 4u         /* routes left at -1 run on the host's cores and are added to
                                 the output (needs moe_hybrid_start) [P1] */

/* status_bits of moe_stats */
#define MOE_STATUS_INVALID_ID 1ull
#define MOE_STATUS_CAPACITY 2ull
#define MOE_STATUS_TIMEOUT 4ull   /* a bounded device wait gave up (reported in every layer) */

typedef struct moe_cache moe_cache; /* opaque */
typedef struct moe_cpu_exec moe_cpu_exec; /* opaque: a cache's hybrid CPU executor */

typedef struct {
  int n_layers;                    /* > 0 */
  int n_experts;                   /* per layer, 1 .. 16384 */
  int n_slots;                     /* per pool, 0 .. 1,048,575 */
  int pool_mode;                   /* moe_pool_mode */
  int hidden, inter;               /* H, I of a routed expert (0, 0 = admission only) */
  int wfmt;                        /* moe_wfmt */
  int shared_inter;                /* I of the shared expert, 0 = none */
  size_t slot_bytes;               /* bytes copied per expert: the blob size, 0 = no storage */
  size_t slot_stride;              /* >= slot_bytes, multiple of 256; 0 = round up slot_bytes */
  void* slot_storage;              /* device, caller-owned, n_pools*n_slots*slot_stride bytes */
  const void* const* host_experts; /* host array [n_layers*n_experts] of pinned host blob
                                      pointers (16-byte aligned; may alias); read at create */
  int max_routes;                  /* routes per admission, 1 .. 16384 */
  int max_rows;                    /* rows per layer call, 1 .. max_routes */
  int max_pred;                    /* predictions per prefetch, 0 .. 4096 (0 = no prefetch) */
  int gather_ctas;                 /* CTAs of the gather kernel, 0 = default (76) */
} moe_cache_desc;

/* Per-layer counters, device-resident, read with moe_read_stats.
 * [P3 Solution]: a step counts once -- calls += 1, lookups += distinct valid
 * ids ("met"), misses += distinct ids not resident -- while decode_freq
 * counts every valid route.  fetched = misses admitted (copied);
 * overflow_routes = valid routes left at -1.  pf_*: prefetch counters [P4
 * Consumer, Eviction guard, Open item 3]: pf_requests = distinct valid
 * predictions = pf_resident + pf_filled + pf_dropped_guard + pf_no_victim. */
typedef struct {
  uint64_t calls, lookups, hits, misses, fetched, overflow_routes, evictions, invalid_routes;
  uint64_t pf_requests, pf_invalid, pf_resident, pf_filled, pf_dropped_guard, pf_no_victim,
           pf_evictions, status_bits;
} moe_stats;

/* Device pointers into the cache's state, for inspection and tests.  Sizes:
 * map, decode_freq, demand_freq, last_demand: n_layers*n_experts;
 * slot_key, stamp, pinned: n_pools*n_slots; clock: n_pools; stats: n_layers;
 * plans and groups as described above. */
typedef struct {
  const int32_t* map;            /* key -> slot in its pool, -1 = not resident */
  const int32_t* slot_key;       /* slot -> key, -1 = empty */
  const uint64_t* stamp;         /* slot -> clock of last touch, 0 = empty */
  const uint8_t* pinned;
  const uint64_t* clock;         /* per pool, starts at 1, +1 per admission */
  const uint32_t* decode_freq;   /* valid routes per key */
  const uint32_t* demand_freq;   /* admissions that demanded the key */
  const uint64_t* last_demand;   /* clock of the last demand, 0 = never */
  const moe_stats* stats;
  const int32_t* plan_demand;
  const int32_t* plan_prefetch;
  const int32_t* groups;
  int n_pools;
} moe_views;

/* Create a cache; every slot starts empty, every clock at 1.  Validates the
 * descriptor (MOE_ERR_CONFIG), translates each host blob pointer to a device
 * address (cudaHostGetDevicePointer; MOE_ERR_CONFIG if a pointer is not
 * pinned, mapped memory), allocates state and scratch (MOE_ERR_CUDA on
 * failure) and creates the events.  Uses the current CUDA device.  It also
 * raises the library kernels' shared-memory limits to what this cache's shapes
 * need (never lowers them, so caches of other shapes stay valid); creates on
 * several threads take turns for that part.  Thread-safe. */
MOE_API int moe_cache_create(const moe_cache_desc* desc, moe_cache** out);

/* Free all cache-owned memory and events after synchronising the device. */
MOE_API int moe_cache_destroy(moe_cache* c);

/* Set-up, synchronous: install n distinct, valid, non-resident experts of
 * `layer` into the lowest empty slots of its pool, stamped with the pool's
 * current clock, and copy their blobs into the slots.  No statistics change.
 * MOE_ERR_INVALID_ARG for a bad / duplicate / resident id, MOE_ERR_CAPACITY
 * when the pool has no empty slot left. */
MOE_API int moe_cache_prefill(moe_cache* c, int layer, const int32_t* h_ids, int n, void* stream);

/* Pin (never evict) or unpin slot `slot` of the pool of `layer` [P4
 * Consumer: pinned slots are never chosen].  Enqueued on `stream`. */
MOE_API int moe_cache_pin(moe_cache* c, int layer, int slot, int pinned, void* stream);

/* Admission of one layer's step, "lru_ensure" [P3 Problem, Solution; P2 What
 * we changed; P1 sections 4-5].  One CTA on `stream`:
 *   clock += 1 for the layer's pool; ids outside [0, E) -> -1 (invalid);
 *   distinct valid ids D (ascending); decode_freq += routes per id;
 *   demand_freq += 1, last_demand = clock for each id of D;
 *   hits: stamp = clock; misses M = D minus hits, ascending;
 *   admitted A = the first min(fetch_cap, |M|) of M (all of M if fetch_cap < 0);
 *   victims: unpinned slots with stamp < clock (never a slot touched by this
 *     admission), ascending (stamp, slot) -- empty slots (stamp 0) first,
 *     lowest index first; the i-th of A takes the i-th victim, evicting its
 *     old expert; the plan lists (slot, layer, expert) in that order;
 *   d_slot_ids[r] = slot of ids[r] if resident now, else -1.
 * d_slot_ids may equal d_ids (in-place rewrite).  n_routes may be 0.
 * MOE_ERR_CAPACITY if n_routes > max_routes. */
MOE_API int moe_admit(moe_cache* c, int layer, const int32_t* d_ids, int32_t* d_slot_ids, int n_routes,
              int fetch_cap, void* stream);

/* Look-ahead prefetch for `layer` [P4 Consumer, Eviction guard].  One CTA on
 * `stream`; the clock does not advance.  Ids outside [0, E) are ignored
 * (pf_invalid), the rest deduplicated (pf_requests); resident ones are left
 * alone (pf_resident).  Each other id, ascending, looks at the first
 * evictable slot (unpinned, stamp < clock, ascending (stamp, slot)); if that
 * slot holds an expert with demand_freq >= 2 and
 *     4 * score(resident) > 5 * score(predicted) + 4 * (4 << 8),
 *     score(key) = (min(demand_freq, 2^24-1) << 8) | recency,
 *     recency = 255 - min(255, clock - last_demand), 0 if never demanded,
 * the prediction is dropped (pf_dropped_guard), never forced into another
 * slot; otherwise the slot is (evicted and) filled, stamped with the current
 * clock, and listed in the prefetch plan.  No evictable slot: pf_no_victim.
 * MOE_ERR_STATE if the cache was created with max_pred = 0. */
MOE_API int moe_prefetch(moe_cache* c, int layer, const int32_t* d_pred, int n, void* stream);

/* The look-ahead producer [llama.cpp fork PR #126 "cuda : MoE look-ahead
 * expert prefetch (PR-A consumer) + LFRU eviction guard", sections What and
 * "Open for PR-P1 (producer)"]: the predicted ids of layer L+1, computed while
 * layer L runs, for moe_prefetch or moe_decode_layer's d_pred.  The pages
 * leave the predictor open; this one applies layer L+1's router to the hidden
 * state layer L has.  For each row b of d_x (bf16 [n_rows][hidden]):
 *   z[e] = sum_h router[e][h] * x[b][h]   (d_router bf16 [n_experts][hidden],
 *          row e = expert e's router weights; exact products, fp32 sums),
 * and d_pred[b*k_pred + r], r = 0..k_pred-1, receives the expert of rank r by
 * z, largest first, a tie going to the lower id, a NaN logit ranking below
 * -inf.  d_pred int32 [n_rows * k_pred] may then be passed whole as
 * (d_pred, n_rows * k_pred): the prefetch admission ignores repeats.
 * Shapes: hidden a multiple of 1024 up to 4096, 1 <= k_pred <= min(32,
 * n_experts), n_rows <= max_rows (else MOE_ERR_UNSUPPORTED / _CAPACITY);
 * d_x and d_router 16-byte aligned, d_pred 4-byte (else MOE_ERR_INVALID_ARG).  One launch on
 * `stream` that waits on nothing; graph-capturable.  Calls on different
 * streams must not overlap (one logit buffer per cache). */
MOE_API int moe_lookahead_predict(moe_cache* c, const void* d_x, const void* d_router, int n_rows,
                                  int k_pred, int32_t* d_pred, void* stream);

/* The gather, "copy_missing" [P2 Problem, What we changed]: copy every entry
 * of the demand or prefetch plan from its pinned host blob into its slot.  The
 * grid reads the device-side count, so the call needs no host sync and its
 * launch does not depend on the miss count.  MOE_ERR_STATE if the cache has no
 * slot storage. */
MOE_API int moe_gather_missing(moe_cache* c, int which, void* stream);

/* Undo the bookings of a plan whose copy failed or was abandoned: each of its
 * slots that still holds the planned expert becomes empty and the expert
 * non-resident.  Statistics are not rewound. */
MOE_API int moe_rollback_plan(moe_cache* c, int which, void* stream);

/* The routed expert FFNs over the slots plus the shared expert and the
 * weighted combine [P2 Problem, What we changed; P1 section 5; P3 Tests]:
 *   out[b] = bf16( sum_j w[b,j] * FFN_slot[b,j](x[b]) + shared(x[b]) ).
 * d_x bf16 [n_rows][H]; d_slot_ids int32 [n_rows][k] (-1 = skip);
 * d_w float32 [n_rows][k]; d_shared_blob / d_shared_gate: device shared
 * expert (NULL = none; requires shared_inter > 0); d_out bf16 [n_rows][H]
 * (must not alias d_x).  MOE_ERR_CAPACITY if n_rows > max_rows or
 * n_rows*k > max_routes. */
MOE_API int moe_routed_experts(moe_cache* c, int layer, const void* d_x, const int32_t* d_slot_ids,
                       const float* d_w, int n_rows, int k, const void* d_shared_blob,
                       const void* d_shared_gate, void* d_out, void* stream);

/* One whole offloaded decode layer [P2 What we changed, order inside one layer]:
 *   compute: admit -> [prefetch layer+1] -> record(ready) -> shared expert + gate
 *            -> wait(done) -> routed FFNs + combine
 *   side:    wait(ready) -> gather (demand) -> record(done) -> gather (prefetch)
 * With flags & MOE_OVERLAP the gather runs on side_stream and the two events
 * fork and join it (capturable: both edges are recorded into the graph).
 * Without it everything runs on compute_stream in the same order (serial
 * mode, also the mode to profile with ncu).  d_slot_ids int32 [n_rows*k]
 * receives the rewritten ids (may equal d_ids).  d_pred/n_pred (NULL/0 = none)
 * are predicted ids of layer+1; their gather is queued on the side stream
 * after this layer's demand gather and is joined by layer+1's own wait.  Must
 * not be mixed with moe_gather_missing(MOE_PLAN_PREFETCH) calls of its own.
 *
 * With flags & MOE_FUSED, for decode-sized steps (at most 16 rows and 64
 * routes, the streaming kernel's shapes, a shared expert of the routed
 * experts' size, at most 4096 experts per layer), the layer is ONE
 * cooperative launch on compute_stream:
 *   - CTA 0 runs the admission (the same algorithm and results as moe_admit,
 *     writing d_slot_ids, the plan and the stats) and then the prefetch
 *     admission of layer+1;
 *   - the other CTAs read the map for the step's experts themselves (a hit
 *     cannot be evicted by its own admission; an installed miss is marked
 *     pending in the map until this launch has copied it in), stream the
 *     resident experts at once and compute the shared and routed experts;
 *   - an uncapped step's misses are copied from pinned host memory into
 *     staging entries (up to max_routes experts within 64 MB, allocated at
 *     create) as soon as they are known and computed from there; each piece
 *     also goes into the expert's slot once the admission has chosen it, and
 *     the pending marks are cleared at the end of the launch; with a fetch cap
 *     they wait for the admission's slots and are copied there directly; the
 *     prefetch plan's experts are copied into their slots in the same launch.
 * The overlap of [P2] (the gather beside the shared expert) happens inside
 * that launch instead of on two streams; side_stream is not used.  If the
 * shapes do not fit, the admission and prefetch run as their own launches
 * followed by one launch for the rest; other shapes fall back to the mode the
 * remaining flags select.  Outputs, slot ids, plans, stats and cache state equal
 * the four-launch path's bit for bit. */
MOE_API int moe_decode_layer(moe_cache* c, int layer, const void* d_x, const int32_t* d_ids,
                     const float* d_w, int32_t* d_slot_ids, int n_rows, int k, int fetch_cap,
                     const int32_t* d_pred, int n_pred, const void* d_shared_blob,
                     const void* d_shared_gate, void* d_out, void* compute_stream,
                     void* side_stream, unsigned flags);

/* ---------------------------------------------------------- hybrid CPU executor
 * [P1 section 4 "How decode works after this PR", section 5 "How routes are
 * split"]: the routes a capped admission leaves at -1 (fetch-cap overflow or
 * no evictable slot) are computed on the host from the pinned host blobs,
 * while the GPU computes the routes that got a slot; the partial outputs are
 * added.  For route r = b*k + j with slot -1 and a valid expert id e:
 *   h = silu(W_g x_b) * (W_u x_b),  cpu[b] = sum_j w[b,j] * (W_d h)   (fp32,
 *   j ascending; rows without such a route give 0),
 * and with MOE_HYBRID the layer output becomes
 *   out[b] = bf16( float(gpu_out[b]) + cpu[b] ),
 * gpu_out being the output moe_decode_layer computes without the flag.
 *
 * moe_hybrid_start: start the cache's executor, a pool of n_threads (1..256)
 * host threads, and its mailbox (mapped pinned memory, max_rows*H inputs and
 * outputs).  The host blob pointers given at create are read by these
 * threads; they must be host-readable (pinned host memory is).  MOE_ERR_STATE
 * if one is running or the cache has no expert shapes / host blobs.
 * moe_hybrid_stop: synchronise the device and stop the pool (also done by
 * moe_cache_destroy).
 *
 * With flags & MOE_HYBRID, moe_decode_layer enqueues, right after the
 * admission, a kernel that posts the step (ids, slot ids, weights, x) to the
 * mailbox with a system-scope release of a job number; the pool takes the
 * job, computes the CPU partial and publishes the number back; after the GPU
 * experts and the combine a second kernel waits for it (bounded: after 1 s it
 * sets MOE_STATUS_TIMEOUT and leaves the GPU partial) and adds the partial.
 * Every step posts a job, even one without -1 routes, so a captured graph
 * does not depend on the hit pattern; both kernels are capturable.  With
 * MOE_FUSED the admission runs as its own launch, followed by the post and
 * the one-launch gather + experts kernel.  MOE_ERR_STATE if no executor runs.
 * A graph captured with MOE_HYBRID holds the executor's mailbox and counter
 * addresses: replay it only while that executor runs (not after
 * moe_hybrid_stop, a later moe_hybrid_start or moe_cache_destroy). */
MOE_API int moe_hybrid_start(moe_cache* c, int n_threads);
MOE_API int moe_hybrid_stop(moe_cache* c);
/* jobs done, CPU routes computed, nanoseconds the coordinator spent on jobs,
 * and on the jobs that had at least one -1 route */
MOE_API int moe_hybrid_counters(moe_cache* c, uint64_t h_out[4]);
/* Test hook: while paused != 0 the executor leaves posted jobs unanswered, so
 * the GPU's bounded wait runs out (MOE_STATUS_TIMEOUT, GPU partial kept);
 * resuming answers the newest posted job. */
MOE_API int moe_hybrid_pause(moe_cache* c, int paused);

/* Test hook, host only (no GPU, no cache): the executor's job protocol over a
 * mailbox in plain host memory.  n_jobs random steps of up to max_rows rows
 * (some ids invalid, about half the routes at -1, a pause every 97th job) are
 * posted the way the GPU posts them, and each answer is compared bit for bit
 * with moe_cpu_experts; *h_mismatches receives the number of differing jobs
 * (a job answered while paused counts as one).  MOE_ERR_STATE if a job goes
 * unanswered for 10 s. */
MOE_API int moe_hybrid_selftest(int wfmt, int hidden, int inter, const void* const* h_blobs,
                                int n_experts, int max_rows, int k, int n_threads, int n_jobs,
                                unsigned seed, long long* h_mismatches);

/* The CPU partial above as a plain host function (no GPU, no cache): h_blobs
 * [n_experts] host blob addresses of one layer; h_x bf16 [n_rows][H]; h_ids,
 * h_slot_ids int32 and h_w float [n_rows][k]; h_out float [n_rows][H].  Uses
 * n_threads host threads (1..256); the result does not depend on n_threads. */
MOE_API int moe_cpu_experts(int wfmt, int hidden, int inter, const void* const* h_blobs,
                            int n_experts, const uint16_t* h_x, const int32_t* h_ids,
                            const int32_t* h_slot_ids, const float* h_w, int n_rows, int k,
                            int n_threads, float* h_out);

/* Test hook, host only: the operations moe_decode_layer enqueues for a layer
 * plan, in order, as "c:op" (compute stream) / "s:op" (side stream) tokens
 * separated by spaces, written to h_out (cap bytes).  The ops are admit, post,
 * prefetch, gather_demand, gather_prefetch, shared, routed, add_cpu,
 * layer_admit, layer_stream, record_ready, wait_ready, record_done and
 * wait_done.  The fork/join events are ready and done.  fail_at >= 0 makes the
 * fail_at-th operation fail with MOE_ERR_CUDA, and the call returns the code
 * the layer would.  MOE_ERR_CAPACITY if the trace does not fit. */
MOE_API int moe_schedule_trace(int one_launch, int fused, int overlap, int pf, int shared,
                               int hybrid, int fail_at, char* h_out, int cap);

/* Host only, no device work: the operations moe_decode_layer would enqueue on
 * cache c for a step of n_rows x k routes, with (shared != 0) or without a
 * shared expert, with (pf != 0) or without predictions, under `flags` -- the
 * same tokens as moe_schedule_trace ("c:layer_admit" alone is the one-launch
 * layer).  Lets a caller (and the tests) confirm which path a shape takes.
 * MOE_ERR_CAPACITY if the trace does not fit in cap bytes. */
MOE_API int moe_decode_layer_plan(moe_cache* c, int n_rows, int k, int shared, int pf,
                                  unsigned flags, char* h_out, int cap);

/* Copy one layer's counters to the host.  Synchronises the device. */
MOE_API int moe_read_stats(moe_cache* c, int layer, moe_stats* h_out);

/* Device pointers into the state (valid until moe_cache_destroy). */
MOE_API int moe_device_views(moe_cache* c, moe_views* out);

/* Which kernels run the routed experts of wide steps (the grouped path: more
 * than 16 rows or 64 routes; the route groups hold each distinct expert's
 * routes).  NVFP4 experts with H and I multiples of 128 have two kernel
 * families: the tensor cores (tcgen05 kind::f16 MMAs of 128 weight rows x up
 * to 32 routes, fp32 accumulators in tensor memory; h is rounded to f16 with a
 * per-route power-of-two scale before the down GEMM) and the CUDA cores (fp32
 * h).  A tensor-core MMA costs the same whatever its route count, so:
 *   MOE_WIDE_AUTO (the default): groups of at least 4 routes on the tensor
 *     cores, smaller groups on the CUDA cores -- the tensor cores only where
 *     the group is a real dense contraction;
 *   MOE_WIDE_CUDA_CORES: every group on the CUDA cores;
 *   MOE_WIDE_TENSOR_CORES: every group on the tensor cores.
 * Other shapes and formats always use the CUDA-core kernels.  Host only;
 * affects calls enqueued afterwards.  MOE_ERR_INVALID_ARG for another mode. */
enum { MOE_WIDE_AUTO = 0, MOE_WIDE_CUDA_CORES = 1, MOE_WIDE_TENSOR_CORES = 2 };
MOE_API int moe_cache_set_wide_path(moe_cache* c, int mode);

/* Test hook: make the next moe_gather_missing call fail with MOE_ERR_INJECTED
 * before it enqueues anything (the plan's bookings stay; the caller is
 * expected to call moe_rollback_plan).  n = 0 clears the request. */
MOE_API int moe_cache_fail_next_gather(moe_cache* c, int n);

/* ---------------------------------------------------------------- no allocation
 * The pages have no counterpart of this call.  It runs the routed expert FFNs
 * and the weighted combine of moe_routed_experts (without the shared expert)
 * over a slot pool the caller owns, and it allocates nothing: no cache handle,
 * no cudaMalloc / cudaFree, no allocator of any library (torch's included).
 *
 * Who needs it: a caller that cannot allocate device memory where it runs the
 * experts.  Examples are a serving engine that reserved its whole memory
 * budget (slot pool, KV cache) at start-up and must not allocate during
 * decode, and code that keeps experts resident by itself and so has no
 * moe_cache whose scratch it could borrow.  Creating a cache allocates state
 * and scratch, and a cudaFree synchronises the device, so neither fits there.
 *
 * Scratch: a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES (1 MiB).
 * Bytes [0, 256) hold the kernel's grid-barrier counter and bytes [256, 1 MiB)
 * hold the fp32 intermediate h [n_rows*k][inter].  A request needs
 * 256 + 4*n_rows*k*inter bytes; a larger one returns MOE_ERR_SCRATCH before
 * anything is enqueued.  Each call clears the counter with a cudaMemsetAsync
 * on `stream` before the kernel; h needs no clearing (every element read is
 * written first in the same launch).
 *
 * Set-up: the first call on each device (that device current) looks up the
 * array's address with cudaGetSymbolAddress and sets the kernel's shared
 * memory limit; a failure returns MOE_ERR_CUDA.  If the first call is the
 * one doing this set-up, make it before any stream capture.  The address is
 * kept per device ordinal for the life of the process and belongs to that
 * device's primary CUDA context: after a cudaDeviceReset of the device it is
 * stale (the context and its array are gone), so do not call this entry point
 * on a device that was reset after its first call.
 *
 * Races: there is one scratch array per device, so calls whose executions
 * overlap on a device (different streams, or threads without ordering) race
 * on it.  Order them on one stream or with events.
 *
 * Arguments: wfmt / hidden / inter as in moe_cache_desc; d_slots the pool
 * base (256-byte aligned), slot s at d_slots + s*slot_stride (multiple of 256,
 * at least the blob size), n_slots > 0; d_x bf16 [n_rows][hidden], 16-byte
 * aligned; d_slot_ids int32 [n_rows][k] (outside [0, n_slots) = skip);
 * d_w float32 [n_rows][k]; d_out bf16 [n_rows][hidden] (not aliasing d_x):
 *   out[b] = bf16( sum_j w[b,j] * FFN_slot[b,j](x[b]) ).
 * d_status: device word that receives MOE_STATUS_TIMEOUT if a bounded wait in
 * the kernel gives up (NULL = not reported).  Only shapes the streaming
 * kernel handles are accepted (among its conditions: hidden % 1024 == 0,
 * inter % 512 == 0, n_rows <= 16, n_rows*k <= 64); others return
 * MOE_ERR_UNSUPPORTED.  Enqueues work only. */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
MOE_API int moe_routed_experts_noalloc(int wfmt, int hidden, int inter, const void* d_slots,
                                       size_t slot_stride, int n_slots, const void* d_x,
                                       const int32_t* d_slot_ids, const float* d_w, int n_rows,
                                       int k, void* d_out, unsigned long long* d_status,
                                       void* stream);

/* Text of an error code; last CUDA error text seen by this thread. */
MOE_API const char* moe_strerror(int err);
MOE_API const char* moe_last_cuda_error(void);
MOE_API int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_CACHE_H */
