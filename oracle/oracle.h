/*
 * oracle.h -- C interface of the CPU oracle for the offloaded-MoE slot cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This header, oracle.cpp and the Python wrapper
 * beside them are the slow, obviously-correct model that the CUDA library is
 * checked against.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark may load it; the product library never does, and the two
 * share no code, header, table or helper.
 *
 * Everything here is single-threaded and follows the pages step by step:
 *  - slot-cache admission ("lru_ensure"): FreeToken PR #680 "fix(moe): admit
 *    a wide offloaded decode step's experts 128 at a time", sections Problem,
 *    Solution and Tests; FreeToken issue #753 "[Perf] Offloaded decode:
 *    overlap the expert-miss gather ...", section What we changed;
 *  - capped fetch with -1 overflow routes: FreeToken PR #491 "refactor(moe):
 *    extract hybrid decode orchestration", sections 4 and 5;
 *  - look-ahead prefetch and the LFRU eviction guard: llama.cpp fork PR #126
 *    "cuda : MoE look-ahead expert prefetch (PR-A consumer) + LFRU eviction
 *    guard", sections Consumer and Eviction guard;
 *  - the layer math (routed SiLU FFN experts, sigmoid-gated shared expert,
 *    weighted combine): FreeToken issue #753, sections Problem and What we
 *    changed.
 *
 * All integers are host-endian; ids and slots are int32, clocks and stamps
 * uint64.  Functions return 0 on success and a negative value on a bad
 * argument; they never abort.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ocache ocache;

/* Statistics, one record per layer; field order is fixed (index constants). */
enum {
  OST_CALLS = 0, OST_LOOKUPS, OST_HITS, OST_MISSES, OST_FETCHED, OST_OVERFLOW_ROUTES,
  OST_EVICTIONS, OST_INVALID_ROUTES, OST_PF_REQUESTS, OST_PF_INVALID, OST_PF_RESIDENT,
  OST_PF_FILLED, OST_PF_DROPPED_GUARD, OST_PF_NO_VICTIM, OST_PF_EVICTIONS, OST_STATUS,
  OST_N
};
/* status bits */
enum { OSTATUS_INVALID_ID = 1, OSTATUS_CAPACITY = 2 };

/* per_layer_pools = 0: one pool of n_slots shared by all layers;
 * per_layer_pools = 1: n_layers pools of n_slots each. */
ocache* oc_create(int n_layers, int n_experts, int n_slots, int per_layer_pools);
void    oc_destroy(ocache* c);

/* Install distinct, valid, non-resident ids of `layer` into the lowest empty
 * slots of its pool, stamped with the pool's current clock.  No statistics. */
int oc_prefill(ocache* c, int layer, const int32_t* ids, int n);
int oc_pin(ocache* c, int layer, int slot, int pinned);

/* One admission.  out_slots[R]: slot id per route, -1 for overflow/invalid.
 * plan: [count, (slot, layer, expert) x count]; capacity 1 + 3*R ints.
 * groups: [n_groups, slot[g] .. , start[g] .. (n_groups+1 entries), route list]
 *   capacity 2 + 3*R ints (see oc_admit in oracle.cpp for the exact layout).
 * split_width > 0 processes the step's distinct experts in queries of that
 * width (the self-check path); widths_out (capacity >= R+1) receives
 * [n_queries, width...]. */
int oc_admit(ocache* c, int layer, const int32_t* ids, int n_routes, int fetch_cap,
             int split_width, int32_t* out_slots, int32_t* plan, int32_t* groups,
             int32_t* widths_out);

/* Look-ahead prefetch for `layer`.  plan as above, capacity 1 + 3*n. */
int oc_prefetch(ocache* c, int layer, const int32_t* pred, int n, int32_t* plan);

/* Undo the bookings of a plan whose copy failed: the filled slots become
 * empty and their keys non-resident.  Statistics are not rewound. */
int oc_rollback(ocache* c, const int32_t* plan);

int oc_stats(const ocache* c, int layer, uint64_t* out /* OST_N */);
int oc_n_pools(const ocache* c);
/* Copies of the whole state; any pointer may be NULL. Sizes: map, decode_freq,
 * demand_freq, last_demand: n_layers*n_experts; slot_key, stamp, pinned:
 * n_pools*n_slots; clock: n_pools. */
int oc_state(const ocache* c, int32_t* map, int32_t* slot_key, uint64_t* stamp,
             uint8_t* pinned, uint64_t* clock, uint32_t* decode_freq,
             uint32_t* demand_freq, uint64_t* last_demand);
/* LRU list of a pool, head first (ordered by (stamp, slot)). */
int oc_lru_order(const ocache* c, int pool, int32_t* out /* n_slots */);

/* ---- expert math, fp64 ---- */
enum { OFMT_BF16 = 0, OFMT_NVFP4 = 1, OFMT_MXFP4 = 2, OFMT_Q4_0 = 3 };

double om_e2m1(int code4);
double om_e4m3(int byte);
double om_e8m0(int byte);
double om_f16(uint16_t bits);
double om_bf16(uint16_t bits);
/* Bytes of one expert blob in the fused six-bank layout. */
uint64_t om_blob_bytes(int fmt, int hidden, int inter);
/* Dequantise one matrix of a blob: which = 0 gate [I,H], 1 up [I,H], 2 down [H,I]. */
int om_dequant(int fmt, const uint8_t* blob, int hidden, int inter, int which, double* out);
/* y[H] = W_d (silu(W_g x) * (W_u x)) in fp64, x given as bf16 bits. */
int om_expert_ffn(int fmt, const uint8_t* blob, int hidden, int inter, const uint16_t* x,
                  double* y);
/* One layer: out[b,:] = sum_j [mask] w[b,j] * FFN(expert ids[b,j])(x_b)
 *                       + sigmoid(x_b . gate_w) * FFN_shared(x_b)  (if shared_blob)
 * blobs[e] is expert e's blob of this layer.  mask (may be NULL = all) selects
 * which routes are summed; ids outside [0, n_experts) contribute nothing. */
int om_layer(int fmt, const uint8_t* const* blobs, int n_experts, int hidden, int inter,
             const uint16_t* x, const int32_t* ids, const float* w, const uint8_t* mask,
             int n_rows, int k, const uint8_t* shared_blob, int shared_inter,
             const uint16_t* shared_gate_w, double* out);

/* The look-ahead producer's prediction [llama.cpp fork PR #126 "cuda : MoE
 * look-ahead expert prefetch (PR-A consumer) + LFRU eviction guard", sections
 * What and "Open for PR-P1 (producer)": the predicted ids of layer L+1, made
 * while layer L runs].  The pages leave the predictor open; the reading here
 * applies layer L+1's router to layer L's hidden state.  For each row b:
 * z[e] = sum_h router[e][h] * x[b][h] in fp64 (both operands bf16 bits, row e
 * of router = expert e), stored in z_out[b*n_experts + e] when z_out is not
 * NULL; pred[b*k + r] = the expert of rank r when the experts are ordered by z
 * descending, then by id ascending, a NaN z ranking after every number.
 * 1 <= k <= n_experts. */
int om_lookahead_predict(const uint16_t* x, const uint16_t* router, int n_rows, int n_experts,
                         int hidden, int k, int32_t* pred, double* z_out);

#ifdef __cplusplus
}
#endif
#endif
