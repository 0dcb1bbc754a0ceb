// oracle.cpp -- plain, single-threaded CPU oracle of the offloaded-MoE slot
// cache and of the layer math.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg, never by the product library.  It shares no
// code with the CUDA path.  Speed is not a goal; every step is written so it
// can be checked against the pages by eye.
//
// Pages followed (titles and sections):
//  [P1] FreeToken PR #491 "refactor(moe): extract hybrid decode orchestration"
//  [P2] FreeToken issue #753 "[Perf] Offloaded decode: overlap the expert-miss
//       gather with the same layer's shared expert, event-ordered inside the
//       CUDA graph"
//  [P3] FreeToken PR #680 "fix(moe): admit a wide offloaded decode step's
//       experts 128 at a time"
//  [P4] llama.cpp fork PR #126 "cuda : MoE look-ahead expert prefetch (PR-A
//       consumer) + LFRU eviction guard"
//
// Readings taken where the pages are silent (each is listed with its reason in
// the design notes): one recency stamp per admission call per pool; victims
// are the eligible slots in ascending (stamp, slot) order, empty slots having
// stamp 0; misses are admitted in ascending expert id and paired with victims
// in that order; the fetch cap admits the lowest expert ids; a capacity
// shortfall behaves like a cap and raises a status bit; the LFRU recency byte
// is 255 - min(255, clock - last_demand) (0 if never demanded) and the guard's
// 1.25x is evaluated in integers as 4*R > 5*P + 4*(4<<8).

#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Cache state
// ---------------------------------------------------------------------------

// One pool of slots.  The LRU order is kept as an explicit doubly linked list
// ordered by (stamp, slot): empty slots (stamp 0) at the head in slot order,
// the most recently touched slots at the tail.
struct Pool {
  uint64_t clock = 1;                 // advanced once per admission of the pool
  std::vector<int32_t> key;           // slot -> layer*E + expert, -1 when empty
  std::vector<uint64_t> stamp;        // slot -> clock of its last touch, 0 when empty
  std::vector<uint8_t> pinned;        // pinned slots are never victims
  std::vector<int> prev, next;        // the list
  int head = -1, tail = -1;

  void init(int S) {
    key.assign(S, -1);
    stamp.assign(S, 0);
    pinned.assign(S, 0);
    prev.assign(S, -1);
    next.assign(S, -1);
    for (int s = 0; s < S; ++s) {
      prev[s] = s - 1;
      next[s] = (s + 1 < S) ? s + 1 : -1;
    }
    head = S > 0 ? 0 : -1;
    tail = S > 0 ? S - 1 : -1;
  }
  // (stamp, slot) order
  bool before(int a, int b) const {
    return stamp[a] < stamp[b] || (stamp[a] == stamp[b] && a < b);
  }
  void unlink(int s) {
    if (prev[s] >= 0) next[prev[s]] = next[s]; else head = next[s];
    if (next[s] >= 0) prev[next[s]] = prev[s]; else tail = prev[s];
    prev[s] = next[s] = -1;
  }
  // Insert s after the last node that precedes it in (stamp, slot) order.
  void insert_sorted(int s) {
    int p = tail;
    while (p >= 0 && before(s, p)) p = prev[p];
    if (p < 0) {  // new head
      prev[s] = -1;
      next[s] = head;
      if (head >= 0) prev[head] = s; else tail = s;
      head = s;
    } else {
      prev[s] = p;
      next[s] = next[p];
      if (next[p] >= 0) prev[next[p]] = s; else tail = s;
      next[p] = s;
    }
  }
  void restamp(int s, uint64_t st) {
    unlink(s);
    stamp[s] = st;
    insert_sorted(s);
  }
  // Walk the list from the head and return up to `want` slots that may be
  // evicted now: not pinned and not touched by the current admission.
  std::vector<int> victims(size_t want) const {
    std::vector<int> v;
    for (int s = head; s >= 0 && v.size() < want; s = next[s]) {
      if (pinned[s]) continue;
      if (stamp[s] >= clock) continue;  // touched in this admission (stamp == clock)
      v.push_back(s);
    }
    return v;
  }
};

}  // namespace

struct ocache {
  int L = 0, E = 0, S = 0;
  bool per_layer = false;
  std::vector<Pool> pools;
  std::vector<int32_t> map;            // key -> slot in its pool, -1 when not resident
  std::vector<uint32_t> decode_freq;   // every valid route        [P3 Solution]
  std::vector<uint32_t> demand_freq;   // distinct demand accesses [P4 Eviction guard]
  std::vector<uint64_t> last_demand;   // clock of the last demand access, 0 = never
  std::vector<uint64_t> stats;         // L * OST_N

  int pool_of(int layer) const { return per_layer ? layer : 0; }
  int32_t key_of(int layer, int e) const { return layer * E + e; }
  uint64_t* st(int layer) { return &stats[(size_t)layer * OST_N]; }
};

namespace {

void plan_init(int32_t* plan) {
  if (plan) plan[0] = 0;
}
void plan_push(int32_t* plan, int slot, int layer, int e) {
  if (!plan) return;
  int32_t n = plan[0];
  plan[1 + 3 * n + 0] = slot;
  plan[1 + 3 * n + 1] = layer;
  plan[1 + 3 * n + 2] = e;
  plan[0] = n + 1;
}

// LFRU score [P4 Eviction guard]: demand frequency in the high bits, a
// recency byte that saturates in the low byte.
uint64_t lfru_score(const ocache* c, int32_t key, uint64_t clock) {
  uint64_t f = c->demand_freq[key];
  if (f > 0xFFFFFFull) f = 0xFFFFFFull;
  uint64_t rec = 0;
  if (c->last_demand[key] != 0) {
    uint64_t age = clock - c->last_demand[key];
    rec = 255 - (age < 255 ? age : 255);
  }
  return (f << 8) | rec;
}

}  // namespace

extern "C" {

ocache* oc_create(int n_layers, int n_experts, int n_slots, int per_layer_pools) {
  if (n_layers <= 0 || n_experts <= 0 || n_slots < 0) return nullptr;
  ocache* c = new ocache;
  c->L = n_layers;
  c->E = n_experts;
  c->S = n_slots;
  c->per_layer = per_layer_pools != 0;
  c->pools.resize(c->per_layer ? n_layers : 1);
  for (auto& p : c->pools) p.init(n_slots);
  size_t K = (size_t)n_layers * n_experts;
  c->map.assign(K, -1);
  c->decode_freq.assign(K, 0);
  c->demand_freq.assign(K, 0);
  c->last_demand.assign(K, 0);
  c->stats.assign((size_t)n_layers * OST_N, 0);
  return c;
}

void oc_destroy(ocache* c) { delete c; }

int oc_n_pools(const ocache* c) { return c ? (int)c->pools.size() : -1; }

int oc_prefill(ocache* c, int layer, const int32_t* ids, int n) {
  if (!c || layer < 0 || layer >= c->L || n < 0 || (n > 0 && !ids)) return -1;
  Pool& P = c->pools[c->pool_of(layer)];
  for (int i = 0; i < n; ++i) {
    int e = ids[i];
    if (e < 0 || e >= c->E) return -2;
    int32_t key = c->key_of(layer, e);
    if (c->map[key] >= 0) return -3;  // duplicate or already resident
    int slot = -1;
    for (int s = 0; s < c->S; ++s)
      if (P.key[s] < 0) { slot = s; break; }
    if (slot < 0) return -4;  // no empty slot
    P.key[slot] = key;
    c->map[key] = slot;
    P.restamp(slot, P.clock);
  }
  return 0;
}

int oc_pin(ocache* c, int layer, int slot, int pinned) {
  if (!c || layer < 0 || layer >= c->L || slot < 0 || slot >= c->S) return -1;
  c->pools[c->pool_of(layer)].pinned[slot] = pinned ? 1 : 0;
  return 0;
}

// One admission ("lru_ensure") of one layer's decode step.
//
// [P3 Problem/Solution]: the step's ids are deduplicated to a sorted list of
// distinct experts, looked up in the expert->slot map, hits refresh recency,
// misses get LRU victims and a copy each; the statistics count the step once
// (distinct experts as lookups, misses, one call) while decode_freq counts
// every route; ids are rewritten in place to slot ids.
// [P2 What we changed]: the admission writes the miss plan that the gather
// reads.  [P1 sections 4-5]: with a fetch cap only some misses are admitted
// and the other routes become -1.
int oc_admit(ocache* c, int layer, const int32_t* ids, int R, int cap, int split_width,
             int32_t* out, int32_t* plan, int32_t* groups, int32_t* widths) {
  if (!c || layer < 0 || layer >= c->L || R < 0 || (R > 0 && (!ids || !out))) return -1;
  Pool& P = c->pools[c->pool_of(layer)];
  uint64_t* st = c->st(layer);
  const int E = c->E;

  // Step 1: one new recency stamp for the whole admission.
  P.clock += 1;
  const uint64_t clk = P.clock;
  st[OST_CALLS] += 1;
  plan_init(plan);

  // Step 2: routes whose id is outside [0, E) take no part; they become -1.
  std::vector<char> valid(R, 0);
  for (int r = 0; r < R; ++r) {
    valid[r] = (ids[r] >= 0 && ids[r] < E);
    if (!valid[r]) {
      st[OST_INVALID_ROUTES] += 1;
      st[OST_STATUS] |= OSTATUS_INVALID_ID;
    }
  }

  // Step 3: sorted distinct experts; per-route and per-expert counters.
  std::vector<int> D;
  for (int r = 0; r < R; ++r)
    if (valid[r]) D.push_back(ids[r]);
  std::sort(D.begin(), D.end());
  D.erase(std::unique(D.begin(), D.end()), D.end());
  for (int r = 0; r < R; ++r)
    if (valid[r]) c->decode_freq[c->key_of(layer, ids[r])] += 1;
  st[OST_LOOKUPS] += D.size();
  for (int e : D) {
    int32_t key = c->key_of(layer, e);
    if (c->demand_freq[key] != 0xFFFFFFFFu) c->demand_freq[key] += 1;
    c->last_demand[key] = clk;
  }

  // Step 4: hits refresh their slot's recency.  All hits of the step are
  // stamped before any victim is chosen, so none of them can be evicted by
  // this admission.
  std::vector<int> M;  // misses, ascending expert id
  for (int e : D) {
    int32_t s = c->map[c->key_of(layer, e)];
    if (s >= 0) {
      P.restamp(s, clk);
      st[OST_HITS] += 1;
    } else {
      M.push_back(e);
    }
  }
  st[OST_MISSES] += M.size();

  // Step 5: the fetch cap admits the lowest expert ids first.
  size_t nA = M.size();
  if (cap >= 0 && nA > (size_t)cap) nA = (size_t)cap;

  // Step 6: victims, in (stamp, slot) order from the head of the list.
  // Single call: one walk for all admitted misses.  Split (self-check path):
  // the distinct experts are taken split_width at a time, and each query's
  // admitted misses walk the list afresh; slots filled by earlier queries now
  // carry this admission's stamp and are skipped by the walk.
  std::vector<int> qbound;  // query boundaries over D
  if (split_width > 0) {
    for (size_t q = 0; q < D.size(); q += split_width) qbound.push_back((int)q);
  } else if (!D.empty()) {
    qbound.push_back(0);
  }
  qbound.push_back((int)D.size());
  if (widths) {
    widths[0] = (int)qbound.size() - 1;
    for (size_t q = 0; q + 1 < qbound.size(); ++q) widths[1 + q] = qbound[q + 1] - qbound[q];
  }

  size_t next_miss = 0;  // index into M of the next miss to admit
  bool short_of_slots = false;
  for (size_t q = 0; q + 1 < qbound.size(); ++q) {
    const int lo = D.empty() ? 0 : D[qbound[q]];
    const int hi = D.empty() ? 0 : D[qbound[q + 1] - 1];
    // this query's admitted misses
    std::vector<int> A;
    while (next_miss < nA && M[next_miss] >= lo && M[next_miss] <= hi) A.push_back(M[next_miss++]);
    if (A.empty() || short_of_slots) continue;
    std::vector<int> V = P.victims(A.size());
    if (V.size() < A.size()) {
      // Not enough evictable slots: the highest expert ids of the rest are
      // not admitted and their routes overflow.
      A.resize(V.size());
      short_of_slots = true;
      st[OST_STATUS] |= OSTATUS_CAPACITY;
    }
    for (size_t i = 0; i < A.size(); ++i) {
      const int s = V[i];
      const int32_t key = c->key_of(layer, A[i]);
      if (P.key[s] >= 0) {
        c->map[P.key[s]] = -1;
        st[OST_EVICTIONS] += 1;
      }
      P.key[s] = key;
      c->map[key] = s;
      P.restamp(s, clk);
      plan_push(plan, s, layer, A[i]);
      st[OST_FETCHED] += 1;
    }
  }

  // Step 7: rewrite every route to its slot, or -1 when its expert did not
  // get one (overflow; the hybrid path computes those routes elsewhere).
  for (int r = 0; r < R; ++r) {
    if (!valid[r]) {
      out[r] = -1;
      continue;
    }
    int32_t s = c->map[c->key_of(layer, ids[r])];
    out[r] = s;
    if (s < 0) st[OST_OVERFLOW_ROUTES] += 1;
  }

  // Step 8: route groups for the routed GEMM: each resident distinct expert in
  // ascending id, its slot, and its routes in ascending route index.
  if (groups) {
    std::vector<int> gslot, gstart, glist;
    for (int e : D) {
      int32_t s = c->map[c->key_of(layer, e)];
      if (s < 0) continue;
      gslot.push_back(s);
      gstart.push_back((int)glist.size());
      for (int r = 0; r < R; ++r)
        if (valid[r] && ids[r] == e) glist.push_back(r);
    }
    gstart.push_back((int)glist.size());
    const int G = (int)gslot.size();
    groups[0] = G;
    for (int g = 0; g < G; ++g) groups[1 + g] = gslot[g];
    for (int g = 0; g <= G; ++g) groups[1 + G + g] = gstart[g];
    for (size_t i = 0; i < glist.size(); ++i) groups[2 + 2 * G + i] = glist[i];
  }
  return 0;
}

// Look-ahead prefetch of predicted experts for `layer` [P4 Consumer, Eviction
// guard].  Ids outside [0, E) are ignored; resident experts are left alone
// (no recency or frequency change); the clock does not advance.  Each other
// prediction, in ascending id, looks at the first evictable slot of the list.
// A resident there with at least 2 demand accesses that is clearly hotter
// than the prediction (score > 1.25 * pred + (4 << 8)) blocks it: the
// prediction is dropped, never forced into another slot.  Otherwise the slot
// is (evicted and) filled with this admission's stamp.
int oc_prefetch(ocache* c, int layer, const int32_t* pred, int n, int32_t* plan) {
  if (!c || layer < 0 || layer >= c->L || n < 0 || (n > 0 && !pred)) return -1;
  Pool& P = c->pools[c->pool_of(layer)];
  uint64_t* st = c->st(layer);
  const uint64_t clk = P.clock;
  plan_init(plan);

  std::vector<int> ids;
  for (int i = 0; i < n; ++i) {
    if (pred[i] < 0 || pred[i] >= c->E) st[OST_PF_INVALID] += 1;
    else ids.push_back(pred[i]);
  }
  std::sort(ids.begin(), ids.end());
  ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
  st[OST_PF_REQUESTS] += ids.size();

  for (int e : ids) {
    const int32_t key = c->key_of(layer, e);
    if (c->map[key] >= 0) {
      st[OST_PF_RESIDENT] += 1;
      continue;
    }
    std::vector<int> v = P.victims(1);
    if (v.empty()) {
      st[OST_PF_NO_VICTIM] += 1;
      continue;
    }
    const int s = v[0];
    const int32_t old = P.key[s];
    if (old >= 0 && c->demand_freq[old] >= 2) {
      const uint64_t R_ = lfru_score(c, old, clk);
      const uint64_t P_ = lfru_score(c, key, clk);
      if (4 * R_ > 5 * P_ + 4 * (4u << 8)) {
        st[OST_PF_DROPPED_GUARD] += 1;
        continue;
      }
    }
    if (old >= 0) {
      c->map[old] = -1;
      st[OST_PF_EVICTIONS] += 1;
    }
    P.key[s] = key;
    c->map[key] = s;
    P.restamp(s, clk);
    plan_push(plan, s, layer, e);
    st[OST_PF_FILLED] += 1;
  }
  return 0;
}

int oc_rollback(ocache* c, const int32_t* plan) {
  if (!c || !plan) return -1;
  for (int i = 0; i < plan[0]; ++i) {
    const int s = plan[1 + 3 * i], layer = plan[2 + 3 * i], e = plan[3 + 3 * i];
    if (layer < 0 || layer >= c->L || s < 0 || s >= c->S || e < 0 || e >= c->E) return -2;
    Pool& P = c->pools[c->pool_of(layer)];
    const int32_t key = c->key_of(layer, e);
    if (P.key[s] != key) continue;
    c->map[key] = -1;
    P.key[s] = -1;
    P.restamp(s, 0);
  }
  return 0;
}

int oc_stats(const ocache* c, int layer, uint64_t* out) {
  if (!c || layer < 0 || layer >= c->L || !out) return -1;
  std::memcpy(out, &c->stats[(size_t)layer * OST_N], sizeof(uint64_t) * OST_N);
  return 0;
}

int oc_state(const ocache* c, int32_t* map, int32_t* slot_key, uint64_t* stamp,
             uint8_t* pinned, uint64_t* clock, uint32_t* decode_freq,
             uint32_t* demand_freq, uint64_t* last_demand) {
  if (!c) return -1;
  const size_t K = c->map.size();
  if (map) std::memcpy(map, c->map.data(), K * sizeof(int32_t));
  if (decode_freq) std::memcpy(decode_freq, c->decode_freq.data(), K * sizeof(uint32_t));
  if (demand_freq) std::memcpy(demand_freq, c->demand_freq.data(), K * sizeof(uint32_t));
  if (last_demand) std::memcpy(last_demand, c->last_demand.data(), K * sizeof(uint64_t));
  for (size_t p = 0; p < c->pools.size(); ++p) {
    const Pool& P = c->pools[p];
    const size_t o = p * (size_t)c->S;
    if (slot_key) std::memcpy(slot_key + o, P.key.data(), c->S * sizeof(int32_t));
    if (stamp) std::memcpy(stamp + o, P.stamp.data(), c->S * sizeof(uint64_t));
    if (pinned) std::memcpy(pinned + o, P.pinned.data(), c->S);
    if (clock) clock[p] = P.clock;
  }
  return 0;
}

int oc_lru_order(const ocache* c, int pool, int32_t* out) {
  if (!c || pool < 0 || pool >= (int)c->pools.size() || !out) return -1;
  int i = 0;
  for (int s = c->pools[pool].head; s >= 0; s = c->pools[pool].next[s]) out[i++] = s;
  return i;
}

// ---------------------------------------------------------------------------
// Expert math in fp64
// ---------------------------------------------------------------------------

// FP4 E2M1 (OCP Microscaling Formats spec): 1 sign bit, 2 exponent bits with
// bias 1, 1 mantissa bit; exponent field 0 encodes the subnormal m * 2^-1.
double om_e2m1(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? m * 0.5 : std::ldexp(1.0 + m * 0.5, e - 1);
  return s ? -mag : mag;
}

// FP8 E4M3 "fn" (OCP 8-bit floating point spec): 1 sign bit, 4 exponent bits
// with bias 7, 3 mantissa bits; exponent 0 is subnormal m/8 * 2^-6; the code
// with all exponent and mantissa bits set is NaN (there is no infinity).
double om_e4m3(int byte) {
  const int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  double mag;
  if (e == 15 && m == 7) mag = NAN;
  else if (e == 0) mag = std::ldexp(m / 8.0, -6);
  else mag = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// E8M0 (OCP Microscaling Formats spec, the shared block scale): 8 exponent
// bits, bias 127, no sign and no mantissa: 2^(e - 127); 0xFF is NaN.
double om_e8m0(int byte) {
  const int e = byte & 255;
  return e == 255 ? NAN : std::ldexp(1.0, e - 127);
}

// IEEE binary16: 1 sign bit, 5 exponent bits with bias 15, 10 mantissa bits;
// exponent 0 is subnormal m * 2^-24, exponent 31 is inf (m = 0) or NaN.
double om_f16(uint16_t bits) {
  const int s = bits >> 15, e = (bits >> 10) & 31, m = bits & 1023;
  double mag;
  if (e == 31) mag = m ? NAN : INFINITY;
  else if (e == 0) mag = std::ldexp((double)m, -24);
  else mag = std::ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -mag : mag;
}

// bfloat16: the upper 16 bits of an IEEE binary32.
double om_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

namespace {

// The fused expert blob, one contiguous copy unit per expert [P2 What we
// changed: "fused copy layout", Correctness: "six-bank NVFP4 row sizes"].
// NVFP4: six banks -- gate, up, down e2m1 codes (two per byte, the even
// element in the low nibble, rows of the reduction dimension), then the gate,
// up, down e4m3 block scales (one per 16 consecutive elements of a row), then
// three fp32 per-matrix global scales padded to 16 bytes.  Gate and up are
// [I, H], down is [H, I].  bf16: gate, up, down, row-major.
// MXFP4 (OCP Microscaling: MXFP4 blocks of 32 e2m1 elements sharing one
// E8M0 scale; FreeToken PR #491, section 7, names MXFP4 among the expert
// formats): the same three code banks, then the gate, up, down E8M0 scales
// (one per 32 consecutive elements of a row); no global scale.
struct Layout {
  uint64_t code[3], scale[3], glob, total;
};
// Q4_0 arithmetic (blocks of 32 weights sharing an fp16 scale d, weight =
// d * (q - 8) for the 4-bit unsigned code q) -- FreeToken PR #491, section 7
// ("What did not change"), names Q4_0 among the expert formats -- laid out in
// banks like the fp4 formats: gate, up, down codes (two per byte, the even element in the low
// nibble), then gate, up, down fp16 scales (one per 32 consecutive elements
// of a row), padded to 16 bytes.
Layout q4_layout(int H, int I) {
  Layout L{};
  const uint64_t ih = (uint64_t)I * H;
  L.code[0] = 0;
  L.code[1] = ih / 2;
  L.code[2] = ih;
  L.scale[0] = 3 * ih / 2;
  L.scale[1] = L.scale[0] + ih / 16;  // 2 bytes per 32 elements
  L.scale[2] = L.scale[1] + ih / 16;
  L.glob = L.scale[2] + ih / 16;
  L.total = (L.glob + 15) / 16 * 16;
  return L;
}
Layout mxfp4_layout(int H, int I) {
  Layout L{};
  const uint64_t ih = (uint64_t)I * H;
  L.code[0] = 0;
  L.code[1] = ih / 2;
  L.code[2] = ih;
  L.scale[0] = 3 * ih / 2;
  L.scale[1] = L.scale[0] + ih / 32;
  L.scale[2] = L.scale[1] + ih / 32;
  L.glob = L.scale[2] + ih / 32;  // no global scales: the blob ends here
  L.total = (L.glob + 15) / 16 * 16;
  return L;
}
Layout nvfp4_layout(int H, int I) {
  Layout L{};
  const uint64_t ih = (uint64_t)I * H;
  L.code[0] = 0;
  L.code[1] = ih / 2;
  L.code[2] = ih;
  L.scale[0] = 3 * ih / 2;
  L.scale[1] = L.scale[0] + ih / 16;
  L.scale[2] = L.scale[1] + ih / 16;
  L.glob = L.scale[2] + ih / 16;
  L.total = L.glob + 16;
  return L;
}

}  // namespace

uint64_t om_blob_bytes(int fmt, int H, int I) {
  if (fmt == OFMT_BF16) return 6ull * H * I;
  if (fmt == OFMT_NVFP4) return nvfp4_layout(H, I).total;
  if (fmt == OFMT_MXFP4) return mxfp4_layout(H, I).total;
  if (fmt == OFMT_Q4_0) return q4_layout(H, I).total;
  return 0;
}

int om_dequant(int fmt, const uint8_t* blob, int H, int I, int which, double* out) {
  if (!blob || !out || which < 0 || which > 2 || H % 32 || I % 32) return -1;
  const int rows = (which == 2) ? H : I;
  const int cols = (which == 2) ? I : H;
  if (fmt == OFMT_BF16) {
    const uint16_t* w = reinterpret_cast<const uint16_t*>(blob) + (uint64_t)which * H * I;
    for (uint64_t i = 0; i < (uint64_t)rows * cols; ++i) {
      uint16_t b;
      std::memcpy(&b, w + i, 2);
      out[i] = om_bf16(b);
    }
    return 0;
  }
  if (fmt == OFMT_Q4_0) {  // element = f16(scale) * (code - 8)
    const Layout L = q4_layout(H, I);
    const uint8_t* codes = blob + L.code[which];
    const uint8_t* scales = blob + L.scale[which];
    for (int n = 0; n < rows; ++n) {
      for (int k = 0; k < cols; ++k) {
        const uint64_t idx = (uint64_t)n * cols + k;
        const uint8_t byte = codes[idx / 2];
        const int q = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
        uint16_t d;
        std::memcpy(&d, scales + 2 * ((uint64_t)n * (cols / 32) + k / 32), 2);
        out[idx] = om_f16(d) * (double)(q - 8);
      }
    }
    return 0;
  }
  if (fmt == OFMT_MXFP4) {  // element = e2m1(code) * 2^(scale - 127)
    const Layout L = mxfp4_layout(H, I);
    const uint8_t* codes = blob + L.code[which];
    const uint8_t* scales = blob + L.scale[which];
    for (int n = 0; n < rows; ++n) {
      for (int k = 0; k < cols; ++k) {
        const uint64_t idx = (uint64_t)n * cols + k;
        const uint8_t byte = codes[idx / 2];
        const int nib = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
        out[idx] = om_e2m1(nib) * om_e8m0(scales[(uint64_t)n * (cols / 32) + k / 32]);
      }
    }
    return 0;
  }
  if (fmt != OFMT_NVFP4) return -1;
  const Layout L = nvfp4_layout(H, I);
  float g;
  std::memcpy(&g, blob + L.glob + 4 * which, 4);
  const uint8_t* codes = blob + L.code[which];
  const uint8_t* scales = blob + L.scale[which];
  for (int n = 0; n < rows; ++n) {
    for (int k = 0; k < cols; ++k) {
      const uint64_t idx = (uint64_t)n * cols + k;
      const uint8_t byte = codes[idx / 2];
      const int nib = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
      const double sc = om_e4m3(scales[(uint64_t)n * (cols / 16) + k / 16]);
      out[idx] = om_e2m1(nib) * sc * (double)g;
    }
  }
  return 0;
}

namespace {

double silu(double v) { return v / (1.0 + std::exp(-v)); }

// y = W_d (silu(W_g x) * (W_u x)); W given dequantised, x in fp64.
void ffn(const double* Wg, const double* Wu, const double* Wd, int H, int I, const double* x,
         double* y) {
  std::vector<double> h(I);
  for (int n = 0; n < I; ++n) {
    double g = 0, u = 0;
    for (int k = 0; k < H; ++k) {
      g += Wg[(uint64_t)n * H + k] * x[k];
      u += Wu[(uint64_t)n * H + k] * x[k];
    }
    h[n] = silu(g) * u;
  }
  for (int n = 0; n < H; ++n) {
    double acc = 0;
    for (int k = 0; k < I; ++k) acc += Wd[(uint64_t)n * I + k] * h[k];
    y[n] = acc;
  }
}

struct Dequantised {
  std::vector<double> g, u, d;
  bool load(int fmt, const uint8_t* blob, int H, int I) {
    g.resize((size_t)I * H);
    u.resize((size_t)I * H);
    d.resize((size_t)H * I);
    return om_dequant(fmt, blob, H, I, 0, g.data()) == 0 &&
           om_dequant(fmt, blob, H, I, 1, u.data()) == 0 &&
           om_dequant(fmt, blob, H, I, 2, d.data()) == 0;
  }
};

}  // namespace

int om_expert_ffn(int fmt, const uint8_t* blob, int H, int I, const uint16_t* x, double* y) {
  if (!blob || !x || !y) return -1;
  Dequantised W;
  if (!W.load(fmt, blob, H, I)) return -1;
  std::vector<double> xd(H);
  for (int k = 0; k < H; ++k) xd[k] = om_bf16(x[k]);
  ffn(W.g.data(), W.u.data(), W.d.data(), H, I, xd.data(), y);
  return 0;
}

// One layer's MoE output [P2 Problem, What we changed; P1 section 5]:
// routed = sum over routes of weight * expert FFN, the shared expert scaled by
// a sigmoid gate computed from the same (original) hidden state, and the final
// sum routed + shared.  A route masked off (the CPU side of a hybrid split, or
// the GPU side) contributes nothing here, so two complementary masks add up to
// the full layer.
int om_layer(int fmt, const uint8_t* const* blobs, int E, int H, int I, const uint16_t* x,
             const int32_t* ids, const float* w, const uint8_t* mask, int B, int k,
             const uint8_t* shared_blob, int Is, const uint16_t* gate_w, double* out) {
  if (!blobs || !x || !ids || !w || !out || B < 0 || k < 0) return -1;
  // Dequantise each distinct expert once (cache by id), and the shared expert.
  std::vector<Dequantised*> cache(E, nullptr);
  Dequantised Sw;
  if (shared_blob && (!gate_w || !Sw.load(fmt, shared_blob, H, Is))) return -3;
  std::vector<double> xd(H), y(H);
  int rc = 0;
  for (int b = 0; b < B && rc == 0; ++b) {
    for (int kk = 0; kk < H; ++kk) xd[kk] = om_bf16(x[(uint64_t)b * H + kk]);
    double* acc = out + (uint64_t)b * H;
    for (int n = 0; n < H; ++n) acc[n] = 0.0;
    for (int j = 0; j < k; ++j) {
      const int r = b * k + j;
      if (mask && !mask[r]) continue;
      const int e = ids[r];
      if (e < 0 || e >= E) continue;
      if (!cache[e]) {
        cache[e] = new Dequantised;
        if (!cache[e]->load(fmt, blobs[e], H, I)) { rc = -2; break; }
      }
      ffn(cache[e]->g.data(), cache[e]->u.data(), cache[e]->d.data(), H, I, xd.data(), y.data());
      for (int n = 0; n < H; ++n) acc[n] += (double)w[r] * y[n];
    }
    if (rc == 0 && shared_blob) {
      double z = 0;
      for (int kk = 0; kk < H; ++kk) z += om_bf16(gate_w[kk]) * xd[kk];
      const double gate = 1.0 / (1.0 + std::exp(-z));
      ffn(Sw.g.data(), Sw.u.data(), Sw.d.data(), H, Is, xd.data(), y.data());
      for (int n = 0; n < H; ++n) acc[n] += gate * y[n];
    }
  }
  for (auto* p : cache) delete p;
  return rc;
}

// The look-ahead producer: layer L+1's router on layer L's hidden state, each
// row's k largest logits (ties and NaN as the header states), in the plain
// order -- every dot product in fp64, then one sort of the row's experts.
int om_lookahead_predict(const uint16_t* x, const uint16_t* router, int B, int E, int H, int k,
                         int32_t* pred, double* z_out) {
  if (!x || !router || !pred || B < 0 || E < 1 || H < 1 || k < 1 || k > E) return -1;
  std::vector<double> z(E);
  std::vector<int> order(E);
  for (int b = 0; b < B; ++b) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += om_bf16(router[(uint64_t)e * H + h]) * om_bf16(x[(uint64_t)b * H + h]);
      z[e] = acc;
      if (z_out) z_out[(uint64_t)b * E + e] = acc;
    }
    for (int e = 0; e < E; ++e) order[e] = e;
    std::sort(order.begin(), order.end(), [&](int a, int c) {
      const bool na = std::isnan(z[a]), nc = std::isnan(z[c]);
      if (na != nc) return nc;              // a number before a NaN
      if (!na && z[a] != z[c]) return z[a] > z[c];
      return a < c;                         // equal (or both NaN): the lower id first
    });
    for (int r = 0; r < k; ++r) pred[(uint64_t)b * k + r] = order[r];
  }
  return 0;
}

}  // extern "C"
