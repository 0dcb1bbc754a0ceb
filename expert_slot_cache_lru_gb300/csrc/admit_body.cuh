// admit_body.cuh -- the admission ("lru_ensure") and the look-ahead prefetch
// as block-wide device routines, templated on the block's thread count NT, so
// that the standalone one-CTA kernels (admit.cu, NT = 1024) and one CTA of the
// fused decode-layer launch (ffn_stream.cu, NT = 512) run the same code.
//
// Admission [FreeToken PR #680 "fix(moe): admit a wide offloaded decode step's
// experts 128 at a time", Problem and Solution; FreeToken issue #753 "[Perf]
// Offloaded decode: overlap the expert-miss gather ...", What we changed;
// FreeToken PR #491 "refactor(moe): extract hybrid decode orchestration",
// sections 4-5].  The pages' kernel deduplicates a query in a [K,K] register
// block, which spills past 128 ids and does not compile past 1,024; here the
// dedup is a shared-memory histogram over the expert ids plus a block prefix
// scan, linear in routes + experts, so one call admits any width.
//
// Victims: the unpinned slots not touched by this admission (stamp < clock),
// ascending (stamp, slot) -- empty slots have stamp 0 and come first.  They
// are found with a block-wide radix select on the stamp (10-bit digits over
// the stamps' actual range, usually one or two passes), then the lowest slot
// indices among the threshold stamp by a prefix scan in slot order.
//
// Prefetch [llama.cpp fork PR #126 "cuda : MoE look-ahead expert prefetch
// (PR-A consumer) + LFRU eviction guard", Consumer and Eviction guard]: the
// same victim routine serves both paths, so they cannot drift (the page's
// shared select_victim / install_fill core).
#pragma once

#include "common.cuh"

namespace moe {
namespace admission {

constexpr int kLoSmem = 512;  // victims ordered in shared memory up to this many
constexpr int kTopMax = 16;   // warp-minimum selection up to this many victims
constexpr int kTopSpt = 8;    // ... over at most this many slots per thread

constexpr int kRadixBins = 1024;  // 10-bit digits

// A map entry with this bit set names a slot whose copy-in has not completed
// (set by an admission inside a layer launch, cleared by the same launch).
constexpr int32_t kMapPending = (int32_t)0x80000000u;

template <int NT>
struct SelSmem {
  int bins[kRadixBins];
  int digit;
  int krem;
  int nvict;
  uint32_t wk[NT / 32][kTopMax];
  unsigned long long lo_t[kLoSmem];
  int lo_s[kLoSmem];
  int vict[kLoSmem];
};

// The victim key of slot s: its stamp when the slot may be evicted, ~0 when it
// is pinned or was touched by this admission (stamp >= clk).  A real stamp is
// a clock value and never ~0.  CACHED reads a copy of the pool held in shared
// memory (filled at kernel entry and patched on hits); otherwise the key is
// derived from the global stamp and pin arrays.
template <bool CACHED>
struct PoolKeys {
  const unsigned long long* sm;  // CACHED: [S]
  const DevState* st;
  size_t base;
  unsigned long long clk;
  __device__ __forceinline__ unsigned long long operator()(int s) const {
    if (CACHED) return sm[s];
    const unsigned long long t = st->stamp[base + s];
    return (st->pinned[base + s] || t >= clk) ? ~0ull : t;
  }
};

// The `want` (<= kTopMax) smallest (stamp, slot) pairs among the evictable
// slots when the evictable stamps span fewer than 2^16 clock values: keys are
// 32-bit, (stamp - oldest) << 16 | slot, unique and ordered like (stamp,
// slot).  Each thread sorts its (at most kTopSpt) keys; each warp takes its
// `want` smallest by repeated warp minimum (redux.sync) and popping the
// winner; warp 0 does the same over the warps' lists.  Returns -1 (in every
// thread) when the stamps span too much for 32-bit keys.
template <bool CACHED, int NT>
__device__ int select_victims_small(const DevState& st, const PoolKeys<CACHED>& key, int want,
                                    int* vict, SelSmem<NT>& sm, BlockScratch& bs) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int S = st.S;
  const int spt = (S + NT - 1) / NT;
  const int s0 = min(S, tid * spt), s1 = min(S, s0 + spt);
  unsigned long long mn = ~0ull, mx = 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = key(s);
    if (t == ~0ull) continue;
    mn = t < mn ? t : mn;
    mx = t > mx ? t : mx;
  }
  unsigned long long smin, smax;
  block_minmax_u64<NT>(mn, mx, bs, &smin, &smax);
  if (smin == ~0ull) return 0;               // nothing evictable
  if (smax - smin >= 0xffffull) return -1;   // too wide for 32-bit keys
  uint32_t k[kTopSpt];
#pragma unroll
  for (int j = 0; j < kTopSpt; ++j) k[j] = 0xffffffffu;
  for (int s = s0; s < s1; ++s) {  // insertion into the sorted k
    const unsigned long long t = key(s);
    if (t == ~0ull) continue;
    uint32_t v = ((uint32_t)(t - smin) << 16) | (uint32_t)s;
#pragma unroll
    for (int j = 0; j < kTopSpt; ++j)
      if (v < k[j]) {
        const uint32_t x = k[j];
        k[j] = v;
        v = x;
      }
  }
  for (int i = 0; i < want; ++i) {  // this warp's `want` smallest
    const uint32_t m = __reduce_min_sync(0xffffffffu, k[0]);
    if (k[0] == m && m != 0xffffffffu) {  // keys are unique: one lane pops its head
#pragma unroll
      for (int j = 0; j < kTopSpt - 1; ++j) k[j] = k[j + 1];
      k[kTopSpt - 1] = 0xffffffffu;
    }
    if (lane == 0) sm.wk[w][i] = m;
  }
  sync_nt<NT>();
  if (w == 0) {
    constexpr int NW = NT / 32;  // one list per warp, lanes past NW hold none
    int h = 0, n = 0;
    uint32_t cur = lane < NW ? sm.wk[lane][0] : 0xffffffffu;
    for (int i = 0; i < want; ++i) {
      const uint32_t m = __reduce_min_sync(0xffffffffu, cur);
      if (m == 0xffffffffu) break;  // fewer evictable slots than wanted (uniform)
      if (cur == m) {
        ++h;
        cur = h < want ? sm.wk[lane][h] : 0xffffffffu;
      }
      if (lane == 0) vict[i] = (int)(m & 0xffffu);
      n = i + 1;
    }
    if (lane == 0) sm.nvict = n;
  }
  sync_nt<NT>();
  return sm.nvict;
}

// Chooses up to `want` victims in pool p and writes them, ascending
// (stamp, slot), to vict[0..n) (shared memory when want <= kLoSmem, else the
// global scratch).  Returns n (the same in every thread).
template <bool CACHED, int NT>
__device__ int select_victims(const DevState& st, const PoolKeys<CACHED>& key, int want,
                              int* vict, SelSmem<NT>& sm, BlockScratch& bs) {
  if (want <= 0) return 0;
  const int tid = threadIdx.x;
  const int S = st.S;
  const int spt = (S + NT - 1) / NT;
  if (want <= kTopMax && spt <= kTopSpt && S <= 65536) {
    const int n = select_victims_small<CACHED, NT>(st, key, want, vict, sm, bs);
    if (n >= 0) return n;
  }
  const int s0 = min(S, tid * spt), s1 = min(S, s0 + spt);

  // pass 0: how many slots may be evicted, and their stamp range
  int ne = 0;
  unsigned long long mn = ~0ull, mx = 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = key(s);
    if (t != ~0ull) {
      ++ne;
      mn = t < mn ? t : mn;
      mx = t > mx ? t : mx;
    }
  }
  const int nE = block_sum<NT>(ne, bs);
  const int n = want < nE ? want : nE;
  if (n == 0) return 0;
  unsigned long long smin, smax;
  block_minmax_u64<NT>(mn, mx, bs, &smin, &smax);

  // radix select of the n-th smallest stamp (with multiplicity)
  unsigned long long prefix = 0;  // over rel = stamp - smin
  int k = n;                      // 1-based rank still to find inside the prefix
  const unsigned long long range = smax - smin;
  if (range > 0) {
    const int nbits = 64 - __clzll((long long)range);
    for (int shift = ((nbits - 1) / 10) * 10; shift >= 0; shift -= 10) {
      for (int i = tid; i < kRadixBins; i += NT) sm.bins[i] = 0;
      sync_nt<NT>();
      for (int s = s0; s < s1; ++s) {
        const unsigned long long t = key(s);
        if (t == ~0ull) continue;
        const unsigned long long rel = t - smin;
        const bool match = (shift + 10 >= 64) || ((rel >> (shift + 10)) == (prefix >> (shift + 10)));
        if (match) atomicAdd(&sm.bins[(rel >> shift) & 1023], 1);
      }
      sync_nt<NT>();
      // bins [tid * BPT, tid * BPT + BPT) belong to this thread, in order
      constexpr int BPT = kRadixBins / NT;
      int cb[BPT], c = 0;
#pragma unroll
      for (int j = 0; j < BPT; ++j) c += (cb[j] = sm.bins[tid * BPT + j]);
      int tot;
      int ex = block_excl_scan<NT>(c, bs, &tot);
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        if (ex < k && k <= ex + cb[j]) {
          sm.digit = tid * BPT + j;
          sm.krem = k - ex;
        }
        ex += cb[j];
      }
      sync_nt<NT>();
      prefix |= (unsigned long long)sm.digit << shift;
      k = sm.krem;
      sync_nt<NT>();
    }
  }
  // k is in [1, n] by construction; the clamp keeps every index below in
  // bounds even if the state were modified concurrently by a misuse.
  k = k < 1 ? 1 : (k > n ? n : k);
  const unsigned long long T = smin + prefix;
  const int below = n - k;  // every evictable slot with stamp < T is a victim
  unsigned long long* lo_t =
      below <= kLoSmem ? sm.lo_t : reinterpret_cast<unsigned long long*>(st.lo_stamp);
  int* lo_s = below <= kLoSmem ? sm.lo_s : st.lo_slot;

  // the k lowest-index evictable slots with stamp == T, in slot order
  int eq = 0, lt = 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = key(s);
    if (t == ~0ull) continue;
    eq += (t == T);
    lt += (t < T);
  }
  int tot;
  int r = block_excl_scan<NT>(eq, bs, &tot);
  int q = below > 0 ? block_excl_scan<NT>(lt, bs, &tot) : 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = key(s);
    if (t == ~0ull) continue;
    if (t == T) {
      if (r < k) vict[below + r] = s;
      ++r;
    } else if (t < T) {
      if (q < below) {
        lo_t[q] = t;
        lo_s[q] = s;
      }
      ++q;
    }
  }
  sync_nt<NT>();
  // order the (few) older victims by (stamp, slot)
  for (int i = tid; i < below; i += NT) {
    const unsigned long long ti = lo_t[i];
    const int si = lo_s[i];
    int rank = 0;
    for (int j = 0; j < below; ++j) {
      const unsigned long long tj = lo_t[j];
      rank += (tj < ti) || (tj == ti && lo_s[j] < si);
    }
    vict[rank] = si;
  }
  sync_nt<NT>();
  return n;
}

// Admission.  CACHED keeps the pool's victim keys and slot keys in shared
// memory for the whole call: they are loaded at entry together with the ids
// and the clock, so the victim search and the install read no global memory.
// Block-shared state of an admission or a prefetch (a static array of the
// standalone kernels; carved from dynamic shared memory where a CTA of a
// larger kernel runs the admission).
template <int NT>
struct AdmitShared {
  BlockScratch bs;
  SelSmem<NT> sel;
  int s_acc[6];  // invalid, distinct, hits, evictions, overflow routes (prefetch: 3)
  unsigned long long s_st[sizeof(moe_stats) / 8];  // the layer's counters
};

// The admission, run by one block of NT threads.  smem_raw holds the [E] x 3
// counters and, when CACHED, the pool's keys (admit_smem_bytes).  Every thread
// calls before_install() after the victims are chosen and before anything is
// installed: no map entry of a requested expert changes before that point.
// An installed miss's map entry is its slot OR-ed with map_or: kMapPending
// marks it as not yet copied in, for readers inside the same launch.
template <bool CACHED, int NT, class Hook>
__device__ void admit_body(const DevState& st, int layer, const int32_t* ids, int32_t* out, int R,
                           int cap, unsigned char* smem_raw, AdmitShared<NT>& sh,
                           Hook&& before_install, int32_t map_or = 0) {
  const int E = st.E, S = st.S;
  unsigned long long* pkey = reinterpret_cast<unsigned long long*>(smem_raw);  // [S] CACHED
  int* pslot = reinterpret_cast<int*>(smem_raw + (CACHED ? (size_t)S * 8 : 0));  // [S] CACHED
  int* cnt = pslot + (CACHED ? S : 0);  // [E] routes per expert
  int* aux = cnt + E;                    // [E] miss rank, -1 otherwise
  int* slot_of = aux + E;                // [E] slot of each requested expert after the call
  BlockScratch& bs = sh.bs;
  int* s_acc = sh.s_acc;
  unsigned long long* s_st = sh.s_st;
  const int tid = threadIdx.x;
  const int p = pool_of(st, layer);
  const size_t pbase = (size_t)p * S;
  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);

  // independent loads first: the first ids, the clock, the layer's counters,
  // this thread's expert state (one expert per thread when E <= 1024), the pool
  uint32_t pf_df = 0, pf_dm = 0;
  int pf_map = -1;
  if (ept == 1 && e0 < e1) {
    const int key = layer * E + e0;
    pf_df = st.decode_freq[key];
    pf_dm = st.demand_freq[key];
    pf_map = st.map[key];
  }
  if (tid < (int)(sizeof(moe_stats) / 8))
    s_st[tid] = reinterpret_cast<const unsigned long long*>(&st.stats[layer])[tid];
  int idv[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = tid + j * NT;
    idv[j] = r < R ? ids[r] : 0;
  }
  const unsigned long long clk = st.clock[p] + 1;  // one recency stamp per admission
  if (CACHED) {
#pragma unroll 4
    for (int s = tid; s < S; s += NT) {
      const unsigned long long t = st.stamp[pbase + s];
      const uint8_t pin = st.pinned[pbase + s];
      const int sk = st.slot_key[pbase + s];
      pkey[s] = pin ? ~0ull : t;  // every stored stamp is below clk
      pslot[s] = sk;
    }
  }
  if (tid < 6) s_acc[tid] = 0;
  for (int e = tid; e < E; e += NT) cnt[e] = 0;
  sync_nt<NT>();

  // histogram of the valid ids; ids outside [0, E) are counted and dropped
  int inv = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = tid + j * NT;
    if (r >= R) continue;
    const int e = idv[j];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else ++inv;
  }
  for (int r = tid + 2 * NT; r < R; r += NT) {
    const int e = ids[r];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else ++inv;
  }
  sync_nt<NT>();

  // distinct experts (contiguous chunk per thread): counters, lookup, hits
  int nd = 0, nh = 0, nm = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    aux[e] = -1;
    slot_of[e] = -1;
    if (c == 0) continue;
    ++nd;
    const int key = layer * E + e;
    const bool pre = ept == 1;  // state loaded at entry
    st.decode_freq[key] = (pre ? pf_df : st.decode_freq[key]) + (uint32_t)c;
    const uint32_t df = pre ? pf_dm : st.demand_freq[key];
    if (df != 0xffffffffu) st.demand_freq[key] = df + 1;
    st.last_demand[key] = clk;
    const int s = pre ? pf_map : st.map[key];
    if (s >= 0) {
      st.stamp[pbase + s] = clk;  // hit: refresh recency; protected from this admission
      if (CACHED) pkey[s] = ~0ull;
      slot_of[e] = s;
      ++nh;
    } else {
      aux[e] = 1;
      ++nm;
    }
  }
  int nM;
  int rank = block_excl_scan<NT>(nm, bs, &nM);  // misses ranked in ascending expert id
  for (int e = e0; e < e1; ++e)
    if (aux[e] >= 0) aux[e] = rank++;
  int nA = (cap >= 0 && cap < nM) ? cap : nM;  // the fetch cap admits the lowest ids
  int* vict = nA <= kLoSmem ? sh.sel.vict : st.vict;
  const PoolKeys<CACHED> keys{pkey, &st, pbase, clk};
  const int nV = select_victims<CACHED, NT>(st, keys, nA, vict, sh.sel, bs);
  const bool short_of_slots = nV < nA;
  nA = nV;
  before_install();

  // install: the i-th admitted miss takes the i-th victim
  int nev = 0;
  for (int e = e0; e < e1; ++e) {
    const int i = aux[e];
    if (i < 0 || i >= nA) continue;
    const int s = vict[i];
    const size_t g = pbase + s;
    const int old = CACHED ? pslot[s] : st.slot_key[g];
    if (old >= 0) {
      st.map[old] = -1;
      ++nev;
    }
    const int key = layer * E + e;
    st.slot_key[g] = key;
    st.map[key] = s | map_or;
    st.stamp[g] = clk;
    slot_of[e] = s;
    st.plan_demand[1 + 3 * i + 0] = s;
    st.plan_demand[1 + 3 * i + 1] = layer;
    st.plan_demand[1 + 3 * i + 2] = e;
  }
  sync_nt<NT>();

  // rewrite routes to slots (in place allowed: each thread reads then writes its own r)
  int ov = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = tid + j * NT;
    if (r >= R) continue;
    const int e = idv[j];
    int o = -1;
    if ((unsigned)e < (unsigned)E) {
      o = slot_of[e];
      ov += (o < 0);
    }
    out[r] = o;
  }
  for (int r = tid + 2 * NT; r < R; r += NT) {
    const int e = ids[r];
    int o = -1;
    if ((unsigned)e < (unsigned)E) {
      o = slot_of[e];
      ov += (o < 0);
    }
    out[r] = o;
  }
  if (inv) atomicAdd(&s_acc[0], inv);
  if (nd) atomicAdd(&s_acc[1], nd);
  if (nh) atomicAdd(&s_acc[2], nh);
  if (nev) atomicAdd(&s_acc[3], nev);
  if (ov) atomicAdd(&s_acc[4], ov);
  sync_nt<NT>();
  if (tid == 0) {  // the counters as loaded at entry, plus this call
    moe_stats v;
    memcpy(&v, s_st, sizeof v);
    v.calls += 1;
    v.lookups += s_acc[1];
    v.hits += s_acc[2];
    v.misses += nM;
    v.fetched += nA;
    v.overflow_routes += s_acc[4];
    v.evictions += s_acc[3];
    v.invalid_routes += s_acc[0];
    if (s_acc[0]) v.status_bits |= MOE_STATUS_INVALID_ID;
    if (short_of_slots) v.status_bits |= MOE_STATUS_CAPACITY;
    st.stats[layer] = v;
    st.plan_demand[0] = nA;
    st.clock[p] = clk;
  }
}

// LFRU score: demand frequency in the high bits, a recency byte saturating
// in the low byte.
__device__ __forceinline__ unsigned long long lfru_score(const DevState& st, int key,
                                                         unsigned long long clk) {
  unsigned long long f = st.demand_freq[key];
  f = f > 0xFFFFFFull ? 0xFFFFFFull : f;
  const unsigned long long ld = st.last_demand[key];
  unsigned long long rec = 0;
  if (ld != 0) {
    const unsigned long long age = clk - ld;
    rec = 255ull - (age < 255ull ? age : 255ull);
  }
  return (f << 8) | rec;
}

// The look-ahead prefetch admission, run by one block of NT threads; smem_i
// holds [E] x 2 ints.
template <int NT>
__device__ void prefetch_body(const DevState& st, int layer, const int32_t* pred, int n,
                              int32_t* plan, int* smem_i, AdmitShared<NT>& sh) {
  const int E = st.E;
  int* cnt = smem_i;      // [E] requested flag, later the candidate list
  int* aux = smem_i + E;  // [E] candidate rank, -1 otherwise
  BlockScratch& bs = sh.bs;
  int* s_acc = sh.s_acc;  // invalid, requests, resident
  const int tid = threadIdx.x;
  const int p = pool_of(st, layer);
  const size_t pbase = (size_t)p * st.S;
  const unsigned long long clk = st.clock[p];  // the clock does not advance

  if (tid < 3) s_acc[tid] = 0;
  for (int e = tid; e < E; e += NT) cnt[e] = 0;
  sync_nt<NT>();
  int inv = 0;
  for (int i = tid; i < n; i += NT) {
    const int e = pred[i];
    if ((unsigned)e < (unsigned)E) cnt[e] = 1;
    else ++inv;
  }
  sync_nt<NT>();
  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int nreq = 0, nres = 0, nq = 0;
  for (int e = e0; e < e1; ++e) {
    aux[e] = -1;
    if (!cnt[e]) continue;
    ++nreq;
    if (st.map[layer * E + e] >= 0) ++nres;  // resident: left alone
    else {
      aux[e] = 1;
      ++nq;
    }
  }
  int nQ;
  int rank = block_excl_scan<NT>(nq, bs, &nQ);
  for (int e = e0; e < e1; ++e)
    if (aux[e] >= 0) {
      cnt[rank] = e;  // candidates in ascending id (cnt of this chunk is no longer needed)
      ++rank;
    }
  if (inv) atomicAdd(&s_acc[0], inv);
  if (nreq) atomicAdd(&s_acc[1], nreq);
  if (nres) atomicAdd(&s_acc[2], nres);
  const PoolKeys<false> keys{nullptr, &st, pbase, clk};
  const int nV = select_victims<false, NT>(st, keys, nQ, st.vict, sh.sel, bs);

  if (tid == 0) {
    // Each candidate, ascending, looks at the current first evictable slot.
    // A fill stamps its slot with the clock, which removes it from the
    // evictable set, so the next one is the next victim in order; a refused
    // prediction leaves the same slot first for the next candidate.
    int idx = 0, m = 0;
    unsigned long long filled = 0, dropped = 0, novict = 0, pfev = 0;
    for (int q = 0; q < nQ; ++q) {
      const int e = cnt[q];
      const int key = layer * E + e;
      if (idx >= nV) {
        ++novict;
        continue;
      }
      const int s = st.vict[idx];
      const size_t g = pbase + s;
      const int old = st.slot_key[g];
      if (old >= 0 && st.demand_freq[old] >= 2u) {
        const unsigned long long Rs = lfru_score(st, old, clk);
        const unsigned long long Ps = lfru_score(st, key, clk);
        if (4ull * Rs > 5ull * Ps + 4ull * (4ull << 8)) {
          ++dropped;
          continue;
        }
      }
      if (old >= 0) {
        st.map[old] = -1;
        ++pfev;
      }
      st.slot_key[g] = key;
      st.map[key] = s;
      st.stamp[g] = clk;
      plan[1 + 3 * m + 0] = s;
      plan[1 + 3 * m + 1] = layer;
      plan[1 + 3 * m + 2] = e;
      ++m;
      ++filled;
      ++idx;
    }
    plan[0] = m;
    moe_stats* S = &st.stats[layer];
    S->pf_invalid += s_acc[0];
    S->pf_requests += s_acc[1];
    S->pf_resident += s_acc[2];
    S->pf_filled += filled;
    S->pf_dropped_guard += dropped;
    S->pf_no_victim += novict;
    S->pf_evictions += pfev;
  }
}

}  // namespace admission
}  // namespace moe
