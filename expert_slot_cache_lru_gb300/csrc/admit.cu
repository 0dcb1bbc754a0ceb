// admit.cu -- slot-cache admission ("lru_ensure") and look-ahead prefetch.
//
// One CTA of 1024 threads per call; no host synchronisation, fixed launch
// shape, so both capture into CUDA graphs at any width.
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
#include "common.cuh"

namespace moe {
namespace {

struct SelSmem {
  int bins[kAdmitThreads];
  int digit;
  int krem;
};

// Chooses up to `want` victims in pool p and writes them, ascending
// (stamp, slot), to st.vict[0..n).  Returns n (the same in every thread).
__device__ int select_victims(const DevState& st, int p, unsigned long long clk, int want,
                              SelSmem& sm, BlockScratch& bs) {
  if (want <= 0) return 0;
  const int tid = threadIdx.x;
  const int S = st.S;
  const size_t base = (size_t)p * S;
  const int spt = (S + kAdmitThreads - 1) / kAdmitThreads;
  const int s0 = min(S, tid * spt), s1 = min(S, s0 + spt);

  // pass 0: how many slots may be evicted, and their stamp range
  int ne = 0;
  unsigned long long mn = ~0ull, mx = 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = st.stamp[base + s];
    if (!st.pinned[base + s] && t < clk) {
      ++ne;
      mn = t < mn ? t : mn;
      mx = t > mx ? t : mx;
    }
  }
  const int nE = block_sum(ne, bs);
  const int n = want < nE ? want : nE;
  if (n == 0) return 0;
  unsigned long long smin, smax;
  block_minmax_u64(mn, mx, bs, &smin, &smax);

  // radix select of the n-th smallest stamp (with multiplicity)
  unsigned long long prefix = 0;  // over rel = stamp - smin
  int k = n;                      // 1-based rank still to find inside the prefix
  const unsigned long long range = smax - smin;
  if (range > 0) {
    const int nbits = 64 - __clzll((long long)range);
    for (int shift = ((nbits - 1) / 10) * 10; shift >= 0; shift -= 10) {
      sm.bins[tid] = 0;
      __syncthreads();
      for (int s = s0; s < s1; ++s) {
        const unsigned long long t = st.stamp[base + s];
        if (st.pinned[base + s] || t >= clk) continue;
        const unsigned long long rel = t - smin;
        const bool match = (shift + 10 >= 64) || ((rel >> (shift + 10)) == (prefix >> (shift + 10)));
        if (match) atomicAdd(&sm.bins[(rel >> shift) & 1023], 1);
      }
      __syncthreads();
      const int c = sm.bins[tid];
      int tot;
      const int ex = block_excl_scan(c, bs, &tot);
      if (ex < k && k <= ex + c) {
        sm.digit = tid;
        sm.krem = k - ex;
      }
      __syncthreads();
      prefix |= (unsigned long long)sm.digit << shift;
      k = sm.krem;
      __syncthreads();
    }
  }
  // k is in [1, n] by construction; the clamp keeps every index below in
  // bounds even if the state were modified concurrently by a misuse.
  k = k < 1 ? 1 : (k > n ? n : k);
  const unsigned long long T = smin + prefix;
  const int below = n - k;  // every evictable slot with stamp < T is a victim

  // the k lowest-index evictable slots with stamp == T, in slot order
  int eq = 0, lt = 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = st.stamp[base + s];
    if (st.pinned[base + s] || t >= clk) continue;
    eq += (t == T);
    lt += (t < T);
  }
  int tot;
  int r = block_excl_scan(eq, bs, &tot);
  int q = below > 0 ? block_excl_scan(lt, bs, &tot) : 0;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long t = st.stamp[base + s];
    if (st.pinned[base + s] || t >= clk) continue;
    if (t == T) {
      if (r < k) st.vict[below + r] = s;
      ++r;
    } else if (t < T) {
      if (q < below) {
        st.lo_stamp[q] = t;
        st.lo_slot[q] = s;
      }
      ++q;
    }
  }
  __syncthreads();
  // order the (few) older victims by (stamp, slot)
  for (int i = tid; i < below; i += kAdmitThreads) {
    const unsigned long long ti = st.lo_stamp[i];
    const int si = st.lo_slot[i];
    int rank = 0;
    for (int j = 0; j < below; ++j) {
      const unsigned long long tj = st.lo_stamp[j];
      rank += (tj < ti) || (tj == ti && st.lo_slot[j] < si);
    }
    st.vict[rank] = si;
  }
  __syncthreads();
  return n;
}

__global__ void __launch_bounds__(kAdmitThreads, 1)
admit_kernel(DevState st, int layer, const int32_t* ids, int32_t* out, int R, int cap) {
  extern __shared__ int smem_i[];
  const int E = st.E;
  int* cnt = smem_i;      // [E] routes per expert
  int* aux = smem_i + E;  // [E] miss rank, -1 otherwise
  __shared__ BlockScratch bs;
  __shared__ SelSmem sel;
  __shared__ unsigned long long s_clk;
  __shared__ int s_acc[6];  // invalid, distinct, hits, evictions, overflow routes
  const int tid = threadIdx.x;
  const int p = pool_of(st, layer);
  const size_t pbase = (size_t)p * st.S;

  if (tid == 0) s_clk = st.clock[p] + 1;  // one recency stamp per admission
  if (tid < 6) s_acc[tid] = 0;
  for (int e = tid; e < E; e += kAdmitThreads) cnt[e] = 0;
  __syncthreads();
  const unsigned long long clk = s_clk;

  // histogram of the valid ids; ids outside [0, E) are counted and dropped
  int inv = 0;
  for (int r = tid; r < R; r += kAdmitThreads) {
    const int e = ids[r];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else ++inv;
  }
  __syncthreads();

  // distinct experts (contiguous chunk per thread): counters, lookup, hits
  const int ept = (E + kAdmitThreads - 1) / kAdmitThreads;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int nd = 0, nh = 0, nm = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    aux[e] = -1;
    if (c == 0) continue;
    ++nd;
    const int key = layer * E + e;
    st.decode_freq[key] += (uint32_t)c;
    const uint32_t df = st.demand_freq[key];
    if (df != 0xffffffffu) st.demand_freq[key] = df + 1;
    st.last_demand[key] = clk;
    const int s = st.map[key];
    if (s >= 0) {
      st.stamp[pbase + s] = clk;  // hit: refresh recency; protected from this admission
      ++nh;
    } else {
      aux[e] = 1;
      ++nm;
    }
  }
  int nM;
  int rank = block_excl_scan(nm, bs, &nM);  // misses ranked in ascending expert id
  for (int e = e0; e < e1; ++e)
    if (aux[e] >= 0) aux[e] = rank++;
  int nA = (cap >= 0 && cap < nM) ? cap : nM;  // the fetch cap admits the lowest ids
  const int nV = select_victims(st, p, clk, nA, sel, bs);
  const bool short_of_slots = nV < nA;
  nA = nV;

  // install: the i-th admitted miss takes the i-th victim
  int nev = 0;
  for (int e = e0; e < e1; ++e) {
    const int i = aux[e];
    if (i < 0 || i >= nA) continue;
    const int s = st.vict[i];
    const size_t g = pbase + s;
    const int old = st.slot_key[g];
    if (old >= 0) {
      st.map[old] = -1;
      ++nev;
    }
    const int key = layer * E + e;
    st.slot_key[g] = key;
    st.map[key] = s;
    st.stamp[g] = clk;
    st.plan_demand[1 + 3 * i + 0] = s;
    st.plan_demand[1 + 3 * i + 1] = layer;
    st.plan_demand[1 + 3 * i + 2] = e;
  }
  __syncthreads();

  // rewrite routes to slots (in place allowed: each thread reads then writes its own r)
  int ov = 0;
  for (int r = tid; r < R; r += kAdmitThreads) {
    const int e = ids[r];
    int o = -1;
    if ((unsigned)e < (unsigned)E) {
      o = st.map[layer * E + e];
      ov += (o < 0);
    }
    out[r] = o;
  }
  if (inv) atomicAdd(&s_acc[0], inv);
  if (nd) atomicAdd(&s_acc[1], nd);
  if (nh) atomicAdd(&s_acc[2], nh);
  if (nev) atomicAdd(&s_acc[3], nev);
  if (ov) atomicAdd(&s_acc[4], ov);
  __syncthreads();
  if (tid == 0) {
    moe_stats* S = &st.stats[layer];
    S->calls += 1;
    S->lookups += s_acc[1];
    S->hits += s_acc[2];
    S->misses += nM;
    S->fetched += nA;
    S->overflow_routes += s_acc[4];
    S->evictions += s_acc[3];
    S->invalid_routes += s_acc[0];
    if (s_acc[0]) S->status_bits |= MOE_STATUS_INVALID_ID;
    if (short_of_slots) S->status_bits |= MOE_STATUS_CAPACITY;
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

__global__ void __launch_bounds__(kAdmitThreads, 1)
prefetch_kernel(DevState st, int layer, const int32_t* pred, int n, int32_t* plan) {
  extern __shared__ int smem_i[];
  const int E = st.E;
  int* cnt = smem_i;      // [E] requested flag, later the candidate list
  int* aux = smem_i + E;  // [E] candidate rank, -1 otherwise
  __shared__ BlockScratch bs;
  __shared__ SelSmem sel;
  __shared__ int s_acc[3];  // invalid, requests, resident
  const int tid = threadIdx.x;
  const int p = pool_of(st, layer);
  const size_t pbase = (size_t)p * st.S;
  const unsigned long long clk = st.clock[p];  // the clock does not advance

  if (tid < 3) s_acc[tid] = 0;
  for (int e = tid; e < E; e += kAdmitThreads) cnt[e] = 0;
  __syncthreads();
  int inv = 0;
  for (int i = tid; i < n; i += kAdmitThreads) {
    const int e = pred[i];
    if ((unsigned)e < (unsigned)E) cnt[e] = 1;
    else ++inv;
  }
  __syncthreads();
  const int ept = (E + kAdmitThreads - 1) / kAdmitThreads;
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
  int rank = block_excl_scan(nq, bs, &nQ);
  for (int e = e0; e < e1; ++e)
    if (aux[e] >= 0) {
      cnt[rank] = e;  // candidates in ascending id (cnt of this chunk is no longer needed)
      ++rank;
    }
  if (inv) atomicAdd(&s_acc[0], inv);
  if (nreq) atomicAdd(&s_acc[1], nreq);
  if (nres) atomicAdd(&s_acc[2], nres);
  const int nV = select_victims(st, p, clk, nQ, sel, bs);

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

__global__ void rollback_kernel(DevState st, int32_t* plan) {
  const int n = plan[0];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int s = plan[1 + 3 * i], layer = plan[2 + 3 * i], e = plan[3 + 3 * i];
    if ((unsigned)layer >= (unsigned)st.L || (unsigned)s >= (unsigned)st.S ||
        (unsigned)e >= (unsigned)st.E)
      continue;
    const size_t g = (size_t)pool_of(st, layer) * st.S + s;
    const int key = layer * st.E + e;
    if (st.slot_key[g] != key) continue;
    st.map[key] = -1;
    st.slot_key[g] = -1;
    st.stamp[g] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) plan[0] = 0;
}

__global__ void pin_kernel(DevState st, size_t g, int v) { st.pinned[g] = (uint8_t)v; }

}  // namespace

size_t admit_smem_bytes(int E) { return 2ull * E * sizeof(int); }

cudaError_t launch_admit(const DevState& st, int layer, const int32_t* ids, int32_t* out, int R,
                         int cap, cudaStream_t s) {
  admit_kernel<<<1, kAdmitThreads, admit_smem_bytes(st.E), s>>>(st, layer, ids, out, R, cap);
  return cudaGetLastError();
}

cudaError_t launch_prefetch(const DevState& st, int layer, const int32_t* pred, int n,
                            int32_t* plan, cudaStream_t s) {
  prefetch_kernel<<<1, kAdmitThreads, admit_smem_bytes(st.E), s>>>(st, layer, pred, n, plan);
  return cudaGetLastError();
}

cudaError_t launch_rollback(const DevState& st, const int32_t* plan, cudaStream_t s) {
  rollback_kernel<<<1, 256, 0, s>>>(st, const_cast<int32_t*>(plan));
  return cudaGetLastError();
}

cudaError_t launch_pin(const DevState& st, int layer, int slot, int pinned, cudaStream_t s) {
  pin_kernel<<<1, 1, 0, s>>>(st, (size_t)pool_of(st, layer) * st.S + slot, pinned);
  return cudaGetLastError();
}

cudaError_t admit_set_smem_limits(int E) {
  const size_t bytes = admit_smem_bytes(E);
  cudaError_t e = cudaFuncSetAttribute(admit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefetch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

}  // namespace moe
