// moe_cache.cu -- host side of the C ABI: descriptor checks, state and
// scratch allocation, and the ordering of kernels, streams and events.
//
// The per-layer order and the fork/join follow FreeToken issue #753 ("[Perf]
// Offloaded decode: overlap the expert-miss gather with the same layer's
// shared expert, event-ordered inside the CUDA graph", What we changed):
//   compute: admit -> record(ready) -> shared expert + gate -> wait(done) -> routed
//   side:    wait(ready) -> gather -> record(done)
// Both events are created with the cache, before any capture; the join is
// made on every exit path once the side stream has been forked, so no side
// work outlives the layer and a capture never ends with an unjoined fork.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"

namespace moe {
cudaError_t admit_set_smem_limits(int E, int S);
cudaError_t gemv_set_smem_limits(int H, int I, int Is, int k_max);
}  // namespace moe

using moe::DevState;
using moe::FfnScratch;

struct moe_cache {
  moe_cache_desc d{};
  int P = 0;
  int device = 0;
  DevState st{};
  FfnScratch sc{};
  void* mem = nullptr;       // one allocation for all state and scratch
  void* stage_mem = nullptr; // staging entries of a layer launch with the admission inside
  size_t mem_bytes = 0;
  cudaEvent_t ev_ready = nullptr, ev_done = nullptr;
  int fail_gathers = 0;
  int gather_grid = 76;
  int down_k_max = 0;        // largest k the down kernel's shared memory was sized for
  int last_pf_layer = 0;     // target layer of the last prefetch enqueued (selects its plan)
  bool stream_ffn = true;    // decode-sized steps use the streaming FFN kernels
  int wide_mode = MOE_WIDE_AUTO;  // which kernels run wide steps (moe_cache_set_wide_path)
  std::vector<const void*> host_ptrs;  // [L*E] host blob addresses, copied at create
  moe_cpu_exec* cpu = nullptr;         // hybrid CPU executor, when started
};

namespace {

thread_local char g_cuda_err[256] = "";
std::mutex g_setup_mu;  // serialises the kernel set-up of moe_cache_create

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_cuda_err, sizeof g_cuda_err, "%.160s: %.80s (%d)", what, cudaGetErrorString(e), (int)e);
  return MOE_ERR_CUDA;
}

#define CK(call)                                     \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t blob_bytes(int fmt, int H, int I) {
  const size_t ih = (size_t)H * I;
  if (fmt == MOE_W_BF16) return 6 * ih;
  if (fmt == MOE_W_NVFP4) return 3 * ih / 2 + 3 * ih / 16 + 16;
  if (fmt == MOE_W_MXFP4) return 3 * ih / 2 + 3 * ih / 32;
  if (fmt == MOE_W_Q4_0) return 3 * ih / 2 + 3 * ih / 16;
  return 0;
}

// Sub-allocator over one device allocation (256-byte aligned pieces).
struct Carve {
  size_t off = 0;
  template <typename T>
  size_t take(size_t n) {
    size_t o = align_up(off, 256);
    off = o + n * sizeof(T);
    return o;
  }
};

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int check_layer(const moe_cache* c, int layer) {
  return (c && layer >= 0 && layer < c->d.n_layers) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_CACHE_ABI_VERSION; }

const char* moe_strerror(int err) {
  switch (err) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CONFIG: return "invalid cache descriptor";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_CAPACITY: return "request exceeds the cache's sizes";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MOE_ERR_STATE: return "call not valid in the cache's state";
    case MOE_ERR_INJECTED: return "injected failure";
    case MOE_ERR_SCRATCH:
      return "request larger than the 1 MiB scratch of moe_routed_experts_noalloc";
    default: return "unknown error";
  }
}

const char* moe_last_cuda_error(void) { return g_cuda_err; }

int moe_cache_create(const moe_cache_desc* desc, moe_cache** out) {
  if (!desc || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const moe_cache_desc& d = *desc;
  if (d.n_layers <= 0 || d.n_experts <= 0 || d.n_experts > 16384 || d.n_slots < 0 ||
      d.n_slots >= (1 << 20) || (d.pool_mode != MOE_POOL_SHARED && d.pool_mode != MOE_POOL_PER_LAYER) ||
      d.max_routes < 1 || d.max_routes > 16384 || d.max_rows < 1 || d.max_rows > d.max_routes ||
      d.max_pred < 0 || d.max_pred > 4096 || d.gather_ctas < 0 || d.gather_ctas > 4096)
    return MOE_ERR_CONFIG;
  if ((long long)d.n_layers * d.n_experts > 0x7fffffffLL) return MOE_ERR_CONFIG;
  if (d.max_pred > 0 && d.n_slots == 0) return MOE_ERR_CONFIG;  // prefetch needs a cache
  const bool compute = d.hidden > 0 || d.inter > 0;
  if (compute) {
    if (d.hidden <= 0 || d.inter <= 0 || d.hidden % 32 || d.inter % 32 || d.shared_inter < 0 ||
        d.shared_inter % 32 ||
        (d.wfmt < MOE_W_BF16 || d.wfmt > MOE_W_Q4_0))
      return MOE_ERR_CONFIG;
    if (d.slot_bytes != blob_bytes(d.wfmt, d.hidden, d.inter)) return MOE_ERR_CONFIG;
    if ((size_t)d.hidden * 4 > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  }
  if (d.slot_bytes > 0) {
    if (!d.slot_storage || !d.host_experts || d.slot_bytes % 16 ||
        (reinterpret_cast<uintptr_t>(d.slot_storage) & 255) || d.n_slots == 0)
      return MOE_ERR_CONFIG;
    if (d.slot_stride && (d.slot_stride < d.slot_bytes || d.slot_stride % 256)) return MOE_ERR_CONFIG;
  }

  moe_cache* c = new (std::nothrow) moe_cache;
  if (!c) return MOE_ERR_CUDA;
  c->d = d;
  if (d.slot_bytes > 0 && !d.slot_stride) c->d.slot_stride = align_up(d.slot_bytes, 256);
  c->P = d.pool_mode == MOE_POOL_PER_LAYER ? d.n_layers : 1;
  c->gather_grid = d.gather_ctas ? d.gather_ctas : 76;
  auto fail = [&](int r) {
    moe_cache_destroy(c);
    return r;
  };
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaGetDevice"));

  const size_t K = (size_t)d.n_layers * d.n_experts;
  const size_t PS = (size_t)c->P * d.n_slots;
  const int vcap = std::max(std::max(d.max_routes, d.max_pred), 1);
  const int I = d.inter, H = d.hidden, Is = d.shared_inter;
  Carve cv;
  const size_t o_map = cv.take<int32_t>(K), o_dfq = cv.take<uint32_t>(K),
               o_dmq = cv.take<uint32_t>(K), o_ld = cv.take<uint64_t>(K),
               o_sk = cv.take<int32_t>(PS), o_stamp = cv.take<uint64_t>(PS),
               o_pin = cv.take<uint8_t>(PS), o_clk = cv.take<uint64_t>(c->P),
               o_stats = cv.take<moe_stats>(d.n_layers),
               o_pd = cv.take<int32_t>(1 + 3 * (size_t)d.max_routes),
               o_pp = cv.take<int32_t>(1 + 3 * (size_t)std::max(d.max_pred, 1)),
               o_pp2 = cv.take<int32_t>(1 + 3 * (size_t)std::max(d.max_pred, 1)),
               o_grp = cv.take<int32_t>(2 + 3 * (size_t)d.max_routes),
               o_vict = cv.take<int32_t>(vcap), o_los = cv.take<uint64_t>(vcap),
               o_lol = cv.take<int32_t>(vcap), o_hb = cv.take<const uint8_t*>(K),
               o_h = cv.take<float>(((size_t)d.max_routes + d.max_rows) * std::max(I, 1)),
               o_gdone = cv.take<int32_t>(std::max(d.max_routes, 1)),
               o_laz = cv.take<float>((size_t)d.max_rows * d.n_experts),
               o_lactr = cv.take<unsigned>(1),
               o_hs = cv.take<float>((size_t)d.max_rows * std::max(Is, 1)),
               o_gate = cv.take<float>(d.max_rows),
               o_ys = cv.take<float>((size_t)d.max_rows * std::max(H, 1)),
               o_x16 = cv.take<uint16_t>((size_t)d.max_rows * std::max(H, 1)),
               o_xinv = cv.take<float>(d.max_rows),
               o_y = cv.take<float>((size_t)d.max_routes * std::max(H, 1)),
               o_h16 = cv.take<uint16_t>((size_t)d.max_routes * std::max(I, 1)),
               o_hinv = cv.take<float>(d.max_routes),
               o_dense = cv.take<int32_t>(1 + (size_t)d.max_routes),
               o_status = cv.take<unsigned long long>(1),
               o_bar = cv.take<unsigned long long>(1),
               o_ep = cv.take<unsigned long long>(1), o_pseq = cv.take<unsigned long long>(1),
               o_bar2 = cv.take<unsigned long long>(1),
               o_sslot = cv.take<unsigned long long>(std::max(d.max_routes, 1));
  c->mem_bytes = align_up(cv.off, 256);
  e = cudaMalloc(&c->mem, c->mem_bytes);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMalloc(state)"));
  uint8_t* m = static_cast<uint8_t*>(c->mem);
  DevState& st = c->st;
  st.L = d.n_layers;
  st.E = d.n_experts;
  st.S = d.n_slots;
  st.P = c->P;
  st.per_layer = d.pool_mode == MOE_POOL_PER_LAYER;
  st.map = reinterpret_cast<int32_t*>(m + o_map);
  st.decode_freq = reinterpret_cast<uint32_t*>(m + o_dfq);
  st.demand_freq = reinterpret_cast<uint32_t*>(m + o_dmq);
  st.last_demand = reinterpret_cast<uint64_t*>(m + o_ld);
  st.slot_key = reinterpret_cast<int32_t*>(m + o_sk);
  st.stamp = reinterpret_cast<uint64_t*>(m + o_stamp);
  st.pinned = m + o_pin;
  st.clock = reinterpret_cast<uint64_t*>(m + o_clk);
  st.stats = reinterpret_cast<moe_stats*>(m + o_stats);
  st.plan_demand = reinterpret_cast<int32_t*>(m + o_pd);
  st.plan_pf[0] = reinterpret_cast<int32_t*>(m + o_pp);
  st.plan_pf[1] = reinterpret_cast<int32_t*>(m + o_pp2);
  st.groups = reinterpret_cast<int32_t*>(m + o_grp);
  st.vict = reinterpret_cast<int32_t*>(m + o_vict);
  st.lo_stamp = reinterpret_cast<uint64_t*>(m + o_los);
  st.lo_slot = reinterpret_cast<int32_t*>(m + o_lol);
  st.vcap = vcap;
  st.host_blob = reinterpret_cast<const uint8_t* const*>(m + o_hb);
  st.slots = static_cast<uint8_t*>(d.slot_storage);
  st.stride = c->d.slot_stride;
  st.slot_bytes = d.slot_bytes;
  st.max_routes = d.max_routes;
  st.max_pred = d.max_pred;
  st.status = reinterpret_cast<unsigned long long*>(m + o_status);
  c->sc.h = reinterpret_cast<float*>(m + o_h);
  c->sc.hs = reinterpret_cast<float*>(m + o_hs);
  c->sc.gate = reinterpret_cast<float*>(m + o_gate);
  c->sc.ys = reinterpret_cast<float*>(m + o_ys);
  c->sc.bar = reinterpret_cast<unsigned long long*>(m + o_bar);
  c->sc.epoch = reinterpret_cast<unsigned long long*>(m + o_ep);
  c->sc.pseq = reinterpret_cast<unsigned long long*>(m + o_pseq);
  c->sc.bar2 = reinterpret_cast<unsigned long long*>(m + o_bar2);
  c->sc.sslot = reinterpret_cast<unsigned long long*>(m + o_sslot);
  c->sc.x16 = reinterpret_cast<uint16_t*>(m + o_x16);
  c->sc.xinv = reinterpret_cast<float*>(m + o_xinv);
  c->sc.y = reinterpret_cast<float*>(m + o_y);
  c->sc.h16 = reinterpret_cast<uint16_t*>(m + o_h16);
  c->sc.hinv = reinterpret_cast<float*>(m + o_hinv);
  c->sc.dense = reinterpret_cast<int32_t*>(m + o_dense);
  c->sc.gdone = reinterpret_cast<int*>(m + o_gdone);
  c->sc.la_z = reinterpret_cast<float*>(m + o_laz);
  c->sc.la_ctr = reinterpret_cast<unsigned*>(m + o_lactr);

  // initial state: nothing resident, every clock at 1
  e = cudaMemset(c->mem, 0, c->mem_bytes);
  if (e == cudaSuccess) e = cudaMemset(st.map, 0xff, K * sizeof(int32_t));
  if (e == cudaSuccess && PS) e = cudaMemset(st.slot_key, 0xff, PS * sizeof(int32_t));
  if (e == cudaSuccess) {
    std::vector<uint64_t> ones(c->P, 1ull);
    e = cudaMemcpy(st.clock, ones.data(), c->P * sizeof(uint64_t), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) return fail(cuda_fail(e, "state init"));

  if (d.slot_bytes > 0) {
    c->host_ptrs.assign(d.host_experts, d.host_experts + K);
    std::vector<const uint8_t*> dev(K);
    for (size_t k = 0; k < K; ++k) {
      const void* hp = d.host_experts[k];
      if (!hp || (reinterpret_cast<uintptr_t>(hp) & 15)) return fail(MOE_ERR_CONFIG);
      void* dp = nullptr;
      e = cudaHostGetDevicePointer(&dp, const_cast<void*>(hp), 0);
      if (e != cudaSuccess) {
        cudaGetLastError();
        std::snprintf(g_cuda_err, sizeof g_cuda_err,
                      "host expert %zu is not pinned, mapped memory: %s", k, cudaGetErrorString(e));
        return fail(MOE_ERR_CONFIG);
      }
      dev[k] = static_cast<const uint8_t*>(dp);
    }
    e = cudaMemcpy(const_cast<const uint8_t**>(st.host_blob), dev.data(), K * sizeof(void*),
                   cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(cuda_fail(e, "host blob table"));
  }

  {
    // kernel attributes and occupancy figures are per kernel, shared by every
    // cache: one create at a time sets them (limits only ever rise)
    std::lock_guard<std::mutex> lock(g_setup_mu);
    e = moe::admit_set_smem_limits(d.n_experts, d.n_slots);
    if (e != cudaSuccess) return fail(cuda_fail(e, "admission shared memory"));
    if (compute) {
      // the down kernel stages k routes' intermediates in shared memory
      c->down_k_max = (int)std::min<size_t>(d.max_routes, (200 * 1024) / ((size_t)I * 4));
      e = moe::gemv_set_smem_limits(H, I, Is, c->down_k_max);
      if (e == cudaSuccess) e = moe::ffn_stream_init();
      if (e == cudaSuccess && moe::lookahead_supported(H, d.n_experts, 1))
        e = moe::lookahead_init(H);
      if (e == cudaSuccess && moe::grouped_supported(d.wfmt, H, I, d.n_experts))
        e = moe::grouped_init(d.n_experts, H, I);
      if (e != cudaSuccess) return fail(cuda_fail(e, "GEMV shared memory"));
    }
  }
  if (compute) {
    // a layer launch with the admission inside copies an uncapped step's misses
    // into staging entries while the admission runs: up to max_routes of them,
    // within 64 MB
    if (d.slot_bytes > 0) {
      const size_t cap = (64ull << 20) / c->d.slot_stride;
      const int n = (int)std::min<size_t>((size_t)d.max_routes, cap);
      if (n > 0) {
        e = cudaMalloc(&c->stage_mem, (size_t)n * c->d.slot_stride);
        if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMalloc(staging)"));
        c->sc.stage = static_cast<uint8_t*>(c->stage_mem);
        c->sc.stage_n = n;
      }
    }
  }
  e = cudaEventCreateWithFlags(&c->ev_ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(cuda_fail(e, "create sync"));
  *out = c;
  return MOE_OK;
}

int moe_cache_destroy(moe_cache* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  int rc = MOE_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) rc = cuda_fail(e, "destroy sync");
  moe::hybrid_stop(c->cpu);
  if (c->ev_ready) cudaEventDestroy(c->ev_ready);
  if (c->ev_done) cudaEventDestroy(c->ev_done);
  if (c->mem) cudaFree(c->mem);
  if (c->stage_mem) cudaFree(c->stage_mem);
  delete c;
  return rc;
}

int moe_cache_prefill(moe_cache* c, int layer, const int32_t* h_ids, int n, void* stream) {
  if (check_layer(c, layer) != MOE_OK || n < 0 || (n > 0 && !h_ids)) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  const moe_cache_desc& d = c->d;
  const int E = d.n_experts, S = d.n_slots;
  const int p = c->P > 1 ? layer : 0;
  CK(cudaDeviceSynchronize());
  std::vector<int32_t> map(E), sk(S);
  uint64_t clk = 0;
  CK(cudaMemcpy(map.data(), c->st.map + (size_t)layer * E, E * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(sk.data(), c->st.slot_key + (size_t)p * S, (size_t)S * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&clk, c->st.clock + p, 8, cudaMemcpyDeviceToHost));
  std::vector<int> slot_of(n);
  int next = 0;
  for (int i = 0; i < n; ++i) {
    const int e = h_ids[i];
    if (e < 0 || e >= E || map[e] >= 0) return MOE_ERR_INVALID_ARG;
    while (next < S && sk[next] >= 0) ++next;
    if (next >= S) return MOE_ERR_CAPACITY;
    map[e] = next;
    sk[next] = layer * E + e;
    slot_of[i] = next;
  }
  // commit: map entries, slot keys, stamps = clock; then the bytes
  CK(cudaMemcpy(c->st.map + (size_t)layer * E, map.data(), E * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->st.slot_key + (size_t)p * S, sk.data(), (size_t)S * 4, cudaMemcpyHostToDevice));
  for (int i = 0; i < n; ++i)
    CK(cudaMemcpy(c->st.stamp + (size_t)p * S + slot_of[i], &clk, 8, cudaMemcpyHostToDevice));
  if (d.slot_bytes > 0) {
    for (int i = 0; i < n; ++i) {
      uint8_t* dst = c->st.slots + ((size_t)p * S + slot_of[i]) * c->st.stride;
      CK(cudaMemcpyAsync(dst, c->host_ptrs[(size_t)layer * E + h_ids[i]], d.slot_bytes,
                         cudaMemcpyHostToDevice, as_stream(stream)));
    }
    CK(cudaStreamSynchronize(as_stream(stream)));
  }
  return MOE_OK;
}

int moe_cache_pin(moe_cache* c, int layer, int slot, int pinned, void* stream) {
  if (check_layer(c, layer) != MOE_OK || slot < 0 || slot >= c->d.n_slots) return MOE_ERR_INVALID_ARG;
  CK(moe::launch_pin(c->st, layer, slot, pinned ? 1 : 0, as_stream(stream)));
  return MOE_OK;
}

int moe_admit(moe_cache* c, int layer, const int32_t* d_ids, int32_t* d_slot_ids, int n_routes,
              int fetch_cap, void* stream) {
  if (check_layer(c, layer) != MOE_OK || n_routes < 0) return MOE_ERR_INVALID_ARG;
  if (n_routes > c->d.max_routes) return MOE_ERR_CAPACITY;
  if (n_routes > 0 && (!d_ids || !d_slot_ids)) return MOE_ERR_INVALID_ARG;
  CK(moe::launch_admit(c->st, layer, d_ids, d_slot_ids, n_routes, fetch_cap, as_stream(stream)));
  return MOE_OK;
}

int moe_prefetch(moe_cache* c, int layer, const int32_t* d_pred, int n, void* stream) {
  if (check_layer(c, layer) != MOE_OK || n < 0 || (n > 0 && !d_pred)) return MOE_ERR_INVALID_ARG;
  if (c->d.max_pred == 0) return MOE_ERR_STATE;
  if (n > c->d.max_pred) return MOE_ERR_CAPACITY;
  CK(moe::launch_prefetch(c->st, layer, d_pred, n, c->st.plan_pf[layer & 1], as_stream(stream)));
  c->last_pf_layer = layer;
  return MOE_OK;
}

int moe_lookahead_predict(moe_cache* c, const void* d_x, const void* d_router, int n_rows,
                          int k_pred, int32_t* d_pred, void* stream) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const moe_cache_desc& d = c->d;
  if (n_rows < 0 || k_pred < 1) return MOE_ERR_INVALID_ARG;
  if (n_rows == 0) return MOE_OK;
  if (!d_x || !d_router || !d_pred || (reinterpret_cast<uintptr_t>(d_x) & 15) ||
      (reinterpret_cast<uintptr_t>(d_router) & 15) || (reinterpret_cast<uintptr_t>(d_pred) & 3))
    return MOE_ERR_INVALID_ARG;
  if (d.hidden == 0) return MOE_ERR_STATE;
  if (n_rows > d.max_rows) return MOE_ERR_CAPACITY;
  if (!moe::lookahead_supported(d.hidden, d.n_experts, k_pred)) return MOE_ERR_UNSUPPORTED;
  CK(moe::launch_lookahead(d_x, d_router, n_rows, d.hidden, d.n_experts, k_pred, c->sc.la_z,
                           c->sc.la_ctr, d_pred, as_stream(stream)));
  return MOE_OK;
}

int moe_gather_missing(moe_cache* c, int which, void* stream) {
  if (!c || (which != MOE_PLAN_DEMAND && which != MOE_PLAN_PREFETCH)) return MOE_ERR_INVALID_ARG;
  if (c->d.slot_bytes == 0) return MOE_ERR_STATE;
  if (which == MOE_PLAN_PREFETCH && c->d.max_pred == 0) return MOE_ERR_STATE;
  if (c->fail_gathers > 0) {
    --c->fail_gathers;
    return MOE_ERR_INJECTED;
  }
  const int32_t* plan =
      which == MOE_PLAN_DEMAND ? c->st.plan_demand : c->st.plan_pf[c->last_pf_layer & 1];
  CK(moe::launch_gather(c->st, plan, c->gather_grid, as_stream(stream)));
  return MOE_OK;
}

int moe_rollback_plan(moe_cache* c, int which, void* stream) {
  if (!c || (which != MOE_PLAN_DEMAND && which != MOE_PLAN_PREFETCH)) return MOE_ERR_INVALID_ARG;
  const int32_t* plan =
      which == MOE_PLAN_DEMAND ? c->st.plan_demand : c->st.plan_pf[c->last_pf_layer & 1];
  CK(moe::launch_rollback(c->st, plan, as_stream(stream)));
  return MOE_OK;
}

static int check_compute(moe_cache* c, int layer, int n_rows, int k, const void* shared_blob,
                         const void* shared_gate) {
  if (check_layer(c, layer) != MOE_OK || n_rows < 0 || k < 0) return MOE_ERR_INVALID_ARG;
  if (c->d.hidden == 0 || c->d.slot_bytes == 0) return MOE_ERR_STATE;
  if (n_rows > c->d.max_rows || (size_t)n_rows * k > (size_t)c->d.max_routes) return MOE_ERR_CAPACITY;
  if (k > c->down_k_max) return MOE_ERR_UNSUPPORTED;
  if (shared_blob && (c->d.shared_inter == 0 || !shared_gate)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

static int run_shared(moe_cache* c, const void* d_x, int n_rows, const void* blob, const void* gate,
                      cudaStream_t s) {
  if (n_rows == 0) return MOE_OK;
  if (c->stream_ffn &&
      moe::ffn_stream_supported(c->d.wfmt, c->d.hidden, c->d.shared_inter, n_rows, n_rows)) {
    CK(moe::launch_shared_stream(c->st, c->d.wfmt, c->d.hidden, c->d.shared_inter, d_x, n_rows,
                                 static_cast<const uint8_t*>(blob), gate, c->sc, c->st.status, s));
    return MOE_OK;
  }
  CK(moe::launch_shared_expert(c->d.wfmt, c->d.hidden, c->d.shared_inter, d_x, n_rows,
                               static_cast<const uint8_t*>(blob), gate, c->sc, s));
  return MOE_OK;
}

static int run_routed(moe_cache* c, int layer, const void* d_x, const int32_t* slot_ids,
                      const float* w, int n_rows, int k, bool with_shared, void* d_out,
                      cudaStream_t s) {
  const moe_cache_desc& d = c->d;
  if (n_rows == 0) return MOE_OK;
  if (c->stream_ffn && moe::ffn_stream_supported(d.wfmt, d.hidden, d.inter, n_rows, n_rows * k)) {
    CK(moe::launch_routed_stream(c->st, d.wfmt, d.hidden, d.inter, layer, d_x, slot_ids, w, n_rows,
                                 k, with_shared ? c->sc.ys : nullptr, d_out, c->sc, c->st.status, s));
    return MOE_OK;
  }
  if (k > 0 && moe::grouped_supported(d.wfmt, d.hidden, d.inter, d.n_experts)) {
    CK(moe::launch_routed_grouped(c->st, d.wfmt, d.hidden, d.inter, layer, d_x, slot_ids, w,
                                  n_rows, k, with_shared ? c->sc.ys : nullptr, d_out, c->sc,
                                  d.max_routes, c->wide_mode, s));
    return MOE_OK;
  }
  if (k > 0)
    CK(moe::launch_routed_up(c->st, d.wfmt, d.hidden, d.inter, layer, d_x, slot_ids, n_rows, k,
                           c->sc, s));
  CK(moe::launch_routed_down_combine(c->st, d.wfmt, d.hidden, d.inter, layer, slot_ids, w,
                                     n_rows, k, with_shared ? c->sc.ys : nullptr, d_out, c->sc, s));
  return MOE_OK;
}

int moe_routed_experts(moe_cache* c, int layer, const void* d_x, const int32_t* d_slot_ids,
                       const float* d_w, int n_rows, int k, const void* d_shared_blob,
                       const void* d_shared_gate, void* d_out, void* stream) {
  int rc = check_compute(c, layer, n_rows, k, d_shared_blob, d_shared_gate);
  if (rc != MOE_OK) return rc;
  if (n_rows == 0) return MOE_OK;
  if (!d_x || !d_out || (k > 0 && (!d_slot_ids || !d_w)) || d_out == d_x) return MOE_ERR_INVALID_ARG;
  if (d_shared_blob && (rc = run_shared(c, d_x, n_rows, d_shared_blob, d_shared_gate, as_stream(stream))))
    return rc;
  return run_routed(c, layer, d_x, d_slot_ids, d_w, n_rows, k, d_shared_blob != nullptr, d_out,
                    as_stream(stream));
}

int moe_routed_experts_noalloc(int wfmt, int hidden, int inter, const void* d_slots,
                               size_t slot_stride, int n_slots, const void* d_x,
                               const int32_t* d_slot_ids, const float* d_w, int n_rows, int k,
                               void* d_out, unsigned long long* d_status, void* stream) {
  if (wfmt < MOE_W_BF16 || wfmt > MOE_W_Q4_0 || hidden <= 0 ||
      inter <= 0 || hidden % 32 ||
      inter % 32 || n_slots <= 0 || n_rows < 0 || k < 0)
    return MOE_ERR_INVALID_ARG;
  if (!d_slots || (reinterpret_cast<uintptr_t>(d_slots) & 255) || slot_stride % 256 ||
      slot_stride < blob_bytes(wfmt, hidden, inter))
    return MOE_ERR_INVALID_ARG;
  if (n_rows == 0) return MOE_OK;
  if (!d_x || !d_out || d_out == d_x || (reinterpret_cast<uintptr_t>(d_x) & 15) ||
      (k > 0 && (!d_slot_ids || !d_w)))
    return MOE_ERR_INVALID_ARG;
  if (256 + (size_t)n_rows * (size_t)k * (size_t)inter * sizeof(float) > MOE_NOALLOC_SCRATCH_BYTES)
    return MOE_ERR_SCRATCH;
  void* scratch = nullptr;
  CK(moe::noalloc_scratch(&scratch));
  if (!moe::ffn_stream_supported(wfmt, hidden, inter, n_rows, n_rows * k)) return MOE_ERR_UNSUPPORTED;
  CK(moe::launch_routed_noalloc(wfmt, hidden, inter, static_cast<const uint8_t*>(d_slots),
                                slot_stride, n_slots, d_x, d_slot_ids, d_w, n_rows, k, d_out,
                                d_status, scratch, as_stream(stream)));
  return MOE_OK;
}

namespace {

// ---------------------------------------------------------------- layer schedule
// The work of one decode layer as operations on two streams, and the order
// they are enqueued in [P2 What we changed, "order inside one layer"; P1
// section 4 for the hybrid post and add].  The same function drives the CUDA
// calls (CudaOps) and, for the host-only schedule test, a recorder
// (moe_schedule_trace).
enum Op {
  kOpAdmit, kOpPost, kOpPrefetch, kOpGatherDemand, kOpGatherPrefetch, kOpShared, kOpRouted,
  kOpAddCpu, kOpLayerAdmit, kOpLayerStream, kOpRecordReady, kOpWaitReady, kOpRecordDone,
  kOpWaitDone, kOpCount
};
const char* const kOpName[kOpCount] = {
    "admit", "post", "prefetch", "gather_demand", "gather_prefetch", "shared", "routed",
    "add_cpu", "layer_admit", "layer_stream", "record_ready", "wait_ready", "record_done",
    "wait_done"};
enum Str { kCompute = 0, kSide = 1 };

struct LayerOps {
  virtual int run(Op op, Str s) = 0;  // MOE_OK or an error code
  virtual ~LayerOps() = default;
};

struct LayerPlan {
  bool one_launch;  // the whole layer, admission included, in one launch
  bool fused;       // the admission, then one launch for the rest
  bool overlap;     // the gather on the side stream, forked and joined by events
  bool pf, shared, hybrid;
};

int schedule_layer(const LayerPlan& p, LayerOps& ops) {
  int rc;
  if (p.one_launch) return ops.run(kOpLayerAdmit, kCompute);
  if ((rc = ops.run(kOpAdmit, kCompute))) return rc;
  if (p.hybrid && (rc = ops.run(kOpPost, kCompute))) return rc;
  if (p.pf && (rc = ops.run(kOpPrefetch, kCompute))) return rc;
  if (p.fused) {
    if ((rc = ops.run(kOpLayerStream, kCompute))) return rc;
    return p.hybrid ? ops.run(kOpAddCpu, kCompute) : MOE_OK;
  }
  if (!p.overlap) {
    if ((rc = ops.run(kOpGatherDemand, kCompute))) return rc;
    if (p.shared && (rc = ops.run(kOpShared, kCompute))) return rc;
    if ((rc = ops.run(kOpRouted, kCompute))) return rc;
    if (p.pf && (rc = ops.run(kOpGatherPrefetch, kCompute))) return rc;
    return p.hybrid ? ops.run(kOpAddCpu, kCompute) : MOE_OK;
  }
  // fork: the side stream waits for the admission, gathers, and records done
  if ((rc = ops.run(kOpRecordReady, kCompute))) return rc;
  if ((rc = ops.run(kOpWaitReady, kSide))) return rc;
  int side = ops.run(kOpGatherDemand, kSide);
  const int rec = ops.run(kOpRecordDone, kSide);
  if (side == MOE_OK && p.pf) side = ops.run(kOpGatherPrefetch, kSide);
  int shared = MOE_OK;
  if (side == MOE_OK && rec == MOE_OK && p.shared) shared = ops.run(kOpShared, kCompute);
  // join, on every path once forked (a capture must not end with an unjoined fork)
  const int join = rec == MOE_OK ? ops.run(kOpWaitDone, kCompute) : rec;
  if (side != MOE_OK) return side;
  if (join != MOE_OK) return join;
  if (shared != MOE_OK) return shared;
  if ((rc = ops.run(kOpRouted, kCompute))) return rc;
  return p.hybrid ? ops.run(kOpAddCpu, kCompute) : MOE_OK;
}

// The operations as CUDA work on the two streams.
struct CudaOps : LayerOps {
  moe_cache* c;
  int layer;
  const void* d_x;
  const int32_t* d_ids;
  const float* d_w;
  int32_t* d_slot_ids;
  int n_rows, k, fetch_cap;
  const int32_t* d_pred;
  int n_pred;
  const void* d_shared_blob;
  const void* d_shared_gate;
  void* d_out;
  cudaStream_t cs, ss;
  int32_t* pf_plan;

  int run(Op op, Str s) override {
    const cudaStream_t st = s == kSide ? ss : cs;
    const moe_cache_desc& dd = c->d;
    const bool pf = d_pred && n_pred > 0;
    switch (op) {
      case kOpAdmit:
        CK(moe::launch_admit(c->st, layer, d_ids, d_slot_ids, n_rows * k, fetch_cap, st));
        return MOE_OK;
      case kOpPost:
        CK(moe::hybrid_post(c->cpu, layer, d_ids, d_slot_ids, d_w, d_x, n_rows, k, st));
        return MOE_OK;
      case kOpPrefetch:
        CK(moe::launch_prefetch(c->st, layer + 1, d_pred, n_pred, pf_plan, st));
        c->last_pf_layer = layer + 1;
        return MOE_OK;
      case kOpGatherDemand:
        CK(moe::launch_gather(c->st, c->st.plan_demand, c->gather_grid, st));
        return MOE_OK;
      case kOpGatherPrefetch:
        CK(moe::launch_gather(c->st, pf_plan, c->gather_grid, st));
        return MOE_OK;
      case kOpShared:
        return run_shared(c, d_x, n_rows, d_shared_blob, d_shared_gate, st);
      case kOpRouted:
        return run_routed(c, layer, d_x, d_slot_ids, d_w, n_rows, k, d_shared_blob != nullptr,
                          d_out, st);
      case kOpAddCpu:
        CK(moe::hybrid_add(c->cpu, d_out, n_rows, c->st.status, st));
        return MOE_OK;
      case kOpLayerAdmit:
        CK(moe::launch_layer_admit(c->st, dd.wfmt, dd.hidden, dd.inter, layer, d_x, d_ids,
                                   d_slot_ids, d_w, n_rows, k, fetch_cap, pf ? d_pred : nullptr,
                                   n_pred, static_cast<const uint8_t*>(d_shared_blob),
                                   d_shared_gate, pf ? pf_plan : nullptr, d_out, c->sc,
                                   c->st.status, st));
        if (pf) c->last_pf_layer = layer + 1;
        return MOE_OK;
      case kOpLayerStream:
        CK(moe::launch_layer_stream(c->st, dd.wfmt, dd.hidden, dd.inter, layer, d_x, d_slot_ids,
                                    d_w, n_rows, k, static_cast<const uint8_t*>(d_shared_blob),
                                    d_shared_gate, c->st.plan_demand, pf ? pf_plan : nullptr,
                                    d_out, c->sc, c->st.status, st));
        return MOE_OK;
      case kOpRecordReady:
        CK(cudaEventRecord(c->ev_ready, st));
        return MOE_OK;
      case kOpWaitReady:
        CK(cudaStreamWaitEvent(st, c->ev_ready, 0));
        return MOE_OK;
      case kOpRecordDone:
        CK(cudaEventRecord(c->ev_done, st));
        return MOE_OK;
      case kOpWaitDone:
        CK(cudaStreamWaitEvent(st, c->ev_done, 0));
        return MOE_OK;
      default:
        return MOE_ERR_INVALID_ARG;
    }
  }
};

// The recorder of the host-only schedule test: "c:op" / "s:op" tokens, and an
// optional operation index that fails.
struct TraceOps : LayerOps {
  std::string out;
  int n = 0, fail_at = -1;
  int run(Op op, Str s) override {
    out += (s == kSide ? "s:" : "c:");
    out += kOpName[op];
    out += ' ';
    return n++ == fail_at ? MOE_ERR_CUDA : MOE_OK;
  }
};

// The plan moe_decode_layer runs for a step of this shape on this cache.
LayerPlan plan_of(const moe_cache* c, int n_rows, int k, bool shared, bool pf, unsigned flags) {
  LayerPlan p{};
  p.overlap = (flags & MOE_OVERLAP) != 0;
  p.hybrid = (flags & MOE_HYBRID) != 0;
  p.pf = pf;
  p.shared = shared;
  const moe_cache_desc& dd = c->d;
  p.fused = (flags & MOE_FUSED) && c->stream_ffn && dd.slot_bytes > 0 &&
            (!shared || dd.shared_inter == dd.inter) &&
            moe::layer_stream_supported(dd.wfmt, dd.hidden, dd.inter, n_rows, k, p.shared);
  // the hybrid post must follow the admission, so a hybrid layer keeps it as
  // its own launch
  p.one_launch = p.fused && !p.hybrid &&
                 moe::layer_admit_supported(c->st, dd.wfmt, dd.hidden, dd.inter, n_rows, k, p.shared);
  return p;
}

}  // namespace

int moe_decode_layer(moe_cache* c, int layer, const void* d_x, const int32_t* d_ids,
                     const float* d_w, int32_t* d_slot_ids, int n_rows, int k, int fetch_cap,
                     const int32_t* d_pred, int n_pred, const void* d_shared_blob,
                     const void* d_shared_gate, void* d_out, void* compute_stream,
                     void* side_stream, unsigned flags) {
  int rc = check_compute(c, layer, n_rows, k, d_shared_blob, d_shared_gate);
  if (rc != MOE_OK) return rc;
  const int R = n_rows * k;
  if (R > 0 && (!d_ids || !d_slot_ids || !d_w)) return MOE_ERR_INVALID_ARG;
  if (!d_x || !d_out || d_out == d_x) return MOE_ERR_INVALID_ARG;
  const bool pf = d_pred && n_pred > 0;
  if (pf && (layer + 1 >= c->d.n_layers || c->d.max_pred == 0)) return MOE_ERR_INVALID_ARG;
  if (pf && n_pred > c->d.max_pred) return MOE_ERR_CAPACITY;
  const LayerPlan p = plan_of(c, n_rows, k, d_shared_blob != nullptr, pf, flags);
  if (p.hybrid && !c->cpu) return MOE_ERR_STATE;
  if (!p.fused && p.overlap && !side_stream) return MOE_ERR_INVALID_ARG;
  CudaOps ops;
  ops.c = c, ops.layer = layer, ops.d_x = d_x, ops.d_ids = d_ids, ops.d_w = d_w;
  ops.d_slot_ids = d_slot_ids, ops.n_rows = n_rows, ops.k = k, ops.fetch_cap = fetch_cap;
  ops.d_pred = d_pred, ops.n_pred = n_pred, ops.d_shared_blob = d_shared_blob;
  ops.d_shared_gate = d_shared_gate, ops.d_out = d_out;
  ops.cs = as_stream(compute_stream), ops.ss = as_stream(side_stream);
  ops.pf_plan = c->st.plan_pf[(layer + 1) & 1];
  return schedule_layer(p, ops);
}

int moe_schedule_trace(int one_launch, int fused, int overlap, int pf, int shared, int hybrid,
                       int fail_at, char* h_out, int cap) {
  if (!h_out || cap < 1) return MOE_ERR_INVALID_ARG;
  LayerPlan p{one_launch != 0, fused != 0, overlap != 0, pf != 0, shared != 0, hybrid != 0};
  TraceOps ops;
  ops.fail_at = fail_at;
  const int rc = schedule_layer(p, ops);
  if ((int)ops.out.size() >= cap) return MOE_ERR_CAPACITY;
  std::memcpy(h_out, ops.out.c_str(), ops.out.size() + 1);
  return rc;
}

int moe_decode_layer_plan(moe_cache* c, int n_rows, int k, int shared, int pf, unsigned flags,
                          char* h_out, int cap) {
  if (!c || !h_out || cap < 1 || n_rows < 0 || k < 0) return MOE_ERR_INVALID_ARG;
  const LayerPlan p = plan_of(c, n_rows, k, shared != 0, pf != 0, flags);
  TraceOps ops;
  const int rc = schedule_layer(p, ops);
  if ((int)ops.out.size() >= cap) return MOE_ERR_CAPACITY;
  std::memcpy(h_out, ops.out.c_str(), ops.out.size() + 1);
  return rc;
}

int moe_hybrid_start(moe_cache* c, int n_threads) {
  if (!c || n_threads < 1 || n_threads > 256) return MOE_ERR_INVALID_ARG;
  if (c->cpu || c->d.hidden <= 0 || c->host_ptrs.empty()) return MOE_ERR_STATE;
  moe::HybridConfig hc{c->d.wfmt, c->d.hidden, c->d.inter, c->d.n_experts, c->d.n_layers,
                       c->d.max_rows, c->d.max_routes, n_threads, c->host_ptrs.data()};
  const int rc = moe::hybrid_start(hc, &c->cpu);
  if (rc <= -1000) return cuda_fail((cudaError_t)(-1000 - rc), "hybrid executor");
  return rc;
}

int moe_hybrid_stop(moe_cache* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (!c->cpu) return MOE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  moe::hybrid_stop(c->cpu);
  c->cpu = nullptr;
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "hybrid stop sync");
}

int moe_hybrid_pause(moe_cache* c, int paused) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (!c->cpu) return MOE_ERR_STATE;
  moe::hybrid_pause(c->cpu, paused != 0);
  return MOE_OK;
}

int moe_hybrid_counters(moe_cache* c, uint64_t h_out[4]) {
  if (!c || !h_out) return MOE_ERR_INVALID_ARG;
  if (!c->cpu) return MOE_ERR_STATE;
  unsigned long long v[4];
  moe::hybrid_counters(c->cpu, v);
  for (int i = 0; i < 4; ++i) h_out[i] = v[i];
  return MOE_OK;
}

int moe_read_stats(moe_cache* c, int layer, moe_stats* h_out) {
  if (check_layer(c, layer) != MOE_OK || !h_out) return MOE_ERR_INVALID_ARG;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(h_out, c->st.stats + layer, sizeof(moe_stats), cudaMemcpyDeviceToHost));
  unsigned long long dev_status = 0;
  CK(cudaMemcpy(&dev_status, c->st.status, sizeof dev_status, cudaMemcpyDeviceToHost));
  h_out->status_bits |= dev_status;
  return MOE_OK;
}

int moe_device_views(moe_cache* c, moe_views* v) {
  if (!c || !v) return MOE_ERR_INVALID_ARG;
  const DevState& st = c->st;
  v->map = st.map;
  v->slot_key = st.slot_key;
  v->stamp = st.stamp;
  v->pinned = st.pinned;
  v->clock = st.clock;
  v->decode_freq = st.decode_freq;
  v->demand_freq = st.demand_freq;
  v->last_demand = st.last_demand;
  v->stats = st.stats;
  v->plan_demand = st.plan_demand;
  v->plan_prefetch = st.plan_pf[c->last_pf_layer & 1];
  v->groups = st.groups;
  v->n_pools = c->P;
  return MOE_OK;
}

int moe_cache_set_wide_path(moe_cache* c, int mode) {
  if (!c || mode < MOE_WIDE_AUTO || mode > MOE_WIDE_TENSOR_CORES) return MOE_ERR_INVALID_ARG;
  c->wide_mode = mode;
  return MOE_OK;
}

int moe_cache_fail_next_gather(moe_cache* c, int n) {
  if (!c || n < 0) return MOE_ERR_INVALID_ARG;
  c->fail_gathers = n;
  return MOE_OK;
}

}  // extern "C"
