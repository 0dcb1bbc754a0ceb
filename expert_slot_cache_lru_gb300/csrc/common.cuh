// common.cuh -- device-side state of the slot cache, block-wide primitives and
// the kernel launchers shared by the translation units of libmoecache.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/moe_cache.h"

namespace moe {

// Raises kern's dynamic shared-memory limit to `bytes` and never lowers it: the
// limit belongs to the kernel, not to a cache, so a cache created later with
// smaller shapes must leave an earlier cache's launches valid.  The caller
// holds moe_cache_create's setup lock (the read and the write are not atomic).
// (The default limit is 48 KiB less the kernel's static shared memory.)
template <typename K>
inline cudaError_t raise_smem_limit(K kern, size_t bytes) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess || (size_t)fa.maxDynamicSharedSizeBytes >= bytes) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Everything a kernel needs to reach the cache state; passed by value.
struct DevState {
  int L, E, S, P;          // layers, experts per layer, slots per pool, pools
  int per_layer;           // 1: pool = layer, 0: one shared pool
  int32_t* map;            // [L*E] key -> slot, -1 = not resident
  uint32_t* decode_freq;   // [L*E]
  uint32_t* demand_freq;   // [L*E]
  uint64_t* last_demand;   // [L*E]
  int32_t* slot_key;       // [P*S] slot -> key, -1 = empty
  uint64_t* stamp;         // [P*S] 0 = empty
  uint8_t* pinned;         // [P*S]
  uint64_t* clock;         // [P]
  moe_stats* stats;        // [L]
  int32_t* plan_demand;    // [1 + 3*max_routes]
  int32_t* plan_pf[2];     // [1 + 3*max(max_pred,1)] each; a prefetch for layer l uses
                           // buffer l & 1, so the gather of one layer's prefetch can still
                           // be reading its plan while the next layer's prefetch is admitted
  int32_t* groups;         // [1 + max_routes + (max_routes+1) + max_routes]
  // victim-selection scratch, [vcap] each
  int32_t* vict;
  uint64_t* lo_stamp;
  int32_t* lo_slot;
  int vcap;
  const uint8_t* const* host_blob;  // [L*E] device-visible addresses of the host blobs
  uint8_t* slots;          // slot storage (NULL: admission only)
  size_t stride;           // bytes between slots
  size_t slot_bytes;       // bytes copied per expert
  int max_routes, max_pred;
  unsigned long long* status;  // device status word (MOE_STATUS_* bits not tied to a layer)
};

__host__ __device__ inline int pool_of(const DevState& st, int layer) {
  return st.per_layer ? layer : 0;
}

constexpr int kAdmitThreads = 1024;  // admission / prefetch: one CTA of 32 warps

// ---------------------------------------------------------------- block helpers
// All helpers are called by every thread of [0, NT) (NT a multiple of 32, at
// most 1024) and synchronise those threads alone (named barrier 1), so a block
// may hold more warps that never take part.

template <int NT>
__device__ __forceinline__ void sync_nt() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

struct BlockScratch {
  int warp_i[32];
  unsigned long long warp_u[32];
  unsigned long long warp_v[32];
};

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive prefix sum over the block in thread order; *total receives the sum.
template <int NT = kAdmitThreads>
__device__ __forceinline__ int block_excl_scan(int v, BlockScratch& bs, int* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) bs.warp_i[w] = incl;
  sync_nt<NT>();
  if (w == 0) {
    int t = lane < NW ? bs.warp_i[lane] : 0;
    t = warp_incl_scan(t);
    bs.warp_i[lane] = t;
  }
  sync_nt<NT>();
  const int excl = incl - v + (w > 0 ? bs.warp_i[w - 1] : 0);
  *total = bs.warp_i[NW - 1];
  sync_nt<NT>();
  return excl;
}

template <int NT = kAdmitThreads>
__device__ __forceinline__ int block_sum(int v, BlockScratch& bs) {
  int total;
  (void)block_excl_scan<NT>(v, bs, &total);
  return total;
}

// Block-wide min and max of 64-bit values.
template <int NT = kAdmitThreads>
__device__ __forceinline__ void block_minmax_u64(unsigned long long mn, unsigned long long mx,
                                                 BlockScratch& bs, unsigned long long* omin,
                                                 unsigned long long* omax) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
    unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  if (lane == 0) {
    bs.warp_u[w] = mn;
    bs.warp_v[w] = mx;
  }
  sync_nt<NT>();
  if (w == 0) {
    mn = lane < NW ? bs.warp_u[lane] : ~0ull;
    mx = lane < NW ? bs.warp_v[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
      unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
      mn = a < mn ? a : mn;
      mx = b > mx ? b : mx;
    }
    if (lane == 0) {
      bs.warp_u[0] = mn;
      bs.warp_v[0] = mx;
    }
  }
  sync_nt<NT>();
  *omin = bs.warp_u[0];
  *omax = bs.warp_v[0];
  sync_nt<NT>();
}

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of the launch.

size_t admit_smem_bytes(int E, int S);
bool admit_cached(int E, int S);  // the admission keeps the pool in shared memory
cudaError_t launch_admit(const DevState& st, int layer, const int32_t* ids, int32_t* out, int R,
                         int cap, cudaStream_t s);
cudaError_t launch_prefetch(const DevState& st, int layer, const int32_t* pred, int n,
                            int32_t* plan, cudaStream_t s);
cudaError_t launch_gather(const DevState& st, const int32_t* plan, int grid, cudaStream_t s);
cudaError_t launch_rollback(const DevState& st, const int32_t* plan, cudaStream_t s);
cudaError_t launch_pin(const DevState& st, int layer, int slot, int pinned, cudaStream_t s);

// Expert math (gemv.cu).
struct FfnScratch {
  float* h;         // [max_routes * I] routed intermediate
  float* hs;        // [max_rows * Is] shared intermediate
  float* gate;      // [max_rows] sigmoid gate of the shared expert
  float* ys;        // [max_rows * H] shared expert output (gated)
  unsigned long long* bar;  // grid-barrier counter of the fused FFN kernel (only grows)
  uint16_t* x16;    // [max_rows * H] x prepared for the grouped kernels
  float* xinv;      // [max_rows] inverse of the per-row x scale
  float* y;         // [max_routes * H] per-route down projections (grouped path)
  uint16_t* h16;    // [max_routes * I] h as f16 for the tensor-core down GEMM
  float* hinv;      // [max_routes] inverse of each route's h scale
  int32_t* dense;   // [1 + max_routes] the groups the tensor-core kernels take: count, ids
  int* gdone;       // [max_routes] pieces of each demand-plan expert copied by a fused layer
  float* la_z;      // [max_rows][n_experts] the look-ahead producer's router logits
  unsigned* la_ctr; // its CTAs done (zero between launches)
  // a fused layer with the admission inside the launch (three counters that only grow)
  unsigned long long* epoch;   // launches (each CTA adds one)
  unsigned long long* pseq;    // the admission's publication sequence
  unsigned long long* bar2;    // grid barrier of the computing CTAs
  unsigned long long* sslot;   // [max_routes] per miss rank: (2j+1) << 32 | slot (~0u: none)
  uint8_t* stage;              // [stage_n] slot-sized areas the step's misses are copied into
  int stage_n;
};

cudaError_t launch_shared_expert(int wfmt, int H, int Is, const void* x, int n_rows,
                                 const uint8_t* blob, const void* gate_w, FfnScratch sc,
                                 cudaStream_t s);
cudaError_t launch_routed_up(const DevState& st, int wfmt, int H, int I, int layer,
                             const void* x, const int32_t* slot_ids, int n_rows, int k,
                             FfnScratch sc, cudaStream_t s);
cudaError_t launch_routed_down_combine(const DevState& st, int wfmt, int H, int I, int layer,
                                       const int32_t* slot_ids, const float* w, int n_rows,
                                       int k, const float* shared_y, void* out, FfnScratch sc,
                                       cudaStream_t s);

// Streaming expert FFNs for decode-sized steps (ffn_stream.cu).
bool ffn_stream_supported(int wfmt, int H, int I, int n_rows, int n_tasks);
cudaError_t ffn_stream_init();

// The look-ahead producer (lookahead.cu).
bool lookahead_supported(int H, int E, int k);
cudaError_t lookahead_init(int H);
cudaError_t launch_lookahead(const void* x, const void* router, int n_rows, int H, int E, int k,
                             float* z, unsigned* ctr, int32_t* pred, cudaStream_t s);
cudaError_t launch_shared_stream(const DevState& st, int wfmt, int H, int Is, const void* x,
                                 int n_rows, const uint8_t* blob, const void* gate_w,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s);
cudaError_t launch_routed_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                 const void* x, const int32_t* slot_ids, const float* w,
                                 int n_rows, int k, const float* shared_y, void* out,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s);

// One launch for a whole decode-sized layer after its admission: the demand
// (and prefetch) gather, the shared expert and the routed experts (ffn_stream.cu).
bool layer_stream_supported(int wfmt, int H, int I, int n_rows, int k, bool shared);
cudaError_t launch_layer_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                const void* x, const int32_t* slot_ids, const float* w,
                                int n_rows, int k, const uint8_t* shared_blob,
                                const void* gate_w, const int32_t* plan0, const int32_t* plan1,
                                void* out, FfnScratch sc, unsigned long long* status,
                                cudaStream_t s);

// One launch for a whole decode-sized layer including its admission: CTA 0
// admits (and prefetch-admits layer + 1 when pred is given) while the other
// CTAs stream the resident experts; the rest as launch_layer_stream.
bool layer_admit_supported(const DevState& st, int wfmt, int H, int I, int n_rows, int k,
                           bool shared);
cudaError_t launch_layer_admit(const DevState& st, int wfmt, int H, int I, int layer,
                               const void* x, const int32_t* ids, int32_t* slot_out,
                               const float* w, int n_rows, int k, int cap, const int32_t* pred,
                               int n_pred, const uint8_t* shared_blob, const void* gate_w,
                               int32_t* plan1, void* out, FfnScratch sc,
                               unsigned long long* status, cudaStream_t s);

// Routed FFNs for wide steps, grouped by expert (grouped.cu).
bool grouped_supported(int wfmt, int H, int I, int E);
cudaError_t grouped_init(int E, int H, int I);
cudaError_t launch_routed_grouped(const DevState& st, int wfmt, int H, int I, int layer,
                                  const void* x, const int32_t* slot_ids, const float* w,
                                  int n_rows, int k, const float* shared_y, void* out,
                                  FfnScratch sc, int max_routes, int wide_mode,
                                  cudaStream_t s);

// The gate/up and down GEMMs of the grouped path on the tensor cores
// (grouped_tc.cu): NVFP4 experts with H and I multiples of 128, for the groups
// group_kernel lists (FfnScratch::dense).  One tcgen05.mma (M 128, K 16) takes about
// 100 cycles to issue whatever its N, i.e. ~20 fp4 weights per cycle per SM,
// half of what HBM delivers to an SM; the CUDA-core kernels reread nothing and
// win while a group has few routes.  In the automatic mode groups of at least
// kTcMinRoutes routes go to the tensor cores and the rest to the CUDA cores (4
// measured best of 3, 4, 6, 8, 12, 16 and 24 on the wide step's Zipf and
// uniform routings).
constexpr int kTcMinRoutes = 4;
bool grouped_tc_supported(int wfmt, int H, int I);
cudaError_t grouped_tc_init();
cudaError_t launch_grouped_tc(const DevState& st, int H, int I, int layer, int k, int n_routes,
                              int max_routes, FfnScratch sc, unsigned long long* status,
                              cudaStream_t s);

// Allocation-free routed FFN (ffn_stream.cu): the scratch is a file-scope
// device array whose address noalloc_scratch looks up once per device.
cudaError_t noalloc_scratch(void** out);
cudaError_t launch_routed_noalloc(int wfmt, int H, int I, const uint8_t* slots, size_t stride,
                                  int n_slots, const void* x, const int32_t* slot_ids,
                                  const float* w, int n_rows, int k, void* out,
                                  unsigned long long* status, void* scratch, cudaStream_t s);

// The hybrid CPU executor (hybrid.cu): a host thread pool computing the
// routes left at -1, fed and joined through a mailbox in mapped host memory.
struct HybridConfig {
  int wfmt, H, I, E, L, max_rows, max_routes, n_threads;
  const void* const* host_blobs;  // [L*E] host addresses of the expert blobs
};
int hybrid_start(const HybridConfig& c, moe_cpu_exec** out, bool host_only = false);  // MOE_OK, MOE_ERR_*, or
                                                               // -1000 - cudaError_t
void hybrid_stop(moe_cpu_exec* x);
void hybrid_counters(const moe_cpu_exec* x, unsigned long long out[4]);
void hybrid_pause(moe_cpu_exec* x, bool paused);
cudaError_t hybrid_post(moe_cpu_exec* x, int layer, const int32_t* ids, const int32_t* slots,
                        const float* w, const void* xin, int n_rows, int k, cudaStream_t s);
cudaError_t hybrid_add(moe_cpu_exec* x, void* out, int n_rows, unsigned long long* status,
                       cudaStream_t s);

}  // namespace moe
