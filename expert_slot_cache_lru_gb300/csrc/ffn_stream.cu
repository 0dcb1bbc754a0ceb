// ffn_stream.cu -- expert FFNs for decode-sized steps, streamed through
// shared memory with bulk asynchronous copies.
//
// What is computed is the same as gemv.cu (FreeToken issue #753 "[Perf]
// Offloaded decode: overlap the expert-miss gather with the same layer's
// shared expert ...", Problem and What we changed: routed experts over the
// slots, a sigmoid-gated shared expert, routed + shared); this file is the
// fast path when every (route, row) of the step fits a small task list.
//
// A decode step moves ~14 MB of weights per layer, which the HBM delivers in
// ~2 us, so the kernel must have megabytes in flight almost at once.  One
// cooperative launch of one CTA per SM computes a whole group of expert FFNs:
// gate/up rows (phase A), a grid-wide barrier, then down rows and the combine
// (phase B).  A producer warp streams the weight rows of both phases through
// a ring of shared-memory stages with cp.async.bulk (completion on per-stage
// mbarriers), so phase-B weights land while phase A computes; sixteen
// consumer warps decode the stages as they land.
//
// Every wait (mbarrier, grid barrier) is bounded (%globaltimer); on a timeout
// the kernel sets MOE_STATUS_TIMEOUT in the cache's device status word, skips
// the remaining work, drains its own copies (again bounded) and returns.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kSW = 16;            // warps per CTA
constexpr int kST = 32 * kSW;      // threads per CTA
constexpr int kMaxStages = 8;      // ring depth
constexpr int kMaxTasks = 64;      // routes per call on this path
constexpr int kXW = 4;             // x words (8 bf16 each) held per consumer thread
constexpr int kYsPre = 2;          // shared-expert outputs prefetched per consumer thread
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_one(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most n of this thread's most recent groups are still pending (n <= 7)
__device__ __forceinline__ void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}
// cooperative copy of `bytes` (multiple of 16) by kST threads, 16 bytes each
__device__ __forceinline__ void copy_async(uint8_t* dst, const uint8_t* src, uint32_t bytes) {
  for (uint32_t o = threadIdx.x * 16; o < bytes; o += kST * 16) cp_async16(dst + o, src + o);
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  while (!mbar_test(bar, parity)) {
    if (now_ns() - t0 > kWaitNs) return false;
  }
  return true;
}

// ------------------------------------------------------------ decode helpers
// NVFP4 decode uses the hardware conversions: cvt.rn.f16x2.e2m1x2 (two FP4
// E2M1 codes of one byte to two exact halves, the low nibble in the low half)
// and cvt.rn.f16x2.e4m3x2 (two FP8 E4M3 block scales).  Products are formed
// exactly: gate/up as fma.rn.f32.f16 (half x half, fp32 accumulate) with x
// held in f16, down as fp32 FMAs with the fp32 intermediate h.

template <int B>
__device__ __forceinline__ uint32_t e2m1x2_h2(uint32_t w) {
  uint32_t h2;
  if (B == 0)
    asm("{ .reg .b8 b0,b1,b2,b3; mov.b32 {b0,b1,b2,b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b0; }"
        : "=r"(h2) : "r"(w));
  else if (B == 1)
    asm("{ .reg .b8 b0,b1,b2,b3; mov.b32 {b0,b1,b2,b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b1; }"
        : "=r"(h2) : "r"(w));
  else if (B == 2)
    asm("{ .reg .b8 b0,b1,b2,b3; mov.b32 {b0,b1,b2,b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b2; }"
        : "=r"(h2) : "r"(w));
  else
    asm("{ .reg .b8 b0,b1,b2,b3; mov.b32 {b0,b1,b2,b3}, %1; cvt.rn.f16x2.e2m1x2 %0, b3; }"
        : "=r"(h2) : "r"(w));
  return h2;
}
// the two halves of a half2 word as fp32 (exact)
__device__ __forceinline__ float2 h2_f32(uint32_t h2) {
  float a, b;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
      : "=f"(a), "=f"(b) : "r"(h2));
  return make_float2(a, b);
}
// two FP8 E4M3 scales (low byte first) as fp32
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t v16) {
  uint32_t h2;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(h2)
      : "r"(v16));
  return h2_f32(h2);
}
// c + w.lo * x.lo + w.hi * x.hi, half operands, fp32 result (exact products)
__device__ __forceinline__ float fma2_h(uint32_t w2, uint32_t x2, float c) {
  float d;
  asm("{ .reg .b16 a0, a1, b0, b1; .reg .f32 t;\n"
      " mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.f16 t, a0, b0, %3;\n fma.rn.f32.f16 %0, a1, b1, t; }"
      : "=f"(d) : "r"(w2), "r"(x2), "f"(c));
  return d;
}
// same with bfloat16 operands
__device__ __forceinline__ float fma2_bf(uint32_t w2, uint32_t x2, float c) {
  float d;
  asm("{ .reg .b16 a0, a1, b0, b1; .reg .f32 t;\n"
      " mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.bf16 t, a0, b0, %3;\n fma.rn.f32.bf16 %0, a1, b1, t; }"
      : "=f"(d) : "r"(w2), "r"(x2), "f"(c));
  return d;
}
// sum_{i<8} e2m1(nibble i of w) * x[i], x as four half2 words (exact products)
__device__ __forceinline__ float dot8_fp4_h(uint32_t w, uint4 x) {
  float a = fma2_h(e2m1x2_h2<0>(w), x.x, 0.f);
  a = fma2_h(e2m1x2_h2<1>(w), x.y, a);
  a = fma2_h(e2m1x2_h2<2>(w), x.z, a);
  return fma2_h(e2m1x2_h2<3>(w), x.w, a);
}
// sum_{i<8} e2m1(nibble i of w) * h[i], h fp32
__device__ __forceinline__ float dot8_fp4_f(uint32_t w, const float* h) {
  float2 f = h2_f32(e2m1x2_h2<0>(w));
  float a = fmaf(f.x, h[0], f.y * h[1]);
  f = h2_f32(e2m1x2_h2<1>(w));
  a = fmaf(f.x, h[2], fmaf(f.y, h[3], a));
  f = h2_f32(e2m1x2_h2<2>(w));
  a = fmaf(f.x, h[4], fmaf(f.y, h[5], a));
  f = h2_f32(e2m1x2_h2<3>(w));
  return fmaf(f.x, h[6], fmaf(f.y, h[7], a));
}
// sum_{i<8} e2m1(nibble i of w) * h[i] with h given as f16 hi + lo parts
// (h = hi + lo to ~22 bits); products exact, fp32 accumulate
__device__ __forceinline__ float dot8_fp4_hl(uint32_t w, const uint32_t* hi, const uint32_t* lo) {
  const uint32_t c0 = e2m1x2_h2<0>(w), c1 = e2m1x2_h2<1>(w), c2 = e2m1x2_h2<2>(w),
                 c3 = e2m1x2_h2<3>(w);
  float a = fma2_h(c0, hi[0], 0.f), b = fma2_h(c0, lo[0], 0.f);
  a = fma2_h(c1, hi[1], a);
  b = fma2_h(c1, lo[1], b);
  a = fma2_h(c2, hi[2], a);
  b = fma2_h(c2, lo[2], b);
  a = fma2_h(c3, hi[3], a);
  b = fma2_h(c3, lo[3], b);
  return a + b;
}
// sum_{i<8} bf16 weights (uint4) * bf16 x (uint4), fp32
__device__ __forceinline__ float dot8_bf16_bf(uint4 w, uint4 x, float a) {
  a = fma2_bf(w.x, x.x, a);
  a = fma2_bf(w.y, x.y, a);
  a = fma2_bf(w.z, x.z, a);
  return fma2_bf(w.w, x.w, a);
}
// sum_{i<8} bf16 weights (uint4) * fp32 h[i]
__device__ __forceinline__ float dot8_bf16_f(uint4 v, const float* x, float a) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a = fmaf(__uint_as_float(w[i] << 16), x[2 * i], a);
    a = fmaf(__uint_as_float(w[i] & 0xffff0000u), x[2 * i + 1], a);
  }
  return a;
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Offsets inside a blob (layout of moe_cache.h).
struct BlobOff {
  size_t code[3], scale[3], glob;  // NVFP4
  size_t mat[3];                   // bf16
  __device__ BlobOff(int H, int I) {
    const size_t ih = (size_t)I * H;
    code[0] = 0;
    code[1] = ih / 2;
    code[2] = ih;
    scale[0] = 3 * ih / 2;
    scale[1] = scale[0] + ih / 16;
    scale[2] = scale[1] + ih / 16;
    glob = scale[2] + ih / 16;
    mat[0] = 0;
    mat[1] = ih * 2;
    mat[2] = ih * 4;
  }
};

// Per-call task list, identical in every CTA: the valid routes in route order,
// with each task's blob, routing weight and fp32 global scales staged in
// shared memory so the compute loops never wait on a global load.
struct Tasks {
  int n;
  int route[kMaxTasks];  // route index r = b*k + j
  const uint8_t* blob[kMaxTasks];
  float wt[kMaxTasks];   // routing weight (1 for the shared expert)
  float gs[kMaxTasks][3];  // NVFP4 global scales of gate, up, down (1 for bf16)
  int valid[kMaxTasks];
};

// Step 1 (threads r < R, one global round trip): which routes have a slot.
// Step 2 (after a __syncthreads): compaction by a prefix count.
// Step 3 (after a __syncthreads): weights and global scales, in parallel.
__device__ void tasks_load(Tasks& tk, const DevState& st, int layer, const int32_t* slot_ids,
                           int R, const uint8_t* fixed_blob) {
  const int r = threadIdx.x;
  if (r < R) {
    const uint8_t* b = fixed_blob;
    if (!b) {
      const int s = slot_ids[r];
      b = (unsigned)s < (unsigned)st.S
              ? st.slots + ((size_t)pool_of(st, layer) * st.S + s) * st.stride
              : nullptr;
    }
    tk.valid[r] = b != nullptr;
    tk.blob[r] = b;  // temporarily indexed by route
  }
}
__device__ void tasks_compact(Tasks& tk, int R) {
  const int r = threadIdx.x;
  const uint8_t* b = r < R ? tk.blob[r] : nullptr;
  int pos = 0;
  if (r < R && tk.valid[r])
    for (int q = 0; q < r; ++q) pos += tk.valid[q];
  __syncthreads();
  if (r < R && tk.valid[r]) {
    tk.route[pos] = r;
    tk.blob[pos] = b;
  }
  if (r == 0) {
    int n = 0;
    for (int q = 0; q < R; ++q) n += tk.valid[q];
    tk.n = n;
  }
}
__device__ void flag_timeout(unsigned long long* status) {
  if (status) atomicOr(status, (unsigned long long)MOE_STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- pipeline
// A CTA walks a list of chunks; a chunk is `rc` consecutive rows of one
// task's matrix (gate+up for the gate/up kernel, down for the down kernel),
// copied with one cp.async.bulk per bank (codes, scales) into a ring stage.
// Warp kSW (the producer) issues the copies; the kSW consumer warps split the
// chunk into rc rows x (kSW / rc) slices of the reduction dimension, combine
// the slices of each row through shared memory in a fixed order, and release
// the stage.  full[s] completes on the copies' bytes, empty[s] on release.

struct Ring {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
};

// The producer's last act: wait (bounded) until every chunk it issued has
// landed, so no copy is still writing shared memory when the CTA exits.
__device__ void producer_drain(Ring& rg, int nstage, int issued) {
  for (int c = issued - nstage < 0 ? 0 : issued - nstage; c < issued; ++c)
    mbar_wait(&rg.full[c % nstage], (uint32_t)((c / nstage) & 1));
}

// Named barrier among the consumer warps only (the producer does not take part).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kSW * 32) : "memory");
}

// rows per chunk: the largest power of two <= 16 whose stage fits `cap` bytes
__host__ __device__ inline int rows_per_chunk(int row_bytes, int cap) {
  int rc = 16;
  while (rc > 1 && rc * row_bytes > cap) rc >>= 1;
  return rc;
}

// ---------------------------------------------------------------- grid barrier
// One CTA per SM, launched cooperatively, so every CTA of the grid is resident.
// `ctr` only grows: each launch adds gridDim.x, and a CTA waits until the count
// reaches the next multiple of gridDim.x.  Release/acquire at GPU scope orders
// the h written before the barrier with the reads after it.  Bounded spin.
__device__ bool grid_barrier(unsigned long long* ctr, unsigned long long* status) {
  __shared__ int s_ok;
  consumers_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned long long old;
    asm volatile("atom.add.release.gpu.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
    const unsigned long long target = (old / gridDim.x + 1) * gridDim.x;
    unsigned long long v = 0;
    const unsigned long long t0 = now_ns();
    int ok = 1;
    for (;;) {
      asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (now_ns() - t0 > kWaitNs) {
        flag_timeout(status);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    s_ok = ok;
  }
  consumers_sync();
  return s_ok != 0;
}

// ---------------------------------------------------------------- fused FFN
// One launch computes a group of expert FFNs for a decode-sized step:
//   phase A (gate/up): rows u of the flattened (task, n) list,
//       h[route][n] = silu(W_g x_b)[n] * (W_u x_b)[n];
//   grid barrier;
//   phase B (down + combine): output rows (b, n),
//       SHARED: ys[b][n] = sigmoid(x_b . w_g) * (W_d h_b)[n]
//       ROUTED: out[b][n] = bf16( sum_j w[b,j] (W_d[slot] h_bj)[n] + ys[b][n] ).
// The producer warp streams the chunks of both phases through one ring of
// stages with cp.async.bulk: phase-B weights arrive during phase A and the
// barrier; after the barrier only h (a few KB, from L2) is read.
//
// Phase A chunk: rcA consecutive rows of one task, gate and up banks.
// Phase B chunk: rcB rows of one batch row b for a group of up to tpc of b's
// tasks.  Consumer warps split a chunk into (task, K slice, row) items, keep
// their slice of x (A) or h (B) in registers, read weights with lane-contiguous
// loads, and combine slice partials through shared memory in a fixed order.
//
// x is staged once per CTA: as f16 for NVFP4 experts (products e2m1 * x exact
// halves-times-halves), scaled per row by a power of two so that max |x| < 2^15
// -- a bf16 value converts to f16 exactly in that range, and the scale is undone
// on the fp32 sums -- or as bf16 for bf16 experts.
struct FusedArgs {
  int H, I, layer, k, R, n_rows;
  const uint16_t* x;
  const int32_t* slot_ids;
  const uint8_t* fixed_blob;   // shared expert blob (SHARED) or null
  const float* w;              // routing weights (ROUTED)
  float* h;                    // [R][I] intermediate
  const uint16_t* gate_w;      // SHARED: gate vector
  float* gate;                 // SHARED: sigmoid gate per row (scratch)
  float* ys;                   // SHARED: output [n_rows][H]; ROUTED: input (may be null)
  __nv_bfloat16* out;          // ROUTED output
  int nstage, stage_bytes, rcA, rcB, tpc;
  unsigned long long* status;
  unsigned long long* bar_ctr;
};

template <int FMT, bool SHARED>
__global__ void __launch_bounds__(kST + 32, 1)
ffn_fused_kernel(DevState st, FusedArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Tasks tk;
  __shared__ Ring rg;
  __shared__ unsigned int xmax[16];  // per row max |x| (float bits, only when > 2^14)
  __shared__ float xscale[16];       // per row power-of-two scale applied to x
  __shared__ float xinv[16];         // per row 1 / scale
  __shared__ float gate_s[16];
  __shared__ int ts[17];             // tasks of batch row b: [ts[b], ts[b+1])
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, k = a.k, n_rows = a.n_rows;

  const int rowB = FMT == MOE_W_NVFP4 ? I / 2 + I / 16 : I * 2;            // down row bytes
  const int nslA = H / 1024, nslB = I / 512;
  const int rcA = a.rcA, rcB = a.rcB, tpc = a.tpc, nstage = a.nstage;

  // ---- prologue: one global round trip for the routes' slots and all of x
  const int nx8 = n_rows * H / 8;
  uint4 xw[kXW];
  if (threadIdx.x < 16) xmax[threadIdx.x] = 0u;
  tasks_load(tk, st, a.layer, a.slot_ids, a.R, a.fixed_blob);
#pragma unroll
  for (int j = 0; j < kXW; ++j) {
    const int i = threadIdx.x + j * kST;
    if (threadIdx.x < kST && i < nx8) xw[j] = reinterpret_cast<const uint4*>(a.x)[i];
  }
  __syncthreads();
  if (FMT == MOE_W_NVFP4) {
#pragma unroll
    for (int j = 0; j < kXW; ++j) {
      const int i = threadIdx.x + j * kST;
      if (threadIdx.x >= kST || i >= nx8) continue;
      const uint32_t wv[4] = {xw[j].x, xw[j].y, xw[j].z, xw[j].w};
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wv[e] << 16)),
                             fabsf(__uint_as_float(wv[e] & 0xffff0000u))));
      if (mx > 16384.f) atomicMax(&xmax[(i * 8) / H], __float_as_uint(mx));
    }
  }
  tasks_compact(tk, a.R);
  if (threadIdx.x == 0) {
    for (int q = 0; q < nstage; ++q) {
      mbar_init(&rg.full[q], 1);
      mbar_init(&rg.empty[q], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int T = tk.n;
  if (threadIdx.x <= n_rows) {  // first task of each batch row (tasks are b-major)
    int t = 0;
    while (t < T && tk.route[t] / k < (int)threadIdx.x) ++t;
    ts[threadIdx.x] = t;
  }
  __syncthreads();

  // phase A rows of this CTA
  const int UA = T * I;
  const int perA = (UA + gridDim.x - 1) / gridDim.x;
  const int u0 = min(UA, perA * blockIdx.x), u1 = min(UA, u0 + perA);
  // phase B output rows of this CTA
  const int UB = n_rows * H;
  const int perB = (UB + gridDim.x - 1) / gridDim.x;
  const int ru0 = min(UB, perB * blockIdx.x), ru1 = min(UB, ru0 + perB);

  // shared memory: x | h [T][I] | y [T][perB] | redA [2][2][nslA*rcA] | redB [2][tpc*nslB*rcB] | ring
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);
  float* hsm = reinterpret_cast<float*>(sm + ((size_t)n_rows * H * 2 + 127) / 128 * 128);
  float* ysm = hsm + (size_t)T * I;
  float* redA = ysm + (size_t)T * perB;
  const int redA_n = nslA * rcA;
  float* redB = redA + 4 * redA_n;
  const int redB_n = tpc * nslB * rcB;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(redB + 2 * redB_n) + 127) / 128 * 128);
  const BlobOff o(H, I);

  // phase B chunk cursor: (b, row block n, task group t0); rows without tasks skipped
  struct Cur {
    int b, n, t0;
  };
  auto b_lo = [&](int b) { return max(ru0 - b * H, 0); };
  auto b_hi = [&](int b) { return min(ru1 - b * H, H); };
  auto settle = [&](Cur& c) -> bool {
    while (c.b * H < ru1) {
      if (ts[c.b] < ts[c.b + 1] && c.n < b_hi(c.b)) {
        if (c.t0 < ts[c.b]) c.t0 = ts[c.b];
        if (c.t0 < ts[c.b + 1]) return true;
        c.t0 = ts[c.b];
        c.n += rcB;
        continue;
      }
      ++c.b;
      if (c.b * H >= ru1) return false;
      c.n = b_lo(c.b);
      c.t0 = ts[c.b];
    }
    return false;
  };
  auto advance = [&](Cur& c) -> bool {
    c.t0 += tpc;
    return settle(c);
  };
  auto start = [&](Cur& c) -> bool {
    if (ru0 >= ru1) return false;
    c.b = ru0 / H;
    c.n = b_lo(c.b);
    c.t0 = ts[c.b];
    return settle(c);
  };

  if (warp == kSW) {  // ================================================ producer
    if (lane == 0) {
      int q = 0;
      bool ok = true;
      auto acquire = [&](int& s) -> bool {  // next stage, free
        s = q % nstage;
        if (q >= nstage && !mbar_wait(&rg.empty[s], (uint32_t)(((q / nstage) - 1) & 1))) {
          flag_timeout(a.status);
          return false;
        }
        fence_proxy_async();
        return true;
      };
      for (int u = u0; u < u1 && ok;) {  // phase A
        const int t = u / I, n = u - t * I;
        const int nr = min(rcA, min(u1 - u, I - n));
        int s;
        if (!(ok = acquire(s))) break;
        uint8_t* dst = ring + (size_t)s * a.stage_bytes;
        const uint8_t* blob = tk.blob[t];
        if (FMT == MOE_W_NVFP4) {
          const uint32_t cb = nr * (H / 2), sb = nr * (H / 16);
          mbar_expect_tx(&rg.full[s], 2 * (cb + sb));
          bulk_g2s(dst, blob + o.code[0] + (size_t)n * (H / 2), cb, &rg.full[s]);
          bulk_g2s(dst + rcA * (H / 2), blob + o.code[1] + (size_t)n * (H / 2), cb, &rg.full[s]);
          bulk_g2s(dst + 2 * rcA * (H / 2), blob + o.scale[0] + (size_t)n * (H / 16), sb, &rg.full[s]);
          bulk_g2s(dst + 2 * rcA * (H / 2) + rcA * (H / 16), blob + o.scale[1] + (size_t)n * (H / 16), sb,
                   &rg.full[s]);
        } else {
          const uint32_t rb = nr * H * 2;
          mbar_expect_tx(&rg.full[s], 2 * rb);
          bulk_g2s(dst, blob + o.mat[0] + (size_t)n * H * 2, rb, &rg.full[s]);
          bulk_g2s(dst + (size_t)rcA * H * 2, blob + o.mat[1] + (size_t)n * H * 2, rb, &rg.full[s]);
        }
        ++q;
        u += nr;
      }
      Cur c;
      for (bool more = ok && start(c); more; more = advance(c)) {  // phase B
        const int nr = min(rcB, b_hi(c.b) - c.n);
        const int t1 = min(c.t0 + tpc, ts[c.b + 1]);
        int s;
        if (!acquire(s)) break;
        uint8_t* dst = ring + (size_t)s * a.stage_bytes;
        mbar_expect_tx(&rg.full[s], (t1 - c.t0) * nr * rowB);
        for (int t = c.t0; t < t1; ++t) {  // stage: task-major, each task rcB rows
          uint8_t* d = dst + (size_t)(t - c.t0) * rcB * rowB;
          const uint8_t* blob = tk.blob[t];
          if (FMT == MOE_W_NVFP4) {
            bulk_g2s(d, blob + o.code[2] + (size_t)c.n * (I / 2), nr * (I / 2), &rg.full[s]);
            bulk_g2s(d + rcB * (I / 2), blob + o.scale[2] + (size_t)c.n * (I / 16), nr * (I / 16),
                     &rg.full[s]);
          } else {
            bulk_g2s(d, blob + o.mat[2] + (size_t)c.n * I * 2, nr * I * 2, &rg.full[s]);
          }
        }
        ++q;
      }
      producer_drain(rg, nstage, q);
    }
    return;
  }

  // ================================================================ consumers
  // per-task constants: loads issued now, stored to shared memory before use
  float cg0 = 1.f, cg1 = 1.f, cg2 = 1.f, cw = 1.f;
  if (threadIdx.x < T) {
    if (!SHARED) cw = a.w[tk.route[threadIdx.x]];
    if (FMT == MOE_W_NVFP4) {
      const float* gp = reinterpret_cast<const float*>(tk.blob[threadIdx.x] + o.glob);
      cg0 = gp[0];
      cg1 = gp[1];
      cg2 = gp[2];
    }
  }
  if (threadIdx.x < n_rows) {
    float sc = 1.f;  // power of two bringing max |x| below 2^15
    const float mx = __uint_as_float(xmax[threadIdx.x]);
    while (mx * sc >= 32768.f) sc *= 0.5f;
    xscale[threadIdx.x] = sc;
    xinv[threadIdx.x] = 1.f / sc;
  }
  consumers_sync();
#pragma unroll
  for (int j = 0; j < kXW; ++j) {  // x into shared memory (f16 for NVFP4, bf16 otherwise)
    const int i = threadIdx.x + j * kST;
    if (i >= nx8) continue;
    if (FMT == MOE_W_NVFP4) {
      const float sc = xscale[(i * 8) / H];
      const uint32_t wv[4] = {xw[j].x, xw[j].y, xw[j].z, xw[j].w};
      uint32_t hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                             __uint_as_float(wv[e] & 0xffff0000u) * sc);
        hv[e] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      reinterpret_cast<uint4*>(xs)[i] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    } else {
      reinterpret_cast<uint4*>(xs)[i] = xw[j];
    }
  }
  if (threadIdx.x < T) {
    tk.gs[threadIdx.x][0] = cg0;
    tk.gs[threadIdx.x][1] = cg1;
    tk.gs[threadIdx.x][2] = cg2;
    tk.wt[threadIdx.x] = cw;
  }
  consumers_sync();
  // the shared expert's sigmoid gate, sigmoid(x_b . w_g), in fp32
  if (SHARED && blockIdx.x == 0 && warp < n_rows) {
    float z = 0.f;
    for (int i0 = lane * 8; i0 < H; i0 += 256) {
      const uint4 gv = *reinterpret_cast<const uint4*>(a.gate_w + i0);
      const uint4 xv = *reinterpret_cast<const uint4*>(a.x + (size_t)warp * H + i0);
      z = dot8_bf16_bf(gv, xv, z);
    }
    z = wsum(z);
    if (lane == 0) a.gate[warp] = 1.f / (1.f + expf(-z));
  }

  bool failed = false;  // a timed-out wait: keep taking part in the barriers, skip the work
  int q = 0;
  // ---------------------------------------------------------------- phase A
  // items (slice sl of 1024, row r), row fastest, contiguous per warp
  //   NVFP4: lane L takes elements [32L, 32L+32) of the slice (16 code bytes)
  //   bf16:  lane L takes elements 8L + 256m + [0, 8), m = 0..3 (4 x 16 bytes)
  {
    uint4 xv[4];
    int xkey = -1;
    for (int u = u0; u < u1; ++q) {
      const int t = u / I, n = u - t * I;
      const int nr = min(rcA, min(u1 - u, I - n));
      const int s = q % nstage;
      if (!failed && !mbar_wait(&rg.full[s], (uint32_t)((q / nstage) & 1))) {
        flag_timeout(a.status);
        failed = true;
      }
      const int b = tk.route[t] / k;
      const uint8_t* stg = ring + (size_t)s * a.stage_bytes;
      float* rd = redA + (size_t)(q & 1) * 2 * redA_n;
      const int items = nslA * nr;
      const int ipw = (items + kSW - 1) / kSW;
      const int i0 = min(items, warp * ipw), i1 = min(items, i0 + ipw);
      int sl = i0 / nr, r = i0 - sl * nr;
      for (int it = i0; it < i1 && !failed; ++it, (++r == nr ? (r = 0, ++sl) : 0)) {
        if (sl * 16 + b != xkey) {  // this batch row's x slice into registers
          const uint16_t* xr = xs + (size_t)b * H + sl * 1024;
#pragma unroll
          for (int m = 0; m < 4; ++m)
            xv[m] = FMT == MOE_W_NVFP4 ? reinterpret_cast<const uint4*>(xr + lane * 32)[m]
                                       : *reinterpret_cast<const uint4*>(xr + lane * 8 + 256 * m);
          xkey = sl * 16 + b;
        }
        float g = 0.f, up = 0.f;
        if (FMT == MOE_W_NVFP4) {
          const int e0 = sl * 1024 + lane * 32;
          const uint4 cgw = *reinterpret_cast<const uint4*>(stg + (size_t)r * (H / 2) + e0 / 2);
          const uint4 cuw = *reinterpret_cast<const uint4*>(stg + (size_t)(rcA + r) * (H / 2) + e0 / 2);
          const uint8_t* sc = stg + (size_t)2 * rcA * (H / 2);
          const float2 sg = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(sc + (size_t)r * (H / 16) + e0 / 16));
          const float2 su =
              e4m3x2_f32(*reinterpret_cast<const uint16_t*>(sc + (size_t)(rcA + r) * (H / 16) + e0 / 16));
          g = fmaf(dot8_fp4_h(cgw.x, xv[0]) + dot8_fp4_h(cgw.y, xv[1]), sg.x, 0.f);
          g = fmaf(dot8_fp4_h(cgw.z, xv[2]) + dot8_fp4_h(cgw.w, xv[3]), sg.y, g);
          up = fmaf(dot8_fp4_h(cuw.x, xv[0]) + dot8_fp4_h(cuw.y, xv[1]), su.x, 0.f);
          up = fmaf(dot8_fp4_h(cuw.z, xv[2]) + dot8_fp4_h(cuw.w, xv[3]), su.y, up);
        } else {
          const uint8_t* rowg = stg + (size_t)r * H * 2 + (size_t)sl * 2048;
          const uint8_t* rowu = stg + (size_t)(rcA + r) * H * 2 + (size_t)sl * 2048;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            g = dot8_bf16_bf(*reinterpret_cast<const uint4*>(rowg + lane * 16 + 512 * m), xv[m], g);
            up = dot8_bf16_bf(*reinterpret_cast<const uint4*>(rowu + lane * 16 + 512 * m), xv[m], up);
          }
        }
        g = wsum(g);
        up = wsum(up);
        if (lane == 0) {
          rd[it] = g;
          rd[redA_n + it] = up;
        }
      }
      consumers_sync();  // every item of the chunk done, stage no longer read
      if (threadIdx.x == 0) mbar_arrive_one(&rg.empty[s]);
      if (threadIdx.x < nr && !failed) {  // one thread per row: slices in a fixed order
        const int rr = threadIdx.x;
        float gs = 0.f, us = 0.f;
        for (int z = 0; z < nslA; ++z) {
          gs += rd[z * nr + rr];
          us += rd[redA_n + z * nr + rr];
        }
        const float xi = FMT == MOE_W_NVFP4 ? xinv[b] : 1.f;
        const float gg = gs * xi * tk.gs[t][0], uu = us * xi * tk.gs[t][1];
        a.h[(size_t)tk.route[t] * I + n + rr] = gg / (1.f + expf(-gg)) * uu;
      }
      u += nr;  // rd is double-buffered: the next chunk writes the other half
    }
  }

  // ---------------------------------------------------------------- barrier
  if (!grid_barrier(a.bar_ctr, a.status)) failed = true;
  {  // every task's h into shared memory: float4 loads, four in flight per thread
    const int n4 = T * I / 4, i4 = I / 4;
    float4* hs4 = reinterpret_cast<float4*>(hsm);
    const float4* h4 = reinterpret_cast<const float4*>(a.h);
    for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * kST) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kST;
        if (i < n4) v[j] = __ldcg(&h4[(size_t)tk.route[i / i4] * i4 + (i % i4)]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i0 + j * kST < n4) hs4[i0 + j * kST] = v[j];
    }
  }
  if (SHARED && threadIdx.x < n_rows) gate_s[threadIdx.x] = __ldcg(&a.gate[threadIdx.x]);
  float ysv[kYsPre];  // the shared expert's output for this thread's combine rows
#pragma unroll
  for (int m = 0; m < kYsPre; ++m) {
    const int ru = ru0 + threadIdx.x + m * kST;
    ysv[m] = (!SHARED && a.ys && ru < ru1) ? a.ys[ru] : 0.f;
  }
  consumers_sync();

  // ---------------------------------------------------------------- phase B
  // items (task j, slice sl of 512, row r), row fastest, contiguous per warp
  //   NVFP4: lane L takes elements [16L, 16L+16) of the slice (8 code bytes)
  //   bf16:  lane L takes elements 8L + 256m + [0, 8), m = 0, 1 (2 x 16 bytes)
  {
    float hv[16];
    int hkey = -1;
    Cur c;
    for (bool more = start(c); more; more = advance(c), ++q) {
      const int nr = min(rcB, b_hi(c.b) - c.n);
      const int t1 = min(c.t0 + tpc, ts[c.b + 1]);
      const int nt = t1 - c.t0;
      const int s = q % nstage;
      if (!failed && !mbar_wait(&rg.full[s], (uint32_t)((q / nstage) & 1))) {
        flag_timeout(a.status);
        failed = true;
      }
      const uint8_t* stg = ring + (size_t)s * a.stage_bytes;
      float* rd = redB + (size_t)(q & 1) * redB_n;
      const int items = nt * nslB * nr;
      const int ipw = (items + kSW - 1) / kSW;
      const int i0 = min(items, warp * ipw), i1 = min(items, i0 + ipw);
      int r = i0 % nr, sl = (i0 / nr) % nslB, j = (i0 / nr) / nslB;
      for (int it = i0; it < i1 && !failed;
           ++it, (++r == nr ? (r = 0, (++sl == nslB ? (sl = 0, ++j) : 0)) : 0)) {
        const int key = (c.t0 + j) * nslB + sl;
        if (key != hkey) {  // task's h slice into registers
          const float* hp = hsm + (size_t)(c.t0 + j) * I + sl * 512;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 v = FMT == MOE_W_NVFP4
                                 ? reinterpret_cast<const float4*>(hp + lane * 16)[m]
                                 : *reinterpret_cast<const float4*>(hp + lane * 8 + 256 * (m >> 1) + 4 * (m & 1));
            hv[4 * m] = v.x;
            hv[4 * m + 1] = v.y;
            hv[4 * m + 2] = v.z;
            hv[4 * m + 3] = v.w;
          }
          hkey = key;
        }
        const uint8_t* tb = stg + (size_t)j * rcB * rowB;
        float p;
        if (FMT == MOE_W_NVFP4) {
          const int e0 = sl * 512 + lane * 16;
          const uint2 cw2 = *reinterpret_cast<const uint2*>(tb + (size_t)r * (I / 2) + e0 / 2);
          const float qd = dot8_fp4_f(cw2.x, hv) + dot8_fp4_f(cw2.y, hv + 8);
          p = qd * e4m3x2_f32(tb[(size_t)rcB * (I / 2) + (size_t)r * (I / 16) + e0 / 16]).x;
        } else {
          const uint8_t* row = tb + (size_t)r * I * 2 + (size_t)sl * 1024;
          p = dot8_bf16_f(*reinterpret_cast<const uint4*>(row + lane * 16), hv, 0.f);
          p = dot8_bf16_f(*reinterpret_cast<const uint4*>(row + lane * 16 + 512), hv + 8, p);
        }
        p = wsum(p);
        if (lane == 0) rd[it] = p;
      }
      consumers_sync();  // stage no longer read; rd complete
      if (threadIdx.x == 0) mbar_arrive_one(&rg.empty[s]);
      if (threadIdx.x < nt * nr && !failed) {  // one thread per (task, row): slices in order
        const int jj = threadIdx.x / nr, rr = threadIdx.x % nr;
        float y = 0.f;
        for (int z = 0; z < nslB; ++z) y += rd[(jj * nslB + z) * nr + rr];
        ysm[(size_t)(c.t0 + jj) * perB + (c.b * H + c.n + rr - ru0)] = y;
      }
    }
  }
  consumers_sync();  // every per-task row result in ysm
  // combine: each output row, its tasks in route order (j ascending), then + ys
  int m = 0;
  for (int ru = ru0 + threadIdx.x; ru < ru1; ru += kST, ++m) {
    const int b = ru / H, n = ru - b * H;
    float acc = 0.f;
    for (int t = ts[b]; t < ts[b + 1]; ++t)
      acc = fmaf(tk.wt[t] * tk.gs[t][2], ysm[(size_t)t * perB + (ru - ru0)], acc);
    if (SHARED) {
      a.ys[(size_t)b * H + n] = gate_s[b] * acc;
    } else {
      const float yv = m < kYsPre ? ysv[m] : (a.ys ? a.ys[ru] : 0.f);
      a.out[(size_t)b * H + n] = __float2bfloat16_rn(a.ys ? acc + yv : acc);
    }
  }
}

int g_num_sms = 0;
constexpr size_t kBudget = 200 * 1024;
constexpr int kStageCapA = 36 * 1024;
constexpr int kStageCapB = 24 * 1024;

size_t round128(size_t v) { return (v + 127) / 128 * 128; }

struct Plan {
  size_t smem;
  int nstage, stage_bytes, rcA, rcB, tpc;
  bool ok;
};

Plan fused_plan(int wfmt, int H, int I, int n_rows, int T) {
  Plan p{};
  const int rowA = wfmt == MOE_W_NVFP4 ? 2 * (H / 2 + H / 16) : 2 * H * 2;
  const int rowB = wfmt == MOE_W_NVFP4 ? I / 2 + I / 16 : I * 2;
  p.rcA = rows_per_chunk(rowA, kStageCapA);
  p.rcB = rows_per_chunk(rowB, kStageCapB);
  p.tpc = kStageCapB / (p.rcB * rowB);
  p.tpc = p.tpc < 1 ? 1 : (p.tpc > 16 ? 16 : p.tpc);
  const size_t sA = (size_t)p.rcA * rowA, sB = (size_t)p.tpc * p.rcB * rowB;
  p.stage_bytes = (int)round128(sA > sB ? sA : sB);
  const int G = g_num_sms > 0 ? g_num_sms : 1;
  const int perB = (n_rows * H + G - 1) / G;
  const size_t fixed = round128((size_t)n_rows * H * 2) +
                       round128(((size_t)T * I + (size_t)T * perB + 4 * (size_t)(H / 1024) * p.rcA +
                                 2 * (size_t)p.tpc * (I / 512) * p.rcB) * 4);
  p.nstage = fixed < kBudget ? (int)((kBudget - fixed) / p.stage_bytes) : 0;
  p.nstage = p.nstage > kMaxStages ? kMaxStages : p.nstage;
  p.smem = fixed + (size_t)p.nstage * p.stage_bytes;
  p.ok = p.nstage >= 1 && H % 1024 == 0 && H / 1024 <= kSW && I % 512 == 0 && I / 512 <= kSW &&
         n_rows * H <= kXW * 8 * kST && p.tpc * p.rcB <= kST && (size_t)p.rcA * rowA <= (size_t)kStageCapA &&
         (size_t)p.rcB * rowB <= (size_t)kStageCapB;
  return p;
}

template <typename K>
cudaError_t launch_coop(K kernel, size_t smem, cudaStream_t s, const DevState& st,
                        const FusedArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(g_num_sms);
  cfg.blockDim = dim3(kST + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, st, a);
}

cudaError_t launch_fused(const DevState& st, int wfmt, bool shared, const FusedArgs& a0,
                         cudaStream_t s) {
  FusedArgs a = a0;
  const Plan p = fused_plan(wfmt, a.H, a.I, a.n_rows, a.R);
  a.nstage = p.nstage;
  a.stage_bytes = p.stage_bytes;
  a.rcA = p.rcA;
  a.rcB = p.rcB;
  a.tpc = p.tpc;
  if (wfmt == MOE_W_NVFP4)
    return shared ? launch_coop(ffn_fused_kernel<MOE_W_NVFP4, true>, p.smem, s, st, a)
                  : launch_coop(ffn_fused_kernel<MOE_W_NVFP4, false>, p.smem, s, st, a);
  return shared ? launch_coop(ffn_fused_kernel<MOE_W_BF16, true>, p.smem, s, st, a)
                : launch_coop(ffn_fused_kernel<MOE_W_BF16, false>, p.smem, s, st, a);
}

}  // namespace

bool ffn_stream_supported(int wfmt, int H, int I, int n_rows, int n_tasks) {
  if (g_num_sms <= 0 || n_tasks > kMaxTasks || n_rows > 16 || n_rows < 1) return false;
  if (H % 256 || I % 256) return false;  // every bulk copy 16-byte aligned and sized
  return fused_plan(wfmt, H, I, n_rows, n_tasks).ok;
}

cudaError_t ffn_stream_init(int wfmt, int H, int I, int Is, int max_rows, int max_tasks) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  auto set = [&](auto kern) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBudget);
  };
  set(ffn_fused_kernel<MOE_W_BF16, true>);
  set(ffn_fused_kernel<MOE_W_NVFP4, true>);
  set(ffn_fused_kernel<MOE_W_BF16, false>);
  set(ffn_fused_kernel<MOE_W_NVFP4, false>);
  (void)wfmt, (void)H, (void)I, (void)Is, (void)max_rows, (void)max_tasks;
  return e;
}

cudaError_t launch_shared_stream(const DevState& st, int wfmt, int H, int Is, const void* x,
                                 int n_rows, const uint8_t* blob, const void* gate_w,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = Is;
  a.layer = 0;
  a.k = 1;
  a.R = n_rows;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = nullptr;
  a.fixed_blob = blob;
  a.w = nullptr;
  a.h = sc.hs;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.gate = sc.gate;
  a.ys = sc.ys;
  a.out = nullptr;
  a.status = status;
  a.bar_ctr = sc.bar;
  return launch_fused(st, wfmt, true, a, s);
}

cudaError_t launch_routed_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                 const void* x, const int32_t* slot_ids, const float* w,
                                 int n_rows, int k, const float* shared_y, void* out,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = I;
  a.layer = layer;
  a.k = k;
  a.R = n_rows * k;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = slot_ids;
  a.fixed_blob = nullptr;
  a.w = w;
  a.h = sc.h;
  a.gate_w = nullptr;
  a.gate = nullptr;
  a.ys = const_cast<float*>(shared_y);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.bar_ctr = sc.bar;
  return launch_fused(st, wfmt, false, a, s);
}

// ---------------------------------------------------------------- allocation-free variant
// moe_routed_experts_noalloc runs ffn_fused_kernel with its scratch in this
// file-scope array instead of memory a cache allocated: bytes [0, 256) hold
// the grid-barrier counter, bytes [256, end) the fp32 intermediate h.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

cudaError_t noalloc_scratch(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess) e = ffn_stream_init(0, 0, 0, 0, 0, 0);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_routed_noalloc(int wfmt, int H, int I, const uint8_t* slots, size_t stride,
                                  int n_slots, const void* x, const int32_t* slot_ids,
                                  const float* w, int n_rows, int k, void* out,
                                  unsigned long long* status, void* scratch, cudaStream_t s) {
  DevState st{};  // just enough state to resolve a slot id to its blob
  st.L = 1;
  st.P = 1;
  st.S = n_slots;
  st.per_layer = 0;
  st.slots = const_cast<uint8_t*>(slots);
  st.stride = stride;
  FfnScratch sc{};
  sc.bar = static_cast<unsigned long long*>(scratch);
  sc.h = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + 256);
  // the barrier waits for the counter's next multiple of the grid size; a launch
  // that gave up after a timeout can leave it elsewhere, so start from zero
  cudaError_t e = cudaMemsetAsync(sc.bar, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  return launch_routed_stream(st, wfmt, H, I, 0, x, slot_ids, w, n_rows, k, nullptr, out, sc,
                              status, s);
}

}  // namespace moe
