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
// ~2 us, so the kernel must have megabytes in flight almost at once.  Each
// warp owns a list of weight rows and keeps a ring of up to 8 of them in
// flight: lane 0 issues cp.async.bulk copies (global -> shared, completion on
// a per-stage mbarrier) and the warp decodes stages as they land.  One CTA
// per SM.  The down-projection kernel is launched as a programmatic
// dependent of the gate/up kernel: it starts while gate/up still runs, loads
// its weights, and waits (griddepcontrol.wait) only before it reads h.
//
// Every wait on an mbarrier is bounded (%globaltimer); on a timeout the kernel
// sets MOE_STATUS_TIMEOUT in the cache's device status word, drains its own
// copies (again bounded) and returns.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kSW = 16;            // warps per CTA
constexpr int kST = 32 * kSW;      // threads per CTA
constexpr int kMaxStages = 8;      // ring depth
constexpr int kMaxTasks = 64;      // routes per call on this path
constexpr int kXW = 4;             // x words (8 bf16 each) held per consumer thread
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
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
template <int FMT>
__device__ void tasks_consts(Tasks& tk, int H, int I, const float* w) {
  const int t = threadIdx.x;
  if (t < tk.n) {
    tk.wt[t] = w ? w[tk.route[t]] : 1.f;
    if (FMT == MOE_W_NVFP4) {
      const size_t ih = (size_t)I * H;
      const float* g = reinterpret_cast<const float*>(tk.blob[t] + 3 * ih / 2 + 3 * (ih / 16));
      tk.gs[t][0] = g[0];
      tk.gs[t][1] = g[1];
      tk.gs[t][2] = g[2];
    } else {
      tk.gs[t][0] = tk.gs[t][1] = tk.gs[t][2] = 1.f;
    }
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

// ---------------------------------------------------------------- gate / up
// Rows u of the flattened (task, n) list -> h[route][n] = silu(g) * u.
//
// x is staged in shared memory once per CTA: as f16 for NVFP4 experts (so the
// products e2m1 * x are exact halves-times-halves), scaled per row by a power
// of two so the largest |x| is below 2^15 -- a bf16 value converts to f16
// exactly in that range, and the scale is undone on the fp32 sums -- or as
// bf16 for bf16 experts.
template <int FMT>
__global__ void __launch_bounds__(kST + 32, 2)
stream_up_kernel(DevState st, int H, int I, int layer, const uint16_t* __restrict__ x, int k,
                 const int32_t* __restrict__ slot_ids, int R, const uint8_t* fixed_blob,
                 float* __restrict__ h, int n_rows, int nstage, int stage_bytes,
                 unsigned long long* status, const uint16_t* __restrict__ gate_w,
                 float* __restrict__ gate_out) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Tasks tk;
  __shared__ Ring rg;
  __shared__ unsigned int xmax[16];  // per row max |x| (float bits, only when > 2^14)
  __shared__ float xscale[16];       // per row power-of-two scale applied to x
  __shared__ float xinv[16];         // per row 1 / scale
  __shared__ float red[16][16][2];   // [row of chunk][K slice]: partials of gate and up
  pdl_launch_dependents();  // the down kernel may start loading its weights now
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = FMT == MOE_W_NVFP4 ? 2 * (H / 2 + H / 16) : 2 * H * 2;
  const int rc = rows_per_chunk(row_bytes, stage_bytes);
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);  // [n_rows][H]
  uint8_t* ring = sm + ((size_t)n_rows * H * 2 + 127) / 128 * 128;

  // One global round trip for the routes' slots and all of x (8 bf16 per
  // thread per uint4, kept in registers); then the compaction; then the
  // producer starts copying while the consumers finish their set-up.
  // (the consumer threads hold x: kXW uint4 each, so n_rows * H <= kXW * 8 * kST)
  const int nx8 = n_rows * H / 8;          // uint4 words of x (H % 256 == 0)
  uint4 xw[kXW];
  if (threadIdx.x < 16) xmax[threadIdx.x] = 0u;
  tasks_load(tk, st, layer, slot_ids, R, fixed_blob);
#pragma unroll
  for (int j = 0; j < kXW; ++j) {
    const int i = threadIdx.x + j * kST;
    if (threadIdx.x < kST && i < nx8) xw[j] = reinterpret_cast<const uint4*>(x)[i];
  }
  __syncthreads();  // xmax zeroed, task loads done
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
  tasks_compact(tk, R);
  if (threadIdx.x == 0) {
    for (int q = 0; q < nstage; ++q) {
      mbar_init(&rg.full[q], 1);
      mbar_init(&rg.empty[q], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();  // tasks, barriers and every row's max |x| ready
  const int T = tk.n;
  const int U = T * I;
  const int per = (U + gridDim.x - 1) / gridDim.x;
  const int u0 = min(U, per * blockIdx.x), u1 = min(U, u0 + per);
  // chunks: rc rows each, never crossing a task boundary
  const BlobOff o(H, I);

  if (warp == kSW) {  // ------------------------------------------ producer
    if (lane == 0) {
      int q = 0;
      for (int u = u0; u < u1;) {
        const int t = u / I, n = u - t * I;
        const int nr = min(rc, min(u1 - u, I - n));
        const int s = q % nstage;
        if (q >= nstage && !mbar_wait(&rg.empty[s], (uint32_t)(((q / nstage) - 1) & 1))) {
          flag_timeout(status);
          break;
        }
        uint8_t* dst = ring + (size_t)s * stage_bytes;
        const uint8_t* blob = tk.blob[t];
        fence_proxy_async();
        if (FMT == MOE_W_NVFP4) {
          const uint32_t cb = nr * (H / 2), sb = nr * (H / 16);
          mbar_expect_tx(&rg.full[s], 2 * (cb + sb));
          bulk_g2s(dst, blob + o.code[0] + (size_t)n * (H / 2), cb, &rg.full[s]);
          bulk_g2s(dst + rc * (H / 2), blob + o.code[1] + (size_t)n * (H / 2), cb, &rg.full[s]);
          bulk_g2s(dst + 2 * rc * (H / 2), blob + o.scale[0] + (size_t)n * (H / 16), sb,
                   &rg.full[s]);
          bulk_g2s(dst + 2 * rc * (H / 2) + rc * (H / 16), blob + o.scale[1] + (size_t)n * (H / 16),
                   sb, &rg.full[s]);
        } else {
          const uint32_t rb = nr * H * 2;
          mbar_expect_tx(&rg.full[s], 2 * rb);
          bulk_g2s(dst, blob + o.mat[0] + (size_t)n * H * 2, rb, &rg.full[s]);
          bulk_g2s(dst + (size_t)rc * H * 2, blob + o.mat[1] + (size_t)n * H * 2, rb, &rg.full[s]);
        }
        ++q;
        u += nr;
      }
      producer_drain(rg, nstage, q);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  if (threadIdx.x < n_rows) {
    float sc = 1.f;  // power of two bringing max |x| below 2^15
    const float mx = __uint_as_float(xmax[threadIdx.x]);
    while (mx * sc >= 32768.f) sc *= 0.5f;
    xscale[threadIdx.x] = sc;
    xinv[threadIdx.x] = 1.f / sc;
  }
  tasks_consts<FMT>(tk, H, I, nullptr);
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
  consumers_sync();
  // the shared expert's sigmoid gate, sigmoid(x_b . w_g), in fp32
  if (gate_w && blockIdx.x == 0 && warp < n_rows) {
    float z = 0.f;
    for (int i0 = lane * 8; i0 < H; i0 += 256) {
      const uint4 gv = *reinterpret_cast<const uint4*>(gate_w + i0);
      const uint4 xv = *reinterpret_cast<const uint4*>(x + (size_t)warp * H + i0);
      z = dot8_bf16_bf(gv, xv, z);
    }
    z = wsum(z);
    if (lane == 0) gate_out[warp] = 1.f / (1.f + expf(-z));
  }
  // Warp = (K slice of 1024 elements, row group).  The warp's slice of x stays
  // in registers for every row it processes; the weights of a row slice are
  // read with lane-contiguous 16-byte loads (no bank conflicts).
  //   NVFP4: lane L takes elements [32L, 32L+32) of the slice (16 code bytes)
  //   bf16:  lane L takes elements 8L + 256j + [0, 8), j = 0..3 (4 x 16 bytes)
  const int nsl = H / 1024;
  const int ngr = kSW / nsl;
  const int my_sl = warp % nsl, my_g = warp / nsl;
  uint4 xv[4];
  int xb = -1;
  bool failed = false;  // a timed-out wait: keep taking part in the barriers, skip the work
  int q = 0;
  for (int u = u0; u < u1; ++q) {
    const int t = u / I, n = u - t * I;
    const int nr = min(rc, min(u1 - u, I - n));
    const int s = q % nstage;
    if (!failed && !mbar_wait(&rg.full[s], (uint32_t)((q / nstage) & 1))) {
      flag_timeout(status);
      failed = true;
    }
    const int b = tk.route[t] / k;
    if (b != xb) {  // this batch row's x slice into registers
      const uint16_t* xr = xs + (size_t)b * H + my_sl * 1024;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        xv[j] = FMT == MOE_W_NVFP4 ? reinterpret_cast<const uint4*>(xr + lane * 32)[j]
                                   : *reinterpret_cast<const uint4*>(xr + lane * 8 + 256 * j);
      xb = b;
    }
    const uint8_t* stg = ring + (size_t)s * stage_bytes;
    for (int r = my_g; r < nr && !failed; r += ngr) {
      float g = 0.f, up = 0.f;
      if (FMT == MOE_W_NVFP4) {
        const int e0 = my_sl * 1024 + lane * 32;
        const uint4 cg = *reinterpret_cast<const uint4*>(stg + (size_t)r * (H / 2) + e0 / 2);
        const uint4 cu = *reinterpret_cast<const uint4*>(stg + (size_t)(rc + r) * (H / 2) + e0 / 2);
        const uint8_t* sc = stg + (size_t)2 * rc * (H / 2);
        const float2 sg = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(sc + (size_t)r * (H / 16) + e0 / 16));
        const float2 su =
            e4m3x2_f32(*reinterpret_cast<const uint16_t*>(sc + (size_t)(rc + r) * (H / 16) + e0 / 16));
        g = fmaf(dot8_fp4_h(cg.x, xv[0]) + dot8_fp4_h(cg.y, xv[1]), sg.x, 0.f);
        g = fmaf(dot8_fp4_h(cg.z, xv[2]) + dot8_fp4_h(cg.w, xv[3]), sg.y, g);
        up = fmaf(dot8_fp4_h(cu.x, xv[0]) + dot8_fp4_h(cu.y, xv[1]), su.x, 0.f);
        up = fmaf(dot8_fp4_h(cu.z, xv[2]) + dot8_fp4_h(cu.w, xv[3]), su.y, up);
      } else {
        const uint8_t* rowg = stg + (size_t)r * H * 2 + (size_t)my_sl * 2048;
        const uint8_t* rowu = stg + (size_t)(rc + r) * H * 2 + (size_t)my_sl * 2048;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          g = dot8_bf16_bf(*reinterpret_cast<const uint4*>(rowg + lane * 16 + 512 * j), xv[j], g);
          up = dot8_bf16_bf(*reinterpret_cast<const uint4*>(rowu + lane * 16 + 512 * j), xv[j], up);
        }
      }
      g = wsum(g);
      up = wsum(up);
      if (lane == 0) {
        red[r][my_sl][0] = g;
        red[r][my_sl][1] = up;
      }
    }
    consumers_sync();  // every slice of every row done, stage no longer read
    if (threadIdx.x == 0) mbar_arrive_one(&rg.empty[s]);
    if (threadIdx.x < nr && !failed) {  // one thread per row: slices in a fixed order
      const int r = threadIdx.x;
      float gs = 0.f, us = 0.f;
      for (int sl = 0; sl < nsl; ++sl) {
        gs += red[r][sl][0];
        us += red[r][sl][1];
      }
      const float xi = FMT == MOE_W_NVFP4 ? xinv[b] : 1.f;
      const float gg = gs * xi * tk.gs[t][0], uu = us * xi * tk.gs[t][1];
      h[(size_t)tk.route[t] * I + n + r] = gg / (1.f + expf(-gg)) * uu;
    }
    consumers_sync();  // red[] reusable
    u += nr;
  }
}

// ---------------------------------------------------------------- down
// SHARED: ys[b][n] = gate[b] * (W_d h_b)[n]  (one task per row b)
// ROUTED: out[b][n] = bf16( sum_j w[b,j] * (W_d[slot] h_bj)[n] + ys[b][n] )
// The CTA's output rows are a range of (b, n); for each batch row b in it the
// chunks are (task of b, rc rows), tasks in route order; the per-task row
// results are kept in shared memory and combined at the end in route order.
template <int FMT, bool SHARED>
__global__ void __launch_bounds__(kST + 32, 2)
stream_down_kernel(DevState st, int H, int I, int layer, int k,
                   const int32_t* __restrict__ slot_ids, int R, const uint8_t* fixed_blob,
                   const float* __restrict__ w, const float* h, const float* gate_in,
                   float* ys, __nv_bfloat16* out, int n_rows, int nstage, int stage_bytes,
                   unsigned long long* status) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Tasks tk;
  __shared__ Ring rg;
  __shared__ float gate_s[16];
  __shared__ int ts[17];  // tasks of batch row b: [ts[b], ts[b+1])
  __shared__ float red[16][16];  // [row of chunk][K slice]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = FMT == MOE_W_NVFP4 ? I / 2 + I / 16 : I * 2;
  const int rc = rows_per_chunk(row_bytes, stage_bytes);
  tasks_load(tk, st, layer, slot_ids, R, fixed_blob);
  __syncthreads();
  tasks_compact(tk, R);
  __syncthreads();
  const int T = tk.n;
  if (threadIdx.x <= n_rows) {  // first task of each batch row (tasks are b-major)
    int a = 0;
    while (a < T && tk.route[a] / k < (int)threadIdx.x) ++a;
    ts[threadIdx.x] = a;
  }
  if (threadIdx.x == 0) {
    for (int q = 0; q < nstage; ++q) {
      mbar_init(&rg.full[q], 1);
      mbar_init(&rg.empty[q], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int U = n_rows * H;
  const int per = (U + gridDim.x - 1) / gridDim.x;
  const int ru0 = min(U, per * blockIdx.x), ru1 = min(U, ru0 + per);
  // shared memory: h of every task [T][I], then y[T][per] (per-task row results), then the ring
  float* hsm = reinterpret_cast<float*>(sm);
  float* ysm = hsm + (size_t)T * I;
  uint8_t* ring = sm + (((size_t)T * I + (size_t)T * per) * 4 + 127) / 128 * 128;
  const BlobOff o(H, I);

  // chunk sequence: for b, for task t of b, for rows [n, n+nr) of b's range
  auto first_chunk = [&](int* b, int* t, int* n) {
    *b = ru0 / H;
    *t = ts[*b];
    *n = ru0 - *b * H;
  };
  // advance to the next chunk; false when done
  auto next_chunk = [&](int* b, int* t, int* n, int nr) -> bool {
    const int nb_end = min(ru1 - *b * H, H);
    *n += nr;
    if (*n < nb_end) return true;
    ++*t;
    *n = max(ru0 - *b * H, 0);
    if (*t < ts[*b + 1]) return true;
    ++*b;
    if (*b * H >= ru1) return false;
    *t = ts[*b];
    *n = 0;
    return true;
  };
  auto valid_chunk = [&](int* b, int* t, int* n) -> bool {  // skip rows without tasks
    while (*b * H < ru1 && *t >= ts[*b + 1]) {
      ++*b;
      if (*b * H >= ru1) return false;
      *t = ts[*b];
      *n = 0;
    }
    return *b * H < ru1 && ru0 < ru1;
  };
  auto rows_of = [&](int b, int n) { return min(rc, min(ru1 - b * H, H) - n); };

  if (warp == kSW) {  // ------------------------------------------ producer
    if (lane == 0) {
      int b, t, n, q = 0;
      first_chunk(&b, &t, &n);
      bool more = valid_chunk(&b, &t, &n);
      while (more) {
        const int nr = rows_of(b, n);
        const int s = q % nstage;
        if (q >= nstage && !mbar_wait(&rg.empty[s], (uint32_t)(((q / nstage) - 1) & 1))) {
          flag_timeout(status);
          break;
        }
        uint8_t* dst = ring + (size_t)s * stage_bytes;
        const uint8_t* blob = tk.blob[t];
        fence_proxy_async();
        if (FMT == MOE_W_NVFP4) {
          const uint32_t cb = nr * (I / 2), sb = nr * (I / 16);
          mbar_expect_tx(&rg.full[s], cb + sb);
          bulk_g2s(dst, blob + o.code[2] + (size_t)n * (I / 2), cb, &rg.full[s]);
          bulk_g2s(dst + rc * (I / 2), blob + o.scale[2] + (size_t)n * (I / 16), sb, &rg.full[s]);
        } else {
          const uint32_t rb = nr * I * 2;
          mbar_expect_tx(&rg.full[s], rb);
          bulk_g2s(dst, blob + o.mat[2] + (size_t)n * I * 2, rb, &rg.full[s]);
        }
        ++q;
        more = next_chunk(&b, &t, &n, nr) && valid_chunk(&b, &t, &n);
      }
      producer_drain(rg, nstage, q);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  tasks_consts<FMT>(tk, H, I, SHARED ? nullptr : w);
  // everything above overlaps the gate/up kernel; its outputs are read only
  // after it has completed
  pdl_wait();
  {  // every task's h into shared memory: float4 loads, four in flight per thread
    const int n4 = T * I / 4, i4 = I / 4;
    float4* hs4 = reinterpret_cast<float4*>(hsm);
    const float4* h4 = reinterpret_cast<const float4*>(h);
    for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * kST) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kST;
        if (i < n4) v[j] = h4[(size_t)tk.route[i / i4] * i4 + (i % i4)];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i0 + j * kST < n4) hs4[i0 + j * kST] = v[j];
    }
  }
  if (SHARED && threadIdx.x < n_rows) gate_s[threadIdx.x] = gate_in[threadIdx.x];
  consumers_sync();

  // Warp = (K slice of 512 elements, row group); the warp's slice of h_t stays
  // in registers while it walks the rows of task t.
  //   NVFP4: lane L takes elements [16L, 16L+16) of the slice (8 code bytes)
  //   bf16:  lane L takes elements 8L + 256j + [0, 8), j = 0, 1 (2 x 16 bytes)
  const int nsl = I / 512;
  const int ngr = kSW / nsl;
  const int my_sl = warp % nsl, my_g = warp / nsl;
  {
    bool failed = false;  // a timed-out wait: keep taking part in the barriers, skip the work
    float hv[16];
    int ht = -1;
    int b, t, n, q = 0;
    first_chunk(&b, &t, &n);
    bool more = valid_chunk(&b, &t, &n);
    while (more) {
      const int nr = rows_of(b, n);
      const int s = q % nstage;
      if (!failed && !mbar_wait(&rg.full[s], (uint32_t)((q / nstage) & 1))) {
        flag_timeout(status);
        failed = true;
      }
      if (t != ht) {  // task t's h slice into registers
        const float* hp = hsm + (size_t)t * I + my_sl * 512;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 v = FMT == MOE_W_NVFP4
                               ? reinterpret_cast<const float4*>(hp + lane * 16)[j]
                               : *reinterpret_cast<const float4*>(hp + lane * 8 + 256 * (j >> 1) + 4 * (j & 1));
          hv[4 * j] = v.x;
          hv[4 * j + 1] = v.y;
          hv[4 * j + 2] = v.z;
          hv[4 * j + 3] = v.w;
        }
        ht = t;
      }
      const uint8_t* stg = ring + (size_t)s * stage_bytes;
      for (int r = my_g; r < nr && !failed; r += ngr) {
        float p;
        if (FMT == MOE_W_NVFP4) {
          const int e0 = my_sl * 512 + lane * 16;
          const uint2 c = *reinterpret_cast<const uint2*>(stg + (size_t)r * (I / 2) + e0 / 2);
          const float qd = dot8_fp4_f(c.x, hv) + dot8_fp4_f(c.y, hv + 8);
          p = qd * e4m3x2_f32(stg[(size_t)rc * (I / 2) + (size_t)r * (I / 16) + e0 / 16]).x;
        } else {
          const uint8_t* row = stg + (size_t)r * I * 2 + (size_t)my_sl * 1024;
          p = dot8_bf16_f(*reinterpret_cast<const uint4*>(row + lane * 16), hv, 0.f);
          p = dot8_bf16_f(*reinterpret_cast<const uint4*>(row + lane * 16 + 512), hv + 8, p);
        }
        p = wsum(p);
        if (lane == 0) red[r][my_sl] = p;
      }
      consumers_sync();
      if (threadIdx.x == 0) mbar_arrive_one(&rg.empty[s]);
      if (threadIdx.x < nr && !failed) {  // one thread per row: slices in a fixed order
        const int r = threadIdx.x;
        float y = 0.f;
        for (int sl = 0; sl < nsl; ++sl) y += red[r][sl];
        ysm[(size_t)t * per + (b * H + n + r - ru0)] = y;
      }
      consumers_sync();
      ++q;
      more = next_chunk(&b, &t, &n, nr) && valid_chunk(&b, &t, &n);
    }
  }
  // combine: each output row, its tasks in route order (j ascending), then + ys
  for (int ru = ru0 + threadIdx.x; ru < ru1; ru += kST) {
    const int b = ru / H, n = ru - b * H;
    float acc = 0.f;
    for (int t = ts[b]; t < ts[b + 1]; ++t)
      acc = fmaf(tk.wt[t] * tk.gs[t][2], ysm[(size_t)t * per + (ru - ru0)], acc);
    if (SHARED) {
      ys[(size_t)b * H + n] = gate_s[b] * acc;
    } else {
      const float yy = ys ? acc + ys[(size_t)b * H + n] : acc;
      out[(size_t)b * H + n] = __float2bfloat16_rn(yy);
    }
  }
}

int g_num_sms = 0;

// Shared-memory budgets: the gate/up kernel and its dependent down kernel are
// sized to fit one SM together (228 KB), so the down kernel can load while
// gate/up still runs.
constexpr size_t kUpBudget = 150 * 1024;
constexpr size_t kDownBudget = 72 * 1024;
constexpr int kUpStageCap = 36 * 1024;
constexpr int kDownStageCap = 16 * 1024;

template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, int grid, size_t smem, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kST + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct Plan {
  size_t smem;
  int nstage, stage_bytes, rc;
  bool ok;
};

Plan up_plan(int wfmt, int H, int n_rows) {
  Plan p{};
  const int row = wfmt == MOE_W_NVFP4 ? 2 * (H / 2 + H / 16) : 2 * H * 2;
  p.rc = rows_per_chunk(row, kUpStageCap);
  p.stage_bytes = (p.rc * row + 127) / 128 * 128;
  const size_t fixed = ((size_t)n_rows * H * 2 + 127) / 128 * 128;
  p.nstage = fixed < kUpBudget ? (int)((kUpBudget - fixed) / p.stage_bytes) : 0;
  p.nstage = p.nstage > kMaxStages ? kMaxStages : p.nstage;
  p.smem = fixed + (size_t)p.nstage * p.stage_bytes;
  p.ok = p.rc * row <= kUpStageCap && p.nstage >= 2 && H % 1024 == 0 && H / 1024 <= kSW &&
         n_rows * H <= kXW * 8 * kST;
  return p;
}

Plan down_plan(int wfmt, int H, int I, int n_rows, int T) {
  Plan p{};
  const int row = wfmt == MOE_W_NVFP4 ? I / 2 + I / 16 : I * 2;
  p.rc = rows_per_chunk(row, kDownStageCap);
  p.stage_bytes = (p.rc * row + 127) / 128 * 128;
  const int per = (n_rows * H + g_num_sms - 1) / (g_num_sms > 0 ? g_num_sms : 1);
  const size_t fixed = (((size_t)T * I + (size_t)T * per) * 4 + 127) / 128 * 128;
  p.nstage = fixed < kDownBudget ? (int)((kDownBudget - fixed) / p.stage_bytes) : 0;
  p.nstage = p.nstage > kMaxStages ? kMaxStages : p.nstage;
  p.smem = fixed + (size_t)p.nstage * p.stage_bytes;
  p.ok = p.rc * row <= kDownStageCap && p.nstage >= 2 && I % 512 == 0 && I / 512 <= kSW;
  return p;
}

}  // namespace

bool ffn_stream_supported(int wfmt, int H, int I, int n_rows, int n_tasks) {
  if (g_num_sms <= 0 || n_tasks > kMaxTasks || n_rows > 16 || n_rows < 1) return false;
  if (H % 256 || I % 256) return false;  // every bulk copy 16-byte aligned and sized
  return up_plan(wfmt, H, n_rows).ok && down_plan(wfmt, H, I, n_rows, n_tasks).ok;
}

cudaError_t ffn_stream_init(int wfmt, int H, int I, int Is, int max_rows, int max_tasks) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  auto set = [&](auto kern, size_t bytes) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  };
  set(stream_up_kernel<MOE_W_BF16>, kUpBudget);
  set(stream_up_kernel<MOE_W_NVFP4>, kUpBudget);
  set(stream_down_kernel<MOE_W_BF16, true>, kDownBudget);
  set(stream_down_kernel<MOE_W_NVFP4, true>, kDownBudget);
  set(stream_down_kernel<MOE_W_BF16, false>, kDownBudget);
  set(stream_down_kernel<MOE_W_NVFP4, false>, kDownBudget);
  (void)wfmt, (void)H, (void)I, (void)Is, (void)max_rows, (void)max_tasks;
  return e;
}

// Shared expert: h_s and the gate via the up kernel, then ys = gate * W_d h_s.
cudaError_t launch_shared_stream(const DevState& st, int wfmt, int H, int Is, const void* x,
                                 int n_rows, const uint8_t* blob, const void* gate_w,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s) {
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const uint16_t* gw = static_cast<const uint16_t*>(gate_w);
  const Plan pu = up_plan(wfmt, H, n_rows), pd = down_plan(wfmt, H, Is, n_rows, n_rows);
  const int grid = g_num_sms;
  const int32_t* none = nullptr;
  cudaError_t e;
  if (wfmt == MOE_W_NVFP4) {
    e = launch_ex(stream_up_kernel<MOE_W_NVFP4>, grid, pu.smem, s, false, st, H, Is, 0, xx, 1,
                  none, n_rows, blob, sc.hs, n_rows, pu.nstage, pu.stage_bytes, status, gw,
                  sc.gate);
    if (e == cudaSuccess)
      e = launch_ex(stream_down_kernel<MOE_W_NVFP4, true>, grid, pd.smem, s, true, st, H, Is, 0, 1,
                    none, n_rows, blob, (const float*)nullptr, (const float*)sc.hs,
                    (const float*)sc.gate, sc.ys, (__nv_bfloat16*)nullptr, n_rows, pd.nstage,
                    pd.stage_bytes, status);
  } else {
    e = launch_ex(stream_up_kernel<MOE_W_BF16>, grid, pu.smem, s, false, st, H, Is, 0, xx, 1,
                  none, n_rows, blob, sc.hs, n_rows, pu.nstage, pu.stage_bytes, status, gw,
                  sc.gate);
    if (e == cudaSuccess)
      e = launch_ex(stream_down_kernel<MOE_W_BF16, true>, grid, pd.smem, s, true, st, H, Is, 0, 1,
                    none, n_rows, blob, (const float*)nullptr, (const float*)sc.hs,
                    (const float*)sc.gate, sc.ys, (__nv_bfloat16*)nullptr, n_rows, pd.nstage,
                    pd.stage_bytes, status);
  }
  return e;
}

cudaError_t launch_routed_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                 const void* x, const int32_t* slot_ids, const float* w,
                                 int n_rows, int k, const float* shared_y, void* out,
                                 FfnScratch sc, unsigned long long* status, cudaStream_t s) {
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const int R = n_rows * k;
  const Plan pu = up_plan(wfmt, H, n_rows), pd = down_plan(wfmt, H, I, n_rows, R);
  const int grid = g_num_sms;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const uint8_t* nob = nullptr;
  const uint16_t* nogw = nullptr;
  float* nogate = nullptr;
  cudaError_t e;
  if (wfmt == MOE_W_NVFP4) {
    e = launch_ex(stream_up_kernel<MOE_W_NVFP4>, grid, pu.smem, s, false, st, H, I, layer, xx, k,
                  slot_ids, R, nob, sc.h, n_rows, pu.nstage, pu.stage_bytes, status, nogw, nogate);
    if (e == cudaSuccess)
      e = launch_ex(stream_down_kernel<MOE_W_NVFP4, false>, grid, pd.smem, s, true, st, H, I,
                    layer, k, slot_ids, R, nob, w, (const float*)sc.h, (const float*)nullptr,
                    const_cast<float*>(shared_y), o, n_rows, pd.nstage, pd.stage_bytes, status);
  } else {
    e = launch_ex(stream_up_kernel<MOE_W_BF16>, grid, pu.smem, s, false, st, H, I, layer, xx, k,
                  slot_ids, R, nob, sc.h, n_rows, pu.nstage, pu.stage_bytes, status, nogw, nogate);
    if (e == cudaSuccess)
      e = launch_ex(stream_down_kernel<MOE_W_BF16, false>, grid, pd.smem, s, true, st, H, I,
                    layer, k, slot_ids, R, nob, w, (const float*)sc.h, (const float*)nullptr,
                    const_cast<float*>(shared_y), o, n_rows, pd.nstage, pd.stage_bytes, status);
  }
  return e;
}

}  // namespace moe
