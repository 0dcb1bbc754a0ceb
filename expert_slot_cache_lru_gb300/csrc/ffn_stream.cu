// ffn_stream.cu -- expert FFNs for decode-sized steps: one launch of thread-
// block clusters per group of experts.
//
// What is computed is the same as gemv.cu (FreeToken issue #753 "[Perf]
// Offloaded decode: overlap the expert-miss gather with the same layer's
// shared expert ...", Problem and What we changed: routed experts over the
// slots, a sigmoid-gated shared expert, routed + shared); this file is the
// fast path when every (route, row) of the step fits a small task list.
//
// A decode step moves ~14 MB of weights per layer, which HBM delivers in ~2 us
// after ~1 us of latency, and the arithmetic per weight is a handful of
// instructions, so the launch is built to have every byte requested within a
// microsecond of entry and to need no grid-wide step:
//   * each task's intermediate I is cut into P parts; a unit (task, part)
//     belongs to one cluster of kCS CTAs, one CTA per SM;
//   * phase A (gate/up): each warp of a CTA owns whole rows of its share of the
//     part; the rows' chunks come into two per-warp shared-memory slots by bulk
//     copies (cp.async.bulk, completing on an mbarrier), and the warp reduces
//     each row; h of a row goes to every CTA of the cluster (distributed shared
//     memory), then one cluster barrier;
//   * phase B (down): each thread of a CTA takes output rows of the CTA's slice
//     of H and dots the part's columns with h; the rows were requested into L2
//     when the unit began;
//   * the last unit to finish a slice (a counter per slice) combines it in a
//     fixed order: routed terms j ascending (each the sum of its parts, p
//     ascending), then the gated shared expert, rounded to bf16 once.
// The one-launch layer (kLayerAdmit) adds a cluster whose CTA 0 runs the
// admission; the CTAs of a missed expert's units copy its bytes from pinned
// host memory while the resident experts compute.
//
// Every wait that depends on another CTA is bounded (%globaltimer): on a
// timeout the kernel sets MOE_STATUS_TIMEOUT in the cache's device status word
// and computes nothing more, keeping every cluster barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "admit_body.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int kW = 16;             // compute warps per CTA
constexpr int kT = 32 * kW;        // compute threads per CTA
// The layer launches (kLayer, kLayerAdmit) add kCW copy warps per CTA: they
// copy the step's missed experts and the next layer's prefetched ones from
// pinned host memory while the compute warps run, so that a copy starts as soon
// as the launch knows its misses and never holds up a unit that hit.  ~280 copy
// warps keep the host link (~205 GB/s of 4 KiB warp reads) busy.
constexpr int kCW = 2;
constexpr int kNW = kW + kCW;      // warps per CTA of a layer launch
constexpr int kMaxRoutes = 64;     // routes per call on this path
constexpr int kMaxTasks = 80;      // routes plus one shared-expert task per row (fused layer)
constexpr int kMaxRows = 16;       // batch rows per call on this path
constexpr int kXW = 4;             // x words (8 elements each) loaded per thread
// Registers per thread: 512 x 104 leaves room on the SM for a gather CTA
// (256 threads x 32 registers), which runs beside the shared-expert launch on
// the side stream.  Each of an SM's four sub-partitions holds 16,384
// registers and a quarter of the warps: the layer launches' 18 warps put five
// on two of them, so those take at most 16,384 / (5 x 32) -> 96.
constexpr int kMaxReg = 104;
constexpr int kMaxRegLayer = 96;
constexpr int max_reg(int mode) { return mode == 2 || mode == 3 ? kMaxRegLayer : kMaxReg; }
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms
constexpr int kPiece = 4096;       // gather unit of the fused layer (one warp, 8 x 16 B per lane)

// What one launch computes: the routed experts, the gated shared expert, or
// (fused layer) both plus the gather of the step's missed experts.
enum { kRouted = 0, kShared = 1, kLayer = 2, kLayerAdmit = 3 };

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
// generic-proxy accesses of shared memory before async-proxy writes to it
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// L2 policy for weight bytes, which every layer reads once: evicted first, so
// the streamed weights do not push the kernels' code, the cache state and the
// activations out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completing `bytes` transactions on `bar`, with an L2 cache policy
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
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
// Bounded wait for the phase of `bar` with the given parity; false on timeout.
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
// an E8M0 block scale (MXFP4): 2^(e - 127), from its exponent bits; 0 is the
// subnormal 2^-127, 255 is NaN
__device__ __forceinline__ float e8m0_f32(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : (e == 255 ? __uint_as_float(0x7fffffffu)
                                                            : __uint_as_float(e << 23));
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
// Q4_0 codes: the 8 unsigned 4-bit codes q of w (even element in the low
// nibble) as four half2 of q - 8, exactly: each q goes into the mantissa of
// an f16 1024 (byte 0x64 above it), then 1032 is subtracted.
__device__ __forceinline__ void q4x8_h2(uint32_t w, uint32_t out[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t m0 = __byte_perm(lo, hi, 0x5140);  // codes 0 1 2 3
  const uint32_t m1 = __byte_perm(lo, hi, 0x7362);  // codes 4 5 6 7
  const uint32_t k = 0x64646464u;
  uint32_t v[4] = {__byte_perm(m0, k, 0x4140), __byte_perm(m0, k, 0x4342),
                   __byte_perm(m1, k, 0x4140), __byte_perm(m1, k, 0x4342)};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&v[j]), bias);
    out[j] = *reinterpret_cast<const uint32_t*>(&r);
  }
}
// sum_{i<8} (q_i - 8) * x[i], x as four half2 words (exact products)
__device__ __forceinline__ float dot8_q4_h(uint32_t w, uint4 x) {
  uint32_t q[4];
  q4x8_h2(w, q);
  float a = fma2_h(q[0], x.x, 0.f);
  a = fma2_h(q[1], x.y, a);
  a = fma2_h(q[2], x.z, a);
  return fma2_h(q[3], x.w, a);
}
// sum_{i<8} (q_i - 8) * h[i], h fp32
__device__ __forceinline__ float dot8_q4_f(uint32_t w, const float* h) {
  uint32_t q[4];
  q4x8_h2(w, q);
  float2 f = h2_f32(q[0]);
  float a = fmaf(f.x, h[0], f.y * h[1]);
  f = h2_f32(q[1]);
  a = fmaf(f.x, h[2], fmaf(f.y, h[3], a));
  f = h2_f32(q[2]);
  a = fmaf(f.x, h[4], fmaf(f.y, h[5], a));
  f = h2_f32(q[3]);
  return fmaf(f.x, h[6], fmaf(f.y, h[7], a));
}
// an fp16 block scale (Q4_0) as fp32, exactly
__device__ __forceinline__ float f16_f32(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
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
  size_t code[3], scale[3], glob;  // NVFP4 and MXFP4 (MXFP4: no global scales)
  size_t mat[3];                   // bf16
  __device__ BlobOff(int H, int I, int fmt) {
    const size_t ih = (size_t)I * H;
    const size_t sb = ih / (fmt == MOE_W_MXFP4 ? 32 : 16);  // scale bytes per matrix
    code[0] = 0;
    code[1] = ih / 2;
    code[2] = ih;
    scale[0] = 3 * ih / 2;
    scale[1] = scale[0] + sb;
    scale[2] = scale[1] + sb;
    glob = scale[2] + sb;
    mat[0] = 0;
    mat[1] = ih * 2;
    mat[2] = ih * 4;
  }
};

// Per-call task list, identical in every CTA: the valid routes in route order.
struct Tasks {
  int n;
  int route[kMaxTasks];            // route index r = b*k + j; R + b for row b's shared task
  int b[kMaxTasks];                // batch row
  int pe[kMaxTasks];               // fused layer: index in the demand plan, -1 = resident,
                                   // kPending = not resident when the launch began
  unsigned char drop[kMaxTasks];   // admission inside: not admitted (fetch cap)
  unsigned char pend[kMaxTasks];   // admission inside: not resident when the launch began
  int slot[kMaxTasks];             // slot id, -1 for the shared expert
  const uint8_t* blob[kMaxTasks];
  float wt[kMaxTasks];             // routing weight x down global scale
  int ubase[kMaxTasks + 1];        // first unit of each task (units of task t: ubase[t] ..)
};

__device__ void flag_timeout(unsigned long long* status) {
  if (status) atomicOr(status, (unsigned long long)MOE_STATUS_TIMEOUT);
}

// x lives in shared memory as 16-byte units, row-major per batch row, with
// unit u of a row stored at u ^ ((u >> 3) & 7): the eight lanes of a quarter
// warp that read units 8L + j (NVFP4, 64 contiguous elements per lane) or
// 32s + L (bf16) then hit eight different bank groups.
__device__ __forceinline__ int xswz(int u) { return u ^ ((u >> 3) & 7); }

// Power of two that brings max |x| of a row below 2^15 (1 when it already is).
// At most 140 halvings, so an infinite input cannot keep the loop going.
__device__ __forceinline__ float x_scale(float mx) {
  float sc = 1.f;
  for (int i = 0; i < 140 && mx * sc >= 32768.f; ++i) sc *= 0.5f;
  return sc;
}

// Two per-lane partial sums -> lane 0 holds both totals (6 shuffles).
__device__ __forceinline__ float2 reduce2(float g, float u, int lane) {
  const bool hi = lane & 16;
  float v = hi ? u : g;
  v += __shfl_xor_sync(0xffffffffu, hi ? g : u, 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return make_float2(v, __shfl_sync(0xffffffffu, v, 16));
}
// Four per-lane partial sums -> lane 8j holds the total of p[j] (6 shuffles).
__device__ __forceinline__ float reduce4(const float p[4], int lane) {
  const bool hi = lane & 16, h8 = lane & 8;
  float k0 = hi ? p[2] : p[0], k1 = hi ? p[3] : p[1];
  k0 += __shfl_xor_sync(0xffffffffu, hi ? p[0] : p[2], 16);
  k1 += __shfl_xor_sync(0xffffffffu, hi ? p[1] : p[3], 16);
  float v = h8 ? k1 : k0;
  v += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ phase A items
// An item is one chunk of CW elements of one gate row and the same chunk of
// the up row, brought into a per-warp shared-memory slot by bulk copies:
//   NVFP4 (CW = 2048): gate codes [1024 B] | up codes [1024 B] | gate scales
//     [128 B] | up scales [128 B] | the blob's 16-byte global-scale record;
//     lane L decodes elements [32L, 32L+32) and [1024+32L, 1024+32L+32);
//   bf16 (CW = 512): gate [1024 B] | up [1024 B]; lane L takes elements
//     8L + [0, 8) and 256 + 8L + [0, 8).
// Every lane reads 16 contiguous bytes per load at a 16-byte lane stride, so
// the shared-memory reads are conflict-free.
template <int FMT>
struct ItemA;
template <>
struct ItemA<MOE_W_NVFP4> {
  static constexpr int CW = 2048;
  static constexpr int BYTES = 2 * 1024 + 2 * 128;
  static __device__ __forceinline__ uint32_t issue(uint8_t* slot, const uint8_t* blob,
                                                   const BlobOff& o, int H, int i, int c,
                                                   uint64_t* bar, uint64_t pol) {
    const size_t cr = (size_t)i * (H / 2) + c * 1024, sr = (size_t)i * (H / 16) + c * 128;
    bulk_g2s(slot, blob + o.code[0] + cr, 1024, bar, pol);
    bulk_g2s(slot + 1024, blob + o.code[1] + cr, 1024, bar, pol);
    bulk_g2s(slot + 2048, blob + o.scale[0] + sr, 128, bar, pol);
    bulk_g2s(slot + 2176, blob + o.scale[1] + sr, 128, bar, pol);
    return BYTES;
  }
  // the gate and up global scales, read with a plain load (a 16-byte bulk copy
  // would cost the SM's bulk-copy unit as much as a 1 KiB one); not through the
  // read-only path, since a fused layer writes the slot earlier in the launch
  static __device__ __forceinline__ float2 glob(const uint8_t* blob, const BlobOff& o) {
    return *reinterpret_cast<const float2*>(blob + o.glob);
  }
  // per-lane partial gate / up sums over the lane's elements of chunk c
  static __device__ __forceinline__ void dot4(const uint8_t* gc, const uint8_t* uc,
                                              const uint8_t* gsc, const uint8_t* usc,
                                              const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(gc + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(gc + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(uc + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(uc + 512 + lane * 16);
    const float2 sg0 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(gsc + lane * 2));
    const float2 sg1 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(gsc + 64 + lane * 2));
    const float2 su0 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(usc + lane * 2));
    const float2 su1 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(usc + 64 + lane * 2));
    const int ua = c * 256 + lane * 4, ub = ua + 128;
    uint4 x0 = xr[xswz(ua)], x1 = xr[xswz(ua + 1)], x2 = xr[xswz(ua + 2)], x3 = xr[xswz(ua + 3)];
    g = fmaf(dot8_fp4_h(g0.x, x0) + dot8_fp4_h(g0.y, x1), sg0.x, g);
    g = fmaf(dot8_fp4_h(g0.z, x2) + dot8_fp4_h(g0.w, x3), sg0.y, g);
    u = fmaf(dot8_fp4_h(u0.x, x0) + dot8_fp4_h(u0.y, x1), su0.x, u);
    u = fmaf(dot8_fp4_h(u0.z, x2) + dot8_fp4_h(u0.w, x3), su0.y, u);
    x0 = xr[xswz(ub)], x1 = xr[xswz(ub + 1)], x2 = xr[xswz(ub + 2)], x3 = xr[xswz(ub + 3)];
    g = fmaf(dot8_fp4_h(g1.x, x0) + dot8_fp4_h(g1.y, x1), sg1.x, g);
    g = fmaf(dot8_fp4_h(g1.z, x2) + dot8_fp4_h(g1.w, x3), sg1.y, g);
    u = fmaf(dot8_fp4_h(u1.x, x0) + dot8_fp4_h(u1.y, x1), su1.x, u);
    u = fmaf(dot8_fp4_h(u1.z, x2) + dot8_fp4_h(u1.w, x3), su1.y, u);
  }
  // the chunk in a per-warp slot
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    dot4(slot, slot + 1024, slot + 2048, slot + 2176, xr, c, lane, g, u);
  }
};
template <>
struct ItemA<MOE_W_BF16> {
  static constexpr int CW = 512;
  static constexpr int BYTES = 2 * 1024;
  static __device__ __forceinline__ uint32_t issue(uint8_t* slot, const uint8_t* blob,
                                                   const BlobOff& o, int H, int i, int c,
                                                   uint64_t* bar, uint64_t pol) {
    const size_t e = ((size_t)i * H + c * 512) * 2;
    bulk_g2s(slot, blob + o.mat[0] + e, 1024, bar, pol);
    bulk_g2s(slot + 1024, blob + o.mat[1] + e, 1024, bar, pol);
    return BYTES;
  }
  static __device__ __forceinline__ void dot4(const uint8_t* gc, const uint8_t* uc,
                                              const uint8_t* gsc, const uint8_t* usc,
                                              const uint4* xr, int c, int lane,
                                             float& gs, float& us) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint4 xv = xr[xswz(c * 64 + 32 * s + lane)];
      gs = dot8_bf16_bf(*reinterpret_cast<const uint4*>(gc + 512 * s + lane * 16), xv, gs);
      us = dot8_bf16_bf(*reinterpret_cast<const uint4*>(uc + 512 * s + lane * 16), xv, us);
    }
  }
  // the chunk in a per-warp slot
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    dot4(slot, slot + 1024, slot, slot, xr, c, lane, g, u);
  }
  static __device__ __forceinline__ float2 glob(const uint8_t*, const BlobOff&) {
    return make_float2(1.f, 1.f);
  }
};
// MXFP4: chunks of 2048 elements as NVFP4; one E8M0 scale per 32 elements, so
// each lane's 32-element block has one scale and no global scale applies:
//   gate codes [1024 B] | up codes [1024 B] | gate scales [64 B] | up scales [64 B].
template <>
struct ItemA<MOE_W_MXFP4> {
  static constexpr int CW = 2048;
  static constexpr int BYTES = 2 * 1024 + 2 * 64;
  static __device__ __forceinline__ uint32_t issue(uint8_t* slot, const uint8_t* blob,
                                                   const BlobOff& o, int H, int i, int c,
                                                   uint64_t* bar, uint64_t pol) {
    const size_t cr = (size_t)i * (H / 2) + c * 1024, sr = (size_t)i * (H / 32) + c * 64;
    bulk_g2s(slot, blob + o.code[0] + cr, 1024, bar, pol);
    bulk_g2s(slot + 1024, blob + o.code[1] + cr, 1024, bar, pol);
    bulk_g2s(slot + 2048, blob + o.scale[0] + sr, 64, bar, pol);
    bulk_g2s(slot + 2112, blob + o.scale[1] + sr, 64, bar, pol);
    return BYTES;
  }
  static __device__ __forceinline__ float2 glob(const uint8_t*, const BlobOff&) {
    return make_float2(1.f, 1.f);
  }
  static __device__ __forceinline__ void dot4(const uint8_t* gc, const uint8_t* uc,
                                              const uint8_t* gsc, const uint8_t* usc,
                                              const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(gc + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(gc + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(uc + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(uc + 512 + lane * 16);
    const float sg0 = e8m0_f32(gsc[lane]), sg1 = e8m0_f32(gsc[32 + lane]);
    const float su0 = e8m0_f32(usc[lane]), su1 = e8m0_f32(usc[32 + lane]);
    const int ua = c * 256 + lane * 4, ub = ua + 128;
    uint4 x0 = xr[xswz(ua)], x1 = xr[xswz(ua + 1)], x2 = xr[xswz(ua + 2)], x3 = xr[xswz(ua + 3)];
    g = fmaf((dot8_fp4_h(g0.x, x0) + dot8_fp4_h(g0.y, x1)) +
             (dot8_fp4_h(g0.z, x2) + dot8_fp4_h(g0.w, x3)), sg0, g);
    u = fmaf((dot8_fp4_h(u0.x, x0) + dot8_fp4_h(u0.y, x1)) +
             (dot8_fp4_h(u0.z, x2) + dot8_fp4_h(u0.w, x3)), su0, u);
    x0 = xr[xswz(ub)], x1 = xr[xswz(ub + 1)], x2 = xr[xswz(ub + 2)], x3 = xr[xswz(ub + 3)];
    g = fmaf((dot8_fp4_h(g1.x, x0) + dot8_fp4_h(g1.y, x1)) +
             (dot8_fp4_h(g1.z, x2) + dot8_fp4_h(g1.w, x3)), sg1, g);
    u = fmaf((dot8_fp4_h(u1.x, x0) + dot8_fp4_h(u1.y, x1)) +
             (dot8_fp4_h(u1.z, x2) + dot8_fp4_h(u1.w, x3)), su1, u);
  }
  // the chunk in a per-warp slot
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    dot4(slot, slot + 1024, slot + 2048, slot + 2112, xr, c, lane, g, u);
  }
};

// Q4_0 (banked): chunks of 2048 elements; one fp16 scale d per 32 elements, so
// each lane's 32-element block has one scale, weight = d * (q - 8):
//   gate codes [1024 B] | up codes [1024 B] | gate scales [128 B] | up scales [128 B].
template <>
struct ItemA<MOE_W_Q4_0> {
  static constexpr int CW = 2048;
  static constexpr int BYTES = 2 * 1024 + 2 * 128;
  static __device__ __forceinline__ uint32_t issue(uint8_t* slot, const uint8_t* blob,
                                                   const BlobOff& o, int H, int i, int c,
                                                   uint64_t* bar, uint64_t pol) {
    const size_t cr = (size_t)i * (H / 2) + c * 1024, sr = (size_t)i * (H / 16) + c * 128;
    bulk_g2s(slot, blob + o.code[0] + cr, 1024, bar, pol);
    bulk_g2s(slot + 1024, blob + o.code[1] + cr, 1024, bar, pol);
    bulk_g2s(slot + 2048, blob + o.scale[0] + sr, 128, bar, pol);
    bulk_g2s(slot + 2176, blob + o.scale[1] + sr, 128, bar, pol);
    return BYTES;
  }
  static __device__ __forceinline__ float2 glob(const uint8_t*, const BlobOff&) {
    return make_float2(1.f, 1.f);
  }
  static __device__ __forceinline__ void dot4(const uint8_t* gc, const uint8_t* uc,
                                              const uint8_t* gsc, const uint8_t* usc,
                                              const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(gc + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(gc + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(uc + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(uc + 512 + lane * 16);
    const uint16_t* scg = reinterpret_cast<const uint16_t*>(gsc);
    const uint16_t* scu = reinterpret_cast<const uint16_t*>(usc);
    const float sg0 = f16_f32(scg[lane]), sg1 = f16_f32(scg[32 + lane]);
    const float su0 = f16_f32(scu[lane]), su1 = f16_f32(scu[32 + lane]);
    const int ua = c * 256 + lane * 4, ub = ua + 128;
    uint4 x0 = xr[xswz(ua)], x1 = xr[xswz(ua + 1)], x2 = xr[xswz(ua + 2)], x3 = xr[xswz(ua + 3)];
    g = fmaf((dot8_q4_h(g0.x, x0) + dot8_q4_h(g0.y, x1)) +
             (dot8_q4_h(g0.z, x2) + dot8_q4_h(g0.w, x3)), sg0, g);
    u = fmaf((dot8_q4_h(u0.x, x0) + dot8_q4_h(u0.y, x1)) +
             (dot8_q4_h(u0.z, x2) + dot8_q4_h(u0.w, x3)), su0, u);
    x0 = xr[xswz(ub)], x1 = xr[xswz(ub + 1)], x2 = xr[xswz(ub + 2)], x3 = xr[xswz(ub + 3)];
    g = fmaf((dot8_q4_h(g1.x, x0) + dot8_q4_h(g1.y, x1)) +
             (dot8_q4_h(g1.z, x2) + dot8_q4_h(g1.w, x3)), sg1, g);
    u = fmaf((dot8_q4_h(u1.x, x0) + dot8_q4_h(u1.y, x1)) +
             (dot8_q4_h(u1.z, x2) + dot8_q4_h(u1.w, x3)), su1, u);
  }
  // the chunk in a per-warp slot
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    dot4(slot, slot + 1024, slot + 2048, slot + 2176, xr, c, lane, g, u);
  }
};

constexpr int kSlotBytes = 2432;
constexpr int kTileGroups = 4;  // tile mode: the CTA's rows in groups, one barrier each
// a gate/up row's code and scale bytes (the whole row, H elements)
__host__ __device__ constexpr int row_code_bytes(int fmt, int H) { return fmt == MOE_W_BF16 ? 2 * H : H / 2; }
__host__ __device__ constexpr int row_scale_bytes(int fmt, int H) {
  return fmt == MOE_W_BF16 ? 0 : (fmt == MOE_W_MXFP4 ? H / 32 : H / 16);
}  // >= ItemA<*>::BYTES, a multiple of 128

// cp.async of 16, 8 or 4 bytes, global -> shared (this thread's own data)
__device__ __forceinline__ void cp16_async(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8_async(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4_async(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// ------------------------------------------------------------ clusters
constexpr int kCS = 4;  // CTAs per cluster: one unit (task, part of I) per cluster

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders the shared-memory writes
// before it (to this CTA or, through DSMEM, to the others) with the reads after it
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// the copy warps' side of the cluster barrier: arrive without waiting (they
// publish nothing through it), and wait for a phase later
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// the compute warps alone (named barrier 1 over kT threads): the copy warps
// of a layer launch never take part
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kT) : "memory"); }
__device__ __forceinline__ bool csync_and(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)v), "n"(kT)
      : "memory");
  return r != 0;
}
// warps 0 and 1 hand the task list and the launch index to the copy warps
// (named barrier 2): the two arrive, the copy warps wait
constexpr int kHandoff = 64 + 32 * kCW;
__device__ __forceinline__ void handoff_arrive() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kHandoff) : "memory");
}
__device__ __forceinline__ void handoff_wait() {
  asm volatile("bar.sync 2, %0;" ::"n"(kHandoff) : "memory");
}
// v into the float at the shared-memory offset of `local`, in CTA `rank` of the cluster
__device__ __forceinline__ void st_cluster_f32(const float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)),
               "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// ------------------------------------------------------------ the launch's arguments
// One launch computes a group of expert FFNs for a decode-sized step.  Tasks
// are (route, expert blob) pairs in route order, plus one shared-expert task
// per batch row in the layer modes.  A task's intermediate I is cut into P
// parts (Pr for a routed task, Ps for a shared-expert task, both fixed by the
// layer's shape so that every launch mode splits a task alike); a unit (task
// t, part p) belongs to one cluster of kCS CTAs:
//   CTA r of the cluster computes h[i] = silu(g_i) * u_i for its I / (P kCS)
//     rows of the part (phase A) and stores them into every CTA of the cluster
//     (distributed shared memory), then a cluster barrier;
//   CTA r then applies the part's columns of the down projection to its
//     H / kCS output rows (phase B): y_tp[n] = sum_{i in part p} W_d[n][i] h[i],
//     and adds w_t * y_tp[n] (w: routing weight, or the shared expert's
//     sigmoid gate, times the down global scale) to the layer's sum for row b
//     as a 64-bit fixed-point integer (2^-32 units, red.add): integer adds give
//     the same bits in any order, so every launch mode and every schedule of
//     the units sums alike;
//   the last unit to finish an output slice (a counter per slice) converts
//     the slice: out[b][n] = bf16(sum), and zeroes the sums.
// No grid-wide barrier and no round trip of h through L2: clusters never wait
// for one another, except for a copy of a missed expert.
struct FusedArgs {
  int H, I, layer, k, R, n_rows;
  const uint16_t* x;
  const int32_t* slot_ids;
  const uint8_t* fixed_blob;   // SHARED: the shared expert's blob
  const float* w;              // routing weights
  const uint16_t* gate_w;      // the shared expert's gate vector
  float* ys;                   // SHARED: output [n_rows][H]; ROUTED: input (may be null)
  __nv_bfloat16* out;          // ROUTED and layer output
  unsigned long long* status;
  int Pr, Ps;                  // parts of I per routed task, per shared-expert task
  int n_units;                 // routes x Pr + shared tasks x Ps, some empty when routes are invalid
  int first_cluster;           // 1 when cluster 0 admits (kLayerAdmit), else 0
  int one_round;               // every unit has a cluster of its own
  unsigned long long* acc;     // [n_rows][H] the layer's fixed-point sums (zero between launches)
  int acc_out;                 // SHARED: convert the sums into ys (else the routed launch adds on)
  int pb_room;                 // shared-memory bytes per thread for a staged phase-B row part
  int tile;                    // phase A as whole tiles: a CTA's gate/up rows by a few large
                               // bulk copies (rows of one chunk), else per-warp chunk slots
  int area;                    // bytes of the phase-A area (the slots, or the largest tile)
  unsigned* slice_cnt;         // [kCS] units done per output slice (the last resets it)
  // fused layer
  const uint8_t* shared_blob;  // shared expert (one extra task per row), null = none
  const int32_t* gplan0;       // demand plan: its experts are copied here and waited on
  const int32_t* gplan1;       // prefetch plan of the next layer (copied only), or null
  int* gdone;                  // [plan entries] pieces copied; zero at entry, reset here
  // fused layer with the admission inside the launch: CTA 0 admits (and
  // prefetch-admits), the other clusters compute
  const int32_t* ids;          // the step's expert ids [R]
  int32_t* slot_out;           // [R] slot ids, written by the admission
  int cap;                     // fetch cap (< 0: none)
  const int32_t* pred;         // the next layer's predicted ids, or null
  int n_pred;
  int adm_cached;              // the admission keeps the pool in shared memory
  unsigned long long* epoch;   // grows by gridDim.x per launch: launch j = old / gridDim.x
  unsigned long long* pseq;    // 2j+1: slot ids and demand plan of launch j out; 2j+2: prefetch plan too
  // [R] launch j's slot of its misses' rank i (ascending id): (2j+1) << 32 | slot,
  // low word ~0u when not admitted; the tag makes an older launch's word stale
  unsigned long long* sslot;
  uint8_t* stage;              // stage_n slot-sized areas the step's misses are copied into
  int stage_n;                 // (0: misses wait for the admission and go to their slots)
};

// ------------------------------------------------------------ waits and copies
// Bounded wait of a warp (lane 0 reads, the warp follows) until *a.pseq >=
// target; then every lane acquires too.  False (and MOE_STATUS_TIMEOUT) on timeout.
__device__ bool wait_seq(const FusedArgs& a, unsigned long long target, int lane) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    int s = 0;  // 1: published, 2: timed out
    if (lane == 0) {
      const unsigned long long v = ld_acquire_u64(a.pseq);
      s = v >= target ? 1 : (now_ns() - t0 > kWaitNs ? 2 : 0);
    }
    s = __shfl_sync(0xffffffffu, s, 0);
    if (s == 1) {
      (void)ld_acquire_u64(a.pseq);
      return true;
    }
    if (s == 2) {
      if (lane == 0) flag_timeout(a.status);
      return false;
    }
    __nanosleep(256);
  }
}
// Bounded wait of a warp until the piece counter reaches n.
__device__ bool wait_count(const int* ctr, int n, unsigned long long* status, int lane) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    int s = 0;  // 1: complete, 2: timed out
    if (lane == 0) {
      int v;
      asm volatile("ld.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      s = v >= n ? 1 : (now_ns() - t0 > kWaitNs ? 2 : 0);
    }
    s = __shfl_sync(0xffffffffu, s, 0);
    if (s == 1) {  // every lane acquires the copies the count covers
      int v;
      asm volatile("ld.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      (void)v;
      return true;
    }
    if (s == 2) {
      if (lane == 0) flag_timeout(status);
      return false;
    }
    __nanosleep(256);
  }
}
__device__ __forceinline__ uint8_t* slot_ptr(const DevState& st, int layer, int s) {
  return st.slots + ((size_t)pool_of(st, layer) * st.S + s) * st.stride;
}
__device__ __forceinline__ int pieces_per_expert(const DevState& st) {
  return max(1, (int)((st.slot_bytes + kPiece - 1) / kPiece));
}
// Piece j of entry i of a plan, from pinned host memory into its slot (a
// warp, 4 KiB); counted in ctr[i] (when given) after the slot holds it.
__device__ void copy_plan_piece(const DevState& st, const int32_t* plan, int i, int j, int* ctr,
                                int lane) {
  const int s = plan[1 + 3 * i], L = plan[2 + 3 * i], e = plan[3 + 3 * i];
  if ((unsigned)s < (unsigned)st.S && (unsigned)L < (unsigned)st.L && (unsigned)e < (unsigned)st.E) {
    const size_t off = (size_t)j * kPiece;
    const int len = (int)min((size_t)kPiece, st.slot_bytes - off);
    const uint4* src = reinterpret_cast<const uint4*>(st.host_blob[L * st.E + e] + off);
    uint4* dst = reinterpret_cast<uint4*>(slot_ptr(st, L, s) + off);
    const int nv = len / 16;
    uint4 v[kPiece / 512];
#pragma unroll
    for (int u = 0; u < kPiece / 512; ++u)
      if (lane + 32 * u < nv) v[u] = src[lane + 32 * u];
#pragma unroll
    for (int u = 0; u < kPiece / 512; ++u)
      if (lane + 32 * u < nv) dst[lane + 32 * u] = v[u];
  }
  __threadfence();  // this lane's stores, before the count that publishes them
  __syncwarp();
  if (ctr && lane == 0) {
    __threadfence();
    atomicAdd(ctr + i, 1);
  }
}
// A staging piece: piece j of the step's missed expert e (staging entry i),
// from pinned host memory into the staging entry and into the slot the
// admission gave the expert (a victim: no task of this step reads it).  While
// the host reads are in flight the warp polls CTA 0's word for the entry (the
// slot, tagged with this launch).  Counted once both copies are written.
__device__ void stage_piece(const DevState& st, const FusedArgs& a, int i, int e, int j,
                            unsigned long long seq0, int lane) {
  const size_t off = (size_t)j * kPiece;
  const int len = (int)min((size_t)kPiece, st.slot_bytes - off);
  const uint4* src = reinterpret_cast<const uint4*>(st.host_blob[a.layer * st.E + e] + off);
  uint4* dst = reinterpret_cast<uint4*>(a.stage + (size_t)i * st.stride + off);
  const int nv = len / 16;
  uint4 v[kPiece / 512];
#pragma unroll
  for (int u = 0; u < kPiece / 512; ++u)
    if (lane + 32 * u < nv) v[u] = src[lane + 32 * u];
  uint32_t sl = ~0u;  // the slot (warp-uniform), ~0u: none or timed out
  {
    const unsigned long long tag = seq0 + 1, t0 = now_ns();
    for (;;) {
      int s = 0;  // 1: this launch's word, 2: timed out
      unsigned long long w = 0;
      if (lane == 0) {
        asm volatile("ld.relaxed.gpu.u64 %0, [%1];" : "=l"(w) : "l"(a.sslot + i) : "memory");
        s = (w >> 32) == (tag & 0xffffffffull) ? 1 : (now_ns() - t0 > kWaitNs ? 2 : 0);
      }
      s = __shfl_sync(0xffffffffu, s, 0);
      if (s == 1) {
        sl = __shfl_sync(0xffffffffu, (uint32_t)w, 0);
        break;
      }
      if (s == 2) {
        if (lane == 0) flag_timeout(a.status);
        break;
      }
      __nanosleep(128);
    }
  }
#pragma unroll
  for (int u = 0; u < kPiece / 512; ++u)
    if (lane + 32 * u < nv) dst[lane + 32 * u] = v[u];
  if (sl < (uint32_t)st.S) {
    uint4* sdst = reinterpret_cast<uint4*>(slot_ptr(st, a.layer, (int)sl) + off);
#pragma unroll
    for (int u = 0; u < kPiece / 512; ++u)
      if (lane + 32 * u < nv) sdst[lane + 32 * u] = v[u];
  }
  __threadfence();  // this lane's stores, before the count that publishes them
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(a.gdone + i, 1);
  }
}

// ------------------------------------------------------------ phase B rows
// A down-projection row's part of I (IP elements) dotted with the part's h
// (fp32, shared memory), one thread per row, 32 elements per step; per-block
// scales as the format defines, no global scale (applied with the routing
// weight).  ldc(c) gives the row part's c-th 16 code bytes (4-bit formats) or
// its c-th 64 bytes as four uint4 (bf16, via ldb), lds(c) the scale bits of
// step c; each step's sum is formed in a fixed order.
template <int FMT, typename LC, typename LS>
__device__ __forceinline__ float rowb_dot(int IP, const float* hp, LC ldc, LS lds) {
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < IP / 32; ++c) {
    float h[32];  // the step's h, by 16-byte shared-memory loads (broadcasts)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = reinterpret_cast<const float4*>(hp + 32 * c)[q];
      h[4 * q] = v.x, h[4 * q + 1] = v.y, h[4 * q + 2] = v.z, h[4 * q + 3] = v.w;
    }
    if (FMT == MOE_W_BF16) {
      uint4 w[4];
      ldc(c, w);
      float q = dot8_bf16_f(w[0], h, 0.f);
      q = dot8_bf16_f(w[1], h + 8, q);
      q = dot8_bf16_f(w[2], h + 16, q);
      q = dot8_bf16_f(w[3], h + 24, q);
      acc += q;
    } else {
      uint4 w[1];
      ldc(c, w);
      const uint32_t sb = lds(c);
      if (FMT == MOE_W_NVFP4) {
        const float2 sc = e4m3x2_f32(sb);
        acc = fmaf(dot8_fp4_f(w[0].x, h) + dot8_fp4_f(w[0].y, h + 8), sc.x, acc);
        acc = fmaf(dot8_fp4_f(w[0].z, h + 16) + dot8_fp4_f(w[0].w, h + 24), sc.y, acc);
      } else if (FMT == MOE_W_MXFP4) {
        acc = fmaf((dot8_fp4_f(w[0].x, h) + dot8_fp4_f(w[0].y, h + 8)) +
                       (dot8_fp4_f(w[0].z, h + 16) + dot8_fp4_f(w[0].w, h + 24)),
                   e8m0_f32(sb), acc);
      } else {  // Q4_0
        acc = fmaf((dot8_q4_f(w[0].x, h) + dot8_q4_f(w[0].y, h + 8)) +
                       (dot8_q4_f(w[0].z, h + 16) + dot8_q4_f(w[0].w, h + 24)),
                   f16_f32(sb), acc);
      }
    }
  }
  return acc;
}
// scale bytes of a down row's part per 32 elements (0 for bf16)
template <int FMT>
__host__ __device__ constexpr int scale_bytes_per32() {
  return FMT == MOE_W_NVFP4 ? 2 : (FMT == MOE_W_Q4_0 ? 2 : (FMT == MOE_W_MXFP4 ? 1 : 0));
}
// the scale bits of step c from `sp` (a row part's scales)
template <int FMT>
__device__ __forceinline__ uint32_t scale_at(const uint8_t* sp, int c) {
  if (FMT == MOE_W_MXFP4) return sp[c];
  return *reinterpret_cast<const uint16_t*>(sp + 2 * c);
}
// Fixed-point term of the layer sum: v * 2^32 rounded to nearest, kept within
// +-2^58 so that any number of terms up to 32 stays inside int64.
constexpr double kFix = 4294967296.0;
__device__ __forceinline__ unsigned long long to_fixed(float v) {
  double d = (double)v * kFix;
  d = fmin(fmax(d, -2.8823037615171174e17), 2.8823037615171174e17);  // +-2^58
  return (unsigned long long)__double2ll_rn(d);
}
__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

constexpr int kPending = -2;
constexpr int kPbWords = 128;  // admission inside: a bitmap over at most 4096 experts
// CTA 0 of a layer launch with the admission inside: the admission of
// a.layer (the same routine as the standalone kernel, on this CTA's threads),
// then the prefetch admission of a.layer + 1 when predictions are given.  It
// needs no word from the computing CTAs: a hit cannot be evicted by its own
// admission, and an installed miss's map entry carries kMapPending until this
// launch has copied it in, so a computing CTA reading the map sees a miss as
// a miss whenever it reads.  It publishes its results with release stores to
// a.pseq: 2j + 1 once the slot ids and the demand plan of launch j are out,
// 2j + 2 once the prefetch plan is too.
__device__ __noinline__ void admit_cta(const DevState& st, const FusedArgs& a, uint8_t* sm,
                                       unsigned long long j) {
  using namespace admission;
  AdmitShared<kT>& sh = *reinterpret_cast<AdmitShared<kT>*>(sm);
  unsigned char* dyn = sm + (sizeof(AdmitShared<kT>) + 127) / 128 * 128;
  auto none = [] {};
  if (a.adm_cached)
    admit_body<true, kT>(st, a.layer, a.ids, a.slot_out, a.R, a.cap, dyn, sh, none, kMapPending);
  else
    admit_body<false, kT>(st, a.layer, a.ids, a.slot_out, a.R, a.cap, dyn, sh, none, kMapPending);
  __threadfence();
  sync_nt<kT>();
  // the slot of each miss rank for the staging copies: the admitted misses are
  // the first entries of the miss list (ascending id), one plan entry each
  if (threadIdx.x < a.R) {
    const int np0 = a.gplan0[0];
    const uint32_t s = threadIdx.x < np0 ? (uint32_t)a.gplan0[1 + 3 * threadIdx.x] : ~0u;
    a.sslot[threadIdx.x] = (2 * j + 1) << 32 | s;
  }
  if (threadIdx.x == 0) st_release_u64(a.pseq, 2 * j + 1);
  if (a.pred && a.n_pred > 0) {
    prefetch_body<kT>(st, a.layer + 1, a.pred, a.n_pred, const_cast<int32_t*>(a.gplan1),
                      reinterpret_cast<int*>(dyn), sh);
    __threadfence();
    sync_nt<kT>();
  }
  if (threadIdx.x == 0) st_release_u64(a.pseq, 2 * j + 2);
}


template <int FMT, int MODE>
__global__ void __maxnreg__(max_reg(MODE))
    ffn_cluster_kernel(DevState st, FusedArgs a) {
  constexpr bool SHARED = MODE == kShared, ADMIT = MODE == kLayerAdmit;
  constexpr bool LAYER = MODE == kLayer || ADMIT;
  constexpr bool FP4 = FMT != MOE_W_BF16;  // 4-bit codes (NVFP4, MXFP4, Q4_0): f16 x
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ unsigned long long s_j;  // admission inside: this launch's index
  __shared__ Tasks tk;
  __shared__ int ts[kMaxRows + 1];         // tasks of batch row b: [ts[b], ts[b+1])
  __shared__ unsigned int xmax[kMaxRows];  // per row max |x| (float bits, only when > 2^14)
  __shared__ float xinv[kMaxRows];         // per row 1 / (power-of-two scale applied to x)
  __shared__ uint64_t bar_a[kW][2];        // per-warp phase-A slot barriers
  __shared__ uint64_t bar_t[kTileGroups];  // tile mode: the row groups' barriers
  __shared__ int s_npend;                  // admission inside: tasks not resident at entry
  __shared__ int s_npx;                    // ... their distinct experts (staging entries)
  __shared__ int s_staged;                 // ... copied into the staging area (else: slots)
  __shared__ unsigned s_pbits[kPbWords];   // ... bitmap of those experts
  __shared__ int s_pexp[kMaxRoutes];       // ... in ascending id: staging entry -> expert
  __shared__ int s_last;                   // this CTA converts its output slice
  __shared__ float s_wsc;                  // the current unit's weight in the layer sum
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const int cl = (int)blockIdx.x / kCS;
  const int H = a.H, I = a.I, k = a.k, n_rows = a.n_rows;
  const BlobOff o(H, I, FMT);
  const bool copier = LAYER && warp >= kW;  // a copy warp
  // every CTA of launch j adds one to a.epoch: j = old / gridDim.x (read
  // after the next barrier of the warps that need it)
  if (ADMIT && threadIdx.x == 32) s_j = atomicAdd(a.epoch, 1ull) / gridDim.x;
  unsigned long long seq0 = 0;  // a.pseq before this launch's admission (set once s_j is read)
  const int ppe = LAYER ? pieces_per_expert(st) : 1;
  const bool pf_plan = LAYER && a.gplan1 && (!ADMIT || (a.pred && a.n_pred > 0));
  // The copy workers, each a warp with an index gw of W, pieces q = gw + i W.
  // Demand copies (the step's misses): the copy warps of every CTA and, with
  // the admission inside, every warp of the admission cluster's CTAs 1..3;
  // prefetch copies: the same and CTA 0's warps once it has admitted.
  const long bx = blockIdx.x;
  const long W_pf = ADMIT ? (long)kCS * kNW + ((long)gridDim.x - kCS) * kCW : (long)gridDim.x * kCW;
  const long gw_pf = !ADMIT ? bx * kCW + (warp - kW)
                     : bx < kCS ? bx * kNW + warp : (long)kCS * kNW + (bx - kCS) * kCW + (warp - kW);
  const long W_d = ADMIT ? W_pf - kNW : W_pf;
  const long gw_d = ADMIT ? gw_pf - kNW : gw_pf;
  // the next layer's prefetched experts
  auto copy_prefetch = [&](long gw, long W) {
    if (!pf_plan) return;
    if (ADMIT && !wait_seq(a, seq0 + 2, lane)) return;
    const int np1 = a.gplan1[0];
    for (long q = gw; q < (long)np1 * ppe; q += W)
      copy_plan_piece(st, a.gplan1, (int)(q / ppe), (int)(q % ppe), nullptr, lane);
  };
  if (ADMIT && blockIdx.x == 0) {  // CTA 0 admits, then copies prefetched experts
    __syncthreads();               // s_j
    seq0 = 2 * s_j;
    if (!copier) admit_cta(st, a, sm, s_j);
    copy_prefetch(gw_pf, W_pf);
    return;
  }
  const int ccl = cl - a.first_cluster, ncl = (int)gridDim.x / kCS - a.first_cluster;

  // ---- entry: the task list (warp 0) and x (everyone) in flight at once
  const int nx8 = n_rows * H / 8;
  uint4 xw[kXW];
#pragma unroll
  for (int j = 0; j < kXW; ++j) {
    const int i = threadIdx.x + j * kT;
    if (!copier && i < nx8) xw[j] = reinterpret_cast<const uint4*>(a.x)[i];
  }
  if (threadIdx.x < kMaxRows) xmax[threadIdx.x] = 0u;
  if (lane == 0 && !copier) {
    mbar_init(&bar_a[warp][0], 1);
    mbar_init(&bar_a[warp][1], 1);
    if (warp == 0)
      for (int g = 0; g < kTileGroups; ++g) mbar_init(&bar_t[g], 1);
    fence_barrier_init();
  }
  // ---- shared memory: x [n_rows][H] | phase-A area (two slots per warp, or a
  // tile) | h [2][IPmax] | staged phase-B row parts [kT][pb_room]
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);
  uint8_t* ring = sm + ((size_t)n_rows * H * 2 + 127) / 128 * 128;
  uint8_t* slots = ring + (size_t)warp * 2 * kSlotBytes;  // this warp's two slots
  const int IPmax = I / min(a.Pr, a.Ps);  // the longest part
  float* hbuf = reinterpret_cast<float*>(ring + (size_t)a.area);  // [2][IPmax]
  uint8_t* pbuf = reinterpret_cast<uint8_t*>(hbuf + 2 * (size_t)IPmax);
  const int pb_room = a.pb_room;
  const uint64_t pol = l2_evict_first();
  constexpr int CW = ItemA<FMT>::CW;
  const int KC = H / CW;  // phase-A chunks per row
  bool failed = false;    // a timed-out wait: the rest computes nothing, but every barrier is kept
  uint32_t ph[2] = {0u, 0u};  // completed phases of the warp's two slot barriers

  // tile mode: the unit's IPC gate and up rows [i0, i0 + IPC) (contiguous in
  // each bank) and their scales, in kTileGroups row groups, by thread 0
  const int RB = row_code_bytes(FMT, H), SB = row_scale_bytes(FMT, H);
  auto issue_tile = [&](const uint8_t* blob, int i0, int IPC, int g_only) {  // g_only < 0: all groups
    const int GR = IPC / kTileGroups;
    uint8_t* gc = ring;
    uint8_t* uc = ring + (size_t)IPC * RB;
    uint8_t* gs = ring + (size_t)2 * IPC * RB;
    uint8_t* us = gs + (size_t)IPC * SB;
    const size_t c0 = FP4 ? o.code[0] : o.mat[0], c1 = FP4 ? o.code[1] : o.mat[1];
    for (int g = 0; g < kTileGroups; ++g) {
      if (g_only >= 0 && g != g_only) continue;
      const size_t r0 = (size_t)i0 + (size_t)g * GR;
      mbar_expect_tx(&bar_t[g], (uint32_t)(GR * (2 * RB + 2 * SB)));
      bulk_g2s(gc + (size_t)g * GR * RB, blob + c0 + r0 * RB, (uint32_t)(GR * RB), &bar_t[g], pol);
      bulk_g2s(uc + (size_t)g * GR * RB, blob + c1 + r0 * RB, (uint32_t)(GR * RB), &bar_t[g], pol);
      if (SB > 0) {
        bulk_g2s(gs + (size_t)g * GR * SB, blob + o.scale[0] + r0 * SB, (uint32_t)(GR * SB),
                 &bar_t[g], pol);
        bulk_g2s(us + (size_t)g * GR * SB, blob + o.scale[1] + r0 * SB, (uint32_t)(GR * SB),
                 &bar_t[g], pol);
      }
    }
  };
  if (warp == 0) {
    const uint8_t* b0 = nullptr;
    const uint8_t* b1 = nullptr;
    int sl0 = -1, sl1 = -1;       // slot ids (admission inside: the map entry at entry)
    int e0 = -1, e1 = -1;         // admission inside: expert ids
    bool v0 = false, v1 = false;  // the route is a task
    auto resolve = [&](int r, int& slot, int& e) -> bool {
      if (a.fixed_blob) return true;
      if (ADMIT) {  // a valid id is a task: resident now, or being admitted by CTA 0
        e = a.ids[r];
        if ((unsigned)e >= (unsigned)st.E) return false;
        slot = st.map[a.layer * st.E + e];  // -1, or kMapPending set: not resident
        return true;
      }
      slot = a.slot_ids[r];
      return (unsigned)slot < (unsigned)st.S;
    };
    if (lane < a.R) v0 = resolve(lane, sl0, e0);
    if (lane + 32 < a.R) v1 = resolve(lane + 32, sl1, e1);
    if (v0) b0 = a.fixed_blob ? a.fixed_blob : (sl0 >= 0 ? slot_ptr(st, a.layer, sl0) : nullptr);
    if (v1) b1 = sl1 >= 0 ? slot_ptr(st, a.layer, sl1) : nullptr;
    int pe0 = -1, pe1 = -1;
    const bool p0 = ADMIT && v0 && sl0 < 0, p1 = ADMIT && v1 && sl1 < 0;  // missed
    if (ADMIT) {
      // the distinct missed experts in ascending id: the staging entries
      const int nw = (st.E + 31) / 32;
      for (int w = lane; w < nw; w += 32) s_pbits[w] = 0;
      __syncwarp();
      if (p0) atomicOr(&s_pbits[e0 >> 5], 1u << (e0 & 31));
      if (p1) atomicOr(&s_pbits[e1 >> 5], 1u << (e1 & 31));
      __syncwarp();
      auto rank_of = [&](int e) {
        int r = __popc(s_pbits[e >> 5] & ((1u << (e & 31)) - 1u));
        for (int w = 0; w < (e >> 5); ++w) r += __popc(s_pbits[w]);
        return r;
      };
      const int x0 = p0 ? rank_of(e0) : -1, x1 = p1 ? rank_of(e1) : -1;
      if (p0) s_pexp[x0] = e0;
      if (p1) s_pexp[x1] = e1;
      int npx = 0;
      for (int w = lane; w < nw; w += 32) npx += __popc(s_pbits[w]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) npx += __shfl_xor_sync(0xffffffffu, npx, off);
      // uncapped steps copy their misses at once into staging entries; with a
      // fetch cap (or too many misses) they wait for the admission's slots
      const bool stg = a.stage && a.cap < 0 && npx <= a.stage_n;
      if (stg) {
        if (p0) b0 = a.stage + (size_t)x0 * st.stride, pe0 = x0;
        if (p1) b1 = a.stage + (size_t)x1 * st.stride, pe1 = x1;
      } else {
        pe0 = p0 ? kPending : -1;
        pe1 = p1 ? kPending : -1;
      }
      const int np = __popc(__ballot_sync(0xffffffffu, p0)) + __popc(__ballot_sync(0xffffffffu, p1));
      if (lane == 0) {
        s_npend = np;
        s_npx = npx;
        s_staged = stg;
      }
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, v0);
    const unsigned m1 = __ballot_sync(0xffffffffu, v1);
    const unsigned lt = (1u << lane) - 1u;
    // valid routes below route index lim
    auto below = [&](int lim) {
      const unsigned a0 = lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u);
      const unsigned a1 = lim >= 64 ? 0xffffffffu : (lim <= 32 ? 0u : ((1u << (lim - 32)) - 1u));
      return __popc(m0 & a0) + __popc(m1 & a1);
    };
    const int spr = (LAYER && a.shared_blob) ? 1 : 0;  // shared tasks per row (after its routes)
    auto put = [&](int p, int r, int b, const uint8_t* blob, int slot, int pe, bool pend) {
      tk.route[p] = r;
      tk.b[p] = b;
      tk.blob[p] = blob;
      tk.slot[p] = slot;
      tk.pe[p] = pe;
      tk.drop[p] = 0;
      tk.pend[p] = pend;
    };
    if (v0) {
      const int b = SHARED ? lane : lane / k;
      put(__popc(m0 & lt) + spr * b, lane, b, b0, SHARED ? -1 : sl0, pe0, p0);
    }
    if (v1) {
      const int b = (lane + 32) / k;
      put(__popc(m0) + __popc(m1 & lt) + spr * b, lane + 32, b, b1, sl1, pe1, p1);
    }
    if (spr && lane < n_rows)
      put(below((lane + 1) * k) + lane, a.R + lane, lane, a.shared_blob, -1, -1, false);
    if (lane == 0) tk.n = __popc(m0) + __popc(m1) + spr * n_rows;
    if (lane <= n_rows) ts[lane] = below(lane * k) + spr * lane;  // first task of row `lane`
  }
  // the step's missed experts: into staging entries (admission inside,
  // uncapped), into the slots the admission gave them (capped), or into the
  // demand plan's slots (kLayer); each piece counted in a.gdone
  auto copy_demand = [&](long gw, long W) {
    if (ADMIT && s_staged) {
      for (long q = gw; q < (long)s_npx * ppe; q += W)
        stage_piece(st, a, (int)(q / ppe), s_pexp[q / ppe], (int)(q % ppe), seq0, lane);
    } else if (ADMIT) {
      if (s_npend > 0 && wait_seq(a, seq0 + 1, lane)) {
        const int np0 = a.gplan0[0];
        for (long q = gw; q < (long)np0 * ppe; q += W)
          copy_plan_piece(st, a.gplan0, (int)(q / ppe), (int)(q % ppe), a.gdone, lane);
      }
    } else if (LAYER && a.gplan0) {
      const int np0 = a.gplan0[0];
      for (long q = gw; q < (long)np0 * ppe; q += W)
        copy_plan_piece(st, a.gplan0, (int)(q / ppe), (int)(q % ppe), a.gdone, lane);
    }
  };
  if (LAYER && warp < 2) handoff_arrive();  // warp 0: the task list; warp 1: s_j
  if (copier) {
    handoff_wait();
    seq0 = ADMIT ? 2 * s_j : 0;
    // the cluster barrier of each unit of this cluster: the copy warps arrive
    // for the first at once, so no unit waits for a copy it does not need
    const int n_u = ccl >= 0 && ccl < a.n_units ? (a.n_units - 1 - ccl) / ncl + 1 : 0;
    if (n_u > 0) cluster_arrive_relaxed();
    copy_demand(gw_d, W_d);
    if (n_u <= 1) copy_prefetch(gw_pf, W_pf);
    for (int i = 0; i < n_u; ++i) {
      if (i > 0) cluster_arrive_relaxed();
      cluster_wait();
    }
    if (n_u > 1) copy_prefetch(gw_pf, W_pf);
    return;
  }
  if (FP4) {  // rows whose |x| reaches 2^14 get a scale below 1
#pragma unroll
    for (int j = 0; j < kXW; ++j) {
      const int i = threadIdx.x + j * kT;
      if (i >= nx8) continue;
      const uint32_t wv[4] = {xw[j].x, xw[j].y, xw[j].z, xw[j].w};
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wv[e] << 16)),
                             fabsf(__uint_as_float(wv[e] & 0xffff0000u))));
      if (mx > 16384.f) atomicMax(&xmax[(i * 8) / H], __float_as_uint(mx));
    }
  }
  csync();  // (1) task list, ts, xmax, s_j
  seq0 = ADMIT ? 2 * s_j : 0;
  if (ADMIT && cl == 0) {  // the admission cluster's CTAs 1..3: copies only
    copy_demand(gw_d, W_d);
    copy_prefetch(gw_pf, W_pf);
    return;
  }
  const int T = tk.n;
  // a routed task has Pr parts, a shared-expert task Ps (in SHARED every task is one)
  auto parts_of = [&](int t) { return (SHARED || tk.route[t] >= a.R) ? a.Ps : a.Pr; };
  if (threadIdx.x == 0) {
    int u = 0;
    for (int t = 0; t < T; ++t) {
      tk.ubase[t] = u;
      u += parts_of(t);
    }
    tk.ubase[T] = u;
  }
  const int npend = ADMIT ? s_npend : 0;
  const int npx = ADMIT ? s_npx : 0;
  const bool staged = ADMIT && s_staged;
  const int n_pl0 = LAYER && !ADMIT && a.gplan0 ? a.gplan0[0] : 0;
  if (LAYER && !ADMIT && warp == 0) {  // the demand plan entry of each task this launch copies in
    for (int t = lane; t < T; t += 32) {
      int pe = -1;
      if (tk.slot[t] >= 0)
        for (int i = 0; i < n_pl0; ++i)
          if (a.gplan0[1 + 3 * i] == tk.slot[t]) pe = i;
      tk.pe[t] = pe;
    }
  }

  // ---- the first unit's first rows requested before x is staged, when its
  // expert is resident at entry (its task list entry is final)
  int early_u = -1;
  if (MODE != kLayer && ccl < a.n_units) {
    int t = 0, u0 = 0;
    while (t < T && u0 + parts_of(t) <= ccl) u0 += parts_of(t++);
    if (t < T && tk.pe[t] == -1 && tk.blob[t]) {
      early_u = ccl;
      const int IP = I / parts_of(t), IPC = IP / kCS;
      const int i0 = (ccl - u0) * IP + (int)crank * IPC;
      if (a.tile) {  // one row group per warp of warps 0..3
        if (lane == 0 && warp < kTileGroups) issue_tile(tk.blob[t], i0, IPC, warp);
      } else {
        const int nit = (IPC > warp ? (IPC - 1 - warp) / kW + 1 : 0) * KC;
        if (lane == 0)
          for (int it = 0; it < min(nit, 2); ++it) {
            mbar_expect_tx(&bar_a[warp][it], ItemA<FMT>::BYTES);
            ItemA<FMT>::issue(slots + it * kSlotBytes, tk.blob[t], o, H, i0 + warp + kW * (it / KC),
                              it % KC, &bar_a[warp][it], pol);
          }
      }
    }
  }

  // ---- x in shared memory: f16 with the row's power-of-two scale (4-bit
  // experts: e2m1 * x products exact in fma.rn.f32.f16), or bf16 as given
#pragma unroll
  for (int j = 0; j < kXW; ++j) {
    const int i = threadIdx.x + j * kT;
    if (i >= nx8) continue;
    const int b = (i * 8) / H, u = i - b * (H / 8);
    uint4 v = xw[j];
    if (FP4) {
      const float sc = x_scale(__uint_as_float(xmax[b]));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                             __uint_as_float(wv[e] & 0xffff0000u) * sc);
        hv[e] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      v = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
    reinterpret_cast<uint4*>(xs)[(size_t)b * (H / 8) + xswz(u)] = v;
  }
  if (threadIdx.x < n_rows)
    xinv[threadIdx.x] = FP4 ? 1.f / x_scale(__uint_as_float(xmax[threadIdx.x])) : 1.f;
  csync();  // (2) x, copy-in entries

  int ul = 0;         // units done by this cluster (selects the h buffer)
  uint32_t tph = 0;   // tile mode: tiles this CTA requested before this unit's
  for (int u = ccl; u < a.n_units; u += ncl, ++ul) {
    int t = 0;  // the unit's task (T: none, an invalid route's unit) and part
    while (t < T && tk.ubase[t + 1] <= u) ++t;
    const int Pt = t < T ? parts_of(t) : 1;
    const int p = t < T ? u - tk.ubase[t] : 0;
    const int IP = I / Pt, IPC = IP / kCS;
    float* hb = hbuf + (size_t)(ul & 1) * IPmax;
    // ---- the unit's blob: resident, or copied in by this launch's copy
    // warps.  Every warp works this out alike (the same shared task list and
    // device words): plans known at entry (kLayer) and staged misses: the
    // task's entry tk.pe; misses that wait for the admission's slots: the plan
    // entry of its slot.  Every unit of a copied expert waits for its pieces.
    const uint8_t* blob = t < T && !failed ? tk.blob[t] : nullptr;
    int wpe = -1;  // the piece counter this unit waits on
    if (LAYER && t < T && tk.pe[t] != -1 && !failed) {
      if (ADMIT && !staged) {  // decided by CTA 0's admission
        if (!wait_seq(a, seq0 + 1, lane)) failed = true;
        const int s = failed ? -1 : a.slot_out[tk.route[t]];
        blob = s >= 0 ? slot_ptr(st, a.layer, s) : nullptr;  // not admitted: no work, no term
        if (s >= 0) {
          const int np = a.gplan0[0];
          for (int i = 0; i < np; ++i)
            if (a.gplan0[1 + 3 * i] == s) wpe = i;
        }
      } else {
        wpe = tk.pe[t];
      }
    }
    if (LAYER && wpe >= 0 && blob && !failed) {  // every piece of the expert copied
      if (!wait_count(a.gdone + wpe, ppe, a.status, lane)) failed = true;
      if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");  // copied bytes -> bulk reads
    }
    if (!csync_and(!failed)) failed = true;
    if (failed) blob = nullptr;

    // ---- phase A: this CTA's rows of the part, each row's chunks on one warp
    const int i0 = p * IP + (int)crank * IPC;
    const int nrw = blob && !a.tile && IPC > warp ? (IPC - 1 - warp) / kW + 1 : 0;
    const int nitA = nrw * KC;
    auto row_of = [&](int it) { return i0 + warp + kW * (it / KC); };
    float2 gsl[2] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
    auto issue_a = [&](int it) {  // lane 0
      const int sl = it & 1;
      mbar_expect_tx(&bar_a[warp][sl], ItemA<FMT>::BYTES);
      ItemA<FMT>::issue(slots + sl * kSlotBytes, blob, o, H, row_of(it), it % KC, &bar_a[warp][sl],
                        pol);
      gsl[sl] = ItemA<FMT>::glob(blob, o);
    };
    if (a.tile) {
      if (lane == 0 && warp < kTileGroups && blob && u != early_u) {
        fence_proxy_async();  // the last unit's tile reads before the new bulk writes
        issue_tile(blob, i0, IPC, warp);
      }
    } else if (lane == 0) {
      if (u == early_u) {  // requested before x was staged
        gsl[0] = gsl[1] = ItemA<FMT>::glob(blob, o);
      } else {
        if (nitA > 0) issue_a(0);
        if (nitA > 1) issue_a(1);
      }
    }
    // phase-B rows of this CTA's slice, the part's columns: staged into shared
    // memory by this thread (cp.async) while phase A runs, or requested into L2
    const int HB = H / kCS;
    const int CBr = FP4 ? IP / 2 : IP * 2;                 // code bytes of a row's part
    const int SBr = (IP / 32) * scale_bytes_per32<FMT>();  // scale bytes of a row's part
    const bool pb_smem = FP4 && HB <= kT && CBr + SBr <= pb_room;
    const int nrow = (int)crank * HB + threadIdx.x;        // the thread's first row
    const uint8_t* rcode = nullptr;
    const uint8_t* rscale = nullptr;
    if (blob && nrow < ((int)crank + 1) * HB) {
      rcode = FP4 ? blob + o.code[2] + (size_t)nrow * (I / 2) + p * IP / 2
                  : blob + o.mat[2] + ((size_t)nrow * I + (size_t)p * IP) * 2;
      if (FP4) {
        const size_t sr = FMT == MOE_W_MXFP4 ? (size_t)nrow * (I / 32) + p * IP / 32
                        : FMT == MOE_W_Q4_0 ? ((size_t)nrow * (I / 32) + p * IP / 32) * 2
                                            : (size_t)nrow * (I / 16) + p * IP / 16;
        rscale = blob + o.scale[2] + sr;
      }
      if (pb_smem) {
        for (int c = 0; c < CBr / 16; ++c)
          cp16_async(pbuf + ((size_t)c * kT + threadIdx.x) * 16, rcode + 16 * c);
        uint8_t* sdst = pbuf + (size_t)(CBr / 16) * kT * 16 + (size_t)threadIdx.x * SBr;
        if (SBr == 16) cp16_async(sdst, rscale);
        else if (SBr == 8) cp8_async(sdst, rscale);
        else if (SBr == 4) cp4_async(sdst, rscale);
        asm volatile("cp.async.commit_group;" ::: "memory");
      } else {
        for (int n = nrow; n < ((int)crank + 1) * HB; n += kT) {
          const uint8_t* rp = FP4 ? blob + o.code[2] + (size_t)n * (I / 2) + p * IP / 2
                                  : blob + o.mat[2] + ((size_t)n * I + (size_t)p * IP) * 2;
          for (int off = 0; off < CBr; off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + off));
        }
      }
    }
    const int tb = t < T ? tk.b[t] : 0;
    const float xi = xinv[tb];
    const uint4* xrow = reinterpret_cast<const uint4*>(xs) + (size_t)tb * (H / 8);
    auto wait_slot = [&](int it) -> bool {
      const int sl = it & 1;
      const bool all = __all_sync(0xffffffffu, mbar_wait(&bar_a[warp][sl], ph[sl] & 1u));
      ++ph[sl];
      if (!all && lane == 0) flag_timeout(a.status);
      return all;
    };
    auto put_h = [&](int it, float gsum, float usum, float2 gs) {  // lane 0: h of a row, to every CTA
      const float gg = gsum * xi * gs.x, uu = usum * xi * gs.y;
      const float h = gg / (1.f + expf(-gg)) * uu;
      const float* dst = hb + (row_of(it) - p * IP);
#pragma unroll
      for (int q = 0; q < kCS; ++q) st_cluster_f32(dst, (uint32_t)q, h);
    };
    if (a.tile && blob) {  // tile mode: warp w's rows [w rpw, (w + 1) rpw), two at a time
      const int rpw = IPC / kW, GR = IPC / kTileGroups;
      const int g = warp * rpw / GR;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_t[g], tph & 1u));
      if (!ok) {
        failed = true;
        if (lane == 0) flag_timeout(a.status);
      }
      const float2 gsc = ItemA<FMT>::glob(blob, o);
      const uint8_t* gcb = ring;
      const uint8_t* ucb = ring + (size_t)IPC * RB;
      const uint8_t* gsb = ring + (size_t)2 * IPC * RB;
      const uint8_t* usb = gsb + (size_t)IPC * SB;
      for (int r = warp * rpw; ok && r < (warp + 1) * rpw; r += 2) {
        float ga = 0.f, ua = 0.f, gb = 0.f, ub = 0.f;
        ItemA<FMT>::dot4(gcb + (size_t)r * RB, ucb + (size_t)r * RB, gsb + (size_t)r * SB,
                         usb + (size_t)r * SB, xrow, 0, lane, ga, ua);
        ItemA<FMT>::dot4(gcb + (size_t)(r + 1) * RB, ucb + (size_t)(r + 1) * RB,
                         gsb + (size_t)(r + 1) * SB, usb + (size_t)(r + 1) * SB, xrow, 0, lane, gb, ub);
        const float pp[4] = {ga, ua, gb, ub};
        const float v = reduce4(pp, lane);
        const float va = __shfl_sync(0xffffffffu, v, 8), vb = __shfl_sync(0xffffffffu, v, 16),
                    vc = __shfl_sync(0xffffffffu, v, 24);
        if (lane == 0) {
          const float* base = hb + (i0 - p * IP);
          const float gg0 = v * xi * gsc.x, uu0 = va * xi * gsc.y;
          const float gg1 = vb * xi * gsc.x, uu1 = vc * xi * gsc.y;
          const float h0 = gg0 / (1.f + expf(-gg0)) * uu0, h1 = gg1 / (1.f + expf(-gg1)) * uu1;
#pragma unroll
          for (int q = 0; q < kCS; ++q) {
            st_cluster_f32(base + r, (uint32_t)q, h0);
            st_cluster_f32(base + r + 1, (uint32_t)q, h1);
          }
        }
      }
    } else {
      float ga = 0.f, ua = 0.f, gb = 0.f, ub = 0.f;
      for (int it = 0; it < nitA; it += 2) {
        const bool two = it + 1 < nitA;
        if (!wait_slot(it)) {
          failed = true;
          if (two) (void)wait_slot(it + 1);  // keep both slots' phases counted
          break;
        }
        ItemA<FMT>::dot(slots, xrow, it % KC, lane, ga, ua);
        const float2 s0 = gsl[0];
        __syncwarp();  // slot 0 read by every lane
        if (it + 2 < nitA && lane == 0) {
          fence_proxy_async();
          issue_a(it + 2);
        }
        float2 s1 = make_float2(1.f, 1.f);
        if (two) {
          if (!wait_slot(it + 1)) {
            failed = true;
            if (it + 2 < nitA) (void)wait_slot(it + 2);
            break;
          }
          ItemA<FMT>::dot(slots + kSlotBytes, xrow, (it + 1) % KC, lane, gb, ub);
          s1 = gsl[1];
          __syncwarp();
          if (it + 3 < nitA && lane == 0) {
            fence_proxy_async();
            issue_a(it + 3);
          }
        }
        if (KC == 1) {  // rows it and it + 1 complete
          const float pp[4] = {ga, ua, gb, ub};
          const float v = reduce4(pp, lane);
          const float va = __shfl_sync(0xffffffffu, v, 8), vb = __shfl_sync(0xffffffffu, v, 16),
                      vc = __shfl_sync(0xffffffffu, v, 24);
          if (lane == 0) {
            put_h(it, v, va, s0);
            if (two) put_h(it + 1, vb, vc, s1);
          }
          ga = ua = gb = ub = 0.f;
        } else if ((it + 1) % KC == KC - 1) {  // the row of items it, it + 1 completes
          const float2 gu = reduce2(ga + gb, ua + ub, lane);
          if (lane == 0) put_h(it + 1, gu.x, gu.y, s1);
          ga = ua = gb = ub = 0.f;
        }
      }
    }
    if (a.tile && blob) ++tph;  // (uniform: blob is the same in every thread)
    // the unit's weight in the layer sum: routing weight (or the shared
    // expert's sigmoid gate) x the down global scale; 0 when the unit adds
    // nothing (no work, or a staged miss the admission did not take)
    if (warp == kW - 1) {
      float wsc = 0.f;
      if (blob) {
        const bool shared_task = SHARED || tk.route[t] >= a.R;
        float cw = 1.f;
        if (shared_task) {  // sigmoid(x_b . w_g) in fp32
          float z = 0.f;
          for (int i0g = lane * 8; i0g < H; i0g += 256) {
            const uint4 gv = *reinterpret_cast<const uint4*>(a.gate_w + i0g);
            const uint4 xv = *reinterpret_cast<const uint4*>(a.x + (size_t)tb * H + i0g);
            z = dot8_bf16_bf(gv, xv, z);
          }
          z = wsum(z);
          cw = 1.f / (1.f + expf(-z));
        } else {
          cw = a.w[tk.route[t]];
        }
        const float c2 = FMT == MOE_W_NVFP4 ? __ldcg(reinterpret_cast<const float*>(blob + o.glob) + 2)
                                            : 1.f;
        wsc = cw * c2;
        if (ADMIT && staged && tk.pend[t]) {  // computed from staging: was it admitted?
          if (!wait_seq(a, seq0 + 1, lane)) failed = true;
          if (failed || a.slot_out[tk.route[t]] < 0) wsc = 0.f;
        }
      }
      if (lane == 0) s_wsc = wsc;
    }
    // h of the whole part in every CTA of the cluster (a failed CTA still takes part)
    cluster_sync();
    if (!csync_and(!failed)) failed = true;

    // ---- phase B: this CTA's output rows, the part's columns, weighted into
    // the layer's fixed-point sums (integer adds: the same bits in any order)
    const float wsc = s_wsc;
    if (blob && !failed && wsc != 0.f) {
      for (int n = nrow; n < ((int)crank + 1) * HB; n += kT) {
        float y;
        if (pb_smem) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          const uint8_t* ssrc = pbuf + (size_t)(CBr / 16) * kT * 16 + (size_t)threadIdx.x * SBr;
          y = rowb_dot<FMT>(
              IP, hb,
              [&](int c, uint4* w) {
                w[0] = *reinterpret_cast<const uint4*>(pbuf + ((size_t)c * kT + threadIdx.x) * 16);
              },
              [&](int c) { return scale_at<FMT>(ssrc, c); });
        } else {
          const uint8_t* rp = FP4 ? blob + o.code[2] + (size_t)n * (I / 2) + p * IP / 2
                                  : blob + o.mat[2] + ((size_t)n * I + (size_t)p * IP) * 2;
          const size_t sr = FMT == MOE_W_MXFP4 ? (size_t)n * (I / 32) + p * IP / 32
                            : FMT == MOE_W_Q4_0 ? ((size_t)n * (I / 32) + p * IP / 32) * 2
                                                : (size_t)n * (I / 16) + p * IP / 16;
          const uint8_t* sp = FP4 ? blob + o.scale[2] + sr : nullptr;
          y = rowb_dot<FMT>(
              IP, hb,
              [&](int c, uint4* w) {
                const uint4* r = reinterpret_cast<const uint4*>(rp);
                if (FMT == MOE_W_BF16) {
                  w[0] = r[4 * c], w[1] = r[4 * c + 1], w[2] = r[4 * c + 2], w[3] = r[4 * c + 3];
                } else {
                  w[0] = r[c];
                }
              },
              [&](int c) { return FP4 ? scale_at<FMT>(sp, c) : 0u; });
        }
        red_add_u64(a.acc + (size_t)tb * H + n, to_fixed(y * wsc));
      }
    } else if (pb_smem && blob) {
      asm volatile("cp.async.wait_all;" ::: "memory");  // no copy left in flight
    }
    // ---- the unit is done for this slice; the last one converts the sums
    __threadfence();  // this thread's adds, before the count that publishes them
    csync();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned old = atomicAdd(&a.slice_cnt[crank], 1u);
      s_last = old == (unsigned)(a.n_units - 1);
      if (s_last) a.slice_cnt[crank] = 0;  // every arrival of this launch is in
    }
    csync();
    if (s_last) {
      __threadfence();
      const int n0 = (int)crank * HB;
      const bool convert = !SHARED || a.acc_out;
      // every unit's adds are in (each fenced them before its count): read
      // the sums, zero them for the next launch, convert
      for (int i0c = threadIdx.x; convert && i0c < n_rows * HB; i0c += 4 * kT) {
        unsigned long long q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int idx = i0c + j * kT;
          if (idx < n_rows * HB) {
            const int b = idx / HB;
            q[j] = __ldcg(a.acc + (size_t)b * H + n0 + (idx - b * HB));
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int idx = i0c + j * kT;
          if (idx >= n_rows * HB) continue;
          const int b = idx / HB;
          const size_t ru = (size_t)b * H + n0 + (idx - b * HB);
          a.acc[ru] = 0ull;
          const float v = (float)((double)(long long)q[j] * (1.0 / kFix));
          if (SHARED)
            a.ys[ru] = v;
          else
            a.out[ru] = __float2bfloat16_rn(a.ys ? v + __ldcg(a.ys + ru) : v);
        }
      }
      // slice 0's last unit: every unit has passed its copy waits and read the
      // map at entry -- reset the piece counters, make the admitted misses'
      // map entries valid for later launches
      if (LAYER && crank == 0) {
        const int n_done = staged ? npx : (ADMIT ? (npend > 0 ? a.gplan0[0] : 0) : n_pl0);
        for (int i = threadIdx.x; i < n_done; i += kT) a.gdone[i] = 0;
        if (ADMIT && npend > 0) {
          if (warp == 0) (void)wait_seq(a, seq0 + 1, lane);
          csync();
          const int np0 = a.gplan0[0];
          for (int i = threadIdx.x; i < np0; i += kT) {
            const int s = a.gplan0[1 + 3 * i], L = a.gplan0[2 + 3 * i], e = a.gplan0[3 + 3 * i];
            if ((unsigned)s < (unsigned)st.S && L == a.layer && (unsigned)e < (unsigned)st.E)
              st.map[a.layer * st.E + e] = s;
          }
        }
      }
      csync();
    }
  }
}

int g_num_sms = 0;
int g_clusters = 0;  // clusters of kCS CTAs resident at once (one CTA per SM)
constexpr size_t kBudget = 200 * 1024;
// every CTA asks for more than half an SM's shared memory, so that the
// clusters spread one CTA per SM (a CTA's bandwidth is its SM's)
constexpr size_t kOneCtaPerSm = 120 * 1024;

size_t round128(size_t v) { return (v + 127) / 128 * 128; }

// tasks per batch row and in all, for a launch of `mode`
int tasks_per_row(int mode, int k, bool shared) {
  return (mode == kLayer || mode == kLayerAdmit) ? k + (shared ? 1 : 0) : k;
}

struct Plan {
  int Pr, Ps, n_units, first_cluster, one_round, grid;
  int pb_room;  // bytes per thread for a staged phase-B row part (0: rows read from L2)
  int tile, area;
  size_t smem;
  bool ok;
};

// Shared memory of CTA 0 in kLayerAdmit: its block state, then the admission's
// [E] x 3 counters (and the pool's keys when cached), or the prefetch's [E] x 2.
size_t admit_cta_smem(int E, int S, bool cached) {
  const size_t adm = 3ull * E * sizeof(int) + (cached ? (size_t)S * 12 : 0);
  return round128(sizeof(admission::AdmitShared<kT>)) + std::max<size_t>(adm, 2ull * E * sizeof(int));
}

bool shape_ok(int wfmt, int H, int I, int n_rows, int T) {
  const int CW = wfmt == MOE_W_BF16 ? 512 : 2048;
  const int KC = H / CW;
  return H % CW == 0 && (KC == 1 || KC % 2 == 0) && I % 128 == 0 && I <= 4096 &&
         H % kCS == 0 && n_rows >= 1 && n_rows <= kMaxRows && T <= kMaxTasks &&
         n_rows * H <= kXW * 8 * kT;
}

// The parts of a layer's tasks, from its shape alone (n_rows x k routes, a
// shared expert or not) so that every launch mode -- the one-launch layer,
// the routed and the shared launches of the four-launch path, the
// allocation-free call -- cuts a task alike and sums alike: powers of two,
// each CTA of a unit keeping at least 32 rows of I, as many as the one-launch
// layer's clusters allow (the resident clusters but the admission's), the
// shared expert halving first.
void parts_of_layer(int I, int n_rows, int k, bool shared, int clusters, int* Pr, int* Ps) {
  const int ncc = std::max(1, clusters - 1), pmax = std::max(1, I / (kCS * 32));
  const long R = (long)n_rows * k, S = shared ? n_rows : 0;
  for (int pr = pmax; pr >= 1; pr /= 2) {
    for (int ps = pr; ps >= std::max(1, pr / 2); ps /= 2) {
      if (R * pr + S * ps <= ncc || (pr == 1 && ps == 1)) {
        *Pr = pr;
        *Ps = ps;
        return;
      }
      if (ps == 1) break;
    }
  }
  *Pr = *Ps = 1;
}

// The launch of `mode` for a layer of n_rows x k routes (shared: the layer
// has a shared expert): its units, grid and shared memory.
Plan plan_of(int mode, int wfmt, int H, int I, int n_rows, int k, bool shared, int clusters) {
  Plan p{};
  const int T = mode == kShared ? n_rows : n_rows * tasks_per_row(mode, k, shared);
  p.ok = shape_ok(wfmt, H, I, n_rows, T) && clusters >= (mode == kLayerAdmit ? 2 : 1);
  if (!p.ok) return p;
  parts_of_layer(I, n_rows, k, shared, clusters, &p.Pr, &p.Ps);
  p.first_cluster = mode == kLayerAdmit ? 1 : 0;
  const int ncc = clusters - p.first_cluster;
  if (mode == kShared)
    p.n_units = n_rows * p.Ps;
  else
    p.n_units = n_rows * k * p.Pr + ((mode == kLayer || mode == kLayerAdmit) && shared ? n_rows * p.Ps : 0);
  p.one_round = p.n_units <= ncc;
  p.grid = (std::min(p.n_units, ncc) + p.first_cluster) * kCS;
  const int ipmax = I / std::min(p.Pr, p.Ps);
  // phase A: tiles when a row is one chunk and the largest unit's rows fit
  const int CW = wfmt == MOE_W_BF16 ? 512 : 2048;
  const size_t tile = (size_t)(ipmax / kCS) * (2 * row_code_bytes(wfmt, H) + 2 * row_scale_bytes(wfmt, H));
  p.tile = H == CW && (ipmax / kCS) % 32 == 0 && tile <= 160 * 1024;
  p.area = (int)round128(p.tile ? tile : (size_t)kW * 2 * kSlotBytes);
  const size_t fixed = round128((size_t)n_rows * H * 2) + (size_t)p.area + 2 * (size_t)ipmax * 4;
  // 4-bit experts with one phase-B row per thread stage the row's part in
  // shared memory: codes IP / 2 bytes, scales up to IP / 16 -- room for the
  // longest part if it fits, else for the routed tasks' parts (the others
  // read their rows from L2)
  p.pb_room = 0;
  if (wfmt != MOE_W_BF16 && H / kCS <= kT) {
    for (const int ip : {ipmax, I / p.Pr}) {
      const int need = ip / 2 + ip / 16;
      if (fixed + (size_t)need * kT <= kBudget) {
        p.pb_room = need;
        break;
      }
    }
  }
  p.smem = std::max(kOneCtaPerSm, fixed + (size_t)p.pb_room * kT);
  p.ok = p.smem <= kBudget;
  return p;
}

// threads per CTA of a launch of `mode`: the layer launches add the copy warps
constexpr int block_threads(int mode) { return mode == kLayer || mode == kLayerAdmit ? 32 * kNW : kT; }

template <typename K>
cudaError_t launch_clusters(K kernel, int mode, const Plan& p, size_t smem, bool coop,
                            cudaStream_t s, const DevState& st, const FusedArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(block_threads(mode));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the grid never exceeds the resident clusters; a launch whose CTAs wait on
  // other clusters (the admission, piece counts) asks for co-residency too
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = coop ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, st, a);
}

template <int FMT>
cudaError_t launch_mode(int mode, const Plan& p, size_t smem, cudaStream_t s, const DevState& st,
                        const FusedArgs& a) {
  switch (mode) {
    case kLayerAdmit:
      return launch_clusters(ffn_cluster_kernel<FMT, kLayerAdmit>, mode, p, smem, true, s, st, a);
    case kLayer:
      return launch_clusters(ffn_cluster_kernel<FMT, kLayer>, mode, p, smem, true, s, st, a);
    case kShared:
      return launch_clusters(ffn_cluster_kernel<FMT, kShared>, mode, p, smem, false, s, st, a);
    default:
      return launch_clusters(ffn_cluster_kernel<FMT, kRouted>, mode, p, smem, false, s, st, a);
  }
}
cudaError_t launch_format(int wfmt, int mode, const Plan& p, size_t smem, cudaStream_t s,
                          const DevState& st, const FusedArgs& a) {
  if (wfmt == MOE_W_NVFP4) return launch_mode<MOE_W_NVFP4>(mode, p, smem, s, st, a);
  if (wfmt == MOE_W_MXFP4) return launch_mode<MOE_W_MXFP4>(mode, p, smem, s, st, a);
  if (wfmt == MOE_W_Q4_0) return launch_mode<MOE_W_Q4_0>(mode, p, smem, s, st, a);
  return launch_mode<MOE_W_BF16>(mode, p, smem, s, st, a);
}

// layer_k, layer_shared: the top-k of the layer these tasks belong to and
// whether it has a shared expert (the routed and shared launches of the
// four-launch path split their tasks as the one-launch layer would)
cudaError_t launch_fused(const DevState& st, int wfmt, int mode, const FusedArgs& a0,
                         int layer_k, bool layer_shared, cudaStream_t s) {
  FusedArgs a = a0;
  const Plan p = plan_of(mode, wfmt, a.H, a.I, a.n_rows, layer_k, layer_shared, g_clusters);
  if (!p.ok) return cudaErrorInvalidValue;
  a.Pr = p.Pr;
  a.Ps = p.Ps;
  a.pb_room = p.pb_room;
  a.tile = p.tile;
  a.area = p.area;
  a.n_units = p.n_units;
  a.first_cluster = p.first_cluster;
  a.one_round = p.one_round;
  size_t smem = p.smem;
  if (mode == kLayerAdmit) smem = std::max(smem, admit_cta_smem(st.E, st.S, a.adm_cached != 0));
  if (smem > kBudget) return cudaErrorInvalidValue;
  return launch_format(wfmt, mode, p, smem, s, st, a);
}

template <int FMT>
cudaError_t set_limits() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto kern) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBudget);
  };
  set(ffn_cluster_kernel<FMT, kShared>);
  set(ffn_cluster_kernel<FMT, kRouted>);
  set(ffn_cluster_kernel<FMT, kLayer>);
  set(ffn_cluster_kernel<FMT, kLayerAdmit>);
  return e;
}

// devices whose limits and cluster count are set (the kernels' attributes are per device)
std::mutex g_init_mu;
bool g_init_done[64] = {};

}  // namespace

bool ffn_stream_supported(int wfmt, int H, int I, int n_rows, int n_tasks) {
  if (g_clusters <= 0 || n_tasks > kMaxRoutes || n_rows < 1) return false;
  const int k = (n_tasks + n_rows - 1) / n_rows;
  return plan_of(kRouted, wfmt, H, I, n_rows, k, false, g_clusters).ok;
}

// Per device: the kernels' shared-memory limits and the number of clusters of
// kCS CTAs that are resident at once with one CTA per SM.
cudaError_t ffn_stream_init() {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_init_mu);
  if (dev >= 0 && dev < 64 && g_init_done[dev]) return cudaSuccess;
  e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = set_limits<MOE_W_BF16>();
  if (e == cudaSuccess) e = set_limits<MOE_W_NVFP4>();
  if (e == cudaSuccess) e = set_limits<MOE_W_MXFP4>();
  if (e == cudaSuccess) e = set_limits<MOE_W_Q4_0>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kCS * std::max(1, g_num_sms / kCS));
  cfg.blockDim = dim3(block_threads(kLayerAdmit));
  cfg.dynamicSmemBytes = kOneCtaPerSm;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, ffn_cluster_kernel<MOE_W_NVFP4, kLayerAdmit>, &cfg);
  if (e != cudaSuccess) return e;
  g_clusters = n;
  if (dev >= 0 && dev < 64) g_init_done[dev] = true;
  return cudaSuccess;
}

int ffn_stream_max_parts(int I) { return std::max(1, I / (kCS * 32)); }

// The split a launch of this shape takes: {parts P, units, clusters in the
// grid (the admission's included), one round (1/0), resident clusters}.
bool ffn_stream_split(int mode_layer, int admit, int wfmt, int H, int I, int n_rows, int k,
                      bool shared, int out[6]) {
  const int mode = admit ? kLayerAdmit : (mode_layer ? kLayer : kRouted);
  const Plan p = plan_of(mode, wfmt, H, I, n_rows, k, shared, g_clusters);
  out[0] = p.Pr, out[1] = p.Ps, out[2] = p.n_units, out[3] = p.grid / kCS, out[4] = p.one_round,
  out[5] = g_clusters;
  return p.ok;
}

cudaError_t launch_shared_stream(const DevState& st, int wfmt, int H, int Is, const void* x,
                                 int n_rows, int k_layer, bool to_ys, const uint8_t* blob,
                                 const void* gate_w, FfnScratch sc, unsigned long long* status,
                                 cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = Is;
  a.layer = 0;
  a.k = 1;
  a.R = n_rows;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.fixed_blob = blob;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.ys = sc.ys;
  a.acc_out = to_ys ? 1 : 0;
  a.status = status;
  a.acc = sc.acc;
  a.slice_cnt = sc.slice_cnt;
  return launch_fused(st, wfmt, kShared, a, k_layer, true, s);
}

cudaError_t launch_routed_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                 const void* x, const int32_t* slot_ids, const float* w,
                                 int n_rows, int k, bool layer_shared, const float* shared_y,
                                 void* out, FfnScratch sc, unsigned long long* status,
                                 cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = I;
  a.layer = layer;
  a.k = k;
  a.R = n_rows * k;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = slot_ids;
  a.w = w;
  a.ys = const_cast<float*>(shared_y);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.acc = sc.acc;
  a.slice_cnt = sc.slice_cnt;
  return launch_fused(st, wfmt, kRouted, a, k, layer_shared, s);
}

bool layer_stream_supported(int wfmt, int H, int I, int n_rows, int k, bool shared) {
  if (g_clusters <= 0 || n_rows < 1 || n_rows > kMaxRows || n_rows * k > kMaxRoutes) return false;
  return plan_of(kLayer, wfmt, H, I, n_rows, k, shared, g_clusters).ok;
}

bool layer_admit_supported(const DevState& st, int wfmt, int H, int I, int n_rows, int k,
                           bool shared) {
  if (st.E > kPbWords * 32 || !layer_stream_supported(wfmt, H, I, n_rows, k, shared)) return false;
  const Plan p = plan_of(kLayerAdmit, wfmt, H, I, n_rows, k, shared, g_clusters);
  return p.ok && std::max(p.smem, admit_cta_smem(st.E, st.S, false)) <= kBudget;
}

cudaError_t launch_layer_admit(const DevState& st, int wfmt, int H, int I, int layer,
                               const void* x, const int32_t* ids, int32_t* slot_out,
                               const float* w, int n_rows, int k, int cap, const int32_t* pred,
                               int n_pred, const uint8_t* shared_blob, const void* gate_w,
                               int32_t* plan1, void* out, FfnScratch sc,
                               unsigned long long* status, cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = I;
  a.layer = layer;
  a.k = k;
  a.R = n_rows * k;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = slot_out;
  a.w = w;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.acc = sc.acc;
  a.slice_cnt = sc.slice_cnt;
  a.shared_blob = shared_blob;
  a.gplan0 = st.plan_demand;
  a.gplan1 = plan1;
  a.gdone = sc.gdone;
  a.ids = ids;
  a.slot_out = slot_out;
  a.cap = cap;
  a.pred = pred;
  a.n_pred = pred ? n_pred : 0;
  a.epoch = sc.epoch;
  a.stage = sc.stage_n > 0 ? sc.stage : nullptr;
  a.stage_n = sc.stage_n;
  a.pseq = sc.pseq;
  a.sslot = sc.sslot;
  const Plan p = plan_of(kLayerAdmit, wfmt, H, I, n_rows, k, shared_blob != nullptr, g_clusters);
  a.adm_cached = admit_cached(st.E, st.S) &&
                 std::max(p.smem, admit_cta_smem(st.E, st.S, true)) <= kBudget;
  return launch_fused(st, wfmt, kLayerAdmit, a, k, shared_blob != nullptr, s);
}

cudaError_t launch_layer_stream(const DevState& st, int wfmt, int H, int I, int layer,
                                const void* x, const int32_t* slot_ids, const float* w,
                                int n_rows, int k, const uint8_t* shared_blob,
                                const void* gate_w, const int32_t* plan0, const int32_t* plan1,
                                void* out, FfnScratch sc, unsigned long long* status,
                                cudaStream_t s) {
  FusedArgs a{};
  a.H = H;
  a.I = I;
  a.layer = layer;
  a.k = k;
  a.R = n_rows * k;
  a.n_rows = n_rows;
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = slot_ids;
  a.w = w;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.acc = sc.acc;
  a.slice_cnt = sc.slice_cnt;
  a.shared_blob = shared_blob;
  a.gplan0 = plan0;
  a.gplan1 = plan1;
  a.gdone = sc.gdone;
  return launch_fused(st, wfmt, kLayer, a, k, shared_blob != nullptr, s);
}
// ---------------------------------------------------------------- allocation-free variant
// moe_routed_experts_noalloc runs ffn_cluster_kernel with its scratch in this
// file-scope array instead of memory a cache allocated: bytes [0, 256) hold
// the output-slice counters, bytes [256, end) the fixed-point layer sums
// [n_rows][H] (int64).
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
    if (e == cudaSuccess) e = ffn_stream_init();
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

// the scratch bytes a call of this shape needs on this device (0: the
// streaming kernel does not take the shape)
size_t noalloc_scratch_bytes(int wfmt, int H, int I, int n_rows, int k) {
  const Plan p = plan_of(kRouted, wfmt, H, I, n_rows, k, false, g_clusters);
  if (!p.ok || n_rows * k > kMaxRoutes) return 0;
  return 256 + (size_t)n_rows * H * sizeof(unsigned long long);
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
  sc.slice_cnt = static_cast<unsigned*>(scratch);
  sc.acc = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(scratch) + 256);
  // the last unit of a slice zeroes its counter and its sums; a launch that
  // gave up after a timeout can leave them elsewhere, so start from zero
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256 + (size_t)n_rows * H * 8, s);
  if (e != cudaSuccess) return e;
  return launch_routed_stream(st, wfmt, H, I, 0, x, slot_ids, w, n_rows, k, false, nullptr, out,
                              sc, status, s);
}

}  // namespace moe
