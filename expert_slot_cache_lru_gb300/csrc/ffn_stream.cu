// ffn_stream.cu -- expert FFNs for decode-sized steps: one cooperative launch
// per group of experts.
//
// What is computed is the same as gemv.cu (FreeToken issue #753 "[Perf]
// Offloaded decode: overlap the expert-miss gather with the same layer's
// shared expert ...", Problem and What we changed: routed experts over the
// slots, a sigmoid-gated shared expert, routed + shared); this file is the
// fast path when every (route, row) of the step fits a small task list.
//
// A decode step moves ~14 MB of weights per layer, which the HBM delivers in
// ~2 us after ~1 us of latency, and the arithmetic per weight is a handful of
// instructions, so the kernel is built to have every byte requested within a
// microsecond of entry and to spend few instructions per weight:
//   * one CTA per SM (cooperative launch), 16 warps;
//   * phase A (gate/up): the rows of the flattened (task, i) list are dealt
//     round-robin over the grid's warps, so every expert (the shared one
//     included) is spread over the whole GPU.  Each warp owns two shared-memory
//     slots; lane 0 fills a slot with the bulk copies (cp.async.bulk) of one
//     item -- a chunk of a gate row and of an up row with their scales --
//     completing on the slot's mbarrier, and requests the next item as soon as
//     the slot is read.  The warp reduces each row itself;
//   * at entry one warp also requests the down-projection rows this CTA needs
//     in phase B, by bulk copies into a staging area on one mbarrier, so they
//     land during phase A;
//   * a grid-wide barrier (h of every task is needed by every CTA);
//   * phase B (down + combine): each warp takes runs of (task, output row)
//     items, reduces four at a time with one butterfly, and the CTA combines
//     its output rows over the tasks in route order.
// The one-launch layer (kLayerAdmit) runs the admission on CTA 0 while the
// other CTAs compute; the step's missed experts are copied from pinned host
// memory by every warp, 4 KiB at a time, as soon as the lookups are done.
//
// Every wait that depends on other CTAs (the grid barrier, the admission's
// publication, a copy's piece count) is bounded (%globaltimer): on a timeout
// the kernel sets MOE_STATUS_TIMEOUT in the cache's device status word and
// skips the remaining work.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "admit_body.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int kW = 16;             // warps per CTA
constexpr int kT = 32 * kW;        // threads per CTA
constexpr int kMaxRoutes = 64;     // routes per call on this path
constexpr int kMaxTasks = 80;      // routes plus one shared-expert task per row (fused layer)
constexpr int kMaxRows = 16;       // batch rows per call on this path
constexpr int kXW = 4;             // x words (8 elements each) loaded per thread
constexpr int kYsPre = 1;          // shared-expert outputs prefetched per thread
// Registers per thread: 512 x 104 leaves room on the SM for a gather CTA
// (256 threads x 32 registers), which runs beside this kernel on the side stream.
constexpr int kMaxReg = 104;
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
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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
  int ord[kMaxTasks];              // phase-A task order (fused layer: copied-in tasks last)
  unsigned char drop[kMaxTasks];   // admission inside: not admitted (fetch cap)
  unsigned char pend[kMaxTasks];   // admission inside: not resident when the launch began
  int slot[kMaxTasks];             // slot id, -1 for the shared expert
  const uint8_t* blob[kMaxTasks];
  float wt[kMaxTasks];             // routing weight x down global scale
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
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(slot + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(slot + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(slot + 1024 + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(slot + 1536 + lane * 16);
    const float2 sg0 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(slot + 2048 + lane * 2));
    const float2 sg1 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(slot + 2048 + 64 + lane * 2));
    const float2 su0 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(slot + 2176 + lane * 2));
    const float2 su1 = e4m3x2_f32(*reinterpret_cast<const uint16_t*>(slot + 2176 + 64 + lane * 2));
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
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& gs, float& us) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint4 xv = xr[xswz(c * 64 + 32 * s + lane)];
      gs = dot8_bf16_bf(*reinterpret_cast<const uint4*>(slot + 512 * s + lane * 16), xv, gs);
      us = dot8_bf16_bf(*reinterpret_cast<const uint4*>(slot + 1024 + 512 * s + lane * 16), xv, us);
    }
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
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(slot + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(slot + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(slot + 1024 + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(slot + 1536 + lane * 16);
    const float sg0 = e8m0_f32(slot[2048 + lane]), sg1 = e8m0_f32(slot[2048 + 32 + lane]);
    const float su0 = e8m0_f32(slot[2112 + lane]), su1 = e8m0_f32(slot[2112 + 32 + lane]);
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
  static __device__ __forceinline__ void dot(const uint8_t* slot, const uint4* xr, int c, int lane,
                                             float& g, float& u) {
    const uint4 g0 = *reinterpret_cast<const uint4*>(slot + lane * 16);
    const uint4 g1 = *reinterpret_cast<const uint4*>(slot + 512 + lane * 16);
    const uint4 u0 = *reinterpret_cast<const uint4*>(slot + 1024 + lane * 16);
    const uint4 u1 = *reinterpret_cast<const uint4*>(slot + 1536 + lane * 16);
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + 2048);
    const float sg0 = f16_f32(sc[lane]), sg1 = f16_f32(sc[32 + lane]);
    const float su0 = f16_f32(sc[64 + lane]), su1 = f16_f32(sc[96 + lane]);
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
};

constexpr int kSlotBytes = 2432;  // >= ItemA<*>::BYTES, a multiple of 128

// ------------------------------------------------------------ phase B items
// One down row of one task: I = 512 m elements.
//   NVFP4: lane L holds elements [16mL, 16mL + 16m): 8m code bytes, m scales.
//   bf16:  lane L holds elements 256s + 8L + [0, 8), s = 0..2m-1.
// h (fp32) for the same elements sits in registers, 16m values per lane.
template <int FMT>
struct ItemB {
  uint4 w[2];   // NVFP4: w[0] = codes (8m bytes), w[1].x = scales; bf16: 2m of these
  uint4 w2[2];  // bf16, m = 2 only
};

// loads one item's lane data from `row` (shared or global, generic address)
template <int FMT>
__device__ __forceinline__ void itemb_load(ItemB<FMT>& it, const uint8_t* codes,
                                           const uint8_t* scales, int m, int lane) {
  if (FMT == MOE_W_NVFP4) {
    if (m == 1) {
      const uint2 cw = *reinterpret_cast<const uint2*>(codes + lane * 8);
      it.w[0] = make_uint4(cw.x, cw.y, 0u, 0u);
      it.w[1].x = scales[lane];
    } else {
      it.w[0] = *reinterpret_cast<const uint4*>(codes + lane * 16);
      it.w[1].x = *reinterpret_cast<const uint16_t*>(scales + lane * 2);
    }
  } else if (FMT == MOE_W_Q4_0) {  // the lane's 16 or 32 elements: one fp16 32-block scale
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(scales);
    if (m == 1) {
      const uint2 cw = *reinterpret_cast<const uint2*>(codes + lane * 8);
      it.w[0] = make_uint4(cw.x, cw.y, 0u, 0u);
      it.w[1].x = sc[lane >> 1];
    } else {
      it.w[0] = *reinterpret_cast<const uint4*>(codes + lane * 16);
      it.w[1].x = sc[lane];
    }
  } else if (FMT == MOE_W_MXFP4) {  // the lane's 16 (m = 1) or 32 elements: one 32-block scale
    if (m == 1) {
      const uint2 cw = *reinterpret_cast<const uint2*>(codes + lane * 8);
      it.w[0] = make_uint4(cw.x, cw.y, 0u, 0u);
      it.w[1].x = scales[lane >> 1];
    } else {
      it.w[0] = *reinterpret_cast<const uint4*>(codes + lane * 16);
      it.w[1].x = scales[lane];
    }
  } else {
    it.w[0] = *reinterpret_cast<const uint4*>(codes + lane * 16);
    it.w[1] = *reinterpret_cast<const uint4*>(codes + 512 + lane * 16);
    if (m == 2) {
      it.w2[0] = *reinterpret_cast<const uint4*>(codes + 1024 + lane * 16);
      it.w2[1] = *reinterpret_cast<const uint4*>(codes + 1536 + lane * 16);
    }
  }
}
template <int FMT>
__device__ __forceinline__ float itemb_dot(const ItemB<FMT>& it, const float* hv, int m) {
  if (FMT == MOE_W_NVFP4) {
    const float2 sc = e4m3x2_f32(it.w[1].x & 0xffffu);
    float p = (dot8_fp4_f(it.w[0].x, hv) + dot8_fp4_f(it.w[0].y, hv + 8)) * sc.x;
    if (m == 2) p = fmaf(dot8_fp4_f(it.w[0].z, hv + 16) + dot8_fp4_f(it.w[0].w, hv + 24), sc.y, p);
    return p;
  } else if (FMT == MOE_W_Q4_0) {
    float p = dot8_q4_f(it.w[0].x, hv) + dot8_q4_f(it.w[0].y, hv + 8);
    if (m == 2) p += dot8_q4_f(it.w[0].z, hv + 16) + dot8_q4_f(it.w[0].w, hv + 24);
    return p * f16_f32(it.w[1].x);
  } else if (FMT == MOE_W_MXFP4) {
    float p = dot8_fp4_f(it.w[0].x, hv) + dot8_fp4_f(it.w[0].y, hv + 8);
    if (m == 2) p += dot8_fp4_f(it.w[0].z, hv + 16) + dot8_fp4_f(it.w[0].w, hv + 24);
    return p * e8m0_f32(it.w[1].x & 0xffu);
  } else {
    float p = dot8_bf16_f(it.w[0], hv, 0.f);
    p = dot8_bf16_f(it.w[1], hv + 8, p);
    if (m == 2) {
      p = dot8_bf16_f(it.w2[0], hv + 16, p);
      p = dot8_bf16_f(it.w2[1], hv + 24, p);
    }
    return p;
  }
}

// ---------------------------------------------------------------- grid barrier
// One CTA per SM, launched cooperatively, so every CTA of the grid is resident.
// `ctr` only grows: each launch adds n (the CTAs taking part), and a CTA waits
// until the count reaches the next multiple of n.  Release/acquire at GPU
// scope orders the h written before the barrier with the reads after it: the
// block barrier orders every thread's writes before thread 0's release add,
// and release is cumulative, so no separate fence is needed.  Bounded spin.
__device__ bool grid_barrier(unsigned long long* ctr, unsigned long long* status, unsigned n) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long old;
    asm volatile("atom.add.release.gpu.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
    const unsigned long long target = (old / n + 1) * n;
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
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---------------------------------------------------------------- fused FFN
// One launch computes a group of expert FFNs for a decode-sized step:
//   phase A (gate/up): rows (task t, i) of the flattened list,
//       h[route_t][i] = silu(W_g x_b)[i] * (W_u x_b)[i];
//   grid barrier;
//   phase B (down + combine) over this CTA's output rows (b, n):
//       SHARED: ys[b][n] = sigmoid(x_b . w_g) * (W_d h_b)[n]
//       ROUTED: out[b][n] = bf16( sum_j w[b,j] (W_d[slot] h_bj)[n] + ys[b][n] ).
// Phase-B items are (task, output row) pairs, b-major then task then row; the
// first `qs` of them are staged in shared memory at entry (cp.async), the rest
// are read from global memory when they are reached.
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
  int qs;                      // phase-B items staged in shared memory
  int htasks;                  // tasks whose h fits the CTA's h buffer (>= its tasks)
  unsigned long long* status;
  unsigned long long* bar_ctr;
  // fused layer
  const uint8_t* shared_blob;  // shared expert (one extra task per row), null = none
  const int32_t* gplan0;       // demand plan: its experts are copied here and waited on
  const int32_t* gplan1;       // prefetch plan of the next layer (copied only), or null
  int* gdone;                  // [plan entries] pieces copied; zero at entry, reset here
  // fused layer with the admission inside the launch: CTA 0 admits (and
  // prefetch-admits), the other CTAs compute
  const int32_t* ids;          // the step's expert ids [R]
  int32_t* slot_out;           // [R] slot ids, written by the admission
  int cap;                     // fetch cap (< 0: none)
  const int32_t* pred;         // the next layer's predicted ids, or null
  int n_pred;
  int adm_cached;              // the admission keeps the pool in shared memory
  unsigned long long* epoch;   // grows by gridDim.x per launch: launch j = old / gridDim.x
  unsigned long long* pseq;    // 2j+1: slot ids and demand plan of launch j out; 2j+2: prefetch plan too
  unsigned long long* bar2;    // grid barrier of the computing CTAs
  // [R] launch j's slot of its misses' rank i (ascending id): (2j+1) << 32 | slot,
  // low word ~0u when not admitted; the tag makes an older launch's word stale
  unsigned long long* sslot;
  uint8_t* stage;              // stage_n slot-sized areas the step's misses are copied into
  int stage_n;                 // (0: misses wait for the admission and go to their slots)
};

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
  __syncthreads();
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
    __syncthreads();
  }
  if (threadIdx.x == 0) st_release_u64(a.pseq, 2 * j + 2);
}

template <int FMT, int MODE>
__global__ void __maxnreg__(kMaxReg) ffn_fused_kernel(DevState st, FusedArgs a) {
  constexpr bool SHARED = MODE == kShared, ADMIT = MODE == kLayerAdmit;
  constexpr bool LAYER = MODE == kLayer || ADMIT;
  constexpr bool FP4 = FMT != MOE_W_BF16;  // 4-bit codes (NVFP4, MXFP4, Q4_0): f16 x
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ unsigned long long s_j;  // admission inside: this launch's index
  if (ADMIT) {  // every CTA of launch j adds one to a.epoch: j = old / gridDim.x
    if (threadIdx.x == 32) s_j = atomicAdd(a.epoch, 1ull) / gridDim.x;
    if (blockIdx.x == 0) {
      __syncthreads();
      admit_cta(st, a, sm, s_j);
      return;
    }
  }
  // the computing CTAs: all of them, or all but CTA 0 when it admits
  const int GF = (int)gridDim.x - (ADMIT ? 1 : 0), cta = (int)blockIdx.x - (ADMIT ? 1 : 0);
  __shared__ Tasks tk;
  __shared__ int ts[kMaxRows + 1];         // tasks of batch row b: [ts[b], ts[b+1])
  __shared__ unsigned int xmax[kMaxRows];  // per row max |x| (float bits, only when > 2^14)
  __shared__ float xinv[kMaxRows];         // per row 1 / (power-of-two scale applied to x)
  __shared__ uint64_t bar_a[kW][2];        // per-warp phase-A slot barriers
  __shared__ uint64_t bar_b;               // the staged phase-B rows
  __shared__ int s_npend;                  // admission inside: tasks not resident at entry
  __shared__ int s_npx;                    // ... their distinct experts (staging entries)
  __shared__ int s_staged;                 // ... copied into the staging area (else: slots)
  __shared__ unsigned s_pbits[kPbWords];   // ... bitmap of those experts
  __shared__ int s_pexp[kMaxRoutes];       // ... in ascending id: staging entry -> expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, k = a.k, n_rows = a.n_rows;
  const int m = I / 512;                                   // 16-element groups per lane (B)
  const int CB = FP4 ? I / 2 : I * 2;                      // down row: code bytes
  const int SB = FMT == MOE_W_MXFP4 ? I / 32 : (FP4 ? I / 16 : 0);  // down row: scale bytes
  constexpr int CW = ItemA<FMT>::CW;
  const int KC = H / CW;                                   // phase-A chunks per row
  const BlobOff o(H, I, FMT);

  // this CTA's output rows (phase B): at most two batch rows (perB <= H)
  const int UB = n_rows * H;
  const int perB = (UB + GF - 1) / GF;
  const int ru0 = min(UB, perB * cta), ru1 = min(UB, ru0 + perB);

  // ---- entry: the slot ids (warp 0) and x (everyone) in flight at once
  const int nx8 = n_rows * H / 8;
  uint4 xw[kXW];
#pragma unroll
  for (int j = 0; j < kXW; ++j) {
    const int i = threadIdx.x + j * kT;
    if (i < nx8) xw[j] = reinterpret_cast<const uint4*>(a.x)[i];
  }
  float ysv[kYsPre];
#pragma unroll
  for (int j = 0; j < kYsPre; ++j) {
    const int ru = ru0 + threadIdx.x + j * kT;
    ysv[j] = (MODE == kRouted && a.ys && ru < ru1) ? a.ys[ru] : 0.f;
  }
  if (threadIdx.x < kMaxRows) xmax[threadIdx.x] = 0u;
  auto slot_blob = [&](int s) -> const uint8_t* {
    return st.slots + ((size_t)pool_of(st, a.layer) * st.S + s) * st.stride;
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
    if (v0) b0 = a.fixed_blob ? a.fixed_blob : (sl0 >= 0 ? slot_blob(sl0) : nullptr);
    if (v1) b1 = sl1 >= 0 ? slot_blob(sl1) : nullptr;
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
  __syncthreads();  // (1) task list, ts, xmax
  const int T = tk.n;
  // fused layer: the demand plan entry of each task whose expert is being
  // copied in by this launch (its rows wait for the copy)
  // (admission inside: the plans are not known yet, see ADMIT below)
  const int n_pl0 = LAYER && !ADMIT && a.gplan0 ? a.gplan0[0] : 0;
  const int n_pl1 = LAYER && !ADMIT && a.gplan1 ? a.gplan1[0] : 0;
  const unsigned long long seq0 = ADMIT ? 2 * s_j : 0;  // a.pseq before this launch's admission
  const int npend = ADMIT ? s_npend : 0;          // tasks whose expert was not resident at entry
  const int npx = ADMIT ? s_npx : 0;              // ... their distinct experts
  const bool staged = ADMIT && s_staged;          // ... copied into staging entries at once
  if (LAYER && warp == 0) {
    if (!ADMIT) {
      for (int t = lane; t < T; t += 32) {
        int pe = -1;
        if (tk.slot[t] >= 0)
          for (int i = 0; i < n_pl0; ++i)
            if (a.gplan0[1 + 3 * i] == tk.slot[t]) pe = i;
        tk.pe[t] = pe;
      }
    }
    __syncwarp();
    // phase-A order: resident tasks, then the ones this launch copies in, so
    // that their rows are the last item of the warps that hold them
    int nres = 0;
    for (int t0 = 0; t0 < T; t0 += 32)
      nres += __popc(__ballot_sync(0xffffffffu, t0 + lane < T && tk.pe[t0 + lane] == -1));
    const unsigned lt = (1u << lane) - 1u;
    for (int t0 = 0, cr = 0, cm = nres; t0 < T; t0 += 32) {
      const int t = t0 + lane;
      const bool res = t < T && tk.pe[t] == -1, mis = t < T && !res;
      const unsigned br = __ballot_sync(0xffffffffu, res), bm = __ballot_sync(0xffffffffu, mis);
      if (res) tk.ord[cr + __popc(br & lt)] = t;
      if (mis) tk.ord[cm + __popc(bm & lt)] = t;
      cr += __popc(br);
      cm += __popc(bm);
    }
  }

  // ---- phase A assignment: whole rows of the flattened (task order, i) list,
  // dealt round-robin over the grid's warps: warp gw takes rows gw, gw + Gw, ...
  const int Gw = GF * kW, gw = cta * kW + warp;
  const int NA = T * I;
  const int nitA = (gw < NA ? (NA - 1 - gw) / Gw + 1 : 0) * KC;
  auto task_of = [&](int it) {  // the task of this warp's item `it`
    const int tp = (gw + (it / KC) * Gw) / I;
    return LAYER ? tk.ord[tp] : tp;
  };
  auto row_of = [&](int it) { return (gw + (it / KC) * Gw) % I; };  // its gate/up row
  // ---- phase-B items of this CTA (staged into shared memory after (2))
  const int bA = ru0 / H, bB = ru1 > ru0 ? (ru1 - 1) / H : bA;
  auto nlo_of = [&](int b) { return max(ru0 - b * H, 0); };
  auto nlen_of = [&](int b) { return min(ru1 - b * H, H) - nlo_of(b); };
  const int cntA = ru1 > ru0 ? (ts[bA + 1] - ts[bA]) * nlen_of(bA) : 0;
  const int cntB = (ru1 > ru0 && bB != bA) ? (ts[bB + 1] - ts[bB]) * nlen_of(bB) : 0;
  const int NQ = cntA + cntB;
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);
  float* ysm = reinterpret_cast<float*>(sm + ((size_t)n_rows * H * 2 + 127) / 128 * 128);
  float* hsm = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ysm) +
                                        ((size_t)a.R * perB * 4 + 127) / 128 * 128);
  uint8_t* ringA = reinterpret_cast<uint8_t*>(hsm) + ((size_t)a.htasks * I * 4 + 127) / 128 * 128;
  uint8_t* slots = ringA + (size_t)warp * 2 * kSlotBytes;  // this warp's two slots
  uint8_t* stC = ringA + (size_t)kW * 2 * kSlotBytes;
  uint8_t* stS = stC + (size_t)a.qs * CB;
  const int qs = min(a.qs, NQ);

  // ---- x in shared memory
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
  if (threadIdx.x < n_rows) {
    xinv[threadIdx.x] = FP4 ? 1.f / x_scale(__uint_as_float(xmax[threadIdx.x])) : 1.f;
  }
  if (lane == 0) {
    mbar_init(&bar_a[warp][0], 1);
    mbar_init(&bar_a[warp][1], 1);
    if (warp == 0) mbar_init(&bar_b, 1);
    fence_barrier_init();
  }
  __syncthreads();  // (2) x, barriers

  // ---- every byte this CTA needs is requested now: each warp's first two
  // phase-A items (bulk copies into its two slots) and the CTA's phase-B rows
  // (bulk copies into the staging area, on one barrier).  No CTA-wide barrier
  // follows until the grid barrier, so each warp computes as soon as its own
  // rows land.
  const uint64_t pol = l2_evict_first();
  // pieces per expert (a fused layer always has slot storage; 1 keeps the others well defined)
  const int ppe = LAYER ? max(1, (int)((st.slot_bytes + kPiece - 1) / kPiece)) : 1;
  // the gate/up global scales of the item in flight on each slot (lane 0)
  float2 gsl0 = make_float2(1.f, 1.f), gsl1 = make_float2(1.f, 1.f);
  auto issue_a = [&](int it, const uint8_t* blob) {  // lane 0
    const int sl = it & 1;
    mbar_expect_tx(&bar_a[warp][sl], ItemA<FMT>::BYTES);
    ItemA<FMT>::issue(slots + sl * kSlotBytes, blob, o, H, row_of(it), it % KC, &bar_a[warp][sl],
                      pol);
    const float2 g = ItemA<FMT>::glob(blob, o);
    gsl0 = sl ? gsl0 : g;
    gsl1 = sl ? g : gsl1;
  };
  // an item of an expert this launch copies in is requested only once the copy
  // is complete (see wait_copied below); every other item as soon as its slot is free
  auto deferred = [&](int it) { return LAYER && tk.pe[task_of(it)] != -1; };
  if (warp == kW - 1) {  // phase-B staging: one lane per (batch row, task) block
    const int nblk = (ru1 > ru0) ? (ts[bA + 1] - ts[bA]) + (bB != bA ? ts[bB + 1] - ts[bB] : 0) : 0;
    uint32_t mine = 0;
    for (int j = lane; j < nblk; j += 32) {
      const int bi = j < ts[bA + 1] - ts[bA] ? 0 : 1;
      const int b = bi ? bB : bA;
      const int t = ts[b] + (bi ? j - (ts[bA + 1] - ts[bA]) : j);
      const int nlen = nlen_of(b), q0 = (bi ? cntA : 0) + (t - ts[b]) * nlen;
      const int cnt = min(nlen, qs - q0);
      if (cnt > 0 && !(LAYER && tk.pe[t] != -1)) mine += (uint32_t)cnt * (CB + SB);
    }
    uint32_t total = mine;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
    if (lane == 0) mbar_expect_tx(&bar_b, total);  // before any of the copies can land
    __syncwarp();
    for (int j = lane; j < nblk; j += 32) {
      const int bi = j < ts[bA + 1] - ts[bA] ? 0 : 1;
      const int b = bi ? bB : bA;
      const int t = ts[b] + (bi ? j - (ts[bA + 1] - ts[bA]) : j);
      const int nlo = nlo_of(b), nlen = nlen_of(b), q0 = (bi ? cntA : 0) + (t - ts[b]) * nlen;
      const int cnt = min(nlen, qs - q0);
      if (cnt <= 0 || (LAYER && tk.pe[t] != -1)) continue;  // copied in by this launch: read later
      const uint8_t* blob = tk.blob[t];
      bulk_g2s(stC + (size_t)q0 * CB,
               blob + (FP4 ? o.code[2] : o.mat[2]) + (size_t)nlo * CB,
               (uint32_t)cnt * CB, &bar_b, pol);
      if (FP4)
        bulk_g2s(stS + (size_t)q0 * SB, blob + o.scale[2] + (size_t)nlo * SB, (uint32_t)cnt * SB,
                 &bar_b, pol);
    }
  }
  // this warp's first two phase-A items are requested before any copy work,
  // so that they land while it copies
  if (lane == 0) {
    if (nitA > 0 && !deferred(0)) issue_a(0, tk.blob[task_of(0)]);
    if (nitA > 1 && !deferred(1)) issue_a(1, tk.blob[task_of(1)]);
  }
  // fused layer: the step's missed experts (and the next layer's prefetches)
  // are copied from pinned host memory in 4 KiB pieces, one per warp at a
  // time, consecutive pieces on consecutive CTAs (so every SM issues host
  // reads).  Each finished piece of a demand entry is counted, and the rows of
  // that expert wait for the full count.  A warp does its pieces before it can
  // wait on any, and a step without misses has no pieces.
  // admission inside: wait (bounded, the whole warp on lane 0's reads) until
  // CTA 0 has published pseq >= target; then every lane acquires too
  auto wait_seq = [&](unsigned long long target) -> bool {
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
  };
  auto copy_piece = [&](long p, int np0) {  // piece p of the demand plan, then the prefetch plan
    const int ei = (int)(p / ppe), j = (int)(p - (long)ei * ppe);
    const bool demand = ei < np0;
    const int32_t* plan = demand ? a.gplan0 : a.gplan1;
    const int i = demand ? ei : ei - np0;
    const int s = plan[1 + 3 * i], L = plan[2 + 3 * i], e = plan[3 + 3 * i];
    if ((unsigned)s < (unsigned)st.S && (unsigned)L < (unsigned)st.L && (unsigned)e < (unsigned)st.E) {
      const size_t off = (size_t)j * kPiece;
      const int len = (int)min((size_t)kPiece, st.slot_bytes - off);
      const uint4* src = reinterpret_cast<const uint4*>(st.host_blob[L * st.E + e] + off);
      uint4* dst = reinterpret_cast<uint4*>(
          st.slots + ((size_t)pool_of(st, L) * st.S + s) * st.stride + off);
      const int nv = len / 16;
      uint4 v[kPiece / 512];
#pragma unroll
      for (int u = 0; u < kPiece / 512; ++u)
        if (lane + 32 * u < nv) v[u] = src[lane + 32 * u];
#pragma unroll
      for (int u = 0; u < kPiece / 512; ++u)
        if (lane + 32 * u < nv) dst[lane + 32 * u] = v[u];
    }
    __syncwarp();
    if (demand && lane == 0) {
      __threadfence();
      atomicAdd(a.gdone + i, 1);
    }
  };
  // a staging piece: piece p of the step's missed experts, from pinned host
  // memory into their staging entry and into the slot the admission gave the
  // expert (a victim: no task of this step reads it), so the end of the launch
  // only has to make the map entries valid.  While the host reads are in
  // flight the warp polls CTA 0's word for the entry (the slot, tagged with
  // this launch); the piece is counted (like the demand plan's pieces) once
  // it is in the staging entry.
  auto stage_piece = [&](long p) {
    const int i = (int)(p / ppe), j = (int)(p - (long)i * ppe);
    const int e = s_pexp[i];
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
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(a.gdone + i, 1);
    }
    if (sl < (uint32_t)st.S) {
      uint4* sdst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(slot_blob((int)sl)) + off);
#pragma unroll
      for (int u = 0; u < kPiece / 512; ++u)
        if (lane + 32 * u < nv) sdst[lane + 32 * u] = v[u];
    }
  };
  const bool pf_plan = a.gplan1 && (!ADMIT || (a.pred && a.n_pred > 0));  // a prefetch plan to copy
  {
    const long p0 = (long)warp * GF + cta;  // this warp's first piece
    if (staged) {  // the misses start crossing the host link now, whatever the admission does
      for (long p = p0; p < (long)npx * ppe; p += Gw) stage_piece(p);
    } else if (ADMIT) {
      // a warp can only get pieces below (misses + predictions) * ppe; the
      // others need not wait for the plans here
      const long bound = (long)(npend + (pf_plan ? a.n_pred : 0)) * ppe;
      if (p0 < bound && wait_seq(seq0 + 1)) {
        const int np0 = a.gplan0[0];
        for (long p = p0; p < (long)np0 * ppe; p += Gw) copy_piece(p, np0);
        if (pf_plan && wait_seq(seq0 + 2)) {
          const long end = (long)(np0 + a.gplan1[0]) * ppe;
          long p = p0;
          while (p < (long)np0 * ppe) p += Gw;
          for (; p < end; p += Gw) copy_piece(p, np0);
        }
      }
    } else if (LAYER && n_pl0 + n_pl1 > 0) {
      const long total = (long)(n_pl0 + n_pl1) * ppe;
      for (long p = p0; p < total; p += Gw) copy_piece(p, n_pl0);
    }
  }

  // per-task combine factor (stored to shared memory before the grid barrier)
  float cw = 1.f, c2 = 1.f;
  if (threadIdx.x < T) {
    if (MODE != kShared && tk.route[threadIdx.x] < a.R) cw = a.w[tk.route[threadIdx.x]];
    if (FMT == MOE_W_NVFP4 && tk.blob[threadIdx.x])  // not yet resident: set after the barrier
      c2 = reinterpret_cast<const float*>(tk.blob[threadIdx.x] + o.glob)[2];
  }

  // the shared expert's sigmoid gate, sigmoid(x_b . w_g), in fp32, by the last
  // CTA (the one least likely to hold phase-A rows), before its phase A
  if ((SHARED || (LAYER && a.shared_blob)) && blockIdx.x == gridDim.x - 1 && warp < n_rows) {
    float z = 0.f;
    for (int i0 = lane * 8; i0 < H; i0 += 256) {
      const uint4 gv = *reinterpret_cast<const uint4*>(a.gate_w + i0);
      const uint4 xv = *reinterpret_cast<const uint4*>(a.x + (size_t)warp * H + i0);
      z = dot8_bf16_bf(gv, xv, z);
    }
    z = wsum(z);
    if (lane == 0) a.gate[warp] = 1.f / (1.f + expf(-z));
  }

  // ---------------------------------------------------------------- phase A
  bool failed = false;  // a timed-out wait: skip the rest
  // the item whose copies are in flight on each of the warp's two slots, -1 =
  // none (warp-uniform: every lane takes the same decisions as lane 0)
  int inflight[2] = {nitA > 0 && !deferred(0) ? 0 : -1, nitA > 1 && !deferred(1) ? 1 : -1};
  // Items are (row, chunk) pairs, alternating between two register buffers;
  // the next item of a buffer is requested as soon as its dot is done.  With
  // one chunk per row (KC = 1) each buffer holds a whole row and the two rows
  // are reduced together; with an even KC a row's chunks alternate buffers and
  // it completes on the second buffer.
  {
    const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
    auto xrow = [&](int it) {
      return xs4 + (size_t)tk.b[task_of(it)] * (H / 8);
    };
    auto store_h = [&](int it, float gsum, float usum, float gs0, float gs1) {  // lane 0
      const int t = task_of(it);
      const float xi = xinv[tk.b[t]];
      const float gg = gsum * xi * gs0, uu = usum * xi * gs1;
      a.h[(size_t)tk.route[t] * I + row_of(it)] = gg / (1.f + expf(-gg)) * uu;
    };
    float ga = 0.f, ua = 0.f, gb = 0.f, ub = 0.f;
    // fused layer: wait (bounded, the whole warp on lane 0's reads) until this
    // launch has copied all of demand-plan entry pe into its slot
    auto wait_copied = [&](int pe) -> bool {
      const int* ctr = a.gdone + pe;
      const unsigned long long t0 = now_ns();
      for (;;) {
        int s = 0;  // 1: complete, 2: timed out
        if (lane == 0) {
          int v;
          asm volatile("ld.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
          s = v >= ppe ? 1 : (now_ns() - t0 > kWaitNs ? 2 : 0);
        }
        s = __shfl_sync(0xffffffffu, s, 0);
        if (s == 1) return true;
        if (s == 2) {
          if (lane == 0) flag_timeout(a.status);
          return false;
        }
        __nanosleep(256);
      }
    };
    // item `it` in its slot (warp-uniform); a deferred item is requested here
    auto wait_a = [&](int it) -> bool {
      const int sl = it & 1;
      if (inflight[sl] != it) {  // deferred: its expert is being copied in by this launch
        const int t = task_of(it);
        const uint8_t* blob = tk.blob[t];
        int pe = tk.pe[t];
        if (ADMIT && !staged) {  // decided by CTA 0's admission
          if (!wait_seq(seq0 + 1)) {
            failed = true;
            return false;
          }
          const int s = a.slot_out[tk.route[t]];
          blob = s >= 0 ? slot_blob(s) : nullptr;
          pe = -1;
          if (s >= 0) {  // its entry in the demand plan
            const int np = a.gplan0[0];
            for (int i0 = 0; i0 < np; i0 += 32) {
              const unsigned hit =
                  __ballot_sync(0xffffffffu, i0 + lane < np && a.gplan0[1 + 3 * (i0 + lane)] == s);
              if (hit) {
                pe = i0 + __ffs(hit) - 1;
                break;
              }
            }
          }
        }
        if (pe >= 0 && !wait_copied(pe)) {
          failed = true;
          return false;
        }
        if (lane == 0) {
          if (blob) {
            fence_proxy_async();  // the slot's previous reads before the new bulk writes
            asm volatile("fence.proxy.async.global;" ::: "memory");  // copied bytes -> bulk reads
            issue_a(it, blob);
          } else {  // not admitted (fetch cap): nothing to copy; its h is never read
            mbar_arrive(&bar_a[warp][sl]);
          }
        }
        inflight[sl] = it;
      }
      const bool all = __all_sync(0xffffffffu, mbar_wait(&bar_a[warp][sl], (uint32_t)((it >> 1) & 1)));
      if (all) {
        inflight[sl] = -1;
      } else {
        failed = true;
        if (lane == 0) flag_timeout(a.status);
      }
      return all;
    };
    for (int it = 0; it < nitA && !failed; it += 2) {
      const bool two = it + 1 < nitA;
      if (!wait_a(it)) break;
      const uint8_t* sa = slots;
      ItemA<FMT>::dot(sa, xrow(it), it % KC, lane, ga, ua);
      const float a0 = gsl0.x, a1 = gsl0.y;
      __syncwarp();  // slot 0 read by every lane
      if (it + 2 < nitA && !deferred(it + 2)) {
        if (lane == 0) {
          fence_proxy_async();
          issue_a(it + 2, tk.blob[task_of(it + 2)]);
        }
        inflight[0] = it + 2;
      }
      float b0 = 1.f, b1 = 1.f;
      if (two) {
        if (!wait_a(it + 1)) break;
        const uint8_t* sb = slots + kSlotBytes;
        ItemA<FMT>::dot(sb, xrow(it + 1), (it + 1) % KC, lane, gb, ub);
        b0 = gsl1.x;
        b1 = gsl1.y;
        __syncwarp();
        if (it + 3 < nitA && !deferred(it + 3)) {
          if (lane == 0) {
            fence_proxy_async();
            issue_a(it + 3, tk.blob[task_of(it + 3)]);
          }
          inflight[1] = it + 3;
        }
      }
      if (KC == 1) {  // rows it and it + 1 complete
        const float p[4] = {ga, ua, gb, ub};
        const float v = reduce4(p, lane);
        const float va = __shfl_sync(0xffffffffu, v, 8), vb = __shfl_sync(0xffffffffu, v, 16),
                    vc = __shfl_sync(0xffffffffu, v, 24);
        if (lane == 0) {
          store_h(it, v, va, a0, a1);
          if (two) store_h(it + 1, vb, vc, b0, b1);
        }
        ga = ua = gb = ub = 0.f;
      } else if ((it + 1) % KC == KC - 1) {  // the row of items it, it + 1 completes
        const float2 gu = reduce2(ga + gb, ua + ub, lane);
        if (lane == 0) store_h(it + 1, gu.x, gu.y, b0, b1);
        ga = ua = gb = ub = 0.f;
      }
    }
    // after a timeout, wait (bounded) for this warp's copies still in flight
    if (failed && lane == 0)
      for (int sl = 0; sl < 2; ++sl)
        if (inflight[sl] >= 0) mbar_wait(&bar_a[warp][sl], (uint32_t)((inflight[sl] >> 1) & 1));
  }
  if (threadIdx.x < T) tk.wt[threadIdx.x] = cw * c2;  // read after the barrier

  // ---------------------------------------------------------------- barrier
  const bool ok = grid_barrier(ADMIT ? a.bar2 : a.bar_ctr, a.status, (unsigned)GF);
  const bool rows_in = mbar_wait(&bar_b, 0);  // the staged phase-B rows (bounded)
  if (!rows_in) flag_timeout(a.status);
  if (!ok || !__syncthreads_and(rows_in)) return;  // timed out: nothing below is trustworthy
  int n_done = staged ? npx : n_pl0;  // piece counters this launch used
  if (ADMIT && npend > 0) {  // the tasks not resident at entry, as CTA 0 admitted them
    if (warp == 0) (void)wait_seq(seq0 + 1);  // bounded
    __syncthreads();
    (void)ld_acquire_u64(a.pseq);
    if (!staged) n_done = a.gplan0[0];
    const int t = threadIdx.x;
    if (t < T && tk.pend[t]) {
      const int s = a.slot_out[tk.route[t]];
      if (s < 0) {
        tk.drop[t] = 1;  // not admitted (fetch cap, no slot): no output term, as in the
                         // two-launch path
      } else if (!staged) {
        int pe = -1;
        for (int i = 0; i < n_done && pe < 0; ++i)
          if (a.gplan0[1 + 3 * i] == s) pe = i;
        tk.blob[t] = slot_blob(s);
        tk.slot[t] = s;
        tk.pe[t] = pe;
      }
    }
    __syncthreads();
  }
  if (LAYER && cta == 0)  // every wait on the copies is behind the barrier
    for (int i = threadIdx.x; i < n_done; i += kT) a.gdone[i] = 0;
  // an expert copied in by this launch: its down global scale is in the slot
  // only now (read by the combine, after the next block barrier)
  if (LAYER && FMT == MOE_W_NVFP4 && threadIdx.x < T && tk.pe[threadIdx.x] >= 0)
    tk.wt[threadIdx.x] = cw * reinterpret_cast<const float*>(tk.blob[threadIdx.x] + o.glob)[2];
  // the gate of this thread's combine row, requested now (written before the barrier)
  const float gate_b = ((SHARED || (LAYER && a.shared_blob)) && ru0 + (int)threadIdx.x < ru1)
                           ? __ldcg(&a.gate[(ru0 + (int)threadIdx.x) / H])
                           : 0.f;
  // h of the tasks this CTA's rows need, read once from L2 into shared memory
  // (every warp reading it from L2 would hammer a few cache lines)
  const int tlo = ru1 > ru0 ? ts[bA] : 0, thi = ru1 > ru0 ? ts[bB + 1] : 0;
  {  // up to kHU loads of each thread in flight before any is stored
    constexpr int kHU = 4;
    float4* h4 = reinterpret_cast<float4*>(hsm);
    const int n4 = (thi - tlo) * I / 4, i4 = I / 4;
    for (int i0 = threadIdx.x; i0 < n4; i0 += kHU * kT) {
      float4 hv4[kHU];
#pragma unroll
      for (int u = 0; u < kHU; ++u) {
        const int i = i0 + u * kT;
        if (i < n4)
          hv4[u] = __ldcg(reinterpret_cast<const float4*>(a.h + (size_t)tk.route[tlo + i / i4] * I) +
                          (i % i4));
      }
#pragma unroll
      for (int u = 0; u < kHU; ++u)
        if (i0 + u * kT < n4) h4[i0 + u * kT] = hv4[u];
    }
  }
  __syncthreads();  // h visible to every warp

  // ---------------------------------------------------------------- phase B
  // warp w takes items [w*ipw, (w+1)*ipw), in runs of up to NG of one task
  // (NG = 4 for NVFP4; 2 for bf16, whose rows hold twice the registers).  The
  // run loop is instantiated for the lane's element count (M = I / 512), and a
  // run whose rows were all staged reads them with shared-memory loads.
  {
    constexpr int NG = FP4 ? 4 : 2;
    const int ipw = (NQ + kW - 1) / kW;
    const int q0w = min(NQ, warp * ipw), q1w = min(NQ, q0w + ipw);
    auto run_b = [&](auto mtag) {
      constexpr int M = decltype(mtag)::value;
      if (q0w >= q1w) return;
      // item q0w: batch row b, task t, row r of the task's nlen rows
      int b = q0w >= cntA ? bB : bA;
      int nlo = nlo_of(b), nlen = nlen_of(b);
      const int qr = q0w - (q0w >= cntA ? cntA : 0);
      int t = ts[b] + qr / nlen, r = qr % nlen;
      float hv[16 * M];
      int ht = -1;
      for (int q = q0w; q < q1w;) {
        const int cnt = min(NG, min(q1w - q, nlen - r));  // items of this run: one task
        if (t != ht) {  // this task's h slice into registers
          const float* hp = hsm + (size_t)(t - tlo) * I;
          if (FP4) {
#pragma unroll
            for (int j = 0; j < 4 * M; ++j) {
              const float4 v = reinterpret_cast<const float4*>(hp + lane * 16 * M)[j];
              hv[4 * j] = v.x, hv[4 * j + 1] = v.y, hv[4 * j + 2] = v.z, hv[4 * j + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int s = 0; s < 2 * M; ++s) {
              const float4 v0 = *reinterpret_cast<const float4*>(hp + 256 * s + 8 * lane);
              const float4 v1 = *reinterpret_cast<const float4*>(hp + 256 * s + 8 * lane + 4);
              hv[8 * s] = v0.x, hv[8 * s + 1] = v0.y, hv[8 * s + 2] = v0.z, hv[8 * s + 3] = v0.w;
              hv[8 * s + 4] = v1.x, hv[8 * s + 5] = v1.y, hv[8 * s + 6] = v1.z, hv[8 * s + 7] = v1.w;
            }
          }
          ht = t;
        }
        ItemB<FMT> itm[NG];
        const bool copied = LAYER && tk.pe[t] != -1;  // copied in by this launch: not staged
        if (ADMIT && tk.drop[t]) {  // not admitted: no rows, no output term (warp-uniform)
        } else if (!copied && q + cnt <= qs) {
#pragma unroll
          for (int j = 0; j < NG; ++j)
            if (j < cnt)
              itemb_load<FMT>(itm[j], stC + (size_t)(q + j) * CB, stS + (size_t)(q + j) * SB, M,
                              lane);
        } else {
          const uint8_t* blob = tk.blob[t];
#pragma unroll
          for (int j = 0; j < NG; ++j) {
            if (j >= cnt) continue;
            const int qq = q + j, n = nlo + r + j;
            if (!copied && qq < qs)
              itemb_load<FMT>(itm[j], stC + (size_t)qq * CB, stS + (size_t)qq * SB, M, lane);
            else
              itemb_load<FMT>(itm[j],
                              blob + (FP4 ? o.code[2] : o.mat[2]) + (size_t)n * CB,
                              blob + o.scale[2] + (size_t)n * SB, M, lane);
          }
        }
        if (!(ADMIT && tk.drop[t])) {
          float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < NG; ++j) p[j] = j < cnt ? itemb_dot<FMT>(itm[j], hv, M) : 0.f;
          const float v = reduce4(p, lane);
          const int j = lane >> 3;
          if ((lane & 7) == 0 && j < cnt) ysm[(size_t)t * perB + (b * H + nlo + r + j - ru0)] = v;
        }
        q += cnt;
        r += cnt;
        if (r == nlen) {  // the task's rows are done: the next task, maybe of the next batch row
          r = 0;
          ++t;
          if (t == ts[b + 1] && b != bB) {
            b = bB;
            nlo = nlo_of(b);
            nlen = nlen_of(b);
          }
        }
      }
    };
    if (m == 1)
      run_b(std::integral_constant<int, 1>{});
    else
      run_b(std::integral_constant<int, 2>{});
  }
  __syncthreads();  // every (task, row) result in ysm
  // combine: each output row, its tasks in route order (j ascending), then + ys
  int mm = 0;
  const bool has_s = LAYER && a.shared_blob;  // row b's last task is the shared expert
  for (int ru = ru0 + threadIdx.x; ru < ru1; ru += kT, ++mm) {
    const int b = ru / H;
    const int te = ts[b + 1] - (has_s ? 1 : 0);
    float acc = 0.f;
    for (int t = ts[b]; t < te; ++t)
      if (!(ADMIT && tk.drop[t])) acc = fmaf(tk.wt[t], ysm[(size_t)t * perB + (ru - ru0)], acc);
    if (LAYER) {  // routed sum (j ascending), then + gate * shared, as in the two-launch path
      float yv = 0.f;
      if (has_s)
        yv = (mm == 0 ? gate_b : __ldcg(&a.gate[b])) * (tk.wt[te] * ysm[(size_t)te * perB + (ru - ru0)]);
      a.out[ru] = __float2bfloat16_rn(has_s ? acc + yv : acc);
    } else if (SHARED) {
      a.ys[ru] = (mm == 0 ? gate_b : __ldcg(&a.gate[b])) * acc;
    } else {
      const float yv = mm < kYsPre ? ysv[mm] : (a.ys ? a.ys[ru] : 0.f);
      a.out[ru] = __float2bfloat16_rn(a.ys ? acc + yv : acc);
    }
  }
  if (ADMIT) {
    // the admitted misses' map entries valid for later launches: every
    // computing CTA read the map, and (staged steps) wrote its pieces into the
    // slots, before the barrier
    if (npend > 0 && cta == 0) {
      const int np0 = a.gplan0[0];
      for (int i = threadIdx.x; i < np0; i += kT) {
        const int s = a.gplan0[1 + 3 * i], L = a.gplan0[2 + 3 * i], e = a.gplan0[3 + 3 * i];
        if ((unsigned)s < (unsigned)st.S && L == a.layer && (unsigned)e < (unsigned)st.E)
          st.map[a.layer * st.E + e] = s;
      }
    }
    // staged steps copy the next layer's prefetches last
    if (staged && pf_plan && wait_seq(seq0 + 2)) {
      const int np0 = a.gplan0[0], np1 = a.gplan1[0];
      for (long p = (long)warp * GF + cta; p < (long)np1 * ppe; p += Gw)
        copy_piece((long)np0 * ppe + p, np0);
    }
  }
}

// SMs of each device, set by ffn_stream_init with that device current (0: not
// set up, the streaming kernels are not used there)
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
std::mutex g_init_mu;
int num_sms() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
  return g_sms[d];
}
constexpr size_t kBudget = 200 * 1024;

size_t round128(size_t v) { return (v + 127) / 128 * 128; }

struct Plan {
  size_t smem;
  int qs, htasks;
  bool ok;
};

// Shared memory: x [n_rows][H] | ysm [T][perB] fp32 | h [htasks][I] fp32 |
// two phase-A slots per warp | staged phase-B rows.  A CTA's output rows span at most two batch rows, so
// it needs the h of at most 2k tasks.
Plan fused_plan(int wfmt, int H, int I, int n_rows, int k, int T, int G) {
  Plan p{};
  const int perB = (n_rows * H + G - 1) / G;
  const int rowB = wfmt == MOE_W_BF16 ? I * 2 : (wfmt == MOE_W_MXFP4 ? I / 2 + I / 32 : I / 2 + I / 16);
  p.htasks = std::min(T, 2 * k);
  const size_t fixed = round128((size_t)n_rows * H * 2) + round128((size_t)T * perB * 4) +
                       round128((size_t)p.htasks * I * 4) + (size_t)kW * 2 * kSlotBytes;
  const int nq = k * perB * 2;  // at most two batch rows of k tasks each
  const size_t room = fixed < kBudget ? kBudget - fixed : 0;
  p.qs = (int)std::min<size_t>((size_t)nq, room / rowB);
  p.smem = fixed + (size_t)p.qs * rowB;
  const int CW = wfmt == MOE_W_BF16 ? 512 : 2048;
  const int KC = H / CW;
  p.ok = fixed <= kBudget && H % CW == 0 && (KC == 1 || KC % 2 == 0) && I % 512 == 0 &&
         I <= 1024 && perB <= H &&
         n_rows * H <= kXW * 8 * kT;
  return p;
}

int grid_of(int mode) {  // computing CTAs (CTA 0 admits in kLayerAdmit)
  const int G = std::max(1, num_sms());
  return mode == kLayerAdmit ? std::max(1, G - 1) : G;
}

// Shared memory of CTA 0 in kLayerAdmit: its block state, then the admission's
// [E] x 3 counters (and the pool's keys when cached), or the prefetch's [E] x 2.
size_t admit_cta_smem(int E, int S, bool cached) {
  const size_t adm = 3ull * E * sizeof(int) + (cached ? (size_t)S * 12 : 0);
  return round128(sizeof(admission::AdmitShared<kT>)) + std::max<size_t>(adm, 2ull * E * sizeof(int));
}

template <typename K>
cudaError_t launch_coop(K kernel, size_t smem, cudaStream_t s, const DevState& st,
                        const FusedArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, st, a);
}

// tasks per batch row and in all, for a launch of `mode`
int tasks_per_row(int mode, int k, bool shared) {
  return (mode == kLayer || mode == kLayerAdmit) ? k + (shared ? 1 : 0) : k;
}

template <int FMT>
cudaError_t launch_mode(int mode, size_t smem, cudaStream_t s, const DevState& st,
                        const FusedArgs& a) {
  switch (mode) {
    case kLayerAdmit: return launch_coop(ffn_fused_kernel<FMT, kLayerAdmit>, smem, s, st, a);
    case kLayer: return launch_coop(ffn_fused_kernel<FMT, kLayer>, smem, s, st, a);
    case kShared: return launch_coop(ffn_fused_kernel<FMT, kShared>, smem, s, st, a);
    default: return launch_coop(ffn_fused_kernel<FMT, kRouted>, smem, s, st, a);
  }
}
cudaError_t launch_format(int wfmt, int mode, size_t smem, cudaStream_t s, const DevState& st,
                          const FusedArgs& a) {
  if (wfmt == MOE_W_NVFP4) return launch_mode<MOE_W_NVFP4>(mode, smem, s, st, a);
  if (wfmt == MOE_W_MXFP4) return launch_mode<MOE_W_MXFP4>(mode, smem, s, st, a);
  if (wfmt == MOE_W_Q4_0) return launch_mode<MOE_W_Q4_0>(mode, smem, s, st, a);
  return launch_mode<MOE_W_BF16>(mode, smem, s, st, a);
}

cudaError_t launch_fused(const DevState& st, int wfmt, int mode, const FusedArgs& a0,
                         cudaStream_t s) {
  FusedArgs a = a0;
  const bool sh = a.shared_blob != nullptr;
  const bool layer = mode == kLayer || mode == kLayerAdmit;
  const int kt = tasks_per_row(mode, a.k, sh);
  const Plan p = fused_plan(wfmt, a.H, a.I, a.n_rows, kt, a.R + (layer && sh ? a.n_rows : 0),
                            grid_of(mode));
  a.qs = p.qs;
  a.htasks = p.htasks;
  size_t smem = p.smem;
  if (mode == kLayerAdmit) smem = std::max(smem, admit_cta_smem(st.E, st.S, a.adm_cached != 0));
  if (smem > kBudget) return cudaErrorInvalidValue;
  return launch_format(wfmt, mode, mode == kLayerAdmit ? smem : p.smem, s, st, a);
}

}  // namespace

bool ffn_stream_supported(int wfmt, int H, int I, int n_rows, int n_tasks) {
  if (num_sms() <= 0 || n_tasks > kMaxRoutes || n_rows > kMaxRows || n_rows < 1) return false;
  const int k = (n_tasks + n_rows - 1) / n_rows;
  return fused_plan(wfmt, H, I, n_rows, k, n_tasks, grid_of(kRouted)).ok;
}

// Per device, once: the kernels' shared-memory limit (a per-device function
// attribute) and the device's SM count.
cudaError_t ffn_stream_init() {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_init_mu);
  if (g_sms[dev] > 0) return cudaSuccess;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto set = [&](auto kern) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBudget);
  };
  set(ffn_fused_kernel<MOE_W_BF16, kShared>);
  set(ffn_fused_kernel<MOE_W_NVFP4, kShared>);
  set(ffn_fused_kernel<MOE_W_BF16, kRouted>);
  set(ffn_fused_kernel<MOE_W_NVFP4, kRouted>);
  set(ffn_fused_kernel<MOE_W_BF16, kLayer>);
  set(ffn_fused_kernel<MOE_W_NVFP4, kLayer>);
  set(ffn_fused_kernel<MOE_W_BF16, kLayerAdmit>);
  set(ffn_fused_kernel<MOE_W_NVFP4, kLayerAdmit>);
  set(ffn_fused_kernel<MOE_W_MXFP4, kShared>);
  set(ffn_fused_kernel<MOE_W_MXFP4, kRouted>);
  set(ffn_fused_kernel<MOE_W_MXFP4, kLayer>);
  set(ffn_fused_kernel<MOE_W_MXFP4, kLayerAdmit>);
  set(ffn_fused_kernel<MOE_W_Q4_0, kShared>);
  set(ffn_fused_kernel<MOE_W_Q4_0, kRouted>);
  set(ffn_fused_kernel<MOE_W_Q4_0, kLayer>);
  set(ffn_fused_kernel<MOE_W_Q4_0, kLayerAdmit>);
  if (e == cudaSuccess) g_sms[dev] = sms;
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
  return launch_fused(st, wfmt, kShared, a, s);
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
  return launch_fused(st, wfmt, kRouted, a, s);
}

bool layer_stream_supported(int wfmt, int H, int I, int n_rows, int k, bool shared) {
  if (num_sms() <= 0 || n_rows < 1 || n_rows > kMaxRows || n_rows * k > kMaxRoutes) return false;
  const int kt = tasks_per_row(kLayer, k, shared);
  const int T = n_rows * kt;
  return T <= kMaxTasks && fused_plan(wfmt, H, I, n_rows, kt, T, grid_of(kLayer)).ok;
}

bool layer_admit_supported(const DevState& st, int wfmt, int H, int I, int n_rows, int k,
                           bool shared) {
  if (num_sms() < 2 || st.E > kPbWords * 32 || !layer_stream_supported(wfmt, H, I, n_rows, k, shared))
    return false;
  const int kt = tasks_per_row(kLayerAdmit, k, shared);
  const Plan p = fused_plan(wfmt, H, I, n_rows, kt, n_rows * kt, grid_of(kLayerAdmit));
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
  a.fixed_blob = nullptr;
  a.w = w;
  a.h = sc.h;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.gate = sc.gate;
  a.ys = nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.bar_ctr = sc.bar;
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
  a.bar2 = sc.bar2;
  a.sslot = sc.sslot;
  const int kt = tasks_per_row(kLayerAdmit, k, shared_blob != nullptr);
  const Plan p = fused_plan(wfmt, H, I, n_rows, kt, n_rows * kt, grid_of(kLayerAdmit));
  a.adm_cached = admit_cached(st.E, st.S) &&
                 std::max(p.smem, admit_cta_smem(st.E, st.S, true)) <= kBudget;
  return launch_fused(st, wfmt, kLayerAdmit, a, s);
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
  a.fixed_blob = nullptr;
  a.w = w;
  a.h = sc.h;
  a.gate_w = static_cast<const uint16_t*>(gate_w);
  a.gate = sc.gate;
  a.ys = nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.bar_ctr = sc.bar;
  a.shared_blob = shared_blob;
  a.gplan0 = plan0;
  a.gplan1 = plan1;
  a.gdone = sc.gdone;
  return launch_fused(st, wfmt, kLayer, a, s);
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
    if (e == cudaSuccess) e = ffn_stream_init();
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
