// grouped.cu -- routed expert FFNs for wide steps, grouped by expert.
//
// What is computed is the routed half of the layer (FreeToken issue #753
// "[Perf] Offloaded decode: overlap the expert-miss gather with the same
// layer's shared expert ...", Problem and What we changed; FreeToken PR #680
// "fix(moe): admit a wide offloaded decode step's experts 128 at a time",
// Tests: a wide step's routes over many distinct experts):
//   out[b] = bf16( sum_j w[b,j] * FFN_slot[b,j](x[b]) + ys[b] ),
// j ascending, routes with slot -1 skipped.
//
// A wide step (hundreds of rows, top-k) routes ~1-10 rows to each of hundreds
// of experts: about two multiply-adds per weight byte, so the work is bound by
// reading every resident expert once from HBM (and, on the CUDA cores, by the
// instructions of the exact products), not by the tensor cores.  The kernels
// therefore group the routes by expert and read each expert's weights once:
//   1. group_kernel   (1 CTA): the CSR of routes per distinct expert, ascending
//      expert id, routes ascending within a group -- the cache's route groups;
//   2. xprep_kernel:  x as f16 (4-bit experts; per-row power-of-two scale so
//      that max |x| < 2^15, undone on the fp32 sums) or bf16 (bf16 experts);
//   3. gate/up:       h[r] = silu(W_g x_b) * (W_u x_b) for every route r of a
//      group -- NVFP4 at H = 1024 JH: gup_warp_kernel (a warp per 8 rows,
//      lanes over K, x in registers); other shapes: gup_staged_kernel /
//      gup_kernel (a thread per row, x broadcast from shared memory);
//   4. down:          y[r] = gs_d * W_d h[r] -- NVFP4 at I = 256 M:
//      gdown_warp_kernel (a warp per 32 rows, h in registers); other shapes:
//      gdown_staged_kernel / gdown_kernel;
//   5. combine_kernel: out[b][n] = bf16( sum_j w[b,j] y[b*k+j][n] + ys[b][n] ).
// Kernels 3 and 4 are persistent (a few CTAs per SM walk the work items), so
// the data-dependent number of groups needs no host round trip.  Expert groups
// of many routes may go to the tensor cores instead (grouped_tc.cu).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGT = 1024;       // group_kernel threads
constexpr int kWT = 256;        // threads of the FFN kernels (8 warps)
constexpr int kNR = 4;          // routes per decode pass

// ------------------------------------------------------------ small helpers

template <int B>
__device__ __forceinline__ uint32_t e2m1x2(uint32_t w) {
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
__device__ __forceinline__ float2 f16x2_f32(uint32_t h2) {
  float a, b;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
      : "=f"(a), "=f"(b) : "r"(h2));
  return make_float2(a, b);
}
// two E4M3 scales (low byte first) as fp32
__device__ __forceinline__ float2 e4m3x2(uint32_t v16) {
  uint32_t h2;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(h2)
      : "r"(v16));
  return f16x2_f32(h2);
}
// c + w.lo * x.lo + w.hi * x.hi with half (or bfloat16) operands, fp32 result
__device__ __forceinline__ float fma2h(uint32_t w2, uint32_t x2, float c) {
  float d;
  asm("{ .reg .b16 a0, a1, b0, b1; .reg .f32 t;\n"
      " mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.f16 t, a0, b0, %3;\n fma.rn.f32.f16 %0, a1, b1, t; }"
      : "=f"(d) : "r"(w2), "r"(x2), "f"(c));
  return d;
}
__device__ __forceinline__ float fma2b(uint32_t w2, uint32_t x2, float c) {
  float d;
  asm("{ .reg .b16 a0, a1, b0, b1; .reg .f32 t;\n"
      " mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.bf16 t, a0, b0, %3;\n fma.rn.f32.bf16 %0, a1, b1, t; }"
      : "=f"(d) : "r"(w2), "r"(x2), "f"(c));
  return d;
}
__device__ __forceinline__ float fp32_of_bf16(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Offsets inside a blob (layout of moe_cache.h): the scale banks hold ih/16
// bytes (NVFP4: e4m3 per 16; Q4_0: fp16 per 32) or ih/32 (MXFP4: E8M0 per 32).
struct Off {
  size_t code[3], scale[3], glob, mat[3];
  __device__ Off(int H, int I, int fmt = MOE_W_NVFP4) {
    const size_t ih = (size_t)I * H;
    const size_t sb = ih / (fmt == MOE_W_MXFP4 ? 32 : 16);
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

// MXFP4 and Q4_0: 32-element blocks.  The scale of block j of a row's scales
// (E8M0 2^(e - 127), 0xFF NaN; or fp16 d), and a block's 32 codes (16 bytes)
// as 16 half2 words: e2m1 values, or q - 8 for Q4_0 (exact in f16).
template <int FMT>
__device__ __forceinline__ float blk32_scale(const uint8_t* scales, int j) {
  if (FMT == MOE_W_MXFP4) {
    const uint32_t e = scales[j];
    return e == 0 ? __uint_as_float(0x00400000u)
                  : (e == 255 ? __uint_as_float(0x7fffffffu) : __uint_as_float(e << 23));
  }
  return __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(scales)[j]));
}
template <int FMT>
__device__ __forceinline__ void blk32_decode(uint4 c, uint32_t d[16]) {
  const uint32_t v[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
    if (FMT == MOE_W_Q4_0) {  // nibbles into the mantissa of f16 1024 + q, minus 1032
      const uint32_t lo = v[wd] & 0x0F0F0F0Fu, hi = (v[wd] >> 4) & 0x0F0F0F0Fu;
      const uint32_t m0 = __byte_perm(lo, hi, 0x5140), m1 = __byte_perm(lo, hi, 0x7362);
      const uint32_t k = 0x64646464u;
      const uint32_t t[4] = {__byte_perm(m0, k, 0x4140), __byte_perm(m0, k, 0x4342),
                             __byte_perm(m1, k, 0x4140), __byte_perm(m1, k, 0x4342)};
      const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&t[q]), bias);
        d[4 * wd + q] = *reinterpret_cast<const uint32_t*>(&r);
      }
    } else {
      d[4 * wd] = e2m1x2<0>(v[wd]);
      d[4 * wd + 1] = e2m1x2<1>(v[wd]);
      d[4 * wd + 2] = e2m1x2<2>(v[wd]);
      d[4 * wd + 3] = e2m1x2<3>(v[wd]);
    }
  }
}

// The route groups buffer: [G, slot[R], start[R + 1], route[R]], R = max_routes.
struct Groups {
  int32_t* base;
  int R;
  __device__ int32_t& G() const { return base[0]; }
  __device__ int32_t* slot() const { return base + 1; }
  __device__ int32_t* start() const { return base + 1 + R; }
  __device__ int32_t* route() const { return base + 2 + 2 * R; }
};

// ------------------------------------------------------------ 1. groups
// hist[e] routes of expert e -> start offsets (ascending e) and group ids;
// routes scattered by an atomic cursor, then each group's (few) routes sorted.
__global__ void __launch_bounds__(kGT) group_kernel(DevState st, int layer,
                                                    const int32_t* __restrict__ slot_ids, int R,
                                                    Groups gr, int dense_from,
                                                    int32_t* __restrict__ dense) {
  extern __shared__ int gsm[];
  const int E = st.E;
  int* off = gsm;          // [E] routes, then start offset, of expert e
  int* cur = gsm + E;      // [E] scatter cursor
  int* eslot = gsm + 2 * E;  // [E] the slot of expert e
  __shared__ BlockScratch bs;
  const int tid = threadIdx.x;
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int e = tid; e < E; e += kGT) {
    off[e] = 0;
    cur[e] = 0;
  }
  __syncthreads();
  for (int r = tid; r < R; r += kGT) {
    const int s = slot_ids[r];
    if ((unsigned)s >= (unsigned)st.S) continue;
    const int e = st.slot_key[pbase + s] - layer * E;
    if ((unsigned)e >= (unsigned)E) continue;  // not this layer's expert: never produced
    atomicAdd(&off[e], 1);
    eslot[e] = s;  // every route of e has the same slot
  }
  __syncthreads();
  const int ept = (E + kGT - 1) / kGT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int nr = 0, ng = 0, nd = 0;
  for (int e = e0; e < e1; ++e) {
    nr += off[e];
    ng += off[e] > 0;
    nd += dense_from > 0 && off[e] >= dense_from;
  }
  int totR, totG, totD;
  int r0 = block_excl_scan<kGT>(nr, bs, &totR);
  int g0 = block_excl_scan<kGT>(ng, bs, &totG);
  int d0 = block_excl_scan<kGT>(nd, bs, &totD);
  for (int e = e0; e < e1; ++e) {
    const int c = off[e];
    if (c > 0) {
      if (dense && dense_from > 0 && c >= dense_from) dense[1 + d0++] = g0;
      gr.slot()[g0] = eslot[e];
      gr.start()[g0] = r0;
      ++g0;
    }
    off[e] = r0;
    r0 += c;
  }
  if (tid == 0) {
    gr.G() = totG;
    gr.start()[totG] = totR;
    if (dense) dense[0] = totD;
  }
  __syncthreads();
  // scatter in ascending route order, 32 routes at a time by warp 0: lanes of
  // the same expert take consecutive places in lane order
  if (tid < 32) {
    for (int b = 0; b < R; b += 32) {
      const int r = b + tid;
      int e = -1;
      if (r < R) {
        const int s = slot_ids[r];
        if ((unsigned)s < (unsigned)st.S) {
          e = st.slot_key[pbase + s] - layer * E;
          if ((unsigned)e >= (unsigned)E) e = -1;
        }
      }
      const unsigned same = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int rank = __popc(same & ((1u << tid) - 1u));
        gr.route()[off[e] + cur[e] + rank] = r;
      }
      __syncwarp();
      if (e >= 0 && tid == 31 - __clz(same)) cur[e] += __popc(same);  // the set's last lane
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------ 2. x
// NVFP4: f16 x with a per-row power-of-two scale (max |x| < 2^15) and its
// inverse; bf16: a copy.  One CTA per row.
template <int FMT>
__global__ void __launch_bounds__(kWT) xprep_kernel(const uint16_t* __restrict__ x, int H,
                                                    uint16_t* __restrict__ x16,
                                                    float* __restrict__ xinv) {
  __shared__ float s_mx[kWT / 32];
  __shared__ float s_sc;
  const int b = blockIdx.x, tid = threadIdx.x;
  const uint16_t* xr = x + (size_t)b * H;
  if (FMT == MOE_W_BF16) {
    for (int i = tid; i < H; i += kWT) x16[(size_t)b * H + i] = xr[i];
    if (tid == 0) xinv[b] = 1.f;
    return;
  }
  float mx = 0.f;
  for (int i = tid; i < H; i += kWT) mx = fmaxf(mx, fabsf(fp32_of_bf16(xr[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) s_mx[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    float m = 0.f;
    for (int w = 0; w < kWT / 32; ++w) m = fmaxf(m, s_mx[w]);
    float sc = 1.f;  // at most 140 halvings, so an infinite input cannot keep it going
    for (int i = 0; i < 140 && m * sc >= 32768.f; ++i) sc *= 0.5f;
    s_sc = sc;
    xinv[b] = 1.f / sc;
  }
  __syncthreads();
  const float sc = s_sc;
  for (int i = tid; i < H; i += kWT)
    x16[(size_t)b * H + i] = __half_as_ushort(__float2half_rn(fp32_of_bf16(xr[i]) * sc));
}

// ------------------------------------------------------------ 3. gate / up
// Work item (group g, 256 rows of I): every lane owns one row i and computes,
// for up to kNR of the group's routes at a time, the whole gate and up dot
// products -- no cross-lane reduction.  The routes' x rows are staged in
// shared memory and read as broadcasts (every lane of a warp reads the same
// address).  NVFP4 weights are decoded once per 16-element block and applied
// to every staged route with exact half-times-half products, fp32 sums.
constexpr int kRowsItem = kWT;  // rows per work item (one per thread)

template <int FMT>
__global__ void __launch_bounds__(kWT) gup_kernel(DevState st, int H, int I, int layer,
                                                  const uint16_t* __restrict__ x16,
                                                  const float* __restrict__ xinv, int k, Groups gr,
                                                  float* __restrict__ h) {
  extern __shared__ __align__(16) uint4 xs[];  // [kNR][H / 8]
  const int G = gr.G();
  const int nch = (I + kRowsItem - 1) / kRowsItem;
  const int Hu = H / 8;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const int i = ch * kRowsItem + threadIdx.x;
    const bool row_ok = i < I;
    const int ii = row_ok ? i : I - 1;  // rows past I compute nothing that is stored
    float gs0 = 1.f, gs1 = 1.f;
    if (FMT == MOE_W_NVFP4) {
      gs0 = reinterpret_cast<const float*>(blob + o.glob)[0];
      gs1 = reinterpret_cast<const float*>(blob + o.glob)[1];
    }
    for (int q0 = ra; q0 < rb; q0 += kNR) {  // up to kNR routes per pass
      const int nq = min(kNR, rb - q0);
      __syncthreads();  // the previous pass's x no longer read
      for (int v = threadIdx.x; v < nq * Hu; v += kWT) {
        const int j = v / Hu, un = v - j * Hu;
        const int b = gr.route()[q0 + j] / k;
        xs[v] = reinterpret_cast<const uint4*>(x16 + (size_t)b * H)[un];
      }
      __syncthreads();
      float ga[kNR] = {0.f, 0.f, 0.f, 0.f}, ua[kNR] = {0.f, 0.f, 0.f, 0.f};
      if (FMT == MOE_W_NVFP4) {
        const uint8_t* gc = blob + o.code[0] + (size_t)ii * (H / 2);
        const uint8_t* uc = blob + o.code[1] + (size_t)ii * (H / 2);
        const uint8_t* gsc = blob + o.scale[0] + (size_t)ii * (H / 16);
        const uint8_t* usc = blob + o.scale[1] + (size_t)ii * (H / 16);
        // two 16-element blocks per step; the next step's words are in flight
        uint4 gwn = *reinterpret_cast<const uint4*>(gc), uwn = *reinterpret_cast<const uint4*>(uc);
        uint32_t sgn = *reinterpret_cast<const uint16_t*>(gsc), sun = *reinterpret_cast<const uint16_t*>(usc);
        for (int blk = 0; blk < H / 16; blk += 2) {
          const uint4 gw = gwn, uw = uwn;
          const float2 sg = e4m3x2(sgn), su = e4m3x2(sun);
          if (blk + 2 < H / 16) {
            gwn = *reinterpret_cast<const uint4*>(gc + (blk + 2) * 8);
            uwn = *reinterpret_cast<const uint4*>(uc + (blk + 2) * 8);
            sgn = *reinterpret_cast<const uint16_t*>(gsc + blk + 2);
            sun = *reinterpret_cast<const uint16_t*>(usc + blk + 2);
          }
          const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w}, uv[4] = {uw.x, uw.y, uw.z, uw.w};
          uint32_t gd[16], ud[16];
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            gd[4 * wd] = e2m1x2<0>(gv[wd]);
            gd[4 * wd + 1] = e2m1x2<1>(gv[wd]);
            gd[4 * wd + 2] = e2m1x2<2>(gv[wd]);
            gd[4 * wd + 3] = e2m1x2<3>(gv[wd]);
            ud[4 * wd] = e2m1x2<0>(uv[wd]);
            ud[4 * wd + 1] = e2m1x2<1>(uv[wd]);
            ud[4 * wd + 2] = e2m1x2<2>(uv[wd]);
            ud[4 * wd + 3] = e2m1x2<3>(uv[wd]);
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const uint4* xr = xs + (size_t)j * Hu + blk * 2;  // 32 elements = 4 units
            const uint4 x0 = xr[0], x1 = xr[1], x2 = xr[2], x3 = xr[3];
            const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                     x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            float p = 0.f, q = 0.f, p2 = 0.f, q2 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              p = fma2h(gd[e], xv[e], p);
              q = fma2h(ud[e], xv[e], q);
              p2 = fma2h(gd[8 + e], xv[8 + e], p2);
              q2 = fma2h(ud[8 + e], xv[8 + e], q2);
            }
            ga[j] = fmaf(p, sg.x, fmaf(p2, sg.y, ga[j]));
            ua[j] = fmaf(q, su.x, fmaf(q2, su.y, ua[j]));
          }
        }
      } else if (FMT == MOE_W_MXFP4 || FMT == MOE_W_Q4_0) {
        // 32-element blocks: codes decoded once, applied to every staged route
        const Off of(H, I, FMT);
        const int sbr = (H / 32) * (FMT == MOE_W_Q4_0 ? 2 : 1);  // scale bytes per row
        const uint8_t* gc = blob + of.code[0] + (size_t)ii * (H / 2);
        const uint8_t* uc = blob + of.code[1] + (size_t)ii * (H / 2);
        const uint8_t* gsc = blob + of.scale[0] + (size_t)ii * sbr;
        const uint8_t* usc = blob + of.scale[1] + (size_t)ii * sbr;
#pragma unroll 2
        for (int blk = 0; blk < H / 32; ++blk) {
          const uint4 gw = *reinterpret_cast<const uint4*>(gc + blk * 16);
          const uint4 uw = *reinterpret_cast<const uint4*>(uc + blk * 16);
          const float sg = blk32_scale<FMT>(gsc, blk), su = blk32_scale<FMT>(usc, blk);
          uint32_t gd[16], ud[16];
          blk32_decode<FMT>(gw, gd);
          blk32_decode<FMT>(uw, ud);
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const uint4* xr = xs + (size_t)j * Hu + blk * 4;  // 32 elements = 4 units
            const uint4 x0 = xr[0], x1 = xr[1], x2 = xr[2], x3 = xr[3];
            const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                     x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            float p = 0.f, q = 0.f, p2 = 0.f, q2 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              p = fma2h(gd[e], xv[e], p);
              q = fma2h(ud[e], xv[e], q);
              p2 = fma2h(gd[8 + e], xv[8 + e], p2);
              q2 = fma2h(ud[8 + e], xv[8 + e], q2);
            }
            ga[j] = fmaf(p + p2, sg, ga[j]);
            ua[j] = fmaf(q + q2, su, ua[j]);
          }
        }
      } else {
        const uint8_t* gm = blob + o.mat[0] + (size_t)ii * H * 2;
        const uint8_t* um = blob + o.mat[1] + (size_t)ii * H * 2;
        for (int un = 0; un < Hu; ++un) {  // 8 elements per step
          const uint4 gw = *reinterpret_cast<const uint4*>(gm + un * 16);
          const uint4 uw = *reinterpret_cast<const uint4*>(um + un * 16);
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const uint4 xv = xs[(size_t)j * Hu + un];
            ga[j] = fma2b(gw.w, xv.w, fma2b(gw.z, xv.z, fma2b(gw.y, xv.y, fma2b(gw.x, xv.x, ga[j]))));
            ua[j] = fma2b(uw.w, xv.w, fma2b(uw.z, xv.z, fma2b(uw.y, xv.y, fma2b(uw.x, xv.x, ua[j]))));
          }
        }
      }
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < kNR; ++j) {
          if (j >= nq) break;
          const int r = gr.route()[q0 + j];
          const float xi = xinv[r / k];
          const float gg = ga[j] * xi * gs0, uu = ua[j] * xi * gs1;
          h[(size_t)r * I + i] = gg / (1.f + expf(-gg)) * uu;
        }
      }
    }
  }
}

// ------------------------------------------------------------ 3b. gate / up, staged
// The NVFP4 gate/up kernel for H a multiple of 64, with the same arithmetic as
// gup_kernel (so the same bits) but a different data path: a work item's 256
// weight rows are streamed through shared memory in stages of 64 elements
// (32 code bytes and 4 scale bytes per row and matrix), kNS stages in flight
// with cp.async.  The copies are coalesced -- two lanes per row, 16 rows per
// warp instruction, whole 32-byte sectors -- where one-row-per-thread global
// loads touch 32 lines per instruction.  Each thread then reads its own row
// from shared memory; the two 16-byte halves of a row's 32 code bytes are
// swapped on every other group of four rows, so a quarter-warp's 16-byte
// reads fall on eight distinct bank groups.
constexpr int kNS = 4;                    // stages in flight
constexpr int kStC = 32 * kRowsItem;      // code bytes per matrix per stage
constexpr int kStS = 4 * kRowsItem;       // scale bytes per matrix per stage

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_stages() {  // all but the kNS - 2 newest groups landed
  asm volatile("cp.async.wait_group %0;" ::"n"(kNS - 2) : "memory");
}
// the 16-byte half c of row r's 32 code bytes within a stage
__device__ __forceinline__ int half_at(int r, int c) { return r * 32 + ((c ^ (r >> 2)) & 1) * 16; }

// Stage s of one matrix's rows [r0, r0 + 256) (clamped to n_rows - 1): codes
// (row stride cb bytes) at dc, scales (row stride sb) at ds.
__device__ __forceinline__ void stage_rows(uint8_t* dc, uint8_t* ds, const uint8_t* codes,
                                           const uint8_t* scales, int r0, int n_rows, int cb,
                                           int sb, int s) {
  const int t = threadIdx.x;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int rr = (t >> 1) + (kRowsItem / 2) * u, c = t & 1;
    const int row = min(r0 + rr, n_rows - 1);
    cp16(dc + half_at(rr, c), codes + (size_t)row * cb + s * 32 + c * 16);
  }
  const int row = min(r0 + t, n_rows - 1);
  cp4(ds + t * 4, scales + (size_t)row * sb + s * 4);
}

__global__ void __launch_bounds__(kWT, 2) gup_staged_kernel(DevState st, int H, int I, int layer,
                                                            const uint16_t* __restrict__ x16,
                                                            const float* __restrict__ xinv,
                                                            int k, Groups gr,
                                                            float* __restrict__ h, int skip_from) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint4* xs = reinterpret_cast<uint4*>(dsm);  // [kNR][H / 8]
  uint8_t* stg = dsm + (size_t)kNR * H * 2;   // [kNS][gate codes | up codes | gate sc | up sc]
  constexpr int kStage = 2 * kStC + 2 * kStS;
  const int G = gr.G();
  const int nch = (I + kRowsItem - 1) / kRowsItem;
  const int Hu = H / 8, nst = H / 64;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  const int t = threadIdx.x;
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    if (skip_from > 0 && rb - ra >= skip_from) continue;  // a dense group: the tensor cores take it
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const int i0 = ch * kRowsItem, i = i0 + t;
    const float gs0 = reinterpret_cast<const float*>(blob + o.glob)[0];
    const float gs1 = reinterpret_cast<const float*>(blob + o.glob)[1];
    auto issue = [&](int s) {
      uint8_t* b = stg + (s % kNS) * kStage;
      stage_rows(b, b + 2 * kStC, blob + o.code[0], blob + o.scale[0], i0, I, H / 2, H / 16, s);
      stage_rows(b + kStC, b + 2 * kStC + kStS, blob + o.code[1], blob + o.scale[1], i0, I, H / 2,
                 H / 16, s);
    };
    for (int q0 = ra; q0 < rb; q0 += kNR) {  // up to kNR routes per pass
      const int nq = min(kNR, rb - q0);
      __syncthreads();  // the previous pass's x and stages no longer read
      for (int v = t; v < nq * Hu; v += kWT) {
        const int j = v / Hu, un = v - j * Hu;
        const int b = gr.route()[q0 + j] / k;
        xs[v] = reinterpret_cast<const uint4*>(x16 + (size_t)b * H)[un];
      }
#pragma unroll
      for (int s = 0; s < kNS - 1; ++s) {
        if (s < nst) issue(s);
        cp_commit();
      }
      float ga[kNR] = {0.f, 0.f, 0.f, 0.f}, ua[kNR] = {0.f, 0.f, 0.f, 0.f};
      for (int s = 0; s < nst; ++s) {
        cp_wait_stages();
        __syncthreads();  // stage s (and, at s = 0, x) visible; stage s - 1 no longer read
        if (s + kNS - 1 < nst) issue(s + kNS - 1);
        cp_commit();
        const uint8_t* b = stg + (s % kNS) * kStage;
        const uint32_t sgw = *reinterpret_cast<const uint32_t*>(b + 2 * kStC + t * 4);
        const uint32_t suw = *reinterpret_cast<const uint32_t*>(b + 2 * kStC + kStS + t * 4);
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // the stage's two block pairs
          const uint4 gw = *reinterpret_cast<const uint4*>(b + half_at(t, c));
          const uint4 uw = *reinterpret_cast<const uint4*>(b + kStC + half_at(t, c));
          const float2 sg = e4m3x2(c ? sgw >> 16 : sgw & 0xffffu);
          const float2 su = e4m3x2(c ? suw >> 16 : suw & 0xffffu);
          const int blk = 4 * s + 2 * c;
          const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w}, uv[4] = {uw.x, uw.y, uw.z, uw.w};
          uint32_t gd[16], ud[16];
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            gd[4 * wd] = e2m1x2<0>(gv[wd]);
            gd[4 * wd + 1] = e2m1x2<1>(gv[wd]);
            gd[4 * wd + 2] = e2m1x2<2>(gv[wd]);
            gd[4 * wd + 3] = e2m1x2<3>(gv[wd]);
            ud[4 * wd] = e2m1x2<0>(uv[wd]);
            ud[4 * wd + 1] = e2m1x2<1>(uv[wd]);
            ud[4 * wd + 2] = e2m1x2<2>(uv[wd]);
            ud[4 * wd + 3] = e2m1x2<3>(uv[wd]);
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const uint4* xr = xs + (size_t)j * Hu + blk * 2;  // 32 elements = 4 units
            const uint4 x0 = xr[0], x1 = xr[1], x2 = xr[2], x3 = xr[3];
            const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                     x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            float p = 0.f, q = 0.f, p2 = 0.f, q2 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              p = fma2h(gd[e], xv[e], p);
              q = fma2h(ud[e], xv[e], q);
              p2 = fma2h(gd[8 + e], xv[8 + e], p2);
              q2 = fma2h(ud[8 + e], xv[8 + e], q2);
            }
            ga[j] = fmaf(p, sg.x, fmaf(p2, sg.y, ga[j]));
            ua[j] = fmaf(q, su.x, fmaf(q2, su.y, ua[j]));
          }
        }
      }
      if (i < I) {
#pragma unroll
        for (int j = 0; j < kNR; ++j) {
          if (j >= nq) break;
          const int r = gr.route()[q0 + j];
          const float xi = xinv[r / k];
          const float gg = ga[j] * xi * gs0, uu = ua[j] * xi * gs1;
          h[(size_t)r * I + i] = gg / (1.f + expf(-gg)) * uu;
        }
      }
    }
  }
}

// ------------------------------------------------------------ 3c. gate / up, warp rows
// The NVFP4 gate/up kernel for H = 1024 JH and I a multiple of kWB, with no
// operand in shared memory.  A warp takes kWB consecutive rows of one group at
// a time (units dealt over the grid's warps group-major, so neighbouring warps
// stream neighbouring rows).  Lane L holds the 16-byte code chunks L, L + 32,
// ... of each row (32 elements each, so every warp load is 512 contiguous
// bytes, and its two block scales as one 16-bit load) and the same elements of
// NQ routes' x in registers, loaded once per unit and pass; the routes left
// after the full passes go one at a time.  Per row the lane decodes each chunk
// once, sums each 16-element block's exact half-times-half products in fp32,
// scales the block sums, and the warp reduces the lanes' gate and up sums of
// every route with shuffles.  The next row's codes are in flight while a row
// computes.
constexpr int kWB = 8;   // rows per warp unit
constexpr int kPfAhead = 3;  // rows (steps) ahead that the warp-row kernels ask L2 to fetch

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// the warp totals of g[q], u[q] (q < NQ): lane 16 q holds route q's gate total
// in gt and its up total in ut
template <int NQ>
__device__ __forceinline__ void warp_gu_totals(const float (&g)[NQ], const float (&u)[NQ],
                                               int lane, float& gt, float& ut) {
  const bool h16 = lane & 16;
  float v;
  if (NQ == 1) {  // lanes < 16 keep g, lanes >= 16 keep u
    v = (h16 ? u[0] : g[0]) + __shfl_xor_sync(0xffffffffu, h16 ? g[0] : u[0], 16);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
  } else {  // lanes < 16 keep route 0, lanes >= 16 route 1; then bit 3 picks g or u
    const float k0 = (h16 ? g[NQ - 1] : g[0]) + __shfl_xor_sync(0xffffffffu, h16 ? g[0] : g[NQ - 1], 16);
    const float k1 = (h16 ? u[NQ - 1] : u[0]) + __shfl_xor_sync(0xffffffffu, h16 ? u[0] : u[NQ - 1], 16);
    const bool h8 = lane & 8;
    v = (h8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
  }
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  gt = v;
  ut = __shfl_xor_sync(0xffffffffu, v, NQ == 1 ? 16 : 8);
}

// one pass of a warp unit over NR routes (rt): kWB rows from row i0 of the
// group's expert (code chunk 0 of row 0 of each bank at gc, uc; scales at gsc, usc)
template <int JH, int NR>
__device__ __forceinline__ void gup_warp_pass(const uint8_t* gc, const uint8_t* uc,
                                              const uint8_t* gsc, const uint8_t* usc,
                                              const uint16_t* __restrict__ x16,
                                              const float* __restrict__ xinv, int k,
                                              const int (&rt)[NR], float gs0, float gs1, int I,
                                              int i0, int lane, float* __restrict__ h) {
  constexpr int H = 1024 * JH;
  // the lane's elements of each route's x
  uint32_t xv[NR][JH][16];
#pragma unroll
  for (int q = 0; q < NR; ++q) {
    const uint4* xp = reinterpret_cast<const uint4*>(x16 + (size_t)(rt[q] / k) * H);
#pragma unroll
    for (int j = 0; j < JH; ++j)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 t = __ldg(xp + (lane + 32 * j) * 4 + v);
        xv[q][j][4 * v] = t.x, xv[q][j][4 * v + 1] = t.y;
        xv[q][j][4 * v + 2] = t.z, xv[q][j][4 * v + 3] = t.w;
      }
  }
  uint4 cg[JH], cu[JH];
  uint32_t sg[JH], su[JH];
  auto load_row = [&](int r, uint4 (&a)[JH], uint4 (&b)[JH], uint32_t (&sa)[JH],
                      uint32_t (&sb)[JH]) {
#pragma unroll
    for (int j = 0; j < JH; ++j) {
      a[j] = __ldcs(reinterpret_cast<const uint4*>(gc + (size_t)r * (H / 2) + 512 * j));
      b[j] = __ldcs(reinterpret_cast<const uint4*>(uc + (size_t)r * (H / 2) + 512 * j));
      sa[j] = __ldcs(reinterpret_cast<const unsigned short*>(gsc + (size_t)r * (H / 16) + 64 * j));
      sb[j] = __ldcs(reinterpret_cast<const unsigned short*>(usc + (size_t)r * (H / 16) + 64 * j));
    }
  };
  auto prefetch_row = [&](int r) {  // into L2, kPfAhead rows before the row's loads
#pragma unroll
    for (int j = 0; j < JH; ++j) {
      prefetch_l2(gc + (size_t)r * (H / 2) + 512 * j);
      prefetch_l2(uc + (size_t)r * (H / 2) + 512 * j);
    }
    prefetch_l2(gsc + (size_t)r * (H / 16));
    prefetch_l2(usc + (size_t)r * (H / 16));
  };
#pragma unroll
  for (int r = 1; r < kPfAhead; ++r) prefetch_row(r);
  load_row(0, cg, cu, sg, su);
#pragma unroll 1
  for (int r = 0; r < kWB; ++r) {
    if (r + kPfAhead < kWB) prefetch_row(r + kPfAhead);
    uint4 ng[JH], nu[JH];
    uint32_t nsg[JH], nsu[JH];
    load_row(min(r + 1, kWB - 1), ng, nu, nsg, nsu);  // the next row in flight
    float ga[NR], ua[NR];
#pragma unroll
    for (int q = 0; q < NR; ++q) ga[q] = ua[q] = 0.f;
#pragma unroll
    for (int j = 0; j < JH; ++j) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {  // gate, then up
        const uint4 c = m ? cu[j] : cg[j];
        const float2 s = e4m3x2(m ? su[j] : sg[j]);
        const uint32_t cv[4] = {c.x, c.y, c.z, c.w};
        uint32_t d[16];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          d[4 * wd] = e2m1x2<0>(cv[wd]);
          d[4 * wd + 1] = e2m1x2<1>(cv[wd]);
          d[4 * wd + 2] = e2m1x2<2>(cv[wd]);
          d[4 * wd + 3] = e2m1x2<3>(cv[wd]);
        }
#pragma unroll
        for (int q = 0; q < NR; ++q) {
          float p = 0.f, p2 = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p = fma2h(d[e], xv[q][j][e], p);
            p2 = fma2h(d[8 + e], xv[q][j][8 + e], p2);
          }
          float& acc = m ? ua[q] : ga[q];
          acc = fmaf(p2, s.y, fmaf(p, s.x, acc));
        }
      }
    }
    float gt, ut;
    warp_gu_totals<NR>(ga, ua, lane, gt, ut);
    const int q = lane >> 4;
    if ((lane & 15) == 0 && q < NR) {
      const int rq = rt[NR == 1 ? 0 : q];
      const float xi = xinv[rq / k];
      const float gg = gt * xi * gs0, uu = ut * xi * gs1;
      h[(size_t)rq * I + i0 + r] = gg / (1.f + expf(-gg)) * uu;
    }
#pragma unroll
    for (int j = 0; j < JH; ++j) cg[j] = ng[j], cu[j] = nu[j], sg[j] = nsg[j], su[j] = nsu[j];
  }
}

template <int JH, int NQ>
__global__ void __launch_bounds__(kWT, 2) gup_warp_kernel(DevState st, int I, int layer,
                                                          const uint16_t* __restrict__ x16,
                                                          const float* __restrict__ xinv, int k,
                                                          Groups gr, float* __restrict__ h,
                                                          int skip_from) {
  constexpr int H = 1024 * JH;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kWT / 32) + (threadIdx.x >> 5), Gw = gridDim.x * (kWT / 32);
  const int G = gr.G(), nb = I / kWB;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int un = gw; un < G * nb; un += Gw) {
    const int g = un / nb, i0 = (un - g * nb) * kWB;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    if (skip_from > 0 && rb - ra >= skip_from) continue;  // a dense group: the tensor cores take it
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const float gs0 = reinterpret_cast<const float*>(blob + o.glob)[0];
    const float gs1 = reinterpret_cast<const float*>(blob + o.glob)[1];
    // this lane's chunk 0 of row i0 in each bank (chunk j is 512 j bytes on)
    const uint8_t* gc = blob + o.code[0] + (size_t)i0 * (H / 2) + lane * 16;
    const uint8_t* uc = blob + o.code[1] + (size_t)i0 * (H / 2) + lane * 16;
    const uint8_t* gsc = blob + o.scale[0] + (size_t)i0 * (H / 16) + lane * 2;
    const uint8_t* usc = blob + o.scale[1] + (size_t)i0 * (H / 16) + lane * 2;
    int q0 = ra;
    for (; NQ > 1 && q0 + NQ <= rb; q0 += NQ) {  // full passes
      int rt[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) rt[q] = gr.route()[q0 + q];
      gup_warp_pass<JH, NQ>(gc, uc, gsc, usc, x16, xinv, k, rt, gs0, gs1, I, i0, lane, h);
    }
    for (; q0 < rb; ++q0) {  // the rest one route at a time
      const int rt[1] = {gr.route()[q0]};
      gup_warp_pass<JH, 1>(gc, uc, gsc, usc, x16, xinv, k, rt, gs0, gs1, I, i0, lane, h);
    }
  }
}

// ------------------------------------------------------------ 4. down
// Work item (group g, 256 rows of H): every lane owns one output row n and
// computes its whole dot product with the h of up to kNR of the group's
// routes, staged in shared memory (broadcast reads).  NVFP4 blocks of 16 are
// decoded once and applied to every staged route in fp32.
template <int FMT>
__global__ void __launch_bounds__(kWT) gdown_kernel(DevState st, int H, int I, int layer,
                                                    Groups gr, const float* __restrict__ h,
                                                    float* __restrict__ y) {
  extern __shared__ __align__(16) float hsm[];  // [kNR][I]
  const int G = gr.G();
  const int nch = (H + kRowsItem - 1) / kRowsItem;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const float gs2 = FMT == MOE_W_NVFP4 ? reinterpret_cast<const float*>(blob + o.glob)[2] : 1.f;
    const int n = ch * kRowsItem + threadIdx.x;
    const bool row_ok = n < H;
    const int nn = row_ok ? n : H - 1;
    for (int q0 = ra; q0 < rb; q0 += kNR) {
      const int nq = min(kNR, rb - q0);
      __syncthreads();
      for (int v = threadIdx.x; v < nq * I / 4; v += kWT) {
        const int j = v / (I / 4), f = v - j * (I / 4);
        reinterpret_cast<float4*>(hsm)[v] =
            __ldcg(reinterpret_cast<const float4*>(h + (size_t)gr.route()[q0 + j] * I) + f);
      }
      __syncthreads();
      float acc[kNR] = {0.f, 0.f, 0.f, 0.f};
      if (FMT == MOE_W_NVFP4) {
        const uint8_t* dc = blob + o.code[2] + (size_t)nn * (I / 2);
        const uint8_t* ds = blob + o.scale[2] + (size_t)nn * (I / 16);
        // two blocks per step; the next step's words are in flight
        uint4 cwn = *reinterpret_cast<const uint4*>(dc);
        uint32_t scn = *reinterpret_cast<const uint16_t*>(ds);
        for (int blk = 0; blk < I / 16; blk += 2) {
          const uint4 cw = cwn;
          const float2 sc = e4m3x2(scn);
          if (blk + 2 < I / 16) {
            cwn = *reinterpret_cast<const uint4*>(dc + (blk + 2) * 8);
            scn = *reinterpret_cast<const uint16_t*>(ds + blk + 2);
          }
          const uint32_t ww[4] = {cw.x, cw.y, cw.z, cw.w};
          float wf[32];
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            const float2 a0 = f16x2_f32(e2m1x2<0>(ww[wd])), a1 = f16x2_f32(e2m1x2<1>(ww[wd]));
            const float2 a2 = f16x2_f32(e2m1x2<2>(ww[wd])), a3 = f16x2_f32(e2m1x2<3>(ww[wd]));
            wf[8 * wd] = a0.x, wf[8 * wd + 1] = a0.y, wf[8 * wd + 2] = a1.x, wf[8 * wd + 3] = a1.y;
            wf[8 * wd + 4] = a2.x, wf[8 * wd + 5] = a2.y, wf[8 * wd + 6] = a3.x, wf[8 * wd + 7] = a3.y;
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)j * I + blk * 16);
            float p = 0.f, p2 = 0.f;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 hv = hp[e4], hv2 = hp[4 + e4];
              p = fmaf(wf[4 * e4], hv.x, p);
              p = fmaf(wf[4 * e4 + 1], hv.y, p);
              p = fmaf(wf[4 * e4 + 2], hv.z, p);
              p = fmaf(wf[4 * e4 + 3], hv.w, p);
              p2 = fmaf(wf[16 + 4 * e4], hv2.x, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 1], hv2.y, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 2], hv2.z, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 3], hv2.w, p2);
            }
            acc[j] = fmaf(p, sc.x, fmaf(p2, sc.y, acc[j]));
          }
        }
      } else if (FMT == MOE_W_MXFP4 || FMT == MOE_W_Q4_0) {
        const Off of(H, I, FMT);
        const int sbr = (I / 32) * (FMT == MOE_W_Q4_0 ? 2 : 1);  // scale bytes per row
        const uint8_t* dc = blob + of.code[2] + (size_t)nn * (I / 2);
        const uint8_t* ds = blob + of.scale[2] + (size_t)nn * sbr;
#pragma unroll 2
        for (int blk = 0; blk < I / 32; ++blk) {
          const uint4 cw = *reinterpret_cast<const uint4*>(dc + blk * 16);
          const float sc = blk32_scale<FMT>(ds, blk);
          uint32_t d2[16];
          blk32_decode<FMT>(cw, d2);
          float wf[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 f = f16x2_f32(d2[e]);
            wf[2 * e] = f.x, wf[2 * e + 1] = f.y;
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)j * I + blk * 32);
            float p = 0.f, p2 = 0.f;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 hv = hp[e4], hv2 = hp[4 + e4];
              p = fmaf(wf[4 * e4], hv.x, p);
              p = fmaf(wf[4 * e4 + 1], hv.y, p);
              p = fmaf(wf[4 * e4 + 2], hv.z, p);
              p = fmaf(wf[4 * e4 + 3], hv.w, p);
              p2 = fmaf(wf[16 + 4 * e4], hv2.x, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 1], hv2.y, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 2], hv2.z, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 3], hv2.w, p2);
            }
            acc[j] = fmaf(p + p2, sc, acc[j]);
          }
        }
      } else {
        const uint8_t* dm = blob + o.mat[2] + (size_t)nn * I * 2;
        for (int wd = 0; wd < I / 8; ++wd) {
          const uint4 v = *reinterpret_cast<const uint4*>(dm + wd * 16);
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)j * I + wd * 8);
            const float4 h0 = hp[0], h1 = hp[1];
            const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[j] = fmaf(fp32_of_bf16(vv[e] & 0xffffu), hv[2 * e], acc[j]);
              acc[j] = fmaf(__uint_as_float(vv[e] & 0xffff0000u), hv[2 * e + 1], acc[j]);
            }
          }
        }
      }
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < kNR; ++j) {
          if (j >= nq) break;
          y[(size_t)gr.route()[q0 + j] * H + n] = acc[j] * gs2;
        }
      }
    }
  }
}

// ------------------------------------------------------------ 4b. down, staged
// The NVFP4 down kernel for I a multiple of 64: gdown_kernel's arithmetic
// over rows streamed through shared memory as in gup_staged_kernel.
__global__ void __launch_bounds__(kWT, 2) gdown_staged_kernel(DevState st, int H, int I,
                                                              int layer, Groups gr,
                                                              const float* __restrict__ h,
                                                              float* __restrict__ y, int skip_from) {
  extern __shared__ __align__(16) uint8_t dsm[];
  float* hsm = reinterpret_cast<float*>(dsm);  // [kNR][I]
  uint8_t* stg = dsm + (size_t)kNR * I * 4;    // [kNS][codes | scales]
  constexpr int kStage = kStC + kStS;
  const int G = gr.G();
  const int nch = (H + kRowsItem - 1) / kRowsItem;
  const int nst = I / 64;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  const int t = threadIdx.x;
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    if (skip_from > 0 && rb - ra >= skip_from) continue;  // a dense group: the tensor cores take it
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const float gs2 = reinterpret_cast<const float*>(blob + o.glob)[2];
    const int n0 = ch * kRowsItem, n = n0 + t;
    auto issue = [&](int s) {
      uint8_t* b = stg + (s % kNS) * kStage;
      stage_rows(b, b + kStC, blob + o.code[2], blob + o.scale[2], n0, H, I / 2, I / 16, s);
    };
    for (int q0 = ra; q0 < rb; q0 += kNR) {
      const int nq = min(kNR, rb - q0);
      __syncthreads();
      for (int v = t; v < nq * I / 4; v += kWT) {
        const int j = v / (I / 4), f = v - j * (I / 4);
        reinterpret_cast<float4*>(hsm)[v] =
            __ldcg(reinterpret_cast<const float4*>(h + (size_t)gr.route()[q0 + j] * I) + f);
      }
#pragma unroll
      for (int s = 0; s < kNS - 1; ++s) {
        if (s < nst) issue(s);
        cp_commit();
      }
      float acc[kNR] = {0.f, 0.f, 0.f, 0.f};
      for (int s = 0; s < nst; ++s) {
        cp_wait_stages();
        __syncthreads();
        if (s + kNS - 1 < nst) issue(s + kNS - 1);
        cp_commit();
        const uint8_t* b = stg + (s % kNS) * kStage;
        const uint32_t scw = *reinterpret_cast<const uint32_t*>(b + kStC + t * 4);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 cw = *reinterpret_cast<const uint4*>(b + half_at(t, c));
          const float2 sc = e4m3x2(c ? scw >> 16 : scw & 0xffffu);
          const int blk = 4 * s + 2 * c;
          const uint32_t ww[4] = {cw.x, cw.y, cw.z, cw.w};
          float wf[32];
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            const float2 a0 = f16x2_f32(e2m1x2<0>(ww[wd])), a1 = f16x2_f32(e2m1x2<1>(ww[wd]));
            const float2 a2 = f16x2_f32(e2m1x2<2>(ww[wd])), a3 = f16x2_f32(e2m1x2<3>(ww[wd]));
            wf[8 * wd] = a0.x, wf[8 * wd + 1] = a0.y, wf[8 * wd + 2] = a1.x, wf[8 * wd + 3] = a1.y;
            wf[8 * wd + 4] = a2.x, wf[8 * wd + 5] = a2.y, wf[8 * wd + 6] = a3.x, wf[8 * wd + 7] = a3.y;
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) {
            if (j >= nq) break;
            const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)j * I + blk * 16);
            float p = 0.f, p2 = 0.f;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 hv = hp[e4], hv2 = hp[4 + e4];
              p = fmaf(wf[4 * e4], hv.x, p);
              p = fmaf(wf[4 * e4 + 1], hv.y, p);
              p = fmaf(wf[4 * e4 + 2], hv.z, p);
              p = fmaf(wf[4 * e4 + 3], hv.w, p);
              p2 = fmaf(wf[16 + 4 * e4], hv2.x, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 1], hv2.y, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 2], hv2.z, p2);
              p2 = fmaf(wf[16 + 4 * e4 + 3], hv2.w, p2);
            }
            acc[j] = fmaf(p, sc.x, fmaf(p2, sc.y, acc[j]));
          }
        }
      }
      if (n < H) {
#pragma unroll
        for (int j = 0; j < kNR; ++j) {
          if (j >= nq) break;
          y[(size_t)gr.route()[q0 + j] * H + n] = acc[j] * gs2;
        }
      }
    }
  }
}

// ------------------------------------------------------------ 4c. down, warp rows
// The NVFP4 down kernel for I = 256 M (M = 1 .. 4), with no operand in shared
// memory.  A warp takes kWD consecutive output rows of one group at a time
// (units dealt as in gup_warp_kernel), 8 / NR rows per step.  Lane L holds
// elements [8ML, 8ML + 8M) of each row (M code words: the warp's M loads
// cover the row's I / 2 bytes) and its one or two block scales, and the same
// elements of NR routes' h in registers.  Each 8-element half block's exact
// e2m1 * h products are summed in fp32 and scaled by the block's e4m3 scale;
// a step's 8 (row, route) lane sums are then reduced across the warp together,
// each shuffle level halving the values a lane keeps.  The next step's rows
// are in flight while a step computes.
constexpr int kWD = 32;  // output rows per warp unit

// the warp totals of v[0 .. NV), NV = 4 or 8: lane L ends with the total of
// value L / (32 / NV)
template <int NV>
__device__ __forceinline__ float warp_sum_scatter(float (&v)[NV], int lane) {
  static_assert(NV == 4 || NV == 8, "four or eight values");
  constexpr int kLv = NV == 8 ? 3 : 2;  // levels at which a lane gives away half its values
#pragma unroll
  for (int l = 0; l < kLv; ++l) {
    const int s = 16 >> l, half = NV >> (l + 1);
    const bool up = lane & s;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? v[i + half] : v[i], send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  float t = v[0];
#pragma unroll
  for (int s = 16 >> kLv; s > 0; s >>= 1) t += __shfl_xor_sync(0xffffffffu, t, s);
  return t;
}

// one pass of a warp unit over NR routes (rt): kWD rows from output row n0
// (this lane's code word 0 of row n0 at cw0, the row's scales at sc0)
template <int M, int NR>
__device__ __forceinline__ void gdown_warp_pass(const uint8_t* cw0, const uint8_t* sc0,
                                                const float* __restrict__ h, const int (&rt)[NR],
                                                float gs2, int H, int n0, int lane,
                                                float* __restrict__ y) {
  constexpr int I = 256 * M, RG = 8 / NR;
  float hv[NR][8 * M];
#pragma unroll
  for (int q = 0; q < NR; ++q) {
    const float4* hp = reinterpret_cast<const float4*>(h + (size_t)rt[q] * I + 8 * M * lane);
#pragma unroll
    for (int v = 0; v < 2 * M; ++v) {
      const float4 t = __ldcg(hp + v);
      hv[q][4 * v] = t.x, hv[q][4 * v + 1] = t.y, hv[q][4 * v + 2] = t.z, hv[q][4 * v + 3] = t.w;
    }
  }
  // the lane's half blocks M L + t (t < M) lie in blocks b0 and, if `two`, b0 + 1
  const int b0 = (M * lane) >> 1;
  const bool two = ((M * lane + M - 1) >> 1) != b0;
  auto load_step = [&](int r0, uint32_t (&cw)[RG][M], uint32_t (&sc)[RG]) {
#pragma unroll
    for (int rr = 0; rr < RG; ++rr) {
      const uint32_t* cr = reinterpret_cast<const uint32_t*>(cw0 + (size_t)(r0 + rr) * (I / 2));
#pragma unroll
      for (int t = 0; t < M; ++t) cw[rr][t] = __ldcs(cr + t);
      const unsigned char* sr = sc0 + (size_t)(r0 + rr) * (I / 16) + b0;
      sc[rr] = __ldcs(sr) | (two ? (uint32_t)__ldcs(sr + 1) << 8 : 0u);
    }
  };
  auto prefetch_step = [&](int r0) {  // into L2, kPfAhead steps before the step's loads
#pragma unroll
    for (int rr = 0; rr < RG; ++rr) {
      prefetch_l2(cw0 + (size_t)(r0 + rr) * (I / 2));
      prefetch_l2(sc0 + (size_t)(r0 + rr) * (I / 16) + b0);
    }
  };
#pragma unroll
  for (int k = 1; k < kPfAhead; ++k)
    if (k * RG < kWD) prefetch_step(k * RG);
  uint32_t cw[RG][M], sc[RG];
  load_step(0, cw, sc);
#pragma unroll 1
  for (int r0 = 0; r0 < kWD; r0 += RG) {
    if (r0 + kPfAhead * RG < kWD) prefetch_step(r0 + kPfAhead * RG);
    uint32_t ncw[RG][M], nsc[RG];
    load_step(min(r0 + RG, kWD - RG), ncw, nsc);  // the next step's rows in flight
    float acc[8];
#pragma unroll
    for (int rr = 0; rr < RG; ++rr) {
      const float2 s = e4m3x2(sc[rr]);
      float a[NR];
#pragma unroll
      for (int q = 0; q < NR; ++q) a[q] = 0.f;
#pragma unroll
      for (int t = 0; t < M; ++t) {
        const float st = ((M * lane + t) >> 1) == b0 ? s.x : s.y;
        float wf[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float2 f = f16x2_f32(b == 0   ? e2m1x2<0>(cw[rr][t])
                                     : b == 1 ? e2m1x2<1>(cw[rr][t])
                                     : b == 2 ? e2m1x2<2>(cw[rr][t])
                                              : e2m1x2<3>(cw[rr][t]));
          wf[2 * b] = f.x, wf[2 * b + 1] = f.y;
        }
#pragma unroll
        for (int q = 0; q < NR; ++q) {
          float p = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) p = fmaf(wf[e], hv[q][8 * t + e], p);
          a[q] = fmaf(p, st, a[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < NR; ++q) acc[rr * NR + q] = a[q];
    }
    const float tot = warp_sum_scatter<8>(acc, lane);
    if ((lane & 3) == 0) {
      const int vi = lane >> 2, rr = vi / NR, q = vi - rr * NR;
      y[(size_t)rt[q] * H + n0 + r0 + rr] = tot * gs2;
    }
#pragma unroll
    for (int rr = 0; rr < RG; ++rr) {
      sc[rr] = nsc[rr];
#pragma unroll
      for (int t = 0; t < M; ++t) cw[rr][t] = ncw[rr][t];
    }
  }
}

template <int M, int NQ>
__global__ void __launch_bounds__(kWT, 2) gdown_warp_kernel(DevState st, int H, int layer,
                                                            Groups gr, const float* __restrict__ h,
                                                            float* __restrict__ y, int skip_from) {
  constexpr int I = 256 * M;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kWT / 32) + (threadIdx.x >> 5), Gw = gridDim.x * (kWT / 32);
  const int G = gr.G(), nb = H / kWD;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int un = gw; un < G * nb; un += Gw) {
    const int g = un / nb, n0 = (un - g * nb) * kWD;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    if (skip_from > 0 && rb - ra >= skip_from) continue;  // a dense group: the tensor cores take it
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const float gs2 = reinterpret_cast<const float*>(blob + o.glob)[2];
    const uint8_t* cw0 = blob + o.code[2] + (size_t)n0 * (I / 2) + 4 * M * lane;
    const uint8_t* sc0 = blob + o.scale[2] + (size_t)n0 * (I / 16);
    int q0 = ra;
    for (; NQ > 1 && q0 + NQ <= rb; q0 += NQ) {  // full passes
      int rt[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) rt[q] = gr.route()[q0 + q];
      gdown_warp_pass<M, NQ>(cw0, sc0, h, rt, gs2, H, n0, lane, y);
    }
    for (; q0 < rb; ++q0) {  // the rest one route at a time
      const int rt[1] = {gr.route()[q0]};
      gdown_warp_pass<M, 1>(cw0, sc0, h, rt, gs2, H, n0, lane, y);
    }
  }
}

// ------------------------------------------------------------ 5. combine
__global__ void __launch_bounds__(kWT) gcombine_kernel(const DevState st, int H, int k,
                                                       const int32_t* __restrict__ slot_ids,
                                                       const float* __restrict__ w,
                                                       const float* __restrict__ y,
                                                       const float* __restrict__ ys, int n_rows,
                                                       __nv_bfloat16* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * kWT + threadIdx.x;
  if (i >= (size_t)n_rows * H) return;
  const int b = (int)(i / H), n = (int)(i % H);
  float acc = 0.f;
  for (int j = 0; j < k; ++j) {
    const int r = b * k + j;
    if ((unsigned)slot_ids[r] >= (unsigned)st.S) continue;
    acc = fmaf(w[r], y[(size_t)r * H + n], acc);
  }
  if (ys) acc += ys[i];
  out[i] = __float2bfloat16_rn(acc);
}

int g_sms = 0;
int g_occ[4][2] = {{1, 1}, {1, 1}, {1, 1}, {1, 1}};  // resident CTAs per SM: [format][gate-up, down]
int g_occ_staged[2] = {1, 1};        // ... of the staged NVFP4 kernels
int g_occ_warp = 1;                   // ... of the warp-row gate/up kernel for the cache's H
int g_occ_dwarp = 1;                  // ... of the warp-row down kernel for the cache's I

size_t gup_staged_smem(int H) { return (size_t)kNR * H * 2 + (size_t)kNS * (2 * kStC + 2 * kStS); }
size_t gdown_staged_smem(int I) { return (size_t)kNR * I * 4 + (size_t)kNS * (kStC + kStS); }
// the staged NVFP4 kernels take whole 64-element stages of every row
bool staged_ok(int H, int I) {
  return H % 64 == 0 && I % 64 == 0 && gup_staged_smem(H) <= 200 * 1024 &&
         gdown_staged_smem(I) <= 200 * 1024;
}

// the warp-row gate/up kernel: H = 1024 JH (two routes per pass up to 2048,
// one above, where two routes' x would not fit in registers)
bool warp_ok(int H, int I) { return H >= 1024 && H <= 4096 && H % 1024 == 0 && I % kWB == 0; }
// the warp-row down kernel: I = 256 M, M = 1 .. 4; H in whole units
bool down_warp_ok(int H, int I) {
  return I >= 256 && I <= 1024 && I % 256 == 0 && H % kWD == 0;
}
template <typename F>
cudaError_t by_m(int I, F f) {
  switch (I / 256) {
    case 1: return f(gdown_warp_kernel<1, 2>);
    case 2: return f(gdown_warp_kernel<2, 2>);
    case 3: return f(gdown_warp_kernel<3, 2>);
    case 4: return f(gdown_warp_kernel<4, 2>);
    default: return cudaErrorInvalidValue;
  }
}
template <typename F>
cudaError_t by_jh(int H, F f) {
  switch (H / 1024) {
    case 1: return f(gup_warp_kernel<1, 2>);
    case 2: return f(gup_warp_kernel<2, 2>);
    case 3: return f(gup_warp_kernel<3, 1>);
    case 4: return f(gup_warp_kernel<4, 1>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool grouped_supported(int wfmt, int H, int I, int E) {
  const bool smem = (size_t)E * 16 <= 200 * 1024 && (size_t)kNR * H * 2 <= 200 * 1024 &&
                    (size_t)kNR * I * 4 <= 200 * 1024;
  if (wfmt == MOE_W_NVFP4 || wfmt == MOE_W_MXFP4 || wfmt == MOE_W_Q4_0)
    return smem && H % 32 == 0 && I % 32 == 0;
  return wfmt == MOE_W_BF16 && smem && H % 8 == 0 && I % 8 == 0;
}

cudaError_t grouped_init(int E, int H, int I) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = raise_smem_limit(group_kernel, (size_t)E * 12);
  auto lim = [&](auto kern, size_t bytes) {
    if (e == cudaSuccess) e = raise_smem_limit(kern, bytes);
  };
  const size_t ub = (size_t)kNR * H * 2, db = (size_t)kNR * I * 4;
  lim(gup_kernel<MOE_W_NVFP4>, ub);
  lim(gup_kernel<MOE_W_BF16>, ub);
  lim(gup_kernel<MOE_W_MXFP4>, ub);
  lim(gup_kernel<MOE_W_Q4_0>, ub);
  lim(gdown_kernel<MOE_W_NVFP4>, db);
  lim(gdown_kernel<MOE_W_BF16>, db);
  lim(gdown_kernel<MOE_W_MXFP4>, db);
  lim(gdown_kernel<MOE_W_Q4_0>, db);
  // persistent grids: as many CTAs as fit on the GPU at once
  auto occ = [&](auto kern, size_t bytes, int* out) {
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kern, kWT, bytes);
    if (*out < 1) *out = 1;
  };
  occ(gup_kernel<MOE_W_BF16>, ub, &g_occ[MOE_W_BF16][0]);
  occ(gup_kernel<MOE_W_NVFP4>, ub, &g_occ[MOE_W_NVFP4][0]);
  occ(gup_kernel<MOE_W_MXFP4>, ub, &g_occ[MOE_W_MXFP4][0]);
  occ(gup_kernel<MOE_W_Q4_0>, ub, &g_occ[MOE_W_Q4_0][0]);
  occ(gdown_kernel<MOE_W_BF16>, db, &g_occ[MOE_W_BF16][1]);
  occ(gdown_kernel<MOE_W_NVFP4>, db, &g_occ[MOE_W_NVFP4][1]);
  occ(gdown_kernel<MOE_W_MXFP4>, db, &g_occ[MOE_W_MXFP4][1]);
  occ(gdown_kernel<MOE_W_Q4_0>, db, &g_occ[MOE_W_Q4_0][1]);
  if (staged_ok(H, I)) {
    lim(gup_staged_kernel, gup_staged_smem(H));
    lim(gdown_staged_kernel, gdown_staged_smem(I));
    occ(gup_staged_kernel, gup_staged_smem(H), &g_occ_staged[0]);
    occ(gdown_staged_kernel, gdown_staged_smem(I), &g_occ_staged[1]);
  }
  if (e == cudaSuccess && warp_ok(H, I))
    e = by_jh(H, [&](auto kern) {
      const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_occ_warp, kern, kWT, 0);
      if (g_occ_warp < 1) g_occ_warp = 1;
      return r;
    });
  if (e == cudaSuccess && down_warp_ok(H, I))
    e = by_m(I, [&](auto kern) {
      const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_occ_dwarp, kern, kWT, 0);
      if (g_occ_dwarp < 1) g_occ_dwarp = 1;
      return r;
    });
  if (e == cudaSuccess && grouped_tc_supported(MOE_W_NVFP4, H, I)) e = grouped_tc_init();
  return e;
}

cudaError_t launch_routed_grouped(const DevState& st, int wfmt, int H, int I, int layer,
                                  const void* x, const int32_t* slot_ids, const float* w,
                                  int n_rows, int k, const float* shared_y, void* out,
                                  FfnScratch sc, int max_routes, int wide_mode,
                                  cudaStream_t s) {
  const int R = n_rows * k;
  Groups gr{st.groups, max_routes};
  const bool tc_any = wide_mode != MOE_WIDE_CUDA_CORES && grouped_tc_supported(wfmt, H, I);
  const bool tc_split = tc_any && wide_mode != MOE_WIDE_TENSOR_CORES && staged_ok(H, I);
  // the tensor cores' groups: those of at least kTcMinRoutes routes (every group
  // when they take them all)
  group_kernel<<<1, kGT, (size_t)st.E * 12, s>>>(st, layer, slot_ids, R, gr,
                                                 tc_any ? (tc_split ? kTcMinRoutes : 1) : 0,
                                                 tc_any ? sc.dense : nullptr);
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const int sms = g_sms > 0 ? g_sms : 1;
  const int fi = wfmt >= MOE_W_BF16 && wfmt <= MOE_W_Q4_0 ? wfmt : MOE_W_BF16;
  const int grid_u = sms * g_occ[fi][0], grid_d = sms * g_occ[fi][1];
  // NVFP4 with both kernel families available: per group by its route count
  // (auto), or all groups on one family (a forced mode)
  const bool tc = tc_any;
  const bool cc = wide_mode != MOE_WIDE_TENSOR_CORES || !tc;
  if (wfmt == MOE_W_NVFP4 && (tc || staged_ok(H, I))) {
    xprep_kernel<MOE_W_NVFP4><<<n_rows, kWT, 0, s>>>(xx, H, sc.x16, sc.xinv);
    const bool split = tc && cc && staged_ok(H, I);
    const int tc_from = !tc ? 0 : (split ? kTcMinRoutes : 1);  // tensor cores: groups >= this
    if (cc && warp_ok(H, I)) {
      const cudaError_t e = by_jh(H, [&](auto kern) {
        kern<<<sms * g_occ_warp, kWT, 0, s>>>(st, I, layer, sc.x16, sc.xinv, k, gr, sc.h, tc_from);
        return cudaGetLastError();
      });
      if (e != cudaSuccess) return e;
    } else if (cc && staged_ok(H, I)) {
      gup_staged_kernel<<<sms * g_occ_staged[0], kWT, gup_staged_smem(H), s>>>(
          st, H, I, layer, sc.x16, sc.xinv, k, gr, sc.h, tc_from);
    }
    if (tc) {
      cudaError_t e = launch_grouped_tc(st, H, I, layer, k, R, max_routes, sc, st.status, s);
      if (e != cudaSuccess) return e;
    }
    if (cc && down_warp_ok(H, I)) {
      const cudaError_t e = by_m(I, [&](auto kern) {
        kern<<<sms * g_occ_dwarp, kWT, 0, s>>>(st, H, layer, gr, sc.h, sc.y, tc_from);
        return cudaGetLastError();
      });
      if (e != cudaSuccess) return e;
    } else if (cc && staged_ok(H, I)) {
      gdown_staged_kernel<<<sms * g_occ_staged[1], kWT, gdown_staged_smem(I), s>>>(
          st, H, I, layer, gr, sc.h, sc.y, tc_from);
    }
  } else if (wfmt == MOE_W_NVFP4 || wfmt == MOE_W_MXFP4 || wfmt == MOE_W_Q4_0) {
    // the CUDA-core kernels of the 4-bit format (x as f16 for every one)
    xprep_kernel<MOE_W_NVFP4><<<n_rows, kWT, 0, s>>>(xx, H, sc.x16, sc.xinv);
    auto run = [&](auto fmt) {
      constexpr int F = decltype(fmt)::value;
      gup_kernel<F><<<grid_u, kWT, (size_t)kNR * H * 2, s>>>(st, H, I, layer, sc.x16, sc.xinv, k,
                                                             gr, sc.h);
      gdown_kernel<F><<<grid_d, kWT, (size_t)kNR * I * 4, s>>>(st, H, I, layer, gr, sc.h, sc.y);
    };
    if (wfmt == MOE_W_MXFP4) run(std::integral_constant<int, MOE_W_MXFP4>{});
    else if (wfmt == MOE_W_Q4_0) run(std::integral_constant<int, MOE_W_Q4_0>{});
    else run(std::integral_constant<int, MOE_W_NVFP4>{});
  } else {
    xprep_kernel<MOE_W_BF16><<<n_rows, kWT, 0, s>>>(xx, H, sc.x16, sc.xinv);
    gup_kernel<MOE_W_BF16><<<grid_u, kWT, (size_t)kNR * H * 2, s>>>(st, H, I, layer, sc.x16,
                                                                    sc.xinv, k, gr, sc.h);
    gdown_kernel<MOE_W_BF16><<<grid_d, kWT, (size_t)kNR * I * 4, s>>>(st, H, I, layer, gr, sc.h,
                                                                     sc.y);
  }
  const size_t n = (size_t)n_rows * H;
  gcombine_kernel<<<(unsigned)((n + kWT - 1) / kWT), kWT, 0, s>>>(
      st, H, k, slot_ids, w, sc.y, shared_y, n_rows, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace moe
