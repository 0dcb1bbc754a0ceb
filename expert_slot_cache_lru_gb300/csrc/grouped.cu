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
// reading every resident expert once from HBM, not by arithmetic.  The kernels
// therefore group the routes by expert and read each expert's weights once:
//   1. group_kernel   (1 CTA): the CSR of routes per distinct expert, ascending
//      expert id, routes ascending within a group -- the cache's route groups;
//   2. xprep_kernel:  x as f16 (NVFP4 experts; per-row power-of-two scale so
//      that max |x| < 2^15, undone on the fp32 sums) or bf16 (bf16 experts);
//   3. gup_kernel:    per (group, 32 rows of I): h[r] = silu(W_g x_b) * (W_u x_b)
//      for every route r of the group -- each weight word is decoded once and
//      applied to up to four routes at a time;
//   4. gdown_kernel:  per (group, 64 rows of H): y[r] = gs_d * W_d h[r];
//   5. combine_kernel: out[b][n] = bf16( sum_j w[b,j] y[b*k+j][n] + ys[b][n] ).
// Kernels 3 and 4 are persistent (a few CTAs per SM walk the work items), so
// the data-dependent number of groups needs no host round trip.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGT = 1024;       // group_kernel threads
constexpr int kWT = 256;        // threads of the FFN kernels (8 warps)
constexpr int kNR = 4;          // routes per decode pass
constexpr int kRowsU = 32;      // rows of I per gate/up work item (4 per warp)
constexpr int kRowsD = 64;      // rows of H per down work item (8 per warp)

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

// Eight per-lane partial sums -> lane 4i holds the total of v[i] (9 shuffles).
__device__ __forceinline__ float reduce8(const float v[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float k[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    k[i] = (b4 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[4 + i], 16);
  float q[2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
    q[i] = (b3 ? k[2 + i] : k[i]) + __shfl_xor_sync(0xffffffffu, b3 ? k[i] : k[2 + i], 8);
  float r = (b2 ? q[1] : q[0]) + __shfl_xor_sync(0xffffffffu, b2 ? q[0] : q[1], 4);
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  return r;
}
// Four per-lane partial sums -> lane 8i holds the total of p[i] (6 shuffles).
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

// Offsets inside a blob (layout of moe_cache.h).
struct Off {
  size_t code[3], scale[3], glob, mat[3];
  __device__ Off(int H, int I) {
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
                                                    Groups gr) {
  extern __shared__ int gsm[];
  const int E = st.E;
  int* off = gsm;          // [E] routes, then start offset, of expert e
  int* cur = gsm + E;      // [E] scatter cursor
  int* eslot = gsm + 2 * E;  // [E] the slot of expert e
  int* gid = gsm + 3 * E;    // [E] group index of expert e (-1 = none)
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
  int nr = 0, ng = 0;
  for (int e = e0; e < e1; ++e) {
    nr += off[e];
    ng += off[e] > 0;
  }
  int totR, totG;
  int r0 = block_excl_scan(nr, bs, &totR);
  int g0 = block_excl_scan(ng, bs, &totG);
  for (int e = e0; e < e1; ++e) {
    const int c = off[e];
    gid[e] = c > 0 ? g0 : -1;
    if (c > 0) {
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
  }
  __syncthreads();
  for (int r = tid; r < R; r += kGT) {
    const int s = slot_ids[r];
    if ((unsigned)s >= (unsigned)st.S) continue;
    const int e = st.slot_key[pbase + s] - layer * E;
    if ((unsigned)e >= (unsigned)E) continue;
    gr.route()[off[e] + atomicAdd(&cur[e], 1)] = r;
  }
  __syncthreads();
  for (int g = tid; g < totG; g += kGT) {  // ascending route index within the group
    int32_t* rt = gr.route();
    const int a = gr.start()[g], b = gr.start()[g + 1];
    for (int i = a + 1; i < b; ++i) {
      const int v = rt[i];
      int j = i - 1;
      while (j >= a && rt[j] > v) {
        rt[j + 1] = rt[j];
        --j;
      }
      rt[j + 1] = v;
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
// Work item (group g, chunk ch of kRowsU rows of I); warp w takes 4 rows.  The
// x rows of up to kNR of the group's routes are staged in shared memory per
// pass (16-byte units, unit u of a row at u ^ ((u >> 3) & 7) so that the
// lanes' reads are conflict-free); each warp keeps the next row's weight words
// in flight while it decodes the current one.
// Lane L covers, per 2048 (NVFP4) / 512 (bf16) elements of a row, the same
// elements as the decode kernel: NVFP4 [32L, 32L+32) and [1024+32L, ...);
// bf16 8L + [0, 8) and 256 + 8L + [0, 8).
__device__ __forceinline__ int xsw(int u) { return u ^ ((u >> 3) & 7); }

template <int FMT>
struct RowU;
template <>
struct RowU<MOE_W_NVFP4> {  // one 2048-element chunk of a gate row and an up row
  uint4 g[2], u[2];
  uint32_t sg[2], su[2];
  __device__ __forceinline__ void load(const uint8_t* blob, const Off& o, int H, int i, int c,
                                       int lane) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const size_t cb = (size_t)i * (H / 2) + c * 1024 + hf * 512 + lane * 16;
      const size_t sb = (size_t)i * (H / 16) + c * 128 + hf * 64 + lane * 2;
      g[hf] = *reinterpret_cast<const uint4*>(blob + o.code[0] + cb);
      u[hf] = *reinterpret_cast<const uint4*>(blob + o.code[1] + cb);
      sg[hf] = *reinterpret_cast<const uint16_t*>(blob + o.scale[0] + sb);
      su[hf] = *reinterpret_cast<const uint16_t*>(blob + o.scale[1] + sb);
    }
  }
  // ga[j] / ua[j] += this chunk's gate / up partial for staged route j < nq
  __device__ __forceinline__ void dot(const uint4* xs, int Hu, int c, int lane, int nq, float* ga,
                                      float* ua) const {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t gv[4] = {g[hf].x, g[hf].y, g[hf].z, g[hf].w};
      const uint32_t uv[4] = {u[hf].x, u[hf].y, u[hf].z, u[hf].w};
      uint32_t gd[16], ud[16];  // decoded once, applied to every route
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
      const float2 sgf = e4m3x2(sg[hf]), suf = e4m3x2(su[hf]);
      const int u0 = c * 256 + hf * 128 + lane * 4;
#pragma unroll
      for (int j = 0; j < kNR; ++j) {
        if (j >= nq) break;
        const uint4* xr = xs + (size_t)j * Hu;
        const uint4 x0 = xr[xsw(u0)], x1 = xr[xsw(u0 + 1)], x2 = xr[xsw(u0 + 2)],
                    x3 = xr[xsw(u0 + 3)];
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
        ga[j] = fmaf(p, sgf.x, fmaf(p2, sgf.y, ga[j]));
        ua[j] = fmaf(q, suf.x, fmaf(q2, suf.y, ua[j]));
      }
    }
  }
};
template <>
struct RowU<MOE_W_BF16> {  // one 512-element chunk of a gate row and an up row
  uint4 g[2], u[2];
  __device__ __forceinline__ void load(const uint8_t* blob, const Off& o, int H, int i, int c,
                                       int lane) {
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const size_t eo = ((size_t)i * H + c * 512 + s2 * 256 + lane * 8) * 2;
      g[s2] = *reinterpret_cast<const uint4*>(blob + o.mat[0] + eo);
      u[s2] = *reinterpret_cast<const uint4*>(blob + o.mat[1] + eo);
    }
  }
  __device__ __forceinline__ void dot(const uint4* xs, int Hu, int c, int lane, int nq, float* ga,
                                      float* ua) const {
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int un = c * 64 + s2 * 32 + lane;
#pragma unroll
      for (int j = 0; j < kNR; ++j) {
        if (j >= nq) break;
        const uint4 xv = xs[(size_t)j * Hu + xsw(un)];
        ga[j] = fma2b(g[s2].w, xv.w, fma2b(g[s2].z, xv.z, fma2b(g[s2].y, xv.y, fma2b(g[s2].x, xv.x, ga[j]))));
        ua[j] = fma2b(u[s2].w, xv.w, fma2b(u[s2].z, xv.z, fma2b(u[s2].y, xv.y, fma2b(u[s2].x, xv.x, ua[j]))));
      }
    }
  }
};

template <int FMT>
__global__ void __launch_bounds__(kWT) gup_kernel(DevState st, int H, int I, int layer,
                                                  const uint16_t* __restrict__ x16,
                                                  const float* __restrict__ xinv, int k, Groups gr,
                                                  float* __restrict__ h) {
  extern __shared__ __align__(16) uint4 xs[];  // [kNR][H / 8]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gr.G();
  const int nch = (I + kRowsU - 1) / kRowsU;
  const int Hu = H / 8;
  constexpr int CW = FMT == MOE_W_NVFP4 ? 2048 : 512;
  const int KC = H / CW;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    float gs0 = 1.f, gs1 = 1.f;
    if (FMT == MOE_W_NVFP4) {
      gs0 = reinterpret_cast<const float*>(blob + o.glob)[0];
      gs1 = reinterpret_cast<const float*>(blob + o.glob)[1];
    }
    const int i0 = ch * kRowsU + warp * (kRowsU / 8);
    const int nrow = max(0, min(kRowsU / 8, I - i0));
    for (int q0 = ra; q0 < rb; q0 += kNR) {  // up to kNR routes per pass
      const int nq = min(kNR, rb - q0);
      __syncthreads();  // the previous pass's x no longer read
      for (int v = threadIdx.x; v < nq * Hu; v += kWT) {
        const int j = v / Hu, un = v - j * Hu;
        const int b = gr.route()[q0 + j] / k;
        xs[(size_t)j * Hu + xsw(un)] = reinterpret_cast<const uint4*>(x16 + (size_t)b * H)[un];
      }
      __syncthreads();
      // rows of this warp; items (row, chunk) with the next one's words in flight
      const int nit = nrow * KC;
      RowU<FMT> cur, nxt;
      if (nit > 0) cur.load(blob, o, H, i0, 0, lane);
      float ga[kNR], ua[kNR];
#pragma unroll
      for (int j = 0; j < kNR; ++j) ga[j] = ua[j] = 0.f;
      for (int it = 0; it < nit; ++it) {
        const int i = i0 + it / KC, c = it % KC;
        if (it + 1 < nit) nxt.load(blob, o, H, i0 + (it + 1) / KC, (it + 1) % KC, lane);
        cur.dot(xs, Hu, c, lane, nq, ga, ua);
        if (c == KC - 1) {  // row i complete
          const float v[8] = {ga[0], ga[1], ga[2], ga[3], ua[0], ua[1], ua[2], ua[3]};
          const float tot = reduce8(v, lane);
          const float upart = __shfl_down_sync(0xffffffffu, tot, 16);  // lane 4j <- u_j
          if (lane < 4 * kNR && (lane & 3) == 0 && (lane >> 2) < nq) {
            const int r = gr.route()[q0 + (lane >> 2)];
            const float xi = xinv[r / k];
            const float gg = tot * xi * gs0, uu = upart * xi * gs1;
            h[(size_t)r * I + i] = gg / (1.f + expf(-gg)) * uu;
          }
#pragma unroll
          for (int j = 0; j < kNR; ++j) ga[j] = ua[j] = 0.f;
        }
        cur = nxt;
      }
    }
  }
}

// ------------------------------------------------------------ 4. down
// Work item (group g, chunk of kRowsD rows of H); warp w takes 8 rows.  h of
// up to kNR of the group's routes is staged in shared memory per pass.
// NVFP4: a row of I elements is I/16 blocks of 16; lane L takes blocks L,
// L+32, ... (8 code bytes and one scale each).  bf16: lane L takes 16-byte
// words L, L+32, ... of the row.  The words of four rows are requested
// before any of them is decoded.
template <int FMT>
__global__ void __launch_bounds__(kWT) gdown_kernel(DevState st, int H, int I, int layer,
                                                    Groups gr, const float* __restrict__ h,
                                                    float* __restrict__ y) {
  extern __shared__ __align__(16) float hsm[];  // [kNR][I]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gr.G();
  const int nch = (H + kRowsD - 1) / kRowsD;
  const Off o(H, I);
  const size_t pbase = (size_t)pool_of(st, layer) * st.S;
  const int nblk = FMT == MOE_W_NVFP4 ? I / 16 : I / 8;  // lane work units per row
  for (int item = blockIdx.x; item < G * nch; item += gridDim.x) {
    const int g = item / nch, ch = item - g * nch;
    const int ra = gr.start()[g], rb = gr.start()[g + 1];
    const uint8_t* blob = st.slots + (pbase + gr.slot()[g]) * st.stride;
    const float gs2 = FMT == MOE_W_NVFP4 ? reinterpret_cast<const float*>(blob + o.glob)[2] : 1.f;
    const int n0 = ch * kRowsD + warp * (kRowsD / 8);
    for (int q0 = ra; q0 < rb; q0 += kNR) {
      const int nq = min(kNR, rb - q0);
      __syncthreads();
      for (int v = threadIdx.x; v < nq * I / 4; v += kWT) {
        const int j = v / (I / 4), f = v - j * (I / 4);
        reinterpret_cast<float4*>(hsm)[v] =
            __ldcg(reinterpret_cast<const float4*>(h + (size_t)gr.route()[q0 + j] * I) + f);
      }
      __syncthreads();
      for (int r4 = 0; r4 < kRowsD / 8; r4 += 4) {  // four rows at a time
        uint2 cw[4][2];
        uint32_t scb[4][2];
        uint4 bw[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int n = n0 + r4 + rr;
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int blk = lane + 32 * bb;
            const bool ok = n < H && blk < nblk;
            if (FMT == MOE_W_NVFP4) {
              cw[rr][bb] = ok ? *reinterpret_cast<const uint2*>(blob + o.code[2] + (size_t)n * (I / 2) + blk * 8)
                              : make_uint2(0u, 0u);
              scb[rr][bb] = ok ? blob[o.scale[2] + (size_t)n * (I / 16) + blk] : 0u;
            } else {
              bw[rr][bb] = ok ? *reinterpret_cast<const uint4*>(blob + o.mat[2] + ((size_t)n * I + blk * 8) * 2)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int n = n0 + r4 + rr;
          const int nn = min(n, H - 1);  // rows past H compute nothing that is stored
          float acc[kNR] = {0.f, 0.f, 0.f, 0.f};
          auto blk_nvfp4 = [&](int blk, uint2 c2, uint32_t sv) {
            const float sc = e4m3x2(sv).x;
            float wf[16];
            const uint32_t ww[2] = {c2.x, c2.y};
#pragma unroll
            for (int wd = 0; wd < 2; ++wd) {
              const float2 a0 = f16x2_f32(e2m1x2<0>(ww[wd])), a1 = f16x2_f32(e2m1x2<1>(ww[wd]));
              const float2 a2 = f16x2_f32(e2m1x2<2>(ww[wd])), a3 = f16x2_f32(e2m1x2<3>(ww[wd]));
              wf[8 * wd] = a0.x, wf[8 * wd + 1] = a0.y, wf[8 * wd + 2] = a1.x, wf[8 * wd + 3] = a1.y;
              wf[8 * wd + 4] = a2.x, wf[8 * wd + 5] = a2.y, wf[8 * wd + 6] = a3.x, wf[8 * wd + 7] = a3.y;
            }
#pragma unroll
            for (int jj = 0; jj < kNR; ++jj) {
              if (jj >= nq) break;
              const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)jj * I + blk * 16);
              float p = 0.f;
#pragma unroll
              for (int e4 = 0; e4 < 4; ++e4) {
                const float4 hv = hp[e4];
                p = fmaf(wf[4 * e4], hv.x, p);
                p = fmaf(wf[4 * e4 + 1], hv.y, p);
                p = fmaf(wf[4 * e4 + 2], hv.z, p);
                p = fmaf(wf[4 * e4 + 3], hv.w, p);
              }
              acc[jj] = fmaf(p, sc, acc[jj]);
            }
          };
          auto blk_bf16 = [&](int blk, uint4 v) {
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int jj = 0; jj < kNR; ++jj) {
              if (jj >= nq) break;
              const float4* hp = reinterpret_cast<const float4*>(hsm + (size_t)jj * I + blk * 8);
              const float4 h0 = hp[0], h1 = hp[1];
              const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[jj] = fmaf(fp32_of_bf16(vv[e] & 0xffffu), hv[2 * e], acc[jj]);
                acc[jj] = fmaf(__uint_as_float(vv[e] & 0xffff0000u), hv[2 * e + 1], acc[jj]);
              }
            }
          };
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {  // the two units loaded above
            const int blk = lane + 32 * bb;
            if (blk >= nblk) continue;
            if (FMT == MOE_W_NVFP4) blk_nvfp4(blk, cw[rr][bb], scb[rr][bb]);
            else blk_bf16(blk, bw[rr][bb]);
          }
          for (int blk = lane + 64; blk < nblk; blk += 32) {  // wider rows: loaded here
            if (FMT == MOE_W_NVFP4)
              blk_nvfp4(blk, *reinterpret_cast<const uint2*>(blob + o.code[2] + (size_t)nn * (I / 2) + blk * 8),
                        blob[o.scale[2] + (size_t)nn * (I / 16) + blk]);
            else
              blk_bf16(blk, *reinterpret_cast<const uint4*>(blob + o.mat[2] + ((size_t)nn * I + blk * 8) * 2));
          }
          const float tot = reduce4(acc, lane);
          if (n < H && (lane & 7) == 0 && (lane >> 3) < nq)
            y[(size_t)gr.route()[q0 + (lane >> 3)] * H + n] = tot * gs2;
        }
      }
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

}  // namespace

bool grouped_supported(int wfmt, int H, int I, int E) {
  const bool smem = (size_t)E * 16 <= 200 * 1024 && (size_t)kNR * H * 2 <= 200 * 1024 &&
                    (size_t)kNR * I * 4 <= 200 * 1024;
  if (wfmt == MOE_W_NVFP4) return smem && H % 2048 == 0 && I % 64 == 0;
  return smem && H % 512 == 0 && I % 8 == 0;
}

cudaError_t grouped_init(int E, int H, int I) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && (size_t)E * 16 > 48 * 1024)
    e = cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((size_t)E * 16));
  auto lim = [&](auto kern, size_t bytes) {
    if (e == cudaSuccess && bytes > 48 * 1024)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  };
  lim(gup_kernel<MOE_W_NVFP4>, (size_t)kNR * H * 2);
  lim(gup_kernel<MOE_W_BF16>, (size_t)kNR * H * 2);
  lim(gdown_kernel<MOE_W_NVFP4>, (size_t)kNR * I * 4);
  lim(gdown_kernel<MOE_W_BF16>, (size_t)kNR * I * 4);
  return e;
}

cudaError_t launch_routed_grouped(const DevState& st, int wfmt, int H, int I, int layer,
                                  const void* x, const int32_t* slot_ids, const float* w,
                                  int n_rows, int k, const float* shared_y, void* out,
                                  FfnScratch sc, int max_routes, cudaStream_t s) {
  const int R = n_rows * k;
  Groups gr{st.groups, max_routes};
  group_kernel<<<1, kGT, (size_t)st.E * 16, s>>>(st, layer, slot_ids, R, gr);
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const int grid = (g_sms > 0 ? g_sms : 1) * 4;
  if (wfmt == MOE_W_NVFP4) {
    xprep_kernel<MOE_W_NVFP4><<<n_rows, kWT, 0, s>>>(xx, H, sc.x16, sc.xinv);
    gup_kernel<MOE_W_NVFP4><<<grid, kWT, (size_t)kNR * H * 2, s>>>(st, H, I, layer, sc.x16,
                                                                     sc.xinv, k, gr, sc.h);
    gdown_kernel<MOE_W_NVFP4><<<grid, kWT, (size_t)kNR * I * 4, s>>>(st, H, I, layer, gr, sc.h,
                                                                      sc.y);
  } else {
    xprep_kernel<MOE_W_BF16><<<n_rows, kWT, 0, s>>>(xx, H, sc.x16, sc.xinv);
    gup_kernel<MOE_W_BF16><<<grid, kWT, (size_t)kNR * H * 2, s>>>(st, H, I, layer, sc.x16,
                                                                    sc.xinv, k, gr, sc.h);
    gdown_kernel<MOE_W_BF16><<<grid, kWT, (size_t)kNR * I * 4, s>>>(st, H, I, layer, gr, sc.h,
                                                                     sc.y);
  }
  const size_t n = (size_t)n_rows * H;
  gcombine_kernel<<<(unsigned)((n + kWT - 1) / kWT), kWT, 0, s>>>(
      st, H, k, slot_ids, w, sc.y, shared_y, n_rows, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace moe
