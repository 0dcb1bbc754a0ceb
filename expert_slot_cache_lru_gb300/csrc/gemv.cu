// gemv.cu -- routed and shared expert FFNs on the CUDA cores (decode-sized
// steps), and the weighted combine.
//
// [FreeToken issue #753 "[Perf] Offloaded decode: overlap the expert-miss
// gather with the same layer's shared expert ...", Problem and What we
// changed]: the shared expert and its sigmoid gate read the original hidden
// state and are computed before the routed experts; the routed experts run
// over the slot ids; the result is routed + shared, in that order.
// [FreeToken PR #491 "refactor(moe): extract hybrid decode orchestration",
// section 5]: a route whose slot id is -1 contributes nothing on the GPU.
//
// Work split: one warp per output row.  Weights stream through 128-bit loads
// (NVFP4: 32 e2m1 codes and their two e4m3 scales per lane per step; bf16:
// 32 elements per lane per step), the activation vector sits in shared memory
// as fp32, and each warp reduces its row with shuffles.  Accumulation is fp32;
// the e2m1 x e4m3 x bf16 products are exact in fp32.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(__half(h));
}

// Two e2m1 codes of one byte (element 2i in the low nibble) as fp32.
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte) {
  __half2_raw h2 = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
  return __half22float2(__half2(h2));
}

// sum_{i<8} e2m1(word nibble i) * xs[i]  (nibble i = element i of the word)
__device__ __forceinline__ float dot8_e2m1(uint32_t w, const float* xs) {
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 f = e2m1x2_to_f32((w >> (8 * b)) & 0xffu);
    acc = fmaf(f.x, xs[2 * b], acc);
    acc = fmaf(f.y, xs[2 * b + 1], acc);
  }
  return acc;
}

// sum_{i<8} bf16(pair words) * xs[i]
__device__ __forceinline__ float dot8_bf16(uint4 v, const float* xs) {
  float acc = 0.f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(w[i] << 16), xs[2 * i], acc);
    acc = fmaf(__uint_as_float(w[i] & 0xffff0000u), xs[2 * i + 1], acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Byte offsets inside an NVFP4 blob (see the layout in moe_cache.h).
struct Nvfp4Off {
  size_t code[3], scale[3], glob;
  __device__ Nvfp4Off(int H, int I) {
    const size_t ih = (size_t)I * H;
    code[0] = 0;
    code[1] = ih / 2;
    code[2] = ih;
    scale[0] = 3 * ih / 2;
    scale[1] = scale[0] + ih / 16;
    scale[2] = scale[1] + ih / 16;
    glob = scale[2] + ih / 16;
  }
};

// Dot of row n of an [rows, K] matrix with the fp32 vector xs[K] (in shared
// memory), partial per lane; the caller reduces.  K is a multiple of 32.
template <int FMT>
__device__ __forceinline__ float row_dot_k32(const uint8_t* blob, int which, int H, int I, int n,
                                             const float* xs, int K) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (FMT == MOE_W_NVFP4) {
    const Nvfp4Off o(H, I);
    const uint8_t* codes = blob + o.code[which] + (size_t)n * (K / 2);
    const uint8_t* scales = blob + o.scale[which] + (size_t)n * (K / 16);
    for (int base = lane * 32; base < K; base += 1024) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + base / 2);
      const uint16_t sc = *reinterpret_cast<const uint16_t*>(scales + base / 16);
      const float* x = xs + base;
      const float p0 = dot8_e2m1(c.x, x) + dot8_e2m1(c.y, x + 8);
      const float p1 = dot8_e2m1(c.z, x + 16) + dot8_e2m1(c.w, x + 24);
      acc = fmaf(p0, e4m3_to_f32((uint8_t)(sc & 0xff)), acc);
      acc = fmaf(p1, e4m3_to_f32((uint8_t)(sc >> 8)), acc);
    }
  } else {
    const size_t mat = (size_t)which * H * I * 2;
    const uint8_t* row = blob + mat + (size_t)n * K * 2;
    for (int base = lane * 32; base < K; base += 1024) {
      const uint4* p = reinterpret_cast<const uint4*>(row + (size_t)base * 2);
      const float* x = xs + base;
      acc += dot8_bf16(p[0], x) + dot8_bf16(p[1], x + 8) + dot8_bf16(p[2], x + 16) +
             dot8_bf16(p[3], x + 24);
    }
  }
  return acc;
}

// Same for K a multiple of 16 with one 16-element block per lane per step
// (the down projection, K = I).
template <int FMT>
__device__ __forceinline__ float row_dot_k16(const uint8_t* blob, int which, int H, int I, int n,
                                             const float* xs, int K) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (FMT == MOE_W_NVFP4) {
    const Nvfp4Off o(H, I);
    const uint8_t* codes = blob + o.code[which] + (size_t)n * (K / 2);
    const uint8_t* scales = blob + o.scale[which] + (size_t)n * (K / 16);
    for (int base = lane * 16; base < K; base += 512) {
      const uint2 c = *reinterpret_cast<const uint2*>(codes + base / 2);
      const float* x = xs + base;
      const float p = dot8_e2m1(c.x, x) + dot8_e2m1(c.y, x + 8);
      acc = fmaf(p, e4m3_to_f32(scales[base / 16]), acc);
    }
  } else {
    const size_t mat = (size_t)which * H * I * 2;
    const uint8_t* row = blob + mat + (size_t)n * K * 2;
    for (int base = lane * 16; base < K; base += 512) {
      const uint4* p = reinterpret_cast<const uint4*>(row + (size_t)base * 2);
      acc += dot8_bf16(p[0], xs + base) + dot8_bf16(p[1], xs + base + 8);
    }
  }
  return acc;
}

template <int FMT>
__device__ __forceinline__ float global_scale(const uint8_t* blob, int H, int I, int which) {
  if (FMT != MOE_W_NVFP4) return 1.f;
  const Nvfp4Off o(H, I);
  return reinterpret_cast<const float*>(blob + o.glob)[which];
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

__device__ __forceinline__ const uint8_t* slot_blob(const DevState& st, int layer, int slot) {
  return st.slots + ((size_t)pool_of(st, layer) * st.S + slot) * st.stride;
}

// h[t][n] = silu(W_g x_b)[n] * (W_u x_b)[n] for task t (a route or a row),
// rows n of this block.  SHARED: task t = row b, fixed blob, plus the gate
// sigmoid(x_b . w_g) computed by the block with blockIdx.x == 0.
template <int FMT, bool SHARED>
__global__ void __launch_bounds__(kThreads)
up_kernel(DevState st, int H, int I, int layer, const uint16_t* __restrict__ x,
          const int32_t* __restrict__ slot_ids, int k, const uint8_t* fixed_blob,
          const uint16_t* __restrict__ gate_w, float* __restrict__ h, float* __restrict__ gate) {
  extern __shared__ float xs[];  // [H]
  const int t = blockIdx.y;
  const int b = SHARED ? t : t / k;
  const uint8_t* blob;
  if (SHARED) {
    blob = fixed_blob;
  } else {
    const int slot = slot_ids[t];
    if ((unsigned)slot >= (unsigned)st.S) return;  // -1 (overflow / invalid): nothing to compute
    blob = slot_blob(st, layer, slot);
  }
  for (int i = threadIdx.x; i < H; i += kThreads) xs[i] = bf16_to_f32(x[(size_t)b * H + i]);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (SHARED && blockIdx.x == 0 && warp == 0) {
    float z = 0.f;
    for (int i = lane; i < H; i += 32) z = fmaf(bf16_to_f32(gate_w[i]), xs[i], z);
    z = warp_sum(z);
    if (lane == 0) gate[b] = 1.f / (1.f + expf(-z));
  }
  const int n = blockIdx.x * kWarps + warp;
  if (n >= I) return;
  float g = row_dot_k32<FMT>(blob, 0, H, I, n, xs, H);
  float u = row_dot_k32<FMT>(blob, 1, H, I, n, xs, H);
  g = warp_sum(g);
  u = warp_sum(u);
  if (lane == 0) {
    g *= global_scale<FMT>(blob, H, I, 0);
    u *= global_scale<FMT>(blob, H, I, 1);
    h[(size_t)t * I + n] = silu(g) * u;
  }
}

// Shared expert down projection, gated: ys[b][n] = gate[b] * (W_d hs_b)[n].
template <int FMT>
__global__ void __launch_bounds__(kThreads)
shared_down_kernel(int H, int I, const uint8_t* blob, const float* __restrict__ hs,
                   const float* __restrict__ gate, float* __restrict__ ys) {
  extern __shared__ float hsm[];  // [I]
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < I; i += kThreads) hsm[i] = hs[(size_t)b * I + i];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + warp;
  if (n >= H) return;
  float y = warp_sum(row_dot_k16<FMT>(blob, 2, H, I, n, hsm, I));
  if (lane == 0) ys[(size_t)b * H + n] = gate[b] * (y * global_scale<FMT>(blob, H, I, 2));
}

// out[b][n] = bf16( sum_j w[b,j] * (W_d[slot_bj] h_bj)[n]  +  ys[b][n] ),
// j ascending, routes with slot -1 skipped.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
down_combine_kernel(DevState st, int H, int I, int layer, const int32_t* __restrict__ slot_ids,
                    const float* __restrict__ w, int k, const float* __restrict__ h,
                    const float* __restrict__ ys, __nv_bfloat16* __restrict__ out) {
  extern __shared__ float hsm[];  // [k][I]
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < k * I; i += kThreads) {
    const int j = i / I;
    hsm[i] = (unsigned)slot_ids[(size_t)b * k + j] < (unsigned)st.S ? h[((size_t)b * k) * I + i] : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + warp;
  if (n >= H) return;
  float acc = 0.f;
  for (int j = 0; j < k; ++j) {
    const int slot = slot_ids[(size_t)b * k + j];
    if ((unsigned)slot >= (unsigned)st.S) continue;
    const uint8_t* blob = slot_blob(st, layer, slot);
    const float p = row_dot_k16<FMT>(blob, 2, H, I, n, hsm + (size_t)j * I, I);
    acc = fmaf(w[(size_t)b * k + j] * global_scale<FMT>(blob, H, I, 2), p, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    if (ys) acc += ys[(size_t)b * H + n];
    out[(size_t)b * H + n] = __float2bfloat16_rn(acc);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t gemv_set_smem_limits(int H, int I, int Is, int k_max) {
  cudaError_t e = cudaSuccess;
  const size_t xb = (size_t)H * 4;
  if (e == cudaSuccess) e = set_smem(up_kernel<MOE_W_BF16, false>, xb);
  if (e == cudaSuccess) e = set_smem(up_kernel<MOE_W_NVFP4, false>, xb);
  if (e == cudaSuccess) e = set_smem(up_kernel<MOE_W_BF16, true>, xb);
  if (e == cudaSuccess) e = set_smem(up_kernel<MOE_W_NVFP4, true>, xb);
  const size_t hb = (size_t)k_max * I * 4;
  if (e == cudaSuccess) e = set_smem(down_combine_kernel<MOE_W_BF16>, hb);
  if (e == cudaSuccess) e = set_smem(down_combine_kernel<MOE_W_NVFP4>, hb);
  const size_t sb = (size_t)Is * 4;
  if (e == cudaSuccess) e = set_smem(shared_down_kernel<MOE_W_BF16>, sb);
  if (e == cudaSuccess) e = set_smem(shared_down_kernel<MOE_W_NVFP4>, sb);
  return e;
}

cudaError_t launch_shared_expert(int wfmt, int H, int Is, const void* x, int n_rows,
                                 const uint8_t* blob, const void* gate_w, FfnScratch sc,
                                 cudaStream_t s) {
  DevState none{};
  const dim3 gu((Is + kWarps - 1) / kWarps, n_rows);
  const dim3 gd((H + kWarps - 1) / kWarps, n_rows);
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const uint16_t* gw = static_cast<const uint16_t*>(gate_w);
  if (wfmt == MOE_W_NVFP4) {
    up_kernel<MOE_W_NVFP4, true><<<gu, kThreads, (size_t)H * 4, s>>>(none, H, Is, 0, xx, nullptr,
                                                                     1, blob, gw, sc.hs, sc.gate);
    shared_down_kernel<MOE_W_NVFP4><<<gd, kThreads, (size_t)Is * 4, s>>>(H, Is, blob, sc.hs,
                                                                         sc.gate, sc.ys);
  } else {
    up_kernel<MOE_W_BF16, true><<<gu, kThreads, (size_t)H * 4, s>>>(none, H, Is, 0, xx, nullptr,
                                                                    1, blob, gw, sc.hs, sc.gate);
    shared_down_kernel<MOE_W_BF16><<<gd, kThreads, (size_t)Is * 4, s>>>(H, Is, blob, sc.hs,
                                                                        sc.gate, sc.ys);
  }
  return cudaGetLastError();
}

cudaError_t launch_routed_up(const DevState& st, int wfmt, int H, int I, int layer,
                             const void* x, const int32_t* slot_ids, int n_rows, int k,
                             FfnScratch sc, cudaStream_t s) {
  const dim3 g((I + kWarps - 1) / kWarps, n_rows * k);
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  if (wfmt == MOE_W_NVFP4)
    up_kernel<MOE_W_NVFP4, false><<<g, kThreads, (size_t)H * 4, s>>>(st, H, I, layer, xx, slot_ids,
                                                                     k, nullptr, nullptr, sc.h,
                                                                     nullptr);
  else
    up_kernel<MOE_W_BF16, false><<<g, kThreads, (size_t)H * 4, s>>>(st, H, I, layer, xx, slot_ids,
                                                                    k, nullptr, nullptr, sc.h,
                                                                    nullptr);
  return cudaGetLastError();
}

cudaError_t launch_routed_down_combine(const DevState& st, int wfmt, int H, int I, int layer,
                                       const int32_t* slot_ids, const float* w, int n_rows,
                                       int k, const float* shared_y, void* out, FfnScratch sc,
                                       cudaStream_t s) {
  const dim3 g((H + kWarps - 1) / kWarps, n_rows);
  const size_t smem = (size_t)k * I * 4;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (wfmt == MOE_W_NVFP4)
    down_combine_kernel<MOE_W_NVFP4><<<g, kThreads, smem, s>>>(st, H, I, layer, slot_ids, w, k,
                                                               sc.h, shared_y, o);
  else
    down_combine_kernel<MOE_W_BF16><<<g, kThreads, smem, s>>>(st, H, I, layer, slot_ids, w, k,
                                                              sc.h, shared_y, o);
  return cudaGetLastError();
}

}  // namespace moe
