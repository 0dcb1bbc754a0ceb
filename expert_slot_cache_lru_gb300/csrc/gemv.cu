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
// (4-bit formats: 32 codes and their scales per lane per step; bf16: 32
// elements per lane per step), the activation vector sits in shared memory
// as fp32, and each warp reduces its row with shuffles.  Accumulation is fp32.
// NVFP4 blocks are 16 codes with an e4m3 scale and a global scale per matrix;
// MXFP4 blocks 32 e2m1 codes with an E8M0 power of two; Q4_0 blocks 32
// unsigned codes q with an fp16 scale d (weight d (q - 8)).
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <type_traits>

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

// sum_{i<8} (q_i - 8) * xs[i], q_i = nibble i of the word (element i)
__device__ __forceinline__ float dot8_q4(uint32_t w, const float* xs) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf((float)((int)((w >> (4 * i)) & 0xFu) - 8), xs[i], acc);
  return acc;
}
// an E8M0 scale: 2^(e - 127); 0xFF is NaN
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u)
                : (e == 255 ? __uint_as_float(0x7fffffffu) : __uint_as_float(e << 23));
}
__device__ __forceinline__ float f16_bits_to_f32(uint16_t v) { return __half2float(__ushort_as_half(v)); }

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

// Byte offsets inside a 4-bit blob (see the layouts in moe_cache.h): three
// code banks, then three scale banks of ih/16 bytes (NVFP4: e4m3 per 16;
// Q4_0: fp16 per 32) or ih/32 (MXFP4: E8M0 per 32), then NVFP4's globals.
struct Nvfp4Off {
  size_t code[3], scale[3], glob;
  __device__ Nvfp4Off(int H, int I, int fmt = MOE_W_NVFP4) {
    const size_t ih = (size_t)I * H;
    const size_t sb = ih / (fmt == MOE_W_MXFP4 ? 32 : 16);
    code[0] = 0;
    code[1] = ih / 2;
    code[2] = ih;
    scale[0] = 3 * ih / 2;
    scale[1] = scale[0] + sb;
    scale[2] = scale[1] + sb;
    glob = scale[2] + sb;
  }
};
// the scale of 32-element block j of a row of MXFP4 or Q4_0 scales
template <int FMT>
__device__ __forceinline__ float scale32(const uint8_t* scales, int j) {
  if (FMT == MOE_W_MXFP4) return e8m0_to_f32(scales[j]);
  return f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scales)[j]);
}
// 32 codes of a 4-bit row dotted with 32 fp32 activations, before the scale
template <int FMT>
__device__ __forceinline__ float dot32_codes(uint4 c, const float* x) {
  if (FMT == MOE_W_Q4_0)
    return (dot8_q4(c.x, x) + dot8_q4(c.y, x + 8)) + (dot8_q4(c.z, x + 16) + dot8_q4(c.w, x + 24));
  return (dot8_e2m1(c.x, x) + dot8_e2m1(c.y, x + 8)) + (dot8_e2m1(c.z, x + 16) + dot8_e2m1(c.w, x + 24));
}

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
  } else if (FMT == MOE_W_MXFP4 || FMT == MOE_W_Q4_0) {
    const Nvfp4Off o(H, I, FMT);
    const uint8_t* codes = blob + o.code[which] + (size_t)n * (K / 2);
    const uint8_t* scales = blob + o.scale[which] + (size_t)n * (K / 32) * (FMT == MOE_W_Q4_0 ? 2 : 1);
    for (int base = lane * 32; base < K; base += 1024) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + base / 2);
      acc = fmaf(dot32_codes<FMT>(c, xs + base), scale32<FMT>(scales, base / 32), acc);
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
  } else if (FMT == MOE_W_MXFP4 || FMT == MOE_W_Q4_0) {
    // 32-element blocks, one per lane per step (K a multiple of 32)
    const Nvfp4Off o(H, I, FMT);
    const uint8_t* codes = blob + o.code[which] + (size_t)n * (K / 2);
    const uint8_t* scales = blob + o.scale[which] + (size_t)n * (K / 32) * (FMT == MOE_W_Q4_0 ? 2 : 1);
    for (int base = lane * 32; base < K; base += 1024) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + base / 2);
      acc = fmaf(dot32_codes<FMT>(c, xs + base), scale32<FMT>(scales, base / 32), acc);
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
  return raise_smem_limit(kernel, bytes);
}

template <int FMT>
cudaError_t set_limits_fmt(size_t xb, size_t hb, size_t sb) {
  cudaError_t e = set_smem(up_kernel<FMT, false>, xb);
  if (e == cudaSuccess) e = set_smem(up_kernel<FMT, true>, xb);
  if (e == cudaSuccess) e = set_smem(down_combine_kernel<FMT>, hb);
  if (e == cudaSuccess) e = set_smem(shared_down_kernel<FMT>, sb);
  return e;
}

// f(std::integral_constant<int, FMT>) for the format wfmt
template <typename F>
cudaError_t by_format(int wfmt, F f) {
  switch (wfmt) {
    case MOE_W_NVFP4: return f(std::integral_constant<int, MOE_W_NVFP4>{});
    case MOE_W_MXFP4: return f(std::integral_constant<int, MOE_W_MXFP4>{});
    case MOE_W_Q4_0: return f(std::integral_constant<int, MOE_W_Q4_0>{});
    default: return f(std::integral_constant<int, MOE_W_BF16>{});
  }
}

}  // namespace

cudaError_t gemv_set_smem_limits(int H, int I, int Is, int k_max) {
  const size_t xb = (size_t)H * 4, hb = (size_t)k_max * I * 4, sb = (size_t)Is * 4;
  cudaError_t e = cudaSuccess;
  for (int f : {MOE_W_BF16, MOE_W_NVFP4, MOE_W_MXFP4, MOE_W_Q4_0})
    if (e == cudaSuccess)
      e = by_format(f, [&](auto fmt) { return set_limits_fmt<decltype(fmt)::value>(xb, hb, sb); });
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
  return by_format(wfmt, [&](auto fmt) {
    constexpr int F = decltype(fmt)::value;
    up_kernel<F, true><<<gu, kThreads, (size_t)H * 4, s>>>(none, H, Is, 0, xx, nullptr, 1, blob,
                                                           gw, sc.hs, sc.gate);
    shared_down_kernel<F><<<gd, kThreads, (size_t)Is * 4, s>>>(H, Is, blob, sc.hs, sc.gate, sc.ys);
    return cudaGetLastError();
  });
}

cudaError_t launch_routed_up(const DevState& st, int wfmt, int H, int I, int layer,
                             const void* x, const int32_t* slot_ids, int n_rows, int k,
                             FfnScratch sc, cudaStream_t s) {
  const dim3 g((I + kWarps - 1) / kWarps, n_rows * k);
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  return by_format(wfmt, [&](auto fmt) {
    up_kernel<decltype(fmt)::value, false><<<g, kThreads, (size_t)H * 4, s>>>(
        st, H, I, layer, xx, slot_ids, k, nullptr, nullptr, sc.h, nullptr);
    return cudaGetLastError();
  });
}

cudaError_t launch_routed_down_combine(const DevState& st, int wfmt, int H, int I, int layer,
                                       const int32_t* slot_ids, const float* w, int n_rows,
                                       int k, const float* shared_y, void* out, FfnScratch sc,
                                       cudaStream_t s) {
  const dim3 g((H + kWarps - 1) / kWarps, n_rows);
  const size_t smem = (size_t)k * I * 4;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  return by_format(wfmt, [&](auto fmt) {
    down_combine_kernel<decltype(fmt)::value><<<g, kThreads, smem, s>>>(st, H, I, layer, slot_ids,
                                                                        w, k, sc.h, shared_y, o);
    return cudaGetLastError();
  });
}

}  // namespace moe
