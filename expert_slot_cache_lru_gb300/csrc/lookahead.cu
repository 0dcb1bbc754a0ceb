// lookahead.cu -- the look-ahead producer: the predicted expert ids of layer
// L + 1, produced while layer L runs.
//
// llama.cpp fork PR #126 "cuda : MoE look-ahead expert prefetch (PR-A
// consumer) + LFRU eviction guard", sections What and "Open for PR-P1
// (producer)": the consumer prefetches the next layer's experts from a list of
// predicted ids; the producer that fills the list is left open there.  This
// one applies layer L + 1's router to the hidden state layer L already has:
//   z[b][e] = sum_h W_r[e][h] x[b][h]     (bf16 operands, exact products,
//                                          fp32 sums in a fixed order)
//   pred[b][0 .. k) = the k experts of largest z[b][.], largest first, a tie
//                     going to the lower id (a NaN logit ranks below -inf).
// The prefetch admission takes the n_rows * k ids as they are (it removes the
// duplicates between rows).
//
// One launch: warp e of the grid computes expert e's logits for every row
// (its router row in registers, x in shared memory, rows in chunks), and the
// last CTA to finish (a counter that it resets) selects each row's top k,
// one warp per row: k rounds of "the largest key below the previous pick" over
// 64-bit keys (ordered logit bits, then the complement of the id), so no
// picked set is kept; up to 512 experts the keys stay in registers.  Nothing
// waits on another CTA.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kLaWarps = 4;
constexpr int kLaThreads = 32 * kLaWarps;
constexpr int kLaChunk = 8;  // rows of x in shared memory at a time (8 x H x 2 bytes)
constexpr int kLaReg = 16;   // logits a lane of the selecting warp keeps in registers

// the order of floats as unsigned integers (larger float, larger key); every
// NaN below -inf
__device__ __forceinline__ uint32_t ordered_bits(float z) {
  if (z != z) return 0u;
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long la_key(float z, int e) {
  return ((unsigned long long)ordered_bits(z) << 32) | (0xffffffffu - (uint32_t)e);
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// each lane holds H / 32 router weights as HV = H / 256 16-byte chunks
// (chunks lane, lane + 32, ...: one coalesced 512-byte load per warp per chunk)
template <int HV>
__global__ void __launch_bounds__(kLaThreads)
lookahead_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ router, int n_rows,
                 int E, int k, float* __restrict__ z, unsigned* __restrict__ ctr,
                 int32_t* __restrict__ pred) {
  constexpr int H = 256 * HV;
  extern __shared__ __align__(16) uint4 xsm[];  // [kLaChunk][H / 8] chunks of 8 bf16
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kLaWarps + warp;
  uint4 wr[HV];
  if (e < E) {
    const uint4* rp = reinterpret_cast<const uint4*>(router + (size_t)e * H);
#pragma unroll
    for (int j = 0; j < HV; ++j) wr[j] = rp[lane + 32 * j];
  }
  for (int b0 = 0; b0 < n_rows; b0 += kLaChunk) {
    const int nb = min(kLaChunk, n_rows - b0);
    __syncthreads();  // the previous chunk no longer read
    const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)b0 * H);
    for (int i = threadIdx.x; i < nb * (H / 8); i += kLaThreads) xsm[i] = xp[i];
    __syncthreads();
    if (e < E) {
      for (int r = 0; r < nb; ++r) {
        const uint4* xr = xsm + (size_t)r * (H / 8);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < HV; ++j) {
          const uint4 wq = wr[j], xq = xr[lane + 32 * j];
          const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w}, xv[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc = fmaf(__uint_as_float(wv[q] << 16), __uint_as_float(xv[q] << 16), acc);
            acc = fmaf(__uint_as_float(wv[q] & 0xffff0000u), __uint_as_float(xv[q] & 0xffff0000u),
                       acc);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) z[(size_t)(b0 + r) * E + e] = acc;
      }
    }
  }
  // the last CTA selects
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(ctr, 1u);
    s_last = old == gridDim.x - 1;
    if (s_last) *ctr = 0;  // every CTA has counted: ready for the next launch
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // up to 32 x kLaReg experts: each lane loads its keys once (one round trip)
  // and the k rounds run from registers; beyond that every round reads L2
  const bool in_regs = E <= 32 * kLaReg;
  for (int b = warp; b < n_rows; b += kLaWarps) {
    const float* zr = z + (size_t)b * E;
    unsigned long long kv[kLaReg];
    if (in_regs) {
#pragma unroll
      for (int j = 0; j < kLaReg; ++j) {
        const int i = lane + 32 * j;
        kv[j] = i < E ? la_key(__ldcg(zr + i), i) : 0ull;  // every real key is above 0
      }
    }
    unsigned long long prev = ~0ull;
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0ull;
      if (in_regs) {
#pragma unroll
        for (int j = 0; j < kLaReg; ++j)
          if (kv[j] < prev && kv[j] > best) best = kv[j];
      } else {
        for (int i = lane; i < E; i += 32) {
          const unsigned long long key = la_key(__ldcg(zr + i), i);
          if (key < prev && key > best) best = key;
        }
      }
      best = warp_max_u64(best);
      if (lane == 0) pred[(size_t)b * k + r] = (int32_t)(0xffffffffu - (uint32_t)(best & 0xffffffffu));
      prev = best;
    }
  }
}

}  // namespace

// H: a multiple of 1024 up to 4096 (the router row in registers)
bool lookahead_supported(int H, int E, int k) {
  return H >= 1024 && H <= 4096 && H % 1024 == 0 && E >= 1 && E <= 65536 && k >= 1 && k <= 32 &&
         k <= E;
}

namespace {
template <typename F>
cudaError_t by_width(int H, F f) {
  switch (H) {
    case 1024: return f(lookahead_kernel<4>);
    case 2048: return f(lookahead_kernel<8>);
    case 3072: return f(lookahead_kernel<12>);
    case 4096: return f(lookahead_kernel<16>);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

// the kernel's shared-memory limit for the cache's H (each H has its own
// kernel, so no other cache lowers it).  Set whatever its size: the static part
// counts against the default 48 KiB too.
cudaError_t lookahead_init(int H) {
  const size_t smem = (size_t)kLaChunk * H * 2;
  return by_width(H, [&](auto kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
}

cudaError_t launch_lookahead(const void* x, const void* router, int n_rows, int H, int E, int k,
                             float* z, unsigned* ctr, int32_t* pred, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const dim3 grid((E + kLaWarps - 1) / kLaWarps);
  const size_t smem = (size_t)kLaChunk * H * 2;
  const uint16_t* xx = static_cast<const uint16_t*>(x);
  const uint16_t* rr = static_cast<const uint16_t*>(router);
  return by_width(H, [&](auto kern) {
    kern<<<grid, kLaThreads, smem, s>>>(xx, rr, n_rows, E, k, z, ctr, pred);
    return cudaGetLastError();
  });
}

}  // namespace moe
