// admit.cu -- the standalone admission and prefetch kernels (one CTA of 1024
// threads per call; no host synchronisation, fixed launch shape, so both
// capture into CUDA graphs at any width), rollback and pinning.  The
// algorithms live in admit_body.cuh.
#include "admit_body.cuh"

namespace moe {
namespace {

using namespace admission;

template <bool CACHED>
__global__ void __launch_bounds__(kAdmitThreads, 1)
admit_kernel(DevState st, int layer, const int32_t* ids, int32_t* out, int R, int cap) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ AdmitShared<kAdmitThreads> sh;
  admit_body<CACHED, kAdmitThreads>(st, layer, ids, out, R, cap, smem_raw, sh, [] {});
}

__global__ void __launch_bounds__(kAdmitThreads, 1)
prefetch_kernel(DevState st, int layer, const int32_t* pred, int n, int32_t* plan) {
  extern __shared__ int smem_i[];
  __shared__ AdmitShared<kAdmitThreads> sh;
  prefetch_body<kAdmitThreads>(st, layer, pred, n, plan, smem_i, sh);
}

__global__ void rollback_kernel(DevState st, int32_t* plan) {
  const int n = plan[0];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int s = plan[1 + 3 * i], layer = plan[2 + 3 * i], e = plan[3 + 3 * i];
    if ((unsigned)layer >= (unsigned)st.L || (unsigned)s >= (unsigned)st.S ||
        (unsigned)e >= (unsigned)st.E)
      continue;
    const size_t g = (size_t)pool_of(st, layer) * st.S + s;
    const int key = layer * st.E + e;
    if (st.slot_key[g] != key) continue;
    st.map[key] = -1;
    st.slot_key[g] = -1;
    st.stamp[g] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) plan[0] = 0;
}

__global__ void pin_kernel(DevState st, size_t g, int v) { st.pinned[g] = (uint8_t)v; }

}  // namespace

// Dynamic shared memory of an admission: [E] x 3 counters, plus the pool's
// victim keys and slot keys when the pool is small enough to keep.
constexpr size_t kAdmitCacheMax = 200 * 1024;
bool admit_cached(int E, int S) { return (size_t)S * 12 + 3ull * E * 4 <= kAdmitCacheMax; }
size_t admit_smem_bytes(int E, int S) {
  return 3ull * E * sizeof(int) + (admit_cached(E, S) ? (size_t)S * 12 : 0);
}

cudaError_t launch_admit(const DevState& st, int layer, const int32_t* ids, int32_t* out, int R,
                         int cap, cudaStream_t s) {
  const size_t smem = admit_smem_bytes(st.E, st.S);
  if (admit_cached(st.E, st.S))
    admit_kernel<true><<<1, kAdmitThreads, smem, s>>>(st, layer, ids, out, R, cap);
  else
    admit_kernel<false><<<1, kAdmitThreads, smem, s>>>(st, layer, ids, out, R, cap);
  return cudaGetLastError();
}

cudaError_t launch_prefetch(const DevState& st, int layer, const int32_t* pred, int n,
                            int32_t* plan, cudaStream_t s) {
  prefetch_kernel<<<1, kAdmitThreads, 2ull * st.E * sizeof(int), s>>>(st, layer, pred, n, plan);
  return cudaGetLastError();
}

cudaError_t launch_rollback(const DevState& st, const int32_t* plan, cudaStream_t s) {
  rollback_kernel<<<1, 256, 0, s>>>(st, const_cast<int32_t*>(plan));
  return cudaGetLastError();
}

cudaError_t launch_pin(const DevState& st, int layer, int slot, int pinned, cudaStream_t s) {
  pin_kernel<<<1, 1, 0, s>>>(st, (size_t)pool_of(st, layer) * st.S + slot, pinned);
  return cudaGetLastError();
}

cudaError_t admit_set_smem_limits(int E, int S) {
  cudaError_t e = raise_smem_limit(admit_kernel<true>, admit_smem_bytes(E, S));
  if (e == cudaSuccess) e = raise_smem_limit(admit_kernel<false>, admit_smem_bytes(E, S));
  if (e != cudaSuccess) return e;
  return raise_smem_limit(prefetch_kernel, 2ull * E * sizeof(int));
}

}  // namespace moe
