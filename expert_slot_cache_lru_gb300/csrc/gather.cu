// gather.cu -- the miss gather ("copy_missing"): copy every planned expert
// blob from pinned, mapped host memory into its device slot.
//
// [FreeToken issue #753 "[Perf] Offloaded decode: overlap the expert-miss
// gather with the same layer's shared expert ...", Problem and What we
// changed]: the gather reads only the miss plan written by the admission and
// writes only slot bytes; replay uses device-side miss counts, fixed
// addresses, no host sync.  A copy engine needs a host-known byte count, so
// inside a captured graph the copy is driven by the SMs: a fixed grid walks
// (plan entry, 64 KiB chunk) pairs read from the device count, each thread
// keeping four 16-byte loads from host memory in flight before it stores.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kGatherThreads = 256;
constexpr size_t kChunk = 64 * 1024;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_host_stream(const uint4* p) { return *p; }

__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(DevState st, const int32_t* plan) {
  const int n = plan[0];
  const size_t bytes = st.slot_bytes;
  const size_t per = (bytes + kChunk - 1) / kChunk;
  const size_t total = (size_t)n * per;
  for (size_t c = blockIdx.x; c < total; c += gridDim.x) {
    const size_t i = c / per, j = c % per;
    const int s = plan[1 + 3 * i], layer = plan[2 + 3 * i], e = plan[3 + 3 * i];
    if ((unsigned)s >= (unsigned)st.S || (unsigned)layer >= (unsigned)st.L ||
        (unsigned)e >= (unsigned)st.E)
      continue;  // never produced by the admission; skip rather than fault
    const size_t off = j * kChunk;
    const size_t len = (bytes - off) < kChunk ? (bytes - off) : kChunk;
    const uint4* src = reinterpret_cast<const uint4*>(st.host_blob[layer * st.E + e] + off);
    uint4* dst = reinterpret_cast<uint4*>(
        st.slots + ((size_t)pool_of(st, layer) * st.S + s) * st.stride + off);
    const size_t nv = len / 16;
    size_t v = threadIdx.x;
    for (; v + (kUnroll - 1) * kGatherThreads < nv; v += kUnroll * kGatherThreads) {
      uint4 t[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) t[u] = ld_host_stream(src + v + u * kGatherThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) dst[v + u * kGatherThreads] = t[u];
    }
    for (; v < nv; v += kGatherThreads) dst[v] = ld_host_stream(src + v);
  }
}

}  // namespace

cudaError_t launch_gather(const DevState& st, const int32_t* plan, int grid, cudaStream_t s) {
  gather_kernel<<<grid, kGatherThreads, 0, s>>>(st, plan);
  return cudaGetLastError();
}

}  // namespace moe
