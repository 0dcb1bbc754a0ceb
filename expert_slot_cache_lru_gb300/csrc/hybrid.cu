// hybrid.cu -- the hybrid CPU executor: the routes a capped admission leaves
// at -1 are computed on the host's cores from the pinned host blobs while the
// GPU computes the others, and the two partial outputs are added.
//
// The order inside one layer follows FreeToken PR #491 ("refactor(moe):
// extract hybrid decode orchestration", section 4, "How decode works after
// this PR", and section 5, "How routes are split"): cache decision -> CPU
// submit -> GPU copy -> GPU experts -> CPU wait -> add the partial results.
// An all-GPU step still submits (an empty job) and waits, so a captured graph
// does not depend on the hit pattern.  The hand-off uses mapped pinned memory
// (the CUDA mechanism the PR names below its executor boundary):
//   - hybrid_post_kernel, right after the admission: copies the step's ids,
//     slot ids, weights and x into a mailbox in mapped host memory and
//     publishes a sequence number with a system-scope release store;
//   - a persistent host thread pool polls the sequence, computes the CPU
//     partial of the -1 routes in fp32 and publishes the same number back;
//   - hybrid_add_kernel, after the GPU's combine: waits (bounded, %globaltimer)
//     for that number and adds the CPU partial to the bf16 output.
// The host math is plain C++ (no intrinsics): every output value is computed
// by one task in a fixed order, so the result does not depend on the thread
// count.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <chrono>
#include <cmath>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace cpu {

// ---------------------------------------------------------------- number formats
// bf16 bits -> fp32 (exact)
inline float bf16f(uint16_t v) {
  const uint32_t u = (uint32_t)v << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// FP4 E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1, no inf / NaN): the
// sixteen codes as fp32, built from the bit fields.
struct E2m1Table {
  float v[16];
  E2m1Table() {
    for (int c = 0; c < 16; ++c) {
      const int e = (c >> 1) & 3, m = c & 1;
      const float mag = e == 0 ? 0.5f * m : std::ldexp(1.f + 0.5f * m, e - 1);
      v[c] = (c & 8) ? -mag : mag;
    }
  }
};
// FP8 E4M3 (1 sign, 4 exponent, 3 mantissa bits, bias 7; exponent 15 with
// mantissa 7 is NaN, there is no inf): the 256 codes as fp32.
struct E4m3Table {
  float v[256];
  E4m3Table() {
    for (int c = 0; c < 256; ++c) {
      const int e = (c >> 3) & 15, m = c & 7;
      float mag;
      if (e == 15 && m == 7)
        mag = NAN;
      else if (e == 0)
        mag = std::ldexp((float)m / 8.f, -6);
      else
        mag = std::ldexp(1.f + (float)m / 8.f, e - 7);
      v[c] = (c & 128) ? -mag : mag;
    }
  }
};
// E8M0 (the MXFP4 block scale: 8 exponent bits, bias 127; 255 is NaN).
struct E8m0Table {
  float v[256];
  E8m0Table() {
    for (int c = 0; c < 256; ++c) v[c] = c == 255 ? NAN : std::ldexp(1.f, c - 127);
  }
};
const E2m1Table kE2m1;
const E4m3Table kE4m3;
const E8m0Table kE8m0;

// ---------------------------------------------------------------- one expert
// Byte offsets of the banks of an expert blob (the layout of moe_cache.h).
struct Banks {
  size_t code[3], scale[3], glob;
  Banks(int H, int I, int fmt) {
    const size_t hi = (size_t)H * I, sb = hi / (fmt == MOE_W_MXFP4 ? 32 : 16);
    code[0] = 0;
    code[1] = hi / 2;
    code[2] = hi;
    scale[0] = 3 * hi / 2;
    scale[1] = scale[0] + sb;
    scale[2] = scale[1] + sb;
    glob = scale[2] + sb;
  }
};

// sum_{c < n} W[c] * x[c] for one bf16 row; n a multiple of 16.  Sixteen
// running sums (element c goes to sum c % 16), added pairwise at the end.
inline float dot_bf16(const uint16_t* w, const float* x, int n) {
  float acc[16] = {0.f};
  for (int c = 0; c < n; c += 16)
    for (int u = 0; u < 16; ++u) acc[u] += bf16f(w[c + u]) * x[c + u];
  for (int s = 8; s > 0; s >>= 1)
    for (int u = 0; u < s; ++u) acc[u] += acc[u + s];
  return acc[0];
}

// The same for one NVFP4 row: per block of 16 elements the e2m1 products are
// summed, then scaled by the block's e4m3 scale; the row's global scale is
// applied by the caller.  Blocks go to four running sums (block b to b % 4).
inline float dot_fp4(const uint8_t* codes, const uint8_t* scales, const float* x, int n) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int blk = 0; blk < n / 16; ++blk) {
    const uint8_t* c = codes + blk * 8;
    const float* xb = x + blk * 16;
    float s = 0.f;
    for (int u = 0; u < 8; ++u) {
      s += kE2m1.v[c[u] & 15] * xb[2 * u];
      s += kE2m1.v[c[u] >> 4] * xb[2 * u + 1];
    }
    acc[blk & 3] += s * kE4m3.v[scales[blk]];
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// The same for one MXFP4 row: per block of 32 elements the e2m1 products are
// summed, then scaled by the block's power of two; blocks go to four sums.
inline float dot_mx(const uint8_t* codes, const uint8_t* scales, const float* x, int n) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int blk = 0; blk < n / 32; ++blk) {
    const uint8_t* c = codes + blk * 16;
    const float* xb = x + blk * 32;
    float s = 0.f;
    for (int u = 0; u < 16; ++u) {
      s += kE2m1.v[c[u] & 15] * xb[2 * u];
      s += kE2m1.v[c[u] >> 4] * xb[2 * u + 1];
    }
    acc[blk & 3] += s * kE8m0.v[scales[blk]];
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// IEEE binary16 bits -> fp32 (exact), from the bit fields
inline float f16f(uint16_t v) {
  const int s = v >> 15, e = (v >> 10) & 31, m = v & 1023;
  float mag;
  if (e == 31)
    mag = m ? NAN : INFINITY;
  else if (e == 0)
    mag = std::ldexp((float)m, -24);
  else
    mag = std::ldexp(1.f + (float)m / 1024.f, e - 15);
  return s ? -mag : mag;
}

// The same for one Q4_0 row (banked): per block of 32 elements the products
// (q - 8) * x are summed, then scaled by the block's fp16 d; four sums.
inline float dot_q4(const uint8_t* codes, const uint8_t* scales, const float* x, int n) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int blk = 0; blk < n / 32; ++blk) {
    const uint8_t* c = codes + blk * 16;
    const float* xb = x + blk * 32;
    float s = 0.f;
    for (int u = 0; u < 16; ++u) {
      s += (float)((int)(c[u] & 15) - 8) * xb[2 * u];
      s += (float)((int)(c[u] >> 4) - 8) * xb[2 * u + 1];
    }
    uint16_t d;
    std::memcpy(&d, scales + 2 * blk, 2);
    acc[blk & 3] += s * f16f(d);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Row `r` of bank `which` (0 gate, 1 up: [I][H]; 2 down: [H][I]) dotted with x.
inline float row_dot(int wfmt, const uint8_t* blob, const Banks& bk, int H, int I, int which,
                     int r, const float* x) {
  const int n = which == 2 ? I : H;
  if (wfmt == MOE_W_BF16) {
    const uint16_t* m = reinterpret_cast<const uint16_t*>(blob) + (size_t)which * H * I;
    return dot_bf16(m + (size_t)r * n, x, n);
  }
  if (wfmt == MOE_W_Q4_0)
    return dot_q4(blob + bk.code[which] + (size_t)r * (n / 2),
                  blob + bk.scale[which] + (size_t)r * (n / 16), x, n);
  if (wfmt == MOE_W_MXFP4)
    return dot_mx(blob + bk.code[which] + (size_t)r * (n / 2),
                  blob + bk.scale[which] + (size_t)r * (n / 32), x, n);
  float g;
  std::memcpy(&g, blob + bk.glob + 4 * which, 4);
  return dot_fp4(blob + bk.code[which] + (size_t)r * (n / 2),
                 blob + bk.scale[which] + (size_t)r * (n / 16), x, n) * g;
}


// ---------------------------------------------------------------- one job
// The CPU partial of one step: for every route r = b*k + j with slot < 0 and
// a valid expert id,
//   h_r = silu(W_g x_b) * (W_u x_b)                     (phase A, fp32)
//   y[b] = sum over those routes of row b, j ascending, of w_r * (W_d h_r)
// (phase B; rows without such a route get 0).  Phase A is split into tasks of
// kRowsA rows of one route, phase B into tasks of kRowsB output rows of one
// batch row; tasks are claimed from atomic counters by any thread taking part.
constexpr int kRowsA = 32, kRowsB = 64;

struct Route {
  int b;                // batch row
  float w;              // routing weight
  const uint8_t* blob;  // host blob of its expert
};

struct Work {
  int wfmt = 0, H = 0, I = 0, n_rows = 0;
  std::vector<Route> routes;  // ascending route index
  std::vector<int> first;     // [n_rows + 1]: routes of row b are [first[b], first[b+1])
  const float* x = nullptr;   // [n_rows][H] fp32
  float* h = nullptr;         // [routes][I]
  float* y = nullptr;         // [n_rows][H] out
  int nA = 0, nB = 0, blkA = 0, blkB = 0;
  std::atomic<int> nextA{0}, nextB{0}, doneA{0}, doneB{0};

  // routes from the step's arrays; blob_of(e) gives expert e's host blob
  template <class BlobOf>
  void setup(int fmt, int hid, int inter, int rows, int k, const int32_t* ids,
             const int32_t* slots, const float* wts, int n_experts, BlobOf blob_of) {
    wfmt = fmt, H = hid, I = inter, n_rows = rows;
    routes.clear();
    first.assign((size_t)rows + 1, 0);
    for (int r = 0; r < rows * k; ++r) {
      const int e = ids[r];
      if (slots[r] >= 0 || e < 0 || e >= n_experts) continue;
      const uint8_t* blob = blob_of(e);
      if (!blob) continue;
      routes.push_back(Route{r / k, wts[r], blob});
      first[(size_t)r / k + 1] += 1;
    }
    for (int b = 0; b < rows; ++b) first[(size_t)b + 1] += first[b];
    blkA = (I + kRowsA - 1) / kRowsA;
    blkB = (H + kRowsB - 1) / kRowsB;
    nA = (int)routes.size() * blkA;
    nB = rows * blkB;
    nextA.store(0, std::memory_order_relaxed);
    nextB.store(0, std::memory_order_relaxed);
    doneA.store(0, std::memory_order_relaxed);
    doneB.store(0, std::memory_order_relaxed);
  }

  void task_a(int t) const {
    const int q = t / blkA, i0 = (t % blkA) * kRowsA, i1 = std::min(I, i0 + kRowsA);
    const Route& rt = routes[(size_t)q];
    const Banks bk(H, I, wfmt);
    const float* xb = x + (size_t)rt.b * H;
    for (int i = i0; i < i1; ++i) {
      const float g = row_dot(wfmt, rt.blob, bk, H, I, 0, i, xb);
      const float u = row_dot(wfmt, rt.blob, bk, H, I, 1, i, xb);
      h[(size_t)q * I + i] = g / (1.f + std::exp(-g)) * u;
    }
  }

  void task_b(int t) const {
    const int b = t / blkB, n0 = (t % blkB) * kRowsB, n1 = std::min(H, n0 + kRowsB);
    const Banks bk(H, I, wfmt);
    for (int n = n0; n < n1; ++n) {
      float acc = 0.f;
      for (int q = first[b]; q < first[(size_t)b + 1]; ++q)
        acc += routes[(size_t)q].w *
               row_dot(wfmt, routes[(size_t)q].blob, bk, H, I, 2, n, h + (size_t)q * I);
      y[(size_t)b * H + n] = acc;
    }
  }

  // take part until no task is left; phase-B tasks wait for the whole of phase A
  void run() {
    for (;;) {
      const int t = nextA.fetch_add(1, std::memory_order_relaxed);
      if (t >= nA) break;
      task_a(t);
      doneA.fetch_add(1, std::memory_order_release);
    }
    if (nextB.load(std::memory_order_relaxed) >= nB) return;
    while (doneA.load(std::memory_order_acquire) < nA) std::this_thread::yield();
    for (;;) {
      const int t = nextB.fetch_add(1, std::memory_order_relaxed);
      if (t >= nB) break;
      task_b(t);
      doneB.fetch_add(1, std::memory_order_release);
    }
  }

  bool complete() const { return doneB.load(std::memory_order_acquire) >= nB; }
};

// x rows as fp32
inline void widen_x(const uint16_t* x, int n, float* out) {
  for (int i = 0; i < n; ++i) out[i] = bf16f(x[i]);
}

// ---------------------------------------------------------------- mailbox
// One step's hand-off in mapped pinned host memory.  The header's two
// sequence words sit on their own 128-byte lines.
struct MailHeader {
  unsigned long long job_seq;   // written by the GPU: jobs posted
  unsigned long long pad0[15];
  unsigned long long done_seq;  // written by the host: the job whose y is complete
  unsigned long long pad1[15];
  int layer, n_rows, k, pad2;
};

inline size_t up16(size_t v) { return (v + 15) / 16 * 16; }

}  // namespace cpu

// byte offsets of the mailbox's arrays (passed to the kernels by value)
struct MailOff {
  size_t ids, slots, w, x, y, bytes;
  MailOff() = default;
  MailOff(int max_routes, int max_rows, int H) {
    ids = 512;
    slots = ids + cpu::up16((size_t)max_routes * 4);
    w = slots + cpu::up16((size_t)max_routes * 4);
    x = w + cpu::up16((size_t)max_routes * 4);
    y = x + cpu::up16((size_t)max_rows * H * 2);
    bytes = y + (size_t)max_rows * H * 4;
  }
};
static_assert(sizeof(cpu::MailHeader) <= 512, "mailbox header");

}  // namespace moe

// The executor: the mailbox, the device job counter and the host threads.
struct moe_cpu_exec {
  int wfmt = 0, H = 0, I = 0, E = 0, L = 0, max_rows = 0, max_routes = 0, n_threads = 0;
  std::vector<const uint8_t*> blobs;  // [L*E] host blob addresses
  uint8_t* mb = nullptr;              // mailbox, host address (mapped, pinned)
  bool host_only = false;             // self-test pool: mailbox in plain host memory, no GPU
  uint8_t* mb_dev = nullptr;          // the same, device address
  moe::MailOff off;
  unsigned long long* d_seq = nullptr;  // device: jobs posted so far
  std::vector<float> xf, h;
  moe::cpu::Work work;
  std::atomic<unsigned long long> gen{0};  // jobs handed to the workers
  std::atomic<unsigned long long> finished{0};  // worker passes over handed jobs
  std::atomic<bool> stop{false};
  std::atomic<bool> paused{false};  // test hook: jobs are left unanswered while set
  std::atomic<unsigned long long> jobs{0}, routes{0}, busy_ns{0};
  std::atomic<unsigned long long> busy_route_ns{0};  // ... of the jobs with -1 routes
  std::vector<std::thread> threads;

  moe::cpu::MailHeader* hdr() { return reinterpret_cast<moe::cpu::MailHeader*>(mb); }
};

namespace moe {
namespace cpu {

// Wait until ready() or stop: spin, then yield while jobs came recently, then
// sleep in 50 us steps.  False on stop.
template <class F>
bool wait_for(F ready, const std::atomic<bool>& stop) {
  using clk = std::chrono::steady_clock;
  const auto t0 = clk::now();
  for (int n = 0; !ready(); ++n) {
    if (stop.load(std::memory_order_relaxed)) return false;
    if (n < 256) continue;
    if (clk::now() - t0 < std::chrono::milliseconds(20))
      std::this_thread::yield();
    else
      std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  return true;
}

// Thread 0: takes each posted job from the mailbox, hands it to the workers
// (a worker never misses a job: the next one is handed out only after every
// worker has finished its pass over the current one), takes part, and
// publishes the job's number once every output row is written.
void coordinator(moe_cpu_exec* x) {
  MailHeader* hd = x->hdr();
  unsigned long long last = 0, handed = 0;
  const unsigned long long nw = (unsigned long long)x->n_threads - 1;
  for (;;) {
    unsigned long long seq = 0;
    // the job number first, then the pause flag: a pause set before a job was
    // posted is then always seen with that job
    if (!wait_for([&] {
          seq = __atomic_load_n(&hd->job_seq, __ATOMIC_ACQUIRE);
          return seq != last && !x->paused.load(std::memory_order_acquire);
        },
                  x->stop))
      return;
    if (!wait_for([&] { return x->finished.load(std::memory_order_acquire) >= handed * nw; },
                  x->stop))
      return;
    const auto t0 = std::chrono::steady_clock::now();
    const int layer = hd->layer, rows = hd->n_rows, k = hd->k;
    Work& w = x->work;
    if (layer >= 0 && layer < x->L && rows >= 0 && rows <= x->max_rows && k >= 0 &&
        (long long)rows * k <= x->max_routes) {
      const auto* ids = reinterpret_cast<const int32_t*>(x->mb + x->off.ids);
      const auto* slots = reinterpret_cast<const int32_t*>(x->mb + x->off.slots);
      const auto* wts = reinterpret_cast<const float*>(x->mb + x->off.w);
      const uint8_t* const* lb = x->blobs.data() + (size_t)layer * x->E;
      w.setup(x->wfmt, x->H, x->I, rows, k, ids, slots, wts, x->E, [&](int e) { return lb[e]; });
      widen_x(reinterpret_cast<const uint16_t*>(x->mb + x->off.x), rows * x->H, x->xf.data());
      w.x = x->xf.data();
      w.h = x->h.data();
      w.y = reinterpret_cast<float*>(x->mb + x->off.y);
    } else {  // a malformed header: an empty job
      w.setup(x->wfmt, x->H, x->I, 0, 0, nullptr, nullptr, nullptr, x->E,
              [](int) { return (const uint8_t*)nullptr; });
    }
    x->gen.store(++handed, std::memory_order_release);
    w.run();
    while (!w.complete()) std::this_thread::yield();
    const auto dt = (unsigned long long)std::chrono::duration_cast<std::chrono::nanoseconds>(
                        std::chrono::steady_clock::now() - t0).count();
    x->routes.fetch_add(w.routes.size(), std::memory_order_relaxed);
    x->jobs.fetch_add(1, std::memory_order_relaxed);
    x->busy_ns.fetch_add(dt, std::memory_order_relaxed);
    if (!w.routes.empty()) x->busy_route_ns.fetch_add(dt, std::memory_order_relaxed);
    __atomic_store_n(&hd->done_seq, seq, __ATOMIC_RELEASE);
    last = seq;
  }
}

void worker(moe_cpu_exec* x) {
  unsigned long long seen = 0;
  for (;;) {
    if (!wait_for([&] { return x->gen.load(std::memory_order_acquire) != seen; }, x->stop)) return;
    seen = x->gen.load(std::memory_order_acquire);
    x->work.run();
    x->finished.fetch_add(1, std::memory_order_release);
  }
}

// ---------------------------------------------------------------- kernels
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
constexpr unsigned long long kHostWaitNs = 1000000000ull;  // 1 s

// One CTA: the step into the mailbox, then its number (system-scope release).
__global__ void hybrid_post_kernel(uint8_t* mb, MailOff off, unsigned long long* d_seq, int layer,
                                   const int32_t* ids, const int32_t* slots, const float* w,
                                   const uint4* x, int R, int nx8, int n_rows, int k) {
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    reinterpret_cast<int32_t*>(mb + off.ids)[i] = ids[i];
    reinterpret_cast<int32_t*>(mb + off.slots)[i] = slots[i];
    reinterpret_cast<float*>(mb + off.w)[i] = w[i];
  }
  for (int i = threadIdx.x; i < nx8; i += blockDim.x) reinterpret_cast<uint4*>(mb + off.x)[i] = x[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    MailHeader* hd = reinterpret_cast<MailHeader*>(mb);
    const unsigned long long seq = *d_seq + 1;
    *d_seq = seq;
    hd->layer = layer;
    hd->n_rows = n_rows;
    hd->k = k;
    __threadfence_system();
    asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(&hd->job_seq), "l"(seq) : "memory");
  }
}

// out += the host's partial, once the host has published this job's number
// (bounded wait; on a timeout the output keeps the GPU partial and the status
// word gets MOE_STATUS_TIMEOUT).  Each thread takes 8 outputs at a time.
__global__ void hybrid_add_kernel(const uint8_t* mb, MailOff off, const unsigned long long* d_seq,
                                  uint16_t* out, int n8, unsigned long long* status) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    const MailHeader* hd = reinterpret_cast<const MailHeader*>(mb);
    const unsigned long long want = *d_seq, t0 = now_ns();
    int good = 0;
    for (;;) {
      unsigned long long v;
      asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(&hd->done_seq) : "memory");
      if (v >= want) {
        good = 1;
        break;
      }
      if (now_ns() - t0 > kHostWaitNs) {
        if (status) atomicOr(status, (unsigned long long)MOE_STATUS_TIMEOUT);
        break;
      }
      __nanosleep(1000);
    }
    ok = good;
  }
  __syncthreads();
  if (!ok) return;
  const float4* y = reinterpret_cast<const float4*>(mb + off.y);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
    uint4 o = reinterpret_cast<const uint4*>(out)[i];
    const float4 y0 = __ldcv(y + 2 * i), y1 = __ldcv(y + 2 * i + 1);
    const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
    uint32_t wv[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(wv[e] << 16) + yv[2 * e];
      const float hi = __uint_as_float(wv[e] & 0xffff0000u) + yv[2 * e + 1];
      const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
      wv[e] = *reinterpret_cast<const uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

}  // namespace cpu
}  // namespace moe

namespace moe {

cudaError_t hybrid_post(moe_cpu_exec* x, int layer, const int32_t* ids, const int32_t* slots,
                        const float* w, const void* xin, int n_rows, int k, cudaStream_t s) {
  cpu::hybrid_post_kernel<<<1, 256, 0, s>>>(x->mb_dev, x->off, x->d_seq, layer, ids, slots, w,
                                            static_cast<const uint4*>(xin), n_rows * k,
                                            n_rows * x->H / 8, n_rows, k);
  return cudaGetLastError();
}

cudaError_t hybrid_add(moe_cpu_exec* x, void* out, int n_rows, unsigned long long* status,
                       cudaStream_t s) {
  const int n8 = n_rows * x->H / 8;
  const int grid = std::min(16, std::max(1, (n8 + 255) / 256));
  cpu::hybrid_add_kernel<<<grid, 256, 0, s>>>(x->mb_dev, x->off, x->d_seq,
                                              static_cast<uint16_t*>(out), n8, status);
  return cudaGetLastError();
}

void hybrid_stop(moe_cpu_exec* x) {
  if (!x) return;
  x->stop.store(true, std::memory_order_relaxed);
  for (std::thread& t : x->threads)
    if (t.joinable()) t.join();
  if (x->mb && x->host_only) std::free(x->mb);
  if (x->mb && !x->host_only) cudaFreeHost(x->mb);
  if (x->d_seq) cudaFree(x->d_seq);
  delete x;
}

int hybrid_start(const HybridConfig& c, moe_cpu_exec** out, bool host_only) {
  moe_cpu_exec* x = new (std::nothrow) moe_cpu_exec();
  if (!x) return MOE_ERR_STATE;
  x->host_only = host_only;
  x->wfmt = c.wfmt, x->H = c.H, x->I = c.I, x->E = c.E, x->L = c.L;
  x->max_rows = c.max_rows, x->max_routes = c.max_routes, x->n_threads = c.n_threads;
  x->blobs.resize((size_t)c.L * c.E);
  for (size_t i = 0; i < x->blobs.size(); ++i)
    x->blobs[i] = static_cast<const uint8_t*>(c.host_blobs[i]);
  x->off = MailOff(c.max_routes, c.max_rows, c.H);
  cudaError_t e = cudaSuccess;
  if (host_only) {  // no device: the caller plays the GPU's part of the protocol
    x->mb = static_cast<uint8_t*>(std::aligned_alloc(4096, (x->off.bytes + 4095) / 4096 * 4096));
    if (!x->mb) {
      hybrid_stop(x);
      return MOE_ERR_STATE;
    }
    std::memset(x->mb, 0, x->off.bytes);
  } else if ((e = cudaHostAlloc(reinterpret_cast<void**>(&x->mb), x->off.bytes,
                                cudaHostAllocMapped)) == cudaSuccess) {
    std::memset(x->mb, 0, x->off.bytes);
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&x->mb_dev), x->mb, 0);
  } else {
    x->mb = nullptr;
  }
  if (e == cudaSuccess && !host_only)
    e = cudaMalloc(reinterpret_cast<void**>(&x->d_seq), sizeof(unsigned long long));
  if (e == cudaSuccess && !host_only) e = cudaMemset(x->d_seq, 0, sizeof(unsigned long long));
  if (e != cudaSuccess) {
    hybrid_stop(x);
    return -1000 - (int)e;  // the caller maps this to MOE_ERR_CUDA
  }
  x->xf.assign((size_t)c.max_rows * c.H, 0.f);
  x->h.assign((size_t)c.max_routes * c.I, 0.f);
  try {
    x->threads.emplace_back(cpu::coordinator, x);
    for (int i = 1; i < c.n_threads; ++i) x->threads.emplace_back(cpu::worker, x);
  } catch (...) {
    hybrid_stop(x);
    return MOE_ERR_STATE;
  }
  *out = x;
  return MOE_OK;
}

void hybrid_pause(moe_cpu_exec* x, bool paused) { x->paused.store(paused, std::memory_order_release); }

void hybrid_counters(const moe_cpu_exec* x, unsigned long long out[4]) {
  out[0] = x->jobs.load(std::memory_order_relaxed);
  out[1] = x->routes.load(std::memory_order_relaxed);
  out[2] = x->busy_ns.load(std::memory_order_relaxed);
  out[3] = x->busy_route_ns.load(std::memory_order_relaxed);
}

}  // namespace moe

extern "C" {

int moe_cpu_experts(int wfmt, int hidden, int inter, const void* const* h_blobs, int n_experts,
                    const uint16_t* h_x, const int32_t* h_ids, const int32_t* h_slot_ids,
                    const float* h_w, int n_rows, int k, int n_threads, float* h_out) {
  if (wfmt < MOE_W_BF16 || wfmt > MOE_W_Q4_0 || hidden <= 0 ||
      inter <= 0 || hidden % 32 ||
      inter % 32 || n_experts <= 0 || !h_blobs || n_rows < 0 || k < 0 || n_threads < 1 ||
      n_threads > 256)
    return MOE_ERR_INVALID_ARG;
  if (n_rows == 0) return MOE_OK;
  if (!h_x || !h_out || (k > 0 && (!h_ids || !h_slot_ids || !h_w))) return MOE_ERR_INVALID_ARG;
  moe::cpu::Work w;
  w.setup(wfmt, hidden, inter, n_rows, k, h_ids, h_slot_ids, h_w, n_experts,
          [&](int e) { return static_cast<const uint8_t*>(h_blobs[e]); });
  std::vector<float> xf((size_t)n_rows * hidden), h(w.routes.size() * (size_t)inter);
  moe::cpu::widen_x(h_x, n_rows * hidden, xf.data());
  w.x = xf.data();
  w.h = h.data();
  w.y = h_out;
  std::vector<std::thread> pool;
  try {
    for (int i = 1; i < n_threads; ++i) pool.emplace_back([&w] { w.run(); });
  } catch (...) {  // fewer threads than asked: the caller's thread finishes the work
  }
  w.run();
  for (std::thread& t : pool) t.join();
  return MOE_OK;
}

// Host-only self-test of the executor's job protocol: a pool over a mailbox in
// plain host memory, fed n_jobs random steps (rows, ids with some invalid,
// slots with about half at -1, weights, x) the way the post kernel feeds it,
// with a pause now and then; every answer is compared bit for bit with
// moe_cpu_experts on the same step.  *h_mismatches receives the number of
// differing output values; MOE_ERR_STATE if a job is not answered in 10 s.
int moe_hybrid_selftest(int wfmt, int hidden, int inter, const void* const* h_blobs,
                        int n_experts, int max_rows, int k, int n_threads, int n_jobs,
                        unsigned seed, long long* h_mismatches) {
  if (wfmt < MOE_W_BF16 || wfmt > MOE_W_Q4_0 || hidden <= 0 || inter <= 0 || hidden % 32 ||
      inter % 32 || n_experts <= 0 || !h_blobs || max_rows < 1 || k < 1 || n_threads < 1 ||
      n_threads > 256 || n_jobs < 0 || !h_mismatches)
    return MOE_ERR_INVALID_ARG;
  moe::HybridConfig hc{wfmt, hidden, inter, n_experts, 1, max_rows, max_rows * k, n_threads,
                       h_blobs};
  moe_cpu_exec* x = nullptr;
  int rc = moe::hybrid_start(hc, &x, true);
  if (rc != MOE_OK) return rc;
  moe::cpu::MailHeader* hd = x->hdr();
  auto* ids = reinterpret_cast<int32_t*>(x->mb + x->off.ids);
  auto* slots = reinterpret_cast<int32_t*>(x->mb + x->off.slots);
  auto* wts = reinterpret_cast<float*>(x->mb + x->off.w);
  auto* xin = reinterpret_cast<uint16_t*>(x->mb + x->off.x);
  const auto* y = reinterpret_cast<const float*>(x->mb + x->off.y);
  uint64_t r = 0x9E3779B97F4A7C15ull ^ seed;
  auto rnd = [&] {  // xorshift64*
    r ^= r >> 12, r ^= r << 25, r ^= r >> 27;
    return (uint32_t)((r * 0x2545F4914F6CDD1Dull) >> 32);
  };
  std::vector<float> ref((size_t)max_rows * hidden);
  long long bad = 0;
  for (int j = 1; j <= n_jobs && rc == MOE_OK; ++j) {
    const int rows = 1 + (int)(rnd() % (unsigned)max_rows);
    for (int q = 0; q < rows * k; ++q) {
      ids[q] = rnd() % 16 == 0 ? n_experts + (int)(rnd() % 3) : (int)(rnd() % (unsigned)n_experts);
      slots[q] = rnd() % 2 ? -1 : (int)(rnd() % 100);
      wts[q] = (float)(rnd() % 1000) / 1000.f;
    }
    for (int i = 0; i < rows * hidden; ++i)  // bf16 values in about [-2, 2)
      xin[i] = (uint16_t)((rnd() % 2 ? 0xC000u : 0x4000u) - 0x100u + (rnd() % 0x200u));
    hd->layer = 0, hd->n_rows = rows, hd->k = k;
    const bool pause = j % 97 == 0;
    if (pause) moe::hybrid_pause(x, true);
    __atomic_store_n(&hd->job_seq, (unsigned long long)j, __ATOMIC_RELEASE);
    if (pause) {
      std::this_thread::sleep_for(std::chrono::milliseconds(2));
      if (__atomic_load_n(&hd->done_seq, __ATOMIC_ACQUIRE) == (unsigned long long)j) ++bad;
      moe::hybrid_pause(x, false);
    }
    const auto t0 = std::chrono::steady_clock::now();
    while (__atomic_load_n(&hd->done_seq, __ATOMIC_ACQUIRE) != (unsigned long long)j) {
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10)) {
        rc = MOE_ERR_STATE;
        break;
      }
      std::this_thread::yield();
    }
    if (rc != MOE_OK) break;
    moe_cpu_experts(wfmt, hidden, inter, h_blobs, n_experts, xin, ids, slots, wts, rows, k, 1,
                    ref.data());
    bad += std::memcmp(ref.data(), y, (size_t)rows * hidden * 4) != 0;
  }
  moe::hybrid_stop(x);
  *h_mismatches = bad;
  return rc;
}

}  // extern "C"
