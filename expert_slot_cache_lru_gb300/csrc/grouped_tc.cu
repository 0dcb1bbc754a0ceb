// grouped_tc.cu -- routed expert FFNs of wide steps on the tensor cores
// (tcgen05, accumulators in tensor memory).
//
// What is computed is the routed half of the layer, as in grouped.cu
// (FreeToken issue #753 "[Perf] Offloaded decode: overlap the expert-miss
// gather with the same layer's shared expert ...", Problem and What we changed;
// FreeToken PR #680 "fix(moe): admit a wide offloaded decode step's experts 128
// at a time", Tests: a wide step's routes over hundreds of distinct experts):
//   h[r]  = silu(W_g x_b) * (W_u x_b)            (r = b*k + j, slot[r] >= 0)
//   y[r]  = W_d h[r]
//   out[b] = bf16( sum_j w[b,j] y[b*k+j] + ys[b] ).
// A wide step routes a few rows to each of hundreds of experts.  Per expert
// the work is a small GEMM: the expert's weight rows against the activations
// of its routes.  Here each such GEMM runs as 128-row weight tiles (M) against
// up to 32 routes (N), with the weight tile as operand A and the routes'
// activations as operand B (K-major, both in shared memory, 128-byte swizzle),
// so that the tensor cores take the multiply-adds and the SMs only decode.
//
// Numbers (NVFP4 experts; the tcgen05 kind::f16 MMA with fp32 accumulation):
//   * A: each weight e2m1(code) * e4m3(scale) decoded to f16 -- exact (at most
//     6 significant bits, exponent within f16's normal range); the fp32 global
//     scale of the matrix multiplies the fp32 accumulator in the epilogue;
//   * B of gate/up: x as f16 with the row's power-of-two scale (xprep_kernel of
//     grouped.cu: a bf16 value below 2^15 converts exactly), undone in the
//     epilogue;
//   * B of down: h rounded to f16 after a per-route power-of-two scale that
//     puts max |h| in [2^14, 2^15) (hprep_kernel), undone in the epilogue --
//     the one rounding this path adds (relative 2^-11 of the route's max |h|).
//
// Kernel shape (one persistent CTA per SM, 13 warps):
//   warps 4..11  producers: for each K-slab of 64 elements, cp.async of the raw
//                codes (32 B per row), scales (4 B per row) and the B rows into
//                a ring of kNR raw stages, kNR - 2 slabs ahead; then decode the
//                raw slab into an operand stage (A: f16, 128 rows x 128 B,
//                swizzled; B: the raw B rows moved over) and signal it.  Slabs
//                go two at a time (a tile has an even number of them), so each
//                warp has two independent decode chains in flight per fence and
//                signal.  Every raw byte is copied and read by the same thread,
//                so a raw stage is free again once its thread has decoded it;
//   warp 12      lane 0 issues the MMAs (4 per slab, K = 16 each) and commits
//                their completion to the stages' "empty" barriers and, after a
//                tile's last slab, to the accumulator's "full" barrier; the
//                warp also allocates and frees the tensor memory;
//   warps 0..3   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//                lanes 32w..32w+31), scales, SiLU gating (gate/up) or the
//                down scales, and the stores.  Two accumulators alternate, so
//                the epilogue of one tile overlaps the MMAs of the next.
// Every wait is bounded (%globaltimer); a timeout sets MOE_STATUS_TIMEOUT,
// raises the CTA's abort flag, drains the copies in flight, and the kernel
// frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kEpiWarps = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kEpiWarps + kProdWarps;   // warp 12
constexpr int kThreads = 32 * (kMmaWarp + 1);      // 416
constexpr int kM = 128;                            // weight rows per tile (MMA M)
constexpr int kNMax = 32;                          // routes per tile (MMA N <= 32)
constexpr int kSlab = 64;                          // K elements per slab (128 B of f16)
constexpr int kNR = 8;                             // raw stages (copies in flight), in pairs
constexpr int kNP = kNR / 2;                       // raw stage pairs
constexpr int kNA = 6;                             // MMA operand stages (even)
constexpr int kRawB = kNMax * 128;                 // B rows of a raw stage (f16, swizzled)
constexpr int kRawC = kM * 32;                     // codes: 32 B per row
constexpr int kRawS = kM * 4;                      // scales: 4 B per row
constexpr int kRawStage = kRawB + kRawC + kRawS;   // 8704
constexpr int kATile = kM * 128;                   // decoded A: 16 KB
constexpr int kAStage = kATile + kRawB;            // A, then the B rows: 20 KB, 1024-multiple
constexpr int kTmemCols = 64;                      // two accumulators of kNMax columns
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;

static_assert(kRawStage % 1024 == 512 && kAStage % 1024 == 0 && kNR % 2 == 0 && kNA % 2 == 0,
              "stage sizes");

enum { kGateUp = 0, kDown = 1 };

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t sa(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups of
// 1024 bytes (stride byte offset), descriptor version 1, start address >> 4.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: D fp32, A and B f16, both K-major, N, M.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
      : "memory");
}
// 32 TMEM lanes x 16 columns of 32 bits: thread t of the warp gets lane
// (base lane + t), columns col .. col + 15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

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
// one E4M3 scale byte as a half2 with both halves equal
__device__ __forceinline__ uint32_t e4m3_h2(uint32_t byte) {
  uint32_t h2;
  const uint32_t v16 = byte | (byte << 8);
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(h2)
      : "r"(v16));
  return h2;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// eight e2m1 codes (one word, even element in the low nibble) times a block
// scale (half2): eight f16 values, exact
__device__ __forceinline__ uint4 dec8(uint32_t w, uint32_t sc2) {
  return make_uint4(hmul2(e2m1x2<0>(w), sc2), hmul2(e2m1x2<1>(w), sc2),
                    hmul2(e2m1x2<2>(w), sc2), hmul2(e2m1x2<3>(w), sc2));
}

// Byte offset of 16-byte chunk c (0..7) of row r in a K-major 128-byte-swizzled
// tile: rows are 128 B apart, chunk c of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Offsets inside an NVFP4 blob (layout of moe_cache.h).
struct Off {
  size_t code[3], scale[3], glob;
  __device__ Off(int H, int I) {
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

// The route groups buffer of the cache: [G, slot[R], start[R + 1], route[R]]
// (the dense groups' ids come from their own list).
struct Groups {
  const int32_t* base;
  int R;
  __device__ int slot(int g) const { return base[1 + g]; }
  __device__ int start(int g) const { return base[1 + R + g]; }
  __device__ int route(int q) const { return base[2 + 2 * R + q]; }
};

struct TcArgs {
  int H, I, k, layer;
  const int32_t* dense;  // [count, group ids ascending]: the groups these kernels take
  Groups gr;
  const uint16_t* act;   // B rows: x16 [rows][H] (gate/up) or h16 [routes][I] (down)
  const float* ainv;     // per B row: 1 / its power-of-two scale (xinv by row, hinv by route)
  float* out;            // gate/up: h [routes][I]; down: y [routes][H]
  unsigned long long* status;
};

// The sequence of tiles a CTA works on, identical for every role: items
// blockIdx.x, + gridDim.x, ... of (listed group, weight-row tile), and within
// an item the group's routes in chunks of kNMax.  What a tile needs from global
// memory (its group's range and slot, the B row a producer thread copies) is
// read once when the cursor reaches the tile, so the per-slab copies need no
// load of their own.
template <int KIND>
struct Cursor {
  const TcArgs* a;
  const DevState* st;
  int item, n_items, n_tiles;  // n_tiles: weight-row tiles per group
  int g, tile, q0, nq, rb;     // current group, tile, first route, routes in the chunk, group end
  int s, n_slab;               // slab within the tile
  int tid;                     // producer thread (0..255) whose B chunk this cursor tracks, or -1
  const uint8_t* blob;         // the group's expert blob
  const uint16_t* bsrc;        // tid's B row (its chunk's row of the chunk), or null
  bool valid;
  __device__ void init(const TcArgs& args, const DevState& state, int t) {
    a = &args;
    st = &state;
    tid = t;
    n_tiles = KIND == kGateUp ? args.I / 64 : args.H / kM;
    n_slab = (KIND == kGateUp ? args.H : args.I) / kSlab;
    n_items = args.dense[0] * n_tiles;
    item = blockIdx.x;
    valid = false;
    start_item();
  }
  __device__ void tile_info() {
    bsrc = nullptr;
    if (tid >= 0 && tid < nq * 8) {
      const int route = a->gr.route(q0 + (tid >> 3));
      const int brow = KIND == kGateUp ? route / a->k : route;
      bsrc = a->act + (size_t)brow * (KIND == kGateUp ? a->H : a->I) + (tid & 7) * 8;
    }
  }
  __device__ void start_item() {
    while (item < n_items) {
      const int d = item / n_tiles;
      g = a->dense[1 + d];
      tile = item - d * n_tiles;
      q0 = a->gr.start(g);
      rb = a->gr.start(g + 1);
      if (q0 < rb) {
        nq = min(kNMax, rb - q0);
        s = 0;
        valid = true;
        blob = st->slots + ((size_t)pool_of(*st, a->layer) * st->S + (size_t)a->gr.slot(g)) *
                               st->stride;
        tile_info();
        return;
      }
      item += gridDim.x;
    }
    valid = false;
  }
  // next route chunk (or next item)
  __device__ void next_tile() {
    q0 += kNMax;
    if (q0 < rb) {
      nq = min(kNMax, rb - q0);
      s = 0;
      tile_info();
      return;
    }
    item += gridDim.x;
    start_item();
  }
  __device__ void next_slab() {
    if (++s == n_slab) next_tile();
  }
};

struct Smem {
  uint64_t a_empty[kNA];
  uint64_t full[kNA];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;        // the MMA thread's last commit: every MMA of the CTA done
  uint32_t tmem_base;
  int abort_flag;
  int epi_ok;            // the epilogue's wait result, shared by its four warps
};

__device__ __forceinline__ void raise_abort(Smem* sm, unsigned long long* status) {
  if (atomicExch(&sm->abort_flag, 1) == 0 && status)
    atomicOr(status, (unsigned long long)MOE_STATUS_TIMEOUT);
}
// bounded wait; false on timeout or when another role gave up
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, Smem* sm,
                                         unsigned long long* status) {
  if (mbar_test(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  while (!mbar_test(b, parity)) {
    if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) return false;
    if (now_ns() - t0 > kWaitNs) {
      raise_abort(sm, status);
      return false;
    }
  }
  return true;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) tc_ffn_kernel(DevState st, TcArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* astg = dsm;                                 // [kNA][kAStage], 1024-aligned
  uint8_t* raw = astg + (size_t)kNA * kAStage;         // [kNR][kRawStage]
  float* ubuf = reinterpret_cast<float*>(raw + (size_t)kNR * kRawStage);  // [64][kNMax + 1]
  Smem* sm = reinterpret_cast<Smem*>(ubuf + 64 * (kNMax + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Off o(a.H, a.I);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&sm->a_empty[i], 1);
      mbar_init(&sm->full[i], kProdWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm->acc_full[i], 1);
      mbar_init(&sm->acc_empty[i], kEpiWarps);
    }
    mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sa(&sm->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp >= kEpiWarps && warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int t = threadIdx.x - 32 * kEpiWarps;  // 0 .. 255
    const int r = t >> 1, half = t & 1;          // A row and which 32 of its 64 elements
    Cursor<KIND> ld, dq;
    ld.init(a, st, t);
    dq.init(a, st, -1);
    const int cb = KIND == kGateUp ? a.H / 2 : a.I / 2;    // code bytes per weight row
    const int sbb = KIND == kGateUp ? a.H / 16 : a.I / 16; // scale bytes per weight row
    // raw copies of the slab at the load cursor into raw stage p
    auto issue = [&](int p) {
      uint8_t* st_ = raw + (size_t)p * kRawStage;
      const uint8_t* blob = ld.blob;
      size_t row;
      const uint8_t* cbase;
      const uint8_t* sbase;
      if (KIND == kGateUp) {  // rows 0-63: gate rows, 64-127: the same up rows
        row = (size_t)ld.tile * 64 + (r & 63);
        cbase = blob + (r < 64 ? o.code[0] : o.code[1]);
        sbase = blob + (r < 64 ? o.scale[0] : o.scale[1]);
      } else {
        row = (size_t)ld.tile * kM + r;
        cbase = blob + o.code[2];
        sbase = blob + o.scale[2];
      }
      cp16(st_ + kRawB + r * 32 + half * 16, cbase + row * cb + ld.s * 32 + half * 16);
      if (half == 0) cp4(st_ + kRawB + kRawC + r * 4, sbase + row * sbb + ld.s * 4);
      // B: chunk t of the nq rows (8 chunks of 16 B per row)
      if (ld.bsrc) cp16(st_ + swz(t >> 3, t & 7), ld.bsrc + ld.s * kSlab);
    };
    // decode raw stage ra into operand stage aa (this thread's row half and B chunk)
    auto decode = [&](int ra, int aa, bool bchunk) {
      const uint8_t* rs = raw + (size_t)ra * kRawStage;
      const uint4 cw = *reinterpret_cast<const uint4*>(rs + kRawB + r * 32 + half * 16);
      uint32_t scw = 0;
      if (half == 0) scw = *reinterpret_cast<const uint32_t*>(rs + kRawB + kRawC + r * 4);
      scw = __shfl_sync(0xffffffffu, scw, lane & ~1);
      const uint32_t s0 = e4m3_h2((scw >> (16 * half)) & 0xffu);
      const uint32_t s1 = e4m3_h2((scw >> (16 * half + 8)) & 0xffu);
      uint8_t* as = astg + (size_t)aa * kAStage;
      *reinterpret_cast<uint4*>(as + swz(r, half * 4 + 0)) = dec8(cw.x, s0);
      *reinterpret_cast<uint4*>(as + swz(r, half * 4 + 1)) = dec8(cw.y, s0);
      *reinterpret_cast<uint4*>(as + swz(r, half * 4 + 2)) = dec8(cw.z, s1);
      *reinterpret_cast<uint4*>(as + swz(r, half * 4 + 3)) = dec8(cw.w, s1);
      if (bchunk) {  // this thread's B chunk, raw stage -> operand stage
        const uint32_t off = swz(t >> 3, t & 7);
        *reinterpret_cast<uint4*>(as + kATile + off) = *reinterpret_cast<const uint4*>(rs + off);
      }
    };
    // the operand stage of slab jj is free once the MMAs of slab jj - kNA are
    // done (lane 0 waits; the warp takes its answer and stays converged)
    auto stage_free = [&](int jj) -> bool {
      bool w = true;
      if (jj >= kNA && lane == 0)
        w = wait_bar(&sm->a_empty[jj % kNA], (uint32_t)(((jj / kNA) - 1) & 1), sm, a.status);
      return __shfl_sync(0xffffffffu, w, 0);
    };
    bool ok = true;
#pragma unroll 1
    for (int p = 0; p < kNP - 1; ++p) {
      if (ld.valid) {
        issue(2 * p);
        ld.next_slab();
        issue(2 * p + 1);
        ld.next_slab();
      }
      cp_commit();
    }
#pragma unroll 1
    for (int j = 0; dq.valid && ok; j += 2) {
      // the pair kNP - 1 ahead goes into the stages this thread decoded last iteration
      if (ld.valid) {
        const int pp = (j / 2 + kNP - 1) % kNP;
        issue(2 * pp);
        ld.next_slab();
        issue(2 * pp + 1);
        ld.next_slab();
      }
      cp_commit();
      cp_wait<kNP - 1>();  // this thread's copies of slabs j, j + 1 have landed
      if (!stage_free(j) || !stage_free(j + 1)) {
        ok = false;
        break;
      }
      const bool bchunk = t < dq.nq * 8;  // slabs j and j + 1 belong to the same tile
      decode(j % kNR, j % kNA, bchunk);
      decode((j + 1) % kNR, (j + 1) % kNA, bchunk);
      fence_async_smem();  // this thread's A and B bytes, before the MMA reads them
      __syncwarp();        // one arrival per warp (256 arrivals on one word serialise)
      if (lane == 0) {
        mbar_arrive(&sm->full[j % kNA]);
        mbar_arrive(&sm->full[(j + 1) % kNA]);
      }
      dq.next_slab();
      dq.next_slab();
    }
    cp_wait_all();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Cursor<KIND> mc;
      mc.init(a, st, -1);
      int j = 0, u = 0;
      bool ok = true;
      uint64_t* last = nullptr;
      while (mc.valid && ok) {
        const int buf = u & 1;
        if (u >= 2 && !wait_bar(&sm->acc_empty[buf], (uint32_t)(((u >> 1) - 1) & 1), sm, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int N = mc.nq <= 16 ? 16 : 32;
        const uint32_t idesc = idesc_f16(kM, N);
        const uint32_t d = tmem + (uint32_t)(buf * kNMax);
        const int ns = mc.n_slab;
        for (int s = 0; s < ns; ++s, ++j) {
          const int aa = j % kNA;
          if (!wait_bar(&sm->full[aa], (uint32_t)((j / kNA) & 1), sm, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sa(astg + (size_t)aa * kAStage);
          const uint32_t b0 = a0 + kATile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(d, sdesc(a0 + kk * 32), sdesc(b0 + kk * 32), idesc, (s | kk) != 0);
          mma_commit(&sm->a_empty[aa]);
          last = &sm->a_empty[aa];
        }
        if (!ok) break;
        mma_commit(&sm->acc_full[buf]);
        ++u;
        mc.next_tile();
      }
      if (last) {  // every MMA issued has finished before the tensor memory is freed
        mma_commit(&sm->drain);  // (bounded, and taken even after an abort)
        const unsigned long long t0 = now_ns();
        while (!mbar_test(&sm->drain, 0) && now_ns() - t0 <= kWaitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp;  // 0..3: TMEM lanes 32*ew ..
    Cursor<KIND> ec;
    ec.init(a, st, -1);
    int u = 0;
    bool ok = true;
    while (ec.valid && ok) {
      const int buf = u & 1;
      // one thread waits and the four warps take its answer together (they
      // share a named barrier below)
      if (threadIdx.x == 0) {
        // a tile's MMAs take microseconds: poll slowly, leaving issue slots to the producers
        while (!mbar_test(&sm->acc_full[buf], (uint32_t)((u >> 1) & 1)) &&
               !*reinterpret_cast<volatile int*>(&sm->abort_flag))
          __nanosleep(256);
        sm->epi_ok = wait_bar(&sm->acc_full[buf], (uint32_t)((u >> 1) & 1), sm, a.status);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (!sm->epi_ok) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v0[16], v1[16];
      const uint32_t taddr = tmem + ((uint32_t)(32 * ew) << 16) + (uint32_t)(buf * kNMax);
      tmem_ld16(taddr, v0);
      if (ec.nq > 16) tmem_ld16(taddr + 16, v1);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->acc_empty[buf]);
      const float* gsc = reinterpret_cast<const float*>(ec.blob + o.glob);
      if (KIND == kGateUp) {
        // warps 2, 3 hold the up rows: through shared memory to warps 0, 1
        if (ew >= 2) {
#pragma unroll
          for (int n = 0; n < kNMax; ++n)
            if (n < ec.nq)
              ubuf[((ew - 2) * 32 + lane) * (kNMax + 1) + n] = __uint_as_float(n < 16 ? v0[n] : v1[n - 16]);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        if (ew < 2) {
          const float gs = gsc[0], us = gsc[1];
          const int i = ec.tile * 64 + ew * 32 + lane;
#pragma unroll
          for (int n = 0; n < kNMax; ++n) {
            if (n >= ec.nq) break;
            const int route = a.gr.route(ec.q0 + n);
            const float xi = a.ainv[route / a.k];
            const float g = __uint_as_float(n < 16 ? v0[n] : v1[n - 16]) * xi * gs;
            const float up = ubuf[(ew * 32 + lane) * (kNMax + 1) + n] * xi * us;
            a.out[(size_t)route * a.I + i] = g / (1.f + expf(-g)) * up;
          }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      } else {
        const float ds = gsc[2];
        const int row = ec.tile * kM + ew * 32 + lane;
#pragma unroll
        for (int n = 0; n < kNMax; ++n) {
          if (n >= ec.nq) break;
          const int route = a.gr.route(ec.q0 + n);
          a.out[(size_t)route * a.H + row] =
              __uint_as_float(n < 16 ? v0[n] : v1[n - 16]) * a.ainv[route] * ds;
        }
      }
      ++u;
      ec.next_tile();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// h [route][I] fp32 -> h16 (f16) with a per-route power-of-two scale that puts
// max |h| in [2^14, 2^15) (1 when the route's h is all zero), hinv = 1 / scale,
// for the routes of the listed groups.  One CTA per listed group, one warp per
// route at a time.
constexpr int kHT = 256;
__global__ void __launch_bounds__(kHT) hprep_kernel(TcArgs a, const float* __restrict__ h,
                                                    uint16_t* __restrict__ h16,
                                                    float* __restrict__ hinv) {
  if ((int)blockIdx.x >= a.dense[0]) return;
  const int g = a.dense[1 + blockIdx.x];
  const int I = a.I, lane = threadIdx.x & 31;
  for (int q = a.gr.start(g) + (threadIdx.x >> 5); q < a.gr.start(g + 1); q += kHT / 32) {
    const int route = a.gr.route(q);
    const float* hr = h + (size_t)route * I;
    float mx = 0.f;
    for (int i = lane; i < I; i += 32) mx = fmaxf(mx, fabsf(hr[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // 2^e with mx * 2^e in [2^14, 2^15): e = 14 - floor(log2(mx)), from the exponent bits
    float sc = 1.f;
    if (mx > 0.f && isfinite(mx)) {
      const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;  // floor(log2) for normals
      sc = ldexpf(1.f, min(max(14 - ex, -126), 127));
    }
    for (int i = lane; i < I; i += 32)
      h16[(size_t)route * I + i] = __half_as_ushort(__float2half_rn(hr[i] * sc));
    if (lane == 0) hinv[route] = 1.f / sc;
  }
}

size_t tc_smem_bytes() {
  return 1024 + (size_t)kNR * kRawStage + (size_t)kNA * kAStage + 64 * (kNMax + 1) * 4 +
         sizeof(Smem);
}

int g_tc_sms = 0;

}  // namespace

bool grouped_tc_supported(int wfmt, int H, int I) {
  // whole 128-row tiles of H, and an even number of 64-element slabs along H and I
  return wfmt == MOE_W_NVFP4 && H % kM == 0 && I % 128 == 0;
}

cudaError_t grouped_tc_init() {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_tc_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_ffn_kernel<kGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_ffn_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_bytes());
  return e;
}

// The gate/up and down GEMMs of the grouped path on the tensor cores, for the
// groups group_kernel listed in sc.dense; the route groups, that list and
// x16/xinv must already be written (group_kernel, xprep_kernel of grouped.cu).
// Leaves y [route][H] of those groups' routes for the combine.
cudaError_t launch_grouped_tc(const DevState& st, int H, int I, int layer, int k, int n_routes,
                              int max_routes, FfnScratch sc, unsigned long long* status,
                              cudaStream_t s) {
  TcArgs a{};
  a.dense = sc.dense;
  a.H = H;
  a.I = I;
  a.k = k;
  a.layer = layer;
  a.gr = Groups{st.groups, max_routes};
  a.status = status;
  const int grid = g_tc_sms > 0 ? g_tc_sms : 1;
  a.act = sc.x16;
  a.ainv = sc.xinv;
  a.out = sc.h;
  tc_ffn_kernel<kGateUp><<<grid, kThreads, tc_smem_bytes(), s>>>(st, a);
  if (n_routes > 0)  // at most one listed group per route
    hprep_kernel<<<n_routes, kHT, 0, s>>>(a, sc.h, sc.h16, sc.hinv);
  a.act = sc.h16;
  a.ainv = sc.hinv;
  a.out = sc.y;
  tc_ffn_kernel<kDown><<<grid, kThreads, tc_smem_bytes(), s>>>(st, a);
  return cudaGetLastError();
}

}  // namespace moe
