// moe_dispatch.cu -- row scatter of token activations into padded per-expert
// buffers, as a bf16 copy or fused with fp8 E4M3 1x128 block quantisation.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Dispatch; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", Quantization):
//   bf16:  expert_x[e][s][:] = x[g][:]            for every (g,k), e = idx, s = slot_of
//   fp8:   per 128-element block b of x[g]: scale = amax/448,
//          q = e4m3_rn_satfinite(x / scale) (all-zero block: scale 0, q 0);
//          the bytes and the H/128 scales go to every (e, s) of the token.
//
// How: work is cut by token, never by expert, so a skewed routing costs the
// same as a uniform one.  The kernel may start while moe_plan is still
// running (programmatic dependent launch): each warp loads its first task
// and only then waits for the plan's slots.  Tasks are software-pipelined:
// the next task's row and routing loads are in flight while this task's
// stores are issued (and, for fp8, while it is quantised).  A warp takes
// one (token, segment) task at a time from a grid sized to fill every SM;
// segments are chosen to divide the row evenly (1024 elements for H = 7168
// or 4096), so all tasks are equal.  Its
// lanes read the segment once with 16-byte loads (all loads issued before
// any store), then write it K times with coalesced 16-byte stores.  In the
// fp8 path each half-warp owns one 128-element block: the absmax is a 4-step
// butterfly over 16 lanes, and the block's scale (amax/448, exactly rounded)
// and its reciprocal are computed once, by the lane that stores the scale,
// and shared by all K copies; neighbouring lanes swap 8-byte halves so every
// store is 16 bytes.  The first task is read and quantised before waiting
// for the plan, which it does not need.
//
// Exact division, cheaply: q must be e4m3(RN(x / scale)).  With r =
// RN(1/scale), x * RN(r * (1 - 2^-20)) and x * RN(r * (1 + 2^-20)), rounded,
// bracket RN(x / scale) (three roundings of at most 2^-24 each cannot close
// a 2^-20 gap).  Rounding to E4M3 is monotone, so where both give the same
// byte, that byte is e4m3(RN(x / scale)); otherwise (a quotient next to an
// E4M3 midpoint, about 1 element in 200 for bf16 inputs) that element alone
// is divided with IEEE __fdiv_rn.  The result is bit-identical to dividing
// every element.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kDispatchThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}

// Routing of one token: lane k < K holds (expert, slot) of entry (g, k).
struct Routes {
  int e, s;
};

__device__ __forceinline__ Routes load_routes(const DispatchParams &p, int64_t g, int lane) {
  Routes r{-1, -1};
  if (lane < p.K) {
    r.e = __ldg(p.topk_idx + g * p.K + lane);
    r.s = __ldg(p.slot_of + g * p.K + lane);
  }
  return r;
}

// Mask of the routed, valid k.  slot -1 marks an entry the plan did not
// route (masked id, or a token beyond its rank's count): skipped silently.
// Other out-of-range entries are skipped and reported once per token.
__device__ __forceinline__ unsigned check_routes(const DispatchParams &p, const Routes &r, int lane,
                                                 bool report) {
  const bool routed = lane < p.K && r.s != -1;
  const bool e_ok = r.e >= 0 && r.e < p.E;
  const bool ok = routed && e_ok && r.s >= 0 && r.s < p.cap;
  if (report && routed && !ok)
    report_status(p.hdr, e_ok ? MOE_ERR_CAPACITY : MOE_ERR_BAD_EXPERT);
  return __ballot_sync(kFull, ok);
}

// Per warp: wait for the plan (programmatic dependency), then read the
// status word it left (one lane, broadcast); false if the warp must write
// nothing.  No block barrier: each warp leaves its pre-wait work on its own.
__device__ __forceinline__ bool wait_plan_ok(const WsHeader *hdr, int lane) {
  pdl_wait_for_previous();
  int32_t st = 0;
  if (lane == 0) st = read_status(hdr);
  return __shfl_sync(0xFFFFFFFFu, st, 0) == MOE_OK;
}

// bf16 copy; U 16-byte chunks per lane per task (a 256*U-element segment).
template <int U>
struct Bf16Task {
  int64_t g;
  int seg;
  uint4 v[U];
};

template <int U>
__device__ __forceinline__ void bf16_load(const DispatchParams &p, int64_t task, int tpr, int lane,
                                          Bf16Task<U> &t) {
  const int cpr = p.H / 8;
  t.g = task / tpr;
  t.seg = (int)(task - t.g * tpr);
  const uint16_t *src = p.x + t.g * p.H;
  const int c0 = t.seg * 32 * U + lane;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = c0 + u * 32;
    t.v[u] = c < cpr ? ld_stream16(src + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
  }
}

template <int U>
__device__ __forceinline__ void bf16_store(const DispatchParams &p, int lane, const Bf16Task<U> &t,
                                           const Routes &r) {
  const int cpr = p.H / 8;
  const unsigned okmask = check_routes(p, r, lane, t.seg == 0);
  const int c0 = t.seg * 32 * U + lane;
  for (int k = 0; k < p.K; ++k) {
    const int e = __shfl_sync(kFull, r.e, k);
    const int s = __shfl_sync(kFull, r.s, k);
    if (!((okmask >> k) & 1u)) continue;
    uint16_t *dst = static_cast<uint16_t *>(p.expert_x) + ((int64_t)e * p.cap + s) * p.H;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < cpr) *reinterpret_cast<uint4 *>(dst + (int64_t)c * 8) = t.v[u];
    }
  }
}

template <int U>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_bf16_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int cpr = p.H / 8;                               // 16-byte chunks per row
  const int tpr = (cpr + 32 * U - 1) / (32 * U);         // tasks per row
  const int64_t ntasks = (int64_t)p.N * tpr;

  // The first task's read of x needs nothing from the plan: issue it before
  // waiting for the plan to finish.
  if (warp0 >= ntasks) return;
  Bf16Task<U> t;
  bf16_load<U>(p, warp0, tpr, lane, t);
  if (!wait_plan_ok(p.hdr, lane)) return;
  Routes r = load_routes(p, t.g, lane);
  // Software pipeline: the next task's loads go out before this task's stores.
  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t next = task + nwarps;
    const bool more = next < ntasks;
    Bf16Task<U> tn;
    Routes rn;
    if (more) {
      bf16_load<U>(p, next, tpr, lane, tn);
      rn = load_routes(p, tn.g, lane);
    }
    bf16_store<U>(p, lane, t, r);
    if (more) {
      t = tn;
      r = rn;
    }
  }
}

// fp8 quantisation; P pairs of 128-element blocks per task.
template <int P>
struct Fp8Raw {      // one task's input, as loaded
  int64_t g;
  int seg;
  uint4 v[P];
};

template <int P>
struct Fp8Task {     // one task's output
  int64_t g;
  int seg;
  uint2 q[P];       // this lane's 8 bytes of block seg*2P + 2*it + half
  uint4 w16[P / 2 > 0 ? P / 2 : 1];   // P even: 16 bytes per lane pair (see fp8_quantise)
  float my_scale;   // lane L < 2P holds the scale of block seg*2P + L
};

template <int P>
__device__ __forceinline__ void fp8_load(const DispatchParams &p, int64_t task, int tpr, int lane,
                                         Fp8Raw<P> &a) {
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int nb = p.H / 128;
  a.g = task / tpr;
  a.seg = (int)(task - a.g * tpr);
  const uint16_t *src = p.x + a.g * p.H;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const int blk = a.seg * 2 * P + it * 2 + half;
    a.v[it] = blk < nb ? ld_stream16(src + (int64_t)blk * 128 + sub * 8) : make_uint4(0, 0, 0, 0);
  }
}

// Quantise one loaded task (needs nothing from the plan).  Each block's
// scale and reciprocal are computed once, by the lane that stores the scale
// (lane L < 2P owns block seg*2P + L), and handed to the half-warp that
// quantises the block by shuffle.  All 32 lanes call it together.
template <int P>
__device__ __forceinline__ void fp8_quantise(const Fp8Raw<P> &a, int lane, Fp8Task<P> &t) {
  const int half = lane >> 4;
  t.g = a.g;
  t.seg = a.seg;
  float am[P];
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const uint32_t w[4] = {a.v[it].x, a.v[it].y, a.v[it].z, a.v[it].w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_lo(w[i]);
      f[2 * i + 1] = bf16_hi(w[i]);
    }
    am[it] = half_warp_amax(f);
  }
  float mine = 0.0f;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const float v = __shfl_sync(kFull, am[it], (lane & 1) * 16);
    if ((lane >> 1) == it) mine = v;
  }
  float my_scale = div448_fast(mine);
  const bool odd = mine != 0.0f && !(mine >= 0x1p-120f && mine <= 3.4028234e38f);
  if (__any_sync(kFull, odd)) {
    if (odd) my_scale = __fdiv_rn(mine, 448.0f);
  }
  const float my_r = mine == 0.0f ? 1.0f : __frcp_rn(my_scale);
  t.my_scale = my_scale;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const uint32_t w[4] = {a.v[it].x, a.v[it].y, a.v[it].z, a.v[it].w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_lo(w[i]);
      f[2 * i + 1] = bf16_hi(w[i]);
    }
    const float scale = __shfl_sync(kFull, my_scale, it * 2 + half);
    const float r = __shfl_sync(kFull, my_r, it * 2 + half);
    t.q[it] = quant_bytes8(f, scale, r, am[it] == 0.0f);
  }
  // Pair neighbouring lanes for 16-byte stores: for each pair of iterations
  // (2j, 2j+1), the even lane of a pair gets iteration 2j's bytes of both
  // lanes and the odd lane iteration 2j+1's.
  if constexpr (P % 2 == 0) {
#pragma unroll
    for (int j = 0; j < P / 2; ++j) {
      const bool even = (lane & 1) == 0;
      const uint2 give = even ? t.q[2 * j + 1] : t.q[2 * j];
      uint2 got;
      got.x = __shfl_xor_sync(kFull, give.x, 1);
      got.y = __shfl_xor_sync(kFull, give.y, 1);
      const uint2 keep = even ? t.q[2 * j] : t.q[2 * j + 1];
      t.w16[j] = even ? make_uint4(keep.x, keep.y, got.x, got.y) : make_uint4(got.x, got.y, keep.x, keep.y);
    }
  }
}

// Write one quantised task to every (expert, slot) of its token.
template <int P>
__device__ __forceinline__ void fp8_store(const DispatchParams &p, int lane, const Fp8Task<P> &t,
                                          const Routes &r) {
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int nb = p.H / 128;
  constexpr int bpt = 2 * P;
  const unsigned okmask = check_routes(p, r, lane, t.seg == 0);
  const int nscale = min(bpt, nb - t.seg * bpt);
  for (int k = 0; k < p.K; ++k) {
    const int e = __shfl_sync(kFull, r.e, k);
    const int s = __shfl_sync(kFull, r.s, k);
    if (!((okmask >> k) & 1u)) continue;
    const int64_t row = (int64_t)e * p.cap + s;
    uint8_t *dst = static_cast<uint8_t *>(p.expert_x) + row * p.H;
    if constexpr (P % 2 == 0) {
      // lane pair (sub & ~1, sub | 1) writes 16 bytes at (sub & ~1) * 8 of
      // block 2j (even lane) or 2j + 1 (odd lane) of its half
#pragma unroll
      for (int j = 0; j < P / 2; ++j) {
        const int blk = t.seg * bpt + (2 * j + (lane & 1)) * 2 + half;
        if (blk < nb)
          *reinterpret_cast<uint4 *>(dst + (int64_t)blk * 128 + (sub & ~1) * 8) = t.w16[j];
      }
    } else {
#pragma unroll
      for (int it = 0; it < P; ++it) {
        const int blk = t.seg * bpt + it * 2 + half;
        if (blk < nb) *reinterpret_cast<uint2 *>(dst + (int64_t)blk * 128 + sub * 8) = t.q[it];
      }
    }
    if (lane < nscale) p.expert_x_scale[row * nb + t.seg * bpt + lane] = t.my_scale;
  }
}

template <int P>
__global__ void __launch_bounds__(kDispatchThreads, P >= 4 ? 3 : 1)
dispatch_fp8_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int nb = p.H / 128;                                  // blocks per row
  const int tpr = (nb + 2 * P - 1) / (2 * P);
  const int64_t ntasks = (int64_t)p.N * tpr;

  // The first task's read and quantisation of x need nothing from the plan:
  // they run before waiting for the plan to finish.  Then software-pipeline
  // the tasks: the next task's x and routing loads are issued before this
  // task's stores, and it is quantised while those stores drain.
  if (warp0 >= ntasks) return;
  Fp8Raw<P> a;
  fp8_load<P>(p, warp0, tpr, lane, a);
  Fp8Task<P> t;
  fp8_quantise<P>(a, lane, t);
  if (!wait_plan_ok(p.hdr, lane)) return;
  Routes r = load_routes(p, a.g, lane);
  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t next = task + nwarps;
    const bool more = next < ntasks;
    Routes rn;
    if (more) {
      fp8_load<P>(p, next, tpr, lane, a);
      rn = load_routes(p, next / tpr, lane);
    }
    fp8_store<P>(p, lane, t, r);
    if (more) {
      fp8_quantise<P>(a, lane, t);
      r = rn;
    }
  }
}

namespace {

// One persistent-grid launch of `kern` over `warp_tasks` equal tasks, allowed
// to start while the plan that precedes it in the stream is still running.
cudaError_t launch_tasks(void (*kern)(DispatchParams), int64_t warp_tasks, const DispatchParams &p,
                         cudaStream_t stream) {
  const int grid = persistent_grid((const void *)kern, kDispatchThreads, warp_tasks);
  return launch_after_previous(kern, grid, kDispatchThreads, p, stream);
}

// Segment size: the largest of 4, 2, 1 units that divides the row evenly
// (4 when nothing does; the last task of a row is then partial).
#ifndef MOE_MAX_UNITS
#define MOE_MAX_UNITS 4
#endif
int pick_units(int units_per_row, int max_units) {
  for (int u : {4, 2, 1})
    if (u <= max_units && units_per_row % u == 0) return u;
  return max_units;
}

// The fp8 path takes up to 4 block pairs per task, with the kernel held to
// 3 resident blocks per SM (80 registers): unbounded it needs 90 and runs 2
// blocks per SM.  Measured at DeepSeek-V3 decode, alternating builds: 4
// pairs at 3 blocks 14.8 us alone and 18.8 us after the plan; 2 pairs
// 16.9 and 21.2 us.
#ifndef MOE_FP8_MAX_PAIRS
#define MOE_FP8_MAX_PAIRS 4
#endif
constexpr int kFp8MaxPairs = MOE_MAX_UNITS < MOE_FP8_MAX_PAIRS ? MOE_MAX_UNITS : MOE_FP8_MAX_PAIRS;

}  // namespace

cudaError_t launch_dispatch_bf16(const DispatchParams &p, cudaStream_t stream) {
  const int cpr = p.H / 8;
  const int U = (cpr % 32 == 0) ? pick_units(cpr / 32, MOE_MAX_UNITS) : MOE_MAX_UNITS;
  const int64_t tasks = (int64_t)p.N * ((cpr + 32 * U - 1) / (32 * U));
  switch (U) {
    case 1: return launch_tasks(dispatch_bf16_kernel<1>, tasks, p, stream);
    case 2: return launch_tasks(dispatch_bf16_kernel<2>, tasks, p, stream);
    default: return launch_tasks(dispatch_bf16_kernel<4>, tasks, p, stream);
  }
}

cudaError_t launch_dispatch_fp8(const DispatchParams &p, cudaStream_t stream) {
  const int nb = p.H / 128;
  const int P = (nb % 2 == 0) ? pick_units(nb / 2, kFp8MaxPairs) : kFp8MaxPairs;
  const int64_t tasks = (int64_t)p.N * ((nb + 2 * P - 1) / (2 * P));
  if (P == 1) return launch_tasks(dispatch_fp8_kernel<1>, tasks, p, stream);
  return launch_tasks(dispatch_fp8_kernel<kFp8MaxPairs>, tasks, p, stream);
}

}  // namespace moe
