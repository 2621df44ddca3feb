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
// stores are issued (and, for fp8, while it is quantised).  A warp takes one (token, segment) task at a time
// from a grid sized to fill every SM; segments are chosen to divide the row
// evenly (1024 elements for H = 7168 or 4096), so all tasks are equal.  Its
// lanes read the segment once with 16-byte loads (all loads issued before
// any store), then write it K times with coalesced 16-byte (bf16) or 8-byte
// (fp8) stores.  In the fp8 path each half-warp owns one 128-element block:
// the absmax is a 4-step butterfly over 16 lanes, and the block's scale is
// computed once and shared by all K copies; the segment's scales are
// gathered into the first lanes and stored as one run per destination row.
//
// Exact division, cheaply: q must be e4m3(RN(x / scale)).  With r =
// RN(1/scale), q~ = RN(x * r) is within 3 binary32 ulps of RN(x / scale)
// (two roundings of 2^-24 each, plus half an ulp).  Rounding to E4M3 is
// monotone, so if q~ moved 4 ulps down and 4 ulps up rounds to the same
// byte, that byte is e4m3(RN(x / scale)); otherwise (a quotient next to an
// E4M3 midpoint, or a zero) the lane divides its 8 elements with IEEE
// __fdiv_rn, behind a warp-wide vote so that the division is a real branch
// taken only when needed.  The result is bit-identical to dividing every
// element.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

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

// Block-wide: wait for the plan (programmatic dependency), then read the
// status word it left; false if the block must write nothing.
__device__ __forceinline__ bool wait_plan_ok(const WsHeader *hdr) {
  __shared__ int32_t s_status;
  pdl_wait_for_previous();
  if (threadIdx.x == 0) s_status = read_status(hdr);
  __syncthreads();
  return s_status == MOE_OK;
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
  Bf16Task<U> t;
  if (warp0 < ntasks) bf16_load<U>(p, warp0, tpr, lane, t);
  if (!wait_plan_ok(p.hdr)) return;
  if (warp0 >= ntasks) return;
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
  uint2 q[P];
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

// Quantise one loaded task (needs nothing from the plan).
template <int P>
__device__ __forceinline__ void fp8_quantise(const Fp8Raw<P> &a, int lane, Fp8Task<P> &t) {
  t.g = a.g;
  t.seg = a.seg;
  t.my_scale = 0.0f;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const uint32_t w[4] = {a.v[it].x, a.v[it].y, a.v[it].z, a.v[it].w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_lo(w[i]);
      f[2 * i + 1] = bf16_hi(w[i]);
    }
    float scale;
    const uint2 q = quantise_block8(f, &scale);
    const uint32_t lo = q.x, hi = q.y;
    t.q[it] = make_uint2(lo, hi);
    const float s_even = __shfl_sync(kFull, scale, 0);
    const float s_odd = __shfl_sync(kFull, scale, 16);
    if (lane == it * 2) t.my_scale = s_even;
    if (lane == it * 2 + 1) t.my_scale = s_odd;
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
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const int blk = t.seg * bpt + it * 2 + half;
      if (blk < nb) *reinterpret_cast<uint2 *>(dst + (int64_t)blk * 128 + sub * 8) = t.q[it];
    }
    if (lane < nscale) p.expert_x_scale[row * nb + t.seg * bpt + lane] = t.my_scale;
  }
}

template <int P>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_fp8_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int nb = p.H / 128;                                  // blocks per row
  const int tpr = (nb + 2 * P - 1) / (2 * P);
  const int64_t ntasks = (int64_t)p.N * tpr;

  // The first task's read of x needs nothing from the plan: issue it before
  // waiting for the plan to finish.  Then software-pipeline the tasks: the
  // next task's x and routing loads are issued before this task's stores,
  // and it is quantised while those stores drain.
  Fp8Raw<P> a;
  if (warp0 < ntasks) fp8_load<P>(p, warp0, tpr, lane, a);
  if (!wait_plan_ok(p.hdr)) return;
  if (warp0 >= ntasks) return;
  Routes r = load_routes(p, a.g, lane);
  Fp8Task<P> t;
  fp8_quantise<P>(a, lane, t);
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
int pick_units(int units_per_row) {
  for (int u : {4, 2, 1})
    if (u <= MOE_MAX_UNITS && units_per_row % u == 0) return u;
  return MOE_MAX_UNITS;
}

}  // namespace

cudaError_t launch_dispatch_bf16(const DispatchParams &p, cudaStream_t stream) {
  const int cpr = p.H / 8;
  const int U = (cpr % 32 == 0) ? pick_units(cpr / 32) : MOE_MAX_UNITS;
  const int64_t tasks = (int64_t)p.N * ((cpr + 32 * U - 1) / (32 * U));
  switch (U) {
    case 1: return launch_tasks(dispatch_bf16_kernel<1>, tasks, p, stream);
    case 2: return launch_tasks(dispatch_bf16_kernel<2>, tasks, p, stream);
    default: return launch_tasks(dispatch_bf16_kernel<4>, tasks, p, stream);
  }
}

cudaError_t launch_dispatch_fp8(const DispatchParams &p, cudaStream_t stream) {
  const int nb = p.H / 128;
  const int P = (nb % 2 == 0) ? pick_units(nb / 2) : MOE_MAX_UNITS;
  const int64_t tasks = (int64_t)p.N * ((nb + 2 * P - 1) / (2 * P));
  switch (P) {
    case 1: return launch_tasks(dispatch_fp8_kernel<1>, tasks, p, stream);
    case 2: return launch_tasks(dispatch_fp8_kernel<2>, tasks, p, stream);
    default: return launch_tasks(dispatch_fp8_kernel<4>, tasks, p, stream);
  }
}

}  // namespace moe
