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
// running (programmatic dependent launch).  By default each warp waits for
// that kernel to complete before its first read of anything, x included:
// the kernel before this one in the stream may be the one writing x.  When
// the caller asserts that x was final before that kernel began (early_x:
// it is moe_plan, or another kernel that leaves x alone), each warp loads
// (fp8: and quantises) its first task first and only then waits for the
// plan's slots.  Tasks are software-pipelined:
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
// store is 16 bytes.
//
// Exact division, cheaply: q must be e4m3(RN(x / scale)).  With y =
// RN(1/scale), RN(x y) corrected once with the exact remainder is RN(x /
// scale) for every bf16 x and every scale in [2^-60, 2^60] (quot2_bf16 in
// moe_common.cuh; checked exhaustively on the CPU).  Blocks with scales
// outside that range divide every element.  The result is bit-identical to
// dividing every element.
#include <cuda_bf16.h>

#include "moe_dispatch_tasks.cuh"

namespace moe {

constexpr int kDispatchThreads = 256;


__device__ __forceinline__ Routes load_routes(const DispatchParams &p, int64_t g, int lane) {
  Routes r{-1, -1};
  if (lane < p.K) {
    r.e = __ldg(p.topk_idx + g * p.K + lane);
    r.s = __ldg(p.slot_of + g * p.K + lane);
  }
  return r;
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
// The same, with the warp's first routes loaded together with the status
// word, so that the two loads are in flight at once (fp8 at DeepSeek-V3
// decode, x read early: 12.55 -> 12.15 us; the bf16 kernel measured 0.7 us
// slower with it and reads the routes after the status).
__device__ __forceinline__ bool wait_plan_ok_routes(const DispatchParams &p, int64_t g, int lane,
                                                    Routes &r) {
  pdl_wait_for_previous();
  int32_t st = 0;
  if (lane == 0) st = read_status(p.hdr);
  r = load_routes(p, g, lane);
  return __shfl_sync(0xFFFFFFFFu, st, 0) == MOE_OK;
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

  // The first task's read of x needs nothing from the plan: with early_x it
  // is issued before waiting for the plan to finish.  Without, the previous
  // kernel may still be writing x, and the wait comes first.
  if (warp0 >= ntasks) return;
  if (!p.early_x) pdl_wait_for_previous();
  TaskCursor cur(warp0, nwarps, tpr);
  Bf16Task<U> t;
  bf16_load<U>(p, cur.g, cur.seg, lane, t);
  if (!wait_plan_ok(p.hdr, lane)) return;
  Routes r = load_routes(p, t.g, lane);
  // Software pipeline: the next task's loads go out before this task's stores.
  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t next = task + nwarps;
    const bool more = next < ntasks;
    cur = cur.next();
    Bf16Task<U> tn;
    Routes rn;
    if (more) {
      bf16_load<U>(p, cur.g, cur.seg, lane, tn);
      rn = load_routes(p, tn.g, lane);
    }
    bf16_store<U>(p, lane, t, r);
    if (more) {
      t = tn;
      r = rn;
    }
  }
}

// MINB: resident blocks per SM the registers are held to (3: 80 registers,
// 4: 64; see launch_dispatch_fp8).  SHORT: H % 128 != 0, the last block of a
// row is short (fp8_load, fp8_store).
template <int P, int MINB, bool SHORT = false>
__global__ void __launch_bounds__(kDispatchThreads, MINB)
dispatch_fp8_kernel(DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kDispatchThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDispatchThreads) >> 5;
  const int nb = SHORT ? (p.H + 127) / 128 : p.H / 128;      // blocks per row
  const int tpr = (nb + 2 * P - 1) / (2 * P);
  const int64_t ntasks = (int64_t)p.N * tpr;

  // The first task's read and quantisation of x need nothing from the plan:
  // with early_x they run before waiting for the plan to finish.  Then software-pipeline
  // the tasks: the next task's x and routing loads are issued before this
  // task's stores, and it is quantised while those stores drain.
  // (The token and segment of a task come from a division here: a
  // TaskCursor's registers would make this kernel spill at its 80.)
  // Without early_x the previous kernel may still be writing x: wait for it
  // before the first read.
  if (warp0 >= ntasks) return;
  if (!p.early_x) pdl_wait_for_previous();
  Fp8Raw<P> a;
  fp8_load<P, SHORT>(p, warp0 / tpr, (int)(warp0 % tpr), lane, a);
  Fp8Task<P> t;
  fp8_quantise<P>(a, lane, t);
  Routes r;
  if (!wait_plan_ok_routes(p, a.g, lane, r)) return;
  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int64_t next = task + nwarps;
    const bool more = next < ntasks;
    // The next kernel may start launching once every warp is on its last
    // task (measured: 13.5 -> 13.1 us alone, 12.5 us when reading x early,
    // at DeepSeek-V3 decode; the bf16 kernel measured slower with it).
    if (!more) pdl_allow_dependents();
    Routes rn;
    if (more) {
      const int64_t g = next / tpr;
      fp8_load<P, SHORT>(p, g, (int)(next - g * tpr), lane, a);
      rn = load_routes(p, g, lane);
    }
    fp8_store<P, SHORT>(p, lane, t, r);
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
  const bool short_blk = p.H % 128 != 0;
  const int nb = (p.H + 127) / 128;
  // a short last block: always kFp8MaxPairs block pairs per task
  const int P = (nb % 2 == 0 && !short_blk) ? pick_units(nb / 2, kFp8MaxPairs) : kFp8MaxPairs;
  const int64_t tasks = (int64_t)p.N * ((nb + 2 * P - 1) / (2 * P));
  if (P == 1) return launch_tasks(dispatch_fp8_kernel<1, 1>, tasks, p, stream);
  // More than 3 tasks per warp at 3 blocks per SM: 4 blocks per SM (64
  // registers, no spills).  Measured on GB300: 15.2 -> 14.1 us at the
  // Mixtral-shaped layer (4.5 tasks per warp), 52.6 -> 52.1 us at Kimi-K2
  // decode (7.9), but 13.45 -> 13.6 us at DeepSeek-V3 decode (2.0).
  const int64_t warps3 = (int64_t)device_sm_count() * 3 * (kDispatchThreads / 32);
  if (short_blk)
    return tasks > 3 * warps3 ? launch_tasks(dispatch_fp8_kernel<kFp8MaxPairs, 4, true>, tasks, p, stream)
                              : launch_tasks(dispatch_fp8_kernel<kFp8MaxPairs, 3, true>, tasks, p, stream);
  if (tasks > 3 * warps3) return launch_tasks(dispatch_fp8_kernel<kFp8MaxPairs, 4>, tasks, p, stream);
  return launch_tasks(dispatch_fp8_kernel<kFp8MaxPairs, 3>, tasks, p, stream);
}

}  // namespace moe
