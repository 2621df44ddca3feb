// moe_common.cuh -- definitions shared by the kernels and the C ABI of
// libmoe_gb300.so: workspace layout, plan geometry, launch parameters and a
// few PTX helpers (acquire/release flags, the global timer).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_dispatch.h"

namespace moe {

// ---------------------------------------------------------------------------
// Plan geometry.  The routed entries are cut into tiles of whole tokens that
// never straddle a rank boundary, so that rank r's offsets are the exclusive
// prefix of tile (r, 0).  One thread block handles one tile.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 512;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanTileEntries = 1024;                          // entries (g,k) per tile, at most
constexpr int kPlanBatchesPerWarp = kPlanTileEntries / (32 * kPlanWarps);  // 2
constexpr int kMaxExperts = 2048;
constexpr int kMaxTopK = 32;
constexpr int kRouterMaxExperts = 1024;   // logits held in registers, 32 per lane at most

struct PlanGeometry {
  int tile_tokens;     // TT: tokens per tile
  int tiles_per_rank;  // ceil(T / TT)
  int num_tiles;       // R * tiles_per_rank
};

inline PlanGeometry plan_geometry(const moe_shape &s) {
  PlanGeometry g;
  if (s.tokens_per_rank == 0) {   // empty batch: no tiles
    g.tile_tokens = 1;
    g.tiles_per_rank = 0;
    g.num_tiles = 0;
    return g;
  }
  int tt = kPlanTileEntries / s.top_k;
  if (tt < 1) tt = 1;
  if (tt > s.tokens_per_rank) tt = s.tokens_per_rank;
  g.tile_tokens = tt;
  g.tiles_per_rank = (s.tokens_per_rank + tt - 1) / tt;
  g.num_tiles = s.num_ranks * g.tiles_per_rank;
  return g;
}

// ---------------------------------------------------------------------------
// Workspace: a 256-byte header, then per-tile flags and per-tile count rows.
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t ticket;      // next tile id to hand out (reset by the last tile)
  uint32_t done;        // tiles finished in the running plan (reset by the last tile)
  uint32_t epoch;       // plan launches so far; tags this launch's flags
  uint32_t err_bits;    // errors seen by the running plan (kErr*)
  int32_t status;       // moe_status of the last plan (and of later dispatch/combine)
  uint32_t debug_flags; // kDebug* test hooks
  uint64_t timeout_ns;  // limit of every wait; 0 = kDefaultTimeoutNs
  uint32_t arrivals;    // fused plan+dispatch: blocks arrived (bits 0-7), blocks whose table
                        // copy timed out (8-15), that saw a bad expert (16-23) or an
                        // over-capacity expert (24-31); reset by the last block to arrive
  uint32_t reserved[55];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr uint32_t kErrBadExpert = 1u;
constexpr uint32_t kErrCapacity = 2u;
constexpr uint32_t kErrTimeout = 4u;
constexpr uint32_t kDebugHoldTile0 = 1u;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
  size_t tags_off;    // uint32 agg_tag[num_tiles], incl_tag[num_tiles]
  size_t rows_off;    // int32 agg[num_tiles][E], incl[num_tiles][E]
  size_t total;
};

inline WsLayout ws_layout(const moe_shape &s) {
  PlanGeometry g = plan_geometry(s);
  WsLayout L;
  L.tags_off = sizeof(WsHeader);
  L.rows_off = L.tags_off + align_up(2 * (size_t)g.num_tiles * sizeof(uint32_t), 256);
  L.total = L.rows_off + align_up(2 * (size_t)g.num_tiles * s.num_experts * sizeof(int32_t), 256);
  return L;
}

// ---------------------------------------------------------------------------
// Kernel parameters.
// ---------------------------------------------------------------------------
struct PlanParams {
  const int32_t *topk_idx;
  const int32_t *num_tokens;   // [R] valid tokens per rank, or null (all T)
  int masked;                  // 1: expert id -1 marks an entry that is not routed
  int32_t *expert_num_tokens;
  int32_t *expert_rank_offsets;
  int32_t *slot_of;
  int32_t *src_of;
  WsHeader *hdr;
  uint32_t *agg_tag;
  uint32_t *incl_tag;
  int32_t *agg;
  int32_t *incl;
  int R, T, E, K, cap;
  int tile_tokens, tiles_per_rank, num_tiles;
  // single-cluster path (filled by launch_plan): one warp per chunk of whole
  // tokens inside one rank
  int chunk_tokens, chunks_per_rank, num_chunks, batches;
};

// Single-cluster plan limits: up to 16 CTAs of 16 warps, one chunk of at
// most 32 * kClusterMaxBatches entries per warp.
constexpr int kClusterMaxCtas = 16;
constexpr int kClusterWarps = 16;
constexpr int kClusterMaxBatches = 8;
constexpr int kClusterMaxExperts = 1024;
constexpr size_t kClusterMaxSmem = 200 * 1024;   // dynamic shared memory per CTA, at most

struct DispatchParams {
  const uint16_t *x;
  const int32_t *topk_idx;
  const int32_t *slot_of;
  void *expert_x;
  float *expert_x_scale;
  WsHeader *hdr;
  int N, H, E, K, cap;
  int scale_t;                 // fp8: scales [E, H/128, cap] instead of [E, cap, H/128]
  int early_x;                 // 1: x is read before waiting for the previous kernel
                               // (the caller asserts it was final before that kernel began)
};

// Plan and dispatch in one launch (moe_plan_dispatch.cu): taken up to
// kFusedMaxEntries routed entries, since every block reads the whole routing
// table, and while the block's tables fit kFusedMaxSmem.
constexpr int64_t kFusedMaxEntries = 16384;
constexpr int kFusedMaxGrid = 255;      // the arrival word counts blocks in 8-bit fields
constexpr size_t kFusedMaxSmem = 200 * 1024;   // the routing table (<= 64 KB) and the block's tables

struct FusedParams {
  DispatchParams d;            // x, expert_x, expert_x_scale, hdr, N, H, E, K, cap
  const int32_t *topk_idx;
  int32_t *expert_num_tokens;
  int32_t *expert_rank_offsets;
  int32_t *slot_of;
  int32_t *src_of;
  int R, T;
  int units;                   // bf16: 16-byte chunks per lane per task; fp8: block pairs
  int tpr;                     // tasks per token row
  int64_t ntasks;              // N * tpr
  int q_tasks;                 // tasks per block, at most (block b: [b*ntasks/grid, (b+1)*ntasks/grid))
  int grid;                    // blocks, one per SM at most
  int owned;                   // experts per block for counts and offsets
  int max_run;                 // routed entries of one block's tokens, at most
  int ebits;                   // bits of the largest expert id
  int vec_idx;                 // topk_idx is 16-byte aligned (16-byte loads)
  int task_elems;              // x elements of one whole task
  size_t stage_off;            // dynamic shared memory offset of the staged second tasks
  size_t smem_bytes;
};

struct CombineParams {
  const uint16_t *expert_y;
  const uint16_t *shared;      // [N, H] bf16 shared-expert output, or null
  const int32_t *topk_idx;
  const int32_t *slot_of;
  const float *topk_weights;
  uint16_t *y;
  WsHeader *hdr;
  int N, H, E, K, cap;
};

struct ActParams {
  const uint16_t *expert_h;          // [E, cap, 2I] bf16: gate | up
  const int32_t *expert_num_tokens;  // [E]
  void *act_q;                       // [E, cap, I] e4m3
  float *act_scale;                  // [E, cap, I/128], or [E, I/128, cap] with scale_t
  WsHeader *hdr;
  int E, cap, I;
  int scale_t;
};

struct RouterParams {
  const float *logits;     // [N, E]
  int32_t *topk_idx;       // [N, K]
  float *topk_weights;     // [N, K]
  int64_t N;
  int E, K;
};

// Valid tokens of rank r: clamp(num_tokens[r], 0, T), or T without num_tokens.
#ifdef __CUDACC__
__device__ __forceinline__ int rank_tokens(const PlanParams &p, int r) {
  if (!p.num_tokens) return p.T;
  const int nt = __ldg(p.num_tokens + r);
  return nt < 0 ? 0 : (nt > p.T ? p.T : nt);
}
#endif

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_plan(const PlanParams &p, cudaStream_t stream);
cudaError_t launch_dispatch_bf16(const DispatchParams &p, cudaStream_t stream);
cudaError_t launch_dispatch_fp8(const DispatchParams &p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
// Fill the launch geometry of the fused plan + dispatch; false when the shape
// is outside the fused path's limits (then run moe_plan and moe_dispatch).
bool plan_dispatch_geometry(const moe_shape &s, FusedParams &p);
cudaError_t launch_plan_dispatch(const FusedParams &p, bool fp8, cudaStream_t stream);
cudaError_t launch_router(const RouterParams &p, cudaStream_t stream);
cudaError_t launch_silu_quant(const ActParams &p, cudaStream_t stream);
cudaError_t launch_set_debug(WsHeader *hdr, uint32_t flags, uint64_t timeout_ns,
                             cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Resident blocks per SM of `kern` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device (cached per kernel and device).
int occupancy_blocks(const void *kern, int threads, size_t smem);

// Persistent grid for `tasks` warp tasks: enough blocks of `threads` for one
// task per warp, at most SMs x resident blocks per SM.
int persistent_grid(const void *kern, int threads, int64_t warp_tasks);

// Launch `kern(params)` allowing a programmatic dependency on the previous
// kernel in `stream` (see pdl_wait_for_previous).
template <typename Params>
cudaError_t launch_after_previous(void (*kern)(Params), int grid, int threads,
                                  const Params &params, cudaStream_t stream) {
#ifndef MOE_PDL
#define MOE_PDL 1
#endif
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, params);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until *flag == want, for at most `deadline` (global timer, ns) and a
// bounded number of polls.  Returns false when the wait ran out.
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, uint32_t want, uint64_t deadline) {
  constexpr uint32_t kMaxPolls = 1u << 26;
  for (uint32_t it = 0; it < kMaxPolls; ++it) {
    if (ld_acquire_gpu(flag) == want) return true;
    if ((it & 15u) == 15u && global_timer_ns() > deadline) return false;
    __nanosleep(32);
  }
  return false;
}

// Barrier `id` (1..15) over the first `n` threads of the block (n a
// multiple of 32; every thread that takes part passes the same id and n).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// named_sync that also returns the AND of `pred` over the n threads.
__device__ __forceinline__ bool named_sync_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\t"
               "setp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, %2, %3, p;\n\t"
               "selp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier without memory ordering: arrive early, wait later
// (used to know that every CTA of the cluster has started).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// A cluster barrier in two halves: every thread's writes before its arrive
// are visible to every thread of the cluster after its wait; work that needs
// nothing from the peers may go in between.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// All threads of all CTAs of the cluster: writes before are visible after.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store an int to the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ void st_dsmem(int32_t *local, uint32_t rank, int32_t v) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Load an int from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ int ld_dsmem(const int32_t *local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// (token, segment) of a warp's tasks task0, task0 + stride, task0 + 2 stride,
// ...: the stride's whole rows and remainder are found once, so stepping to
// the next task needs no 64-bit division.  32-bit fields: tokens are below
// 2^31 (N*K < 2^31) and the stride is a grid's warps.
struct TaskCursor {
  int g, seg, dg, dseg, tpr;
  __device__ __forceinline__ TaskCursor(int64_t task0, int64_t stride, int tpr_) {
    tpr = tpr_;
    const int64_t g0 = task0 / tpr_;
    g = (int)g0;
    seg = (int)(task0 - g0 * tpr_);
    dg = (int)(stride / tpr_);
    dseg = (int)(stride - (int64_t)dg * tpr_);
  }
  __device__ __forceinline__ TaskCursor next() const {
    TaskCursor n = *this;
    n.g += dg;
    n.seg += dseg;
    if (n.seg >= tpr) {
      n.seg -= tpr;
      ++n.g;
    }
    return n;
  }
};

// Lanes of this warp whose key equals this lane's key (keys < 2^bits, or -1
// for "no key", which matches only other -1 lanes).  Every lane executes
// every ballot (no lane leaves early), as the full-warp ballots require.
__device__ __forceinline__ unsigned peers_with_same_key(int key, int bits) {
  const unsigned none = __ballot_sync(0xFFFFFFFFu, key < 0);
  unsigned m = ~none;
  for (int b = 0; b < bits; ++b) {
    const int bit = (key >> b) & 1;
    const unsigned set = __ballot_sync(0xFFFFFFFFu, bit);
    m &= bit ? set : ~set;
  }
  return key < 0 ? none : m;
}

// --- bulk copy global -> shared with an mbarrier (one CTA) ---
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive on `bar` announcing `bytes` of asynchronous copies, then copy
// `bytes` (a multiple of 16, both addresses 16-byte aligned) from global
// `src` to shared `dst`; the copy completes the announced bytes.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` for at most `deadline` (global timer,
// ns) and a bounded number of polls; false when the wait ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t deadline) {
  constexpr uint32_t kMaxPolls = 1u << 24;
  for (uint32_t it = 0; it < kMaxPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() > deadline) return false;
  }
  return false;
}

// Programmatic dependent launch.  The plan and activation kernels allow the
// next kernel in the stream to be scheduled as soon as all their blocks have
// started (measured: the dispatch, combine and router kernels ran slower
// when their successors started early, so they do not), and every kernel but
// the plan's is launched as such a dependent: it may do work that needs
// nothing from the previous kernel (dispatch loads and quantises x rows; the
// activation stages its table) and then waits here until the previous kernel
// has completed and its writes are visible.  No kernel writes anything
// before that wait.  Without a programmatic dependency the wait returns at
// once.
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_for_previous() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --- 1x128 E4M3 quantisation shared by dispatch and the activation kernel ---
// bf16 halves of a 32-bit word -> float (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four floats -> four E4M3 bytes, the first in the low byte: round to
// nearest even, finite overflow saturated to +-448 (cvt ... e4m3x2 puts its
// first source operand in the upper byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// max(|a|, |b|) of each bf16 half of two packed words (the result's sign
// bits are the XOR of the inputs' and carry nothing); a NaN half loses to a
// number, as in fmaxf.
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest |x| of a 128-element block held by a half-warp as raw bf16, 4
// words per lane (lanes 0-15 one block, 16-31 the next), NaN ignored and 0 for
// a block of NaNs, as fmaxf from 0 gives.  The tree and the butterfly run on
// packed pairs; the two halves meet at the end.  All 32 lanes call it together.
__device__ __forceinline__ float half_warp_amax_bf16(uint4 v) {
  uint32_t m = bf16x2_max_abs(bf16x2_max_abs(v.x, v.y), bf16x2_max_abs(v.z, v.w));
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) m = bf16x2_max_abs(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  return fmaxf(fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m))), 0.0f);
}

// Largest |x| of a 128-element block held by a half-warp, 8 values per lane
// (lanes 0-15 one block, 16-31 the next); all 32 lanes call it together.
__device__ __forceinline__ float half_warp_amax(const float (&f)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  return amax;
}

// --- E4M3 bytes e4m3(RN(x / scale)) of fp32 x by a bracketing window ---
// (the activation's values; bf16 x takes the corrected quotient below).
// With r = RN(1 / scale), x is multiplied by r scaled down and up by 2^-20
// (quant_window4), which brackets RN(x / scale); where both ends give the
// same byte, that byte is exact (sampled in tests/window_check.c).  Where
// they differ -- a quotient next to an E4M3 midpoint, rare for fp32 values --
// that element alone is divided with IEEE __fdiv_rn.  If 1/scale overflows
// (r > 3e38) every element is divided.
__device__ __forceinline__ uint32_t e4m3_byte(float v) { return e4m3x4(v, 0.0f, 0.0f, 0.0f) & 0xFFu; }

// The bytes by IEEE division of every element.
__device__ __forceinline__ uint2 quant_bytes8_exact(const float (&f)[8], float scale) {
  return make_uint2(e4m3x4(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale), __fdiv_rn(f[2], scale),
                           __fdiv_rn(f[3], scale)),
                    e4m3x4(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale), __fdiv_rn(f[6], scale),
                           __fdiv_rn(f[7], scale)));
}

// Fast E4M3 words of 4 values from rl = RN(r * (1 - 2^-20)) and
// rh = RN(r * (1 + 2^-20)), r = RN(1 / scale): lo = e4m3(RN(x * rl)) and
// hi = e4m3(RN(x * rh)).  RN(x * rl) is at most x/scale * (1 - 2^-20) *
// (1 + 2^-24)^3 < x/scale * (1 - 2^-24) in magnitude, below RN(x / scale),
// and RN(x * rh) above it likewise; rounding to E4M3 is monotone, so a byte
// where lo and hi agree is e4m3(RN(x / scale)).  (Below the normal range
// every candidate rounds to a zero of x's sign.)
// (x0 * s, x1 * s), each rounded to nearest even (IEEE binary32, no flush
// to zero): one packed two-lane multiply of sm_100-class GPUs.
__device__ __forceinline__ void fmul2_rn(float x0, float x1, float s, float &y0, float &y1) {
  uint64_t a, b, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(s));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(r));
}

__device__ __forceinline__ void quant_window4(float a, float b, float c, float d, float rl, float rh,
                                              uint32_t &lo, uint32_t &hi) {
  float al, bl, cl, dl, ah, bh, ch, dh;
  fmul2_rn(a, b, rl, al, bl);
  fmul2_rn(c, d, rl, cl, dl);
  fmul2_rn(a, b, rh, ah, bh);
  fmul2_rn(c, d, rh, ch, dh);
  lo = e4m3x4(al, bl, cl, dl);
  hi = e4m3x4(ah, bh, ch, dh);
}

// rl and rh of quant_window4.
__device__ __forceinline__ float2 quant_window_r(float r) {
  return make_float2(__fmul_rn(r, 1.0f - 0x1p-20f), __fmul_rn(r, 1.0f + 0x1p-20f));
}

// Replace the bytes of lo where lo and hi differ by the divided ones.
__device__ __forceinline__ uint32_t quant_patch4(uint32_t lo, uint32_t hi, float a, float b, float c,
                                                 float d, float scale) {
  const uint32_t diff = lo ^ hi;
  if (diff & 0x000000FFu) lo = (lo & 0xFFFFFF00u) | e4m3_byte(__fdiv_rn(a, scale));
  if (diff & 0x0000FF00u) lo = (lo & 0xFFFF00FFu) | (e4m3_byte(__fdiv_rn(b, scale)) << 8);
  if (diff & 0x00FF0000u) lo = (lo & 0xFF00FFFFu) | (e4m3_byte(__fdiv_rn(c, scale)) << 16);
  if (diff & 0xFF000000u) lo = (lo & 0x00FFFFFFu) | (e4m3_byte(__fdiv_rn(d, scale)) << 24);
  return lo;
}

// --- RN(x / scale) for bf16 x, with no division and no branch ---
// q0 = RN(x y) with y = RN(1/scale) is off by up to about 1.5 units in the
// last place; one correction with the exact remainder (Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 1990): e = RN(scale q0 - x), q = RN(q0 - e y).  For bf16 x (8
// significant bits) and y = RN(1/scale), q = RN(x / scale) exactly: checked
// for every finite bf16 x with |x/scale| < 1024 against every binary32 scale
// in [1, 2) (2.95e11 cases), and at scale exponents -60 to 60 on every 64th
// significand (tests/quotient_check.c).  Scaling x and scale by the same
// power of two changes no rounding while every intermediate stays normal,
// which holds for scale in [2^-60, 2^60]; a quotient below 2^-12 comes out
// below 2^-10 in magnitude, an E4M3 zero of x's sign.  The steps run on -x and
// -y: with x - scale q0 as the remainder, x = -0 would come out +0.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// Two-lane packed multiply and fused multiply-add of sm_100-class GPUs, each
// lane rounded to nearest even (IEEE binary32, no flush to zero).
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Scales whose quotients the correction gives exactly.
__device__ __forceinline__ bool quot_scale_ok(float scale) {
  return scale >= 0x1p-60f && scale <= 0x1p60f;
}

// RN(x / scale) of the two bf16 halves of w; s2 = (scale, scale), ny2 =
// (-y, -y) with y = RN(1/scale), scale within quot_scale_ok.
__device__ __forceinline__ float2 quot2_bf16(uint32_t w, uint64_t s2, uint64_t ny2) {
  const uint32_t nw = w ^ 0x80008000u;                 // -x, both halves
  const uint64_t nx = pack2(__uint_as_float(nw << 16), __uint_as_float(nw & 0xFFFF0000u));
  const uint64_t q0 = fmul2(nx, ny2);                   // x y
  const uint64_t e = ffma2(s2, q0, nx);                 // scale q0 - x
  return unpack2(ffma2(e, ny2, q0));                    // q0 - e y
}

// One lane's 8 E4M3 bytes e4m3(RN(x / scale)) of its 16-byte chunk v of a
// block, as two little-endian words; scale within quot_scale_ok.
__device__ __forceinline__ uint2 quant_bytes8_bf16(uint4 v, float scale, float ny) {
  const uint64_t s2 = pack2(scale, scale);
  const uint64_t ny2 = pack2(ny, ny);
  const float2 a = quot2_bf16(v.x, s2, ny2);
  const float2 b = quot2_bf16(v.y, s2, ny2);
  const float2 c = quot2_bf16(v.z, s2, ny2);
  const float2 d = quot2_bf16(v.w, s2, ny2);
  return make_uint2(e4m3x4(a.x, a.y, b.x, b.y), e4m3x4(c.x, c.y, d.x, d.y));
}

// The same bytes for any scale: outside quot_scale_ok every element is
// divided (zero: the block's amax is 0, all bytes 0).
__device__ __forceinline__ uint2 quant_bytes8_bf16_any(uint4 v, float scale, float ny, bool zero) {
  if (zero) return make_uint2(0u, 0u);
  if (quot_scale_ok(scale)) return quant_bytes8_bf16(v, scale, ny);
  const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
  return quant_bytes8_exact(f, scale);
}

// A lane's P blocks of 8 values (block it: scale[it], r[it] = RN(1/scale),
// zero[it]: its amax is 0) to E4M3 bytes, exact: the window bytes, then, if
// any lane of the warp has a byte whose window ends disagree (one vote),
// each such byte alone divided.  1/scale overflowing (r > 3e38) divides the
// whole block.  For fp32 inputs, where such bytes are rare enough that one
// vote per task beats a branch per word.  All 32 lanes call it together.
template <int P>
__device__ __forceinline__ void quantise_blocks(const float (&f)[P][8], const float (&scale)[P],
                                                const float (&r)[P], const bool (&zero)[P],
                                                uint2 (&q)[P]) {
  uint32_t hi[P][2];
  bool any = false;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    if (zero[it]) {
      q[it] = make_uint2(0u, 0u);
      hi[it][0] = hi[it][1] = 0u;
    } else if (!(r[it] <= 3.0e38f)) {
      q[it] = quant_bytes8_exact(f[it], scale[it]);
      hi[it][0] = q[it].x;
      hi[it][1] = q[it].y;
    } else {
      const float2 rw = quant_window_r(r[it]);
      quant_window4(f[it][0], f[it][1], f[it][2], f[it][3], rw.x, rw.y, q[it].x, hi[it][0]);
      quant_window4(f[it][4], f[it][5], f[it][6], f[it][7], rw.x, rw.y, q[it].y, hi[it][1]);
      any |= (q[it].x != hi[it][0]) | (q[it].y != hi[it][1]);
    }
  }
  if (__any_sync(0xFFFFFFFFu, any)) {
#pragma unroll
    for (int it = 0; it < P; ++it) {
      if (q[it].x != hi[it][0])
        q[it].x = quant_patch4(q[it].x, hi[it][0], f[it][0], f[it][1], f[it][2], f[it][3], scale[it]);
      if (q[it].y != hi[it][1])
        q[it].y = quant_patch4(q[it].y, hi[it][1], f[it][4], f[it][5], f[it][6], f[it][7], scale[it]);
    }
  }
}

// amax / 448 rounded to nearest: q0 = RN(amax * RN(1/448)), then one
// correction with the exact remainder (the method for divisors known in
// advance of Brisebarre, Muller and Raina, IEEE Trans. Computers 2004).
// Checked against IEEE division for every binary32 amax in [2^-120, FLT_MAX]
// (tests/div448_check.c); smaller and non-finite amax (subnormal quotients,
// inf) take __fdiv_rn.
__device__ __forceinline__ float div448_fast(float amax) {
  const float y = 1.0f / 448.0f;
  const float q0 = __fmul_rn(amax, y);
  const float r = __fmaf_rn(-q0, 448.0f, amax);
  return __fmaf_rn(r, y, q0);
}


// The status the dispatch and combine kernels see; read once per block.
__device__ __forceinline__ int32_t read_status(const WsHeader *hdr) {
  return *reinterpret_cast<const volatile int32_t *>(&hdr->status);
}

// Record a data error found by dispatch/combine (first error wins).
__device__ __forceinline__ void report_status(WsHeader *hdr, int32_t code) {
  atomicCAS(reinterpret_cast<int *>(&hdr->status), 0, code);
}
#endif

}  // namespace moe
