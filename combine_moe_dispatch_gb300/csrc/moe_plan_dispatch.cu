// moe_plan_dispatch.cu -- the plan and the dispatch in one launch.
//
// What it computes: exactly what moe_plan followed by moe_dispatch computes
// (moe_plan.cu, moe_dispatch.cu): counts, per-rank offsets, stable slots,
// return addresses, and the bf16 or fp8 expert rows ("Efficient and portable
// mixture-of-experts communication", Dispatch; "Enabling trillion-parameter
// models on AWS EFA", Send and Receive Buffers; "Lower latency and higher
// throughput with multi-node DeepSeek deployment", Quantization).
//
// Why: at decode sizes the plan is a chain of short dependent steps (load the
// routes, rank, exchange counts, scan, write) whose latency, and the kernel
// boundary after it, is a third of plan + dispatch.  Here no block waits for
// another: each finds the slots it needs from the routing table itself.
//
// How: block b takes the contiguous run of (token, segment) tasks
// [b*n/G, (b+1)*n/G) (n tasks, G blocks, one per SM), so its tokens form one
// range [g_lo, g_hi] and its routed entries the run [g_lo*K, (g_hi+1)*K).
// The slot of an entry (g, k) with expert e is the number of entries of e
// before the run plus the number of entries of e inside the run before
// (g, k).  Block b also owns the experts [b*O, (b+1)*O) and writes their
// counts and offsets rows.  The kernel is a programmatic dependent of the
// previous kernel: its blocks may be scheduled while that kernel drains, and
// wait for it before reading anything.
//   1. Thread 0 starts one bulk copy (cp.async.bulk, completed on an
//      mbarrier, waited for with a time limit) of the whole routing table
//      into shared memory, and every warp issues the loads of its first
//      task's x segment.  The copy engine leaves the SM's load pipeline to
//      the x loads; when the table went through that pipeline as plain
//      loads, it waited behind them (about 2 us at DeepSeek-V3 decode).
//      bf16: each warp's second task is bulk-copied into shared memory too.
//   2-4 are the planner warps' work (all warps for bf16, 12 of 24 for fp8);
//      for fp8 the other warps quantise their first task meanwhile, so the
//      first stores wait for the longer of the plan and the quantisation,
//      not for their sum.
//   2. The planners mark the experts of the run in a shared byte table.
//   3. Warp 0 ranks the run stably (one ballot per bit of the expert id finds
//      the lanes with the same expert; a shared per-expert counter carries
//      the count across 32-entry batches).  Meanwhile the other planners
//      scan the entries before the run in shared memory: one whose expert is
//      marked adds one to that expert's count.
//   4. slot = count before the run + rank in the run, kept in shared memory;
//      a slot at or beyond cap is the capacity error (every entry is in some
//      block's run, so the runs see every expert that overflows).
//   5. After one block barrier the warps run their tasks as moe_dispatch
//      does, software-pipelined, with the routes read from shared memory
//      (the planners first quantise their own first task).  A warp starting
//      its last task lets the next kernel in the stream begin to launch.
//   6. The block's first warp to run out of tasks adds the block's arrival
//      and error bits to one workspace word; the last block to arrive writes
//      the status word (no block waits for another).  Issued by a warp with
//      stores still to make, that contended atomic delayed it by ~0.8 us.
//      The same warp writes slot_of and src_of for the tokens whose first
//      segment the block holds (stores issued before the tasks would wait
//      behind the x loads).
//   7. The warps that run out of tasks claim 128-entry chunks of the table
//      and count the owned experts' entries per rank; the warp that
//      completes the last chunk writes the owners' counts and offsets rows.
//      The block's slowest warp, which sets its end, mostly finds no chunk
//      left.
// Every block copies and scans all N*K routes, which pays only while the
// table is small: the fused path is taken up to kFusedMaxEntries routed
// entries (at Kimi-K2 decode, 32768 entries, two launches measured faster);
// larger shapes run moe_plan and moe_dispatch as two launches.  One block per
// SM, as many threads as the dispatch kernels keep resident per SM (768 for
// fp8, or 1024 when that would give a warp more than two tasks; 1024 for
// bf16).
//
// Data errors: the status word ends up exactly as moe_plan would set it, and
// the plan outputs are those of moe_plan.  But no block waits for the
// outcome of the others, so the rows of entries whose expert is in range and
// whose slot is below cap may already have been written when the status
// reports an error; moe_dispatch would write none.
#include <cuda_bf16.h>

#include "moe_dispatch_tasks.cuh"

namespace moe {

// bf16 and fp8 tasks behind one interface: load (no routing needed), prep
// (fp8: quantise; bf16: nothing), store to the K rows.
// Warps of a block that make the plan (the rest quantise meanwhile): all of
// them for bf16, which has nothing to quantise; a part for fp8.
#ifndef MOE_FUSED_PLAN_WARPS
#define MOE_FUSED_PLAN_WARPS 12
#endif

template <int U>
struct Bf16Path {
  using Raw = Bf16Task<U>;
  using Out = Bf16Task<U>;
  static constexpr int kPlanWarps = 0;   // all
  static constexpr bool kStage2 = true;
  static __device__ __forceinline__ void load(const DispatchParams &p, const TaskCursor &c,
                                              int lane, Raw &a) {
    bf16_load<U>(p, c.g, c.seg, lane, a);
  }
  // the task from its copy in shared memory (s: the task's first element)
  static __device__ __forceinline__ void load_staged(const DispatchParams &p, const TaskCursor &c,
                                                     int lane, const uint16_t *s, Raw &a) {
    const int cpr = p.H / 8;
    a.g = c.g;
    a.seg = c.seg;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c16 = c.seg * 32 * U + lane + u * 32;
      a.v[u] = c16 < cpr ? *reinterpret_cast<const uint4 *>(s + (lane + u * 32) * 8)
                         : make_uint4(0, 0, 0, 0);
    }
  }
  static __device__ __forceinline__ void prep(const Raw &a, int, Out &t) { t = a; }
  static __device__ __forceinline__ void store(const DispatchParams &p, int lane, const Out &t,
                                               const Routes &r) {
    bf16_store<U>(p, lane, t, r);
  }
};

template <int P, bool SHORT = false>   // SHORT: H % 128 != 0 (fp8_load, fp8_store)
struct Fp8Path {
  using Raw = Fp8Raw<P>;
  using Out = Fp8Task<P>;
  static constexpr int kPlanWarps = MOE_FUSED_PLAN_WARPS;
  static constexpr bool kStage2 = false;
  static __device__ __forceinline__ void load(const DispatchParams &p, const TaskCursor &c,
                                              int lane, Raw &a) {
    fp8_load<P, SHORT>(p, c.g, c.seg, lane, a);
  }
  static __device__ __forceinline__ void load_staged(const DispatchParams &p, const TaskCursor &c,
                                                     int lane, const uint16_t *s, Raw &a) {
    const int half = lane >> 4, sub = lane & 15, nb = p.H / 128;
    a.g = c.g;
    a.seg = c.seg;
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const int blk = c.seg * 2 * P + it * 2 + half;
      const bool in = SHORT ? blk * 128 + sub * 8 < p.H : blk < nb;
      a.v[it] = in ? *reinterpret_cast<const uint4 *>(s + (it * 2 + half) * 128 + sub * 8)
                   : make_uint4(0, 0, 0, 0);
    }
  }
  static __device__ __forceinline__ void prep(const Raw &a, int lane, Out &t) {
    fp8_quantise<P>(a, lane, t);
  }
  static __device__ __forceinline__ void store(const DispatchParams &p, int lane, const Out &t,
                                               const Routes &r) {
    fp8_store<P, SHORT>(p, lane, t, r);
  }
};

// Routes of token g from the block's run: lane k < K holds (expert, slot);
// slot -1 (a bad id, or a slot at or beyond cap) makes the store skip it.
__device__ __forceinline__ Routes run_routes(const int32_t *s_rexp, const int32_t *s_rslot,
                                             int64_t g, int64_t g_lo, int K, int cap, int lane) {
  Routes r{-1, -1};
  if (lane < K) {
    const int i = (int)(g - g_lo) * K + lane;
    r.e = s_rexp[i];
    const int s = s_rslot[i];
    r.s = (r.e >= 0 && s < cap) ? s : -1;
  }
  return r;
}

// Status of a block, as one atomic add to the workspace's arrival word:
// bits 0-7 count the blocks that arrived, 8-15 those whose wait for the
// routing table ran out, 16-23 those that saw a bad expert id, 24-31 those
// that saw an expert over capacity (8-bit fields: at most 255 blocks).
__device__ __forceinline__ uint32_t arrival_code(uint32_t err) {
  return 1u | ((err & kErrTimeout) ? 1u << 8 : 0u) | ((err & kErrBadExpert) ? 1u << 16 : 0u) |
         ((err & kErrCapacity) ? 1u << 24 : 0u);
}

// Called by the one thread of a block that made the block's add, with the
// arrival word after that add: the last block to arrive writes the status
// word and resets the count.
__device__ __forceinline__ void finish_status(WsHeader *hdr, uint32_t arrived) {
  if ((arrived & 0xFFu) != gridDim.x) return;
  hdr->status = ((arrived >> 8) & 0xFFu)    ? MOE_ERR_TIMEOUT
                : ((arrived >> 16) & 0xFFu) ? MOE_ERR_BAD_EXPERT
                : (arrived >> 24)           ? MOE_ERR_CAPACITY
                                            : MOE_OK;
  hdr->arrivals = 0;
}


template <class Path, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
plan_dispatch_kernel(FusedParams p) {
  constexpr int kWarps = THREADS / 32;
  // planner warps: warp 0 ranks the run, the others scan the prefix
  constexpr int kPlanWarps = (Path::kPlanWarps > 0 && Path::kPlanWarps < kWarps) ? Path::kPlanWarps : kWarps;
  static_assert(kPlanWarps >= 2, "one warp ranks, at least one scans");
  constexpr int kPlanThreads = kPlanWarps * 32;
  constexpr int kScanThreads = kPlanThreads - 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ uint32_t s_err, s_fin, s_fail, s_chunk, s_chunk_done;
  __shared__ __align__(8) uint64_t s_xbar[Path::kStage2 ? kWarps : 1];   // per warp: its staged second task
  const int E = p.d.E, K = p.d.K, R = p.R, cap = p.d.cap;
  const int total = p.d.N * K;
  const size_t tab_bytes = ((size_t)total * 4 + 15) & ~(size_t)15;
  int32_t *s_tab = reinterpret_cast<int32_t *>(smem);                      // [N*K] the routing table
  uint8_t *s_code = smem + tab_bytes;                                      // [E] expert used by the run
  int32_t *s_pre = reinterpret_cast<int32_t *>(s_code + ((E + 15) & ~15)); // [E] entries before the run
  int32_t *s_loc = s_pre + E;                                              // [E] ranking counters
  int32_t *s_ocnt = s_loc + E;                                             // [O][R] owned experts per rank
  int32_t *s_rexp = s_ocnt + p.owned * R;                                  // [run] expert, -1 if bad
  int32_t *s_rslot = s_rexp + p.max_run;                                   // [run] rank, then slot

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool planner = warp < kPlanWarps;
  // block b: tasks [b * ntasks / grid, (b + 1) * ntasks / grid), so that the
  // runs differ by one task at most and every SM gets a block
  const int64_t t0 = (int64_t)blockIdx.x * p.ntasks / p.grid;
  const int64_t t1 = ((int64_t)blockIdx.x + 1) * p.ntasks / p.grid;
  const int64_t g_lo = t0 / p.tpr, g_hi = (t1 - 1) / p.tpr;
  const int lo_ent = (int)(g_lo * K);
  const int run = (int)(g_hi - g_lo + 1) * K;
  const int own0 = blockIdx.x * p.owned;

  // The shared-memory set-up (the barrier, the zeroed tables and counters)
  // reads nothing from global memory.  fp8 runs it before the wait for the
  // previous kernel (a programmatic dependency), so that it overlaps that
  // kernel's tail: 15.67 -> 15.22 us at DeepSeek-V3 decode, 15.95 -> 15.55
  // us at the Mixtral-shaped layer.  bf16 measured slower with it (22.3 ->
  // 23.6 us; its build then spilled) and runs it after.
  constexpr bool kEarlySetup = !Path::kStage2;
  auto zero_tables = [&]() {
    for (int i = tid; i < E; i += THREADS) {
      s_code[i] = 0;
      s_pre[i] = 0;
      s_loc[i] = 0;
    }
    for (int i = tid; i < p.owned * R; i += THREADS) s_ocnt[i] = 0;
    if (tid == 0) {
      s_err = 0;
      s_fin = 0;
      s_fail = 0;
      s_chunk = 0;
      s_chunk_done = 0;
    }
  };
  if constexpr (kEarlySetup) {
    if (tid == 0) mbar_init(&s_bar, 1);
    zero_tables();
  }
  // nothing in global memory is read before the previous kernel completes
  pdl_wait_for_previous();

  // 1. the routing table into shared memory: one bulk copy of its 16-byte
  //    part by the copy engine (it leaves the SM's load pipeline to the x
  //    loads), plain loads for the rest (all of it when the table is not
  //    16-byte aligned); the first task's x loads, which need nothing from
  //    the routing
  const int nbulk = p.vec_idx ? (total & ~3) : 0;
  if (tid == 0) {
    if constexpr (!kEarlySetup) mbar_init(&s_bar, 1);
    if (nbulk > 0) bulk_copy_g2s(s_tab, p.topk_idx, (uint32_t)nbulk * 4u, &s_bar);
  }
  for (int q = nbulk + tid; q < total; q += THREADS) s_tab[q] = __ldg(p.topk_idx + q);
  const int64_t my0 = t0 + warp;
  const bool has0 = my0 < t1;
  TaskCursor cur(my0, kWarps, p.tpr);
  typename Path::Raw a;
  if (has0) Path::load(p.d, cur, lane, a);
  // bf16: the warp's second task is copied into shared memory now, by the
  // copy engine, so x is read while the plan runs, before the stores start,
  // instead of between them.  (For fp8 it measured slower: the copies delay
  // the routing table, and the quantisers wait for the first task's x.)
  const uint16_t *s_x2 = reinterpret_cast<const uint16_t *>(smem + p.stage_off) +
                         (size_t)warp * p.task_elems;
  const bool has1 = Path::kStage2 && my0 + kWarps < t1;
  if (Path::kStage2 && lane == 0) {
    mbar_init(&s_xbar[warp], 1);
    if (has1) {
      const TaskCursor c1 = cur.next();
      const int64_t e0 = (int64_t)c1.seg * p.task_elems;
      const int64_t n = min((int64_t)p.task_elems, (int64_t)p.d.H - e0);
      bulk_copy_g2s(const_cast<uint16_t *>(s_x2), p.d.x + (int64_t)c1.g * p.d.H + e0,
                    (uint32_t)(n * 2), &s_xbar[warp]);
    }
  }
  bool stage_pending = has1;   // the copy may still be in flight
  if constexpr (!kEarlySetup) zero_tables();
  __syncthreads();   // also publishes the barriers' initialisation and the zeroed tables

  // 2-4 run on the planner warps alone (named barrier 1); the other warps
  // quantise their first task (fp8) meanwhile, as soon as its x lands, so
  // that the first stores wait for the plan or the quantisation, whichever
  // ends later, instead of for both one after the other.
  typename Path::Out t;
  uint32_t err = 0;
  if (planner) {
    const bool ok = nbulk == 0 || mbar_wait_bounded(&s_bar, 0, global_timer_ns() + kDefaultTimeoutNs);
    const bool tab_ok = named_sync_and(1, kPlanThreads, ok);
    if (tid == 0) s_fail = tab_ok ? 0u : 1u;
    if (tab_ok) {
      // 2. mark the run's experts
      for (int i = tid; i < run; i += kPlanThreads) {
        const int e = s_tab[lo_ent + i];
        const bool in = (unsigned)e < (unsigned)E;
        s_rexp[i] = in ? e : -1;
        if (in) s_code[e] = 1;   // every writer stores the same value
        else err |= kErrBadExpert;
      }
      named_sync(1, kPlanThreads);

      // 3. rank the run (warp 0) / count the entries before the run (the
      //    other planner warps)
      if (warp == 0) {
        const unsigned lt = (1u << lane) - 1u;
        for (int i0 = 0; i0 < run; i0 += 32) {
          const int i = i0 + lane;
          const int e = i < run ? s_rexp[i] : -1;
          const unsigned same = peers_with_same_key(e, p.ebits);
          const int before = __popc(same & lt);
          const int base = e >= 0 ? s_loc[e] : 0;
          __syncwarp();
          if (e >= 0 && before == 0) s_loc[e] = base + __popc(same);
          __syncwarp();
          if (i < run) s_rslot[i] = base + before;
        }
      } else {
        // An entry before the run whose expert the run uses adds one to
        // that expert's count before the run.  Only the prefix is read, and
        // nothing else is counted here: the owned experts' per-rank counts
        // are needed only for the offsets rows, written after the tasks.  A
        // bad id is reported by its own run's block.
        auto count_pre = [&](int e) {
          if ((unsigned)e < (unsigned)E && s_code[e]) atomicAdd(&s_pre[e], 1);
        };
        const int4 *t4 = reinterpret_cast<const int4 *>(s_tab);
        const int n4 = lo_ent >> 2;
        for (int j = tid - 32; j < n4; j += kScanThreads) {
          const int4 w = t4[j];
          count_pre(w.x);
          count_pre(w.y);
          count_pre(w.z);
          count_pre(w.w);
        }
        for (int q = 4 * n4 + tid - 32; q < lo_ent; q += kScanThreads) count_pre(s_tab[q]);
      }
      named_sync(1, kPlanThreads);

      // 4. slots (in shared memory only: the plan outputs are written after
      //    the tasks, so no store here waits behind the x loads in flight);
      //    errors.  An expert over capacity has an entry with slot cap, in
      //    some block's run: the runs' slots alone find every capacity error.
      for (int i = tid; i < run; i += kPlanThreads) {
        const int e = s_rexp[i];
        const int slot = e >= 0 ? s_pre[e] + s_rslot[i] : -1;
        if (e >= 0 && slot >= cap) err |= kErrCapacity;
        s_rslot[i] = slot;
      }
      if (err) atomicOr(&s_err, err);
    }
  } else if (has0) {
    Path::prep(a, lane, t);
  }
  __syncthreads();
  if (s_fail) {
    // the table copy did not land in time: wait once more (bounded) so that
    // no copy into this block's shared memory is left in flight, report,
    // and write nothing
    if (stage_pending) mbar_wait_bounded(&s_xbar[warp], 0, global_timer_ns() + kDefaultTimeoutNs);
    if (tid == 0) {
      mbar_wait_bounded(&s_bar, 0, global_timer_ns() + kDefaultTimeoutNs);
      const uint32_t code = arrival_code(kErrTimeout);
      finish_status(p.d.hdr, atomicAdd(&p.d.hdr->arrivals, code) + code);
    }
    return;
  }
  if (planner && has0) Path::prep(a, lane, t);   // the planners' first task, after the plan

  // 5. the tasks, software-pipelined as in moe_dispatch, starting from the
  //    first task quantised above.
  if (has0) {
    Routes r = run_routes(s_rexp, s_rslot, a.g, g_lo, K, cap, lane);
    int64_t task = my0;
    for (; task < t1; task += kWarps) {
      const int64_t next = task + kWarps;
      const bool more = next < t1;
      if (!more) pdl_allow_dependents();   // the next kernel may start launching
      cur = cur.next();
      typename Path::Raw an;
      const bool staged = has1 && task == my0;   // the next task is the one in shared memory
      if (more && !staged) Path::load(p.d, cur, lane, an);
      Path::store(p.d, lane, t, r);
      if (more) {
        if (staged) {
          // every lane waits for the copy (bounded); if any lane's wait ran
          // out, the warp reads x from global memory instead
          const bool in = mbar_wait_bounded(&s_xbar[warp], 0, global_timer_ns() + kDefaultTimeoutNs);
          if (__all_sync(kFull, in)) {
            stage_pending = false;
            Path::load_staged(p.d, cur, lane, s_x2, an);
          } else {
            Path::load(p.d, cur, lane, an);
          }
        }
        Path::prep(an, lane, t);
        r = run_routes(s_rexp, s_rslot, cur.g, g_lo, K, cap, lane);
      }
    }
  }
  // A copy not seen to complete (a wait that ran out): wait for it again,
  // bounded, so that none is left in flight when the block exits; report a
  // copy that still has not landed.
  if (stage_pending) {
    const bool in = mbar_wait_bounded(&s_xbar[warp], 0, global_timer_ns() + kDefaultTimeoutNs);
    if (!__all_sync(kFull, in) && lane == 0) report_status(p.d.hdr, MOE_ERR_TIMEOUT);
  }

  // 6-7 are shared out among the warps that finish their tasks first, so
  // that the block's slowest warp, which sets its end, does none of it: a
  // share per thread (with a block barrier before the offsets rows) cost
  // 1.1 us of the fp8 call at DeepSeek-V3 decode.
  //
  // 6. The block's first warp to run out of tasks carries its arrival and
  //    errors in one atomic (all blocks add to one word, so its round trip
  //    delays no warp that still has stores to issue), and writes slot_of
  //    and src_of of the tokens whose segment 0 is in this block.
  const unsigned first = __shfl_sync(kFull, lane == 0 ? atomicAdd(&s_fin, 1u) : 0u, 0);
  if (first == 0u) {
    if (lane == 0) {
      const uint32_t code = arrival_code(s_err);
      finish_status(p.d.hdr, atomicAdd(&p.d.hdr->arrivals, code) + code);
    }
    const int64_t gw0 = (t0 + p.tpr - 1) / p.tpr;
    const int64_t gw1 = (t1 + p.tpr - 1) / p.tpr;
    for (int i = lane; i < run; i += 32) {
      const int64_t g = g_lo + i / K;
      if (g >= gw0 && g < gw1) {
        const int e = s_rexp[i], slot = s_rslot[i], q = lo_ent + i;
        p.slot_of[q] = slot;
        if (e >= 0 && slot < cap) p.src_of[(int64_t)e * cap + slot] = q;
      }
    }
  }

  // 7. The owned experts' entries per rank, over the whole table, in
  //    128-entry chunks (4 per lane) that the warps claim as they run out of
  //    tasks; the warp that completes the last chunk writes the owners'
  //    counts and offsets rows.  Few entries belong to the owned experts,
  //    so an entry costs a compare; only those take an atomic.
  const int tk = p.T * K;      // entries per rank
  const int nchunks = (total + 127) / 128;
  unsigned mine = 0;   // chunks this warp counted
  for (;;) {
    const unsigned c = __shfl_sync(kFull, lane == 0 ? atomicAdd(&s_chunk, 1u) : 0u, 0);
    if (c >= (unsigned)nchunks) break;
    const int q0 = (int)c * 128 + 4 * lane;   // this lane's 4 entries
    int ev[4];
    if (q0 + 4 <= total) {
      const int4 w = *reinterpret_cast<const int4 *>(s_tab + q0);
      ev[0] = w.x;
      ev[1] = w.y;
      ev[2] = w.z;
      ev[3] = w.w;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) ev[u] = q0 + u < total ? s_tab[q0 + u] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const unsigned o = (unsigned)(ev[u] - own0);
      if ((unsigned)ev[u] < (unsigned)E && o < (unsigned)p.owned)
        atomicAdd(&s_ocnt[o * R + (q0 + u) / tk], 1);
    }
    ++mine;
  }
  if (mine == 0u) return;
  // One fence per warp: its counts are in before its chunks are reported
  // done.  The warp whose report completes the last chunk has every count.
  __threadfence_block();
  __syncwarp();
  const unsigned done = __shfl_sync(kFull, lane == 0 ? atomicAdd(&s_chunk_done, mine) + mine : 0u, 0);
  if (done != (unsigned)nchunks) return;
  __threadfence_block();
  for (int j = 0; j < p.owned; ++j) {
    const int e = own0 + j;
    if (e >= E) break;
    int32_t *row = p.expert_rank_offsets + (int64_t)e * (R + 1);
    int sum = 0;
    for (int r0 = 0; r0 < R; r0 += 32) {
      const int r = r0 + lane;
      const int cnt = r < R ? atomicAdd(&s_ocnt[j * R + r], 0) : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += v;
      }
      if (r < R) row[r] = sum + incl - cnt;
      sum += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
      row[R] = sum;
      p.expert_num_tokens[e] = sum;
    }
  }
}

namespace {

constexpr int kFusedFp8Threads = 768;    // 3 x 256: the fp8 dispatch's residency per SM
// fp8 with more than two tasks per warp at 768 threads: 1024 threads (64
// registers, 4 bytes of spill).  Measured: Mixtral-shaped layer (108 tasks
// per block) 16.5 -> 16.0 us; DeepSeek-V3 decode (48) 15.9 against 15.95 us.
constexpr int kFusedFp8ThreadsWide = 1024;
constexpr int kFusedBf16Threads = 1024;  // 4 x 256: the bf16 dispatch's residency per SM

template <class Path, int THREADS>
cudaError_t launch_fused(const FusedParams &p, cudaStream_t stream) {
  auto kern = plan_dispatch_kernel<Path, THREADS>;
  if (p.smem_bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
  }
  // A programmatic dependent of the previous kernel: its blocks may be
  // scheduled while that kernel drains (the previous kernels of this library
  // let their dependents launch when their warps start their last task),
  // and wait for it to complete before reading anything.  Measured at
  // DeepSeek-V3 decode in graphs of back-to-back calls, with the other
  // kernels' late trigger: fp8 16.6 -> 15.5 us, bf16 24.0 -> 23.3 us.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Task size of the fused kernel: up to 4 block pairs (fp8) or 4 chunks per
// lane (bf16), 1024 elements.  Half-size tasks, which start the first
// stores after half the quantisation, measured slower at DeepSeek-V3
// decode: fp8 18.7 against 17.3 us, bf16 25.8 against 24.0 us.
#ifndef MOE_FUSED_FP8_MAX_PAIRS
#define MOE_FUSED_FP8_MAX_PAIRS 4
#endif
#ifndef MOE_FUSED_BF16_MAX_UNITS
#define MOE_FUSED_BF16_MAX_UNITS 4
#endif
constexpr int kFusedFp8MaxPairs = MOE_FUSED_FP8_MAX_PAIRS;
constexpr int kFusedBf16MaxUnits = MOE_FUSED_BF16_MAX_UNITS;

bool plan_dispatch_geometry(const moe_shape &s, FusedParams &p) {
  const int64_t N = (int64_t)s.num_ranks * s.tokens_per_rank;
  if (N < 1 || N * s.top_k > kFusedMaxEntries) return false;
  const bool fp8 = s.payload != MOE_PAYLOAD_BF16;
  int tpr;
  if (fp8) {
    // a short last block (H % 128 != 0): always kFusedFp8MaxPairs pairs per task
    const int nb = (s.hidden + 127) / 128;
    const int P = (nb % 2 == 0 && s.hidden % 128 == 0) ? pick_units(nb / 2, kFusedFp8MaxPairs)
                                                        : kFusedFp8MaxPairs;
    tpr = (nb + 2 * P - 1) / (2 * P);
    p.units = P;
  } else {
    const int cpr = s.hidden / 8;
    const int U = (cpr % 32 == 0) ? pick_units(cpr / 32, kFusedBf16MaxUnits) : kFusedBf16MaxUnits;
    tpr = (cpr + 32 * U - 1) / (32 * U);
    p.units = U;
  }
  const int64_t ntasks = N * tpr;
  const int64_t sms = device_sm_count() < kFusedMaxGrid ? device_sm_count() : kFusedMaxGrid;
  const int grid = (int)(ntasks < sms ? ntasks : sms);
  const int64_t q = (ntasks + grid - 1) / grid;   // tasks of a block, at most
  const int owned = (s.num_experts + grid - 1) / grid;
  const int64_t max_run = (q / tpr + 2) * s.top_k;
  const size_t tab = ((size_t)(N * s.top_k) * 4 + 15) & ~(size_t)15;
  size_t smem = tab + (size_t)((s.num_experts + 15) & ~15) + 8 * (size_t)s.num_experts +
                4 * (size_t)owned * s.num_ranks + 8 * (size_t)max_run;
  // one whole task of x per warp, for the staged second tasks
  p.task_elems = fp8 ? 2 * p.units * 128 : 256 * p.units;
  p.stage_off = (smem + 15) & ~(size_t)15;
  if (!fp8) smem = p.stage_off + (size_t)(kFusedBf16Threads / 32) * p.task_elems * 2;
  if (smem > kFusedMaxSmem) return false;
  p.R = s.num_ranks;
  p.T = s.tokens_per_rank;
  p.tpr = tpr;
  p.ntasks = ntasks;
  p.q_tasks = (int)q;
  p.grid = grid;
  p.owned = owned;
  p.max_run = (int)max_run;
  int bits = 1;
  while ((1 << bits) < s.num_experts) ++bits;
  p.ebits = bits;
  p.smem_bytes = smem;
  return true;
}

cudaError_t launch_plan_dispatch(const FusedParams &p, bool fp8, cudaStream_t stream) {
  // The kernel's task size must be the one the geometry was made for: the
  // tasks per row (p.tpr) come from it, and the kernel indexes the blocks
  // of a task with its own size.
  if (fp8) {
    const bool wide = p.q_tasks > 2 * (kFusedFp8Threads / 32);
    if (p.d.H % 128 != 0) {   // a short last block: built for kFusedFp8MaxPairs only
      if (p.units != kFusedFp8MaxPairs) return cudaErrorInvalidValue;
      return wide ? launch_fused<Fp8Path<kFusedFp8MaxPairs, true>, kFusedFp8ThreadsWide>(p, stream)
                  : launch_fused<Fp8Path<kFusedFp8MaxPairs, true>, kFusedFp8Threads>(p, stream);
    }
    switch (p.units) {
      case 1: return wide ? launch_fused<Fp8Path<1>, kFusedFp8ThreadsWide>(p, stream)
                          : launch_fused<Fp8Path<1>, kFusedFp8Threads>(p, stream);
      case 2: return wide ? launch_fused<Fp8Path<2>, kFusedFp8ThreadsWide>(p, stream)
                          : launch_fused<Fp8Path<2>, kFusedFp8Threads>(p, stream);
      case 4: return wide ? launch_fused<Fp8Path<4>, kFusedFp8ThreadsWide>(p, stream)
                          : launch_fused<Fp8Path<4>, kFusedFp8Threads>(p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.units) {
    case 1: return launch_fused<Bf16Path<1>, kFusedBf16Threads>(p, stream);
    case 2: return launch_fused<Bf16Path<2>, kFusedBf16Threads>(p, stream);
    case 4: return launch_fused<Bf16Path<4>, kFusedBf16Threads>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
