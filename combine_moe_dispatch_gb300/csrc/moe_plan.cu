// moe_plan.cu -- per-expert counts, per-rank offsets and stable slots.
//
// What it computes ("Efficient and portable mixture-of-experts
// communication", Dispatch; "Enabling trillion-parameter models on AWS EFA",
// Send and Receive Buffers, Dispatch and Combine): for routed entries (g, k)
// in ascending order,
//   count[e]      = #{(g,k) : idx = e}
//   offsets[e][r] = #{(g,k) : idx = e, g < r*T}     (r = 0..R)
//   slot_of[g,k]  = #{(g',k') before (g,k) : same expert}
//   src_of[e][slot_of[g,k]] = g*K + k
//
// How (single pass, one launch): the entries are cut into tiles of whole
// tokens inside one rank; each thread block takes the next tile id from a
// ticket counter, so every tile it may wait for has already started.
//   1. Stable local ranks: warp w ranks its 32-entry batches with
//      __match_any_sync (equal experts in one batch) on top of a warp-private
//      per-expert counter; an exclusive scan over the warps turns these into
//      ranks inside the tile and gives the tile histogram h_t.
//   2. The block publishes h_t, waits (bounded) until every earlier tile has
//      published its histogram, takes the nearest earlier tile that already
//      published its inclusive prefix, and adds the histograms in between:
//      base_t = inclusive[j] + sum_{j<i<t} h_i.  It then publishes its own
//      inclusive prefix base_t + h_t.  (A look-back over whole count vectors
//      instead of single values; the waits never depend on later tiles.)
//   3. slot = base_t[e] + local rank; slot_of is written coalesced, src_of
//      only below cap.  Tile (r, 0) writes offsets[.][r] = base_t, the last
//      tile writes the counts and offsets[.][R].
//   4. The last block to finish turns the error bits into the status word,
//      resets the ticket and done counters and advances the epoch that tags
//      every flag, so the next launch needs no clearing pass.
#include "moe_common.cuh"

namespace moe {

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(PlanParams p) {
  extern __shared__ int32_t smem[];
  const int E = p.E;
  int32_t *wc = smem;                          // [kPlanWarps][E] warp counters -> warp bases
  int32_t *s_base = smem + kPlanWarps * E;     // [E] exclusive prefix of this tile
  int32_t *s_h = s_base + E;                   // [E] histogram of this tile
  __shared__ uint32_t s_tile, s_epoch, s_err;
  __shared__ int s_j;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  WsHeader *hdr = p.hdr;

  if (tid == 0) {
    s_tile = atomicAdd(&hdr->ticket, 1u);
    s_epoch = *reinterpret_cast<volatile uint32_t *>(&hdr->epoch);
    s_err = 0;
    s_j = -1;
  }
  for (int i = tid; i < kPlanWarps * E; i += kPlanThreads) wc[i] = 0;
  __syncthreads();

  // A tile id beyond the grid can only come from a workspace that was never
  // zeroed; such a block touches no array and reports a timeout.
  const bool stale = s_tile >= (uint32_t)p.num_tiles;
  const uint32_t t = stale ? 0u : s_tile;
  const uint32_t tag = (s_epoch & 0x7FFFFFFFu) + 1u;     // never 0 (0 = cleared)
  const uint64_t tmo = hdr->timeout_ns ? hdr->timeout_ns : kDefaultTimeoutNs;
  const bool hold = (hdr->debug_flags & kDebugHoldTile0) && t == 0;

  if (stale) {
    if (tid == 0) s_err = kErrTimeout;
  } else {
    const int r = (int)(t / (uint32_t)p.tiles_per_rank);
    const int j = (int)(t % (uint32_t)p.tiles_per_rank);
    const int64_t g0 = (int64_t)r * p.T + (int64_t)j * p.tile_tokens;
    const int tok = min(p.tile_tokens, p.T - j * p.tile_tokens);
    const int n_ent = tok * p.K;
    const int64_t ent0 = g0 * p.K;
    const int epw = ((n_ent + kPlanWarps * 32 - 1) / (kPlanWarps * 32)) * 32;  // entries per warp
    const unsigned lt_mask = (1u << lane) - 1u;

    // 1. stable ranks inside the warp's share of the tile
    int lrank[kPlanBatchesPerWarp];
    int lexp[kPlanBatchesPerWarp];
  #pragma unroll
    for (int b = 0; b < kPlanBatchesPerWarp; ++b) {
      const int pl = warp * epw + b * 32 + lane;
      const bool valid = (b * 32 < epw) && pl < n_ent;
      int e = valid ? __ldg(p.topk_idx + ent0 + pl) : -1;
      const bool ok = valid && e >= 0 && e < E;
      if (valid && !ok) atomicOr(&s_err, kErrBadExpert);
      const int key = ok ? e : -1;
      const unsigned same = __match_any_sync(0xFFFFFFFFu, key);
      const int before = __popc(same & lt_mask);
      const int wbase = ok ? wc[warp * E + e] : 0;
      __syncwarp();
      if (ok && before == 0) wc[warp * E + e] = wbase + __popc(same);
      __syncwarp();
      lrank[b] = wbase + before;
      lexp[b] = ok ? e : -1;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kPlanThreads) {
      int run = 0;
  #pragma unroll
      for (int w = 0; w < kPlanWarps; ++w) {
        const int c = wc[w * E + e];
        wc[w * E + e] = run;
        run += c;
      }
      s_h[e] = run;
    }
    __syncthreads();

    // 2. publish the histogram, then find this tile's exclusive prefix
    for (int e = tid; e < E; e += kPlanThreads) p.agg[(int64_t)t * E + e] = s_h[e];
    __threadfence();
    __syncthreads();
    if (tid == 0 && !hold) st_release_gpu(&p.agg_tag[t], tag);

    const uint64_t deadline = global_timer_ns() + tmo;
    for (uint32_t i = tid; i < t; i += kPlanThreads)
      if (!wait_flag(&p.agg_tag[i], tag, deadline)) atomicOr(&s_err, kErrTimeout);
    for (uint32_t i = tid; i < t; i += kPlanThreads)
      if (ld_acquire_gpu(&p.incl_tag[i]) == tag) atomicMax(&s_j, (int)i);
    __threadfence();
    __syncthreads();
    const int jn = s_j;
    for (int e = tid; e < E; e += kPlanThreads) {
      int b = jn >= 0 ? __ldcg(p.incl + (int64_t)jn * E + e) : 0;
      for (int i = jn + 1; i < (int)t; ++i) b += __ldcg(p.agg + (int64_t)i * E + e);
      s_base[e] = b;
      p.incl[(int64_t)t * E + e] = b + s_h[e];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0 && !hold) st_release_gpu(&p.incl_tag[t], tag);

    // 3. slots, return addresses, offsets, counts
  #pragma unroll
    for (int b = 0; b < kPlanBatchesPerWarp; ++b) {
      const int pl = warp * epw + b * 32 + lane;
      const bool valid = (b * 32 < epw) && pl < n_ent;
      if (!valid) continue;
      const int e = lexp[b];
      if (e < 0) {
        p.slot_of[ent0 + pl] = -1;
        continue;
      }
      const int slot = s_base[e] + wc[warp * E + e] + lrank[b];
      p.slot_of[ent0 + pl] = slot;
      if (slot >= 0 && slot < p.cap) p.src_of[(int64_t)e * p.cap + slot] = (int32_t)(ent0 + pl);
      else atomicOr(&s_err, kErrCapacity);
    }
    if (j == 0)
      for (int e = tid; e < E; e += kPlanThreads)
        p.expert_rank_offsets[(int64_t)e * (p.R + 1) + r] = s_base[e];
    if ((int)t == p.num_tiles - 1)
      for (int e = tid; e < E; e += kPlanThreads) {
        const int tot = s_base[e] + s_h[e];
        p.expert_num_tokens[e] = tot;
        p.expert_rank_offsets[(int64_t)e * (p.R + 1) + p.R] = tot;
      }
  }  // !stale

  // 4. the last block publishes the status and resets the counters
  __syncthreads();
  if (tid == 0) {
    if (s_err) atomicOr(&hdr->err_bits, s_err);
    __threadfence();
    const uint32_t d = atomicAdd(&hdr->done, 1u);
    if (d == (uint32_t)p.num_tiles - 1u) {
      __threadfence();
      const uint32_t bits = atomicExch(&hdr->err_bits, 0u);
      int32_t st = MOE_OK;
      if (bits & kErrTimeout) st = MOE_ERR_TIMEOUT;
      else if (bits & kErrBadExpert) st = MOE_ERR_BAD_EXPERT;
      else if (bits & kErrCapacity) st = MOE_ERR_CAPACITY;
      hdr->status = st;
      hdr->ticket = 0;
      hdr->done = 0;
      __threadfence();
      atomicAdd(&hdr->epoch, 1u);
    }
  }
}

__global__ void set_debug_kernel(WsHeader *hdr, uint32_t flags, uint64_t timeout_ns) {
  hdr->debug_flags = flags;
  hdr->timeout_ns = timeout_ns;
}

cudaError_t launch_plan(const PlanParams &p, cudaStream_t stream) {
  const size_t smem = (size_t)(kPlanWarps + 2) * p.E * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<p.num_tiles, kPlanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_set_debug(WsHeader *hdr, uint32_t flags, uint64_t timeout_ns,
                             cudaStream_t stream) {
  set_debug_kernel<<<1, 1, 0, stream>>>(hdr, flags, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
