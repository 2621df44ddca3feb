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
  pdl_allow_dependents();

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
    const int routed_ent = max(0, min(tok, rank_tokens(p, r) - j * p.tile_tokens)) * p.K;
    const unsigned lt_mask = (1u << lane) - 1u;

    // 1. stable ranks inside the warp's share of the tile
    int lrank[kPlanBatchesPerWarp];
    int lexp[kPlanBatchesPerWarp];
  #pragma unroll
    for (int b = 0; b < kPlanBatchesPerWarp; ++b) {
      const int pl = warp * epw + b * 32 + lane;
      const bool valid = (b * 32 < epw) && pl < n_ent;
      int e = (valid && pl < routed_ent) ? __ldg(p.topk_idx + ent0 + pl) : -1;
      const bool routed = valid && pl < routed_ent && !(p.masked && e == -1);
      const bool ok = routed && e >= 0 && e < E;
      if (routed && !ok) atomicOr(&s_err, kErrBadExpert);
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

// ---------------------------------------------------------------------------
// Single-cluster plan.  When every rank-aligned chunk fits one warp and all
// chunks fit 16 CTAs of 16 warps, the whole plan runs in one thread-block
// cluster and the cross-tile step goes through distributed shared memory:
//   1. warp w of CTA c ranks chunk 16c + w stably: for each 32-entry batch,
//      the lanes holding the same expert are found with one ballot per bit
//      of the expert id, on top of a warp-private per-expert counter;
//   2. an exclusive scan over the CTA's 16 warps gives each warp's base in
//      the CTA and the CTA histogram h_c;
//   3. every CTA stores h_c (and its error bits) into row c of every peer's
//      shared table (after a split cluster barrier, arrived at entry, shows
//      that every peer has started), then one cluster barrier makes the table
//      complete in every CTA: base_c = sum of rows < c, totals = sum of all
//      rows, read locally.  No CTA reads a peer's memory, so none has to
//      outlive that barrier for the others;
//   4. slot = base_c + warp base + rank in warp.  The CTA's return addresses
//      are staged in shared memory in (expert, slot) order and written out
//      as contiguous runs.  Each CTA owns a block of rows (experts) of the
//      offsets matrix: the CTA where rank r starts pushed its in-CTA prefix
//      for rank r into the row owner's shared memory before the barrier,
//      and each owner writes its rows and counts as one contiguous run
//      (stores from many CTAs into the same few sectors of that small
//      matrix serialise).  The last CTA writes the status word.
// The barrier is the hardware cluster barrier over co-scheduled CTAs; the
// kernel has no flags, counters or spin-waits in global memory.
// ---------------------------------------------------------------------------

// Exclusive scan of in[0..n) into out[0..n) by the whole block (n <= 2 *
// blockDim.x); returns the total.  Starts and ends with __syncthreads.
__device__ __forceinline__ int block_exclusive_scan(const int32_t *in, int32_t *out, int n) {
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  const int a = 2 * tid < n ? in[2 * tid] : 0;
  const int b = 2 * tid + 1 < n ? in[2 * tid + 1] : 0;
  int incl = a + b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += v;
    }
    if (lane < nw) s_warp[lane] = w;            // inclusive over warps
    if (lane == nw - 1) s_total = w;
  }
  __syncthreads();
  const int excl = incl - a - b + (warp > 0 ? s_warp[warp - 1] : 0);
  if (2 * tid < n) out[2 * tid] = excl;
  if (2 * tid + 1 < n) out[2 * tid + 1] = excl + a;
  __syncthreads();
  return s_total;
}

__global__ void __launch_bounds__(kClusterWarps * 32)
plan_cluster_kernel(PlanParams p) {
  extern __shared__ int32_t smem[];
  const int E = p.E;
  // CTA c owns experts [c * rows, (c + 1) * rows): it gathers every CTA's
  // counts of them, hands each CTA its base, and writes their counts and
  // offsets rows.
  const int rows = (E + (int)gridDim.x - 1) / (int)gridDim.x;
  int32_t *wc = smem;                             // [16][E] warp counters -> warp bases
  int32_t *s_hist = wc + kClusterWarps * E;       // [E] this CTA's histogram
  int32_t *s_base = s_hist + E;                   // [E] this CTA's base (written by the owners)
  int32_t *s_eoff = s_base + E;                   // [E] this CTA's entries before expert e
  int32_t *s_own = s_eoff + E;                    // [ncta][rows] owned experts' counts, row c from CTA c
  int32_t *s_tot = s_own + kClusterMaxCtas * rows;   // [rows] owned experts' totals
  int32_t *s_stage = s_tot + rows;                // [2][16*32*8] (entry id, expert) in slot order
  int32_t *s_offs = s_stage + 2 * kClusterWarps * 32 * kClusterMaxBatches;
                                                  // [R][rows] rank-start prefixes of owned experts
  __shared__ int32_t s_err[kClusterMaxCtas];      // last CTA: bad-expert bits, entry c from CTA c
  __shared__ int32_t s_cap[kClusterMaxCtas];      // last CTA: capacity bits, entry c from owner c
  __shared__ int32_t s_cta_err, s_cta_cap;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nthreads = kClusterWarps * 32;
  const uint32_t cta = cluster_cta_rank();
  const uint32_t ncta = gridDim.x;
  pdl_allow_dependents();
  // Peers' shared memory may be written only once every CTA of the cluster
  // has started: arrive now, wait just before the first remote store.
  cluster_arrive_relaxed();

  // 1. this warp's chunk; its routing loads go out before anything else
  const int chunk = (int)cta * kClusterWarps + warp;
  const bool has_chunk = chunk < p.num_chunks;
  int r = 0, j = 0, n_ent = 0;
  int64_t ent0 = 0;
  if (has_chunk) {
    r = chunk / p.chunks_per_rank;
    j = chunk % p.chunks_per_rank;
    const int64_t g0 = (int64_t)r * p.T + (int64_t)j * p.chunk_tokens;
    n_ent = min(p.chunk_tokens, p.T - j * p.chunk_tokens) * p.K;
    ent0 = g0 * p.K;
  }
  // entries of tokens beyond the rank's valid count are not routed
  const int routed_ent = has_chunk
      ? max(0, min(n_ent / p.K, rank_tokens(p, r) - j * p.chunk_tokens)) * p.K : 0;
  int e_in[kClusterMaxBatches];
#pragma unroll
  for (int b = 0; b < kClusterMaxBatches; ++b) {
    const int pl = b * 32 + lane;
    e_in[b] = (b < p.batches && pl < routed_ent) ? __ldg(p.topk_idx + ent0 + pl) : -1;
  }
  for (int i = tid; i < kClusterWarps * E; i += nthreads) wc[i] = 0;
  if (tid == 0) {
    s_cta_err = 0;
    s_cta_cap = 0;
  }
  int32_t my_err = 0;
  __syncthreads();

  int bits = 1;
  while ((1 << bits) < E) ++bits;
  const unsigned lt_mask = (1u << lane) - 1u;
  int lrank[kClusterMaxBatches];
  int lexp[kClusterMaxBatches];
#pragma unroll
  for (int b = 0; b < kClusterMaxBatches; ++b) {
    lrank[b] = 0;
    lexp[b] = -1;
    if (b >= p.batches) continue;                       // warp-uniform
    const int pl = b * 32 + lane;
    const int e = e_in[b];
    const bool routed = pl < routed_ent && !(p.masked && e == -1);
    const bool ok = routed && e >= 0 && e < E;
    if (routed && !ok) my_err |= (int32_t)kErrBadExpert;
    const unsigned same = peers_with_same_key(ok ? e : -1, bits);
    const int before = __popc(same & lt_mask);
    const int wbase = ok ? wc[warp * E + e] : 0;
    __syncwarp();
    if (ok && before == 0) wc[warp * E + e] = wbase + __popc(same);
    __syncwarp();
    lrank[b] = wbase + before;
    lexp[b] = ok ? e : -1;
  }
  my_err = __reduce_or_sync(0xFFFFFFFFu, my_err);
  if (lane == 0 && my_err) atomicOr(&s_cta_err, my_err);
  __syncthreads();
  cluster_wait();

  // 2. scan over the CTA's warps (all 16 counters loaded before any store)
  const int first_rank_warp =
      (p.chunks_per_rank - ((int)cta * kClusterWarps) % p.chunks_per_rank) % p.chunks_per_rank;
  for (int e = tid; e < E; e += nthreads) {
    int c[kClusterWarps];
#pragma unroll
    for (int w = 0; w < kClusterWarps; ++w) c[w] = wc[w * E + e];
    int run = 0;
#pragma unroll
    for (int w = 0; w < kClusterWarps; ++w) {
      const int cw = c[w];
      wc[w * E + e] = run;                         // exclusive prefix over the CTA's warps
      run += cw;
    }
    s_hist[e] = run;
    // 3a. to the owner of e: this CTA's count of e, and the in-CTA prefix
    //     of every chunk of this CTA that starts a rank
    const uint32_t owner = (uint32_t)(e / rows);
    const int oe = e - (int)owner * rows;
    st_dsmem(s_own + (int)cta * rows + oe, owner, run);
    for (int w = first_rank_warp; w < kClusterWarps; w += p.chunks_per_rank) {
      const int ch = (int)cta * kClusterWarps + w;
      if (ch >= p.num_chunks) break;
      st_dsmem(s_offs + (ch / p.chunks_per_rank) * rows + oe, owner, wc[w * E + e]);
    }
  }
  if (tid == 0) st_dsmem(s_err + cta, ncta - 1, s_cta_err);
  const bool last = cta == ncta - 1;

  // 3b. cluster barrier (every owner gets its experts' counts from every
  //     CTA), with this CTA's own scan, which needs nothing from the peers,
  //     between the two halves
  cluster_arrive_release();
  const int n_cta = block_exclusive_scan(s_hist, s_eoff, E);
  cluster_wait_acquire();

  // 3c. owners: each CTA's base for the owned experts (pushed to that CTA),
  //     the totals (counts), the capacity check, and the offsets rows
  const int e0 = (int)cta * rows, e1 = min(E, e0 + rows);
  int32_t cap_err = 0;
  for (int e = e0 + tid; e < e1; e += nthreads) {
    int run = 0;
    for (uint32_t c = 0; c < ncta; ++c) {
      const int h = s_own[(int)c * rows + (e - e0)];
      s_own[(int)c * rows + (e - e0)] = run;       // exclusive over CTAs
      st_dsmem(s_base + e, c, run);
      run += h;
    }
    p.expert_num_tokens[e] = run;
    s_tot[e - e0] = run;
    if (run > p.cap) cap_err = (int32_t)kErrCapacity;
  }
  cap_err = __reduce_or_sync(0xFFFFFFFFu, cap_err);
  if (lane == 0 && cap_err) atomicOr(&s_cta_cap, cap_err);
  __syncthreads();                                 // s_own, s_tot, s_cta_cap complete
  if (tid == 0) st_dsmem(s_cap + cta, ncta - 1, s_cta_cap);
  // 3d. cluster barrier (every CTA gets its bases for all experts, the last
  //     CTA every error bit; no remote access follows), with the owned
  //     offsets rows, which need nothing from the peers, between the halves
  cluster_arrive_release();
  {
    // offsets[e][r] = (counts of the CTAs before the one where rank r
    // starts) + (in-CTA prefix pushed by that CTA); rows [e0, e1) of the
    // matrix, one contiguous run
    const int R1 = p.R + 1;
    for (int i = tid; i < (e1 - e0) * R1; i += nthreads) {
      const int e = e0 + i / R1, rr = i % R1;
      const int cr = (rr * p.chunks_per_rank) / kClusterWarps;   // CTA where rank rr starts
      p.expert_rank_offsets[(int64_t)e0 * R1 + i] =
          rr == p.R ? s_tot[e - e0] : s_own[cr * rows + (e - e0)] + s_offs[rr * rows + (e - e0)];
    }
  }

  cluster_wait_acquire();

  // 4. slots; return addresses staged in (expert, slot) order so that the
  //    src_of rows go out as contiguous runs
  int32_t *stage_v = s_stage;
  int32_t *stage_e = s_stage + kClusterWarps * 32 * kClusterMaxBatches;
#pragma unroll
  for (int b = 0; b < kClusterMaxBatches; ++b) {
    if (b >= p.batches) continue;
    const int pl = b * 32 + lane;
    if (pl >= n_ent) continue;
    const int e = lexp[b];
    if (e < 0) {
      p.slot_of[ent0 + pl] = -1;
      continue;
    }
    const int local = wc[warp * E + e] + lrank[b];       // rank among this CTA's entries of e
    p.slot_of[ent0 + pl] = s_base[e] + local;
    stage_v[s_eoff[e] + local] = (int32_t)(ent0 + pl);
    stage_e[s_eoff[e] + local] = e;
  }
  __syncthreads();
  for (int i = tid; i < n_cta; i += nthreads) {
    const int e = stage_e[i];
    const int slot = s_base[e] + (i - s_eoff[e]);
    if (slot < p.cap) p.src_of[(int64_t)e * p.cap + slot] = stage_v[i];
  }
  if (last) {
    int32_t err = tid < (int)ncta ? (s_err[tid] | s_cap[tid]) : 0;
    err = __reduce_or_sync(0xFFFFFFFFu, err);
    if (tid == 0)
      p.hdr->status = (err & kErrBadExpert) ? MOE_ERR_BAD_EXPERT
                      : (err & kErrCapacity) ? MOE_ERR_CAPACITY : MOE_OK;
  }
}

__global__ void set_debug_kernel(WsHeader *hdr, uint32_t flags, uint64_t timeout_ns) {
  hdr->debug_flags = flags;
  hdr->timeout_ns = timeout_ns;
}

namespace {

// Chunking for the single-cluster path: the fewest entries per warp (so the
// most CTAs, which share the scattered stores) such that all rank-aligned
// chunks fit 16 CTAs of 16 warps.
bool cluster_geometry(PlanParams &p) {
  if (p.E > kClusterMaxExperts) return false;
  for (int max_ctas : {kClusterMaxCtas})
  for (int b = 1; b <= kClusterMaxBatches; ++b) {
    int tw = (32 * b) / p.K;
    if (tw < 1) continue;
    if (tw > p.T) tw = p.T;
    const int cpr = (p.T + tw - 1) / tw;
    const int64_t nc = (int64_t)p.R * cpr;
    if (nc <= (int64_t)max_ctas * kClusterWarps) {
      p.chunk_tokens = tw;
      p.chunks_per_rank = cpr;
      p.num_chunks = (int)nc;
      p.batches = (tw * p.K + 31) / 32;
      return true;
    }
  }
  return false;
}

struct ClusterFit {
  int ctas = 0;
  size_t smem = 0;
  int ok = -1;   // -1 unknown, 0 no, 1 yes
};
ClusterFit cluster_fit_cache[64];

// Can a cluster of `ctas` blocks with `smem` bytes each be scheduled?
cudaError_t cluster_fits(int ctas, size_t smem, bool *fits) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  ClusterFit &c = cluster_fit_cache[(dev >= 0 && dev < 64) ? dev : 0];
  if (c.ok >= 0 && c.ctas == ctas && c.smem == smem) {
    *fits = c.ok == 1;
    return cudaSuccess;
  }
  if (ctas > 8) {
    e = cudaFuncSetAttribute(plan_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(plan_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kClusterWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, plan_cluster_kernel, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  c.ctas = ctas;
  c.smem = smem;
  c.ok = n > 0 ? 1 : 0;
  *fits = n > 0;
  return cudaSuccess;
}

cudaError_t launch_plan_cluster(const PlanParams &p, int ctas, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kClusterWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_cluster_kernel, p);
}

}  // namespace

cudaError_t launch_plan(const PlanParams &p_in, cudaStream_t stream) {
  PlanParams p = p_in;
  if (cluster_geometry(p)) {
    const int ctas = (p.num_chunks + kClusterWarps - 1) / kClusterWarps;
    const size_t rows = (size_t)((p.E + ctas - 1) / ctas);
    const size_t csmem = ((size_t)(kClusterWarps + 3) * p.E + (kClusterMaxCtas + 1) * rows +
                          (size_t)p.R * rows + 2 * kClusterWarps * 32 * kClusterMaxBatches) *
                         sizeof(int32_t);
    bool fits = false;
    cudaError_t e = csmem <= kClusterMaxSmem ? cluster_fits(ctas, csmem, &fits) : cudaSuccess;
    if (e != cudaSuccess) return e;
    if (fits) {
      e = launch_plan_cluster(p, ctas, csmem, stream);
      if (e != cudaSuccess) return e;
      return cudaGetLastError();
    }
  }
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
