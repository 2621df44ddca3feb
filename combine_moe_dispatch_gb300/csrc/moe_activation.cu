// moe_activation.cu -- SiLU(gate) * up with 1x128 E4M3 re-quantisation over
// the padded per-expert buffers, driven by the per-expert token counts.
//
// What it computes ("Lower latency and higher throughput with multi-node
// DeepSeek deployment", Quantization): between the two expert GEMMs, for
// expert e and row s < clamp(expert_num_tokens[e], 0, cap),
//   a = SiLU(gate) * up,  gate, up = the two halves of expert_h[e][s],
// then one scale per 128 elements of a (amax/448) and the E4M3 bytes
// e4m3(RN(a / scale)) -- the same rule as the fp8 dispatch.  Rows at or
// beyond the count are not touched, so the kernel stays correct inside a CUDA
// graph whatever the routing (the pages: kernels must read the per-expert
// counts rather than plan their work from the buffer sizes).
//
// SiLU(g) = g / (1 + e^-g) in binary32, with e^x by a fixed sequence of IEEE
// operations (Cody-Waite reduction with a two-part ln 2, a degree-7 Taylor
// polynomial by Horner with fused multiply-adds, exact scaling by 2^n), so
// every byte is reproducible.  The gate is bf16, so SiLU(g) is a function of
// 16 bits, and the kernel looks it up instead of evaluating it:
//  * 2^-25 <= |g| < 128: a table of the 8192 values, generated at build time
//    by silu_table_gen.cpp with that sequence and staged in shared memory;
//  * |g| < 2^-25: e^-g rounds to exactly 1, so SiLU(g) = g / 2 = g * 0.5;
//  * |g| >= 128: for g > 0, e^-g is below 2^-25 (or 0), so 1 + e^-g == 1 and
//    SiLU(g) = g; for g < 0, e^-g = +inf and g / inf = -0, which g * 0 also
//    gives (with NaN for g = -inf, as the division does).
// The product with up and the quantisation are evaluated as written.
//
// How: persistent grid; each block stages the table (before waiting on the
// previous kernel, which it does not depend on) and scans the clamped counts
// into a prefix in shared memory; then each warp takes a contiguous range of
// (row, segment) tasks over the populated rows only (its first task's expert
// by binary search, the next ones by walking forward).  A task is 2P blocks
// of 128 elements: each half-warp loads 8 gate and 8 up values per lane per
// block pair (16-byte loads), and the loads of a warp's next task are issued
// before the current one is computed.  Each block's scale
// and reciprocal are computed once, by the lane that stores the scale, and
// handed to the half-warp that quantises the block by shuffle.
#include "moe_common.cuh"

namespace moe {

constexpr int kActThreads = 256;
constexpr unsigned kWarpAll = 0xFFFFFFFFu;
constexpr int kSiluTabEntries = 8192;   // sign x 32 binades x 128 mantissas
constexpr int kSiluTabE0 = 102;         // biased exponent of 2^-25

__device__ __align__(16) const uint32_t g_silu_table[kSiluTabEntries] = {
#include "silu_table.inc"
};

// SiLU(g) for the bf16 pattern h (in the low 16 bits), every case of the
// file comment.
__device__ __forceinline__ float silu_bf16(uint32_t h, const float *s_tab) {
  const float g = __uint_as_float(h << 16);
  const int t = (int)(h & 0x7FFFu) - (kSiluTabE0 << 7);
  const bool in_tab = (unsigned)t < (unsigned)(kSiluTabEntries / 2);
  const float tab = s_tab[(in_tab ? (uint32_t)t : 0u) | ((h >> 15) << 12)];
  const float small = __fmul_rn(g, 0.5f);
  const float large = g > 0.0f ? g : __fmul_rn(g, 0.0f);
  return in_tab ? tab : (t < 0 ? small : large);
}

// Table lookups of SiLU for the 8 bf16 gates in gw (two per word, low half
// first).  Both halves of a word are indexed at once: with the sign bits
// cleared, adding 0x4D00 to each half (no carry can cross) maps the table's
// magnitudes [102 << 7, 134 << 7) to [0x8000, 0x9000), so a half is in the
// table iff its top nibble is 1000b, and its low 12 bits are the index (the
// sign adds 4096).  The byte offset is masked into range, so every lookup is
// in bounds; *outside collects the words a caller must redo exactly
// (silu_bf16) when (*outside & 0xF000F000) != 0.
__device__ __forceinline__ void silu8_table(const uint4 &g, const float *s_tab, float (&sv)[8],
                                            uint32_t &outside) {
  const unsigned char *tab = reinterpret_cast<const unsigned char *>(s_tab);
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t d = (gw[i] & 0x7FFF7FFFu) + 0x4D004D00u;
    outside |= d ^ 0x80008000u;
    const uint32_t o0 = ((d << 2) & 0x3FFCu) | ((gw[i] >> 1) & 0x4000u);
    const uint32_t o1 = ((d >> 14) & 0x3FFCu) | ((gw[i] >> 17) & 0x4000u);
    sv[2 * i] = *reinterpret_cast<const float *>(tab + o0);
    sv[2 * i + 1] = *reinterpret_cast<const float *>(tab + o1);
  }
}


// Exclusive prefix of clamp(count[e], 0, cap) over e into out[0..E], by the
// whole block (any E).
__device__ void count_prefix(const int32_t *count, int E, int cap, int32_t *out) {
  __shared__ int32_t s_warp[kActThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + kActThreads - 1) / kActThreads;     // consecutive entries per thread
  const int e0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) local += min(max(__ldg(count + e), 0), cap);
  }
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(kWarpAll, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  int run = before + incl - local;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E) {
      out[e] = run;
      run += min(max(__ldg(count + e), 0), cap);
    }
  }
  if (tid == kActThreads - 1) out[E] = run;
  __syncthreads();
}

// The expert whose populated rows hold row number rg: the last e with
// prefix[e] <= rg.
__device__ __forceinline__ int populated_expert(const int32_t *s_prefix, int E, int rg) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= rg) lo = mid;
    else hi = mid;
  }
  return lo;
}

// The 2P blocks of task (row, seg): lane (half, sub) loads elements
// [blk * 128 + sub * 8, + 8) of block blk = seg * 2P + 2 * it + half of the
// gate and the up half.  EXACT: the row is a whole number of tasks, so every
// block exists; otherwise blocks past the row read as zeros.  SHORT
// (I % 128 != 0, I % 16 == 0): the last block is short, and a lane's 8
// elements past the row's end read as zeros.
template <int P, bool EXACT, bool SHORT = false>
__device__ __forceinline__ void load_task(const ActParams &p, int64_t row, int seg, int half, int sub,
                                          int nb, uint4 (&gv)[P], uint4 (&uv)[P]) {
  const uint16_t *gate = p.expert_h + row * 2 * p.I + (int64_t)seg * (2 * P * 128) + half * 128 + sub * 8;
  const uint16_t *up = gate + p.I;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const int blk = seg * 2 * P + it * 2 + half;
    const bool ok = SHORT ? blk * 128 + sub * 8 < p.I : (EXACT || blk < nb);
    gv[it] = ok ? __ldcs(reinterpret_cast<const uint4 *>(gate + it * 256)) : make_uint4(0, 0, 0, 0);
    uv[it] = ok ? __ldcs(reinterpret_cast<const uint4 *>(up + it * 256)) : make_uint4(0, 0, 0, 0);
  }
}

// One task: SiLU(gate) * up for the 2P blocks in gv/uv, the block scales
// (computed once each, by lanes 0 .. 2P-1, which also store them) and the
// E4M3 bytes.  All 32 lanes call it together.
template <int P, bool EXACT, bool TS, bool SHORT = false>
__device__ __forceinline__ void act_task(const ActParams &p, const float *s_tab, int64_t row, int seg,
                                         int lane, int nb, const uint4 (&gv)[P], const uint4 (&uv)[P]) {
  const int half = lane >> 4;
  const int sub = lane & 15;
  constexpr int bpt = 2 * P;
  float a[P][8];
  uint32_t outside = 0;
#pragma unroll
  for (int it = 0; it < P; ++it) silu8_table(gv[it], s_tab, a[it], outside);
  if (__any_sync(kWarpAll, (outside & 0xF000F000u) != 0)) {   // a gate outside the table: exact cases
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const uint32_t gw[4] = {gv[it].x, gv[it].y, gv[it].z, gv[it].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[it][2 * i] = silu_bf16(gw[i] & 0xFFFFu, s_tab);
        a[it][2 * i + 1] = silu_bf16(gw[i] >> 16, s_tab);
      }
    }
  }
  float am[P];
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const uint32_t uw[4] = {uv[it].x, uv[it].y, uv[it].z, uv[it].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[it][2 * i] = __fmul_rn(a[it][2 * i], bf16_lo(uw[i]));
      a[it][2 * i + 1] = __fmul_rn(a[it][2 * i + 1], bf16_hi(uw[i]));
    }
    am[it] = half_warp_amax(a[it]);
  }
  // lane L < 2P owns block seg*2P + L: amax from half L & 1 of pair L >> 1
  float mine = 0.0f;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const float v = __shfl_sync(kWarpAll, am[it], (lane & 1) * 16);
    if ((lane >> 1) == it) mine = v;
  }
  float my_scale = div448_fast(mine);
  const bool tiny = mine != 0.0f && !(mine >= 0x1p-120f && mine <= 3.4028234e38f);
  if (__any_sync(kWarpAll, tiny)) {
    if (tiny) my_scale = __fdiv_rn(mine, 448.0f);
  }
  const float my_r = mine == 0.0f ? 1.0f : __frcp_rn(my_scale);

  // bytes from RN(a * r) where provably exact, else by division (per element)
  uint2 q[P];
  float scale[P], r[P];
  bool zero[P];
#pragma unroll
  for (int it = 0; it < P; ++it) {
    scale[it] = __shfl_sync(kWarpAll, my_scale, it * 2 + half);
    r[it] = __shfl_sync(kWarpAll, my_r, it * 2 + half);
    zero[it] = am[it] == 0.0f;
  }
  quantise_blocks<P>(a, scale, r, zero, q);
  uint8_t *qrow = static_cast<uint8_t *>(p.act_q) + row * p.I + (int64_t)seg * (bpt * 128) + half * 128 + sub * 8;
#pragma unroll
  for (int it = 0; it < P; ++it) {
    const int blk = seg * bpt + it * 2 + half;
    const bool in = SHORT ? blk * 128 + sub * 8 < p.I : (EXACT || blk < nb);
    if (in) *reinterpret_cast<uint2 *>(qrow + it * 256) = q[it];
  }
  if (lane < min(bpt, nb - seg * bpt)) {
    const int blk = seg * bpt + lane;
    int64_t at = row * nb + blk;                      // [E, cap, I/128]
    if (TS) {                                         // [E, I/128, cap]; E * cap < 2^31
      const int e = (int)row / p.cap, s = (int)row - e * p.cap;
      at = ((int64_t)e * nb + blk) * p.cap + s;
    }
    p.act_scale[at] = my_scale;
  }
}

// Walks a warp's contiguous range of (populated row, segment) tasks.
struct ActCursor {
  int64_t row;
  int rg, seg, e;
  __device__ __forceinline__ void next(const int32_t *s_prefix, int E, int cap, int tpr) {
    if (++seg == tpr) {
      seg = 0;
      ++rg;
      while (e + 1 < E && s_prefix[e + 1] <= rg) ++e;   // experts without rows are skipped
    }
    row = (int64_t)e * cap + (rg - s_prefix[e]);
  }
};

template <int P, bool EXACT, bool TS, bool SHORT = false>
__global__ void __launch_bounds__(kActThreads, P >= 2 ? 3 : 1)
silu_quant_kernel(ActParams p) {
  __shared__ __align__(16) float s_tab[kSiluTabEntries];
  extern __shared__ __align__(16) int32_t s_prefix[];                  // [E + 1]
  __shared__ int32_t s_status;
  pdl_allow_dependents();
  for (int i = threadIdx.x; i < kSiluTabEntries / 4; i += kActThreads)
    reinterpret_cast<uint4 *>(s_tab)[i] = __ldg(reinterpret_cast<const uint4 *>(g_silu_table) + i);
  pdl_wait_for_previous();
  if (threadIdx.x == 0) s_status = read_status(p.hdr);
  count_prefix(p.expert_num_tokens, p.E, p.cap, s_prefix);   // ends with __syncthreads
  if (s_status != MOE_OK) return;

  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int64_t warp0 = ((int64_t)blockIdx.x * kActThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kActThreads) >> 5;
  const int nb = SHORT ? (p.I + 127) / 128 : p.I / 128;   // SHORT: the last block is short
  const int tpr = (nb + 2 * P - 1) / (2 * P);
  // each warp takes a contiguous range of tasks, so the row and its expert
  // advance incrementally from one task to the next
  const int64_t ntasks = (int64_t)s_prefix[p.E] * tpr;
  const int64_t per_warp = (ntasks + nwarps - 1) / nwarps;
  const int64_t t0 = warp0 * per_warp;
  const int64_t t1 = min(ntasks, t0 + per_warp);
  if (t0 >= t1) return;
  int n = (int)(t1 - t0);                                    // tasks left, the current one included

  ActCursor c;
  c.rg = (int)(t0 / tpr);
  c.seg = (int)(t0 - (int64_t)c.rg * tpr);
  c.e = populated_expert(s_prefix, p.E, c.rg);
  c.row = (int64_t)c.e * p.cap + (c.rg - s_prefix[c.e]);
  // two register buffers in turn: the next task's rows load while this one computes
  uint4 ga[P], ua[P], gb[P], ub[P];
  load_task<P, EXACT, SHORT>(p, c.row, c.seg, half, sub, nb, ga, ua);
  for (;;) {
    ActCursor nc = c;
    nc.next(s_prefix, p.E, p.cap, tpr);
    if (n > 1) load_task<P, EXACT, SHORT>(p, nc.row, nc.seg, half, sub, nb, gb, ub);
    act_task<P, EXACT, TS, SHORT>(p, s_tab, c.row, c.seg, lane, nb, ga, ua);
    if (--n == 0) break;
    c = nc;
    nc.next(s_prefix, p.E, p.cap, tpr);
    if (n > 1) load_task<P, EXACT, SHORT>(p, nc.row, nc.seg, half, sub, nb, ga, ua);
    act_task<P, EXACT, TS, SHORT>(p, s_tab, c.row, c.seg, lane, nb, gb, ub);
    if (--n == 0) break;
    c = nc;
  }
}

namespace {
template <int P, bool EXACT, bool TS, bool SHORT = false>
cudaError_t launch_p(const ActParams &p, cudaStream_t stream) {
  const size_t smem = (size_t)(p.E + 1) * sizeof(int32_t);
  // enough warps for every row of every expert at full capacity, capped at a full device
  const int64_t tasks = (int64_t)p.E * p.cap * (((p.I + 127) / 128 + 2 * P - 1) / (2 * P));
  const int grid =
      persistent_grid((const void *)silu_quant_kernel<P, EXACT, TS, SHORT>, kActThreads, tasks);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kActThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, silu_quant_kernel<P, EXACT, TS, SHORT>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

template <bool TS>
cudaError_t launch_layout(const ActParams &p, cudaStream_t stream) {
  if (p.I % 128 != 0) return launch_p<1, false, TS, true>(p, stream);   // a short last block
  const int nb = p.I / 128;
  if (nb % 4 == 0) return launch_p<2, true, TS>(p, stream);
  if (nb % 2 == 0) return launch_p<1, true, TS>(p, stream);
  return launch_p<1, false, TS>(p, stream);
}

cudaError_t launch_silu_quant(const ActParams &p, cudaStream_t stream) {
  // the scale layout is a template parameter: the default layout's kernel
  // carries no code for the other
  return p.scale_t ? launch_layout<true>(p, stream) : launch_layout<false>(p, stream);
}

}  // namespace moe
