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
// SiLU(g) = g / (1 + e^-g) with e^x computed by a fixed sequence of IEEE
// binary32 operations (Cody-Waite reduction with a two-part ln 2, a degree-7
// Taylor polynomial in Horner form with fused multiply-adds, exact scaling by
// 2^n), so that the result, and therefore every quantised byte, is
// reproducible bit for bit on any implementation of the same steps.
//
// How: persistent grid; each block scans the clamped counts into a prefix in
// shared memory, then warps take (row, segment) tasks over the populated rows
// only and find a task's expert by binary search.  A task is 1024 elements
// of a (8 blocks of 128): each half-warp loads 8 gate and 8 up values per
// lane (16-byte loads), computes a in registers and quantises its block.
#include <math.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kActThreads = 256;
constexpr unsigned kWarpAll = 0xFFFFFFFFu;

// e^x; +inf above 88.72 and 0 below -87.33 (the steps of the file comment).
__device__ __forceinline__ float exp_fixed(float x) {
  const float xc = fminf(fmaxf(x, -87.33f), 88.72f);
  const float n = rintf(__fmul_rn(xc, 1.44269502f));          // log2(e)
  float r = __fmaf_rn(-n, 0.693145751953125f, xc);           // ln2, high 16 bits
  r = __fmaf_rn(-n, 1.42860677e-06f, r);                     // ln2, low part
  float p = 1.98412701e-04f;                                 // 1/7!
  p = __fmaf_rn(p, r, 1.38888892e-03f);                      // 1/6!
  p = __fmaf_rn(p, r, 8.33333377e-03f);                      // 1/5!
  p = __fmaf_rn(p, r, 4.16666679e-02f);                      // 1/4!
  p = __fmaf_rn(p, r, 1.66666672e-01f);                      // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  int ni = (int)n;
  const bool big = ni > 127;                                 // 2^128 is not a float
  p = big ? __fmul_rn(p, 2.0f) : p;
  ni = big ? ni - 1 : ni;
  const float v = __fmul_rn(p, __int_as_float((ni + 127) << 23));
  return x > 88.72f ? __int_as_float(0x7F800000) : (x < -87.33f ? 0.0f : v);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp_fixed(-g))), u);
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

template <int P>
__global__ void __launch_bounds__(kActThreads)
silu_quant_kernel(ActParams p) {
  extern __shared__ int32_t s_prefix[];                     // [E + 1]
  __shared__ int32_t s_status;
  pdl_wait_for_previous();
  if (threadIdx.x == 0) s_status = read_status(p.hdr);
  count_prefix(p.expert_num_tokens, p.E, p.cap, s_prefix);
  if (s_status != MOE_OK) return;

  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int64_t warp0 = ((int64_t)blockIdx.x * kActThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kActThreads) >> 5;
  const int nb = p.I / 128;
  constexpr int bpt = 2 * P;
  const int tpr = (nb + bpt - 1) / bpt;
  const int64_t ntasks = (int64_t)s_prefix[p.E] * tpr;

  for (int64_t task = warp0; task < ntasks; task += nwarps) {
    const int rg = (int)(task / tpr);
    const int seg = (int)(task - (int64_t)rg * tpr);
    int lo = 0, hi = p.E;                                   // last e with prefix[e] <= rg
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= rg) lo = mid;
      else hi = mid;
    }
    const int64_t row = (int64_t)lo * p.cap + (rg - s_prefix[lo]);
    const uint16_t *gate = p.expert_h + row * 2 * p.I;
    const uint16_t *up = gate + p.I;
    uint4 gv[P], uv[P];
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const int blk = seg * bpt + it * 2 + half;
      const int64_t off = (int64_t)blk * 128 + sub * 8;
      gv[it] = blk < nb ? __ldcs(reinterpret_cast<const uint4 *>(gate + off)) : make_uint4(0, 0, 0, 0);
      uv[it] = blk < nb ? __ldcs(reinterpret_cast<const uint4 *>(up + off)) : make_uint4(0, 0, 0, 0);
    }
    float my_scale = 0.0f;
    uint8_t *qrow = static_cast<uint8_t *>(p.act_q) + row * p.I;
#pragma unroll
    for (int it = 0; it < P; ++it) {
      const uint32_t gw[4] = {gv[it].x, gv[it].y, gv[it].z, gv[it].w};
      const uint32_t uw[4] = {uv[it].x, uv[it].y, uv[it].z, uv[it].w};
      float a[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[2 * i] = silu_mul(bf16_lo(gw[i]), bf16_lo(uw[i]));
        a[2 * i + 1] = silu_mul(bf16_hi(gw[i]), bf16_hi(uw[i]));
      }
      float scale;
      const uint2 q = quantise_block8(a, &scale);
      const int blk = seg * bpt + it * 2 + half;
      if (blk < nb) *reinterpret_cast<uint2 *>(qrow + (int64_t)blk * 128 + sub * 8) = q;
      const float s_even = __shfl_sync(kWarpAll, scale, 0);
      const float s_odd = __shfl_sync(kWarpAll, scale, 16);
      if (lane == it * 2) my_scale = s_even;
      if (lane == it * 2 + 1) my_scale = s_odd;
    }
    if (lane < min(bpt, nb - seg * bpt)) p.act_scale[row * nb + seg * bpt + lane] = my_scale;
  }
}

namespace {
template <int P>
cudaError_t launch_p(const ActParams &p, cudaStream_t stream) {
  const size_t smem = (size_t)(p.E + 1) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(silu_quant_kernel<P>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // enough warps for every row of every expert at full capacity, capped at a full device
  const int64_t tasks = (int64_t)p.E * p.cap * ((p.I / 128 + 2 * P - 1) / (2 * P));
  const int grid = persistent_grid((const void *)silu_quant_kernel<P>, kActThreads, tasks);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, silu_quant_kernel<P>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_silu_quant(const ActParams &p, cudaStream_t stream) {
  const int nb = p.I / 128;
  if (nb % 8 == 0) return launch_p<4>(p, stream);
  if (nb % 4 == 0) return launch_p<2>(p, stream);
  return launch_p<1>(p, stream);
}

}  // namespace moe
