// moe_api.cu -- the C ABI of libmoe_gb300.so (declared in moe_dispatch.h):
// host-side argument checks, workspace sizing and kernel launches.  Every
// check here happens before anything is enqueued, so a rejected call leaves
// the stream and the caller's buffers untouched.
#include <stdint.h>

#include <mutex>

#include "moe_common.cuh"

namespace moe {

int device_sm_count() {
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

int occupancy_blocks(const void *kern, int threads, size_t smem) {
  struct Entry {
    const void *kern;
    int dev, threads;
    size_t smem;
    int blocks;
  };
  static Entry cache[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].kern == kern && cache[i].dev == dev && cache[i].threads == threads &&
        cache[i].smem == smem)
      return cache[i].blocks;
  int v = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem) != cudaSuccess || v < 1) {
    cudaGetLastError();
    v = 1;
  }
  if (used < 64) cache[used++] = Entry{kern, dev, threads, smem, v};
  return v;
}

int persistent_grid(const void *kern, int threads, int64_t warp_tasks) {
  const int64_t want = (warp_tasks + threads / 32 - 1) / (threads / 32);
  const int64_t cap = (int64_t)device_sm_count() * occupancy_blocks(kern, threads, 0);
  const int64_t g = want < cap ? want : cap;
  return (int)(g < 1 ? 1 : g);
}

namespace {

moe_status check_shape(const moe_shape *s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->num_ranks <= 0 || s->tokens_per_rank < 0 || s->hidden <= 0 || s->num_experts <= 0 ||
      s->top_k <= 0 || s->capacity <= 0)
    return MOE_ERR_INVALID_ARG;
  if (s->payload != MOE_PAYLOAD_BF16 && s->payload != MOE_PAYLOAD_FP8_E4M3 &&
      s->payload != MOE_PAYLOAD_FP8_E4M3_TSCALE)
    return MOE_ERR_INVALID_ARG;
  if (s->top_k > kMaxTopK || s->num_experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  const int64_t N = (int64_t)s->num_ranks * s->tokens_per_rank;
  if (N * s->top_k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)s->num_experts * s->capacity >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (s->hidden % 8 != 0) return MOE_ERR_UNSUPPORTED;
  // fp8: rows of any multiple of 16 elements (the last 128-element scale
  // block may be short); each 16-byte store is then all in or all past a row
  if (s->payload != MOE_PAYLOAD_BF16 && s->hidden % 16 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

WsHeader *header(void *ws) { return static_cast<WsHeader *>(ws); }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_shape *shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return ws_layout(*shape).total;
}

moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return MOE_ERR_ALIGNMENT;
  return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream));
}

static moe_status plan_common(const moe_shape *shape, const int32_t *topk_idx,
                              const int32_t *num_tokens, int masked, int32_t *expert_num_tokens,
                              int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of,
                              void *workspace, size_t workspace_bytes, void *stream);

moe_status moe_plan(const moe_shape *shape, const int32_t *topk_idx, int32_t *expert_num_tokens,
                    int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of,
                    void *workspace, size_t workspace_bytes, void *stream) {
  return plan_common(shape, topk_idx, nullptr, 0, expert_num_tokens, expert_rank_offsets, slot_of,
                     src_of, workspace, workspace_bytes, stream);
}

moe_status moe_plan_masked(const moe_shape *shape, const int32_t *topk_idx,
                           const int32_t *num_tokens, int32_t *expert_num_tokens,
                           int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of,
                           void *workspace, size_t workspace_bytes, void *stream) {
  if (num_tokens && ((uintptr_t)num_tokens & 3u)) return MOE_ERR_ALIGNMENT;
  return plan_common(shape, topk_idx, num_tokens, 1, expert_num_tokens, expert_rank_offsets,
                     slot_of, src_of, workspace, workspace_bytes, stream);
}

static moe_status plan_common(const moe_shape *shape, const int32_t *topk_idx,
                              const int32_t *num_tokens, int masked, int32_t *expert_num_tokens,
                              int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of,
                              void *workspace, size_t workspace_bytes, void *stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const bool empty = shape->tokens_per_rank == 0;   // topk_idx, slot_of may then be NULL
  if ((!empty && (!topk_idx || !slot_of)) || !expert_num_tokens || !expert_rank_offsets || !src_of)
    return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < ws_layout(*shape).total) return MOE_ERR_WORKSPACE;
  if (!aligned(topk_idx, 4) || !aligned(expert_num_tokens, 4) || !aligned(expert_rank_offsets, 4) ||
      !aligned(slot_of, 4) || !aligned(src_of, 4) || !aligned(workspace, 16))
    return MOE_ERR_ALIGNMENT;

  const PlanGeometry g = plan_geometry(*shape);
  const WsLayout L = ws_layout(*shape);
  cudaStream_t s = (cudaStream_t)stream;
  if (g.num_tiles == 0) {   // empty batch: zero counts and offsets, status OK
    if (cudaMemsetAsync(expert_num_tokens, 0, sizeof(int32_t) * shape->num_experts, s) != cudaSuccess ||
        cudaMemsetAsync(expert_rank_offsets, 0,
                        sizeof(int32_t) * shape->num_experts * (shape->num_ranks + 1), s) != cudaSuccess ||
        cudaMemsetAsync(&header(workspace)->status, 0, sizeof(int32_t), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  char *base = static_cast<char *>(workspace);
  PlanParams p;
  p.topk_idx = topk_idx;
  p.num_tokens = num_tokens;
  p.masked = masked;
  p.expert_num_tokens = expert_num_tokens;
  p.expert_rank_offsets = expert_rank_offsets;
  p.slot_of = slot_of;
  p.src_of = src_of;
  p.hdr = header(workspace);
  p.agg_tag = reinterpret_cast<uint32_t *>(base + L.tags_off);
  p.incl_tag = p.agg_tag + g.num_tiles;
  p.agg = reinterpret_cast<int32_t *>(base + L.rows_off);
  p.incl = p.agg + (size_t)g.num_tiles * shape->num_experts;
  p.R = shape->num_ranks;
  p.T = shape->tokens_per_rank;
  p.E = shape->num_experts;
  p.K = shape->top_k;
  p.cap = shape->capacity;
  p.tile_tokens = g.tile_tokens;
  p.tiles_per_rank = g.tiles_per_rank;
  p.num_tiles = g.num_tiles;
  return from_cuda(launch_plan(p, s));
}

moe_status moe_dispatch(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                        const int32_t *slot_of, void *expert_x, float *expert_x_scale,
                        void *workspace, void *stream) {
  return moe_dispatch_ex(shape, x, topk_idx, slot_of, expert_x, expert_x_scale, workspace, stream, 0u);
}

moe_status moe_dispatch_ex(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                           const int32_t *slot_of, void *expert_x, float *expert_x_scale,
                           void *workspace, void *stream, uint32_t flags) {
  if ((flags & ~(uint32_t)MOE_DISPATCH_EARLY_X) != 0u) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->tokens_per_rank == 0) return MOE_OK;   // empty batch: nothing to read or write
  const bool fp8 = shape->payload != MOE_PAYLOAD_BF16;
  if (!x || !topk_idx || !slot_of || !expert_x || (fp8 && !expert_x_scale))
    return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(expert_x, 16) || !aligned(topk_idx, 4) || !aligned(slot_of, 4) ||
      (fp8 && !aligned(expert_x_scale, 4)) || !aligned(workspace, 16))
    return MOE_ERR_ALIGNMENT;
  DispatchParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.topk_idx = topk_idx;
  p.slot_of = slot_of;
  p.expert_x = expert_x;
  p.expert_x_scale = fp8 ? expert_x_scale : nullptr;
  p.hdr = header(workspace);
  p.N = shape->num_ranks * shape->tokens_per_rank;
  p.H = shape->hidden;
  p.E = shape->num_experts;
  p.K = shape->top_k;
  p.cap = shape->capacity;
  p.scale_t = shape->payload == MOE_PAYLOAD_FP8_E4M3_TSCALE;
  p.early_x = (flags & MOE_DISPATCH_EARLY_X) ? 1 : 0;
  cudaStream_t s = (cudaStream_t)stream;
  return from_cuda(fp8 ? launch_dispatch_fp8(p, s) : launch_dispatch_bf16(p, s));
}

moe_status moe_plan_dispatch(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                             int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                             int32_t *slot_of, int32_t *src_of, void *expert_x,
                             float *expert_x_scale, void *workspace, size_t workspace_bytes,
                             void *stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const bool fp8 = shape->payload != MOE_PAYLOAD_BF16;
  const bool empty = shape->tokens_per_rank == 0;
  if (!empty && (!x || !expert_x || (fp8 && !expert_x_scale))) return MOE_ERR_INVALID_ARG;
  if (!empty && (!aligned(x, 16) || !aligned(expert_x, 16) || (fp8 && !aligned(expert_x_scale, 4))))
    return MOE_ERR_ALIGNMENT;
  FusedParams f;
  if (empty || !plan_dispatch_geometry(*shape, f)) {
    // outside the fused path's limits: the plan, then the dispatch
    st = plan_common(shape, topk_idx, nullptr, 0, expert_num_tokens, expert_rank_offsets, slot_of,
                     src_of, workspace, workspace_bytes, stream);
    if (st != MOE_OK || empty) return st;
    // The kernel before the dispatch is this call's own plan, an ordinary
    // launch that began after every earlier kernel (whatever wrote x) had
    // completed, and that never writes x: the dispatch may read x early.
    return moe_dispatch_ex(shape, x, topk_idx, slot_of, expert_x, expert_x_scale, workspace,
                           stream, MOE_DISPATCH_EARLY_X);
  }
  if (!topk_idx || !slot_of || !expert_num_tokens || !expert_rank_offsets || !src_of)
    return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < ws_layout(*shape).total) return MOE_ERR_WORKSPACE;
  if (!aligned(topk_idx, 4) || !aligned(expert_num_tokens, 4) || !aligned(expert_rank_offsets, 4) ||
      !aligned(slot_of, 4) || !aligned(src_of, 4) || !aligned(workspace, 16))
    return MOE_ERR_ALIGNMENT;
  f.d.x = static_cast<const uint16_t *>(x);
  f.d.topk_idx = topk_idx;
  f.d.slot_of = slot_of;
  f.d.expert_x = expert_x;
  f.d.expert_x_scale = fp8 ? expert_x_scale : nullptr;
  f.d.hdr = header(workspace);
  f.d.N = shape->num_ranks * shape->tokens_per_rank;
  f.d.H = shape->hidden;
  f.d.E = shape->num_experts;
  f.d.K = shape->top_k;
  f.d.cap = shape->capacity;
  f.d.scale_t = shape->payload == MOE_PAYLOAD_FP8_E4M3_TSCALE;
  f.d.early_x = 1;   // unused: the fused kernel is an ordinary launch
  f.topk_idx = topk_idx;
  f.expert_num_tokens = expert_num_tokens;
  f.expert_rank_offsets = expert_rank_offsets;
  f.slot_of = slot_of;
  f.src_of = src_of;
  f.vec_idx = aligned(topk_idx, 16) ? 1 : 0;
  return from_cuda(launch_plan_dispatch(f, fp8, (cudaStream_t)stream));
}

static moe_status combine_common(const moe_shape *shape, const void *expert_y,
                                 const int32_t *topk_idx, const int32_t *slot_of,
                                 const float *topk_weights, const void *shared, void *y,
                                 void *workspace, void *stream);

moe_status moe_combine(const moe_shape *shape, const void *expert_y, const int32_t *topk_idx,
                       const int32_t *slot_of, const float *topk_weights, void *y,
                       void *workspace, void *stream) {
  return combine_common(shape, expert_y, topk_idx, slot_of, topk_weights, nullptr, y, workspace,
                        stream);
}

moe_status moe_combine_shared(const moe_shape *shape, const void *expert_y,
                              const int32_t *topk_idx, const int32_t *slot_of,
                              const float *topk_weights, const void *shared_y, void *y,
                              void *workspace, void *stream) {
  if (shape && shape->tokens_per_rank > 0) {
    if (!shared_y) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)shared_y % 16 != 0) return MOE_ERR_ALIGNMENT;
  }
  return combine_common(shape, expert_y, topk_idx, slot_of, topk_weights, shared_y, y, workspace,
                        stream);
}

static moe_status combine_common(const moe_shape *shape, const void *expert_y,
                                 const int32_t *topk_idx, const int32_t *slot_of,
                                 const float *topk_weights, const void *shared, void *y,
                                 void *workspace, void *stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->tokens_per_rank == 0) return MOE_OK;   // empty batch: nothing to read or write
  if (!expert_y || !topk_idx || !slot_of || !topk_weights || !y) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!aligned(expert_y, 16) || !aligned(y, 16) || !aligned(topk_idx, 4) || !aligned(slot_of, 4) ||
      !aligned(topk_weights, 4) || !aligned(workspace, 16))
    return MOE_ERR_ALIGNMENT;
  CombineParams p;
  p.expert_y = static_cast<const uint16_t *>(expert_y);
  p.shared = static_cast<const uint16_t *>(shared);
  p.topk_idx = topk_idx;
  p.slot_of = slot_of;
  p.topk_weights = topk_weights;
  p.y = static_cast<uint16_t *>(y);
  p.hdr = header(workspace);
  p.N = shape->num_ranks * shape->tokens_per_rank;
  p.H = shape->hidden;
  p.E = shape->num_experts;
  p.K = shape->top_k;
  p.cap = shape->capacity;
  return from_cuda(launch_combine(p, (cudaStream_t)stream));
}

moe_status moe_router_topk(const moe_shape *shape, const float *logits, int32_t *topk_idx,
                           float *topk_weights, void *stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->top_k > shape->num_experts || shape->num_experts > kRouterMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (shape->tokens_per_rank == 0) return MOE_OK;   // empty batch
  if (!logits || !topk_idx || !topk_weights) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_weights, 4))
    return MOE_ERR_ALIGNMENT;
  RouterParams p;
  p.logits = logits;
  p.topk_idx = topk_idx;
  p.topk_weights = topk_weights;
  p.N = (int64_t)shape->num_ranks * shape->tokens_per_rank;
  p.E = shape->num_experts;
  p.K = shape->top_k;
  return from_cuda(launch_router(p, (cudaStream_t)stream));
}

moe_status moe_silu_mul_quant(const moe_shape *shape, int32_t intermediate, const void *expert_h,
                              const int32_t *expert_num_tokens, void *act_q, float *act_scale,
                              void *workspace, void *stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (intermediate <= 0) return MOE_ERR_INVALID_ARG;
  // rows of any multiple of 16 elements: the last 128-element scale block may
  // be short, and every 8-byte store of a row is then wholly inside it
  if (intermediate % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)shape->num_experts * shape->capacity * 2 * intermediate >= ((int64_t)1 << 46))
    return MOE_ERR_UNSUPPORTED;
  if (!expert_h || !expert_num_tokens || !act_q || !act_scale) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!aligned(expert_h, 16) || !aligned(act_q, 16) || !aligned(expert_num_tokens, 4) ||
      !aligned(act_scale, 4) || !aligned(workspace, 16))
    return MOE_ERR_ALIGNMENT;
  ActParams p;
  p.expert_h = static_cast<const uint16_t *>(expert_h);
  p.expert_num_tokens = expert_num_tokens;
  p.act_q = act_q;
  p.act_scale = act_scale;
  p.hdr = header(workspace);
  p.E = shape->num_experts;
  p.cap = shape->capacity;
  p.I = intermediate;
  p.scale_t = shape->payload == MOE_PAYLOAD_FP8_E4M3_TSCALE;
  return from_cuda(launch_silu_quant(p, (cudaStream_t)stream));
}

moe_status moe_read_status(const void *workspace, void *stream, moe_status *out) {
  if (!workspace || !out) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&v, &static_cast<const WsHeader *>(workspace)->status, sizeof v,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *out = (moe_status)v;
  return MOE_OK;
}

const char *moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_BAD_EXPERT: return "expert id out of range";
    case MOE_ERR_CAPACITY: return "expert capacity exceeded";
    case MOE_ERR_TIMEOUT: return "wait between thread blocks timed out";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

moe_status moe_workspace_set_debug(void *workspace, uint32_t flags, uint64_t timeout_ns,
                                   void *stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_set_debug(header(workspace), flags, timeout_ns, (cudaStream_t)stream));
}

}  // extern "C"
