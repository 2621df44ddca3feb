// moe_plan_noalloc.cu -- moe_plan for callers that cannot allocate device
// memory.  The plan kernel's scratch (the workspace header, per-tile flags
// and per-tile count rows) lives in a file-scope static device array instead
// of a caller-provided workspace.
//
// Who needs it: code that is handed only its inputs and outputs and has no
// way to obtain scratch memory -- for example a plugin whose host framework
// owns every device allocation, or a latency-critical caller that must not
// call cudaMalloc because it can synchronise the device.
//
// Costs and limits: every GPU that loads this library holds the array
// (kNoAllocScratchBytes) until the process exits; shapes whose workspace
// would exceed it are rejected.  All calls on a device share the array, so
// two calls that may run at the same time on the GPU (different streams
// without ordering between them) race and must not be issued.
#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;   // 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_plan_scratch[kNoAllocScratchBytes];

// Device address of g_plan_scratch, looked up with that device current.  In
// host code the symbol itself is only a host-side stand-in, so kernels must
// be given this address, never the symbol.  Only a successful lookup is
// kept: a lookup that failed (for example one made while the stream was
// being captured) is tried again by the next call.
std::mutex g_mutex;
void *g_addr[kMaxDevices];

cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_plan_scratch);
    if (e != cudaSuccess) {
      // clear the error the failed lookup recorded, so that the next
      // launch check of this thread does not mistake it for its own
      (void)cudaGetLastError();
      return e;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_plan_noalloc(const moe_shape *shape, const int32_t *topk_idx,
                                       int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                                       int32_t *slot_of, int32_t *src_of, int32_t *status_out,
                                       void *stream) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  // Shape checks and the size of the scratch this shape needs.
  const size_t need = moe_workspace_size(shape);
  if (need == 0)
    return (shape->num_ranks <= 0 || shape->tokens_per_rank < 0 || shape->hidden <= 0 ||
            shape->num_experts <= 0 || shape->top_k <= 0 || shape->capacity <= 0 ||
            (shape->payload != MOE_PAYLOAD_BF16 && shape->payload != MOE_PAYLOAD_FP8_E4M3 &&
             shape->payload != MOE_PAYLOAD_FP8_E4M3_TSCALE))
               ? MOE_ERR_INVALID_ARG
               : MOE_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  // An empty batch (T = 0) reads no routes and writes no slots: topk_idx and
  // slot_of may then be NULL, as for moe_plan.
  const bool empty = shape->tokens_per_rank == 0;
  if ((!empty && (!topk_idx || !slot_of)) || !expert_num_tokens || !expert_rank_offsets ||
      !src_of || !status_out)
    return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)status_out & 3u) != 0) return MOE_ERR_ALIGNMENT;

  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;

  // The array keeps the previous call's contents.  The counters in the
  // header and the per-tile flags must start at zero: clear them (the count
  // rows are always written before they are read).
  const WsLayout L = ws_layout(*shape);
  if (cudaMemsetAsync(scratch, 0, L.rows_off, s) != cudaSuccess) return MOE_ERR_CUDA;

  moe_status st = moe_plan(shape, topk_idx, expert_num_tokens, expert_rank_offsets, slot_of,
                           src_of, scratch, kNoAllocScratchBytes, stream);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(status_out, &static_cast<WsHeader *>(scratch)->status, sizeof(int32_t),
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
