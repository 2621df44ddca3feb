// pdl_producer.cu -- test support for the dispatch ordering test (built by
// tests/test_gpu_ordering.py with nvcc, never part of the library).
//
// produce_x stands for a kernel that computes the dispatch's input x and,
// like many GEMM kernels in serving stacks, lets the next kernel in the
// stream start at once (griddepcontrol.launch_dependents at entry).  It then
// sleeps for a bounded time and only afterwards copies the new x into place,
// so a dependent that read x without waiting for it would see the old rows.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void produce_x(uint4 *x, const uint4 *src, long long n16, unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  // bounded both by the global timer and by the number of polls
  for (int i = 0; i < 200000; ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= delay_ns) break;
    __nanosleep(500);
  }
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    x[i] = src[i];
}

// Copy n16 16-byte words from src to x on `stream` after delay_ns; 64 blocks
// of 256 threads, all resident at once, so every block reaches the trigger.
extern "C" int launch_produce_x(void *x, const void *src, long long n16, unsigned long long delay_ns,
                                void *stream) {
  produce_x<<<64, 256, 0, (cudaStream_t)stream>>>(static_cast<uint4 *>(x),
                                                  static_cast<const uint4 *>(src), n16, delay_ns);
  return (int)cudaGetLastError();
}
