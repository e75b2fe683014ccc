// Test kernels for the library's bounded mbarrier waits (mla_device.cuh):
// every wait in the decode and indexer kernels gives up after a bounded
// number of polls, sets a bit in a fault word the host can read, and
// returns, so that a phase that never completes costs an error status, not
// a hung GPU.  Built and run only by tests/test_gpu_bounded_wait.py.
//
//   mode 0: nothing ever arrives on the barrier        -> wait returns false, fault bit set
//   mode 1: another warp sets the CTA's abort flag     -> wait returns false, no fault bit
//   mode 2: another warp arrives after a short delay   -> wait returns true, no fault bit
#include <cstdint>

#include "mla_device.cuh"

namespace {

constexpr unsigned int kTestFault = 0x40u;

__device__ __forceinline__ void spin_cycles(long long n) {
  const long long t0 = clock64();
  while (clock64() - t0 < n) {
  }
}

__global__ void wait_probe_kernel(int mode, unsigned int* fault_word, int* ok_out, long long* cycles_out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mla::mbar_init(&bar, 1);
    abort_flag = 0;
    mla::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const long long t0 = clock64();
    const bool ok = mode == 0 ? mla::mbar_wait_bounded(&bar, 0u, fault_word, kTestFault)
                              : mla::mbar_wait_or_abort(&bar, 0u, &abort_flag, fault_word, kTestFault);
    if (lane == 0) {
      ok_out[0] = ok ? 1 : 0;
      cycles_out[0] = clock64() - t0;
    }
  } else if (lane == 0) {
    spin_cycles(200000);  // ~0.1 ms: the waiter is polling by then
    if (mode == 1) *reinterpret_cast<volatile int*>(&abort_flag) = 1;
    if (mode == 2) mla::mbar_arrive(&bar);
  }
}

}  // namespace

// Runs one probe launch (one CTA of two warps) and copies its results back.
// Returns the CUDA error of the launch and synchronisation (0 = success).
extern "C" int wait_probe(int mode, unsigned int* fault_host, int* ok_host, long long* cycles_host) {
  unsigned int* fault = nullptr;
  int* ok = nullptr;
  long long* cycles = nullptr;
  cudaError_t e = cudaMalloc(&fault, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMalloc(&ok, sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&cycles, sizeof(long long));
  if (e == cudaSuccess) e = cudaMemset(fault, 0, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemset(ok, 0xFF, sizeof(int));
  if (e == cudaSuccess) {
    wait_probe_kernel<<<1, 64>>>(mode, fault, ok, cycles);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(fault_host, fault, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(ok_host, ok, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(cycles_host, cycles, sizeof(long long), cudaMemcpyDeviceToHost);
  cudaFree(fault);
  cudaFree(ok);
  cudaFree(cycles);
  return static_cast<int>(e);
}
