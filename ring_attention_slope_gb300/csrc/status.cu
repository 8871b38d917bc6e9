// Device status word and the bounded-wait self-test.
//
// Kernels never spin without a limit: a barrier wait that runs out records
// {kStatusTimeout, site} here and the kernel returns.  The host reads and
// clears the word through slope_device_status().
#include <atomic>

#include "kernels.cuh"
#include "sm103_ptx.cuh"
#include "waits.cuh"

namespace slope {

// {code, site}; one copy per device that loads the library.
__device__ int g_slope_status[2];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int*> g_status_ptr[kMaxDevices];

// One block waits on a barrier that nothing ever arrives on; the bounded wait
// must run out, record the timeout and let the kernel return normally.
__global__ void timeout_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(&bar, 0, &abort_flag, status, limit_ns, 99);
  __syncthreads();
}

}  // namespace

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* ptr = g_status_ptr[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_slope_status) != cudaSuccess) return nullptr;
    ptr = static_cast<int*>(addr);
    g_status_ptr[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

cudaError_t launch_timeout_selftest(uint64_t limit_ns, int* status, cudaStream_t stream) {
  timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace slope
