// Device status word, the attention kernel's work-tile counters and the
// bounded-wait self-test.
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

// Work-tile counters of the attention launches that claim their tiles at run time, handed
// out round robin, one per launch.  Each is 0 between launches: the launch's last CTA to
// claim past the end puts it back (see the attention kernel's scheduler warp).  A counter
// is shared only by launches kTileCounterSlots apart.  On one stream those never run at
// once: a launch's CTAs start only after the previous grid's have all started, each holds
// an SM until that previous grid is done, and the device has far fewer SMs than slots.
// Across streams two such launches would have to be queued or running at the same time.
__device__ uint32_t g_slope_tile_counters[kTileCounterSlots];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int*> g_status_ptr[kMaxDevices];
std::atomic<uint32_t*> g_counters_ptr[kMaxDevices];
std::atomic<uint32_t> g_counter_next[kMaxDevices];

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

uint32_t* claim_tile_counter() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint32_t* base = g_counters_ptr[dev].load(std::memory_order_acquire);
  if (base == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_slope_tile_counters) != cudaSuccess) return nullptr;
    base = static_cast<uint32_t*>(addr);
    g_counters_ptr[dev].store(base, std::memory_order_release);
  }
  return base + g_counter_next[dev].fetch_add(1, std::memory_order_relaxed) % kTileCounterSlots;
}

cudaError_t launch_timeout_selftest(uint64_t limit_ns, int* status, cudaStream_t stream) {
  timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace slope
