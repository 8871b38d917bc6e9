// Exact log-sum-exp merge of attention partials computed over disjoint key
// sets: the combination step that turns the per-device partials of Ring
// Attention (Moreh, "Optimizing long-context prefill on multiple
// older-generation GPU nodes", section "Introduction to Context Parallelism",
// Ring Attention item) into the attention over all keys.
//
//   L   = m + log sum_k exp(lse_k - m),  m = max_k lse_k   (all -inf -> -inf)
//   out = sum_k exp(lse_k - L) * out_k   (partials with lse_k = -inf are not read)
//
// Bandwidth-bound: dv/16 threads share one (row, head); each reads the n
// log-sum-exp values of the row, then issues predicated 16-byte streaming
// loads of its 64 bytes of every live partial, two partials at a time, and
// writes bf16 or fp32.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.cuh"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

// NMAX: compile-time bound on the number of partials (2, 4, 8, 16 or 32), so that the
// per-thread log-sum-exp array fits in few registers when n is small and more warps stay
// resident to hide the two dependent loads (lse, then partials): five blocks of 256 threads
// per SM at 3 or 4 partials, four at n <= 8 otherwise.  Measured on one GB300 against the old
// fixed bound of 32: 2 partials 2.6 -> 6.8 TB/s, 8 partials 5.3 -> 6.7 TB/s, 16 partials
// 6.4 -> 7.0 TB/s.  Five blocks instead of four (no spills) took the merge of the
// 128-token-window ring (three planes, most rows -inf in two of them) from 0.80 to 0.88 of
// the copy rate, but the two-plane merge of the chunked layout from 1.01 to 0.96.
// IN_BF16: the partials are bf16 (each thread then reads 4 columns = 8 bytes per float4
// position), halving the bytes read; accumulation stays fp32.
template <int DV, bool OUT_BF16, int NMAX, bool IN_BF16>
__global__ void __launch_bounds__(kMergeThreads, NMAX == 4 ? 5 : NMAX <= 8 ? 4 : 2)
    lse_merge_kernel(const __grid_constant__ MergeParams p) {
  // DV/16 threads per (row, head), four float4 columns each: thread q owns float4
  // columns q, q+kTpp, q+2 kTpp, q+3 kTpp, so that each load instruction of a warp reads
  // contiguous runs of kTpp * 16 bytes.
  constexpr int kTpp = DV / 16;
  constexpr int kVec = 4;  // float4s per thread per partial
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const int64_t pair = gtid / kTpp;
  const int q = static_cast<int>(gtid % kTpp);
  if (pair >= p.S * p.H) return;
  const int64_t row = pair / p.H;
  const int h = static_cast<int>(pair - row * p.H);

  constexpr int kBatch = 2;  // partials loaded together (more resident warps beat bigger batches)
  float lk[NMAX];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < NMAX; ++k) {
    lk[k] = -INFINITY;
    if (k < p.n) {
      lk[k] = __ldg(p.lses[k] + row * p.l_srow[k] + h * p.l_shead[k]);
      mx = fmaxf(mx, lk[k]);
    }
  }

  float4 acc[kVec];
#pragma unroll
  for (int j = 0; j < kVec; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < NMAX; ++k)
      if (k < p.n) sum += ex2_approx((lk[k] - mx) * kLog2e);
    L = mx + lg2_approx(sum) * kLn2;
#pragma unroll
    for (int b = 0; b < NMAX; b += kBatch) {
      if (b >= p.n) break;
      float4 v[kBatch][kVec];
      float w[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int k = b + i;
        const bool live = k < p.n && lk[k] != -INFINITY;
        w[i] = live ? ex2_approx((lk[k] - L) * kLog2e) : 0.f;
        const int64_t eoff = row * p.o_srow[k] + h * p.o_shead[k];
        if constexpr (IN_BF16) {
          const uint2* src = live ? reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.outs[k]) + eoff)
                                  : nullptr;
#pragma unroll
          for (int j = 0; j < kVec; ++j) {
            const uint2 r = live ? __ldcs(src + q + kTpp * j) : make_uint2(0u, 0u);
            v[i][j] = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                                  __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
          }
        } else {
          const float4* src = live ? reinterpret_cast<const float4*>(static_cast<const float*>(p.outs[k]) + eoff)
                                   : nullptr;
#pragma unroll
          for (int j = 0; j < kVec; ++j)
            v[i][j] = live ? __ldcs(src + q + kTpp * j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          acc[j].x = fmaf(w[i], v[i][j].x, acc[j].x);
          acc[j].y = fmaf(w[i], v[i][j].y, acc[j].y);
          acc[j].z = fmaf(w[i], v[i][j].z, acc[j].z);
          acc[j].w = fmaf(w[i], v[i][j].w, acc[j].w);
        }
    }
  }

#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const int64_t col = 4 * (q + kTpp * j);
    if (OUT_BF16) {
      __nv_bfloat16* base = static_cast<__nv_bfloat16*>(p.out);
      const uint2 packed = make_uint2(pack_bf16x2(acc[j].x, acc[j].y), pack_bf16x2(acc[j].z, acc[j].w));
      *reinterpret_cast<uint2*>(base + row * p.out_srow + h * p.out_shead + col) = packed;
    } else {
      float* base = static_cast<float*>(p.out);
      *reinterpret_cast<float4*>(base + row * p.out_srow + h * p.out_shead + col) = acc[j];
    }
  }
  if (q == 0 && p.lse != nullptr) p.lse[row * p.lse_srow + h * p.lse_shead] = L;
}

template <int DV, bool BF16, int NMAX, bool IN_BF16>
cudaError_t launch_n(const MergeParams& p, cudaStream_t stream) {
  const int64_t threads = p.S * p.H * (DV / 16);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + kMergeThreads - 1) / kMergeThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  lse_merge_kernel<DV, BF16, NMAX, IN_BF16><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int DV, bool BF16, bool IN_BF16>
cudaError_t launch_in(const MergeParams& p, cudaStream_t stream) {
  static_assert(kMaxMerge == 32, "plane-count bounds below");
  if (p.n <= 2) return launch_n<DV, BF16, 2, IN_BF16>(p, stream);
  if (p.n <= 4) return launch_n<DV, BF16, 4, IN_BF16>(p, stream);
  if (p.n <= 8) return launch_n<DV, BF16, 8, IN_BF16>(p, stream);
  if (p.n <= 16) return launch_n<DV, BF16, 16, IN_BF16>(p, stream);
  return launch_n<DV, BF16, 32, IN_BF16>(p, stream);
}

template <int DV, bool BF16>
cudaError_t launch_impl(const MergeParams& p, cudaStream_t stream) {
  return p.in_bf16 ? launch_in<DV, BF16, true>(p, stream) : launch_in<DV, BF16, false>(p, stream);
}

// Writes -inf into every element of the listed planes (coalesced 4-byte stores; each plane
// is split over gridDim.x blocks, blockIdx.y picks the plane).
__global__ void __launch_bounds__(256) lse_fill_kernel(const __grid_constant__ FillParams p) {
  float* const plane = p.base + static_cast<int64_t>(p.planes[blockIdx.y]) * p.plane_elems;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.plane_elems; i += stride)
    plane[i] = -INFINITY;
}

}  // namespace

cudaError_t launch_lse_fill(const FillParams& p, cudaStream_t stream) {
  if (p.n <= 0 || p.plane_elems <= 0) return cudaSuccess;
  if (p.n > kMaxMerge) return cudaErrorInvalidValue;
  // about 4 resident blocks per SM in total, split over the planes
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t per_plane = std::max<int64_t>(1, std::min<int64_t>((p.plane_elems + 255) / 256, (4LL * sms + p.n - 1) / p.n));
  lse_fill_kernel<<<dim3(static_cast<unsigned>(per_plane), static_cast<unsigned>(p.n)), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.dv == 64) return p.out_bf16 ? launch_impl<64, true>(p, stream) : launch_impl<64, false>(p, stream);
  if (p.dv == 128) return p.out_bf16 ? launch_impl<128, true>(p, stream) : launch_impl<128, false>(p, stream);
  if (p.dv == 192) return p.out_bf16 ? launch_impl<192, true>(p, stream) : launch_impl<192, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace slope
