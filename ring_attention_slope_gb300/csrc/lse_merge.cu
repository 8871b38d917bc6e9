// Exact log-sum-exp merge of attention partials computed over disjoint key
// sets: the combination step that turns the per-device partials of Ring
// Attention (Moreh, "Optimizing long-context prefill on multiple
// older-generation GPU nodes", section "Introduction to Context Parallelism",
// Ring Attention item) into the attention over all keys.
//
//   L   = m + log sum_k exp(lse_k - m),  m = max_k lse_k   (all -inf -> -inf)
//   out = sum_k exp(lse_k - L) * out_k   (partials with lse_k = -inf are not read)
//
// Bandwidth-bound: each thread owns 4 consecutive output elements of one
// (row, head); it reads the n log-sum-exp values of its row first, then issues
// the (predicated) 16-byte streaming loads of all live partials in batches of
// 8 so that many loads are in flight, and writes bf16 or fp32.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int DV, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int kTpr = DV / 4;  // threads per (row, head)
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const int64_t pair = gtid / kTpr;
  const int c4 = static_cast<int>(gtid % kTpr);
  if (pair >= p.S * p.H) return;
  const int64_t row = pair / p.H;
  const int h = static_cast<int>(pair % p.H);

  float lk[kMaxMerge];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMaxMerge; ++k) {
    lk[k] = -INFINITY;
    if (k < p.n) {
      lk[k] = __ldg(p.lses[k] + row * p.l_srow[k] + h * p.l_shead[k]);
      mx = fmaxf(mx, lk[k]);
    }
  }

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxMerge; ++k)
      if (k < p.n) sum += ex2_approx((lk[k] - mx) * kLog2e);
    L = mx + lg2_approx(sum) * kLn2;
#pragma unroll
    for (int b = 0; b < kMaxMerge; b += 8) {
      if (b >= p.n) break;
      float4 v[8];
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = b + i;
        const bool live = k < p.n && lk[k] != -INFINITY;
        w[i] = live ? ex2_approx((lk[k] - L) * kLog2e) : 0.f;
        v[i] = live ? __ldcs(reinterpret_cast<const float4*>(p.outs[k] + row * p.o_srow[k] + h * p.o_shead[k]) + c4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc.x = fmaf(w[i], v[i].x, acc.x);
        acc.y = fmaf(w[i], v[i].y, acc.y);
        acc.z = fmaf(w[i], v[i].z, acc.z);
        acc.w = fmaf(w[i], v[i].w, acc.w);
      }
    }
  }

  if (OUT_BF16) {
    __nv_bfloat16* base = static_cast<__nv_bfloat16*>(p.out);
    uint2 packed = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    *reinterpret_cast<uint2*>(base + row * p.out_srow + h * p.out_shead + 4 * c4) = packed;
  } else {
    float* base = static_cast<float*>(p.out);
    *reinterpret_cast<float4*>(base + row * p.out_srow + h * p.out_shead + 4 * c4) = acc;
  }
  if (c4 == 0 && p.lse != nullptr) p.lse[row * p.lse_srow + h * p.lse_shead] = L;
}

template <int DV, bool BF16>
cudaError_t launch_impl(const MergeParams& p, cudaStream_t stream) {
  const int64_t threads = p.S * p.H * (DV / 4);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + kMergeThreads - 1) / kMergeThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  lse_merge_kernel<DV, BF16><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.dv == 64) return p.out_bf16 ? launch_impl<64, true>(p, stream) : launch_impl<64, false>(p, stream);
  if (p.dv == 128) return p.out_bf16 ? launch_impl<128, true>(p, stream) : launch_impl<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace slope
