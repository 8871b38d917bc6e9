// C ABI of libslope (declared in include/slope.h): argument validation, the
// work decomposition of context-parallel prefill, TMA tensor maps and the
// kernel launches.  The library allocates no device memory.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "slope.h"

using namespace slope;

namespace {

constexpr int kMaxRanks = 32;
constexpr int64_t kMaxSeq = int64_t(1) << 30;
// Bound on the global positions slope_attn_partial accepts: the kernel forms differences of a query
// and a key position, less the window, in 32-bit integers, which then stay within +-1.5 * 2^30.
constexpr int64_t kMaxPos = int64_t(1) << 28;
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// ---------------------------------------------------------------- argument checks

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local char g_last_error[256] = "";

// Records the text of a failing CUDA call and returns SLOPE_ERR_CUDA.
slope_status cuda_fail(const char* where, cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return SLOPE_ERR_CUDA;
}
slope_status cuda_fail(const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", where);
  return SLOPE_ERR_CUDA;
}

// bf16 [S, H, d] readable by TMA: innermost stride 1, other strides multiples of 8 elements.
slope_status check_qkv(const slope_tensor* t) {
  if (t == nullptr) return SLOPE_ERR_NULL;
  if (t->dtype != SLOPE_BF16) return SLOPE_ERR_DTYPE;
  if (t->ndim != 3) return SLOPE_ERR_SHAPE;
  if (t->shape[0] < 0 || t->shape[1] <= 0 || t->shape[2] <= 0 || t->shape[0] > kMaxSeq || t->shape[1] > 65535)
    return SLOPE_ERR_SHAPE;
  if (t->shape[0] > 0 && t->data == nullptr) return SLOPE_ERR_NULL;
  if (t->stride[2] != 1) return SLOPE_ERR_STRIDE;
  if (t->stride[0] <= 0 || t->stride[1] <= 0 || t->stride[0] % 8 || t->stride[1] % 8) return SLOPE_ERR_STRIDE;
  if (!aligned(t->data, 16)) return SLOPE_ERR_STRIDE;
  return SLOPE_OK;
}

// [S, H, dv] output, fp32 (or bf16 when allowed); 16-byte vector stores.
slope_status check_out(const slope_tensor* t, int64_t S, int64_t H, int64_t dv, bool allow_bf16) {
  if (t == nullptr) return SLOPE_ERR_NULL;
  if (t->dtype != SLOPE_F32 && !(allow_bf16 && t->dtype == SLOPE_BF16)) return SLOPE_ERR_DTYPE;
  if (t->ndim != 3 || t->shape[0] != S || t->shape[1] != H || t->shape[2] != dv) return SLOPE_ERR_SHAPE;
  if (S > 0 && t->data == nullptr) return SLOPE_ERR_NULL;
  if (t->stride[2] != 1 || t->stride[0] <= 0 || t->stride[1] <= 0) return SLOPE_ERR_STRIDE;
  if (t->stride[0] % 4 || t->stride[1] % 4) return SLOPE_ERR_STRIDE;
  if (!aligned(t->data, t->dtype == SLOPE_F32 ? 16 : 8)) return SLOPE_ERR_STRIDE;
  return SLOPE_OK;
}

// fp32 [H, S], any positive strides.
slope_status check_lse(const slope_tensor* t, int64_t H, int64_t S) {
  if (t == nullptr) return SLOPE_ERR_NULL;
  if (t->dtype != SLOPE_F32) return SLOPE_ERR_DTYPE;
  if (t->ndim != 2 || t->shape[0] != H || t->shape[1] != S) return SLOPE_ERR_SHAPE;
  if (S > 0 && t->data == nullptr) return SLOPE_ERR_NULL;
  if (t->stride[0] <= 0 || t->stride[1] <= 0) return SLOPE_ERR_STRIDE;
  if (!aligned(t->data, 4)) return SLOPE_ERR_STRIDE;
  return SLOPE_OK;
}

uint64_t wait_limit_ns() {
  static const uint64_t limit = [] {
    const char* e = std::getenv("SLOPE_WAIT_LIMIT_NS");
    if (e != nullptr) {
      const unsigned long long v = std::strtoull(e, nullptr, 10);
      if (v >= 1000ull && v <= 60000000000ull) return static_cast<uint64_t>(v);
    }
    return kDefaultWaitLimitNs;
  }();
  return limit;
}

float resolve_scale(float scale, int64_t dqk) {
  return scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(dqk)));
}

// ---------------------------------------------------------------- TMA tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 3-D view {d, H, S} of a bf16 [S, H, d] tensor; box = 64 columns x 1 head x 128 rows,
// 128-byte swizzle (the layout the tcgen05 descriptors expect); out-of-range rows read 0.
bool make_map(CUtensorMap* m, const slope_tensor* t) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  std::memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(t->shape[2]), static_cast<cuuint64_t>(t->shape[1]),
                        static_cast<cuuint64_t>(t->shape[0])};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(t->stride[1]) * 2, static_cast<cuuint64_t>(t->stride[0]) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockN)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {dv, H, rows} of an fp32 or bf16 output with row/head strides in elements;
// box = 128 bytes of columns (32 fp32 or 64 bf16) x 1 head x 32 rows (one softmax warp's
// rows), 128-byte swizzle, written by TMA stores from the attention kernel's epilogue.
// Returns false if the map cannot be built (the kernel then stores directly).
bool make_out_map(CUtensorMap* m, void* base, bool bf16, int64_t rows, int64_t H, int64_t dv, int64_t srow,
                  int64_t shead) {
  auto enc = encode_fn();
  if (enc == nullptr || rows <= 0 || rows > 0x7fffffffLL) return false;
  const cuuint64_t esize = bf16 ? 2 : 4;
  if ((srow * esize) % 16 != 0 || (shead * esize) % 16 != 0 || !aligned(base, 16)) return false;
  std::memset(m, 0, sizeof(*m));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dv), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(shead) * esize, static_cast<cuuint64_t>(srow) * esize};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- work decomposition

struct Range {
  int64_t row0, len;
};
struct PItem {
  int launch, plane;
  int64_t q_row0, q_len;
  int n_kv;
  Range kv[kMaxKvRanges];
  int hg = 0, n_hg = 1;  // query heads [hg*Hq/n_hg, (hg+1)*Hq/n_hg)
};
struct Plan {
  std::vector<PItem> items;  // grouped by launch, in launch order
  int n_launches = 0;
  int n_planes = 0;
  bool direct = false;     // the items write the final output (no partials, no merge)
  int n_head_groups = 1;   // Ulysses degree (query-head groups); must divide Hkv
};

// Restricts keys [k0, k1) to those some query in [q0, q1) can see (positions = rows).
bool trim(int64_t q0, int64_t q1, int64_t& k0, int64_t& k1, int causal, int64_t window) {
  if (causal) k1 = std::min(k1, q1);
  if (window > 0) k0 = std::max(k0, q0 - window + 1);
  return k1 > k0;
}

slope_status chunk_list(int64_t S, int n_chunks, const int64_t* chunk_sizes, std::vector<int64_t>& sizes) {
  sizes.clear();
  if (n_chunks < 1 || n_chunks > 4096) return SLOPE_ERR_LAYOUT;
  if (chunk_sizes != nullptr) {
    int64_t sum = 0;
    for (int c = 0; c < n_chunks; ++c) {
      if (chunk_sizes[c] <= 0) return SLOPE_ERR_LAYOUT;
      sum += chunk_sizes[c];
      sizes.push_back(chunk_sizes[c]);
    }
    if (sum != S) return SLOPE_ERR_LAYOUT;
  } else {
    const int64_t c = (S + n_chunks - 1) / n_chunks;
    int64_t left = S;
    for (int i = 0; i < n_chunks; ++i) {
      const int64_t sz = std::min(c, left);
      if (sz <= 0) return SLOPE_ERR_LAYOUT;
      sizes.push_back(sz);
      left -= sz;
    }
  }
  return SLOPE_OK;
}

// Ring layouts: at step t rank r holds the keys/values of rank (r - t) mod N; each
// of r's query sub-chunks attends to the visible parts of those sub-chunks and
// writes partial plane t.  Chunked: chunk [s, e) gives (Q_c, KV[0, s)) -> plane 0
// and (Q_c, KV[s, e)) -> plane 1, one launch per chunk.  Ulysses: after the
// all-to-all, rank u holds every token of head group u of N and computes the whole
// attention of those heads: one item per rank, written as the final output.
slope_status build_base_plan(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                             int64_t window, bool fused, Plan& plan) {
  plan = Plan();
  if (S <= 0 || S > kMaxSeq) return SLOPE_ERR_SHAPE;
  if (window < 0) return SLOPE_ERR_SHAPE;
  if (layout == SLOPE_LAYOUT_CONTIGUOUS || layout == SLOPE_LAYOUT_ZIGZAG) {
    const int N = n_chunks;
    if (N < 1 || N > kMaxRanks) return SLOPE_ERR_LAYOUT;
    const bool zz = layout == SLOPE_LAYOUT_ZIGZAG;
    const int64_t parts = zz ? 2 * N : N;
    if (S % parts != 0) return SLOPE_ERR_LAYOUT;
    const int64_t sub = S / parts;
    auto owned = [&](int r, int64_t* out) -> int {
      out[0] = r;
      if (!zz) return 1;
      out[1] = 2 * N - 1 - r;
      return 2;
    };
    if (fused) {
      // Every ring step of rank r visits one of the ranks' blocks, so over the whole ring each of
      // r's query sub-chunks meets every key block once: their union is all S keys, of which the
      // masks leave one range.  One item per sub-chunk runs its online softmax over that range and
      // writes the final output.
      for (int r = 0; r < N; ++r) {
        int64_t qa[2];
        const int nq = owned(r, qa);
        for (int i = 0; i < nq; ++i) {
          PItem it{};
          it.launch = r;
          it.plane = 0;
          it.q_row0 = qa[i] * sub;
          it.q_len = sub;
          int64_t k0 = 0, k1 = S;
          if (trim(it.q_row0, it.q_row0 + sub, k0, k1, causal, window)) it.kv[it.n_kv++] = Range{k0, k1 - k0};
          plan.items.push_back(it);
        }
      }
      plan.n_launches = N;
      plan.n_planes = 1;
      plan.direct = true;
      return SLOPE_OK;
    }
    for (int t = 0; t < N; ++t) {
      for (int r = 0; r < N; ++r) {
        const int src = ((r - t) % N + N) % N;
        int64_t qa[2], kb[2];
        const int nq = owned(r, qa), nk = owned(src, kb);
        for (int i = 0; i < nq; ++i) {
          PItem it{};
          it.launch = t;
          it.plane = t;
          it.q_row0 = qa[i] * sub;
          it.q_len = sub;
          it.n_kv = 0;
          for (int j = 0; j < nk; ++j) {
            int64_t k0 = kb[j] * sub, k1 = k0 + sub;
            if (trim(it.q_row0, it.q_row0 + sub, k0, k1, causal, window)) it.kv[it.n_kv++] = Range{k0, k1 - k0};
          }
          plan.items.push_back(it);
        }
      }
    }
    plan.n_launches = N;
    plan.n_planes = N;
    return SLOPE_OK;
  }
  if (layout == SLOPE_LAYOUT_CHUNKED) {
    std::vector<int64_t> sizes;
    slope_status st = chunk_list(S, n_chunks, chunk_sizes, sizes);
    if (st != SLOPE_OK) return st;
    if (fused) {
      // chunk [s, e): its prefix partial and its diagonal partial in one item over keys [0, e)
      int64_t s0 = 0;
      for (size_t c = 0; c < sizes.size(); ++c) {
        const int64_t s1 = s0 + sizes[c];
        PItem it{};
        it.launch = static_cast<int>(c);
        it.plane = 0;
        it.q_row0 = s0;
        it.q_len = s1 - s0;
        int64_t k0 = 0, k1 = S;
        if (trim(s0, s1, k0, k1, causal, window)) it.kv[it.n_kv++] = Range{k0, k1 - k0};
        plan.items.push_back(it);
        s0 = s1;
      }
      plan.n_launches = static_cast<int>(sizes.size());
      plan.n_planes = 1;
      plan.direct = true;
      return SLOPE_OK;
    }
    int64_t s0 = 0;
    for (size_t c = 0; c < sizes.size(); ++c) {
      const int64_t s1 = s0 + sizes[c];
      PItem pre{}, own{};
      pre.launch = own.launch = static_cast<int>(c);
      pre.plane = 0;
      own.plane = 1;
      pre.q_row0 = own.q_row0 = s0;
      pre.q_len = own.q_len = s1 - s0;
      int64_t k0 = 0, k1 = s0;
      if (trim(s0, s1, k0, k1, causal, window)) pre.kv[pre.n_kv++] = Range{k0, k1 - k0};
      k0 = s0;
      k1 = s1;
      if (trim(s0, s1, k0, k1, causal, window)) own.kv[own.n_kv++] = Range{k0, k1 - k0};
      plan.items.push_back(pre);
      plan.items.push_back(own);
      s0 = s1;
    }
    plan.n_launches = static_cast<int>(sizes.size());
    plan.n_planes = 2;
    return SLOPE_OK;
  }
  if (layout == SLOPE_LAYOUT_ULYSSES) {
    const int N = n_chunks;
    if (N < 1 || N > kMaxRanks) return SLOPE_ERR_LAYOUT;
    for (int u = 0; u < N; ++u) {
      PItem it{};
      it.launch = u;
      it.plane = 0;
      it.q_row0 = 0;
      it.q_len = S;
      it.hg = u;
      it.n_hg = N;
      int64_t k0 = 0, k1 = S;
      if (trim(0, S, k0, k1, causal, window)) it.kv[it.n_kv++] = Range{k0, k1 - k0};
      plan.items.push_back(it);
    }
    plan.n_launches = N;
    plan.n_planes = 1;
    plan.direct = true;
    plan.n_head_groups = N;
    return SLOPE_OK;
  }
  return SLOPE_ERR_LAYOUT;
}

// Partial plans: each item keeps only the query rows that see at least one of its keys (the
// hull of those rows over its key ranges, with the ranges trimmed again to them), and an item
// whose rows see none is dropped.  Rows left out of every item of a plane keep the -inf lse
// that the call writes into the partial planes before the attention launches, so the merge
// skips them without the attention kernel visiting them.  Positions are row indices here.
void keep_rows_that_see_keys(Plan& plan, int causal, int64_t window) {
  std::vector<PItem> kept;
  kept.reserve(plan.items.size());
  for (const PItem& it : plan.items) {
    const int64_t q0 = it.q_row0, q1 = it.q_row0 + it.q_len;
    int64_t lo = q1, hi = q0 - 1;  // hull of the live rows
    for (int r = 0; r < it.n_kv; ++r) {
      const int64_t k0 = it.kv[r].row0, k1 = k0 + it.kv[r].len;
      // row i sees a key of [k0, k1) iff (!causal || i >= k0) && (window == 0 || i - window + 1 <= k1 - 1)
      const int64_t a = causal ? std::max(q0, k0) : q0;
      const int64_t b = window > 0 ? std::min(q1 - 1, k1 + window - 2) : q1 - 1;
      if (a <= b) {
        lo = std::min(lo, a);
        hi = std::max(hi, b);
      }
    }
    if (lo > hi) continue;
    PItem t = it;
    t.q_row0 = lo;
    t.q_len = hi - lo + 1;
    t.n_kv = 0;
    for (int r = 0; r < it.n_kv; ++r) {
      int64_t k0 = it.kv[r].row0, k1 = k0 + it.kv[r].len;
      if (trim(lo, hi + 1, k0, k1, causal, window)) t.kv[t.n_kv++] = Range{k0, k1 - k0};
    }
    kept.push_back(t);
  }
  plan.items = std::move(kept);
}

// The layout word: the base layout in the low 8 bits and, for the ring and chunked layouts, a
// Ulysses degree u in bits 8-15 (0 or 1: none).  Ulysses x Ring: each of the base plan's items
// is split into u items, one per query-head group (the ranks of one Ulysses group after the
// all-to-all), which write the same partial planes.
slope_status build_plan(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                        int64_t window, unsigned flags, Plan& plan) {
  const unsigned word = static_cast<unsigned>(layout);
  if (word >> 16) return SLOPE_ERR_LAYOUT;
  const slope_layout base = static_cast<slope_layout>(word & 0xffu);
  const int u = static_cast<int>((word >> 8) & 0xffu);
  slope_status st =
      build_base_plan(S, n_chunks, base, chunk_sizes, causal, window, (flags & SLOPE_CP_FUSED) != 0, plan);
  if (st == SLOPE_OK && !plan.direct) keep_rows_that_see_keys(plan, causal, window);
  if (st != SLOPE_OK || u <= 1) return st;
  if (base == SLOPE_LAYOUT_ULYSSES || u > kMaxRanks) {
    plan = Plan();
    return SLOPE_ERR_LAYOUT;
  }
  std::vector<PItem> split;
  split.reserve(plan.items.size() * static_cast<size_t>(u));
  for (const PItem& it : plan.items)
    for (int g = 0; g < u; ++g) {
      PItem c = it;
      c.hg = g;
      c.n_hg = u;
      split.push_back(c);
    }
  plan.items = std::move(split);
  plan.n_head_groups = u;
  return SLOPE_OK;
}

// Rough work estimate (visible pairs x share of the heads) used to order items heaviest first.
double item_work(const PItem& it, int causal) {
  double w = 0;
  for (int r = 0; r < it.n_kv; ++r) {
    const bool diag = causal && it.kv[r].row0 + it.kv[r].len > it.q_row0;
    w += static_cast<double>(it.q_len) * static_cast<double>(it.kv[r].len) * (diag ? 0.5 : 1.0);
  }
  return w / it.n_hg;
}

// The attention kernel pairs two query heads of one KV group on the same 128 rows as the two
// Q tiles of a work tile when a KV head serves an even number of query heads (both tiles then
// take the same steps); otherwise its Q tiles are 256 consecutive rows of one head.
bool pair_heads(int64_t Hq, int64_t Hkv) { return (Hq / Hkv) % 2 == 0; }

// Packs items into launch parameter blocks (<= kMaxItems each), heaviest first.  Returns
// false if a block has more work tiles than a launch indexes (2^31 - 1).
bool pack_items(std::vector<PItem> items, int causal, int64_t Hq, bool pair,
                std::vector<std::vector<WorkItem>>& out) {
  const int64_t rows_per_tile = pair ? kBlockM : kRowsPerCta;
  std::stable_sort(items.begin(), items.end(),
                   [&](const PItem& a, const PItem& b) { return item_work(a, causal) > item_work(b, causal); });
  out.clear();
  for (size_t i = 0; i < items.size(); i += kMaxItems) {
    std::vector<WorkItem> group;
    int64_t begin = 0;
    for (size_t j = i; j < std::min(items.size(), i + kMaxItems); ++j) {
      const PItem& s = items[j];
      WorkItem w{};
      w.q_row0 = static_cast<int32_t>(s.q_row0);
      w.q_len = static_cast<int32_t>(s.q_len);
      w.out_row0 = static_cast<int32_t>(s.q_row0);
      w.plane = s.plane;
      w.n_kv = s.n_kv;
      for (int r = 0; r < s.n_kv; ++r) w.kv[r] = KvRange{static_cast<int32_t>(s.kv[r].row0),
                                                        static_cast<int32_t>(s.kv[r].len)};
      w.n_blocks = static_cast<int32_t>((s.q_len + rows_per_tile - 1) / rows_per_tile);
      w.h_begin = static_cast<int32_t>(s.hg * (Hq / s.n_hg));
      w.h_count = static_cast<int32_t>(Hq / s.n_hg);
      w.tile_begin = static_cast<int32_t>(begin);
      begin += static_cast<int64_t>(w.n_blocks) * (pair ? w.h_count / 2 : w.h_count);
      if (begin > 0x7fffffffLL) return false;
      group.push_back(w);
    }
    out.push_back(std::move(group));
  }
  return true;
}

// ---------------------------------------------------------------- launches

struct Timing {
  void** events = nullptr;
  int capacity = 0;
  int count = 0;
  int* kinds = nullptr;
};

cudaError_t record(Timing* tm, bool before, int kind, cudaStream_t stream) {
  if (tm == nullptr) return cudaSuccess;
  if (before) {
    if (tm->count >= tm->capacity) return cudaErrorInvalidValue;
    if (tm->kinds != nullptr) tm->kinds[tm->count] = kind;
    return cudaEventRecord(static_cast<cudaEvent_t>(tm->events[2 * tm->count]), stream);
  }
  cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(tm->events[2 * tm->count + 1]), stream);
  ++tm->count;
  return e;
}

// dependent: this launch follows another attention launch of the same call in the stream (see
// launch_attn_partial); never the first launch of a call, which may follow a kernel that reads
// what this one writes.  Launches timed with events run the ordinary way.
slope_status run_attention(const std::vector<WorkItem>& group, int dqk, int dv, const CUtensorMap& tq,
                           const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, AttnParams base,
                           bool dependent, Timing* tm, cudaStream_t stream) {
  base.n_items = static_cast<int32_t>(group.size());
  for (size_t i = 0; i < group.size(); ++i) base.items[i] = group[i];
  cudaError_t e;
  if ((e = record(tm, true, 0, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  if ((e = launch_attn_partial(dqk, dv, tq, tk, tv, to, base, dependent && tm == nullptr, stream)) != cudaSuccess)
    return cuda_fail("attention kernel launch", e);
  if ((e = record(tm, false, 0, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  return SLOPE_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WorkspaceLayout {
  size_t out_bytes, lse_offset, total;
};
// Partial planes (fp32, or bf16 under SLOPE_CP_BF16_PARTIALS), then the fp32 lse planes.
// A direct plan (Ulysses) keeps no partials: the workspace holds only an lse plane,
// written when the caller passes no lse.
WorkspaceLayout workspace_layout(int64_t S, int64_t Hq, int64_t dv, int n_planes, unsigned flags, bool direct) {
  WorkspaceLayout w;
  const size_t elem = (flags & SLOPE_CP_BF16_PARTIALS) ? 2 : sizeof(float);
  w.out_bytes = direct ? 0 : static_cast<size_t>(S) * Hq * dv * elem;
  w.lse_offset = round_up(w.out_bytes * n_planes, 256);
  w.total = w.lse_offset + round_up(static_cast<size_t>(S) * Hq * sizeof(float) * n_planes, 256);
  return w;
}

// Known flags, alone or together where they mean something: bf16 partials exist only without
// SLOPE_CP_FUSED, which keeps no partials.
bool flags_valid(unsigned flags) {
  const unsigned known = SLOPE_CP_BF16_PARTIALS | SLOPE_CP_FUSED;
  if (flags & ~known) return false;
  return (flags & known) != known;
}

// Every argument check of cp_prefill_impl, with no side effect; fills `plan`.
slope_status cp_prefill_check(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int n_chunks,
                              slope_layout layout, const int64_t* chunk_sizes, int causal, int64_t window,
                              unsigned flags, const slope_tensor* out, const slope_tensor* lse,
                              const void* workspace, size_t workspace_bytes, Plan& plan) {
  slope_status st;
  if (!flags_valid(flags)) return SLOPE_ERR_UNSUPPORTED;
  if ((st = check_qkv(q)) != SLOPE_OK || (st = check_qkv(k)) != SLOPE_OK || (st = check_qkv(v)) != SLOPE_OK)
    return st;
  const int64_t S = q->shape[0], Hq = q->shape[1], dqk = q->shape[2];
  const int64_t Hkv = k->shape[1], dv = v->shape[2];
  if (k->shape[0] != S || v->shape[0] != S || v->shape[1] != Hkv || k->shape[2] != dqk) return SLOPE_ERR_SHAPE;
  if (Hq % Hkv != 0) return SLOPE_ERR_SHAPE;
  if (!attn_partial_supported(static_cast<int>(dqk), static_cast<int>(dv))) return SLOPE_ERR_UNSUPPORTED;
  if (window < 0 || window > kMaxSeq) return SLOPE_ERR_SHAPE;
  if ((st = check_out(out, S, Hq, dv, true)) != SLOPE_OK) return st;
  if (lse != nullptr && (st = check_lse(lse, Hq, S)) != SLOPE_OK) return st;
  if (S == 0) return SLOPE_ERR_SHAPE;
  if ((st = build_plan(S, n_chunks, layout, chunk_sizes, causal, window, flags, plan)) != SLOPE_OK) return st;
  if (plan.n_planes > kMaxMerge) return SLOPE_ERR_UNSUPPORTED;
  if (Hkv % plan.n_head_groups != 0) return SLOPE_ERR_LAYOUT;  // whole KV heads per Ulysses rank
  if (plan.direct) {
    // the attention kernel writes out itself (bf16 16 bytes at a time)
    if (out->dtype == SLOPE_BF16 && (out->stride[0] % 8 || out->stride[1] % 8 || !aligned(out->data, 16)))
      return SLOPE_ERR_STRIDE;
  }
  const WorkspaceLayout wl = workspace_layout(S, Hq, dv, plan.n_planes, flags, plan.direct);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < wl.total) return SLOPE_ERR_WORKSPACE;
  return SLOPE_OK;
}

slope_status cp_prefill_impl(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int n_chunks,
                             slope_layout layout, const int64_t* chunk_sizes, int causal, int64_t window,
                             float scale, unsigned flags, slope_tensor* out, slope_tensor* lse, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream, Timing* tm) {
  slope_status st;
  Plan plan;
  if ((st = cp_prefill_check(q, k, v, n_chunks, layout, chunk_sizes, causal, window, flags, out, lse, workspace,
                             workspace_bytes, plan)) != SLOPE_OK)
    return st;
  const int64_t S = q->shape[0], Hq = q->shape[1], dqk = q->shape[2];
  const int64_t Hkv = k->shape[1], dv = v->shape[2];
  const WorkspaceLayout wl = workspace_layout(S, Hq, dv, plan.n_planes, flags, plan.direct);
  const bool bf16_partials = (flags & SLOPE_CP_BF16_PARTIALS) != 0;
  int* status = device_status_ptr();
  if (status == nullptr) return cuda_fail("device status word (cudaGetSymbolAddress)");

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q) || !make_map(&tk, k) || !make_map(&tv, v)) return cuda_fail("cuTensorMapEncodeTiled");

  void* planes = workspace;  // fp32 or bf16 elements
  float* lse_planes = reinterpret_cast<float*>(static_cast<char*>(workspace) + wl.lse_offset);
  AttnParams base{};
  base.Hq = static_cast<int32_t>(Hq);
  base.group = static_cast<int32_t>(Hq / Hkv);
  base.pair_heads = pair_heads(Hq, Hkv) ? 1 : 0;
  base.causal = causal ? 1 : 0;
  base.window = static_cast<int32_t>(window);
  base.q_pos_off = 0;
  base.kv_pos_off = 0;
  base.write_empty_out = 0;  // the merge never reads partials whose lse is -inf
  base.scale_log2 = resolve_scale(scale, dqk) * 1.44269504088896340736f;
  base.out = static_cast<float*>(planes);  // the kernel reinterprets it as bf16 under out_bf16
  base.out_srow = Hq * dv;
  base.out_shead = dv;
  base.out_splane = S * Hq * dv;
  base.lse = lse_planes;
  base.lse_srow = Hq;
  base.lse_shead = 1;
  base.lse_splane = S * Hq;
  base.status = status;
  base.wait_limit_ns = wait_limit_ns();
  CUtensorMap to;
  if (plan.direct) {
    // the items write the final out (and lse, else the workspace's lse plane) themselves
    base.write_empty_out = 1;
    base.out = static_cast<float*>(out->data);
    base.out_srow = out->stride[0];
    base.out_shead = out->stride[1];
    base.out_splane = 0;
    base.out_plane_rows = 0;
    base.out_bf16 = out->dtype == SLOPE_BF16 ? 1 : 0;
    base.out_tma =
        make_out_map(&to, out->data, base.out_bf16 != 0, S, Hq, dv, out->stride[0], out->stride[1]) ? 1 : 0;
    if (lse != nullptr) {
      base.lse = static_cast<float*>(lse->data);
      base.lse_srow = lse->stride[1];
      base.lse_shead = lse->stride[0];
    }
    base.lse_splane = 0;
  } else {
    base.out_plane_rows = S;
    base.out_bf16 = bf16_partials ? 1 : 0;
    base.out_tma =
        make_out_map(&to, planes, bf16_partials, static_cast<int64_t>(plan.n_planes) * S, Hq, dv, Hq * dv, dv) ? 1 : 0;
  }
  if (!base.out_tma) to = tq;  // never used

  // A plane none of whose items sees a key (ring steps that a sliding window leaves
  // empty) is neither computed nor merged: its partials would all be out = 0 and
  // lse = -inf, which the merge ignores.  Plane 0 is always kept, so that the merge
  // writes -inf / 0 for rows that see nothing at all.
  std::vector<char> plane_live(static_cast<size_t>(plan.n_planes), 0);
  plane_live[0] = 1;
  for (const PItem& it : plan.items)
    if (it.n_kv > 0) plane_live[static_cast<size_t>(it.plane)] = 1;
  if (!plan.direct) {
    // the live planes' lse starts at -inf: rows that no item covers read as empty partials
    FillParams fp{};
    fp.base = lse_planes;
    fp.plane_elems = S * Hq;
    for (int pl = 0; pl < plan.n_planes; ++pl)
      if (plane_live[static_cast<size_t>(pl)]) fp.planes[fp.n++] = pl;
    cudaError_t e;
    if ((e = record(tm, true, 2, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
    if ((e = launch_lse_fill(fp, stream)) != cudaSuccess) return cuda_fail("lse fill kernel launch", e);
    if ((e = record(tm, false, 2, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  }

  // Ring steps / chunks in order.  Their partials are independent of each other on one GPU
  // (every step reads only the inputs and writes its own plane), so consecutive steps share
  // a kernel launch up to the launch's item limit: each partial is computed by the same code
  // as in a launch of its own, with fewer launch prologues and tails.
  size_t i = 0;
  int launched = 0;  // attention launches of this call so far
  std::vector<std::vector<WorkItem>> groups;
  for (int l = 0; l < plan.n_launches;) {
    std::vector<PItem> items;
    for (; l < plan.n_launches; ++l) {
      std::vector<PItem> step_items;
      size_t j = i;
      for (; j < plan.items.size() && plan.items[j].launch == l; ++j)
        if (plane_live[static_cast<size_t>(plan.items[j].plane)]) step_items.push_back(plan.items[j]);
      if (!items.empty() && items.size() + step_items.size() > static_cast<size_t>(kMaxItems)) break;
      items.insert(items.end(), step_items.begin(), step_items.end());
      i = j;
    }
    if (items.empty()) continue;
    if (!pack_items(items, causal, Hq, base.pair_heads != 0, groups)) return SLOPE_ERR_UNSUPPORTED;
    for (const auto& g : groups) {
      if ((st = run_attention(g, static_cast<int>(dqk), static_cast<int>(dv), tq, tk, tv, to, base, launched > 0, tm,
                              stream)) != SLOPE_OK)
        return st;
      ++launched;
    }
  }
  if (plan.direct) return SLOPE_OK;

  MergeParams mp{};
  mp.n = 0;
  mp.H = static_cast<int32_t>(Hq);
  mp.dv = static_cast<int32_t>(dv);
  mp.S = S;
  mp.in_bf16 = bf16_partials ? 1 : 0;
  for (int pl = 0; pl < plan.n_planes; ++pl) {
    if (!plane_live[static_cast<size_t>(pl)]) continue;
    const int m = mp.n++;
    mp.outs[m] = static_cast<const char*>(planes) + static_cast<size_t>(pl) * wl.out_bytes;
    mp.lses[m] = lse_planes + static_cast<int64_t>(pl) * S * Hq;
    mp.o_srow[m] = Hq * dv;
    mp.o_shead[m] = dv;
    mp.l_srow[m] = Hq;
    mp.l_shead[m] = 1;
  }
  mp.out = out->data;
  mp.out_bf16 = out->dtype == SLOPE_BF16 ? 1 : 0;
  mp.out_srow = out->stride[0];
  mp.out_shead = out->stride[1];
  mp.lse = lse != nullptr ? static_cast<float*>(lse->data) : nullptr;
  mp.lse_srow = lse != nullptr ? lse->stride[1] : 0;
  mp.lse_shead = lse != nullptr ? lse->stride[0] : 0;
  cudaError_t e;
  if ((e = record(tm, true, 1, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  if ((e = launch_lse_merge(mp, stream)) != cudaSuccess) return cuda_fail("merge kernel launch", e);
  if ((e = record(tm, false, 1, stream)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  return SLOPE_OK;
}

// ---------------------------------------------------------------- fixed scratch (no allocation)

// Partials of slope_cp_prefill_static_scratch: one array per device that loads the library.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
std::atomic<void*> g_static_scratch_ptr[64];

// Device address of the scratch array for the current device, looked up once per device.
void* static_scratch_ptr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail("cudaGetDevice", e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    cuda_fail("fixed scratch: device index out of range");
    return nullptr;
  }
  void* ptr = g_static_scratch_ptr[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cuda_fail("cudaGetSymbolAddress(fixed scratch)", e);
      return nullptr;
    }
    g_static_scratch_ptr[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

}  // namespace

// ==================================================================== exported

// ---------------------------------------------------------------- host-buffer prefill

namespace {

// A dense (row-major, no padding) tensor: the host copy and its device buffer are then
// one contiguous block each, moved by one cudaMemcpyAsync.
bool dense(const slope_tensor* t) {
  if (t->ndim == 3) return t->stride[2] == 1 && t->stride[1] == t->shape[2] && t->stride[0] == t->shape[1] * t->shape[2];
  if (t->ndim == 2) return t->stride[1] == 1 && t->stride[0] == t->shape[1];
  return false;
}
bool same_shape(const slope_tensor* a, const slope_tensor* b) {
  if (a->ndim != b->ndim || a->dtype != b->dtype) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}
size_t tensor_bytes(const slope_tensor* t) {
  size_t n = t->dtype == SLOPE_BF16 ? 2 : 4;
  for (int i = 0; i < t->ndim; ++i) n *= static_cast<size_t>(t->shape[i]);
  return n;
}

// Ordering between calls that reuse one set of device buffers, keyed by (device, q buffer):
// `in_ready`  the input copies into the buffers are done,
// `consumed`  the compute that read them (and wrote out/lse) is done,
// `drained`   the output copies that read out/lse are done.
struct BufferSetEvents {
  int device = -1;
  const void* key = nullptr;
  cudaEvent_t in_ready = nullptr, consumed = nullptr, drained = nullptr;
  bool used = false;  // events hold the records of an earlier call
};
constexpr int kBufferSets = 16;
std::mutex g_buffer_sets_mutex;
BufferSetEvents g_buffer_sets[kBufferSets];
int g_buffer_sets_next = 0;

// The entry of (device, key), creating it (or taking the oldest slot) if absent.  A slot
// taken from another buffer set first waits (on the host) for that set's last call to
// finish, so a later call on the evicted set starts with no work of its own pending.
BufferSetEvents* buffer_set(int device, const void* key) {
  for (auto& b : g_buffer_sets)
    if (b.device == device && b.key == key) return &b;
  BufferSetEvents& b = g_buffer_sets[g_buffer_sets_next];
  g_buffer_sets_next = (g_buffer_sets_next + 1) % kBufferSets;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return nullptr;
  if (b.in_ready != nullptr) {
    // the slot's events belong to b.device: work on them with that device current, and
    // make `cur` current again on every path
    const bool switched = b.device != cur;
    if (switched && cudaSetDevice(b.device) != cudaSuccess) return nullptr;
    const cudaError_t sync = b.used ? cudaEventSynchronize(b.drained) : cudaSuccess;
    if (sync == cudaSuccess && b.device != device) {
      cudaEventDestroy(b.in_ready);
      cudaEventDestroy(b.consumed);
      cudaEventDestroy(b.drained);
      b.in_ready = b.consumed = b.drained = nullptr;
    }
    if (switched && cudaSetDevice(cur) != cudaSuccess) return nullptr;
    if (sync != cudaSuccess) return nullptr;
  }
  b.used = false;
  b.key = key;
  b.device = device;
  if (b.in_ready == nullptr &&
      (cudaEventCreateWithFlags(&b.in_ready, cudaEventDisableTiming) != cudaSuccess ||
       cudaEventCreateWithFlags(&b.consumed, cudaEventDisableTiming) != cudaSuccess ||
       cudaEventCreateWithFlags(&b.drained, cudaEventDisableTiming) != cudaSuccess)) {
    b.device = -1;
    b.key = nullptr;
    return nullptr;
  }
  return &b;
}

}  // namespace

// One NVTX range around each public call that queues GPU work, named after the call, so that
// Nsight tools group its launches (ncu --nvtx).  With no tool attached a push or pop is a check
// of a function pointer.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

extern "C" {

slope_status slope_attn_partial(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int64_t q_off,
                                int64_t kv_off, int causal, int64_t window, float scale, slope_tensor* out,
                                slope_tensor* lse, void* stream) {
  const CallRange range("slope_attn_partial");
  slope_status st;
  if ((st = check_qkv(q)) != SLOPE_OK) return st;
  if (k == nullptr || v == nullptr) return SLOPE_ERR_NULL;
  if (k->dtype != SLOPE_BF16 || v->dtype != SLOPE_BF16) return SLOPE_ERR_DTYPE;
  if (k->ndim != 3 || v->ndim != 3) return SLOPE_ERR_SHAPE;
  const int64_t Sq = q->shape[0], Hq = q->shape[1], dqk = q->shape[2];
  const int64_t Skv = k->shape[0], Hkv = k->shape[1], dv = v->shape[2];
  if (Skv > 0) {
    if ((st = check_qkv(k)) != SLOPE_OK || (st = check_qkv(v)) != SLOPE_OK) return st;
  } else if (k->shape[1] <= 0 || v->shape[1] <= 0 || v->shape[2] <= 0 || k->shape[0] < 0) {
    return SLOPE_ERR_SHAPE;
  }
  if (v->shape[0] != Skv || v->shape[1] != Hkv || k->shape[2] != dqk) return SLOPE_ERR_SHAPE;
  if (Hq % Hkv != 0) return SLOPE_ERR_SHAPE;
  if (!attn_partial_supported(static_cast<int>(dqk), static_cast<int>(dv))) return SLOPE_ERR_UNSUPPORTED;
  if (window < 0 || window > kMaxSeq) return SLOPE_ERR_SHAPE;
  // every query and key position within [-2^28, 2^28]
  if (q_off < -kMaxPos || q_off + Sq > kMaxPos || kv_off < -kMaxPos || kv_off + Skv > kMaxPos) return SLOPE_ERR_SHAPE;
  if ((st = check_out(out, Sq, Hq, dv, true)) != SLOPE_OK) return st;
  // bf16 rows are written 16 bytes at a time
  if (out->dtype == SLOPE_BF16 && (out->stride[0] % 8 || out->stride[1] % 8 || !aligned(out->data, 16)))
    return SLOPE_ERR_STRIDE;
  if ((st = check_lse(lse, Hq, Sq)) != SLOPE_OK) return st;
  if (Sq == 0) return SLOPE_OK;
  int* status = device_status_ptr();
  if (status == nullptr) return cuda_fail("device status word (cudaGetSymbolAddress)");

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q)) return cuda_fail("cuTensorMapEncodeTiled");
  if (Skv > 0) {
    if (!make_map(&tk, k) || !make_map(&tv, v)) return cuda_fail("cuTensorMapEncodeTiled");
  } else {
    tk = tq;  // never read: an item with no key range issues no K/V load
    tv = tq;
  }
  PItem it{};
  it.q_row0 = 0;
  it.q_len = Sq;
  it.plane = 0;
  it.n_kv = 0;
  if (Skv > 0) {
    // positions of the query block / key block
    int64_t k0 = kv_off, k1 = kv_off + Skv;
    if (trim(q_off, q_off + Sq, k0, k1, causal, window)) it.kv[it.n_kv++] = Range{k0 - kv_off, k1 - k0};
  }
  std::vector<std::vector<WorkItem>> groups;
  if (!pack_items({it}, causal, Hq, pair_heads(Hq, Hkv), groups)) return SLOPE_ERR_UNSUPPORTED;

  AttnParams base{};
  base.Hq = static_cast<int32_t>(Hq);
  base.group = static_cast<int32_t>(Hq / Hkv);
  base.pair_heads = pair_heads(Hq, Hkv) ? 1 : 0;
  base.causal = causal ? 1 : 0;
  base.window = static_cast<int32_t>(window);
  base.q_pos_off = static_cast<int32_t>(q_off);
  base.kv_pos_off = static_cast<int32_t>(kv_off);
  base.write_empty_out = 1;
  base.scale_log2 = resolve_scale(scale, dqk) * 1.44269504088896340736f;
  base.out = static_cast<float*>(out->data);
  base.out_srow = out->stride[0];
  base.out_shead = out->stride[1];
  base.out_splane = 0;
  base.lse = static_cast<float*>(lse->data);
  base.lse_srow = lse->stride[1];
  base.lse_shead = lse->stride[0];
  base.lse_splane = 0;
  base.status = status;
  base.wait_limit_ns = wait_limit_ns();
  CUtensorMap to;
  base.out_plane_rows = 0;
  base.out_bf16 = out->dtype == SLOPE_BF16 ? 1 : 0;
  base.out_tma = make_out_map(&to, out->data, base.out_bf16 != 0, Sq, Hq, dv, out->stride[0], out->stride[1]) ? 1 : 0;
  if (!base.out_tma) to = tq;  // never used
  return run_attention(groups[0], static_cast<int>(dqk), static_cast<int>(dv), tq, tk, tv, to, base, false, nullptr,
                       static_cast<cudaStream_t>(stream));
}

slope_status slope_lse_merge(const slope_tensor* outs, const slope_tensor* lses, int n, slope_tensor* out,
                             slope_tensor* lse, void* stream) {
  const CallRange range("slope_lse_merge");
  if (outs == nullptr || lses == nullptr || out == nullptr) return SLOPE_ERR_NULL;
  if (n < 1 || n > kMaxMerge) return SLOPE_ERR_SHAPE;
  if (out->ndim != 3) return SLOPE_ERR_SHAPE;
  const int64_t S = out->shape[0], H = out->shape[1], dv = out->shape[2];
  if (!merge_dv_supported(dv)) return SLOPE_ERR_UNSUPPORTED;
  if (S < 0 || S > kMaxSeq || H <= 0 || H > 65535) return SLOPE_ERR_SHAPE;
  slope_status st;
  if ((st = check_out(out, S, H, dv, true)) != SLOPE_OK) return st;
  if (lse != nullptr && (st = check_lse(lse, H, S)) != SLOPE_OK) return st;
  MergeParams mp{};
  for (int i = 0; i < n; ++i) {
    if ((st = check_out(&outs[i], S, H, dv, true)) != SLOPE_OK) return st;
    if (outs[i].dtype != outs[0].dtype) return SLOPE_ERR_DTYPE;  // one dtype for all partials
    if ((st = check_lse(&lses[i], H, S)) != SLOPE_OK) return st;
    mp.outs[i] = outs[i].data;
    mp.o_srow[i] = outs[i].stride[0];
    mp.o_shead[i] = outs[i].stride[1];
    mp.lses[i] = static_cast<const float*>(lses[i].data);
    mp.l_srow[i] = lses[i].stride[1];
    mp.l_shead[i] = lses[i].stride[0];
  }
  if (S == 0) return SLOPE_OK;
  mp.n = n;
  mp.H = static_cast<int32_t>(H);
  mp.dv = static_cast<int32_t>(dv);
  mp.S = S;
  mp.in_bf16 = outs[0].dtype == SLOPE_BF16 ? 1 : 0;
  mp.out = out->data;
  mp.out_bf16 = out->dtype == SLOPE_BF16 ? 1 : 0;
  mp.out_srow = out->stride[0];
  mp.out_shead = out->stride[1];
  mp.lse = lse != nullptr ? static_cast<float*>(lse->data) : nullptr;
  mp.lse_srow = lse != nullptr ? lse->stride[1] : 0;
  mp.lse_shead = lse != nullptr ? lse->stride[0] : 0;
  const cudaError_t e = launch_lse_merge(mp, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SLOPE_OK : cuda_fail("merge kernel launch", e);
}

size_t slope_cp_prefill_workspace_size_ex(int64_t S, int64_t Hq, int64_t dv, int n_chunks, slope_layout layout,
                                          const int64_t* chunk_sizes, unsigned flags) {
  if (S <= 0 || S > kMaxSeq || Hq <= 0 || !merge_dv_supported(dv)) return 0;
  if (!flags_valid(flags)) return 0;
  Plan plan;
  if (build_plan(S, n_chunks, layout, chunk_sizes, 1, 0, flags, plan) != SLOPE_OK) return 0;
  return workspace_layout(S, Hq, dv, plan.n_planes, flags, plan.direct).total;
}

size_t slope_cp_prefill_workspace_size(int64_t S, int64_t Hq, int64_t dv, int n_chunks, slope_layout layout,
                                       const int64_t* chunk_sizes) {
  return slope_cp_prefill_workspace_size_ex(S, Hq, dv, n_chunks, layout, chunk_sizes, 0u);
}

slope_status slope_cp_prefill(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int n_chunks,
                              slope_layout layout, const int64_t* chunk_sizes, int causal, int64_t window,
                              float scale, slope_tensor* out, slope_tensor* lse, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const CallRange range("slope_cp_prefill");
  return cp_prefill_impl(q, k, v, n_chunks, layout, chunk_sizes, causal, window, scale, 0u, out, lse, workspace,
                         workspace_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

slope_status slope_cp_prefill_ex(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int n_chunks,
                                 slope_layout layout, const int64_t* chunk_sizes, int causal, int64_t window,
                                 float scale, unsigned flags, slope_tensor* out, slope_tensor* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const CallRange range("slope_cp_prefill_ex");
  return cp_prefill_impl(q, k, v, n_chunks, layout, chunk_sizes, causal, window, scale, flags, out, lse, workspace,
                         workspace_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

slope_status slope_cp_prefill_static_scratch(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                             int n_chunks, slope_layout layout, const int64_t* chunk_sizes,
                                             int causal, int64_t window, float scale, slope_tensor* out,
                                             slope_tensor* lse, void* stream) {
  const CallRange range("slope_cp_prefill_static_scratch");
  if (q == nullptr || v == nullptr) return SLOPE_ERR_NULL;
  if (q->ndim != 3 || v->ndim != 3) return SLOPE_ERR_SHAPE;
  const size_t need = slope_cp_prefill_workspace_size(q->shape[0], q->shape[1], v->shape[2], n_chunks, layout,
                                                      chunk_sizes);
  if (need > kStaticScratchBytes) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "fixed scratch holds %zu bytes; this request needs %zu (use slope_cp_prefill with a workspace)",
                  kStaticScratchBytes, need);
    return SLOPE_ERR_WORKSPACE;
  }
  void* scratch = static_scratch_ptr();
  if (scratch == nullptr) return SLOPE_ERR_CUDA;
  return slope_cp_prefill(q, k, v, n_chunks, layout, chunk_sizes, causal, window, scale, out, lse, scratch,
                          kStaticScratchBytes, stream);
}

slope_status slope_cp_prefill_timed(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                    int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                                    int64_t window, float scale, slope_tensor* out, slope_tensor* lse,
                                    void* workspace, size_t workspace_bytes, void* stream, void** events,
                                    int n_event_pairs, int* n_launches, int* launch_kind) {
  const CallRange range("slope_cp_prefill_timed");
  if (events == nullptr || n_launches == nullptr) return SLOPE_ERR_NULL;
  Timing tm;
  tm.events = events;
  tm.capacity = n_event_pairs;
  tm.kinds = launch_kind;
  // count launches first so that a short event array is an argument error, not a partial run
  if (q != nullptr && q->ndim == 3) {
    Plan plan;
    if (build_plan(q->shape[0], n_chunks, layout, chunk_sizes, causal, window, 0u, plan) == SLOPE_OK) {
      int needed = 2;  // the lse fill and the merge
      size_t i = 0;
      for (int l = 0; l < plan.n_launches; ++l) {
        size_t c = 0;
        while (i < plan.items.size() && plan.items[i].launch == l) ++i, ++c;
        needed += static_cast<int>((c + kMaxItems - 1) / kMaxItems);
      }
      if (needed > n_event_pairs) return SLOPE_ERR_SHAPE;
    }
  }
  slope_status st = cp_prefill_impl(q, k, v, n_chunks, layout, chunk_sizes, causal, window, scale, 0u, out, lse,
                                    workspace, workspace_bytes, static_cast<cudaStream_t>(stream), &tm);
  *n_launches = tm.count;
  return st;
}

slope_status slope_cp_prefill_host(const slope_tensor* q_host, const slope_tensor* k_host,
                                   const slope_tensor* v_host, slope_tensor* out_host, slope_tensor* lse_host,
                                   const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                   slope_tensor* out, slope_tensor* lse, int n_chunks, slope_layout layout,
                                   const int64_t* chunk_sizes, int causal, int64_t window, float scale,
                                   void* workspace, size_t workspace_bytes, void* copy_in_stream,
                                   void* compute_stream, void* copy_out_stream) {
  const CallRange range("slope_cp_prefill_host");
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr || q == nullptr ||
      k == nullptr || v == nullptr || out == nullptr)
    return SLOPE_ERR_NULL;
  if ((lse_host == nullptr) != (lse == nullptr)) return SLOPE_ERR_NULL;
  const slope_tensor* pairs[5][2] = {{q_host, q}, {k_host, k}, {v_host, v}, {out_host, out}, {lse_host, lse}};
  for (auto& pr : pairs) {
    if (pr[0] == nullptr) continue;
    if (!same_shape(pr[0], pr[1])) return SLOPE_ERR_SHAPE;
    if (!dense(pr[0]) || !dense(pr[1])) return SLOPE_ERR_STRIDE;
    if (tensor_bytes(pr[0]) > 0 && pr[0]->data == nullptr) return SLOPE_ERR_NULL;
  }
  // every check of the compute runs before anything is queued
  Plan probe;
  slope_status st = cp_prefill_check(q, k, v, n_chunks, layout, chunk_sizes, causal, window, 0u, out, lse, workspace,
                                     workspace_bytes, probe);
  if (st != SLOPE_OK) return st;
  if (out->dtype != SLOPE_BF16 && out->dtype != SLOPE_F32) return SLOPE_ERR_DTYPE;
  int device = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&device)) != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  auto s_in = static_cast<cudaStream_t>(copy_in_stream);
  auto s_c = static_cast<cudaStream_t>(compute_stream);
  auto s_out = static_cast<cudaStream_t>(copy_out_stream);
  std::lock_guard<std::mutex> guard(g_buffer_sets_mutex);
  BufferSetEvents* b = buffer_set(device, q->data);
  if (b == nullptr) return cuda_fail("cudaEventCreateWithFlags (buffer-set events)");
  // inputs: after the previous compute on these buffers has read them
  if (b->used && (e = cudaStreamWaitEvent(s_in, b->consumed, 0)) != cudaSuccess)
    return cuda_fail("cudaStreamWaitEvent", e);
  for (int i = 0; i < 3; ++i)
    if ((e = cudaMemcpyAsync(const_cast<void*>(pairs[i][1]->data), pairs[i][0]->data, tensor_bytes(pairs[i][0]),
                             cudaMemcpyHostToDevice, s_in)) != cudaSuccess)
      return cuda_fail("cudaMemcpyAsync (host to device)", e);
  if ((e = cudaEventRecord(b->in_ready, s_in)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  // compute: after the inputs, and after the previous output copies have read out/lse
  if ((e = cudaStreamWaitEvent(s_c, b->in_ready, 0)) != cudaSuccess) return cuda_fail("cudaStreamWaitEvent", e);
  if (b->used && (e = cudaStreamWaitEvent(s_c, b->drained, 0)) != cudaSuccess)
    return cuda_fail("cudaStreamWaitEvent", e);
  st = cp_prefill_impl(q, k, v, n_chunks, layout, chunk_sizes, causal, window, scale, 0u, out, lse, workspace,
                       workspace_bytes, s_c, nullptr);
  if (st != SLOPE_OK) return st;
  if ((e = cudaEventRecord(b->consumed, s_c)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  // outputs: after the compute
  if ((e = cudaStreamWaitEvent(s_out, b->consumed, 0)) != cudaSuccess) return cuda_fail("cudaStreamWaitEvent", e);
  for (int i = 3; i < 5; ++i) {
    if (pairs[i][0] == nullptr) continue;
    if ((e = cudaMemcpyAsync(pairs[i][0]->data, pairs[i][1]->data, tensor_bytes(pairs[i][1]),
                             cudaMemcpyDeviceToHost, s_out)) != cudaSuccess)
      return cuda_fail("cudaMemcpyAsync (device to host)", e);
  }
  if ((e = cudaEventRecord(b->drained, s_out)) != cudaSuccess) return cuda_fail("cudaEventRecord", e);
  b->used = true;
  return SLOPE_OK;
}

int64_t slope_cp_prefill_plan_ex(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes,
                                 int causal, int64_t window, unsigned flags, slope_plan_item* items, int64_t capacity,
                                 int32_t* n_launches, int32_t* n_planes) {
  if (!flags_valid(flags)) return SLOPE_ERR_UNSUPPORTED;
  Plan plan;
  slope_status st = build_plan(S, n_chunks, layout, chunk_sizes, causal, window, flags, plan);
  if (st != SLOPE_OK) return st;
  if (capacity > 0 && items == nullptr) return SLOPE_ERR_NULL;
  for (int64_t i = 0; i < static_cast<int64_t>(plan.items.size()) && i < capacity; ++i) {
    const PItem& p = plan.items[i];
    slope_plan_item& o = items[i];
    std::memset(&o, 0, sizeof(o));
    o.launch = p.launch;
    o.plane = p.plane;
    o.q_row0 = p.q_row0;
    o.q_len = p.q_len;
    o.n_kv = p.n_kv;
    for (int r = 0; r < p.n_kv; ++r) {
      o.kv_row0[r] = p.kv[r].row0;
      o.kv_len[r] = p.kv[r].len;
    }
    o.head_group = p.hg;
    o.n_head_groups = p.n_hg;
  }
  if (n_launches != nullptr) *n_launches = plan.n_launches;
  if (n_planes != nullptr) *n_planes = plan.n_planes;
  return static_cast<int64_t>(plan.items.size());
}

int64_t slope_cp_prefill_plan(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                              int64_t window, slope_plan_item* items, int64_t capacity, int32_t* n_launches,
                              int32_t* n_planes) {
  return slope_cp_prefill_plan_ex(S, n_chunks, layout, chunk_sizes, causal, window, 0u, items, capacity, n_launches,
                                  n_planes);
}

slope_status slope_device_status(void* stream, int* site) {
  if (site != nullptr) *site = 0;
  cudaError_t e;
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail("cudaStreamSynchronize", e);
  int* ptr = device_status_ptr();
  if (ptr == nullptr) return cuda_fail("device status word (cudaGetSymbolAddress)");
  int word[2] = {0, 0};
  if ((e = cudaMemcpy(word, ptr, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail("cudaMemcpy", e);
  if (word[0] == 0) return SLOPE_OK;
  const int zero[2] = {0, 0};
  if ((e = cudaMemcpy(ptr, zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail("cudaMemcpy", e);
  if (site != nullptr) *site = word[1];
  return SLOPE_ERR_TIMEOUT;
}

slope_status slope_debug_timeout_selftest(uint64_t limit_ns, void* stream) {
  const CallRange range("slope_debug_timeout_selftest");
  if (limit_ns < 1000ull || limit_ns > 5000000000ull) return SLOPE_ERR_SHAPE;
  int* ptr = device_status_ptr();
  if (ptr == nullptr) return cuda_fail("device status word (cudaGetSymbolAddress)");
  const cudaError_t e = launch_timeout_selftest(limit_ns, ptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SLOPE_OK : cuda_fail("self-test kernel launch", e);
}

const char* slope_status_string(slope_status s) {
  switch (s) {
    case SLOPE_OK: return "ok";
    case SLOPE_ERR_NULL: return "null pointer";
    case SLOPE_ERR_DTYPE: return "wrong dtype";
    case SLOPE_ERR_SHAPE: return "bad or inconsistent shape";
    case SLOPE_ERR_STRIDE: return "bad stride or alignment";
    case SLOPE_ERR_LAYOUT: return "layout does not divide the sequence";
    case SLOPE_ERR_CUDA: return "CUDA error";
    case SLOPE_ERR_TIMEOUT: return "bounded device wait timed out";
    case SLOPE_ERR_UNSUPPORTED: return "unsupported configuration";
    case SLOPE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

const char* slope_version(void) { return "slope-gb300 0.1.0 (sm_103a)"; }

const char* slope_last_error(void) { return g_last_error; }

}  // extern "C"
