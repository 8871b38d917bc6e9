// Parameter blocks shared by the host launcher and the two kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "slope.h"

namespace slope {

// ---------------------------------------------------------------- attention partial (K1)

constexpr int kBlockM = 128;      // query rows per Q tile (= TMEM lanes)
constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kQTiles = 2;        // Q tiles per CTA at most; a CTA's Q tiles share every K/V tile
constexpr int kRowsPerCta = kBlockM * kQTiles;  // rows of a one-head work tile with two Q tiles
constexpr int kMaxItems = 32;     // work items per launch
constexpr int kMaxKvRanges = 2;   // key/value ranges per item

struct KvRange {
  int32_t row0;  // first key row (in the k/v tensors)
  int32_t len;   // keys in the range
};

// One query block of a range of query heads, and the key/value ranges it attends to in
// this launch.  Its work tiles are (row block, head unit) pairs, where a head unit is one
// head (the CTA's two Q tiles are 256 consecutive rows of it) or, with
// AttnParams::pair_heads, two heads of one KV group (the two Q tiles are the same 128
// rows of both).  Tiles run unit group by unit group (AttnParams::head_group units each),
// and in a group row blocks from the last one down with the group's units inner.
struct WorkItem {
  int32_t q_row0;      // first query row (in q)
  int32_t q_len;       // query rows
  int32_t out_row0;    // output row of q_row0
  int32_t plane;       // output plane
  int32_t n_kv;        // 0..kMaxKvRanges
  int32_t tile_begin;  // first work tile of this item (prefix sum over items of n_blocks * head units)
  int32_t n_blocks;    // ceil(q_len / rows per work tile): 128 with pair_heads or one Q tile per
                       // CTA (the launcher recounts for that kernel), else kRowsPerCta
  int32_t h_begin;     // first query head
  int32_t h_count;     // query heads (whole KV-head groups)
  KvRange kv[kMaxKvRanges];
};
static_assert(sizeof(WorkItem) % 4 == 0, "work items are copied as 32-bit words");

struct AttnParams {
  int32_t n_items;
  int32_t total_tiles;      // work tiles (sum over items of row blocks x heads); set by the launcher
  int32_t head_group;       // head units per tile group (divides every item's unit count; 0 = one group
                            // per item); set by the launcher
  int32_t pair_heads;       // 1: a work tile's two Q tiles are two heads of one KV group on the same
                            // 128 rows (needs an even Hq / Hkv); 0: 256 consecutive rows of one head
  int32_t Hq;
  int32_t group;            // Hq / Hkv
  int32_t causal;
  int32_t window;           // 0 = none
  int32_t q_pos_off;        // global position of q row 0
  int32_t kv_pos_off;       // global position of k row 0
  int32_t write_empty_out;  // write zeros to out for rows that see no key
  float scale_log2;         // softmax scale * log2(e)
  float* out;               // output planes: fp32 partials, or bf16 when out_bf16
  int64_t out_srow, out_shead, out_splane;  // in elements
  int32_t out_bf16;         // 1: out holds bf16 (a final output, not a partial)
  int32_t out_tma;          // 1: full 32-row warp chunks of out go through the O tensor map
  int64_t out_plane_rows;   // rows per plane in the O tensor map's outer dimension
  float* lse;               // fp32 log-sum-exp planes
  int64_t lse_srow, lse_shead, lse_splane;
  int* status;              // device status word {code, site}
  uint32_t* tile_counter;   // 0 at launch: work tiles claimed so far (kernels that claim them at run
                            // time); set by the launcher
  uint64_t wait_limit_ns;   // bound on every barrier wait
  WorkItem items[kMaxItems];
};

// ---------------------------------------------------------------- merge (K2)

constexpr int kMaxMerge = 32;
constexpr int kMergeThreads = 256;

struct MergeParams {
  int32_t n;
  int32_t H;
  int32_t dv;
  int32_t out_bf16;
  int64_t S;
  int32_t in_bf16;  // partials are bf16 (else fp32)
  const void* outs[kMaxMerge];
  const float* lses[kMaxMerge];
  int64_t o_srow[kMaxMerge], o_shead[kMaxMerge];
  int64_t l_srow[kMaxMerge], l_shead[kMaxMerge];
  void* out;
  int64_t out_srow, out_shead;
  float* lse;  // may be null
  int64_t lse_srow, lse_shead;
};

// -inf into whole fp32 lse planes: base + planes[i] * plane_elems, i < n.
struct FillParams {
  float* base;
  int64_t plane_elems;
  int32_t n;
  int32_t planes[kMaxMerge];
};

// Status codes written into the device status word.
constexpr int kStatusTimeout = 1;

// Host-side launchers (defined in attn_partial.cu / lse_merge.cu / status.cu).
// dependent: launch as a programmatic dependent of the previous kernel in the stream, which
// must be another attention launch of the same decomposition (one that writes none of what
// this one reads or writes).
cudaError_t launch_attn_partial(int dqk, int dv, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to, const AttnParams& p, bool dependent,
                                cudaStream_t stream);
bool attn_partial_supported(int dqk, int dv);
cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_lse_fill(const FillParams& p, cudaStream_t stream);
// Head sizes the merge kernel is built for (64, 128 and 192).
inline bool merge_dv_supported(long long dv) { return dv == 64 || dv == 128 || dv == 192; }
cudaError_t launch_timeout_selftest(uint64_t limit_ns, int* status, cudaStream_t stream);
int* device_status_ptr();  // per current device; nullptr on failure
// Work-tile counters for attention launches that claim tiles at run time (a ring in static device
// memory, each 0 between launches).
constexpr int kTileCounterSlots = SLOPE_TILE_COUNTERS;
uint32_t* claim_tile_counter();  // the next counter of the current device; nullptr on failure

}  // namespace slope
