// Partial attention kernel (ring steps / chunked-prefill chunks, or the whole
// sequence in one launch).
//
// Computes, for every work item (a block of query rows and up to two
// key/value row ranges), softmax attention restricted to the visible keys of
// those ranges and writes the normalised output plus its natural-log
// log-sum-exp: the per-device partial of Ring Attention (Moreh, "Optimizing
// long-context prefill on multiple older-generation GPU nodes", section
// "Introduction to Context Parallelism", Ring Attention item), combined later
// by the log-sum-exp merge.  Over the whole sequence with bf16 output the same
// launch is the complete attention (no partials, no merge).
//
// Persistent grid of CTAs that walk work tiles, heaviest first.  With two Q tiles per CTA
// (windows up to 4096 keys, and dqk >= 128) one CTA holds an SM and a work tile is one item x 128
// query rows x two query heads of one KV group, or x 256 rows of one head; with one Q tile
// (d = 64 otherwise) two CTAs share an SM, each with 6 warps (softmax 0-3, TMA 4,
// MMA 5), 256 TMEM columns and half the shared memory, and a work tile is 128 rows of one
// head.  At d = 64 a CTA takes every gridDim.x-th tile; at dqk >= 128 the CTAs claim tiles
// at run time.  The launch's items sit in shared memory.  With two Q tiles:
//   warps 0-3   online softmax of Q tile 0 (one query row per thread = TMEM lane),
//   warps 4-7   online softmax of Q tile 1; each also runs its tile's epilogue,
//               which stages O in shared memory (32-row x 128-byte boxes per
//               warp, fp32 or bf16) and writes it with TMA stores.
//   warp 8      TMA producer: Q tiles once per work tile, then K and V tiles
//               through a ring of shared-memory slots (128-byte swizzle).
//   warps 9-10  MMA issuers, one per Q tile: S_t = Q_t K^T (SS, K-major) into
//               TMEM, then O_t += P_t V (P from TMEM, V MN-major); warp 9 also
//               owns the 512-column TMEM allocation.
//   warp 11     idle, or, where tiles are claimed at run time, the scheduler: it takes the
//               next work tile from the launch's global counter and hands its index to
//               the other roles through one shared-memory word.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+dv), O_1 after it (one Q tile:
// S [0,128), O [128,192), P [192,256)).
// With dv = 64 the last 128 columns hold P_0 and P_1 (bf16 pairs, 64 columns
// each), so the MMA warp issues S(n+1) = Q K(n+1)^T before O += P(n) V(n) and
// the softmax of step n+1 starts while PV(n) still runs.  With dv = 128 TMEM is
// full: P_t overwrites the first 64 columns of S_t, S(n+1) waits for PV(n), and
// the two softmax warps of each SM sub-partition take turns on the exponentials.
// The load of S returns each 32-column quarter's maximum (tcgen05.ld.red), which
// is the row max of a fully visible tile.  Scores live in the log2 domain
// (scale * log2 e folded into one FMA); the running max is only moved when it
// grows by more than 8 (factor 256), which keeps every p <= 256 and makes most O
// rescales unnecessary; the final normalisation uses the same max, so the
// result is exact either way.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.cuh"
#include "sm103_ptx.cuh"
#include "waits.cuh"

namespace slope {
namespace {

constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 64 bf16 (128 bytes)
// 12 warps put 3 warps on each SM sub-partition (16K registers each), which caps
// a thread at 168 registers.
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units
// Of every 16 element pairs of a score row, this many take 2^x on the FMA pipe
// (softmax_pair_poly) instead of the MUFU unit.  With two softmax warps per SM
// sub-partition, 2 ex2 cost 8 MUFU cycles and the polynomial pair about 14 more FMA-pipe
// cycles and 8 more issue slots than the MUFU pair.  That paid while the row max was a
// tree of 3-input max instructions (kernel TFLOP/s on the causal 32K zigzag workload:
// 0 -> 745, 1 -> 749, 2 -> 765, 3 -> 696); since the TMEM load takes the row max, the
// MUFU-only loop is fastest (0 -> 954, 1 -> 927, 2 -> 917, 3 -> 885), so the
// polynomial is compiled out.  With pairs on the polynomial, a masked score (-inf)
// gives 2^-125 instead of 0: once a row has seen a key its sum l is >= 1 and the term
// is far below bf16 resolution; before that the row's max is -inf and the first
// visible key rescales l and O by 0; a row that never sees a key writes 0.
constexpr int kPolyPairsPer16 = 0;

// QT: Q tiles per CTA.  Two share every K/V tile and one CTA holds the SM (all 512 TMEM
// columns, 12 warps); with one, two CTAs share the SM (256 columns and about 100 KB of shared
// memory each, 6 warps each), and one CTA's work-tile boundary (last PV, epilogue, next Q load)
// overlaps the other CTA's steps instead of stalling both Q tiles at once.
template <int DQK, int DV, int QT = 2>
struct K1Cfg {
  static_assert(DQK % 64 == 0 && DV % 64 == 0, "head dims are multiples of 64");
  static_assert(QT == 1 || QT == 2, "one or two Q tiles per CTA");
  static constexpr int kQTiles = QT;
  static constexpr int kTmaWarp = 4 * QT;  // warps 0 .. 4 QT - 1 are the softmax warpgroups
  static constexpr int kMmaWarp = kTmaWarp + 1;
  static constexpr int kSchedWarp = kMmaWarp + QT;  // warp 11 with two Q tiles
  // roles that read each claimed work tile: the TMA thread, the MMA issuers and the softmax warps
  static constexpr int kTileReaders = 1 + QT + 4 * QT;
  static constexpr int kThreads = QT == 2 ? 384 : 192;
  static constexpr int kMinBlocks = QT == 2 ? 1 : 2;
  static constexpr uint32_t kTmemCols = QT == 2 ? 512 : 256;
  static constexpr int kQChunks = DQK / 64;
  static constexpr int kVChunks = DV / 64;
  static constexpr int kQTileBytes = kQChunks * kChunkBytes;
  static constexpr int kKTileBytes = kQChunks * kChunkBytes;
  static constexpr int kVTileBytes = kVChunks * kChunkBytes;
  static constexpr int kSlotBytes = kKTileBytes > kVTileBytes ? kKTileBytes : kVTileBytes;
  // Work tiles claimed at run time from a global counter, in tile order, instead of the fixed
  // w = blockIdx.x + k * gridDim.x.  Each CTA then takes the next tile when it has room for
  // one, so the CTAs in flight always hold a window of about one grid's width of consecutive
  // tiles: with one query head per KV head that keeps few heads' K/V in use at a time, which
  // L2 holds, where the fixed order drifts apart (tile costs differ by row block) and spreads
  // the CTAs over many heads.
  static constexpr bool kDynamicTiles = DQK >= 128;
  // 128 KB of K/V slots: 8 of 16 KB at d = 64, 4 of 32 KB with a 128-column K or V tile, 2 of 48 KB at 192
  // (measured on the causal 32K zigzag workload: a second Q buffer, which leaves room for only
  // 6 slots at d = 64, cost 2.5%); 64 KB (4 slots at d = 64) with one Q tile per CTA
  static constexpr int kSlots = (QT == 2 ? 131072 : 65536) / kSlotBytes;
  static_assert(QT == 2 || !kDynamicTiles, "claimed tiles run with two Q tiles per CTA");
  static constexpr int kNumBars = 1 + 2 * kSlots + 6 * QT + 1 + 4 * QT + (kDynamicTiles ? 2 : 0);
  // epilogue staging: 32-row x 32-column fp32 boxes (4 KB each, 128-byte swizzle), two per
  // softmax warp where shared memory allows (the second box is written while the first
  // one's store still reads), else one
  static constexpr int kStageOffset = QT * kQTileBytes + kSlots * kSlotBytes;
  static constexpr int kStageBufs = QT == 2 && kStageOffset + 2 * 4 * QT * 4096 + 2048 <= 232448 ? 2 : 1;
  static constexpr int kStageBytes = kStageBufs * 4 * QT * 4096;
  static constexpr int kBarOffset = kStageOffset + kStageBytes;
  // the launch's work items, copied from the kernel parameters (read on every work tile)
  static constexpr int kItemsOffset = kBarOffset + ((8 * kNumBars + 16 + 15) / 16) * 16;
  static constexpr int kSmemBytes = 1024 + kItemsOffset + kMaxItems * static_cast<int>(sizeof(WorkItem));
  static constexpr uint32_t kColO = QT * kBlockN;
  static constexpr uint32_t kColP = kColO + QT * DV;  // separate P columns, if they fit
  static constexpr bool kSepP = kColP + QT * (kBlockN / 2) <= kTmemCols;
  // one CTA per SM, or two (each within half of the SM's 228 KB less 1 KB reserved per CTA)
  static_assert(kSmemBytes <= (QT == 2 ? 232448 : 115712), "shared memory budget");
  static_assert(kColO + QT * DV <= kTmemCols, "TMEM budget");
  // TMEM column of P_t
  __device__ static constexpr uint32_t col_p(int t) { return kSepP ? kColP + t * (kBlockN / 2) : t * kBlockN; }
  // The two softmax warps of an SM sub-partition take turns on their exponentials where P
  // overwrites S (dv = 128).  Measured (kernel TFLOP/s): MLA shape 192/128 1141 -> 1220
  // with turns; at dv = 64 turns cost more than they save (causal 32K zigzag 956 -> 920).
  static constexpr bool kTurns = !kSepP;
  // Head-grouped tile order (see tile_head_group) for the wider head sizes, where MLA-shaped
  // attention (one query head per KV head) runs; at d = 64 the ungrouped decode is kept, which
  // measured 2% faster on the GQA workloads (where grouping would not change the order).
  static constexpr bool kGroupedTiles = DQK >= 128;
};

__device__ __forceinline__ int floor_div(int a, int b) {
  int q = a / b;
  if ((a % b) != 0 && (a < 0)) --q;
  return q;
}

struct TileGeom {
  int rows[kQTiles];  // valid query rows of each tile (0 = tile unused)
  int qa[kQTiles];    // global position of the tile's first row
  int qb[kQTiles];    // global position of its last valid row
};

struct Step {
  int krow;       // first key row of the K/V tile
  int kpos;       // its global position
  int valid;      // keys of the range inside the tile (<= 128)
  uint32_t part;  // bit t: Q tile t sees at least one key of the tile
  uint32_t full;  // bit t: Q tile t sees every key of the tile (no masking)
};

// Enumerates the K/V tiles of an item that at least one Q tile of this CTA can
// see, in the same order for every role.  f returns false to stop (abort).
template <int QT = kQTiles, typename F>
__device__ __forceinline__ bool for_each_step(const WorkItem& it, const AttnParams& p, const TileGeom& g, F&& f) {
  const int qa_min = g.qa[0];
  const int qb_max = QT == 2 && g.rows[1] > 0 ? g.qb[1] : g.qb[0];
  for (int r = 0; r < it.n_kv; ++r) {
    // select instead of a dynamic index: keeps the ranges in registers
    const int row0 = r == 0 ? it.kv[0].row0 : it.kv[1].row0;
    const int len = r == 0 ? it.kv[0].len : it.kv[1].len;
    const int kpos0 = p.kv_pos_off + row0;
    int lo = 0, hi = (len + kBlockN - 1) / kBlockN - 1;
    if (p.causal) hi = min(hi, floor_div(qb_max - kpos0, kBlockN));
    if (p.window > 0) lo = max(lo, floor_div(qa_min - p.window + 1 - kpos0, kBlockN));
    for (int j = lo; j <= hi; ++j) {
      Step s;
      s.krow = row0 + j * kBlockN;
      s.kpos = kpos0 + j * kBlockN;
      s.valid = min(kBlockN, len - j * kBlockN);
      const int klast = s.kpos + s.valid - 1;
      s.part = 0;
      s.full = 0;
#pragma unroll
      for (int t = 0; t < QT; ++t) {
        if (g.rows[t] <= 0) continue;
        const bool vis = (!p.causal || s.kpos <= g.qb[t]) && (p.window == 0 || g.qa[t] - klast < p.window);
        if (!vis) continue;
        s.part |= 1u << t;
        const bool full = s.valid == kBlockN && (!p.causal || klast <= g.qa[t]) &&
                          (p.window == 0 || g.qb[t] - s.kpos < p.window);
        if (full) s.full |= 1u << t;
      }
      if (s.part && !f(s)) return false;
    }
  }
  return true;
}

// The K/V tiles of one key range that a single Q tile (rows at positions qa..qb)
// sees: j in [lo, hi], and among them the ones it sees in full (no masked key): j in
// [flo, fhi].  Step for step these are the tiles of for_each_step whose part bit for
// that Q tile is set, with its full bit; the softmax warps walk them directly, which
// keeps their per-step loop state to a few registers.
struct TileRange {
  int kpos0, len, lo, hi, flo, fhi;
};
__device__ __forceinline__ TileRange tile_range(int row0, int len, int qa, int qb, const AttnParams& p) {
  TileRange R;
  R.kpos0 = p.kv_pos_off + row0;
  R.len = len;
  const int last = (len + kBlockN - 1) / kBlockN - 1;
  R.hi = p.causal ? min(last, floor_div(qb - R.kpos0, kBlockN)) : last;
  R.lo = 0;
  if (p.window > 0) {
    R.lo = max(0, floor_div(qa - p.window + 1 - R.kpos0, kBlockN));
    // a short last tile: its own last key decides
    if (R.lo == last && qa - (R.kpos0 + len - 1) >= p.window) R.lo = last + 1;
  }
  R.fhi = (len % kBlockN == 0) ? last : last - 1;
  if (p.causal) R.fhi = min(R.fhi, floor_div(qa - R.kpos0 - (kBlockN - 1), kBlockN));
  R.flo = R.lo;
  if (p.window > 0) R.flo = max(R.flo, floor_div(qb - R.kpos0 - p.window, kBlockN) + 1);
  return R;
}

// True if at least one Q tile of the work tile sees at least one key.  Work tiles
// without any (for example ring steps that a sliding window leaves empty) only need
// their -inf log-sum-exp written by the softmax warps: the TMA and MMA warps skip them,
// Q load and all, and count only the others in their Q-buffer phases.
template <int QT = kQTiles>
__device__ __forceinline__ bool has_steps(const WorkItem& it, const AttnParams& p, const TileGeom& g) {
  bool any = false;
  for_each_step<QT>(it, p, g, [&](const Step&) -> bool {
    any = true;
    return false;
  });
  return any;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// One unit of work: an item's block of query rows for one head unit, i.e. 256 rows of one
// head (Q tile t = rows 128t..128t+127 of the block) or, with pair_heads, 128 rows of two
// heads of one KV group (Q tile t = head h + t).  With a pair the two Q tiles see exactly
// the same keys under the same masks, so they take the same steps and reach the end of the
// work tile together; 256 rows of one head give the second Q tile one more (diagonal) step.
struct Tile {
  WorkItem itm;
  int blk, h, g;  // row block, first head of the unit, KV head
  TileGeom geo;
};

// First row (within the item) and head of Q tile t of a work tile (QT Q tiles per CTA; with one,
// a work tile is 128 rows of one head).
template <int QT>
__device__ __forceinline__ int tile_row0(const AttnParams& p, const Tile& T, int t) {
  if constexpr (QT == 1) return T.blk * kBlockM;
  return p.pair_heads ? T.blk * kBlockM : T.blk * kRowsPerCta + t * kBlockM;
}
__device__ __forceinline__ int tile_head(const AttnParams& p, const Tile& T, int t) {
  return p.pair_heads ? T.h + t : T.h;
}

// Work tile w -> (item, row block, head unit).  Consecutive w are the units of one row
// block (K/V shared in L2 by a KV group); items come heaviest first and an item's
// later (heavier under the causal mask) row blocks before its earlier ones.
// `ii` carries the item index from the caller's previous work tile: a CTA visits its
// tiles in increasing w, so the item index never decreases and the scan resumes there.
// kGrouped: tiles run unit group by unit group (p.head_group units each); otherwise every
// unit of an item is inner to its row blocks.
template <bool kGrouped, int QT>
__device__ __forceinline__ void decode_tile(const AttnParams& p, const WorkItem* items, int w, Tile& T, int& ii) {
  const int ushift = p.pair_heads;  // head units per item = h_count >> ushift
  while (ii < p.n_items - 1 && w >= items[ii].tile_begin + items[ii].n_blocks * (items[ii].h_count >> ushift)) ++ii;
  T.itm = items[ii];
  const int local = w - T.itm.tile_begin;
  int unit;
  if constexpr (kGrouped) {
    const int hg = p.head_group;
    const int per_group = T.itm.n_blocks * hg;
    const int grp = local / per_group;
    const int rem = local - grp * per_group;
    T.blk = T.itm.n_blocks - 1 - rem / hg;
    unit = grp * hg + rem % hg;
  } else {
    const int hu = T.itm.h_count >> ushift;
    T.blk = T.itm.n_blocks - 1 - local / hu;
    unit = local % hu;
  }
  T.h = T.itm.h_begin + (unit << ushift);
  T.g = T.h / p.group;
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    const int r0 = tile_row0<QT>(p, T, t);
    T.geo.rows[t] = max(0, min(kBlockM, T.itm.q_len - r0));
    T.geo.qa[t] = p.q_pos_off + T.itm.q_row0 + r0;
    T.geo.qb[t] = T.geo.qa[t] + T.geo.rows[t] - 1;
  }
  if constexpr (QT == 1) {  // the second slot of the geometry stays unused
    T.geo.rows[1] = 0;
    T.geo.qa[1] = T.geo.qa[0];
    T.geo.qb[1] = T.geo.qb[0];
  }
}

// Loop bounds of a CTA's work tiles: w = blockIdx.x, blockIdx.x + gridDim.x, ... in the fixed
// order; with tiles claimed at run time the loop variable is set inside the loop instead.
template <bool kDynamic>
__device__ __forceinline__ int first_tile() {
  return kDynamic ? 0 : static_cast<int>(blockIdx.x);
}
template <bool kDynamic>
__device__ __forceinline__ int tile_stride() {
  return kDynamic ? 0 : static_cast<int>(gridDim.x);
}

// For a CTA that computes no more tiles of a launch whose tiles are claimed at run time:
// claims until an index past the end comes back, so that each CTA takes exactly one of those
// (total .. total + gridDim.x - 1); the CTA handed the last one is the launch's last claim
// and puts the counter back to 0 for the next launch that uses it.
__device__ __forceinline__ void release_tiles(const AttnParams& p, int total) {
  for (;;) {
    const uint32_t w = atomicAdd(p.tile_counter, 1u);
    if (w >= static_cast<uint32_t>(total)) {
      if (w == static_cast<uint32_t>(total) + gridDim.x - 1) atomicExch(p.tile_counter, 0u);
      return;
    }
  }
}

template <int DQK, int DV, int QT>
__global__ void __launch_bounds__(K1Cfg<DQK, DV, QT>::kThreads, K1Cfg<DQK, DV, QT>::kMinBlocks)
    attn_partial_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ AttnParams p) {
  using C = K1Cfg<DQK, DV, QT>;
  constexpr int kQTiles = C::kQTiles;  // Q tiles of this CTA
  constexpr int kTmaWarp = C::kTmaWarp, kMmaWarp = C::kMmaWarp, kSchedWarp = C::kSchedWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sSlot = smem + kQTiles * C::kQTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* bar_q = bars;
  uint64_t* bar_full = bars + 1;
  uint64_t* bar_empty = bar_full + C::kSlots;
  uint64_t* bar_s = bar_empty + C::kSlots;
  uint64_t* bar_p = bar_s + kQTiles;
  uint64_t* bar_o = bar_p + kQTiles;
  uint64_t* bar_ofree = bar_o + kQTiles;
  uint64_t* bar_qempty = bar_ofree + kQTiles;
  uint64_t* bar_drain = bar_qempty + 1;  // one per MMA issuer
  uint64_t* bar_sfree = bar_drain + kQTiles;  // softmax t has loaded S_t into registers
  uint64_t* bar_turn = bar_sfree + kQTiles;    // [t * 4 + wq]: softmax warp (t, wq) may exponentiate
  uint64_t* bar_tfull = bar_turn + 4 * kQTiles;  // the scheduler published the next work tile
  uint64_t* bar_tfree = bar_tfull + 1;           // every reader has taken it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_turn + 4 * kQTiles + (C::kDynamicTiles ? 2 : 0));
  volatile int* cta_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* sTileIdx = reinterpret_cast<volatile int*>(tmem_slot + 2);  // claimed tile, -1 = none left

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = p.total_tiles;

  // The next attention launch of a decomposition (independent of this one: it reads the same
  // inputs and writes other partial planes) may take each SM this grid leaves, as soon as
  // every CTA of this grid has started.
  pdl_launch_dependents();

  // ---- a CTA scheduled after a timeout elsewhere does nothing
  if (threadIdx.x == 0) *cta_abort = (*reinterpret_cast<volatile int*>(p.status) != 0) ? 1 : 0;
  __syncthreads();
  if (*cta_abort) {
    if (C::kDynamicTiles && threadIdx.x == 0) release_tiles(p, total);
    pdl_wait();
    return;
  }

  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == kMmaWarp * 32) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kQTiles);  // one commit per MMA issuer
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_ofree[t], 4);
    }
    mbar_init(bar_qempty, kQTiles);
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bar_drain[t], 1);
      mbar_init(&bar_sfree[t], 4);  // one arrival per softmax warp
      for (int q = 0; q < 4; ++q) mbar_init(&bar_turn[t * 4 + q], 1);  // lane 0 of the partner warp
    }
    if (C::kDynamicTiles) {
      mbar_init(bar_tfull, 1);
      mbar_init(bar_tfree, C::kTileReaders);
    }
    fence_barrier_init();
  }
  // work items into shared memory: dynamically indexed parameter reads miss the constant cache
  WorkItem* sItems = reinterpret_cast<WorkItem*>(smem + C::kItemsOffset);
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.items);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sItems);
    const int words = p.n_items * static_cast<int>(sizeof(WorkItem) / 4);
    for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
  }
  if (threadIdx.x == kTmaWarp * 32) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint64_t limit = p.wait_limit_ns;

  // The tile loops run w = blockIdx.x, blockIdx.x + gridDim.x, ... (a fixed order), or, with
  // tiles claimed at run time, take_tile() sets w at the top of each pass to the k-th tile the
  // scheduler warp claimed (-1 after the last; false if the wait for it ran out) and the loop
  // header only keeps the loop going.  `warp_wide`: the whole warp calls and lane 0 arrives.
  auto take_tile = [&](int k, int& w, bool warp_wide) -> bool {
    bool ok = wait_bounded(bar_tfull, k & 1, cta_abort, p.status, limit, 17);
    if (warp_wide) ok = warp_all(ok);
    if (!ok) return false;
    w = *sTileIdx;
    if (warp_wide) __syncwarp();
    if (!warp_wide || lane == 0) mbar_arrive(bar_tfree);
    return true;
  };

  if (C::kDynamicTiles && warp == kSchedWarp) {
    // ================================================================ scheduler
    // Claims work tiles one at a time: the next once every role has taken the previous one, so
    // the CTA holds at most the tile it computes and the one it loads.  After the last tile (or
    // once the CTA gave up on a wait) it still claims until it is handed an index past the end,
    // so that every CTA takes exactly one of those and the counter can be put back to 0.
    if (lane == 0) {
      bool live = true;
      for (int k = 0;; ++k) {
        if (live && k > 0 && !wait_bounded(bar_tfree, (k - 1) & 1, cta_abort, p.status, limit, 18)) live = false;
        if (!live) {
          release_tiles(p, total);
          break;
        }
        const uint32_t w = atomicAdd(p.tile_counter, 1u);
        const bool end = w >= static_cast<uint32_t>(total);
        *sTileIdx = end ? -1 : static_cast<int>(w);
        mbar_arrive(bar_tfull);
        if (end) {
          if (w == static_cast<uint32_t>(total) + gridDim.x - 1) atomicExch(p.tile_counter, 0u);
          break;
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // ================================================================ TMA producer
    if (lane == 0) {
      uint32_t cnt = 0;
      int wt = 0;
      bool ok = true;
      int item_hint = 0;
      int k = 0;
      for (int w = first_tile<C::kDynamicTiles>(); w < total; w += tile_stride<C::kDynamicTiles>()) {
        if constexpr (C::kDynamicTiles) {
          if (!take_tile(k++, w, false)) {
            ok = false;
            break;
          }
          if (w < 0) break;
        }
        Tile T;
        decode_tile<C::kGroupedTiles, C::kQTiles>(p, sItems, w, T, item_hint);
        if (!has_steps<kQTiles>(T.itm, p, T.geo)) continue;
        // Q of the previous work tile is in use until its last S MMAs are done
        if (wt > 0 && !wait_bounded(bar_qempty, (wt - 1) & 1, cta_abort, p.status, limit, 11)) {
          ok = false;
          break;
        }
        const int nq = kQTiles == 2 && T.geo.rows[1] > 0 ? 2 : 1;
        mbar_arrive_expect_tx(bar_q, nq * C::kQTileBytes);
        for (int t = 0; t < nq; ++t)
          for (int c = 0; c < C::kQChunks; ++c)
            tma_load_3d(sQ + t * C::kQTileBytes + c * kChunkBytes, &tm_q, bar_q, 64 * c, tile_head(p, T, t),
                        T.itm.q_row0 + tile_row0<C::kQTiles>(p, T, t));
        ++wt;  // Q loads issued
        ok = for_each_step<kQTiles>(T.itm, p, T.geo, [&](const Step& s) -> bool {
          {  // K tile
            const uint32_t slot = cnt % C::kSlots, ph = (cnt / C::kSlots) & 1;
            if (!wait_bounded(&bar_empty[slot], ph ^ 1, cta_abort, p.status, limit, 1)) return false;
            mbar_arrive_expect_tx(&bar_full[slot], C::kKTileBytes);
            for (int c = 0; c < C::kQChunks; ++c)
              tma_load_3d(sSlot + slot * C::kSlotBytes + c * kChunkBytes, &tm_k, &bar_full[slot], 64 * c, T.g,
                          s.krow);
            ++cnt;
          }
          {  // V tile
            const uint32_t slot = cnt % C::kSlots, ph = (cnt / C::kSlots) & 1;
            if (!wait_bounded(&bar_empty[slot], ph ^ 1, cta_abort, p.status, limit, 2)) return false;
            mbar_arrive_expect_tx(&bar_full[slot], C::kVTileBytes);
            for (int c = 0; c < C::kVChunks; ++c)
              tma_load_3d(sSlot + slot * C::kSlotBytes + c * kChunkBytes, &tm_v, &bar_full[slot], 64 * c, T.g,
                          s.krow);
            ++cnt;
          }
          return true;
        });
        if (!ok) break;
      }
      if (!ok) {
        // let the loads already issued land before the CTA gives up its shared memory
        if (wt > 0) wait_final(bar_q, (wt - 1) & 1, limit);
        for (uint32_t s = 0; s < C::kSlots && s < cnt; ++s) {
          const uint32_t last = s + ((cnt - 1 - s) / C::kSlots) * C::kSlots;
          wait_final(&bar_full[s], (last / C::kSlots) & 1, limit);
        }
      }
    }
  } else if (warp == kMmaWarp || (kQTiles == 2 && warp == kMmaWarp + 1)) {
    // ================================================================ MMA issuers
    // One issuing thread per Q tile (warps on different SM sub-partitions), so each
    // tile's MMAs wait only on that tile's softmax.  Per step j issuer t issues
    // S_t(j) = Q_t K(j)^T and then (separate-P layout) O_t += P_t(j-1) V(j-1); with
    // P inside S_t (dv = 128) O_t += P_t(j) V(j) once softmax t has written P_t(j).
    // Every issuer commits once per K/V fill and per work tile (those barriers
    // count one arrival per issuer), whether or not its tile used the step.
    if (lane == 0) {
      const int t = warp - kMmaWarp;
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, DV, 0, 1);
      constexpr uint32_t kDescHi = smem_desc_hi(1024, kSwizzle128B);
      const uint32_t qlo = smem_desc_lo(smem_u32(sQ + t * C::kQTileBytes), 16);
      const uint32_t d_s = tmem + t * kBlockN, d_o = tmem + C::kColO + t * DV, a_p = tmem + C::col_p(t);
      uint32_t cnt = 0;
      int n = 0;    // S MMAs issued for this tile, over all work tiles
      int pvw = 0;  // work tiles whose first PV into O_t has been issued
      // separate-P order: the previous step's V slot and whether this tile used it
      bool pend = false, pend_part = false, pend_first = false;
      uint32_t pend_vslot = 0, pend_vph = 0;
      int pend_k = 0;

      auto issue_qk = [&](uint32_t kslot) {
        const uint32_t klo = smem_desc_lo(smem_u32(sSlot + kslot * C::kSlotBytes), 16);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_lh(d_s, qlo + off, kDescHi, klo + off, kDescHi, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s[t]);
      };
      // The first PV of a work tile overwrites O_t: it waits until the previous work
      // tile's epilogue has read O_t.
      auto issue_pv = [&](uint32_t vslot, bool first) -> bool {
        if (first) {
          if (pvw > 0) {
            if (!wait_bounded(&bar_ofree[t], (pvw - 1) & 1, cta_abort, p.status, limit, 12)) return false;
            tc_fence_after_sync();
          }
          ++pvw;
        }
        const uint32_t vlo = smem_desc_lo(smem_u32(sSlot + vslot * C::kSlotBytes), kChunkBytes);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_lh(d_o, a_p + kk * 8, vlo + ((kk * 2048) >> 4), kDescHi, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bar_o[t]);
        return true;
      };
      // separate-P: PV of the previous step (if this tile used it), then release its V slot
      // (an issuer waits for every fill it releases, used or not, so that it can never
      // commit for a later fill of a slot before the other issuer released the earlier)
      auto flush = [&]() -> bool {
        if (!pend) return true;
        if (!wait_bounded(&bar_full[pend_vslot], pend_vph, cta_abort, p.status, limit, 6)) return false;
        if (pend_part) {
          if (!wait_bounded(&bar_p[t], pend_k & 1, cta_abort, p.status, limit, 7)) return false;
          tc_fence_after_sync();
          if (!issue_pv(pend_vslot, pend_first)) return false;
        }
        mma_commit(&bar_empty[pend_vslot]);
        pend = false;
        return true;
      };

      bool ok = true;
      int wt = 0;
      int item_hint = 0;
      int k = 0;
      for (int w = first_tile<C::kDynamicTiles>(); w < total && ok; w += tile_stride<C::kDynamicTiles>()) {
        if constexpr (C::kDynamicTiles) {
          if (!take_tile(k++, w, false)) {
            ok = false;
            break;
          }
          if (w < 0) break;
        }
        Tile T;
        decode_tile<C::kGroupedTiles, C::kQTiles>(p, sItems, w, T, item_hint);
        if (!has_steps<kQTiles>(T.itm, p, T.geo)) continue;
        if (!wait_bounded(bar_q, wt & 1, cta_abort, p.status, limit, 3)) {
          ok = false;
          break;
        }
        ++wt;
        tc_fence_after_sync();
        bool first = true;  // first PV of this work tile still due
        ok = for_each_step<kQTiles>(T.itm, p, T.geo, [&](const Step& s) -> bool {
          const uint32_t kslot = cnt % C::kSlots, kph = (cnt / C::kSlots) & 1;
          ++cnt;
          const uint32_t vslot = cnt % C::kSlots, vph = (cnt / C::kSlots) & 1;
          ++cnt;
          const bool part = (s.part >> t) & 1;
          if (!wait_bounded(&bar_full[kslot], kph, cta_abort, p.status, limit, 4)) return false;
          if (part) {
            if (n > 0) {
              // separate P: S_t is free as soon as softmax t has loaded it into registers
              // (bar_sfree), so S_t(j) overlaps softmax t's work on step j-1; P inside
              // S_t: once the previous PV has consumed P_t
              uint64_t* b = C::kSepP ? &bar_sfree[t] : &bar_o[t];
              if (!wait_bounded(b, (n - 1) & 1, cta_abort, p.status, limit, 5)) return false;
            }
            tc_fence_after_sync();
            issue_qk(kslot);
          }
          mma_commit(&bar_empty[kslot]);
          if (C::kSepP) {
            if (!flush()) return false;
            pend = true;
            pend_part = part;
            pend_first = part && first;
            pend_vslot = vslot;
            pend_vph = vph;
            pend_k = n;
            if (part) {
              first = false;
              ++n;
            }
          } else {
            if (!wait_bounded(&bar_full[vslot], vph, cta_abort, p.status, limit, 6)) return false;
            if (part) {
              if (!wait_bounded(&bar_p[t], n & 1, cta_abort, p.status, limit, 7)) return false;
              tc_fence_after_sync();
              if (!issue_pv(vslot, first)) return false;
              first = false;
              ++n;
            }
            mma_commit(&bar_empty[vslot]);
          }
          return true;
        });
        // this issuer's S MMAs of the work tile are issued: Q may be reloaded once done
        mma_commit(bar_qempty);
        // the tile's last PV goes out now, not behind the next tile's first S MMA (which
        // waits for the next Q load): the epilogue waits for that PV
        if (ok && C::kSepP) ok = flush();
      }
      if (ok) flush();
      // every MMA of this issuer (and the arrivals its commits make) completes before teardown
      mma_commit(&bar_drain[t]);
      wait_final(&bar_drain[t], 0, limit);
    }
  } else if (warp < kTmaWarp) {
    // ================================================================ softmax + epilogue
    const int t = kQTiles == 2 ? warp >> 2 : 0;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * kBlockN;
    const uint32_t tP = tmem + lane_base + C::col_p(t);
    const uint32_t tO = tmem + lane_base + C::kColO + t * DV;
    uint8_t* const sStage = smem + C::kStageOffset + warp * (C::kStageBufs * 4096);  // this warp's boxes
    // Where C::kTurns holds, the softmax warps of the two Q tiles that share an SM
    // sub-partition (same wq) take turns on their exponentials, which the sub-partition's
    // MUFU unit bounds: one warp
    // exponentiates alone while the other loads S, stores P and waits for the MMAs.
    // Turn k of tile 0 waits for tile 1's turn k-1, turn k of tile 1 for tile 0's turn k.
    // Both take one turn per step of whichever tile has more steps in the work tile; the
    // tile with fewer steps passes its extra turns without work, so the turns stay paired.
    int turn = 0;
    auto take_turn = [&]() -> bool {
      if (t == 0 && turn == 0) return true;
      const uint32_t par = static_cast<uint32_t>(t == 0 ? turn - 1 : turn) & 1u;
      return warp_all(wait_bounded(&bar_turn[t * 4 + wq], par, cta_abort, p.status, limit, 13));
    };
    auto pass_turn = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_turn[(t ^ 1) * 4 + wq]);
      ++turn;
    };
    const float sl2 = p.scale_log2;
    int n = 0;  // steps (= PVs) of this Q tile over all work tiles
    bool ok = true;
    int item_hint = 0;
    int k = 0;
    for (int w = first_tile<C::kDynamicTiles>(); w < total && ok; w += tile_stride<C::kDynamicTiles>()) {
      if constexpr (C::kDynamicTiles) {
        if (!take_tile(k++, w, true)) {
          ok = false;
          break;
        }
        if (w < 0) break;
      }
      Tile T;
      decode_tile<C::kGroupedTiles, C::kQTiles>(p, sItems, w, T, item_hint);
      const int rows_t = t == 0 ? T.geo.rows[0] : T.geo.rows[1];
      // turns of this work tile: the step count of the tile with more steps
      int n_turns = 0;
      if (C::kTurns) {
        int cnt[2] = {0, 0};
#pragma unroll
        for (int u = 0; u < kQTiles; ++u) {
          if (T.geo.rows[u] <= 0) continue;
          for (int r = 0; r < T.itm.n_kv; ++r) {
            const TileRange R = tile_range(r == 0 ? T.itm.kv[0].row0 : T.itm.kv[1].row0,
                                           r == 0 ? T.itm.kv[0].len : T.itm.kv[1].len, T.geo.qa[u], T.geo.qb[u], p);
            cnt[u] += max(0, R.hi - R.lo + 1);
          }
        }
        n_turns = max(cnt[0], cnt[1]);
      }
      int taken = 0;  // turns taken in this work tile
      if (rows_t <= 0) {
        if constexpr (C::kTurns) {
          for (; taken < n_turns && ok; ++taken) {
            ok = take_turn();
            if (ok) pass_turn();
          }
        }
        continue;
      }
      const int q_pos = (t == 0 ? T.geo.qa[0] : T.geo.qa[1]) + row;
      float m_used = -INFINITY;  // running max in log2-scaled units
      float l = 0.f;             // running sum of exp2(s*sl2 - m_used)
      int nl = 0;                // steps of this work tile
      const int qa_t = t == 0 ? T.geo.qa[0] : T.geo.qa[1];
      const int qb_t = qa_t + rows_t - 1;
      auto step = [&](const bool full, const int kpos, const int valid) -> bool {
        if (!warp_all(wait_bounded(&bar_s[t], n & 1, cta_abort, p.status, limit, 8))) return false;
        tc_fence_after_sync();
        // S_t with the maximum of each 32-column quarter of the row (taken by the load)
        uint32_t r0[32], r1[32], r2[32], r3[32];
        float q0 = tmem_ld32_max(tS + 0, r0);
        float q1 = tmem_ld32_max(tS + 32, r1);
        float q2 = tmem_ld32_max(tS + 64, r2);
        float q3 = tmem_ld32_max(tS + 96, r3);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        reg_fence(r2);
        reg_fence(r3);
        reg_fence(q0);
        reg_fence(q1);
        reg_fence(q2);
        reg_fence(q3);
        float sv[128];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(r0[i]);
          sv[32 + i] = __uint_as_float(r1[i]);
          sv[64 + i] = __uint_as_float(r2[i]);
          sv[96 + i] = __uint_as_float(r3[i]);
        }
        float mx = fmax3(q0, q1, fmaxf(q2, q3));  // row max of a fully visible tile
        if (!full) {
          // the row's visible columns of this tile form one interval [lo, hi]: c < valid,
          // causal kpos + c <= q_pos, window q_pos - (kpos + c) < window
          int lo = p.window > 0 ? max(0, q_pos - kpos - p.window + 1) : 0;
          int hi = p.causal ? min(valid - 1, q_pos - kpos) : valid - 1;
          if (hi < lo) lo = hi = kBlockN;  // nothing visible: every c - lo is negative
          const uint32_t span = static_cast<uint32_t>(hi - lo);
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (static_cast<uint32_t>(c - lo) > span) sv[c] = -INFINITY;
          // row max over the visible scores, per 32-column quarter: a quarter wholly visible
          // to this lane keeps the load's maximum, a hidden one gives -inf; only a quarter
          // that some lane of the warp sees in part takes a max over the masked scores
          float qm[4] = {q0, q1, q2, q3};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool all_vis = lo <= 32 * j && 32 * j + 31 <= hi;
            const bool none_vis = hi < 32 * j || lo > 32 * j + 31;
            if (__any_sync(0xffffffffu, !all_vis && !none_vis)) {
              float a = fmax3(sv[32 * j], sv[32 * j + 1], sv[32 * j + 2]);
              float b = fmax3(sv[32 * j + 3], sv[32 * j + 4], sv[32 * j + 5]);
#pragma unroll
              for (int i = 6; i < 30; i += 4) {
                a = fmax3(a, sv[32 * j + i], sv[32 * j + i + 1]);
                b = fmax3(b, sv[32 * j + i + 2], sv[32 * j + i + 3]);
              }
              qm[j] = fmax3(a, b, fmaxf(sv[32 * j + 30], sv[32 * j + 31]));
            } else {
              qm[j] = all_vis ? qm[j] : -INFINITY;
            }
          }
          mx = fmax3(qm[0], qm[1], fmaxf(qm[2], qm[3]));
        }
        const float m_new = mx * sl2;
        const bool need = m_new > m_used + kRescaleThreshold;
        // per-lane update without a branch; the warp-wide vote (needed only for the O
        // rescale after the exponentials) stays off the path to the exponentials
        const float alpha = need ? ex2_approx(m_used - m_new) : 1.f;
        m_used = need ? m_new : m_used;
        l *= alpha;
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // p = exp2(s * sl2 - m), packed to bf16 pairs; row sum in fp32 (four packed chains)
        if constexpr (C::kTurns) {
          if (!take_turn()) return false;
        }
        const uint64_t sl2v = pack_f32x2(sl2, sl2), negm = pack_f32x2(-msub, -msub);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[64];
        const Exp2Poly poly = exp2_poly_consts();
        // P is stored in 16-column chunks while later pairs are still being exponentiated.
        // Over S_t (dv = 128) each chunk goes out when done; in its own columns (dv = 64) the
        // previous PV must have read P first, which it has by three quarters of the loop.
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          pk[i] = (i & 15) < kPolyPairsPer16
                      ? softmax_pair_poly(sv[2 * i], sv[2 * i + 1], sl2v, negm, acc[i & 3], poly)
                      : softmax_pair(sv[2 * i], sv[2 * i + 1], sl2v, negm, acc[i & 3]);
          if (C::kSepP && i == 15) {  // S_t is in registers: the next S MMA of this tile may overwrite it
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_sfree[t]);
          }
          if ((i & 15) == 15) {
            const int c = i >> 4;  // chunk c of P is complete
            if constexpr (!C::kSepP) {
              tmem_st16(tP + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * c]));
            } else if (c == 2) {
              if (n > 0) {
                if (!warp_all(wait_bounded(&bar_o[t], (n - 1) & 1, cta_abort, p.status, limit, 9))) return false;
                tc_fence_after_sync();
              }
#pragma unroll
              for (int cc = 0; cc < 3; ++cc)
                tmem_st16(tP + cc * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * cc]));
            } else if (c == 3) {
              tmem_st16(tP + 48, *reinterpret_cast<const uint32_t(*)[16]>(&pk[48]));
            }
          }
        }
        const float2 c0 = unpack_f32x2(acc[0]), c1 = unpack_f32x2(acc[1]);
        const float2 c2 = unpack_f32x2(acc[2]), c3 = unpack_f32x2(acc[3]);
        l += ((c0.x + c0.y) + (c1.x + c1.y)) + ((c2.x + c2.y) + (c3.x + c3.y));
        if constexpr (C::kTurns) {
          pass_turn();
          ++taken;
        }
        const bool any_need = __any_sync(0xffffffffu, need);
        // O_t holds the previous PV's result here.  Separate P: the P store above waited for
        // that PV.  P inside S_t: the issuer sent S_t(n) only after PV(n-1) completed, and the
        // commit behind bar_s tracks every earlier MMA of that issuer.
        if (any_need && nl > 0) {
#pragma unroll 1
          for (int c = 0; c < DV / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_ld_wait();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + c * 16, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p[t]);
        ++n;
        ++nl;
        return true;
      };
      // the item's fields are read from shared memory where they are used, rather than kept in
      // registers across the steps, which need every register they can get
      const WorkItem& sit = sItems[item_hint];
      for (int r = 0; r < sit.n_kv && ok; ++r) {
        const KvRange kr = sit.kv[r];
        const TileRange R = tile_range(kr.row0, kr.len, qa_t, qb_t, p);
        for (int j = R.lo; j <= R.hi && ok; ++j)
          ok = step(j >= R.flo && j <= R.fhi, R.kpos0 + j * kBlockN, min(kBlockN, R.len - j * kBlockN));
      }
      // the other tile's extra steps: pass the turns before this tile's epilogue
      if constexpr (C::kTurns) {
        for (; taken < n_turns && ok; ++taken) {
          ok = take_turn();
          if (ok) pass_turn();
        }
      }
      if (!ok) break;

      // ---- epilogue: out = O / l, lse = ln(sum exp(scaled scores))
      // What does not depend on O (the row's 1/l, its lse, the output address) is done before
      // the wait for the tile's last PV.
      const bool valid_row = row < rows_t;
      const int head = tile_head(p, T, t);
      const int64_t orow = static_cast<int64_t>(sit.out_row0) + tile_row0<C::kQTiles>(p, T, t) + row;
      const int64_t plane = sit.plane;
      if (valid_row) {
        p.lse[plane * p.lse_splane + orow * p.lse_srow + static_cast<int64_t>(head) * p.lse_shead] =
            l > 0.f ? (m_used + lg2_approx(l)) * kLn2 : -INFINITY;
      }
      // a row that saw no key keeps m = -inf; its l holds only the clamped 2^-125
      // terms of the polynomial pairs, and its output is 0
      const float inv = (l > 0.f && m_used > -INFINITY) ? 1.f / l : 0.f;
      float* op = p.out + plane * p.out_splane + orow * p.out_srow + static_cast<int64_t>(head) * p.out_shead;
      // A warp whose 32 rows are all valid writes O through shared memory and TMA stores
      // (one 32 x 32 box per 32 columns): each thread's row lies a whole output row apart
      // from its neighbour's, so direct stores would touch 32 cache lines per instruction.
      const bool via_tma = p.out_tma && __all_sync(0xffffffffu, valid_row);
      if (nl > 0) ok = warp_all(wait_bounded(&bar_o[t], (n - 1) & 1, cta_abort, p.status, limit, 10));
      if (!ok) break;
      if (nl > 0) {
        tc_fence_after_sync();
        if (p.out_bf16) {
          // bf16 output: two 32-column TMEM loads fill one 64-column (128-byte) box row
          __nv_bfloat16* bp = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              (plane * p.out_splane + orow * p.out_srow + static_cast<int64_t>(head) * p.out_shead);
#pragma unroll
          for (int g = 0; g < DV / 64; ++g) {
            uint32_t wv[32];
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const int c = 2 * g + hlf;
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
              reg_fence(o);
              if (c == DV / 32 - 1) {  // O_t is read: the next work tile's first PV may overwrite it
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_ofree[t]);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i)
                wv[16 * hlf + i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            }
            if (via_tma) {
              uint8_t* const box = sStage + (g % C::kStageBufs) * 4096;
              if (lane == 0) {
                if (C::kStageBufs == 2)
                  bulk_wait_read_allbut1();
                else
                  bulk_wait_read_all();
              }
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<uint4*>(box + lane * 128 + ((i ^ (lane & 7)) * 16)) =
                    make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
              fence_proxy_async_shared();
              __syncwarp();
              if (lane == 0) {
                const int64_t z = plane * p.out_plane_rows + orow;  // row of lane 0
                tma_store_3d(&tm_o, box, 64 * g, head, static_cast<int>(z));
                bulk_commit();
              }
            } else if (valid_row) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<uint4*>(bp + 64 * g + 8 * i) =
                    make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
            }
          }
        } else {
          // fp32 output, as many 32-column chunks at a time as there are staging boxes: each is
          // loaded from TMEM and written to its box in turn, and the group's boxes then share one
          // proxy fence and one bulk group of TMA stores
          constexpr int kG = C::kStageBufs;
          static_assert((DV / 32) % kG == 0, "whole groups of chunks");
#pragma unroll
          for (int c0 = 0; c0 < DV / 32; c0 += kG) {
            if (via_tma) {
              // the stores that last used these boxes have read them
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll
            for (int b = 0; b < kG; ++b) {
              const int c = c0 + b;
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
              reg_fence(o);
              if (c == DV / 32 - 1) {  // O_t is read: the next work tile's first PV may overwrite it
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_ofree[t]);
              }
              if (via_tma) {
                // row `lane` of the box: 16-byte chunk i at chunk position i ^ (lane & 7) (128-byte swizzle)
                uint8_t* const box = sStage + b * 4096;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 v = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                               __uint_as_float(o[4 * i + 2]) * inv,
                                               __uint_as_float(o[4 * i + 3]) * inv);
                  *reinterpret_cast<float4*>(box + lane * 128 + ((i ^ (lane & 7)) * 16)) = v;
                }
              } else if (valid_row) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 v = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                               __uint_as_float(o[4 * i + 2]) * inv,
                                               __uint_as_float(o[4 * i + 3]) * inv);
                  *reinterpret_cast<float4*>(op + c * 32 + 4 * i) = v;
                }
              }
            }
            if (via_tma) {
              fence_proxy_async_shared();
              __syncwarp();
              if (lane == 0) {
                const int64_t z = plane * p.out_plane_rows + orow;  // row of lane 0
#pragma unroll
                for (int b = 0; b < kG; ++b)
                  tma_store_3d(&tm_o, sStage + b * 4096, 32 * (c0 + b), head, static_cast<int>(z));
                bulk_commit();
              }
            }
          }
        }
      } else if (p.write_empty_out && valid_row) {
        if (p.out_bf16) {
          __nv_bfloat16* bp = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              (plane * p.out_splane + orow * p.out_srow + static_cast<int64_t>(head) * p.out_shead);
#pragma unroll
          for (int i = 0; i < DV / 8; ++i) *reinterpret_cast<uint4*>(bp + 8 * i) = make_uint4(0u, 0u, 0u, 0u);
        } else {
#pragma unroll
          for (int i = 0; i < DV / 4; ++i) *reinterpret_cast<float4*>(op + 4 * i) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    // the O stores of this warp complete before the CTA releases its shared memory
    if (lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // Launched as a dependent of the previous attention launch, this grid finishes only after
  // that one has: a kernel queued after the last launch (the merge) then sees every launch's
  // partials.
  pdl_wait();
}

// CTAs per launch: one persistent CTA per SM (each holds the SM's whole TMEM),
// or fewer when there are fewer work tiles.
int resident_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 1;
  return sms;
}

int gcd_int(int a, int b) {
  while (b != 0) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Head units (heads, or head pairs with pair_heads) per tile group.  With every unit of an
// item inner to its row blocks, the resident CTAs work on about grid / units row blocks at a
// time.  When a KV head serves few query heads (Hq / Hkv < 4, as in MLA-shaped attention),
// that is about one CTA per KV head, so each CTA streams its own K/V tiles from DRAM.  A group
// of units just large enough to give the grid one group's row blocks puts many CTAs on the
// same heads, and they then share those heads' K/V tiles in L2.  With tiles claimed at run
// time the CTAs in flight hold about one grid's width of consecutive tiles whatever the group,
// and groups of one unit (an item's tiles head by head) put the fewest heads in that window.
// With larger GQA groups the query heads of a KV head already share its tiles, and one group
// of all the units is kept.
int tile_head_group(const AttnParams& p, long long grid, bool dynamic_tiles) {
  int common = 0, max_blocks = 1;
  for (int i = 0; i < p.n_items; ++i) {
    common = gcd_int(common, p.items[i].h_count >> p.pair_heads);
    max_blocks = std::max(max_blocks, static_cast<int>(p.items[i].n_blocks));
  }
  if (common <= 0) return 1;
  if (p.group >= 4) return common;
  if (dynamic_tiles) return 1;
  const long long want = (grid + max_blocks - 1) / max_blocks;
  for (int hg = 1; hg < common; ++hg)
    if (common % hg == 0 && hg >= want) return hg;
  return common;
}

template <int DQK, int DV, int QT = 2>
cudaError_t launch_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                        AttnParams p, bool dependent, cudaStream_t stream) {
  using C = K1Cfg<DQK, DV, QT>;
  if (p.n_items <= 0) return cudaSuccess;
  long long tiles;
  if constexpr (QT == 1) {
    // one Q tile per CTA: work tiles of 128 rows of one head, counted here (the plan counts
    // them for two Q tiles)
    p.pair_heads = 0;
    tiles = 0;
    for (int i = 0; i < p.n_items; ++i) {
      WorkItem& it = p.items[i];
      it.n_blocks = (it.q_len + kBlockM - 1) / kBlockM;
      if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      it.tile_begin = static_cast<int32_t>(tiles);
      tiles += static_cast<long long>(it.n_blocks) * it.h_count;
    }
  } else {
    const WorkItem& last = p.items[p.n_items - 1];
    tiles = static_cast<long long>(last.tile_begin) +
            static_cast<long long>(last.n_blocks) * (last.h_count >> p.pair_heads);
  }
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.total_tiles = static_cast<int32_t>(tiles);
  const long long grid = std::min<long long>(tiles, resident_ctas() * C::kMinBlocks);
  p.head_group = C::kGroupedTiles ? tile_head_group(p, grid, C::kDynamicTiles) : 0;
  if (C::kDynamicTiles) {
    p.tile_counter = claim_tile_counter();
    if (p.tile_counter == nullptr) return cudaErrorInvalidDevice;
  }
  cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<DQK, DV, QT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if constexpr (QT == 1) {  // the whole shared-memory carve-out, so that two CTAs fit on an SM
    e = cudaFuncSetAttribute(attn_partial_kernel<DQK, DV, QT>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_partial_kernel<DQK, DV, QT>, tq, tk, tv, to, p);
}

}  // namespace

// (dqk, dv) in {64, 128, 192} x {64, 128}.  dv = 192 is not built: the two Q tiles' O
// accumulators (2 x 192 TMEM columns) and their S tiles (2 x 128) would need 640 of the 512
// columns of an SM's tensor memory.
bool attn_partial_supported(int dqk, int dv) {
  return (dqk == 64 || dqk == 128 || dqk == 192) && (dv == 64 || dv == 128);
}

// Windows up to this many keys run with two Q tiles per CTA at d = 64 (see launch_attn_partial).
constexpr int kTwoTileMaxWindow = 4096;

cudaError_t launch_attn_partial(int dqk, int dv, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const AttnParams& p, bool dependent, cudaStream_t stream) {
  if (dqk == 64 && dv == 64) {
    // one Q tile per CTA and two CTAs per SM, except with a sliding window of up to 4096 keys, whose
    // short work tiles run faster two to a CTA.  Measured: the causal 32K zigzag-8 ring +2.7%, the
    // 32K single launch +7.2%, the 100K zigzag-16 ring +1.8%; the 100K window-128 ring -22%; on the
    // 32K ring with windows of 128 .. 4096 keys the two-tile kernel leads by 28% .. 1%, at 8192 the
    // one-tile kernel by 1%.
    if (p.window > 0 && p.window <= kTwoTileMaxWindow)
      return launch_impl<64, 64, 2>(tq, tk, tv, to, p, dependent, stream);
    return launch_impl<64, 64, 1>(tq, tk, tv, to, p, dependent, stream);
  }
  if (dqk == 64 && dv == 128) return launch_impl<64, 128>(tq, tk, tv, to, p, dependent, stream);
  if (dqk == 128 && dv == 64) return launch_impl<128, 64>(tq, tk, tv, to, p, dependent, stream);
  if (dqk == 128 && dv == 128) return launch_impl<128, 128>(tq, tk, tv, to, p, dependent, stream);
  if (dqk == 192 && dv == 64) return launch_impl<192, 64>(tq, tk, tv, to, p, dependent, stream);
  if (dqk == 192 && dv == 128) return launch_impl<192, 128>(tq, tk, tv, to, p, dependent, stream);
  return cudaErrorInvalidValue;
}

}  // namespace slope
