/*
 * slope.h - C ABI of libslope: context-parallel causal GQA prefill attention
 * on one GB300 (sm_103a).
 *
 * The method: the SLOPE prefill engine (Moreh, "Optimizing long-context
 * prefill on multiple older-generation GPU nodes", section "Introduction to
 * Context Parallelism") splits a prompt along the sequence dimension; every op
 * but attention is per-token, and attention is computed by Ring Attention:
 * each device attends its share of the queries to the key/value block it
 * currently holds while key/value blocks circulate between neighbours.  The
 * SGLang pipeline-parallelism article ("SGLang Pipeline Parallelism: 1M-token
 * context ...", TL;DR) processes long prompts as chunked prefill with
 * 12K-token chunks, each chunk attending to the growing key/value prefix.
 *
 * This library computes exactly that attention on one GPU: the ring's steps
 * (or the chunks) run in order, each step emitting a partial output plus its
 * log-sum-exp, and the partials are combined by an exact log-sum-exp merge.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are described by slope_tensor: a DEVICE pointer, a dtype, a rank
 *    and shape/stride in ELEMENTS.  The innermost stride must be 1.
 *  - Q is [Sq, Hq, dqk], K is [Skv, Hkv, dqk], V is [Skv, Hkv, dv], all bf16,
 *    token-major (batch 1).  Row and head strides of Q/K/V must be multiples
 *    of 8 elements (16 bytes) and the data pointer 16-byte aligned, because
 *    the kernels read them with the Tensor Memory Accelerator.
 *  - Supported head sizes: dqk in {64, 128, 192} with dv in {64, 128}; other
 *    pairs return SLOPE_ERR_UNSUPPORTED.  dv = 192 is refused because the
 *    attention kernel keeps two 128-row query tiles per SM, each with a 128-
 *    column score tile and a dv-column output accumulator in tensor memory:
 *    2 x (128 + 192) = 640 columns, more than the 512 an SM has.  The merge
 *    alone (slope_lse_merge) takes dv in {64, 128, 192}.  Hq must be a
 *    multiple of Hkv; query head h reads key/value head h / (Hq / Hkv).
 *  - Masks use GLOBAL token positions: key j is visible to query i iff
 *    (!causal || pos(j) <= pos(i)) && (window == 0 || pos(i) - pos(j) < window).
 *  - scale <= 0 selects 1/sqrt(dqk).  lse is the natural log of the sum of
 *    exp(scale * q.k) over the visible keys.  A query row that sees no key
 *    gets out = 0 and lse = -inf (never NaN).
 *  - The library never allocates or frees device memory; the caller owns
 *    every buffer, including the workspace.  Host arrays passed in are read
 *    during the call only.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and does not synchronise.  Argument errors are returned
 *    before anything is launched and leave the outputs untouched; a failed
 *    launch returns SLOPE_ERR_CUDA.  Kernel waits are bounded: a wait that
 *    runs out records SLOPE_ERR_TIMEOUT in a device status word that
 *    slope_device_status() reports.
 *  - Calls are thread-safe (no mutable library state besides the device
 *    status word, the work-tile counters below and a lazily resolved driver
 *    entry point).
 *  - Attention launches with dqk >= 128 (the MLA-shaped heads) claim their
 *    work tiles at run time from a counter in static device memory, one of
 *    SLOPE_TILE_COUNTERS per device handed out round robin, which every
 *    launch leaves at 0 (also one whose CTAs found the status word set).
 *    Launches on one stream never share one; across streams, keep fewer
 *    than SLOPE_TILE_COUNTERS such launches queued or running at a time.
 *    A launch recorded into a CUDA graph keeps the counter it was given for
 *    every replay, so replays of one such graph must not overlap.
 */
#define SLOPE_TILE_COUNTERS 4096
#ifndef SLOPE_H
#define SLOPE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SLOPE_API __attribute__((visibility("default")))
#else
#define SLOPE_API
#endif

typedef enum {
  SLOPE_OK = 0,
  SLOPE_ERR_NULL = -1,        /* a required pointer is NULL                         */
  SLOPE_ERR_DTYPE = -2,       /* wrong element type                                 */
  SLOPE_ERR_SHAPE = -3,       /* inconsistent or unsupported shape                  */
  SLOPE_ERR_STRIDE = -4,      /* innermost stride != 1, or misaligned stride/pointer */
  SLOPE_ERR_LAYOUT = -5,      /* layout/chunking does not divide the sequence        */
  SLOPE_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed                   */
  SLOPE_ERR_TIMEOUT = -7,     /* a bounded device wait ran out                       */
  SLOPE_ERR_UNSUPPORTED = -8, /* valid request outside what the kernels implement    */
  SLOPE_ERR_WORKSPACE = -9    /* workspace missing, too small or misaligned          */
} slope_status;

typedef enum { SLOPE_BF16 = 0, SLOPE_F32 = 1 } slope_dtype;

typedef struct {
  void* data;        /* device pointer                                */
  slope_dtype dtype; /* element type                                  */
  int32_t ndim;      /* 2 or 3                                        */
  int64_t shape[3];  /* sizes, outermost first                        */
  int64_t stride[3]; /* strides in elements; stride[ndim-1] must be 1 */
} slope_tensor;

typedef enum {
  SLOPE_LAYOUT_CONTIGUOUS = 0, /* ring of n ranks, rank r owns tokens [r*S/n, (r+1)*S/n)          */
  SLOPE_LAYOUT_ZIGZAG = 1,     /* ring of n ranks, rank r owns sub-chunks r and 2n-1-r of S/(2n)  */
  SLOPE_LAYOUT_CHUNKED = 2,    /* chunked prefill: chunk c attends to all earlier tokens + itself */
  SLOPE_LAYOUT_ULYSSES = 3,    /* n ranks, rank u owns every token of query-head group u of n     */
  /* Not a layout: widens the enum's range to 16 bits, so that a layout word carrying a Ulysses
   * degree (SLOPE_ULYSSES_DEGREE below) is a valid value of this type in C++ as well as in C. */
  SLOPE_LAYOUT_WORD_MAX_ = 0xffff
} slope_layout;

/*
 * Ulysses x Ring: a layout word may carry a Ulysses degree u in bits 8-15 on top of
 * SLOPE_LAYOUT_CONTIGUOUS, SLOPE_LAYOUT_ZIGZAG or SLOPE_LAYOUT_CHUNKED, e.g.
 * SLOPE_LAYOUT_ZIGZAG | SLOPE_ULYSSES_DEGREE(4) (0 or 1: none).  The Moreh post
 * ("Introduction to Context Parallelism") combines the two schemes: after the
 * all-to-all each of u groups holds every token of its query-head group, and the
 * ring (or the chunks) runs within each group.  Every ring step's (or chunk's)
 * partial is then computed as u head-group items that write the same partial
 * planes, so the result equals the layout without the degree.  u must divide Hkv
 * (else SLOPE_ERR_LAYOUT), 2 <= u <= 32, and SLOPE_LAYOUT_ULYSSES takes none.
 */
#define SLOPE_ULYSSES_DEGREE(u) ((slope_layout)(((unsigned)(u) & 0xffu) << 8))

/*
 * Partial attention of one query block against one key/value block
 * (Ring Attention item: a device attends its partial queries to the partial
 * keys/values it holds).
 *
 *   q   bf16 [Sq, Hq, dqk]    k bf16 [Skv, Hkv, dqk]    v bf16 [Skv, Hkv, dv]
 *   q_off / kv_off: global positions of q row 0 / k row 0 (the masks use them).
 *       Every position must lie in [-2^28, 2^28]: q_off >= -2^28, q_off + Sq <= 2^28,
 *       and the same for kv_off and Skv (else SLOPE_ERR_SHAPE), because the kernel
 *       takes differences of a query and a key position, less the window, in 32-bit
 *       integers.
 *   causal, window, scale: see the conventions above.
 *   out fp32 or bf16 [Sq, Hq, dv]: the softmax-normalised output over the
 *       visible keys of this block (0 for rows that see none).  Innermost
 *       stride 1, pointer 16-byte aligned; row and head strides multiples of
 *       4 elements (fp32) or 8 elements (bf16).  With q, k and v covering the
 *       whole sequence (q_off = kv_off = 0) and bf16 out, this one launch is
 *       the whole attention: every query tile runs the online softmax over
 *       all of its visible keys, with no partials and no merge (the fused
 *       single-GPU form of the ring).
 *   lse fp32, rank 2 [Hq, Sq] (any strides): natural-log log-sum-exp of the
 *       scaled scores over the visible keys of this block (-inf if none).
 * Sq == 0 is a no-op.  Returns SLOPE_OK or an error status.
 */
SLOPE_API slope_status slope_attn_partial(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                int64_t q_off, int64_t kv_off, int causal, int64_t window, float scale,
                                slope_tensor* out, slope_tensor* lse, void* stream);

/*
 * Exact log-sum-exp merge of n partials computed over disjoint key sets
 * (the combination step of Ring Attention):
 *   L   = log sum_k exp(lse_k)            (max-shifted; all -inf gives -inf)
 *   out = sum_k exp(lse_k - L) * out_k     (partials with lse_k = -inf are skipped)
 *
 *   outs[k] fp32 or bf16 [S, H, dv], dv in {64, 128, 192}, all of one dtype (else SLOPE_ERR_DTYPE);
 *        lses[k] fp32 rank 2 [H, S] (any strides), 1 <= n <= 32.  bf16 partials
 *        are widened to fp32 as they are read; the sums run in fp32 either way.
 *   out: bf16 or fp32 [S, H, dv] (innermost stride 1, row/head strides multiples
 *        of 4 elements; pointers 16-byte aligned for fp32, 8-byte for bf16, for
 *        out and every outs[k]).
 *   lse: fp32 [H, S], or NULL to skip writing it.
 * `outs` and `lses` are host arrays of n descriptors.
 */
SLOPE_API slope_status slope_lse_merge(const slope_tensor* outs, const slope_tensor* lses, int n, slope_tensor* out,
                             slope_tensor* lse, void* stream);

/*
 * Whole context-parallel prefill attention of one layer on one GPU.
 *
 *   q bf16 [S, Hq, dqk], k bf16 [S, Hkv, dqk], v bf16 [S, Hkv, dv] (positions 0..S-1).
 *   layout SLOPE_LAYOUT_CONTIGUOUS / SLOPE_LAYOUT_ZIGZAG: a ring of n_chunks
 *     simulated ranks.  At ring step t rank r holds the keys/values of rank
 *     (r - t) mod n_chunks; every step computes one partial per (rank, step),
 *     and a final merge launch combines each row's partials.  Steps run in
 *     order, consecutive steps sharing an attention-kernel launch up to 32
 *     work items (two per rank and step in ZIGZAG, one in CONTIGUOUS); each
 *     partial is the same as in a launch of its own.  A step in which no query
 *     sees any key (possible only with a window) is skipped, and so is its
 *     partial in the merge.  CONTIGUOUS needs S % n_chunks == 0,
 *     ZIGZAG needs S % (2*n_chunks) == 0.  1 <= n_chunks <= 32.
 *   layout SLOPE_LAYOUT_CHUNKED: n_chunks query chunks, sizes chunk_sizes[0..n)
 *     (summing to S), or NULL for ceil(S/n_chunks) with a shorter last chunk.
 *     Chunk [s, e) yields two partials - against keys [0, s) and, causally,
 *     against [s, e) - computed chunk by chunk, in order (consecutive chunks
 *     sharing a launch up to 32 work items), then merged.
 *   layout SLOPE_LAYOUT_ULYSSES: the head-sharded scheme (Moreh, section
 *     "Introduction to Context Parallelism": an all-to-all hands each device
 *     all tokens of a subset of the heads).  Rank u of n_chunks holds query
 *     heads [u*Hq/n, (u+1)*Hq/n) and key/value heads [u*Hkv/n, (u+1)*Hkv/n) of
 *     every token and computes their whole attention; there are no partials
 *     and no merge: the ranks' items (one each, consecutive ranks sharing a
 *     launch up to 32) write out and lse directly.  Hkv % n_chunks == 0 (GQA
 *     limits the Ulysses degree to the number of key/value heads, as the page
 *     notes), else SLOPE_ERR_LAYOUT; 1 <= n_chunks <= 32.  A bf16 out then
 *     needs row/head strides that are multiples of 8 elements and a 16-byte
 *     aligned pointer.
 *   causal, window, scale: as above.  out: bf16 or fp32 [S, Hq, dv];
 *   lse: fp32 [Hq, S] or NULL.
 *   workspace: device buffer of at least slope_cp_prefill_workspace_size()
 *     bytes, 256-byte aligned; it holds the fp32 partials between the
 *     attention launches and the merge (for ULYSSES only an lse plane, used
 *     when lse is NULL).
 */
SLOPE_API slope_status slope_cp_prefill(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v, int n_chunks,
                              slope_layout layout, const int64_t* chunk_sizes, int causal, int64_t window,
                              float scale, slope_tensor* out, slope_tensor* lse, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * slope_cp_prefill for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call; it exists for users of this library.
 *
 * Some callers cannot call cudaMalloc: code that runs inside a fixed memory
 * budget reserved up front (a serving process whose device memory is all
 * handed to its own pools), or code on a latency-critical path where an
 * allocation would synchronise the device.  This variant takes no workspace:
 * the fp32 partials live in a fixed scratch array of 64 MiB (67108864 bytes)
 * that the library holds on every GPU that loads it, until the process exits.
 *
 * Same arguments and results as slope_cp_prefill, without workspace and
 * workspace_bytes.  A request whose partials need more than 64 MiB (see
 * slope_cp_prefill_workspace_size) returns SLOPE_ERR_WORKSPACE, before any
 * launch, with the sizes in slope_last_error().  The call allocates nothing
 * and calls no allocating routine.
 *
 * The first call on a device looks up the scratch array's device address
 * (with that device current) and keeps it; make that first call before any
 * stream capture.  The 64 MiB are committed on a device when the library's
 * module is loaded there; with CUDA's lazy module loading (the default since
 * CUDA 12.2) that happens at that first call.  A caller that reserves the rest
 * of the device memory for its own pools should therefore make the first call
 * before reserving them, or the first call may fail with SLOPE_ERR_CUDA (out of
 * memory).  Every call on a device shares the one array and it keeps
 * the last call's contents (nothing in it needs to start at zero: each call
 * writes every partial the merge reads).  Calls whose work overlaps on the
 * GPU (for example on two streams) race on the array and give wrong results;
 * order them on one stream or with events.
 */
SLOPE_API slope_status slope_cp_prefill_static_scratch(const slope_tensor* q, const slope_tensor* k,
                                                       const slope_tensor* v, int n_chunks, slope_layout layout,
                                                       const int64_t* chunk_sizes, int causal, int64_t window,
                                                       float scale, slope_tensor* out, slope_tensor* lse,
                                                       void* stream);

/* Workspace bytes slope_cp_prefill needs for these sizes (0 on invalid arguments). */
SLOPE_API size_t slope_cp_prefill_workspace_size(int64_t S, int64_t Hq, int64_t dv, int n_chunks, slope_layout layout,
                                       const int64_t* chunk_sizes);

/* Flags of slope_cp_prefill_ex. */
#define SLOPE_CP_BF16_PARTIALS 1u /* keep the partial outputs in bf16 (lse stays fp32)            */
#define SLOPE_CP_FUSED 2u         /* merge each rank's / chunk's partials online, in the kernel    */

/*
 * slope_cp_prefill with options.  flags = 0 is slope_cp_prefill exactly.
 *
 * SLOPE_CP_BF16_PARTIALS: each partial output travels from the attention
 * launches to the merge rounded to bf16 (round to nearest even) instead of
 * fp32: half the workspace and half the bytes the merge reads.  The partial
 * log-sum-exps stay fp32 and the merge sums in fp32.  The pages name Ring
 * Attention (Moreh, section "Introduction to Context Parallelism") without
 * fixing the precision in which a step's partial result is kept; the merge is
 * the exact one of slope_lse_merge either way.  Since the merge weights are
 * positive and sum to 1, rounding each partial once more moves the final
 * output by at most one bf16 rounding (relative 2^-8) of the largest partial
 * element, before the output's own rounding when out is bf16.
 *
 * SLOPE_CP_FUSED: the ring and chunked layouts without partial planes and
 * without the merge launch.  Over a whole ring, each query sub-chunk of rank r
 * meets every key/value block once (Moreh, section "Introduction to Context
 * Parallelism", Ring Attention item: the blocks circulate until every device
 * has seen all of them), so its partials cover disjoint key sets whose union
 * is every key; under the masks that union is one contiguous key range.  With
 * this flag each query sub-chunk (ZIGZAG: two per rank; CONTIGUOUS: one) or
 * chunk (CHUNKED: its prefix and its diagonal) is one work item whose online
 * softmax runs over that range, key tiles in ascending order, and writes out
 * and lse directly: the same attention as the partials and the exact merge,
 * up to the order in which fp32 sums are taken.  The items of all ranks (or
 * chunks) share attention launches up to 32 items each.  A Ulysses degree in
 * the layout word still splits every item by head group.  SLOPE_LAYOUT_ULYSSES
 * already writes out directly; the flag changes nothing there.  A bf16 out
 * needs row/head strides that are multiples of 8 elements and a 16-byte
 * aligned pointer.  The workspace then holds only an lse plane (used when lse
 * is NULL).  Together with SLOPE_CP_BF16_PARTIALS (no partials to keep)
 * the call returns SLOPE_ERR_UNSUPPORTED.
 *
 * Unknown flag bits return SLOPE_ERR_UNSUPPORTED.  The workspace must hold
 * slope_cp_prefill_workspace_size_ex(..., flags) bytes (the flags = 0 size is
 * always enough).
 */
SLOPE_API slope_status slope_cp_prefill_ex(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                           int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                                           int64_t window, float scale, unsigned flags, slope_tensor* out,
                                           slope_tensor* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes slope_cp_prefill_ex needs for these sizes and flags (0 on invalid arguments). */
SLOPE_API size_t slope_cp_prefill_workspace_size_ex(int64_t S, int64_t Hq, int64_t dv, int n_chunks,
                                                    slope_layout layout, const int64_t* chunk_sizes, unsigned flags);

/*
 * slope_cp_prefill on inputs and outputs in host memory: the same attention
 * (Moreh, "Optimizing long-context prefill on multiple older-generation GPU
 * nodes", section "Introduction to Context Parallelism"), with the copies
 * to and from the GPU queued by the library, on three caller streams:
 *   copy_in_stream   host q/k/v -> the device buffers q/k/v,
 *   compute_stream   slope_cp_prefill on the device buffers (after the copies),
 *   copy_out_stream  device out/lse -> host out/lse (after the compute).
 *
 *   q_host, k_host, v_host, out_host, lse_host: host tensors (pinned memory
 *     for asynchronous copies), each dense (row-major, no padding) and of the
 *     same shape and dtype as its device buffer.  lse_host and lse are both
 *     NULL or both given.
 *   q, k, v, out, lse: caller-owned device buffers, dense; the other
 *     arguments are those of slope_cp_prefill.
 *
 * Nothing is allocated.  The call returns once the work is queued: the host
 * inputs must stay valid and unchanged until copy_in_stream has passed this
 * call, and the host outputs are valid once copy_out_stream has.  Two calls with
 * different device buffers overlap: the second call's input copies run while
 * the first computes, and the first call's output copies while the second
 * computes (the workspace is shared safely: both computes run on
 * compute_stream).  A call that reuses the device buffers of an earlier call
 * (same device, same q buffer) is ordered after it by events: its input
 * copies wait until the earlier compute has read the inputs, and its compute
 * waits until the earlier output copies have read out/lse.  The library
 * tracks 16 such buffer sets per process; taking a slot from a 17th set first
 * waits on the host for the oldest set's last call.  Argument errors return
 * a status before anything is queued.
 */
SLOPE_API slope_status slope_cp_prefill_host(const slope_tensor* q_host, const slope_tensor* k_host,
                                             const slope_tensor* v_host, slope_tensor* out_host,
                                             slope_tensor* lse_host, const slope_tensor* q, const slope_tensor* k,
                                             const slope_tensor* v, slope_tensor* out, slope_tensor* lse,
                                             int n_chunks, slope_layout layout, const int64_t* chunk_sizes,
                                             int causal, int64_t window, float scale, void* workspace,
                                             size_t workspace_bytes, void* copy_in_stream, void* compute_stream,
                                             void* copy_out_stream);

/*
 * Same as slope_cp_prefill, and additionally records a pair of CUDA events
 * around every kernel launch it makes, on `stream`: events[2*i] before launch
 * i and events[2*i+1] after it.  events is a host array of 2*n_event_pairs
 * cudaEvent_t handles created by the caller.  On return *n_launches holds the
 * number of launches made and launch_kind[i] (if non-NULL, n_event_pairs
 * entries) is 0 for an attention-partial launch, 1 for the merge and 2 for
 * the fill that sets the live partial planes' lse to -inf before the
 * attention launches.
 * Returns SLOPE_ERR_SHAPE if n_event_pairs is smaller than the launch count.
 */
SLOPE_API slope_status slope_cp_prefill_timed(const slope_tensor* q, const slope_tensor* k, const slope_tensor* v,
                                    int n_chunks, slope_layout layout, const int64_t* chunk_sizes, int causal,
                                    int64_t window, float scale, slope_tensor* out, slope_tensor* lse,
                                    void* workspace, size_t workspace_bytes, void* stream, void** events,
                                    int n_event_pairs, int* n_launches, int* launch_kind);

/*
 * Host-only view of the work decomposition slope_cp_prefill performs (no GPU
 * needed).  One entry per (launch, query block): the query rows, the partial
 * plane written and the key/value row ranges attended in that launch
 * (after dropping blocks the mask hides entirely).  In the ring and chunked
 * layouts an entry keeps only the query rows that see at least one of its
 * keys, and a block none of whose rows sees a key has no entry: the call first
 * sets the lse of every live partial plane to -inf, so rows in no entry of a
 * plane are empty partials the merge skips.  A plane with no entry is neither
 * launched nor merged (plane 0 always is).  Ulysses and fused entries cover
 * every row (they write the final output).
 */
typedef struct {
  int32_t launch;     /* attention launch index (ring step or chunk)      */
  int32_t plane;      /* partial plane written                             */
  int64_t q_row0;     /* first query row                                   */
  int64_t q_len;      /* number of query rows                              */
  int32_t n_kv;       /* number of key/value ranges (0..2)                 */
  int64_t kv_row0[2]; /* first key row of each range                       */
  int64_t kv_len[2];  /* length of each range                              */
  int32_t head_group;    /* the entry covers query heads [g*Hq/n, (g+1)*Hq/n)  */
  int32_t n_head_groups; /* n: 1 (all heads) except in SLOPE_LAYOUT_ULYSSES    */
} slope_plan_item;

/*
 * Fills up to `capacity` items (items may be NULL when capacity is 0) and
 * returns the total number of items, or a negative slope_status.  *n_launches
 * and *n_planes (if non-NULL) receive the attention-launch and partial-plane
 * counts.
 */
SLOPE_API int64_t slope_cp_prefill_plan(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes,
                              int causal, int64_t window, slope_plan_item* items, int64_t capacity,
                              int32_t* n_launches, int32_t* n_planes);

/*
 * slope_cp_prefill_plan for the decomposition slope_cp_prefill_ex performs with
 * these flags (SLOPE_CP_FUSED: one item per query sub-chunk or chunk, each over
 * its whole visible key range, one plane written directly).  Unknown or
 * conflicting flags return SLOPE_ERR_UNSUPPORTED.
 */
SLOPE_API int64_t slope_cp_prefill_plan_ex(int64_t S, int n_chunks, slope_layout layout, const int64_t* chunk_sizes,
                                           int causal, int64_t window, unsigned flags, slope_plan_item* items,
                                           int64_t capacity, int32_t* n_launches, int32_t* n_planes);

/*
 * Dynamic chunk sizing for SLOPE_LAYOUT_CHUNKED (host only, no GPU needed).
 *
 * The SGLang pipeline-parallelism article (TL;DR, caption of its throughput
 * figure) runs chunked prefill with dynamic chunking from an initial chunk of
 * 12288 tokens with a smoothing factor of 0.65, but stops before giving the
 * algorithm.  This call implements one reading of those two numbers: later
 * chunks shrink as the key prefix grows, towards the size whose attention cost
 * (visible query-key pairs: row i sees i + 1 keys, or min(i + 1, window))
 * equals the first chunk's, smoothed exponentially with factor sigma:
 *   n_0 = min(initial, S);
 *   n_c = round(sigma * n*(s_c) + (1 - sigma) * n_{c-1}), then rounded down to
 *         a multiple of align (at least align), the last chunk clipped to S,
 * where s_c is the chunk's first token and n*(s) the largest n >= 1 with
 * cost(s, n) <= cost(0, n_0).  Sizes never grow; sigma = 0 gives fixed chunks
 * of n_0, sigma = 1 chunks of equal cost.
 *
 *   S (1..2^30), initial >= 1, 0 <= sigma <= 1, window >= 0 (0 = none),
 *   1 <= align <= initial: else SLOPE_ERR_SHAPE.  sizes: host array of
 *   `capacity` entries (NULL when capacity is 0), filled with the first
 *   min(count, capacity) sizes.
 * Returns the number of chunks (their sizes sum to S), or a negative
 * slope_status.  Pass the sizes to slope_cp_prefill as chunk_sizes.
 */
SLOPE_API int64_t slope_dck_chunk_sizes(int64_t S, int64_t initial, double sigma, int64_t window, int64_t align,
                                        int64_t* sizes, int64_t capacity);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: SLOPE_OK, or SLOPE_ERR_TIMEOUT if a bounded kernel wait ran
 * out since the last query (the kernel that saw it skipped its remaining work
 * and released its tensor memory).  *site (if non-NULL) receives the code of
 * the wait that ran out (0 when none).
 */
SLOPE_API slope_status slope_device_status(void* stream, int* site);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing will ever complete, with the given limit in nanoseconds
 * (1e3..5e9).  The wait runs out, records SLOPE_ERR_TIMEOUT in the device
 * status word and the kernel returns normally; no fault, no hang.
 */
SLOPE_API slope_status slope_debug_timeout_selftest(uint64_t limit_ns, void* stream);

/*
 * Text of the last CUDA runtime/driver failure that made a call of this
 * library (in the calling thread) return SLOPE_ERR_CUDA, or "" if none.
 * The pointer stays valid until the next call from the same thread.
 */
SLOPE_API const char* slope_last_error(void);

/* Static description of a status code. */
SLOPE_API const char* slope_status_string(slope_status s);

/* Library version string. */
SLOPE_API const char* slope_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SLOPE_H */
