/*
 * rf.h -- C ABI of librf.so: fused online-softmax attention for one GB300.
 *
 * The library computes the cascaded reduction behind safe-softmax attention
 * -- row maximum, then the sum of exp(s - max), then the normalised P.V, with
 * s = scale * Q K^T -- in one pass over K and V, keeping a running maximum,
 * a running sum and an output accumulator on chip and rescaling them by
 * exp(m_old - m_new) at every key tile. Scores are never written to memory.
 *
 * Sources (page title, section):
 *  - RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions
 *    on AI Accelerators -- technical summary section 1 (attention is a safe
 *    softmax followed by a GEMM, a cascade of reductions), section 2 (formal
 *    definition d_i = (+) F_i(X[l], D_i); feasibility: decomposable F_i,
 *    commutative monoid, distributivity; incremental form with O(1) state),
 *    section 3 (single-segment strategy in one CTA; multi-segment strategy
 *    that partitions the input and merges partial results; FlashAttention
 *    and FlashDecoding are special cases).
 *  - Riepilogo Tecnico: FLASHLIGHT -- Metodologia items 2-4 (the max of the
 *    softmax fused into Q K^T, the online softmax by rescaling with
 *    e^(x-y) = e^x / e^y, small dimensions eliminated by tiling).
 *  - Accelerating Sparse Transformer Inference on GPU (STOF) -- Méthodologie,
 *    unified MHA module (row-compressed lists of block-sparse outer tiles;
 *    masked tiles skipped entirely rather than zeroed after the fact).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    allocates no device memory, never synchronises (except rf_device_status),
 *    and enqueues its kernels on the given stream; calls return at enqueue.
 *  - Layouts are dense row-major, last dimension contiguous:
 *      q, o : [B, H,   Sq, d]      k, v : [B, Hkv, Sk, d]      lse : [B, H, Sq]
 *  - Query head h reads key/value head h / (H / Hkv) (grouped-query heads).
 *  - Causal masking is bottom-right aligned: row i sees key j iff
 *    j <= i + (Sk - Sq).
 *  - lse is the natural-log log-sum-exp of the scaled, masked scores of a row.
 *    A row that sees no key gets O = 0 and lse = -inf.
 *  - Every call returns an rf_status. Invalid arguments are detected on the
 *    host and no kernel is launched; rf_last_error() then describes the
 *    problem (thread-local string, valid until the next call on the thread).
 *  - Data-dependent faults found on the device (a block list that is out of
 *    range or not ascending; a pipeline wait that ran out of time) never trap:
 *    the kernel records a code in a device status word and skips the work.
 *    rf_device_status() reads and clears it.
 */
#ifndef RF_H_
#define RF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *rf_stream;

typedef enum {
  RF_OK = 0,
  RF_ERR_INVALID = 1,      /* bad argument (host) or malformed block list (device) */
  RF_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head dim outside {64,128} for bf16) */
  RF_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  RF_ERR_TIMEOUT = 4       /* a device-side wait gave up (recorded in the device status word) */
} rf_status;

typedef enum {
  RF_F32 = 0,   /* float32 in, float32 out, float32 arithmetic */
  RF_BF16 = 1   /* bfloat16 in and out, float32 accumulation */
} rf_dtype;

/*
 * Block-sparse tile lists (STOF's outer-tile row-compressed format).
 * Tiles are 128 x 128 (query tile i covers rows [128 i, 128 i + 128), key
 * tile j covers keys [128 j, 128 j + 128)). For query tile i of head n the
 * listed key tiles are col_idx[row_ptr[n * nqt + i] .. row_ptr[n * nqt + i + 1]),
 * in strictly ascending order, each in [0, nkt). Unlisted tiles are skipped
 * entirely; listed tiles are attended in full (and, with causal, under the
 * causal element mask).
 *  per_head = 0: one list set shared by every (b, h); row_ptr has nqt + 1 entries.
 *  per_head = 1: B*H list sets back to back, head n = b * H + h;
 *                row_ptr has B*H*nqt + 1 entries.
 * Inner level (the same page's two-level format, optional): with tile_bits
 * non-NULL, tile_bits[n] (int32, parallel to col_idx) is -1 for a full tile
 * and otherwise the index P of the tile's bitmaps, bits[256 P .. 256 P + 255]:
 * one uint64 per 8 x 8 inner block, blocks row-major over the tile's 16 x 16,
 * bit 8 r + c = element (r, c) of the block (1 = attended). A partial tile is
 * attended only where its bit is set (and, with causal, causally visible).
 * tile_bits = NULL: every listed tile is full (bits is ignored).
 * Work order (optional): cta_order, as rf_blockmask_cta_order writes it, is
 * the order in which rf_attn_fwd's tensor-core kernel takes its work items
 * (bf16 only; the other kernels ignore it). NULL: head-major order. Entries
 * outside [0, items) are skipped and reported through rf_device_status.
 * row_ptr, col_idx, tile_bits, bits and cta_order are device pointers owned
 * by the caller; the struct itself is read on the host during the call only.
 * Zero-initialise the struct so that fields added later read as absent.
 */
typedef struct {
  int tile_q;                /* must be 128 */
  int tile_k;                /* must be 128 */
  int nqt;                   /* must be ceil(Sq / 128) */
  int nkt;                   /* must be ceil(Sk / 128) */
  const int32_t *row_ptr;    /* device */
  const int32_t *col_idx;    /* device */
  int per_head;              /* 0 or 1 */
  const int32_t *tile_bits;  /* device, parallel to col_idx; NULL: all tiles full */
  const uint64_t *bits;      /* device, 256 words per partial tile */
  const int32_t *cta_order;  /* device, optional: see rf_blockmask_cta_order; NULL: head-major */
} rf_blockmask;

/*
 * Row softmax: y[r, :] = exp(x[r, :] - max) / sum(exp(x[r, :] - max)).
 * The pure two-reduction cascade of the RedFuser page's problem statement
 * (maximum, then sum of exponentials). A row that fits one CTA (up to
 * 64 KB: cols <= 16384 for f32) is held in shared memory between the
 * reductions and the write: one read and one write of x per element in HBM.
 * A longer row is split over a cluster of 2..8 CTAs (64 KB or more each).
 * They exchange (max, sum) pairs through distributed shared memory
 * (multi-segment strategy), then read their slice a second time, mostly from
 * L2 where the first read left it.
 *  x, y : [rows, cols] row-major, dtype dt (RF_F32 or RF_BF16); may alias.
 *  rows >= 0, cols >= 0 (either 0: nothing is launched, RF_OK).
 * A row whose entries are all -inf yields zeros. Errors: RF_ERR_INVALID for
 * NULL pointers with nonzero sizes or negative sizes.
 */
rf_status rf_softmax_rows(const void *x, void *y, int64_t rows, int64_t cols,
                          rf_dtype dt, rf_stream stream);

/*
 * Attention forward (prefill), single-segment incremental form per query tile.
 *  q [B,H,Sq,d], k/v [B,Hkv,Sk,d] (dtype dt), o [B,H,Sq,d] (dtype dt),
 *  lse [B,H,Sq] float32 (may be NULL: not written).
 *  scale > 0 and finite (scores are scale * q.k).
 *  causal: 0 or 1.  blockmask: NULL for dense, else tile lists as above.
 * Supported: RF_BF16 with d in {64, 128} (tensor-core kernel: TMA-staged K/V
 * tiles, tcgen05 MMAs into tensor memory); RF_F32 with d % 4 == 0 and
 * d <= 256 (exact SIMT kernel, one warp per query row).
 * Pointers must be 16-byte aligned. B, H, Hkv >= 1; H % Hkv == 0;
 * 0 <= Sq, Sk <= 2^30 (Sq == 0: nothing launched; Sk == 0: O = 0,
 * lse = -inf).
 * Errors: RF_ERR_INVALID (NULL/misaligned pointers, bad sizes, H % Hkv,
 * scale <= 0, blockmask fields inconsistent with Sq/Sk); RF_ERR_UNSUPPORTED
 * (dtype/d combination not listed above).
 */
rf_status rf_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                      int causal, const rf_blockmask *blockmask, rf_dtype dt,
                      rf_stream stream);

/*
 * Attention forward on HOST buffers, the copies overlapped with the kernels.
 * Computes exactly what rf_attn_fwd computes (same arguments, same results),
 * but q, k, v are read from and o, lse written to host memory. The work is
 * cut into chunks of whole (batch, key/value-head group) slices -- independent
 * problems, so no merge is needed (the single-segment strategy per chunk) --
 * and chunk c's copy in, its kernel and the copy out of chunk c - 1 run
 * concurrently on internal streams (one for copies in, one for copies out,
 * two for the kernels, so that consecutive chunks' kernels overlap).
 *  q, k, v, o, lse: host pointers in rf_attn_fwd's layouts; page-locked
 *      memory (cudaHostAlloc, torch pin_memory) lets the copies run
 *      asynchronously, pageable memory works but serialises them. lse may be
 *      NULL. Must not change (q, k, v) or be read (o, lse) until the work on
 *      `stream` is done.
 *  ws: device workspace of at least rf_attn_fwd_host_workspace_bytes(...)
 *      bytes, 256-byte aligned, owned by the caller (two chunks in flight);
 *      no other call may use it until this one's work on `stream` is done.
 *  blockmask: as for rf_attn_fwd (device lists); its cta_order is not used
 *             (each chunk of heads runs in head-major order).
 * Ordering: the copies start after the work already queued on `stream`, and
 * work queued on `stream` afterwards starts after the last copy out; the host
 * is not blocked (except by pageable copies). The library creates four streams
 * and a few events per device on first use and keeps them.
 * Errors: those of rf_attn_fwd; RF_ERR_INVALID for NULL host pointers or a
 * short or misaligned workspace, or while the visited-tile debug buffer is
 * set; RF_ERR_CUDA if a copy or stream operation fails.
 */
rf_status rf_attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                           int causal, const rf_blockmask *blockmask, rf_dtype dt, void *ws,
                           size_t ws_bytes, rf_stream stream);

/* Bytes of device workspace rf_attn_fwd_host needs for these sizes (two
 * chunks of Q, K, V, O and LSE); 0 for invalid arguments. */
size_t rf_attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int Sq, int Sk, int d,
                                        rf_dtype dt);

/*
 * Split-K decode (multi-segment strategy; FlashDecoding as a special case).
 * One query row per head: q [B,H,1,d], k/v [B,Hkv,Sk,d], o [B,H,1,d], all
 * dtype dt (RF_BF16); lse [B,H,1] float32 (may be NULL). The keys are cut
 * into nsplit contiguous splits of Sk / nsplit keys (the last split takes the
 * remainder); each split's partial (O_s normalised within the split, lse_s)
 * goes to the workspace, then rf_splitk_merge combines them on the same
 * stream. Every query head of a key/value group shares one pass over K/V.
 *  ws: device workspace of at least rf_decode_workspace_bytes(B,H,nsplit,d)
 *      bytes, 16-byte aligned, owned by the caller; ws_bytes its size.
 *      Layout: o_part float32 [B*H, nsplit, d] followed by lse_part float32
 *      [B*H, nsplit].
 *  1 <= nsplit <= Sk; d in {64, 128}; H % Hkv == 0; H / Hkv <= 16.
 * Errors: RF_ERR_INVALID, RF_ERR_UNSUPPORTED (dt != RF_BF16 or d).
 */
rf_status rf_attn_decode_splitk(const void *q, const void *k, const void *v, void *o,
                                float *lse, int B, int H, int Hkv, int Sk, int d,
                                float scale, int nsplit, float *ws, size_t ws_bytes,
                                rf_dtype dt, rf_stream stream);

/*
 * Split-K decode without a caller workspace (no counterpart on the pages:
 * an addition for callers that cannot allocate device memory, e.g. a plug-in
 * inside a host process whose runtime owns all device memory, or a serving
 * loop that forbids allocation after start-up).
 * Same arguments, results and errors as rf_attn_decode_splitk, minus ws and
 * ws_bytes: the partials live in a 16 MiB array inside the library's device
 * image, reserved on every GPU that loads the library until the process
 * exits. Allocates nothing (no cudaMalloc/cudaFree, no allocating library
 * call).
 *  - Sizes whose workspace, rf_decode_workspace_bytes(B,H,nsplit,d), exceeds
 *    16 MiB (16777216 bytes) are rejected with RF_ERR_INVALID.
 *  - Invalid arguments are rejected as by rf_attn_decode_splitk, before any
 *    CUDA call.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress) and caches it for the current context;
 *    after cudaDeviceReset, or when the device's context is created again,
 *    the next call looks it up again. Make the first call in a context
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's partials. A successful call writes every partial before reading
 *    it, so nothing needs clearing; calls that overlap on the GPU (different
 *    streams, or concurrent host threads) race on it and must be serialised
 *    by the caller.
 *  - When rf_device_status reports RF_ERR_TIMEOUT after a call, a partials
 *    CTA gave up before writing its split, and that call's O and LSE are
 *    undefined (they may combine an earlier call's partials).
 */
rf_status rf_attn_decode_splitk_noalloc(const void *q, const void *k, const void *v, void *o,
                                        float *lse, int B, int H, int Hkv, int Sk, int d,
                                        float scale, int nsplit, rf_dtype dt, rf_stream stream);

/*
 * The partials step of rf_attn_decode_splitk alone (multi-segment strategy,
 * RedFuser section 3: the per-segment results before the merge). Writes into
 * ws, laid out as rf_attn_decode_splitk's workspace,
 *   o_part float32 [B*H, nsplit, d] (each split's O, normalised within it),
 *   then lse_part float32 [B*H, nsplit] (natural log; -inf for no key),
 * and launches nothing else. A rank holding a contiguous shard of the keys
 * computes its partials with this call, merges them (rf_splitk_merge with
 * out_dt RF_F32), exchanges the per-rank results and merges those with
 * rf_splitk_merge_strided. Arguments and errors as rf_attn_decode_splitk.
 */
rf_status rf_attn_decode_partials(const void *q, const void *k, const void *v, float *ws,
                                  size_t ws_bytes, int B, int H, int Hkv, int Sk, int d,
                                  float scale, int nsplit, rf_dtype dt, rf_stream stream);

/* Bytes of workspace rf_attn_decode_splitk needs: 4 * B*H*nsplit*(d + 1),
 * rounded up to 256. Returns 0 for non-positive arguments. */
size_t rf_decode_workspace_bytes(int B, int H, int nsplit, int d);

/*
 * Log-sum-exp merge of split partials (multi-segment strategy, merge step):
 *   LSE = log sum_s exp(lse_s),   O = sum_s exp(lse_s - LSE) * O_s.
 *  o_part float32 [rows, nsplit, d], lse_part float32 [rows, nsplit] (device);
 *  o [rows, d] of dtype out_dt; lse float32 [rows] (may be NULL).
 * Partials with lse_s = -inf contribute nothing (their O_s is not read and
 * may hold any bits, NaN included); a row whose partials are all -inf gets
 * O = 0 and LSE = -inf. rows >= 0, nsplit >= 1, 1 <= d <= 1024.
 */
rf_status rf_splitk_merge(const float *o_part, const float *lse_part, void *o, float *lse,
                          int64_t rows, int nsplit, int d, rf_dtype out_dt,
                          rf_stream stream);

/*
 * The same merge over partials laid out with explicit element strides:
 * partial s of row r is the d floats at o_part + s * o_split_stride +
 * r * o_row_stride, with its lse at lse_part[s * lse_split_stride +
 * r * lse_row_stride]. rf_splitk_merge is the row-major case
 * (o strides d and nsplit * d, lse strides 1 and nsplit). The split-major
 * case [nsplit, rows, d] (o strides rows * d and d, lse strides rows and 1)
 * is what an all-gather of per-rank partials produces when the keys are
 * sharded across GPUs (RedFuser, section 3, multi-segment strategy:
 * partition the input, then merge the partial results), so it is merged
 * without a transposing copy. Strides >= 0; other rules as rf_splitk_merge.
 */
rf_status rf_splitk_merge_strided(const float *o_part, const float *lse_part, void *o, float *lse,
                                  int64_t rows, int nsplit, int d, int64_t o_split_stride,
                                  int64_t o_row_stride, int64_t lse_split_stride,
                                  int64_t lse_row_stride, rf_dtype out_dt, rf_stream stream);

/*
 * Build block-sparse tile lists from a dense tile mask on the device.
 *  dense: uint8 [nheads, nqt, nkt] (nonzero = tile present), device.
 *  row_ptr: int32 [nheads*nqt + 1] (device, written): exclusive scan of the
 *           per-row counts; row_ptr[nheads*nqt] = total nnz.
 *  col_idx: int32 [col_cap] (device, written): column indices of each row in
 *           ascending order. If nnz > col_cap, entries past col_cap are not
 *           written (row_ptr still holds the true counts) and the device
 *           status word records RF_ERR_INVALID.
 * One list set per head, in the layout rf_blockmask expects (per_head = 1
 * when nheads > 1). nheads, nqt, nkt >= 1; col_cap >= 0.
 */
rf_status rf_blockmask_build(const uint8_t *dense, int nheads, int nqt, int nkt,
                             int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                             rf_stream stream);

/*
 * Build the two-level (outer lists + inner 8 x 8 bitmaps) mask of a dense
 * element mask on the device (STOF page, two-level storage format).
 *  dense: uint8 [nheads, Sq, Sk] (nonzero = attend), device.
 *  An outer 128 x 128 tile is listed if it holds a nonzero element; it is
 *  full (tile_bits = -1) if every element of it inside the Sq x Sk matrix is
 *  nonzero, else partial, with 256 bitmap words (bits outside the matrix 0).
 *  row_ptr: int32 [nheads*nqt + 1]; col_idx, tile_bits: int32 [nheads*nqt*nkt]
 *  (capacity for every tile; entries past row_ptr[last] are unspecified);
 *  bits: uint64 [bits_cap * 256], partial tiles numbered in list order; a
 *  mask with more than bits_cap partial tiles records RF_ERR_INVALID in the
 *  device status word and leaves the extra bitmaps unwritten. bits = NULL:
 *  only the lists are built (tile_bits still numbers the partial tiles), no
 *  error is recorded, and n_partial tells how large bits must be. n_partial
 *  (device int32, may be NULL) receives the number of partial tiles.
 * nheads, Sq, Sk >= 1, bits_cap >= 0; nqt = ceil(Sq/128), nkt = ceil(Sk/128).
 */
rf_status rf_blockmask_build_elements(const uint8_t *dense, int nheads, int Sq, int Sk,
                                      int32_t *row_ptr, int32_t *col_idx, int32_t *tile_bits,
                                      uint64_t *bits, int64_t bits_cap, int32_t *n_partial,
                                      rf_stream stream);

/*
 * Row-wise attention: the same operation and arguments as rf_attn_fwd, by
 * STOF's row-wise kernel (Accelerating Sparse Transformer Inference on GPU,
 * Méthodologie, unified MHA module, dual-kernel strategy: Q split into rows,
 * warp-level shuffles, no synchronisation between warps). One warp per query
 * row visits only the row's visible keys -- all keys of a full listed tile,
 * the set bits of a partial tile's inner bitmaps, up to the causal limit --
 * in float32 (bf16 inputs widened exactly; P is not rounded), so its work is
 * proportional to the visible pairs rather than to the listed tiles. For
 * highly sparse masks on short sequences. d must be 64 or 128 (f32 or bf16).
 * The rf_debug_set_visited test aid does not apply to this kernel.
 * Errors: those of rf_attn_fwd; RF_ERR_UNSUPPORTED for d outside {64, 128}.
 */
rf_status rf_attn_fwd_rowwise(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int Hkv, int Sq, int Sk, int d, float scale,
                              int causal, const rf_blockmask *blockmask, rf_dtype dt,
                              rf_stream stream);

/*
 * Inputs of the kernel selector below, counted on the device from the tile
 * lists themselves (STOF, Méthodologie, unified MHA module: the selection is
 * taken from the mask's sparsity, which the lists already encode).
 *  bm     : the lists as rf_attn_fwd takes them (NULL: dense), for an
 *           attention of B x H heads, Sq queries, Sk keys, causal 0/1.
 *  counts : device int64[3], caller-owned, overwritten on the stream with
 *           counts[0] = listed tiles that hold a visible pair (tiles the
 *                       attention kernels process), over all B*H heads;
 *           counts[1] = how many of them are partial (two-level masks);
 *           counts[2] = visible (query, key) pairs over all heads, after the
 *                       causal limit and the inner bitmaps.
 *           A list shared by all heads (per_head 0) counts once per head.
 * Asynchronous: read counts after the stream has reached the call. Out-of-
 * range tile indices are skipped and reported through rf_device_status.
 * Errors: RF_ERR_INVALID (bad sizes or list fields, counts NULL or not
 * 8-byte aligned), RF_ERR_CUDA.
 */
rf_status rf_blockmask_counts(const rf_blockmask *bm, int B, int H, int Sq, int Sk, int causal,
                              int64_t *counts, rf_stream stream);

#define RF_KERNEL_BLOCKWISE 0  /* rf_attn_fwd */
#define RF_KERNEL_ROWWISE 1    /* rf_attn_fwd_rowwise */

/*
 * STOF's kernel selection (same page, unified MHA module): an analytic model
 * of both kernels' times from the mask's sparsity and the sequence length.
 *  listed_tiles : 128 x 128 tiles listed over all B*H heads (a shared mask
 *                 counts once per head); partial_tiles: how many of them are
 *                 partial (two-level masks), 0 <= partial <= listed;
 *  visible_pairs: visible (query, key) pairs over all heads (after causal);
 *  num_sms      : streaming multiprocessors of the device (152 on GB300).
 * rf_attn_choose_kernel returns RF_KERNEL_BLOCKWISE or RF_KERNEL_ROWWISE
 * (the smaller estimate), or -1 for invalid arguments (B, H, Sq >= 1,
 * Sk >= 0, d in {64, 128}, counts >= 0, num_sms >= 1). rf_attn_estimate_us
 * writes both estimates in microseconds (RF_ERR_INVALID on bad arguments or
 * NULL outputs). Pure host functions: no CUDA call.
 */
int rf_attn_choose_kernel(int B, int H, int Sq, int Sk, int d, int64_t listed_tiles,
                          int64_t partial_tiles, int64_t visible_pairs, int num_sms);
int rf_attn_estimate_us(int B, int H, int Sq, int Sk, int d, int64_t listed_tiles,
                        int64_t partial_tiles, int64_t visible_pairs, int num_sms,
                        double *block_us, double *row_us);

/*
 * Work order of rf_attn_fwd's tensor-core (bf16) kernel for a block-sparse or
 * two-level mask. The kernel's work items are double items x in [0, items),
 * items = B * H * ceil(pairs / 2) with pairs = ceil(nqt / 2): item x of head
 * x / ceil(pairs / 2) holds the query-tile pair counted j = x % ceil(pairs / 2)
 * from the top and the pair counted j from the bottom (about equal causal
 * work). By default CTA c takes item c, head-major, so that a head's K and V
 * stay in L2 while its CTAs run. A mask whose query tiles differ a lot in
 * listed tiles (global tokens: query rows that attend to every key, as in
 * STOF's sparse patterns) then leaves one long CTA per head spread over the
 * grid, and the last of them sets the kernel's end. This call writes order[c]
 * = the item CTA c takes: the items whose listed tiles exceed twice the mean
 * first, then the others, both in head-major order (a stable partition, so a
 * mask without such items keeps the default order).
 *  bm    : the lists (row_ptr required; its cta_order field is ignored);
 *  B, H, Sq: the attention the order is for (nqt = ceil(Sq/128) = bm->nqt);
 *  order : device int32 [cap], cap >= rf_blockmask_cta_order_len(B, H, Sq).
 * Listed tiles are counted before any causal truncation. Asynchronous on the
 * stream. Errors: RF_ERR_INVALID (bad sizes or fields, order NULL or short),
 * RF_ERR_CUDA.
 */
int64_t rf_blockmask_cta_order_len(int B, int H, int Sq);
rf_status rf_blockmask_cta_order(const rf_blockmask *bm, int B, int H, int Sq, int32_t *order,
                                 int64_t cap, rf_stream stream);

/*
 * Multi-head latent attention (MLA) decode, absorbed form (RedFuser page,
 * section 4: MLA is one of the evaluated workloads, compared with FlashMLA;
 * section 3: multi-segment strategy). Each batch element has one query
 * token of 128 heads and one latent key-value head:
 *  q   : bf16 [B, 128, 576] (512 latent + 64 rotary columns per head);
 *  kv  : bf16 [B, Sk, 576], shared by the 128 heads; the values are its
 *        first 512 columns;
 *  o   : bf16 [B, 128, 512]; lse: float [B, 128] (natural log) or NULL;
 *  s = scale * q . kv over all 576 columns; o = softmax(s) v.
 * The keys are cut into nsplit contiguous segments (floor(Sk/nsplit) keys,
 * the last one takes the remainder; 1 <= nsplit <= Sk). One CTA per SM, half
 * of them per half of the value columns, takes a contiguous run of the
 * B * nsplit segments; the segments of one batch element within a run are
 * folded into one partial (O, LSE), computed on the tensor cores and stored
 * in the slot of the first of them (the other slots get LSE = -inf). The
 * partials are merged by log-sum-exp (rf_splitk_merge) in the caller's
 * workspace (float, >= rf_mla_decode_workspace_bytes bytes: o_part
 * [B*128, nsplit, 512] then lse_part [B*128, nsplit]). So nsplit sets the
 * granularity at which keys are dealt to the SMs. All pointers
 * device, 16-byte aligned (lse 4). Errors: RF_ERR_INVALID for bad sizes,
 * NULL or misaligned pointers, a short workspace; a device wait that gives
 * up records RF_ERR_TIMEOUT in the device status word.
 */
size_t rf_mla_decode_workspace_bytes(int B, int nsplit);
rf_status rf_mla_decode(const void *q, const void *kv, void *o, float *lse, int B, int Sk,
                        float scale, int nsplit, float *ws, size_t ws_bytes, rf_stream stream);

/*
 * Mixture-of-Experts top-k softmax routing (RedFuser page, section 1: MoE
 * routing is a cascade of reductions; section 4: one of its workloads).
 * For each token t: p = softmax(logits[t, :]) over the E experts (maximum,
 * then sum of exponentials), then the k experts with the largest p in
 * descending order, ties going to the lower expert index (exp is increasing,
 * so the selection is taken on the logits themselves, as given).
 *  logits : [T, E] row-major, dtype dt (RF_F32 or RF_BF16), device.
 *  idx    : int32 [T, k], device, written (expert indices, descending p).
 *  w      : float [T, k], device, written: p of the selected experts, or,
 *           with renorm = 1, p divided by the sum of the k selected p.
 *  lse    : float [T], device, may be NULL: max + log(sum of exponentials).
 *  T >= 0 (0: nothing launched), 1 <= E <= 1024, 1 <= k <= min(E, 32).
 * One warp per token reads the token's logits once. Errors: RF_ERR_INVALID
 * for NULL pointers, sizes out of range or a bad dtype.
 */
rf_status rf_moe_route(const void *logits, int64_t T, int E, int k, int renorm, int32_t *idx,
                       float *w, float *lse, rf_dtype dt, rf_stream stream);

/*
 * Per-row moments and normalisation (RedFuser page, section 1:
 * normalisation layers; the Korean page's variance workload): the mean, then
 * the population variance sum((x - mean)^2) / n, which needs the mean, and
 * optionally y = (x - mean) / sqrt(var + eps). The two reductions run in one
 * read of x: each thread folds its elements into a (count, mean, M2) state
 * and the states merge pairwise (Chan, Golub and LeVeque), the incremental
 * form of the two-pass definition.
 *  x    : [rows, cols] row-major, dtype dt (RF_F32 or RF_BF16), device.
 *  mean, var : float [rows], device, each may be NULL.
 *  y    : [rows, cols], dtype dt, device, may be NULL (statistics only);
 *         may alias x.
 *  rows >= 0, cols >= 0 (either 0: nothing launched); rows <= 2^31 - 1;
 *  eps >= 0 and finite. A row is read once more from L2 when y is written.
 * Errors: RF_ERR_INVALID for NULL x with nonzero sizes, bad dtype or eps.
 */
rf_status rf_row_moments(const void *x, int64_t rows, int64_t cols, float eps, float *mean,
                         float *var, void *y, rf_dtype dt, rf_stream stream);

/*
 * Moment of inertia of point sets (the Korean RedFuser page's results: a
 * non-ML cascaded reduction): for each set of n point masses, the total mass
 * M = sum m_i and the centre of mass c = sum m_i r_i / M (reduction 1), then
 * the moment of inertia about the centre of mass I = sum m_i |r_i - c|^2
 * (reduction 2, which needs c), in one read of the points: mass-weighted
 * (W, c, M2) states merged pairwise (the weighted form of Chan, Golub and
 * LeVeque's merge).
 *  points : float [sets, n, 3] (x, y, z of each point), device.
 *  masses : float [sets, n], device, or NULL for unit masses.
 *  total_mass : float [sets]; center: float [sets, 3]; inertia: float [sets];
 *               device, each may be NULL.
 *  sets >= 0 (0: nothing launched), n >= 0; a set of total mass 0 (or
 *  n = 0) gives M = 0, c = 0, I = 0. Errors: RF_ERR_INVALID for NULL points
 *  with n > 0, negative sizes, or misaligned pointers.
 */
rf_status rf_moment_of_inertia(const float *points, const float *masses, int64_t sets, int64_t n,
                               float *total_mass, float *center, float *inertia,
                               rf_stream stream);

/*
 * Per-row FP8 quantisation (RedFuser page, sections 1 and 4: FP8 quantisation
 * followed by GEMM is a cascade of reductions). For each row of x:
 * amax = max |x| (reduction 1); codes = E4M3(float32(x) * (448 / amax)),
 * rounded to nearest even and saturated at 448 (4 exponent bits, bias 7,
 * 3 mantissa bits); scale = amax / 448. An all-zero row gives codes 0 and
 * scale 1. The row is read once (staged in shared memory).
 *  x     : [rows, K] row-major, RF_F32 or RF_BF16, device, 16-byte aligned.
 *  q     : uint8 [rows, K] E4M3 codes, device, 16-byte aligned.
 *  scale : float [rows], device.
 *  rows >= 0 (0: nothing launched); K a positive multiple of 16 with
 *  K * element size <= 64 KB (RF_ERR_UNSUPPORTED otherwise).
 */
rf_status rf_rowquant_e4m3(const void *x, int64_t rows, int64_t K, uint8_t *q, float *scale,
                           rf_dtype dt, rf_stream stream);

/*
 * GEMM over E4M3 codes with per-row and per-column scales (reduction 2 of the
 * cascade above): C[m, n] = sa[m] * sw[n] * sum_k A[m, k] W[n, k], products
 * accumulated in float32 by tcgen05.mma kind::f8f6f4 tiles of 128 x 256, C
 * rounded to bf16.
 *  a  : uint8 [M, K] codes (K-major), w: uint8 [N, K] codes (K-major),
 *       c: bf16 [M, N]; device, 16-byte aligned.
 *  sa : float [M], sw: float [N]; device.
 *  M a multiple of 128, N of 256, K a positive multiple of 128
 *  (RF_ERR_UNSUPPORTED otherwise); M or N = 0: nothing launched.
 * Errors: RF_ERR_INVALID for NULL or misaligned pointers; a device wait that
 * gives up records RF_ERR_TIMEOUT in the device status word.
 */
rf_status rf_fp8_gemm(const uint8_t *a, const float *sa, const uint8_t *w, const float *sw,
                      void *c, int M, int N, int K, rf_stream stream);

/*
 * Test aid: when visited is non-NULL, every later rf_attn_fwd on this host
 * thread sets visited[((b*H + h) * nqt + qt) * nkt + kt] = 1 for each
 * 128 x 128 tile (qt, kt) whose scores it computes. The caller zeroes the
 * uint8 buffer (device, >= B*H*nqt*nkt bytes; visited_len its size).
 * NULL turns it off. The skip set is checked bit-exactly against the set of
 * tiles holding at least one visible (query, key) pair.
 */
rf_status rf_debug_set_visited(uint8_t *visited, int64_t visited_len);

/*
 * Test aid (fault injection without a GPU fault): every later call on this
 * host thread that reaches the named site skips one step there, so that a
 * bounded device wait runs out. 0 turns it off.
 *  site 1: rf_softmax_rows, a row that one CTA holds on chip (cols * element
 *          size <= 64 KB, 16-byte aligned): CTA 0 arms the barrier of its
 *          first shared-memory copy but never issues the copy. Its waits give
 *          up after the device wait limit (2 s), it records a timeout in the
 *          device status word (rf_device_status then returns RF_ERR_TIMEOUT),
 *          waits (bounded) for its own copies in flight and exits; the other
 *          CTAs and later calls are unaffected.
 * Errors: RF_ERR_INVALID for an unknown site.
 */
rf_status rf_debug_inject_fault(int site);

/*
 * Synchronises the stream, then reads and clears the device status word of
 * the current device. *code receives the raw code (0 = nothing recorded).
 * Returns RF_OK, RF_ERR_TIMEOUT (a wait gave up), RF_ERR_INVALID (a malformed
 * device-side list), or RF_ERR_CUDA.
 */
rf_status rf_device_status(rf_stream stream, int *code);

/* Thread-local description of the last error returned on this thread. */
const char *rf_last_error(void);

/* ABI version, currently 1. */
int rf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RF_H_ */
