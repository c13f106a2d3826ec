/*
 * bsattn.h -- C ABI of the frame-aligned block-sparse attention forward for
 * B300 (sm_103a).  Library: libbsattn.so (block_sparse_video_row_b300/).
 *
 * The operation (web pages on HeyGen's Avatar IV port to Trillium TPUs):
 *  - Attention in a video super-resolution transformer whose block mask, at
 *    frame granularity, says which key/value blocks each query block reads.
 *    Block edges coincide with frame edges and the block size is any multiple
 *    of 16, so no element predicate, tail pass or padding exists
 *    ("HeyGen Avatar IV on Trillium TPU" deep-dive, section 把 block 縮到 16 /
 *    "shrink the block to 16"; "Optimizing HeyGen's Avatar IV diffusion model
 *    for Google Cloud TPUs", section "How it works").
 *  - The softmax uses a precomputed per-row upper bound on the logits in place
 *    of the running max: m_i = scale * |q_i| * max over allowed keys |k_j|,
 *    which holds by Cauchy-Schwarz, so exp(S - m_i) accumulates with no
 *    rescaling (deep-dive, section 拿掉 softmax 的序列相依 / "remove softmax's
 *    serial dependency"; "How is HeyGen optimizing AI video on Google Cloud
 *    TPUs", section "Innovating Beyond Serial Dependencies").  Following the
 *    deep-dive's eligibility check with fallback to online softmax (same
 *    section), work units holding a row whose bound is far above any plausible
 *    logit are sent to a running-max (online softmax) launch of the same kernel
 *    template, and rows whose exponentials underflow anyway are detected and
 *    rerun in that launch.
 *
 * Tensors: Q and O are bf16, contiguous [B, H, L, D] with L = nb * block_size;
 * K and V are [B, H, L_kv, D] with L_kv = nb_kv * block_size; 16-byte-aligned
 * base addresses, on the device that was current at layout creation.  Row i of
 * head (b, h) belongs to block i / block_size, key j to block j / block_size.
 * The block mask is one [nb, nb_kv] uint8 matrix (row-major, nonzero = query
 * block qb reads key block kb), shared by every batch entry and head, or, with
 * BSATTN_MASK_PER_HEAD, one such matrix per head (shared by the batch entries).
 * Self-attention over one chunk has L_kv = L (bsattn_create_layout); a streamed
 * chunk whose queries also read earlier context frames has L_kv > L
 * (bsattn_create_layout_rect; the pages stream their output chunk by chunk,
 * deep-dive, opening section).
 *
 * Ownership: the caller owns every tensor it passes (Q, K, V, O, LSE and the
 * metadata buffers).  A layout owns its host plan and its device buffers (the
 * allowed-block table, the work list and a small workspace for the underflow
 * guard), allocated by bsattn_create_layout and freed by bsattn_destroy.  The
 * mask is copied; the caller may free it after create.
 *
 * Streams: bsattn_row_bounds and bsattn_forward enqueue work on `stream` and
 * never synchronise.  A layout keeps per-call state in its workspace, so calls
 * with the same layout must not overlap on the GPU (use one stream per layout).
 *
 * Errors: argument errors are returned before any work is enqueued.  Device-
 * side conditions (a bounded wait that ran out, which the kernel reports and
 * returns from instead of hanging; with BSATTN_DEBUG_CHECKS, a work unit that the
 * device checks rejected) are recorded in a device status word that
 * bsattn_query_stats returns.
 */
#ifndef BSATTN_H
#define BSATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bounded waits: every wait inside the kernels gives up after a wall-clock limit
 * (the environment variable BSATTN_TIMEOUT_MS, read when a layout is created;
 * default 4000 ms), records BSATTN_ERR_TIMEOUT in the layout's status word and
 * returns, so a stalled pipeline never hangs the GPU. */

/* Concurrency: a layout holds one guard workspace (counters, unit flags, fallback
 * list), reset by every bsattn_forward, and bsattn_forward_host keeps its staging,
 * streams and chunk layouts in the layout.  Calls on one layout must therefore be
 * ordered: issue them on one stream (or order the streams with events) and from one
 * host thread at a time.  Use one layout per concurrent stream.  Different layouts are
 * independent. */

/* A cudaStream_t, passed through unchanged (NULL = the legacy default stream). */
typedef struct CUstream_st *bsattn_stream_t;

typedef struct bsattn_layout_s *bsattn_layout_t;

typedef enum {
    BSATTN_OK = 0,
    BSATTN_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned pointer, plan-only layout */
    BSATTN_ERR_UNALIGNED_BLOCK = 2, /* block_size not a multiple of 16, or L not a multiple of it */
    BSATTN_ERR_UNSUPPORTED = 3,     /* D other than 64 or 128, or sizes beyond the limits below */
    BSATTN_ERR_CUDA = 4,            /* a CUDA runtime / driver call failed */
    BSATTN_ERR_OOM = 5,             /* device allocation failed at create */
    BSATTN_ERR_TIMEOUT = 6,         /* a bounded device wait ran out (reported by query_stats) */
    BSATTN_ERR_DEVICE = 7,          /* no usable sm_103 (B300) device */
    BSATTN_ERR_INDEX = 8            /* device checks found a work unit or key tile out of range */
} bsattn_status;

/* flags */
enum {
    /* bsattn_forward (the default): an eligibility check of every work unit (its
       rows' bounds m_i at most BSATTN_ELIGIBLE_BOUND), the bound softmax over the
       eligible units with the underflow guard on their rows, then one online-max
       launch over the other units and the units holding a flagged row. */
    BSATTN_BOUND = 0,
    /* bsattn_forward: run the online-max (running max + rescale) kernel over
       every work unit instead; the A/B baseline of the same kernel. */
    BSATTN_ONLINE_MAX = 1,
    /* bsattn_forward: skip the online-max launch (testing only: rows of units
       that failed the eligibility check or hold a guard-flagged row keep an
       undefined value; with N(0,1)-like data there are none). */
    BSATTN_NO_FALLBACK = 2,
    /* bsattn_forward: every unit passes the eligibility check (the bound softmax
       for every row whatever its bound); the guard and the rerun still apply. */
    BSATTN_BOUND_ONLY = 4,
    /* bsattn_forward, testing only: the first work unit of every CTA never gets
       its query tiles, so the kernel's bounded waits run out (after the layout's
       wait limit, BSATTN_TIMEOUT_MS at create, default 4000 ms); the kernel
       returns, bsattn_query_stats reports BSATTN_ERR_TIMEOUT and o is undefined.
       The GPU context stays usable. */
    BSATTN_DEBUG_STALL = 0x100,
    /* bsattn_forward (and bsattn_forward_host): device-side index checks.  Before
       any role of the kernel uses a work unit, it checks the unit (head, query
       block, query tiles against the frame) and every key tile the unit reads
       (start and width against L_kv, 16-aligned, width 16..128) against the
       layout's tables.  A unit that fails is skipped by every role (its rows of o
       and lse are left as they were), bit BSATTN_ERR_INDEX is recorded in the
       layout's status word and bsattn_query_stats reports it.  Nothing traps.
       Costs one pass over the unit's tile list per role; off by default. */
    BSATTN_DEBUG_CHECKS = 0x200,
    /* bsattn_forward, testing only, and only together with BSATTN_DEBUG_CHECKS:
       the device checks see the first key tile of every CTA's first work unit as
       starting at L_kv (past the last key), so they reject that unit. */
    BSATTN_DEBUG_PLANT_INDEX = 0x400,
    /* bsattn_create_layout: build the host plan only, touch no device; such a
       layout can be inspected (info/export) but not run. */
    BSATTN_PLAN_ONLY = 0x10,
    /* bsattn_create_layout(_rect): one block mask per head.  block_mask then holds
       H masks, [H][nb][nb_kv] bytes, and head h of every batch reads mask h. */
    BSATTN_MASK_PER_HEAD = 0x20
};

/* Eligibility of a row for the bound softmax, in nats: a work unit holding a row
   with a larger Cauchy-Schwarz bound is computed by the online-max launch.
   Every unmasked logit satisfies S_ij >= -m_i, so the denominator of a bound row
   is at least exp(-2 m_i): a row with m_i <= 22 can never trip the guard, and
   above 64 a row passes it only if its best logit lies within 44 nats of a
   bound of more than 64, which the data this kernel serves rarely shows. */
#define BSATTN_ELIGIBLE_BOUND 64.0f

/* Limits checked by bsattn_create_layout. */
#define BSATTN_MAX_NB 4096            /* frames (blocks) per sequence, query or key side */
#define BSATTN_MAX_ROWS 2147483647LL  /* B * H * L and B * H * L_kv */

/*
 * Build a layout for one problem shape and block mask.
 *   out         receives the handle (set to NULL on error).
 *   B, H        batch and heads (>= 1).
 *   L           tokens per sequence (frames x tokens per frame), a multiple of block_size.
 *   D           head dimension: 64 or 128.
 *   block_size  tokens per frame block: a multiple of 16 (>= 16).
 *   block_mask  host pointer, nb * nb bytes, nb = L / block_size (row-major by query
 *               block, 1 = attend); H * nb * nb bytes with BSATTN_MASK_PER_HEAD.
 *   flags       0, or BSATTN_PLAN_ONLY and/or BSATTN_MASK_PER_HEAD.
 * The plan: the allowed key blocks of each query block in ascending order;
 * the key tiles of each query block (its allowed blocks grouped into runs of
 * consecutive frames, each run cut into tiles of 128 keys and one last tile of
 * the remaining keys: a multiple of 16, because frames are, so every tile is
 * an exactly sized MMA with no element mask or padding and none reaches into a
 * masked frame); query tiles of 128 rows that never straddle a frame edge (the
 * last tile of a frame may be partial); and a work list of pairs of query
 * tiles of one frame.  When a frame has an odd number of query tiles and its
 * last one holds at most 64 rows (a 3600-token frame: 28 tiles and 16 rows),
 * the tails of up to 8 consecutive frames are packed into one query tile (row
 * group g = the g-th frame) while each added frame costs fewer key tiles than
 * its own tail unit: that tile reads every key frame of its frames, in tiles cut
 * at frame edges, each marked with the row groups allowed to read it (a row
 * still reads exactly its own frames).  Every unit has a cost (100 per key tile for a unit of two query
 * tiles, 83 for one tile, whose softmax cannot overlap another tile's MMAs,
 * plus 150 per unit).  A device layout deals the units to its persistent CTAs
 * (one per SM) by that cost, each to the least-loaded CTA, in the order that
 * bsattn_layout_schedule describes.
 * The plan follows the frame-aligned layout of the deep-dive's section 把 block 縮到 16
 * (blocks whose edges are frame edges, any multiple of 16 tokens, so that no element
 * predicate, tail pass or padding is needed).
 * Returns BSATTN_OK, INVALID_ARG, UNALIGNED_BLOCK, UNSUPPORTED, CUDA, OOM or DEVICE.
 */
bsattn_status bsattn_create_layout(bsattn_layout_t *out, int32_t B, int32_t H, int64_t L, int32_t D,
                                   int32_t block_size, const uint8_t *block_mask, int32_t flags);

/*
 * The same for a streamed chunk: L query tokens (the chunk) reading L_kv >= L key
 * tokens (context frames and the chunk; L_kv < L returns BSATTN_ERR_UNSUPPORTED).  block_mask is nb * nb_kv bytes
 * (H * nb * nb_kv with BSATTN_MASK_PER_HEAD), nb = L / block_size, nb_kv = L_kv / block_size, row-major by
 * query block.
 * Q and O are [B, H, L, D], K and V [B, H, L_kv, D], qnorm and rowbound
 * [B, H, L], kmax [B, H, nb_kv].  bsattn_create_layout(..., L, ...) equals
 * bsattn_create_layout_rect(..., L, L, ...).  Returns as bsattn_create_layout.
 */
bsattn_status bsattn_create_layout_rect(bsattn_layout_t *out, int32_t B, int32_t H, int64_t L, int64_t L_kv,
                                        int32_t D, int32_t block_size, const uint8_t *block_mask, int32_t flags);

/*
 * The Cauchy-Schwarz row bounds (the precomputed norm table of the deep-dive,
 * section 拿掉 softmax 的序列相依).  All pointers are device pointers.
 *   q, k      bf16 [B, H, L, D] and [B, H, L_kv, D].
 *   scale     the softmax scale (usually 1/sqrt(D)); pass the same value to bsattn_forward.
 *   qnorm     out, fp32 [B, H, L]: |q_i|.
 *   kmax      out, fp32 [B, H, nb_kv]: the largest |k_j| of each key block.
 *   rowbound  out, fp32 [B, H, L]: m_i = (scale * |q_i|) * max over allowed kb of kmax[kb],
 *             each product rounded to fp32 (0 for a row that reads no block).
 * Norms use one fixed fp32 rounding order: the D elements split into 16
 * contiguous chunks, fmaf over each chunk in order, the chunk sums combined
 * pairwise at distances 8, 4, 2, 1, then a correctly rounded sqrt; so the
 * results are reproducible bit for bit.  Enqueued on `stream`; returns
 * BSATTN_OK, INVALID_ARG or CUDA.
 */
bsattn_status bsattn_row_bounds(bsattn_layout_t lay, const void *q, const void *k, float scale,
                                float *qnorm, float *kmax, float *rowbound, bsattn_stream_t stream);

/*
 * The same row bounds from per-token norms that the caller's own kernels already
 * produced, so Q and K are not read again.  The deep-dive (section
 * 拿掉 softmax 的序列相依) feeds the kernel a small precomputed norm table by
 * scalar prefetch, and "How is HeyGen optimizing AI video on Google Cloud TPUs"
 * (section "Innovating Beyond Serial Dependencies") fuses stages through explicit
 * layout contracts: a QK-norm, RoPE or projection epilogue that writes Q and K
 * can write their norms beside them, and this call then reads 4 bytes per token
 * instead of 2 * D.  All pointers are device pointers.
 *   qnorm     in, fp32 [B, H, L]: |q_i| for each query row.
 *   knorm     in, fp32 [B, H, L_kv]: |k_j| for each key row.
 *   scale     the softmax scale; pass the same value to bsattn_forward.
 *   kmax      out, fp32 [B, H, nb_kv]: the largest knorm of each key block (the
 *             maximum starts at 0, so negative and NaN entries never win it).
 *   rowbound  out, fp32 [B, H, L]: (scale * qnorm_i) * max over allowed kb of kmax[kb],
 *             each product rounded to fp32, exactly as bsattn_row_bounds forms it.
 * Given the norms bsattn_row_bounds computes, the outputs equal its outputs bit for
 * bit.  Norms rounded another way also work: the softmax is exact for any shift
 * that keeps its exponentials in range, and bsattn_forward's guard reruns, with the
 * online max, every row whose denominator underflowed or overflowed.
 * Enqueued on `stream`; returns BSATTN_OK, INVALID_ARG or CUDA.
 */
bsattn_status bsattn_row_bounds_from_norms(bsattn_layout_t lay, const float *qnorm, const float *knorm, float scale,
                                           float *kmax, float *rowbound, bsattn_stream_t stream);

/*
 * The attention forward.  All pointers are device pointers.
 *   q         bf16 [B, H, L, D] in; k, v bf16 [B, H, L_kv, D] in.
 *   o         bf16 [B, H, L, D] out (every row is written; rows that read no block get 0).
 *   scale     softmax scale (the value given to bsattn_row_bounds).
 *   rowbound  fp32 [B, H, L] from bsattn_row_bounds (unused with BSATTN_ONLINE_MAX; may be NULL then).
 *   lse       optional fp32 [B, H, L] out: the natural log of the softmax denominator,
 *             ln sum_j exp(scale * q_i . k_j) over allowed keys (-inf for rows that read nothing).
 *   flags     BSATTN_BOUND (0), BSATTN_ONLINE_MAX, BSATTN_NO_FALLBACK, BSATTN_BOUND_ONLY,
 *             BSATTN_DEBUG_CHECKS, and the testing flags BSATTN_DEBUG_STALL and
 *             BSATTN_DEBUG_PLANT_INDEX (the latter only with BSATTN_DEBUG_CHECKS).
 * BSATTN_BOUND computes P = exp(scale * S - m_i) with no running max, rounds P
 * to bf16 for the P.V product and sums the denominator from the same rounded
 * values.  Before it, a small kernel checks every work unit (one or two 128-row
 * query tiles of a frame): a unit holding a row with m_i > BSATTN_ELIGIBLE_BOUND
 * (the deep-dive's eligibility check, section 拿掉 softmax 的序列相依) is left to
 * the online-max launch that follows, whole (BSATTN_BOUND_ONLY turns the check
 * off).  A bound row is flagged when its denominator is below 2^-64 or not
 * finite, and every work unit holding a flagged row is recomputed by that
 * online-max launch too, on the same stream (no host synchronisation).  The
 * launches: a counter clear, the check, the bound kernel and the online-max
 * kernel; each exits at once when it has nothing to do.  The bound and
 * online-max kernels are programmatic dependent launches: each may be scheduled
 * while the kernel before it runs, and waits for that kernel's completion before
 * it reads or writes anything, so stream order holds as for plain launches.
 * Enqueued on `stream`; returns BSATTN_OK, INVALID_ARG or CUDA.
 */
bsattn_status bsattn_forward(bsattn_layout_t lay, const void *q, const void *k, const void *v, void *o,
                             float scale, const float *rowbound, float *lse, int32_t flags,
                             bsattn_stream_t stream);

/*
 * Row bounds and forward for tensors in host memory: the whole path of
 * bsattn_row_bounds + bsattn_forward, including the copies.
 *   q, k, v   host bf16 [B, H, L, D] in; o host bf16 [B, H, L, D] out.  Page-locked
 *             (pinned) memory lets the copies run asynchronously and overlap the
 *             kernels; pageable memory works but the copies then serialise.
 *   scale, flags  as for bsattn_forward (BSATTN_ONLINE_MAX skips the row bounds;
 *             the testing flags are refused).
 *   lse       optional host fp32 [B, H, L] out, as for bsattn_forward.
 *   pairs_per_chunk  (batch, head) pairs per pipeline chunk; 0 picks about twelve
 *             chunks.
 * The (batch, head) pairs are processed in chunks: copy-in, kernels and copy-out
 * run on three streams owned by the layout, with two sets of device staging
 * buffers, so the copies of one chunk overlap the kernels of the next.  The first
 * call (and a call with another chunk size) allocates the staging, about
 * 8 * pairs_per_chunk * L * D bytes plus metadata, with the chunk layouts and
 * streams; bsattn_destroy frees them.  Results equal bsattn_forward's on the same
 * inputs.  The work is ordered after earlier work on `stream`, and `stream` waits
 * for the last copy-out: synchronise `stream` before reading o.  Guard counters of
 * the whole call are reported by bsattn_query_stats.  Returns BSATTN_OK,
 * INVALID_ARG, OOM or CUDA.
 */
bsattn_status bsattn_forward_host(bsattn_layout_t lay, const void *q, const void *k, const void *v, void *o,
                                  float scale, float *lse, int32_t flags, int32_t pairs_per_chunk,
                                  bsattn_stream_t stream);

/*
 * bsattn_forward_noalloc -- the forward of bsattn_forward for callers that may not
 * allocate device memory.  The pages have no counterpart: this is a deployment
 * convenience of this library.
 *
 * Some callers cannot call cudaMalloc: a plugin whose host framework owns all
 * device memory through its own fixed arena, or a streaming loop that must not
 * take cudaMalloc's implicit device synchronisation between chunks.  Creating a
 * layout allocates the work plan and the guard workspace on the device; this
 * entry point needs no layout.  It builds the plan on the host for each call and
 * keeps plan and workspace in one static device array of
 * BSATTN_NOALLOC_SCRATCH_BYTES (1 MiB) inside the library, which every GPU that
 * loads the library holds until the process exits.  It calls no allocating CUDA
 * or library routine.
 *   q, k, v, o, scale, rowbound, lse, flags: as for bsattn_forward (device pointers;
 *             rowbound from bsattn_row_bounds or any equal bound).  flags: BSATTN_BOUND,
 *             BSATTN_ONLINE_MAX, BSATTN_NO_FALLBACK, BSATTN_BOUND_ONLY, BSATTN_MASK_PER_HEAD
 *             (one mask per head, as at layout creation) and the testing flag
 *             BSATTN_DEBUG_STALL.
 *   B, H, L, D, block_size, block_mask: as for bsattn_create_layout (mask on the host).
 *             Self-attention only: K and V have L rows per head, like Q (there is no
 *             streamed-chunk form with L_kv > L; use a layout for that).
 * The work units are dealt to one persistent CTA per SM by the same cost model as a
 * device layout, so the kernels run exactly as under bsattn_forward and the output is
 * bit-identical to it.
 * Limits: the array holds an 8-int guard header, 28 bytes per schedule slot (16 for
 * the slot, 4 each for its guard flag, its fallback-list entry and its eligibility;
 * the slots are the work units dealt to the CTAs, padded with empty slots to a
 * multiple of the SM count), the key-tile index of 4 * (n_segments + 1) bytes
 * (bsattn_layout_info) and 8 bytes per key tile, each of the four parts rounded up to
 * 256 bytes.  That is
 * about 37,000 slots (the 720p chunk uses about 4,700, the 1080p chunk about
 * 10,000); a larger problem returns BSATTN_ERR_UNSUPPORTED before any device work.
 * The first call on a device (with that device current) looks up the array's
 * device address.  Each call copies the plan and zeroed guard counters and status into
 * the array with one cudaMemcpyAsync from a host buffer that lives only during the
 * call, on `stream`, so the call may wait for work already queued on that stream,
 * and it cannot be captured in a CUDA graph: on a capturing stream it returns
 * BSATTN_ERR_UNSUPPORTED before any work (use a layout and bsattn_forward there).
 * All calls share the array and it keeps the last call's contents: calls whose GPU
 * work overlaps (other streams, other host threads) race.  A bounded device wait that
 * runs out leaves the rows of the units it stopped unwritten; bsattn_noalloc_query
 * reports it.  Returns BSATTN_OK, INVALID_ARG, UNALIGNED_BLOCK, UNSUPPORTED, CUDA or
 * DEVICE.
 */
#define BSATTN_NOALLOC_SCRATCH_BYTES (1 << 20)
bsattn_status bsattn_forward_noalloc(const void *q, const void *k, const void *v, void *o, int32_t B, int32_t H,
                                     int64_t L, int32_t D, int32_t block_size, const uint8_t *block_mask,
                                     float scale, const float *rowbound, float *lse, int32_t flags,
                                     bsattn_stream_t stream);

/*
 * Statistics of the last bsattn_forward_noalloc on the current device, read from its
 * static array without allocating: synchronises `stream`, then copies the guard
 * header with cudaMemcpy.  Outputs as for bsattn_query_stats (each nullable), but for
 * the last call only: every call clears the header, device status included.  Returns
 * BSATTN_OK, CUDA or DEVICE.
 */
bsattn_status bsattn_noalloc_query(int64_t *fallback_rows, int64_t *fallback_units, int32_t *device_status,
                                   bsattn_stream_t stream);

/* Free the layout's device buffers (plan tables, workspace, the host-tensor path's staging
 * and streams) and its host plan: the end of the layout created for one chunk shape and
 * frame mask (deep-dive, section 把 block 縮到 16).  Synchronises the layout's own
 * streams; work the caller queued on other streams must be complete.  NULL is ignored. */
void bsattn_destroy(bsattn_layout_t lay);

/* ---- helpers ----------------------------------------------------------------------------- */

/* A static, human-readable name for a status code. */
const char *bsattn_status_string(bsattn_status st);

/*
 * Statistics of the last bsattn_forward on this layout.  Synchronises `stream`.
 *   fallback_rows   rows flagged by the underflow guard (nullable).
 *   fallback_units  work units rerun with the online-max kernel (nullable).
 *   device_status   BSATTN_OK; BSATTN_ERR_TIMEOUT if a bounded device wait ran
 *                   out since the layout was created; else BSATTN_ERR_INDEX if
 *                   the device checks (BSATTN_DEBUG_CHECKS) rejected a work unit
 *                   since then (nullable).
 */
bsattn_status bsattn_query_stats(bsattn_layout_t lay, int64_t *fallback_rows, int64_t *fallback_units,
                                 int32_t *device_status, bsattn_stream_t stream);

/*
 * The eligibility check of the last bsattn_forward on this layout (the deep-dive's
 * per-head check, section 拿掉 softmax 的序列相依, made per work unit).  Synchronises
 * `stream`.
 *   bound_units   work units whose rows all had m_i <= BSATTN_ELIGIBLE_BOUND, computed
 *                 by the bound softmax (nullable).
 *   online_units  work units sent to the online-max launch (nullable).
 * Both 0 after a BSATTN_ONLINE_MAX forward, which checks nothing.  For
 * bsattn_forward_host, summed over the call's chunks.
 */
bsattn_status bsattn_query_eligibility(bsattn_layout_t lay, int64_t *bound_units, int64_t *online_units,
                                       bsattn_stream_t stream);

/* Plan summary of a layout (host only). */
typedef struct {
    int32_t B, H, D, block_size, nb;
    int64_t L;
    int32_t nnz_blocks;        /* allowed (query block, key block) pairs, summed over the masks */
    int32_t kv_tile;           /* keys per full key tile (128) */
    int32_t key_tiles;         /* key tiles over all query blocks of all masks */
    int32_t q_tiles_per_block; /* ceil(block_size / 128) */
    int32_t n_units;           /* work units (pairs of query tiles of one frame) */
    int64_t mma_rows;          /* query rows the MMAs process, partial tiles included */
    double useful_flop;        /* 4 * block_size^2 * D * B * (allowed pairs summed over the H heads) */
    int64_t L_kv;              /* key tokens per sequence (L for self-attention) */
    int32_t nb_kv;             /* key blocks */
    int32_t mask_heads;        /* masks in the plan: 1, or H with BSATTN_MASK_PER_HEAD */
    int32_t n_segments;        /* key-tile segments: mask_heads * nb, then one per packed-tail tile */
    int32_t tail_units;        /* work units that are packed tails of several frames (see create) */
} bsattn_layout_info_t;

bsattn_status bsattn_layout_info(bsattn_layout_t lay, bsattn_layout_info_t *info);

/*
 * Copy the plan to host arrays (any may be NULL).  Query block qb of mask m is
 * segment s = m * nb + qb (m = 0 for a shared mask; m = h with BSATTN_MASK_PER_HEAD):
 *   row_ptr  int32 [mask_heads * nb + 1], col_idx int32 [nnz_blocks]: allowed key blocks of
 *            segment s in col_idx[row_ptr[s] .. row_ptr[s+1]), ascending;
 *   units    int32 [n_units * 4]: (b * H + h, query block, first query tile, tiles in the unit (1 or 2)),
 *            in (b * H + h, query block, first query tile) order; a packed-tail unit (see
 *            bsattn_create_layout) is (b * H + h, first frame, its segment, -frames) and follows the
 *            units of its last frame;
 *   tile_ptr int32 [n_segments + 1], tiles int32 [key_tiles * 2]: the key tiles of segment s are
 *            (tiles[2t], tiles[2t+1]) = (first key within the head, width) for t in [tile_ptr[s], tile_ptr[s+1]);
 *            segments from mask_heads * nb on are packed-tail tiles, whose width words carry in bits
 *            16..23 the row groups (frames) allowed to read the tile.
 */
bsattn_status bsattn_layout_export(bsattn_layout_t lay, int32_t *row_ptr, int32_t *col_idx, int32_t *units,
                                   int32_t *tile_ptr, int32_t *tiles);

/*
 * The schedule a device layout runs for `grid` persistent CTAs (host only; a device
 * layout uses grid = the SM count, or fewer CTAs when it has fewer units).  The units
 * are taken in plan order, (head, frame, tile), so that the CTAs running at any one time
 * work on one or two heads and read each K/V tile from DRAM about once; the last
 * 4 * grid units (all of them, when there are fewer) are taken by cost instead, largest
 * first.  Each unit goes to the least-loaded CTA by the cost model of
 * bsattn_create_layout.  Slot k * grid + c holds CTA c's k-th unit as 4 int32 in the
 * format of `units` above; empty slots are (0, 0, 0, 0).
 *   grid     >= 1.
 *   slots    host int32 [*n_slots * 4] out, or NULL to learn the size.
 *   n_slots  out: slots, a multiple of grid.
 * Returns BSATTN_OK, INVALID_ARG or OOM.
 */
bsattn_status bsattn_layout_schedule(bsattn_layout_t lay, int32_t grid, int32_t *slots, int32_t *n_slots);

#ifdef __cplusplus
}
#endif

#endif /* BSATTN_H */
