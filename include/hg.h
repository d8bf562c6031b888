/*
 * hg.h - C ABI of the vocab-parallel LM-head logits gather on a two-parity
 * Lamport mailbox, for TP virtual ranks on one GPU.
 *
 * The operation (vLLM API page
 * "vllm.models.kimi_k3.nvidia.specialized_decode.runtime.logits_gather",
 * module docstring and class HeadGather): each of TP ranks holds an [M, W]
 * BF16 logits shard (W = V / TP vocab columns). Seen as 32-bit words, rank r's
 * row m is stored into the same row of each rank's mailbox (the pushing rank's
 * own included), starting at word column r * W / 2: NCCL's all-gather order. A mailbox word
 * that has not arrived holds the sentinel, the BF16 pair (+0, -0) = 0x80000000
 * (low half +0, high half -0); a data word equal to the sentinel is sent as
 * (+0, +0) = 0x00000000, every other word moves unchanged. Each rank polls its
 * mailbox row until no sentinel word is left, copies the row to its [M, V]
 * output and writes the sentinel back (re-arms). Two mailbox parities
 * alternate per call, so that a push never lands in a row that the previous
 * call may still be reading.
 *
 * On one GPU the TP ranks are virtual: every rank has its own shard, mailbox
 * and output allocation on the same device, and one kernel launch runs all of
 * them.
 *
 * Conventions for every entry point:
 *  - Return value: HG_OK (0) or one of the HG_ERR_* codes below.
 *  - "device pointer": memory of the device that was current at hg_create;
 *    the caller keeps that device current for every later call.
 *  - Calls on one handle are not thread-safe; every gather of a handle runs on
 *    one stream, in call order (the class docstring's one-stream assumption).
 *  - A call that returns an error other than HG_ERR_TIMEOUT changed nothing:
 *    neither the parity nor any mailbox nor any output.
 */
#ifndef HG_H_
#define HG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *hg_stream_t;

/* Opaque, library-owned state of one gather: the mailboxes, the parity, the
 * device status word and the launch shapes. */
typedef struct hg_handle hg_handle;

enum {
  HG_OK = 0,
  HG_ERR_ARG = 1,      /* invalid argument: NULL, misaligned, out of range */
  HG_ERR_ROWS = 2,     /* row count M not served by this handle (where
                          HeadGather.__call__ falls back to the stock gather) */
  HG_ERR_CAPTURE = 3,  /* stream is capturing a CUDA graph (HeadGather also
                          falls back to the stock gather under capture) */
  HG_ERR_CUDA = 4,     /* a CUDA runtime call failed (allocation, launch) */
  HG_ERR_TIMEOUT = 5,  /* a poll gave up: some pushed word never arrived */
  HG_ERR_STATE = 6     /* the handle holds an unrecovered device error;
                          call hg_rearm before gathering again */
};

/* Largest TP supported by one handle. */
#define HG_MAX_TP 32

/* Optional settings of hg_create_ex. Zero in any field selects the default. */
typedef struct hg_options {
  uint64_t poll_timeout_ns; /* bound of every poll; default 1e9 (1 s) */
  int elems_per_lane;       /* 16-byte vectors (or words) per lane per unit:
                               1 to 6 for tp <= 16, 1 or 2 above; default
                               chosen per row count */
  int ctas;                 /* CTAs of the gather kernel (32 * tp threads each);
                               default chosen per row count; clamped to what is
                               co-resident. Also caps the grid of
                               hg_gather_fused (default one CTA per SM) */
  int prefetch;             /* 0: chosen per row count (off unless tuned), 1: the
                               next push's shard loads are issued one iteration
                               ahead of its stores (overlapping a poll), 2: off */
  int cooperative;          /* 0 (default): programmatic dependent launch, the
                               next call's launch overlaps this one; 1:
                               cooperative launch, the runtime itself checks
                               that every CTA is co-resident (no overlap) */
  int device_parity;        /* 0 (default): the host keeps the parity and calls
                               on a capturing stream are refused
                               (HG_ERR_CAPTURE); 1: the parity lives in device
                               memory, each call's kernel reads it and flips it
                               once every CTA has read it, so calls may be
                               captured into a CUDA graph and replayed; the
                               host learns the parity only at hg_sync */
  int autotune;             /* 0 (default): launch shapes from a fixed rule; 1:
                               hg_create_ex times candidate shapes (elements
                               per lane, CTAs, prefetch) of hg_gather for every
                               served row count on the device and keeps the
                               fastest (hg_gather_stats keeps the fixed rule)
                               (the fixed rule's shape unless another is
                               faster by at least 3 %, in the sweep and again
                               head to head). The
                               candidates honour the fields above that are
                               set. The timed calls rotate over inputs and
                               outputs in a zero-filled pool of max(256 MB,
                               tp * M * (W + tp * W) * 2 bytes) that is freed
                               before returning; row counts above 16, and those
                               whose one set would exceed 1 GB, keep the fixed
                               rule. It costs
                               tens of milliseconds per served row count at the
                               decode sizes and changes no result, only speed */
  int timeline_calls;       /* 0 (default): off; n > 0: a measurement build of
                               the gather records, for each of the last n
                               calls of hg_gather, hg_gather_stats and
                               hg_gather_fused, per CTA when it started, when
                               its wait for the previous kernel returned and
                               when each warp finished (hg_timeline). Needs shard_cols % 8 == 0,
                               tp <= 16 and no prefetch; it costs a few stores
                               per CTA and changes no result */
} hg_options;

/*
 * hg_create - allocate and arm the mailboxes of one gather
 * (HeadGather.__init__: LamportRows(group, device, (2, cap, words * tp),
 * PAIR_SENT), parity = 0, device synchronised before returning).
 *
 *   tp          virtual ranks, 1 <= tp <= HG_MAX_TP
 *   shard_cols  W, BF16 columns per rank; even (W % 8 == 0 selects the 16-byte
 *               vector path, other even W a 4-byte word path)
 *   cap         mailbox rows per parity, >= max(rows)
 *   rows        the served row counts, each in [1, cap] (HeadGather's `rows`);
 *               NULL with nrows == 0 serves every M in [1, cap]
 *   out         receives the handle
 *
 * Allocates, on the current device, tp mailboxes of 2 * cap * tp * W BF16
 * each (parity-major, then row, then column) plus a status word, fills every
 * mailbox word with 0x80000000 and synchronises the device. The handle owns
 * that memory until hg_destroy. Errors: HG_ERR_ARG (bad sizes, rows out of
 * range, size overflow), HG_ERR_CUDA (no device, allocation failure).
 */
int hg_create(int tp, int shard_cols, int cap, const int *rows, int nrows, hg_handle **out);

/* hg_create with settings; opt may be NULL. Same contract as hg_create. */
int hg_create_ex(int tp, int shard_cols, int cap, const int *rows, int nrows,
                 const hg_options *opt, hg_handle **out);

/* Free the mailboxes and the handle; waits for the device first. NULL is a
 * no-op. Always returns HG_OK unless freeing fails (HG_ERR_CUDA).
 * The pages have no counterpart: HeadGather's mailbox lives as long as the
 * model that installed it. */
int hg_destroy(hg_handle *h);

/*
 * hg_gather - one gather call (HeadGather.__call__ and the kernel of the module
 * docstring): push, poll, copy, re-arm, for every virtual rank, in one
 * persistent kernel launch on `stream`. Asynchronous.
 *
 *   shard_ptrs  tp device pointers; shard_ptrs[r] is rank r's [M, W] BF16
 *               shard, row-major, rows contiguous (row stride W); 16-byte
 *               aligned on the vector path, 4-byte aligned otherwise; read only
 *   out_ptrs    tp device pointers; out_ptrs[d] is rank d's [M, tp * W] BF16
 *               output, row-major, fully overwritten; same alignment rule; must
 *               not overlap a shard or another output
 *   M           rows this call; must be a served row count
 *   stream      the stream every gather of this handle runs on
 *
 * Uses parity hg_parity(h), then flips it. The caller owns the shards and the
 * outputs; the library owns the mailboxes.
 *
 * The launch may start while the previous kernel on `stream` still runs (a
 * programmatic dependent launch). Before it waits for that kernel to
 * complete, each CTA asks L2 to prefetch the first bytes of shard it will
 * read (on the vector path). That is a cache hint only: every value the
 * gather reads is read after the previous kernel has completed, so the
 * shards may be that kernel's output.
 *
 * Co-residency: the kernel's CTAs wait on one another's pushes, so its whole
 * grid must become resident. The grid is sized for an otherwise idle GPU.
 * Kernels running concurrently on other streams can hold SM resources and
 * keep part of the grid from starting until they release them; the call is
 * delayed that long, and if that exceeds the poll bound (for example a
 * persistent kernel on another stream, including another gather: two gathers
 * on different streams can each hold the slots the other needs) it reports
 * HG_ERR_TIMEOUT at hg_sync.
 * Issue such work on the same stream, or create the handle with
 * hg_options.cooperative = 1, where the runtime itself guarantees
 * co-residency (at the cost of the launch overlap). Errors, all before any device work
 * and with no parity flip: HG_ERR_ARG (NULL handle or pointer, misaligned
 * pointer), HG_ERR_ROWS (M not served), HG_ERR_CAPTURE (stream capturing,
 * unless the handle has device_parity), HG_ERR_CUDA (launch failed; parity
 * not flipped). A poll that times out on the
 * device is reported by the next hg_sync; until hg_rearm every later gather
 * of the handle does no device work.
 */
int hg_gather(hg_handle *h, const void *const *shard_ptrs, void *const *out_ptrs, int M,
              hg_stream_t stream);

/*
 * hg_gather_host - hg_gather whose shards and outputs may live in page-locked
 * host memory (cudaHostAlloc, cudaMallocHost or cudaHostRegister), as well as
 * in device memory of the handle's device. The pages define the gather on
 * device buffers only; this entry point is this library's end-to-end form for
 * a host that holds the logits: the same kernel reads the shards from host
 * memory and writes the outputs into host memory directly over the
 * host-device link (no staging copies), while the mailboxes stay in device
 * memory. Same arguments, contract and errors as hg_gather, plus:
 *
 *   no L2 prefetch of the shards before the wait (the host may still be
 *   writing them);
 *   every pointer is checked with cudaPointerGetAttributes and replaced by its
 *   device-side address; pageable host memory, memory of another device and
 *   unknown addresses give HG_ERR_ARG before any device work.
 *
 * The outputs are complete in host memory once the stream has passed the
 * call (e.g. after hg_sync or a stream synchronisation).
 */
int hg_gather_host(hg_handle *h, const void *const *shard_ptrs, void *const *out_ptrs, int M,
                   hg_stream_t stream);

/* Wait for `stream`, then read the device status word. Returns HG_OK,
 * HG_ERR_TIMEOUT (a poll gave up; mailbox contents undefined until hg_rearm)
 * or HG_ERR_CUDA. Failure detection of this library; the pages have no
 * counterpart (their polls are unbounded). */
int hg_sync(hg_handle *h, hg_stream_t stream);

/* Recovery after an error: refill every mailbox word of both parities with
 * the sentinel, re-arm the statistics cells and the fused producer's split
 * cells, clear the status words and set the parity to 0 (host and device
 * copies), on `stream`, asynchronously. It restores the state that
 * HeadGather.__init__ leaves (mailboxes armed with PAIR_SENT, parity 0);
 * recovery itself has no counterpart on the pages. */
int hg_rearm(hg_handle *h, hg_stream_t stream);

/* Parity the next hg_gather uses (0 or 1; starts at 0, flips per served call
 * as `self.parity ^= 1` in HeadGather.__call__), or -1 for NULL. With
 * device_parity, the parity as of the last hg_sync or hg_rearm. */
int hg_parity(const hg_handle *h);

/* Rank `rank`'s mailbox for inspection: device pointer to [2][cap][tp * W]
 * BF16 (parity-major) and its size in bytes. Owned by the handle; read it only
 * while no gather is in flight. Errors: HG_ERR_ARG. Test surface: the layout
 * is that of LamportRows(group, device, (2, cap, words * tp), PAIR_SENT) in
 * HeadGather.__init__, but the pages expose no accessor. */
int hg_mailbox(const hg_handle *h, int rank, const void **dev_ptr, size_t *bytes);

/* Launch shape that hg_gather uses for row count M: CTAs, threads per CTA,
 * elements per lane and whether the next push's shard loads are issued one
 * iteration ahead (1) or not (0). Any output pointer may be NULL. Errors:
 * HG_ERR_ARG, HG_ERR_ROWS. Inspection only; the pages' counterpart,
 * gather_ctas(m, ...) in HeadGather.__init__, is named but not printed. */
int hg_launch_shape(const hg_handle *h, int M, int *ctas, int *threads, int *elems_per_lane,
                    int *prefetch);

/* One CTA's record in the timeline of hg_options.timeline_calls: %globaltimer
 * nanoseconds at entry (before the kernel waits for the previous kernel on
 * the stream), once that wait returned, and when warp d finished (d < tp;
 * warps of CTAs that gave up record nothing); for tp <= 14, warp_done[14]
 * holds instead the index of the SM the CTA ran on. In hg_gather_stats calls with
 * tp < 16, warp_done[15] holds when warp 0 finished its share of the gather
 * and turned to reducing the statistics of its rows, and for tp <= 8 warp 0
 * also records in warp_done[8..12]: its first poll complete, its first
 * outputs stored, its first unit folded, and (CTAs g < M, reducing row g) all
 * of row g's cells arrived and folded, and row g's statistics written. hg_gather_fused calls
 * (one CTA per SM; recorded when the handle's grid records have room for it)
 * use the same slots differently: entry; set-up done (tensor memory and
 * barriers ready); warp_done[i] (i < 8): the epilogue has pushed its item i;
 * warp_done[8 + j] (j < 6): it has consumed the neighbour CTA's item j inside
 * its loop; warp_done[14]: the epilogue loop is done; warp_done[15]: the CTA
 * is done. */
#define HG_TIMELINE_SLOTS 18
typedef struct hg_timeline_record {
  uint64_t entry;
  uint64_t waited;
  uint64_t warp_done[HG_TIMELINE_SLOTS - 2];
} hg_timeline_record;

/*
 * hg_timeline - the timeline of a handle created with timeline_calls = n:
 * device pointer to [n][ctas] hg_timeline_record (ctas = the largest grid of
 * any served row count; a call of a smaller grid fills its first CTAs), and
 * the index of the record the next call writes (calls fill records 0, 1, ...
 * in call order and wrap around after n). Read it only while no gather of the
 * handle is in flight. A measurement surface with no counterpart on the
 * pages. Errors: HG_ERR_ARG (NULL, or a handle without a timeline).
 */
int hg_timeline(const hg_handle *h, const hg_timeline_record **dev_ptr, int *calls, int *ctas,
                int *next);

/*
 * hg_probe - measurement kernels that bound the gather's latency from below;
 * no counterpart on the pages. Both are launched as the gather is (a
 * programmatic dependent launch of `ctas` CTAs of `threads` threads, a
 * multiple of 32, at most 512) on `stream`:
 *
 *   kind 0  empty: wait for the previous kernel, let the next one launch,
 *           return. The cost of one dependent launch of that grid.
 *   kind 1  handoff: warp w of CTA g stores one 16-byte vector per lane into
 *           its slot, lets the next kernel launch, polls the slot of CTA
 *           g + 1 (mod ctas) until it arrives (relaxed loads, bounded by 1 s),
 *           stores it to an output and re-arms that slot: the gather's push,
 *           poll, copy and re-arm for one vector per lane and no shard read.
 *
 *   scratch  device buffer of hg_probe_scratch_bytes(ctas, threads) bytes,
 *            16-byte aligned, owned by the caller; kind 1 needs it armed by
 *            kind 2 (fill the slots with the sentinel, clear the status word)
 *            once before its first launch, and leaves it armed; the status
 *            word (the last 4 bytes) becomes 1 if a poll gave up.
 *
 * Errors: HG_ERR_ARG (kind, sizes, NULL or misaligned scratch), HG_ERR_CUDA.
 */
int hg_probe(int kind, int ctas, int threads, void *scratch, hg_stream_t stream);

/* Bytes of the scratch buffer of hg_probe for that grid. */
size_t hg_probe_scratch_bytes(int ctas, int threads);

/*
 * Test hook for failure detection: make rank `rank`'s push skip its rows in
 * every later gather, plain, with statistics or fused (the fused producer
 * still computes and optionally stores that rank's logits) (rank = -1 turns
 * it off). The pollers of the other ranks
 * then wait for words that never arrive and give up after the poll bound;
 * hg_sync reports HG_ERR_TIMEOUT. No device fault, trap or endless wait is
 * involved. Errors: HG_ERR_ARG. No counterpart on the pages.
 */
int hg_debug_skip_push(hg_handle *h, int rank);

/*
 * hg_gather_fused - the vocab-parallel LM head and the gather in one kernel
 * (API page, module docstring: the lm_head's [M, V / TP] logits per rank, then
 * the gather). For every rank r:
 *   logits_r[m][n] = bf16_rn(sum_k hidden_r[m][k] * weight_r[n][k])
 * with fp32 accumulation on the tensor cores; the GEMM's epilogue pushes the
 * bf16 words straight into every rank's mailbox (sentinel rewrite included),
 * and the same launch polls, copies to out_ptrs and re-arms, exactly as
 * hg_gather does on those logits. Asynchronous on `stream`; uses parity
 * hg_parity(h), then flips it.
 *
 *   hidden_ptrs  tp device pointers to [M, K] bf16, row-major, 16-byte aligned
 *   weight_ptrs  tp device pointers to [W, K] bf16 (nn.Linear layout: vocab
 *                rows, hidden columns), row-major, 16-byte aligned
 *   logits_ptrs  NULL, or tp device pointers (each may be NULL) that receive
 *                rank r's bf16 logits [M, W] as computed (before the rewrite)
 *   out_ptrs     tp device pointers to [M, tp * W] bf16, as for hg_gather
 *   M            rows: served by the handle and <= 16
 *   K            hidden size: a positive multiple of 64
 *
 * Requires tp <= 16 and W a multiple of 128. One CTA per SM (a cooperative
 * launch; hg_options.ctas caps the grid). When the vocab tiles do not divide
 * evenly over the CTAs, the last tiles are split along K over several CTAs,
 * whose fp32 partials meet in the handle's split cells; the sum of the parts
 * may round differently from one accumulation over K (fp32), which the
 * logits tolerance covers, and the gathered outputs are always exactly the
 * gather of the returned logits. Errors, before any device work and with no
 * parity flip: HG_ERR_ARG, HG_ERR_ROWS, HG_ERR_CAPTURE, HG_ERR_STATE,
 * HG_ERR_CUDA (launch or tensor-map encoding failed). A wait that times out is
 * reported by hg_sync, as for hg_gather; hg_rearm also re-arms the split
 * cells.
 */
int hg_gather_fused(hg_handle *h, const void *const *hidden_ptrs, const void *const *weight_ptrs,
                    void *const *logits_ptrs, void *const *out_ptrs, int M, int K,
                    hg_stream_t stream);

/*
 * hg_stock_gather - the baseline without a mailbox: the rank-order concat of
 * NCCL's all-gather (the page's stock LogitsProcessor gather: all-gather into
 * [TP, M, V / TP], then a copy to [M, V]) done as tp * tp cudaMemcpy2DAsync
 * copies on `stream`. Moves every word unchanged (no sentinel rewrite).
 * Pointers and layouts as in hg_gather (no alignment rule beyond 2 bytes).
 * Errors: HG_ERR_ARG, HG_ERR_CUDA.
 */
int hg_stock_gather(int tp, int shard_cols, const void *const *shard_ptrs,
                    void *const *out_ptrs, int M, hg_stream_t stream);

/* Largest mailbox that one hg_gather_static call may use, in bytes:
 * tp * M * tp * shard_cols * 2 (every rank's [M, V] BF16 rows, one parity).
 * At TP8, V=163840 (shard_cols 20480) that is up to M = 9 rows. */
#define HG_STATIC_MAILBOX_BYTES (24u * 1024u * 1024u)

/*
 * hg_gather_static - hg_gather for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point: their gather always owns a
 * mailbox allocated at construction.
 *
 * Some callers cannot call cudaMalloc: a serving engine whose caching
 * allocator has already reserved the GPU's free memory, a plug-in inside a
 * host framework that forbids allocations outside its own allocator, or a
 * latency-critical loop that cannot pay for cudaMalloc/cudaFree's implicit
 * device synchronisation. This call allocates nothing. Its mailbox and status
 * words live in a fixed __device__ array inside the library
 * (HG_STATIC_MAILBOX_BYTES + 256 bytes), which every GPU that loads the
 * library holds until the process exits.
 *
 *   tp, shard_cols  as for hg_create (1 <= tp <= HG_MAX_TP, shard_cols even)
 *   shard_ptrs      tp device pointers to [M, shard_cols] BF16, as for hg_gather
 *   out_ptrs        tp device pointers to [M, tp * shard_cols] BF16, as for
 *                   hg_gather
 *   M               rows, >= 1, with tp * M * tp * shard_cols * 2 <=
 *                   HG_STATIC_MAILBOX_BYTES
 *   status_out      optional device pointer to one int32 that receives, in
 *                   stream order, 0 on success or 1 if a poll gave up; NULL: not
 *                   reported
 *   stream          the stream of the call
 *
 * Same result as hg_gather on the same shards. The call works on the device
 * that is current when it is made: `stream` and every pointer must belong to
 * that device (a stream of another device gives HG_ERR_ARG). The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current), so make that first call before any stream capture. Every call
 * shares the array and finds it as the previous call left it: each call clears
 * the status words and re-arms its mailbox region before gathering, on
 * `stream`. Calls whose device work overlaps (other streams or threads) race on
 * the array. No parity state is kept. Errors, before any device work:
 * HG_ERR_ARG (bad sizes, NULL or misaligned pointers, a mailbox larger than
 * HG_STATIC_MAILBOX_BYTES, or a stream of another device), HG_ERR_CUDA
 * (device lookup or launch failed).
 */
int hg_gather_static(int tp, int shard_cols, const void *const *shard_ptrs,
                     void *const *out_ptrs, int M, int *status_out, hg_stream_t stream);

/* Sampler statistics of one gathered row (over its V bf16 values x_c). */
typedef struct hg_row_stats {
  float max_logit;  /* max_c x_c */
  int argmax;       /* smallest c with x_c == max_logit */
  float sum_exp;    /* sum of exp(x_c - max_logit) over x_c != -inf */
  float logsumexp;  /* max_logit + log(sum_exp) */
} hg_row_stats;

/*
 * hg_gather_stats - hg_gather plus sampler statistics of every gathered row,
 * folded where each unit is pushed and reduced per row inside the same kernel. The API page's module docstring
 * notes that the sentinel rewrite leaves every value a sampler uses
 * unchanged, so these are the sampler's statistics of the gathered row. Same
 * arguments, contract and errors as hg_gather (tp <= 16), plus
 *
 *   stats  device pointer to M hg_row_stats, written in stream order: for
 *          row m, over its V = tp * W bf16 values x_c (rank-order columns),
 *          max_logit = max x_c, argmax = the smallest c attaining it,
 *          sum_exp = sum of exp(x_c - max_logit) over x_c != -inf (fp32,
 *          any summation order), logsumexp = max_logit + log(sum_exp).
 *          Rows holding NaN or +inf give unspecified statistics.
 */
int hg_gather_stats(hg_handle *h, const void *const *shard_ptrs, void *const *out_ptrs, int M,
                    hg_row_stats *stats, hg_stream_t stream);

/* Human-readable text of a status code; never NULL. No counterpart on the
 * pages (HeadGather reports failures as Python exceptions). */
const char *hg_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* HG_H_ */
