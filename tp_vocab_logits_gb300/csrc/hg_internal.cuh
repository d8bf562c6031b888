// Internal declarations shared by the gather library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "hg.h"

namespace hg {

// Sentinel word: the BF16 pair (+0, -0), +0 in the low half (column 2k), -0 in
// the high half (column 2k+1); a data word equal to it is sent as (+0, +0).
// (vLLM API page "...runtime.logits_gather", module docstring.)
constexpr uint32_t kSentinel = 0x80000000u;
constexpr uint32_t kSentAs = 0x00000000u;

// Device status block. status[0]: kDevOk or kDevTimeout; status[1..3]: where
// a poll gave up (unit index, consumer rank, first word offset).
enum DevStatus : int { kDevOk = 0, kDevTimeout = 1 };
constexpr int kStatusWords = 8;

// Row statistics of one unit's values (max, first argmax, sum of exp(x -
// max)), 16 bytes. The cells are Lamport cells: armed with the
// sentinel in every word, written with relaxed stores (a word equal to the
// sentinel written as zero, as in the gather), polled and re-armed by the
// row's reducer (warp 0 of CTA m mod G for row m).
struct RowPartial {
  float max;
  int arg;
  float sum;
  int mark;  // 1 once written
};

// Arguments of one gather launch. Element = 16-byte vector (vector path) or
// one 32-bit word (word path).
struct GatherArgs {
  const void* shard[HG_MAX_TP];  // rank r's [M][wv] elements
  void* out[HG_MAX_TP];          // rank d's [M][tp * wv] elements
  void* box[HG_MAX_TP];          // rank d's mailbox, parity in use: [cap][tp * wv]
  int* status;                   // device status words (kStatusWords)
  unsigned long long timeout_ns;
  int tp;
  int wv;         // elements per rank-row
  int M;          // rows of this call
  int chunks;     // units per rank-row: ceil(wv / (32 * vpt)), or a balanced count
  // Balanced chunks (chunk_q > 0): chunk c of a rank-row holds chunk_q
  // elements, plus one for c < chunk_r (chunk_q = wv / chunks, chunk_r = wv %
  // chunks), at most 32 * vpt; chunk_q = 0: chunks of 32 * vpt elements, the
  // last one ragged.
  int chunk_q = 0;
  int chunk_r = 0;
  int skip_rank;  // test hook: rank whose push is skipped (-1: none)
  // Device-resident parity: nullptr when box[] already points at the parity in
  // use. Otherwise box[] points at parity 0, parity p adds p * parity_stride
  // elements, and parity_words holds parity_entries copies of the parity.
  // Warp d of CTA g reads copy g * tp + d; when done it flips copies
  // g * tp + d + k * G * tp, so every copy flips exactly once per call for any
  // grid size, with no coordination between CTAs.
  int* parity_words = nullptr;
  int parity_entries = 0;
  size_t parity_stride = 0;
  // Row statistics (kernels built with them only): one cell per unit, the [M]
  // output, and the shard width in bf16 columns.
  RowPartial* partials = nullptr;
  hg_row_stats* stats = nullptr;
  int shard_cols = 0;
  // When the next kernel on the stream may start launching: 0 early (once the
  // first loads are issued), 1 late (once each warp's work is done).
  int late_trigger = 0;
  // 1: before waiting on the previous kernel, each CTA prefetches its first
  // push unit of the shards into L2 (shards in device memory only).
  int l2_prefetch = 0;
  // Timeline record of this call (kernels built with it only): CTA g writes
  // %globaltimer readings into timeline[g * kTimelineSlots + k]: k = 0 at
  // entry, 1 once the wait for the previous kernel has returned, 2 + d when
  // warp d has finished (the statistics reducer included).
  unsigned long long* timeline = nullptr;
};

// 64-bit slots of one CTA's timeline record (entry, after the wait, one end
// time per warp for up to 16 warps).
constexpr int kTimelineSlots = 2 + 16;

// Launch shape of one row count: CTAs (32 * tp threads each), elements per lane
// per unit, and whether the next push's shard loads are issued one iteration
// ahead.
struct LaunchShape {
  int ctas = 0;
  int vpt = 1;
  bool pref = false;
  bool stats = false;  // the kernel also folds row statistics
  bool late = false;   // trigger the next launch late (see trigger_late)
  bool timeline = false;  // the kernel writes a timeline record (16-byte vector
                          // path, tp <= 16, no prefetch)
  bool balanced = false;  // balanced chunks (GatherArgs::chunk_q); tuner candidates only
};

// The kernel indexes units with int: a CTA's push index t * G + g runs up to
// N + 3G (the shard loads of iteration t + 1 included), so a launch of N units
// on at most max_ctas CTAs must keep N + 3 * max_ctas within int.
inline bool units_fit_int(long long units, long long max_ctas) {
  return units + 3 * max_ctas <= 0x7fffffffLL;
}

// When to let the next kernel on the stream start launching, for a grid of
// `ctas` CTAs that loops over `units` units with at most `max_ctas`
// co-resident: early (the next grid fits beside this one, or this launch runs
// many iterations) or late, once each warp's work is done (the next grid
// cannot fit beside this one and this launch is short: launched early, its
// CTAs would take the free slots unevenly). Measured at TP8, V=163840: M=2
// 4.33 us late against 4.97 early, M=4 6.48 against 6.95, M=1 (early) 3.29
// against 3.41, M=64 (early) 91.0 against 93.6.
inline bool trigger_late(long long ctas, long long units, long long max_ctas) {
  const long long iters = (units + ctas - 1) / ctas;
  return 2 * ctas > max_ctas && iters <= 4;
}

// Elements per lane a gather kernel exists for: 1..6 for tp <= 16, 1..2 above.
inline int max_vpt(int tp) { return tp <= 16 ? 6 : 2; }

// Elements per lane of the fixed launch rule for M rows: 3 for up to three rows
// at tp <= 8, where the call is latency-bound and smaller units put more
// CTAs in flight; 4 otherwise (2 for tp > 16, whose CTAs have 1024 threads).
// Graph-replayed at TP8, V=163840, M=3: 4.88 us with 3 (608 CTAs) against 5.21
// with 4 (480 CTAs). From four rows on the host may widen the units when that
// leaves the busiest SM fewer vectors to move (widen_units).
inline int default_vpt(int tp, int M) {
  if (tp > 16) return 2;
  return (tp <= 8 && M <= 3) ? 3 : 4;
}

// Elements per lane of the statistics kernel (tp <= 16) for M rows: 3 up to
// eight rows at tp <= 8, where the smaller units shorten each unit's fold and
// the reducer still polls a row's cells in one wait; 4 otherwise. (TP8,
// V=163840, M=1: 3.79 us graph-replayed, against 3.91 / 4.24 / 4.80 us with 4 /
// 5 / 6 elements per lane and 4.46 us with 2; M=8: 10.87 us against 11.15 / 11.51
// with 4 / 5; M=7: 9.84 against 10.10 / 10.42 / 12.08 with 4 / 5 / 6.)
inline int stats_vpt(int tp, int M) { return (tp <= 8 && M <= 8) ? 3 : 4; }

// Largest co-resident CTAs per SM of the gather kernel for this shape.
cudaError_t gather_occupancy(const LaunchShape& s, bool vec16, int tp, int* ctas_per_sm);

// The fixed rule's unit widening (hg_lib.cu): from four rows on, for launches
// of at most four rounds, replace *s (the default width's shape: vpt, ctas,
// late) and *chunks with the width whose busiest SM moves the fewest vectors.
cudaError_t widen_units(int tp, int wv, int M, int sms, bool vec16, LaunchShape* s,
                        int* chunks);

// Launch of the gather kernel. cooperative: the runtime guarantees that all
// CTAs are co-resident (or fails the launch); otherwise a programmatic
// dependent launch (the kernel waits for its predecessor before any access).
cudaError_t launch_gather(const GatherArgs& a, const LaunchShape& s, bool vec16,
                          cudaStream_t stream, bool cooperative);

// Fill n 32-bit words with v.
cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t v, cudaStream_t stream);

namespace fused {

// Largest TP of the fused producer (its kernel argument block holds two tensor
// maps per rank).
constexpr int kFusedMaxTp = 16;

// Kernel arguments of the fused LM-head producer + gather.
struct FusedArgs {
  CUtensorMap tm_w[kFusedMaxTp];  // rank r's weight [W, K] bf16, box [128, 64]
  CUtensorMap tm_h[kFusedMaxTp];  // rank r's hidden [M, K] bf16, box [16, 64]
  void* box[kFusedMaxTp];         // rank d's mailbox, parity in use: [cap][V] bf16
  void* out[kFusedMaxTp];         // rank d's output [M][V] bf16
  void* logits[kFusedMaxTp];      // optional: rank r's bf16 logits [M][W] (nullptr: none)
  int* status;                    // device status words
  unsigned long long timeout_ns;
  int tp, W, K, M;
  int tiles_per_rank;             // W / 128
  // Device-resident parity (see GatherArgs): box[] then points at parity 0 and
  // parity p adds p * parity_stride_words 32-bit words; CTA g reads copy g and
  // flips copies g + k * G.
  int* parity_words;
  int parity_entries;
  size_t parity_stride_words;
  // Work split: every CTA takes full_waves whole tiles (tiles g + k * G);
  // the `tail` remaining tiles are split along K into `split` parts (split
  // 1: tail tile j is taken whole by CTA j). Part p of tail tile j runs on
  // CTA j * split + p; parts 1.. hand their fp32 partials to part 0 through
  // split_cells ([tail][split - 1][128 rows][16] words, armed with
  // kSplitArmed).
  int full_waves;
  int tail;
  int split;
  uint32_t* split_cells;
  int skip_rank;  // test hook: rank whose mailbox pushes are skipped (-1: none)
  // Timeline record of this call (nullptr: none): CTA g writes %globaltimer
  // readings into timeline[g * kTimelineSlots + k] (see kFusedTl*).
  unsigned long long* timeline;
};

// Slots of a fused call's timeline record per CTA: entry, set-up done (TMEM
// allocated, barriers ready), item i pushed by the epilogue (i < 8), the
// neighbour's item j consumed inside the epilogue loop (j < 6), the
// epilogue loop done, the CTA done.
constexpr int kFusedTlEntry = 0, kFusedTlSetup = 1, kFusedTlPush = 2, kFusedTlPushN = 8,
              kFusedTlConsume = 10, kFusedTlConsumeN = 6, kFusedTlLoopDone = 16,
              kFusedTlDone = 17;

// Armed word of a split cell, and the word a partial with that bit pattern
// is written as (both NaNs).
constexpr uint32_t kSplitArmed = 0xffffffffu;
constexpr uint32_t kSplitArmedAs = 0x7fffffffu;
// Words of one split cell (128 rows x 16 fp32 columns) and the most parts a
// tail tile is split into.
constexpr size_t kSplitCellWords = 128 * 16;
constexpr int kMaxSplit = 4;

// Host-side description of one fused call.
struct FusedLaunch {
  const void* const* hidden;  // tp device pointers, [M, K] bf16
  const void* const* weight;  // tp device pointers, [W, K] bf16
  void* const* logits;        // nullptr, or tp device pointers (entries may be nullptr)
  void* box[HG_MAX_TP];
  void* const* out;
  int* status;
  unsigned long long timeout_ns;
  int tp, W, K, M;
  int* parity_words = nullptr;  // device-resident parity copies (nullptr: box[] resolved)
  int parity_entries = 0;
  size_t parity_stride_words = 0;
  uint32_t* split_cells = nullptr;  // armed split cells (nullptr: tail tiles are not split)
  size_t split_cell_count = 0;      // cells available (each kSplitCellWords words)
  int max_ctas = 0;                 // cap on the grid (0: one CTA per SM)
  int skip_rank = -1;               // test hook: rank whose pushes are skipped
  unsigned long long* timeline = nullptr;  // record of this call (nullptr: none)
  int timeline_ctas = 0;                   // CTAs the record has room for
};

// Limits of the fused path: TP, rows, K granularity, W granularity.
int fused_limits(int* max_tp, int* max_m, int* k_multiple, int* w_multiple);

// Cooperative launch of the fused kernel (one CTA per SM at most).
cudaError_t fused_launch(const FusedLaunch& l, cudaStream_t stream, int sms);

// Split cells a handle needs for any fused call on a device with `sms` SMs.
size_t split_cells_needed(int sms);

}  // namespace fused

}  // namespace hg
