// Host side of the C ABI declared in include/hg.h: handle, mailboxes, parity,
// argument checks, launch shapes and the stock baseline.
//
// The per-call logic follows HeadGather (vLLM API page "vllm.models.kimi_k3.
// nvidia.specialized_decode.runtime.logits_gather"): unserved row counts and
// graph capture are refused before any state changes (__call__'s eligibility
// test); otherwise the call uses the current parity, flips it, and launches
// one kernel.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "hg_internal.cuh"

struct hg_handle {
  int device = -1;
  int sms = 0;
  int tp = 0;
  int W = 0;       // shard columns
  int wv = 0;      // elements per rank-row (16-byte vectors or words)
  bool vec16 = false;
  int cap = 0;
  std::vector<char> served;  // served[M]
  int parity = 0;
  size_t box_bytes = 0;      // bytes of one rank's mailbox, both parities
  size_t parity_elems = 0;   // elements of one parity of one mailbox
  void* box[HG_MAX_TP] = {};
  int* status = nullptr;     // device status words
  unsigned long long timeout_ns = 1000000000ull;
  int skip_rank = -1;
  bool failed = false;       // hg_sync saw a device error; cleared by hg_rearm
  bool cooperative = false;  // cooperative launch instead of programmatic dependent launch
  bool device_parity = false;  // parity lives on the device; calls may be captured
  int* parity_words = nullptr;  // copies of the device-resident parity
  int parity_entries = 0;
  std::vector<hg::LaunchShape> shape;  // launch shape per M (index M)
  std::vector<int> chunks;             // units per rank-row per M
  std::vector<hg::LaunchShape> shape_stats;  // the same for hg_gather_stats (tp <= 16)
  std::vector<int> chunks_stats;
  hg::RowPartial* partials = nullptr;  // statistics cells: one per unit of the largest call
  size_t partial_count = 0;
  uint32_t* split_cells = nullptr;  // fused calls: split cells of the tail tiles (armed)
  size_t split_cell_count = 0;
  int max_ctas = 0;                 // hg_options.ctas: also caps the fused grid
  unsigned long long* timeline = nullptr;  // [timeline_calls][timeline_ctas] records
  int timeline_calls = 0;
  int timeline_ctas = 0;
  long long timeline_next = 0;      // calls recorded so far
};

namespace hg {

// From four rows on, where the call moves enough bytes that the busiest SM
// sets its time, wider units may load that SM with fewer vectors: CTA i
// takes units i, i + G, ..., and SM j holds CTAs j, j + S, ... (the launch
// spreads CTAs over the SMs in turn). Take the width whose busiest SM moves
// the fewest vectors (ties keep the narrower), for launches of at most four
// rounds. TP8, V=163840, graph-replayed: M=4 6 per lane on 448 CTAs (576
// vectors on the busiest SM against 640 with 4) 5.88 against 6.07-6.11 us;
// M=7 5 per lane (960 against 1024) 9.11 against 9.53-9.56 us; M=8 5 per
// lane (1120 against 1152) 10.36-10.37 against 10.49-10.52 us; M=5 and M=6
// keep 4 (768 and 896, against 800 and 960 with 5: 7.42 and 8.23 against
// 7.01-7.03 and 8.02-8.04 us). Past four rounds five of six sweep points got
// slower. Up to three rows at tp <= 8 the chain of vectors per lane sets the
// time instead, and the narrow rule stays.
cudaError_t widen_units(int tp, int wv, int M, int sms, bool vec16, LaunchShape* s,
                        int* chunks) {
  if (M < 4) return cudaSuccess;
  int per_sm = 0;
  cudaError_t e = gather_occupancy(*s, vec16, tp, &per_sm);
  if (e != cudaSuccess) return e;
  const long long S = sms;
  const long long maxg = (long long)per_sm * S;
  const long long units = (long long)M * tp * *chunks;
  if (per_sm < 1 || units > 4 * maxg) return cudaSuccess;
  auto busiest = [S](long long U, long long Gc, int v) {
    long long worst = 0;
    for (long long j = 0; j < S && j < Gc; ++j) {
      long long load = 0;
      for (long long i = j; i < Gc; i += S) load += (U - 1 - i) / Gc + 1;
      if (load > worst) worst = load;
    }
    return worst * 32LL * v;
  };
  long long best = busiest(units, units < maxg ? units : maxg, s->vpt);
  const LaunchShape base = *s;
  for (int v = base.vpt + 1; v <= max_vpt(tp); ++v) {
    LaunchShape c = base;
    c.vpt = v;
    int pv = 0;
    if (gather_occupancy(c, vec16, tp, &pv) != cudaSuccess || pv < 1) continue;
    const long long mv = (long long)pv * S;
    const int cv = (wv + 32 * v - 1) / (32 * v);
    const long long uv = (long long)M * tp * cv;
    if (!units_fit_int(uv, mv)) continue;
    const long long gv = uv < mv ? uv : mv;
    const long long load = busiest(uv, gv, v);
    if (load < best) {
      best = load;
      c.ctas = (int)gv;
      c.late = trigger_late(gv, uv, mv);
      *s = c;
      *chunks = cv;
    }
  }
  return cudaSuccess;
}

}  // namespace hg

namespace {

using hg::GatherArgs;

constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

void free_handle(hg_handle* h) {
  if (!h) return;
  for (int d = 0; d < HG_MAX_TP; ++d)
    if (h->box[d]) cudaFree(h->box[d]);
  if (h->status) cudaFree(h->status);
  if (h->parity_words) cudaFree(h->parity_words);
  if (h->partials) cudaFree(h->partials);
  if (h->split_cells) cudaFree(h->split_cells);
  if (h->timeline) cudaFree(h->timeline);
  delete h;
}

// Range checks of the launch-shape options.
int check_shape_options(const hg_handle* h, const hg_options* opt) {
  if (!opt) return HG_OK;
  const int v = opt->elems_per_lane;
  if (v < 0 || v > hg::max_vpt(h->tp) || opt->ctas < 0 || opt->prefetch < 0 ||
      opt->prefetch > 2)
    return HG_ERR_ARG;
  if (opt->autotune < 0 || opt->autotune > 1) return HG_ERR_ARG;
  if (opt->timeline_calls < 0) return HG_ERR_ARG;
  if (opt->timeline_calls > 0 && (!h->vec16 || h->tp > 16 || opt->prefetch == 1))
    return HG_ERR_ARG;
  return HG_OK;
}

// Co-resident CTAs of shape s on the whole device.
int max_grid(const hg_handle* h, const hg::LaunchShape& s, long long* g) {
  int per_sm = 0;
  if (hg::gather_occupancy(s, h->vec16, h->tp, &per_sm) != cudaSuccess || per_sm < 1)
    return HG_ERR_CUDA;
  *g = (long long)per_sm * h->sms;
  return HG_OK;
}

// Launch shape for M rows by the fixed rule, unless the options force part of
// it: one CTA = one warp per virtual rank; each lane carries default_vpt(tp, M)
// elements (3 for up to three rows at tp <= 8, 4 otherwise, 2 for CTAs of 1024
// threads; the statistics kernel: stats_vpt), widened from four rows on when
// that leaves the busiest SM fewer vectors (widen_units); one CTA per unit up
// to the co-resident maximum, beyond which the CTAs loop over the units; no
// prefetch.
// The best shape depends on tp, W and M in ways no simple rule captures, so
// hg_options.autotune can time the candidates instead. The grid never exceeds
// the co-resident CTA count, which the kernel's cross-CTA polls need.
int plan_one(hg_handle* h, int M, const hg_options* opt, bool stats, hg::LaunchShape* out,
             int* chunks_out) {
  const int forced_vpt = opt ? opt->elems_per_lane : 0;
  const int forced_ctas = opt ? opt->ctas : 0;
  hg::LaunchShape s;
  s.stats = stats;
  // The statistics kernel has its own rule: its reducer polls one cell per
  // unit (TP8, V=163840: 3 per lane measured 6.1-6.2 us at M=1 and 14.8 us at
  // M=8, against 6.5 and 15.6 us with 4).
  s.vpt = forced_vpt ? forced_vpt : (stats ? hg::stats_vpt(h->tp, M) : hg::default_vpt(h->tp, M));
  s.pref = opt && opt->prefetch == 1;
  const int chunks = (h->wv + 32 * s.vpt - 1) / (32 * s.vpt);
  const long long units = (long long)M * h->tp * chunks;
  if (units > 0x7fffffffLL) return HG_ERR_ARG;
  long long want = forced_ctas ? forced_ctas : units;
  if (want > units) want = units;
  long long maxg = 0;
  const int st = max_grid(h, s, &maxg);
  if (st != HG_OK) return st;
  if (!hg::units_fit_int(units, maxg)) return HG_ERR_ARG;
  long long G = want < maxg ? want : maxg;
  if (G < 1) G = 1;
  s.ctas = (int)G;
  s.late = hg::trigger_late(G, units, maxg);
  *out = s;
  *chunks_out = chunks;
  if (!stats && !forced_vpt && !forced_ctas && !s.pref &&
      hg::widen_units(h->tp, h->wv, M, h->sms, h->vec16, out, chunks_out) != cudaSuccess)
    return HG_ERR_CUDA;
  return HG_OK;
}

// Shapes of every served M, for hg_gather and (tp <= 16) hg_gather_stats, and
// the number of statistics cells the largest stats call needs.
int plan_shapes(hg_handle* h, const hg_options* opt) {
  const int chk = check_shape_options(h, opt);
  if (chk != HG_OK) return chk;
  h->shape.assign(h->cap + 1, hg::LaunchShape());
  h->chunks.assign(h->cap + 1, 0);
  h->shape_stats.assign(h->cap + 1, hg::LaunchShape());
  h->chunks_stats.assign(h->cap + 1, 0);
  h->partial_count = 0;
  for (int M = 1; M <= h->cap; ++M) {
    if (!h->served[M]) continue;
    int st = plan_one(h, M, opt, false, &h->shape[M], &h->chunks[M]);
    if (st != HG_OK) return st;
    if (h->tp <= 16) {
      st = plan_one(h, M, opt, true, &h->shape_stats[M], &h->chunks_stats[M]);
      if (st != HG_OK) return st;
      const size_t cells = (size_t)M * h->tp * h->chunks_stats[M];  // one per unit
      if (cells > h->partial_count) h->partial_count = cells;
    }
  }
  return HG_OK;
}

}  // namespace

extern "C" {

namespace {
// Defined below, next to gather_impl, whose calls it times.
int autotune_shapes(hg_handle* h, const hg_options* opt);
}  // namespace

const char* hg_strerror(int status) {
  switch (status) {
    case HG_OK: return "ok";
    case HG_ERR_ARG: return "invalid argument";
    case HG_ERR_ROWS: return "row count not served by this gather";
    case HG_ERR_CAPTURE: return "stream is capturing a CUDA graph";
    case HG_ERR_CUDA: return "CUDA runtime error";
    case HG_ERR_TIMEOUT: return "mailbox poll timed out";
    case HG_ERR_STATE: return "gather holds an unrecovered device error; re-arm it";
    default: return "unknown status";
  }
}

int hg_create_ex(int tp, int shard_cols, int cap, const int* rows, int nrows,
                 const hg_options* opt, hg_handle** out) {
  if (!out) return HG_ERR_ARG;
  *out = nullptr;
  if (tp < 1 || tp > HG_MAX_TP || shard_cols < 2 || shard_cols % 2 != 0 || cap < 1)
    return HG_ERR_ARG;
  if (nrows < 0 || (nrows > 0 && !rows)) return HG_ERR_ARG;
  const long long V = (long long)tp * shard_cols;
  const long long words_per_row = V / 2;
  if (words_per_row > (1LL << 30) || (long long)cap * words_per_row > (1LL << 40))
    return HG_ERR_ARG;

  hg_handle* h = new (std::nothrow) hg_handle;
  if (!h) return HG_ERR_CUDA;
  h->tp = tp;
  h->W = shard_cols;
  h->vec16 = shard_cols % 8 == 0;
  h->wv = h->vec16 ? shard_cols / 8 : shard_cols / 2;
  h->cap = cap;
  h->served.assign(cap + 1, 0);
  if (nrows == 0) {
    for (int m = 1; m <= cap; ++m) h->served[m] = 1;
  } else {
    for (int i = 0; i < nrows; ++i) {
      if (rows[i] < 1 || rows[i] > cap) { delete h; return HG_ERR_ARG; }
      h->served[rows[i]] = 1;
    }
  }
  h->timeout_ns = opt && opt->poll_timeout_ns ? opt->poll_timeout_ns : kDefaultTimeoutNs;
  h->cooperative = opt && opt->cooperative;
  h->device_parity = opt && opt->device_parity;
  h->max_ctas = opt ? opt->ctas : 0;

  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return HG_ERR_CUDA;
  }
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (h->cooperative && !coop) { delete h; return HG_ERR_CUDA; }

  int st = plan_shapes(h, opt);
  if (st != HG_OK) { delete h; return st; }

  // Mailboxes: [2 parities][cap rows][V] bf16 per rank, armed with the sentinel.
  const size_t row_bytes = (size_t)V * 2;
  h->box_bytes = 2 * (size_t)cap * row_bytes;
  h->parity_elems = (size_t)cap * tp * h->wv;
  for (int d = 0; d < tp; ++d) {
    if (cudaMalloc(&h->box[d], h->box_bytes) != cudaSuccess) { free_handle(h); return HG_ERR_CUDA; }
    if (hg::launch_fill_u32(static_cast<uint32_t*>(h->box[d]), h->box_bytes / 4, hg::kSentinel,
                            nullptr) != cudaSuccess) {
      free_handle(h);
      return HG_ERR_CUDA;
    }
  }
  if (h->partial_count) {
    // Statistics cells, armed with the sentinel (Lamport cells).
    if (cudaMalloc(&h->partials, h->partial_count * sizeof(hg::RowPartial)) != cudaSuccess ||
        hg::launch_fill_u32(reinterpret_cast<uint32_t*>(h->partials), h->partial_count * 4,
                            hg::kSentinel, nullptr) != cudaSuccess) {
      free_handle(h);
      return HG_ERR_CUDA;
    }
  }
  {
    // Split cells of the fused producer's tail tiles, armed (handles whose
    // shape the fused call accepts).
    int max_tp = 0, max_m = 0, k_mult = 0, w_mult = 0;
    hg::fused::fused_limits(&max_tp, &max_m, &k_mult, &w_mult);
    if (tp <= max_tp && h->vec16 && shard_cols % w_mult == 0) {
      h->split_cell_count = hg::fused::split_cells_needed(h->sms);
      const size_t words = h->split_cell_count * hg::fused::kSplitCellWords;
      if (cudaMalloc(&h->split_cells, words * sizeof(uint32_t)) != cudaSuccess ||
          hg::launch_fill_u32(h->split_cells, words, hg::fused::kSplitArmed, nullptr) !=
              cudaSuccess) {
        free_handle(h);
        return HG_ERR_CUDA;
      }
    }
  }
  if (cudaMalloc(&h->status, hg::kStatusWords * sizeof(int)) != cudaSuccess ||
      cudaMemset(h->status, 0, hg::kStatusWords * sizeof(int)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    free_handle(h);
    return HG_ERR_CUDA;
  }
  if (opt && opt->autotune) {
    st = autotune_shapes(h, opt);
    if (st != HG_OK) { free_handle(h); return st; }
  }
  if (opt && opt->timeline_calls > 0) {
    // Timeline records: the measurement build of the kernel (no prefetch; the
    // tuner may have chosen it, so it is switched off for these shapes). Its
    // grid must stay co-resident with the measurement build's own occupancy.
    int max_ctas = 0;
    for (int M = 1; M <= cap; ++M) {
      if (!h->served[M]) continue;
      for (int k = 0; k < 2; ++k) {
        hg::LaunchShape& sh = k == 0 ? h->shape[M] : h->shape_stats[M];
        const int chunks = k == 0 ? h->chunks[M] : h->chunks_stats[M];
        sh.pref = false;
        sh.timeline = true;
        long long maxg = 0;
        st = max_grid(h, sh, &maxg);
        if (st != HG_OK) { free_handle(h); return st; }
        if (sh.ctas > maxg) sh.ctas = (int)maxg;
        sh.late = hg::trigger_late(sh.ctas, (long long)M * tp * chunks, maxg);
        max_ctas = std::max(max_ctas, sh.ctas);
      }
    }
    h->timeline_calls = opt->timeline_calls;
    h->timeline_ctas = max_ctas;
    const size_t bytes = (size_t)h->timeline_calls * max_ctas * hg::kTimelineSlots * 8;
    if (cudaMalloc(&h->timeline, bytes) != cudaSuccess ||
        cudaMemset(h->timeline, 0, bytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
      free_handle(h);
      return HG_ERR_CUDA;
    }
  }
  if (h->device_parity) {
    // One copy per reader: warp d of CTA g of a gather reads copy g * tp + d,
    // CTA g of a fused call (at most one CTA per SM) reads copy g.
    int max_ctas = 0;
    for (int M = 1; M <= cap; ++M) {
      if (h->served[M] && h->shape[M].ctas > max_ctas) max_ctas = h->shape[M].ctas;
      if (h->served[M] && h->shape_stats[M].ctas > max_ctas) max_ctas = h->shape_stats[M].ctas;
    }
    h->parity_entries = max_ctas * tp > h->sms ? max_ctas * tp : h->sms;
    if (cudaMalloc(&h->parity_words, (size_t)h->parity_entries * sizeof(int)) != cudaSuccess ||
        cudaMemset(h->parity_words, 0, (size_t)h->parity_entries * sizeof(int)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
      free_handle(h);
      return HG_ERR_CUDA;
    }
  }
  *out = h;
  return HG_OK;
}

int hg_create(int tp, int shard_cols, int cap, const int* rows, int nrows, hg_handle** out) {
  return hg_create_ex(tp, shard_cols, cap, rows, nrows, nullptr, out);
}

int hg_destroy(hg_handle* h) {
  if (!h) return HG_OK;
  int st = cudaDeviceSynchronize() == cudaSuccess ? HG_OK : HG_ERR_CUDA;
  free_handle(h);
  return st;
}

namespace {

// device_shards: the shards are device memory, whose first units the kernel
// may prefetch into L2 before it waits on the previous kernel (not for
// page-locked host memory, which the host may still be writing).
int gather_impl(hg_handle* h, const void* const* shard_ptrs, void* const* out_ptrs, int M,
                hg_row_stats* stats, hg_stream_t stream, bool device_shards) {
  if (!h || !shard_ptrs || !out_ptrs) return HG_ERR_ARG;
  if (stats && (h->tp > 16 || !h->partials)) return HG_ERR_ARG;
  if (M < 1 || M > h->cap || !h->served[M]) return HG_ERR_ROWS;
  if (h->failed) return HG_ERR_STATE;
  const size_t align = h->vec16 ? 16 : 4;
  GatherArgs a;
  for (int r = 0; r < h->tp; ++r) {
    if (!shard_ptrs[r] || !out_ptrs[r] || !aligned(shard_ptrs[r], align) ||
        !aligned(out_ptrs[r], align))
      return HG_ERR_ARG;
    a.shard[r] = shard_ptrs[r];
    a.out[r] = out_ptrs[r];
  }
  if (!h->device_parity) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return HG_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return HG_ERR_CAPTURE;
  }

  const size_t esz = h->vec16 ? 16 : 4;
  const int host_parity = h->device_parity ? 0 : h->parity;
  for (int d = 0; d < h->tp; ++d)
    a.box[d] = static_cast<char*>(h->box[d]) + (size_t)host_parity * h->parity_elems * esz;
  if (h->device_parity) {
    a.parity_words = h->parity_words;
    a.parity_entries = h->parity_entries;
    a.parity_stride = h->parity_elems;
  }
  for (int d = h->tp; d < HG_MAX_TP; ++d) {
    a.shard[d] = nullptr;
    a.out[d] = nullptr;
    a.box[d] = nullptr;
  }
  a.status = h->status;
  a.timeout_ns = h->timeout_ns;
  a.tp = h->tp;
  a.wv = h->wv;
  a.M = M;
  a.chunks = stats ? h->chunks_stats[M] : h->chunks[M];
  if ((stats ? h->shape_stats[M] : h->shape[M]).balanced) {
    a.chunk_q = h->wv / a.chunks;
    a.chunk_r = h->wv % a.chunks;
  }
  a.skip_rank = h->skip_rank;
  a.l2_prefetch = device_shards ? 1 : 0;
  if (stats) {
    a.partials = h->partials;
    a.stats = stats;
    a.shard_cols = h->W;
  }
  const hg::LaunchShape& shape = stats ? h->shape_stats[M] : h->shape[M];
  if (h->timeline)
    a.timeline = h->timeline + (size_t)(h->timeline_next % h->timeline_calls) *
                                   h->timeline_ctas * hg::kTimelineSlots;
  if (hg::launch_gather(a, shape, h->vec16, stream, h->cooperative) != cudaSuccess)
    return HG_ERR_CUDA;
  if (h->timeline) ++h->timeline_next;
  if (!h->device_parity) h->parity ^= 1;
  return HG_OK;
}

// One candidate launch shape of the autotuner.
struct Candidate {
  hg::LaunchShape s;
  int chunks = 0;
  float us = 1e30f;
};

// Candidate shapes of row count M: every allowed (elements per lane,
// prefetch) pair, each on one CTA per unit (capped at the co-resident
// maximum) and on k CTAs per SM for every k below the co-resident count
// that leaves CTAs looping over units. Prefetch only with two or more
// iterations (otherwise it is the same kernel work as without).
int tune_candidates(hg_handle* h, int M, const hg_options* opt, std::vector<Candidate>* out) {
  std::vector<int> vpts;
  if (opt->elems_per_lane) vpts.push_back(opt->elems_per_lane);
  else for (int v = 1; v <= hg::max_vpt(h->tp); ++v) vpts.push_back(v);
  std::vector<bool> prefs;
  if (opt->prefetch == 0 || opt->prefetch == 2) prefs.push_back(false);
  if (opt->prefetch == 0 || opt->prefetch == 1) prefs.push_back(true);
  for (int vpt : vpts) {
    for (bool pref : prefs) {
      Candidate c;
      c.s.vpt = vpt;
      c.s.pref = pref;
      c.chunks = (h->wv + 32 * vpt - 1) / (32 * vpt);
      const long long units = (long long)M * h->tp * c.chunks;
      if (units > 0x7fffffffLL) continue;
      long long maxg = 0;
      const int st = max_grid(h, c.s, &maxg);
      if (st != HG_OK) return st;
      if (!hg::units_fit_int(units, maxg)) continue;
      std::vector<long long> grids;
      if (opt->ctas) {
        long long g = opt->ctas < units ? opt->ctas : units;
        grids.push_back(g < maxg ? g : maxg);
      } else {
        grids.push_back(units < maxg ? units : maxg);
        for (long long g = h->sms; g < maxg && g < units; g += h->sms) grids.push_back(g);
      }
      for (long long g : grids) {
        const long long iters = (units + g - 1) / g;
        if (pref && iters < 2) continue;
        c.s.ctas = (int)g;
        c.s.late = hg::trigger_late(g, units, maxg);
        out->push_back(c);
      }
      // Balanced chunks (one wave, no prefetch, grid not forced): the chunk
      // counts, up to twice the fixed one, for which the units fill a whole
      // number of CTAs per SM, each chunk within 32 * vpt elements. With fixed
      // chunks the grid can leave some SMs with one CTA more than others.
      if (!pref && !opt->ctas) {
        for (long long cc = c.chunks + 1; cc <= 2LL * c.chunks; ++cc) {
          const long long u = (long long)M * h->tp * cc;
          if (u > maxg) break;
          if (u % h->sms != 0 || h->wv / cc < 1) continue;
          Candidate b = c;
          b.chunks = (int)cc;
          b.s.balanced = true;
          b.s.ctas = (int)u;
          b.s.late = hg::trigger_late(u, u, maxg);
          out->push_back(b);
        }
      }
    }
  }
  return HG_OK;
}

// hg_options.autotune: time the candidate shapes of every served row count
// (whose inputs and outputs, one set, stay within kSetLimit) and keep the
// fastest. Timing: calls back to back on a private stream, as a decode loop
// issues them, rotating over as many sets of inputs and outputs as fit in a
// zero-filled pool of at least kPoolBytes (more than twice the L2), so that
// they stream from HBM as in a long run of calls. Each measurement is 2 calls
// of warm-up, then a block of calls timed with events, sized to about
// kBlockUs of device time (4 to 32 calls); three rounds over all candidates,
// interleaved so that a slow stretch of the device does not fall on one
// candidate alone, the fastest block of each candidate kept. The calls gather
// real data through the handle's mailboxes, which every call leaves armed;
// the parity is reset to 0 afterwards.
int autotune_shapes(hg_handle* h, const hg_options* opt) {
  constexpr size_t kSetLimit = 1ull << 30;
  constexpr size_t kPoolBytes = 256ull << 20;
  // Row counts above this keep the fixed rule: tuning pays at decode sizes,
  // and at large row counts the fixed rule is near the memory roofline (TP8,
  // V=163840: 0.97-1.21 of the measured HBM copy rate from M = 32 on).
  constexpr int kMaxTunedRows = 16;
  constexpr float kBlockUs = 300.f;
  constexpr int kRounds = 3;
  constexpr float kMargin = 0.03f;
  constexpr int kConfirm = 4;  // even: the median is the mean of the middle two
  const size_t V = (size_t)h->tp * h->W;
  // One set: tp shards [M][W], then tp outputs [M][V], each 16-byte aligned.
  auto set_bytes = [&](int M) { return (size_t)h->tp * M * (h->W + V) * 2; };
  int maxM = 0;
  for (int M = 1; M <= h->cap && M <= kMaxTunedRows; ++M)
    if (h->served[M] && set_bytes(M) <= kSetLimit) maxM = M;
  if (maxM == 0) return HG_OK;
  const size_t pool_bytes = set_bytes(maxM) > kPoolBytes ? set_bytes(maxM) : kPoolBytes;
  char* pool = nullptr;
  cudaStream_t stream = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  const bool saved_dp = h->device_parity;
  h->device_parity = false;  // host parity while tuning: parity copies do not exist yet
  int rc = HG_OK;
  if (cudaMalloc(&pool, pool_bytes) != cudaSuccess || cudaMemset(pool, 0, pool_bytes) != cudaSuccess ||
      cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    rc = HG_ERR_CUDA;
  std::vector<const void*> shard(h->tp);
  std::vector<void*> out(h->tp);
  int call = 0;
  auto run = [&](int M, const Candidate& c, int calls) {
    h->shape[M] = c.s;
    h->chunks[M] = c.chunks;
    const size_t sb = set_bytes(M);
    const int sets = (int)(pool_bytes / sb);
    for (int i = 0; i < calls; ++i, ++call) {
      char* base = pool + (size_t)(call % sets) * sb;
      for (int r = 0; r < h->tp; ++r) {
        shard[r] = base + (size_t)r * M * h->W * 2;
        out[r] = base + (size_t)h->tp * M * h->W * 2 + (size_t)r * M * V * 2;
      }
      const int st = gather_impl(h, shard.data(), out.data(), M, nullptr, stream, true);
      if (st != HG_OK) return st;
    }
    return (int)HG_OK;
  };
  for (int M = 1; M <= maxM && rc == HG_OK; ++M) {
    if (!h->served[M]) continue;
    std::vector<Candidate> cand;
    rc = tune_candidates(h, M, opt, &cand);
    if (rc != HG_OK) break;
    if (cand.empty()) continue;  // nothing to time (e.g. prefetch forced, one wave): fixed rule
    Candidate fixed;  // the fixed rule's shape, as planned before tuning
    fixed.s = h->shape[M];
    fixed.chunks = h->chunks[M];
    // Time `calls` calls of candidate c (after 2 of warm-up), in us per call.
    auto timed = [&](const Candidate& c, int calls, float* us) {
      int st = run(M, c, 2);
      if (st != HG_OK) return st;
      if (cudaEventRecord(e0, stream) != cudaSuccess) return (int)HG_ERR_CUDA;
      st = run(M, c, calls);
      if (st != HG_OK) return st;
      float ms = 0.f;
      if (cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
        return (int)HG_ERR_CUDA;
      *us = ms * 1000.f / calls;
      return (int)HG_OK;
    };
    if (call == 0) rc = run(M, cand[0], 200);  // clocks up before the first timing
    float est = 0.f;
    if (rc == HG_OK) rc = timed(cand[0], 8, &est);  // block size from the first candidate
    int block = est > 0.f ? (int)(kBlockUs / est) : 32;
    block = block < 4 ? 4 : (block > 32 ? 32 : block);
    for (int round = 0; round < kRounds && rc == HG_OK; ++round) {
      for (Candidate& c : cand) {
        float us = 0.f;
        rc = timed(c, block, &us);
        if (rc != HG_OK) break;
        if (us < c.us) c.us = us;
      }
    }
    if (rc != HG_OK) break;
    // The fixed rule's shape stays unless a candidate is faster by at least
    // kMargin: differences below that are within run-to-run noise.
    const Candidate* fastest = &cand[0];
    const Candidate* rule = nullptr;
    for (const Candidate& c : cand) {
      if (c.us < fastest->us) fastest = &c;
      if (c.s.vpt == fixed.s.vpt && c.s.ctas == fixed.s.ctas && c.s.pref == fixed.s.pref &&
          c.s.balanced == fixed.s.balanced)
        rule = &c;
    }
    const Candidate* best =
        (rule && fastest->us > rule->us * (1.f - kMargin)) ? rule : fastest;
    if (rule && best != rule) {
      // Confirm head to head: kConfirm alternating blocks of the rule's shape
      // and the challenger; the challenger's median must beat the rule's by
      // kMargin, else the rule's shape stays.
      float tr[kConfirm], tc[kConfirm];
      for (int k = 0; k < kConfirm && rc == HG_OK; ++k) {
        rc = timed(*rule, block, &tr[k]);
        if (rc == HG_OK) rc = timed(*best, block, &tc[k]);
      }
      if (rc != HG_OK) break;
      std::sort(tr, tr + kConfirm);
      std::sort(tc, tc + kConfirm);
      const float mr = 0.5f * (tr[kConfirm / 2 - 1] + tr[kConfirm / 2]);
      const float mc = 0.5f * (tc[kConfirm / 2 - 1] + tc[kConfirm / 2]);
      if (mc > mr * (1.f - kMargin)) best = rule;
    }
    h->shape[M] = best->s;
    h->chunks[M] = best->chunks;
  }
  if (stream) {
    int status = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpy(&status, h->status, sizeof status, cudaMemcpyDeviceToHost) != cudaSuccess) {
      if (rc == HG_OK) rc = HG_ERR_CUDA;
    } else if (status != hg::kDevOk && rc == HG_OK) {
      rc = HG_ERR_TIMEOUT;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (stream) cudaStreamDestroy(stream);
  if (pool) cudaFree(pool);
  h->device_parity = saved_dp;
  h->parity = 0;
  return rc;
}

}  // namespace

int hg_gather(hg_handle* h, const void* const* shard_ptrs, void* const* out_ptrs, int M,
              hg_stream_t stream) {
  return gather_impl(h, shard_ptrs, out_ptrs, M, nullptr, stream, true);
}

namespace {

// Device-side address of p, which must be page-locked host memory or device
// memory of device `dev` (HG_ERR_ARG otherwise).
int device_view(const void* p, int dev, void** out) {
  if (!p) return HG_ERR_ARG;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return HG_ERR_ARG;
  }
  if (!at.devicePointer) return HG_ERR_ARG;
  if (at.type == cudaMemoryTypeHost) {
    *out = at.devicePointer;
    return HG_OK;
  }
  if ((at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev) {
    *out = at.devicePointer;
    return HG_OK;
  }
  return HG_ERR_ARG;  // pageable host memory or another device's memory
}

}  // namespace

int hg_gather_host(hg_handle* h, const void* const* shard_ptrs, void* const* out_ptrs, int M,
                   hg_stream_t stream) {
  if (!h || !shard_ptrs || !out_ptrs) return HG_ERR_ARG;
  const void* sh[HG_MAX_TP];
  void* ou[HG_MAX_TP];
  for (int r = 0; r < h->tp; ++r) {
    void* p = nullptr;
    if (device_view(shard_ptrs[r], h->device, &p) != HG_OK) return HG_ERR_ARG;
    sh[r] = p;
    if (device_view(out_ptrs[r], h->device, &ou[r]) != HG_OK) return HG_ERR_ARG;
  }
  return gather_impl(h, sh, ou, M, nullptr, stream, false);
}

int hg_gather_stats(hg_handle* h, const void* const* shard_ptrs, void* const* out_ptrs, int M,
                    hg_row_stats* stats, hg_stream_t stream) {
  if (!stats) return HG_ERR_ARG;
  return gather_impl(h, shard_ptrs, out_ptrs, M, stats, stream, true);
}

int hg_sync(hg_handle* h, hg_stream_t stream) {
  if (!h) return HG_ERR_ARG;
  int st[hg::kStatusWords] = {};
  int par = 0;
  if (cudaMemcpyAsync(st, h->status, sizeof st, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      (h->device_parity && cudaMemcpyAsync(&par, h->parity_words, sizeof par,
                                           cudaMemcpyDeviceToHost, stream) != cudaSuccess) ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return HG_ERR_CUDA;
  if (h->device_parity) h->parity = par & 1;
  if (st[0] == hg::kDevOk) return HG_OK;
  h->failed = true;
  return HG_ERR_TIMEOUT;
}

int hg_rearm(hg_handle* h, hg_stream_t stream) {
  if (!h) return HG_ERR_ARG;
  for (int d = 0; d < h->tp; ++d)
    if (hg::launch_fill_u32(static_cast<uint32_t*>(h->box[d]), h->box_bytes / 4, hg::kSentinel,
                            stream) != cudaSuccess)
      return HG_ERR_CUDA;
  if (cudaMemsetAsync(h->status, 0, hg::kStatusWords * sizeof(int), stream) != cudaSuccess)
    return HG_ERR_CUDA;
  if (h->parity_words &&
      cudaMemsetAsync(h->parity_words, 0, (size_t)h->parity_entries * sizeof(int), stream) !=
          cudaSuccess)
    return HG_ERR_CUDA;
  if (h->partials &&
      hg::launch_fill_u32(reinterpret_cast<uint32_t*>(h->partials), h->partial_count * 4,
                          hg::kSentinel, stream) != cudaSuccess)
    return HG_ERR_CUDA;
  if (h->split_cells &&
      hg::launch_fill_u32(h->split_cells, h->split_cell_count * hg::fused::kSplitCellWords,
                          hg::fused::kSplitArmed, stream) != cudaSuccess)
    return HG_ERR_CUDA;
  h->parity = 0;
  h->failed = false;
  return HG_OK;
}

int hg_parity(const hg_handle* h) { return h ? h->parity : -1; }

int hg_mailbox(const hg_handle* h, int rank, const void** dev_ptr, size_t* bytes) {
  if (!h || rank < 0 || rank >= h->tp || !dev_ptr || !bytes) return HG_ERR_ARG;
  *dev_ptr = h->box[rank];
  *bytes = h->box_bytes;
  return HG_OK;
}

int hg_launch_shape(const hg_handle* h, int M, int* ctas, int* threads, int* elems_per_lane,
                    int* prefetch) {
  if (!h) return HG_ERR_ARG;
  if (M < 1 || M > h->cap || !h->served[M]) return HG_ERR_ROWS;
  const hg::LaunchShape& s = h->shape[M];
  if (ctas) *ctas = s.ctas;
  if (threads) *threads = 32 * h->tp;
  if (elems_per_lane) *elems_per_lane = s.vpt;
  if (prefetch) *prefetch = s.pref ? 1 : 0;
  return HG_OK;
}

int hg_timeline(const hg_handle* h, const hg_timeline_record** dev_ptr, int* calls, int* ctas,
                int* next) {
  static_assert(sizeof(hg_timeline_record) == hg::kTimelineSlots * 8, "timeline record layout");
  if (!h || !h->timeline || !dev_ptr) return HG_ERR_ARG;
  *dev_ptr = reinterpret_cast<const hg_timeline_record*>(h->timeline);
  if (calls) *calls = h->timeline_calls;
  if (ctas) *ctas = h->timeline_ctas;
  if (next) *next = (int)(h->timeline_next % h->timeline_calls);
  return HG_OK;
}

int hg_debug_skip_push(hg_handle* h, int rank) {
  if (!h || rank < -1 || rank >= h->tp) return HG_ERR_ARG;
  h->skip_rank = rank;
  return HG_OK;
}

int hg_gather_fused(hg_handle* h, const void* const* hidden_ptrs, const void* const* weight_ptrs,
                    void* const* logits_ptrs, void* const* out_ptrs, int M, int K,
                    hg_stream_t stream) {
  if (!h || !hidden_ptrs || !weight_ptrs || !out_ptrs) return HG_ERR_ARG;
  int max_tp = 0, max_m = 0, k_mult = 0, w_mult = 0;
  hg::fused::fused_limits(&max_tp, &max_m, &k_mult, &w_mult);
  if (h->tp > max_tp || !h->vec16 || h->W % w_mult != 0 || K < k_mult || K % k_mult != 0)
    return HG_ERR_ARG;
  if (M < 1 || M > h->cap || !h->served[M]) return HG_ERR_ROWS;
  if (M > max_m) return HG_ERR_ARG;
  if (h->failed) return HG_ERR_STATE;
  for (int r = 0; r < h->tp; ++r) {
    if (!hidden_ptrs[r] || !weight_ptrs[r] || !out_ptrs[r] || !aligned(hidden_ptrs[r], 16) ||
        !aligned(weight_ptrs[r], 16) || !aligned(out_ptrs[r], 16))
      return HG_ERR_ARG;
    if (logits_ptrs && logits_ptrs[r] && !aligned(logits_ptrs[r], 4)) return HG_ERR_ARG;
  }
  if (!h->device_parity) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return HG_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return HG_ERR_CAPTURE;
  }

  hg::fused::FusedLaunch l;
  l.hidden = hidden_ptrs;
  l.weight = weight_ptrs;
  l.logits = logits_ptrs;
  l.out = out_ptrs;
  const int host_parity = h->device_parity ? 0 : h->parity;
  for (int d = 0; d < h->tp; ++d)
    l.box[d] = static_cast<char*>(h->box[d]) + (size_t)host_parity * h->parity_elems * 16;
  if (h->device_parity) {
    l.parity_words = h->parity_words;
    l.parity_entries = h->parity_entries;
    l.parity_stride_words = h->parity_elems * 4;  // 16-byte elements
  }
  l.status = h->status;
  l.timeout_ns = h->timeout_ns;
  l.tp = h->tp;
  l.W = h->W;
  l.K = K;
  l.M = M;
  l.split_cells = h->split_cells;
  l.split_cell_count = h->split_cell_count;
  l.max_ctas = h->max_ctas;
  l.skip_rank = h->skip_rank;
  if (h->timeline) {
    l.timeline = h->timeline + (size_t)(h->timeline_next % h->timeline_calls) *
                                   h->timeline_ctas * hg::kTimelineSlots;
    l.timeline_ctas = h->timeline_ctas;
  }
  if (hg::fused::fused_launch(l, stream, h->sms) != cudaSuccess) return HG_ERR_CUDA;
  if (h->timeline) ++h->timeline_next;
  if (!h->device_parity) h->parity ^= 1;
  return HG_OK;
}

int hg_stock_gather(int tp, int shard_cols, const void* const* shard_ptrs, void* const* out_ptrs,
                    int M, hg_stream_t stream) {
  if (tp < 1 || tp > HG_MAX_TP || shard_cols < 1 || M < 0 || !shard_ptrs || !out_ptrs)
    return HG_ERR_ARG;
  for (int r = 0; r < tp; ++r)
    if (!shard_ptrs[r] || !out_ptrs[r]) return HG_ERR_ARG;
  if (M == 0) return HG_OK;
  const size_t wbytes = (size_t)shard_cols * 2;
  const size_t vbytes = wbytes * tp;
  for (int d = 0; d < tp; ++d)
    for (int r = 0; r < tp; ++r)
      if (cudaMemcpy2DAsync(static_cast<char*>(out_ptrs[d]) + r * wbytes, vbytes, shard_ptrs[r],
                            wbytes, wbytes, (size_t)M, cudaMemcpyDeviceToDevice,
                            stream) != cudaSuccess)
        return HG_ERR_CUDA;
  return HG_OK;
}

}  // extern "C"
