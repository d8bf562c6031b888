// Persistent gather kernel: push, poll, copy and re-arm for every virtual rank
// in one launch.
//
// Operation (vLLM API page "vllm.models.kimi_k3.nvidia.specialized_decode.
// runtime.logits_gather", module docstring and class HeadGather): rank r's
// shard row m, seen as 32-bit words with the sentinel (+0, -0) sent as
// (+0, +0), lands at row m, word column r * W / 2 of every rank's mailbox;
// each rank polls its mailbox row until no sentinel word is left, copies it to
// its [M, V] output and writes the sentinel back.
//
// Work decomposition. A CTA has one warp per virtual rank d (blockDim.x = 32 *
// tp); warp d owns rank d's mailbox and output. A unit is (row m, source rank
// r, chunk c): 32 * VPT consecutive elements (16-byte vectors, or 32-bit words
// when W % 8 != 0) of rank r's row m, VPT per lane. Units are dealt
// round-robin to the CTAs. In iteration t, CTA g pushes unit t*G + g (warp d
// reads the shard elements, through L1, and stores them into mailbox d) and
// consumes the unit that CTA g+1 (mod G) pushed in iteration t-1 (warp d polls
// mailbox d, then writes out[d] and re-arms). Every poll therefore waits on
// words that another CTA stores, and a push never depends on a poll, so with
// all CTAs resident every wait ends. The host never launches more CTAs than
// can be co-resident; each wait is also bounded in time by %globaltimer and
// gives up with an error in the status word instead of spinning on. The
// one-iteration lag keeps a pushed unit in L2 until it is polled and decouples
// neighbouring CTAs.
//
// Polling: load every element of the unit, check, re-load only what still
// holds a sentinel word; the loads land in the result registers directly.
// PREF: the shard loads of the next push are issued one iteration ahead, so
// that their latency overlaps this iteration's poll (multi-iteration
// launches). Outputs are written with evict-first stores: the caller reads
// them once, and L2 is better spent on the mailboxes.
//
// Memory ordering. Pushes, polls and re-arms are relaxed at gpu scope (morally
// strong, per-word single-copy atomic; a vector access is one access per
// 32-bit word), so a polled word is either still the sentinel or the pushed
// data word, never a mix. A word is re-armed by the thread that read it, after
// reading it (same-address coherence). Calls are ordered by kernel boundaries
// (a programmatic dependent launch waits for the previous kernel's completion
// before any access); two calls in a row use different mailbox parities.

#include "hg_internal.cuh"

namespace hg {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <typename V>
struct Elem;

// 16-byte vector of four words.
template <>
struct Elem<uint4> {
  static constexpr int kWords = 4;
  static __device__ __forceinline__ uint32_t word(const uint4& v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
  }
  static __device__ __forceinline__ uint4 ld_shard(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
  }
  static __device__ __forceinline__ uint4 ld_poll(const uint4* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
  }
  static __device__ __forceinline__ void st_relaxed(uint4* p, uint4 v) {
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
  }
  static __device__ __forceinline__ void st_out(uint4* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
  }
  static __device__ __forceinline__ bool arrived(uint4 v) {
    return v.x != kSentinel && v.y != kSentinel && v.z != kSentinel && v.w != kSentinel;
  }
  static __device__ __forceinline__ uint32_t rw(uint32_t x) {
    return x == kSentinel ? kSentAs : x;
  }
  static __device__ __forceinline__ uint4 rewrite(uint4 v) {
    return make_uint4(rw(v.x), rw(v.y), rw(v.z), rw(v.w));
  }
  static __device__ __forceinline__ uint4 sentinel() {
    return make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  }
};

// One 32-bit word (shards whose width is not a multiple of 8 columns).
template <>
struct Elem<uint32_t> {
  static constexpr int kWords = 1;
  static __device__ __forceinline__ uint32_t word(uint32_t v, int) { return v; }
  static __device__ __forceinline__ uint32_t ld_shard(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
  static __device__ __forceinline__ uint32_t ld_poll(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  }
  static __device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
  }
  static __device__ __forceinline__ void st_out(uint32_t* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
  }
  static __device__ __forceinline__ bool arrived(uint32_t v) { return v != kSentinel; }
  static __device__ __forceinline__ uint32_t rewrite(uint32_t v) {
    return v == kSentinel ? kSentAs : v;
  }
  static __device__ __forceinline__ uint32_t sentinel() { return kSentinel; }
};

// Element offsets of unit u for this lane's slot 0 (slot v adds 32 * v).
struct UnitPos {
  int r;       // source rank
  int idx;     // element index of slot 0 within the rank-row
  int lim;     // end of the unit's elements within the rank-row (exclusive)
  size_t src;  // offset in rank r's shard
  size_t dst;  // offset in a mailbox parity and in an output
};

template <int VPT>
__device__ __forceinline__ UnitPos unit_pos(const GatherArgs& a, int u, int lane) {
  const int per_row = a.tp * a.chunks;
  const int m = u / per_row;
  const int rem = u - m * per_row;
  const int r = rem / a.chunks;
  const int c = rem - r * a.chunks;
  // Chunk c covers elements [start, lim) of the rank-row: 32 * VPT elements
  // from c * 32 * VPT (the last chunk ragged), or, with balanced chunks
  // (a.chunk_q > 0), chunk_q elements, plus one for the first chunk_r chunks.
  int start, lim;
  if (a.chunk_q > 0) {
    start = c * a.chunk_q + min(c, a.chunk_r);
    lim = start + a.chunk_q + (c < a.chunk_r ? 1 : 0);
  } else {
    start = c * 32 * VPT;
    lim = min(start + 32 * VPT, a.wv);
  }
  UnitPos p;
  p.r = r;
  p.lim = lim;
  p.idx = start + lane;
  p.src = (size_t)m * a.wv + p.idx;
  p.dst = (size_t)m * a.tp * a.wv + (size_t)r * a.wv + p.idx;
  return p;
}

// Record where a poll gave up (the first one wins).
__device__ __forceinline__ void record_timeout(const GatherArgs& a, int u, int d, size_t dst) {
  if (atomicCAS(a.status, kDevOk, kDevTimeout) == kDevOk) {
    a.status[1] = u;
    a.status[2] = d;
    a.status[3] = (int)dst;
  }
}

template <typename V, int VPT>
__device__ __forceinline__ void issue_polls(const V* box, const UnitPos& p, unsigned todo,
                                            V (&q)[VPT]) {
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    if (todo >> v & 1) q[v] = Elem<V>::ld_poll(box + p.dst + 32 * v);
}

// Poll this lane's elements of unit u in mailbox `box` until none holds a
// sentinel word; res receives the data. poll_begin issues the first loads
// (so that other work can overlap their round trip); poll_finish waits. A
// lane that waits too long (or sees an error raised elsewhere) gives up; the
// warp leaves together (vote). poll_finish returns false when the warp gave
// up. The status word is loaded together with each round of re-polls and
// looked at in the next round, so that a retry costs one memory round trip,
// not two.
template <typename V, int VPT>
__device__ __forceinline__ unsigned poll_begin(const GatherArgs& a, const V* box,
                                               const UnitPos& p, V (&res)[VPT]) {
  unsigned todo = 0;  // bit v: slot v still waits
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    if (p.idx + 32 * v < p.lim) todo |= 1u << v;
  issue_polls<V, VPT>(box, p, todo, res);
  return todo;
}

template <typename V, int VPT>
__device__ __forceinline__ bool poll_finish(const GatherArgs& a, const V* box, const UnitPos& p,
                                            int u, int d, unsigned todo, V (&res)[VPT]) {
  unsigned long long t_wait = 0;
  bool gave_up = false;
  int status = kDevOk;  // as loaded with the previous round of polls
  for (;;) {
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if ((todo >> v & 1) && Elem<V>::arrived(res[v])) todo &= ~(1u << v);
    if (todo) {
      const unsigned long long now = globaltimer_ns();
      if (t_wait == 0) t_wait = now;
      if (now - t_wait > a.timeout_ns || status != kDevOk) {
        record_timeout(a, u, d, p.dst);
        gave_up = true;
        todo = 0;
      }
    }
    if (__all_sync(kFull, todo == 0)) break;
    issue_polls<V, VPT>(box, p, todo, res);
    status = ld_relaxed_s32(a.status);
  }
  return !__any_sync(kFull, gave_up);
}

// ---- Row statistics (max, first argmax, sum of exp(x - max)) -------------
//
// Every step here is branch-free (comparisons feed selects, never jumps): a
// per-value condition that diverges inside a warp costs tens of cycles of
// divergence handling, and a fold touches 24 values per lane. A warp's
// result comes from each lane's own (max, first argmax, sum of exp(x - lane
// max)), then one warp max (redux.sync on an order-preserving key), one warp
// min over the lanes that hold that max (the first argmax), and a shuffle sum
// of the lanes' sums rescaled to the warp max.

constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kNoColumn = 0x7fffffff;

// Unsigned key of a float whose unsigned order is the float order (-0 below
// +0; NaNs at the ends), and back.
__device__ __forceinline__ unsigned order_key(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (mx, arg, s) <- its combination with (mx2, arg2, s2), where s is a sum of
// exp(x - mx) over finite x (0 when mx is -inf); ties keep the smaller
// column. Both exponentials are taken before the selects.
__device__ __forceinline__ void combine_partial(float& mx, int& arg, float& s, float mx2,
                                                int arg2, float s2) {
  const float m = fmaxf(mx, mx2);
  const int a = mx > mx2 ? arg : (mx2 > mx ? arg2 : min(arg, arg2));
  const float e1 = __expf(mx - m);
  const float e2 = __expf(mx2 - m);
  const float t1 = mx != kNegInf ? s * e1 : 0.f;
  const float t2 = mx2 != kNegInf ? s2 * e2 : 0.f;
  mx = m;
  arg = a;
  s = t1 + t2;
}

// Warp-wide (max, first argmax, sum of exp(x - max)) from every lane's own
// (lane_mx, lane_arg, lane_s), lane_s relative to lane_mx; every lane
// receives the result.
__device__ __forceinline__ void warp_stats(float lane_mx, int lane_arg, float lane_s, float& mx,
                                           int& arg, float& s) {
  mx = key_float(__reduce_max_sync(kFull, order_key(lane_mx)));
  const unsigned cand = lane_mx == mx ? (unsigned)lane_arg : (unsigned)kNoColumn;
  arg = (int)__reduce_min_sync(kFull, cand);
  const float e = __expf(lane_mx - mx);
  float t = lane_mx != kNegInf ? lane_s * e : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(kFull, t, off);
  s = t;
}

// Statistics of unit u's values, folded by one warp from its rank's copy
// (every rank's copy holds the same values). Per lane: the max (a tree of fmaxf),
// then in one pass the sum of exp(x - lane max) and the smallest column
// holding the lane max; then warp_stats. Lane 0 writes the result into cell u
// with one relaxed 16-byte store.
template <typename V, int VPT>
__device__ __forceinline__ void unit_stats(const GatherArgs& a, const UnitPos& p, int u,
                                           const V (&res)[VPT]) {
  using E = Elem<V>;
  // Pass 1: the lane max over the words (each word: the larger half), two
  // interleaved chains of fmaxf. Words of a vector beyond the row count as
  // two -inf values.
  float m0 = kNegInf, m1 = kNegInf;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const bool ok = p.idx + 32 * v < p.lim;
#pragma unroll
    for (int k = 0; k < E::kWords; ++k) {
      const uint32_t w = E::word(res[v], k);
      const float m = fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
      if ((v * E::kWords + k) & 1) m1 = fmaxf(m1, ok ? m : kNegInf);
      else m0 = fmaxf(m0, ok ? m : kNegInf);
    }
  }
  const float lm = fmaxf(m0, m1);
  // Pass 2, from the words again: the sum of exp(x - lane max) and the
  // smallest column holding the lane max.
  int la = kNoColumn;
  float ls = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const bool ok = p.idx + 32 * v < p.lim;
    const int col0 = p.r * a.shard_cols + (p.idx + 32 * v) * (2 * E::kWords);
#pragma unroll
    for (int k = 0; k < E::kWords; ++k) {
      const uint32_t w = E::word(res[v], k);
      const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
      const float e = __expf(lo - lm) + __expf(hi - lm);  // exp(-inf) = 0; lm = -inf: below
      ls += ok ? e : 0.f;
      const int c = hi == lm ? col0 + 2 * k + 1 : kNoColumn;
      la = ok ? min(la, lo == lm ? col0 + 2 * k : c) : la;
    }
  }
  if (lm == kNegInf) ls = 0.f;
  float mx, s;
  int arg;
  warp_stats(lm, la, ls, mx, arg, s);
  if ((threadIdx.x & 31) == 0) {
    // A Lamport cell: no word may equal the sentinel, so a -0.0 max is
    // written as +0.0 (the same value); the other words cannot be it.
    uint4 w;
    w.x = __float_as_uint(mx) == kSentinel ? 0u : __float_as_uint(mx);
    w.y = (uint32_t)arg;
    w.z = __float_as_uint(s);
    w.w = 1u;
    Elem<uint4>::st_relaxed(reinterpret_cast<uint4*>(a.partials + u), w);
  }
}

// Warp 0 of CTA g, once its own units are done: for rows g, g + G, ..., poll
// the row's cells until all have arrived (bounded), fold them, write the row's
// statistics and re-arm the cells. BATCH cells per lane are in flight at once,
// so a row of up to 32 * BATCH cells costs one wait. Rows are reduced by
// different CTAs in parallel.
// A cell is written once per call, by the warp that folded its unit, and a
// reducer waits on cells without anyone ever waiting on a reducer, so neither
// a CTA barrier nor any atomic is involved: the cells carry their own
// arrival, as mailbox words do.
// TL: lane 0 also records, for the first row, when all its cells had arrived
// and been folded across the warp, and when its statistics were written
// (timeline slots of warps 11 and 12, tp <= 8).
template <int BATCH, bool TL>
__device__ __forceinline__ void finish_stats(const GatherArgs& a, int g, int G) {
  const int lane = (int)threadIdx.x & 31;
  const int per_row = a.tp * a.chunks;  // cells (units) per row
  const uint4 armed = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  for (int m = g; m < a.M; m += G) {
    uint4* q = reinterpret_cast<uint4*>(a.partials + (size_t)m * per_row);
    float mx = kNegInf, s = 0.f;
    int arg = kNoColumn;
    bool gave_up = false;
    for (int base = lane; base < per_row && !gave_up; base += BATCH * 32) {
      // A batch of cells in flight; the ones still armed are re-loaded
      // together (never one at a time), until all have arrived (bounded).
      uint4 v[BATCH];
      unsigned todo = 0;
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        if (base + 32 * k < per_row) {
          v[k] = Elem<uint4>::ld_poll(q + base + 32 * k);
          todo |= 1u << k;
        }
      }
      const unsigned valid = todo;
      unsigned long long t0 = 0;
      int status = kDevOk;  // loaded with the previous round of polls
      for (;;) {
#pragma unroll
        for (int k = 0; k < BATCH; ++k)
          if ((todo >> k & 1) && Elem<uint4>::arrived(v[k])) todo &= ~(1u << k);
        if (!todo) break;
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (now - t0 > a.timeout_ns || status != kDevOk) {
          record_timeout(a, -1, -1, (size_t)base);
          gave_up = true;
          break;
        }
#pragma unroll
        for (int k = 0; k < BATCH; ++k)
          if (todo >> k & 1) v[k] = Elem<uint4>::ld_poll(q + base + 32 * k);
        status = ld_relaxed_s32(a.status);
      }
      if (gave_up) break;
      // The batch: its max (a tree), then in one pass its smallest column at
      // that max and its sum rescaled to it (independent exponentials).
      float km[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k)
        km[k] = (valid >> k & 1) ? __uint_as_float(v[k].x) : kNegInf;
      float tm[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) tm[k] = km[k];
#pragma unroll
      for (int step = 1; step < BATCH; step <<= 1)
#pragma unroll
        for (int k = 0; k + step < BATCH; k += 2 * step) tm[k] = fmaxf(tm[k], tm[k + step]);
      const float bm = tm[0];
      int ba = kNoColumn;
      float bs = 0.f;
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const float e = __expf(km[k] - bm);
        bs += (km[k] != kNegInf) ? __uint_as_float(v[k].z) * e : 0.f;
        ba = ((valid >> k & 1) && km[k] == bm) ? min(ba, (int)v[k].y) : ba;
      }
      if (base == lane) {  // the first batch (the only one up to 32 * BATCH cells)
        mx = bm;
        arg = ba;
        s = bs;
      } else {
        combine_partial(mx, arg, s, bm, ba, bs);
      }
    }
    float rm, rs;
    int ra;
    warp_stats(mx, arg, s, rm, ra, rs);
    if (__any_sync(kFull, gave_up)) return;
    if constexpr (TL) {
      if (m == g && lane == 0 && a.tp <= 8)
        a.timeline[(size_t)g * kTimelineSlots + 2 + 11] = globaltimer_ns();
    }
    if (lane == 0) {
      hg_row_stats r;
      r.max_logit = rm;
      r.argmax = ra;
      r.sum_exp = rs;
      r.logsumexp = rm + logf(rs);
      a.stats[m] = r;
      if constexpr (TL) {
        if (m == g && a.tp <= 8) a.timeline[(size_t)g * kTimelineSlots + 2 + 12] = globaltimer_ns();
      }
    }
    // Re-arm the row's cells once its statistics are written: stored inside
    // the fold, the re-arms held the fold back (0.3 us per call at one row).
    for (int c = lane; c < per_row; c += 32) Elem<uint4>::st_relaxed(q + c, armed);
  }
}

// VPT: elements per lane per unit. PREF: the next push's shard loads are
// issued one iteration ahead. MAXT: largest CTA (32 * tp). STATS: one warp
// also folds each pushed unit into a statistics cell (the push of iteration
// t: warp t mod tp), and warp 0 of CTA g folds the cells of rows g, g + G,
// ...
// TL: the kernel records when each CTA starts, passes the wait and when each
// of its warps finishes (a measurement build; the others record nothing).
template <typename V, int VPT, bool PREF, int MAXT, bool STATS, bool TL>
__device__ __forceinline__ void gather_body(const GatherArgs& a) {
  using E = Elem<V>;
  unsigned long long tl_entry = 0;
  if constexpr (TL) tl_entry = globaltimer_ns();
  const int lane = (int)threadIdx.x & 31;
  const int d = (int)threadIdx.x >> 5;  // this warp's rank: mailbox and output
  const int N = a.M * a.tp * a.chunks;  // units
  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  const int cons = (g + 1 == G) ? 0 : g + 1;  // the CTA whose pushes we consume
  const int iters = (N + G - 1) / G;
  // The first push's position needs only the arguments: compute it before
  // the wait, off the path that starts when the previous kernel completes.
  UnitPos p0{};
  const bool push0 = iters > 0 && g < N;
  if (push0) p0 = unit_pos<VPT>(a, g, lane);
  // This warp's pointers come from the kernel arguments, which no kernel
  // writes, so they may be read before the wait.
  const V* const src0 =
      reinterpret_cast<const V*>(a.shard[push0 ? p0.r : 0]) + (push0 ? p0.src : 0);
  V* const box0 = reinterpret_cast<V*>(a.box[d]);
  V* const out = reinterpret_cast<V*>(a.out[d]);
  // Before the wait, only an L2 prefetch of that unit (16-byte vectors), so
  // that its DRAM round trip overlaps the previous kernel. It brings no value
  // into the SM, and every access to device memory goes through L2, so the
  // loads after the wait still see what the previous kernel writes to the
  // shards. The unit is contiguous: 32 * VPT vectors from lane 0's first,
  // fewer in a ragged last chunk.
  if constexpr (sizeof(V) == 16) {
    if (a.l2_prefetch && threadIdx.x == 0 && push0 && p0.r != a.skip_rank) {
      const int n = p0.lim - p0.idx;  // from lane 0's first element
      if (n > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src0), "r"(n * 16)
                     : "memory");
    }
  }
  // With the early trigger this launch usually starts while the previous
  // kernel still runs: have the pointers in registers before the wait (the
  // empty asm takes them as operands), off the path that starts when that
  // kernel completes. With the late trigger it starts as the previous kernel
  // ends; there the loads keep the compiler's schedule (forcing them, or
  // moving them after the wait, measured slower at two rows).
  if (!a.late_trigger) asm volatile("" ::"l"(src0), "l"(box0), "l"(out));
  // Programmatic dependent launch: wait until the previous kernel on the
  // stream has completed and its memory is visible. Apart from the L2
  // prefetch, nothing reads or writes global memory before the wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (TL) {
    if (threadIdx.x == 0) {
      unsigned long long* rec = a.timeline + (size_t)blockIdx.x * kTimelineSlots;
      rec[0] = tl_entry;
      rec[1] = globaltimer_ns();
      // The SM this CTA runs on, in the slot of warp 14 (a CTA of tp <= 14
      // warps has none).
      if (a.tp <= 14) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        rec[2 + 14] = smid;
      }
    }
  }

  // The first push's shard loads do not depend on the parity: start them
  // before anything else, so that their latency overlaps the parity and
  // status reads.
  V x0[VPT];
  if (push0 && p0.r != a.skip_rank) {
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if (p0.idx + 32 * v < p0.lim) x0[v] = E::ld_shard(src0 + 32 * v);
  }
  // Device-resident parity: this warp's own copy (one load per warp of one
  // address, so every lane sees the same value).
  const int reader = g * a.tp + d;
  int parity = 0;
  if (a.parity_words) parity = ld_relaxed_s32(a.parity_words + reader);
  // Let the next kernel on the stream start launching (it waits for this one
  // to complete before it touches memory): here, or once this warp's work is
  // done (late_trigger).
  if (!a.late_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // One load per warp of one address: every lane sees the same value.
  if (ld_relaxed_s32(a.status) != kDevOk) return;  // unrecovered error: no work

  V* const box = box0 + (size_t)parity * a.parity_stride;

  // Iteration 0's push, from the loads started above.
  if (push0 && p0.r != a.skip_rank) {
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if (p0.idx + 32 * v < p0.lim) E::st_relaxed(box + p0.dst + 32 * v, E::rewrite(x0[v]));
    // Statistics: warp 0 folds iteration 0's unit right after its push, before
    // its first polls. Folded between issuing the polls and waiting for them,
    // the fold held the first consumer step back by more than its own length
    // (0.5 / 0.8 / 1.1 µs more per call at 1 / 4 / 8 rows).
    if (STATS && d == 0) {
      unit_stats<V, VPT>(a, p0, g, x0);
      // Statistics timeline (tp <= 8: the slot of warp 10): when warp 0 had
      // folded iteration 0's push.
      if constexpr (TL) {
        if (lane == 0 && a.tp <= 8)
          a.timeline[(size_t)g * kTimelineSlots + 2 + 10] = globaltimer_ns();
      }
    }
  }

  // Shard loads of a push: with PREF issued one iteration ahead (during the
  // previous iteration's poll), otherwise right before the push's stores.
  V xn[VPT];
  UnitPos pn{};
  bool pushn = false;
  auto load_push = [&](int t) {
    const int u = t * G + g;
    pushn = t < iters && u < N;
    if (!pushn) return;
    pn = unit_pos<VPT>(a, u, lane);
    if (pn.r == a.skip_rank) {
      pushn = false;
      return;
    }
    const V* src = reinterpret_cast<const V*>(a.shard[pn.r]) + pn.src;
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if (pn.idx + 32 * v < pn.lim) xn[v] = E::ld_shard(src + 32 * v);
  };
  if (PREF) load_push(1);

  for (int t = 1; t <= iters; ++t) {
    if (!PREF) load_push(t);
    if (pushn) {
#pragma unroll
      for (int v = 0; v < VPT; ++v)
        if (pn.idx + 32 * v < pn.lim) E::st_relaxed(box + pn.dst + 32 * v, E::rewrite(xn[v]));
      // Statistics are folded where the values already sit in registers: at
      // the push. Every warp pushes the same unit (into its own rank's
      // mailbox), so the fold of iteration t's push goes to warp t mod tp and
      // no warp falls behind by one fold per iteration. The values are the
      // shard's own words: a sentinel word (+0, -0) that the push sends as
      // (+0, +0) holds the same two values to every comparison, sum and exp.
      if (STATS && d == t % a.tp) unit_stats<V, VPT>(a, pn, t * G + g, xn);
    }
    if (PREF) load_push(t + 1);
    const int uc = (t - 1) * G + cons;
    if (uc < N) {
      const UnitPos p = unit_pos<VPT>(a, uc, lane);
      V res[VPT];
      const unsigned todo = poll_begin<V, VPT>(a, box, p, res);
      // Statistics timeline (tp <= 8: the slots of warps 8 and 9): when warp
      // 0's first poll completed and its stores were issued.
      constexpr bool kTlStats = TL && STATS;
      const bool tl_here = kTlStats && t == 1 && d == 0 && lane == 0 && a.tp <= 8;
      if (!poll_finish<V, VPT>(a, box, p, uc, d, todo, res)) return;
      if (kTlStats && tl_here) a.timeline[(size_t)g * kTimelineSlots + 2 + 8] = globaltimer_ns();
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (p.idx + 32 * v < p.lim) {
          E::st_out(out + p.dst + 32 * v, res[v]);
          E::st_relaxed(box + p.dst + 32 * v, E::sentinel());
        }
      }
      if (kTlStats && tl_here) a.timeline[(size_t)g * kTimelineSlots + 2 + 9] = globaltimer_ns();
    }
  }
  if (a.late_trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.parity_words) {
    // Flip this warp's share of the parity copies: copies reader + k * G * tp,
    // so that every copy flips exactly once per call whatever the grid size.
    // None of them but this warp's own is read in this call, and that one was
    // read above by this warp.
    const int stride = G * a.tp;
    for (int e = reader + lane * stride; e < a.parity_entries; e += 32 * stride)
      asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(a.parity_words + e),
                   "r"(parity ^ 1)
                   : "memory");
  }
  // Warp 0 of CTA g: rows g, g + G, ... Eight cells per lane cover a row of
  // TP8 V=163840 at 3 elements per lane (216 cells) in one wait; wider units
  // leave fewer cells and fewer free registers.
  if constexpr (TL && STATS) {
    // When warp 0 turns to the statistics reducer (the slot of warp 15,
    // which a statistics CTA of tp <= 15 warps does not have).
    if (d == 0 && lane == 0 && a.tp < 16)
      a.timeline[(size_t)g * kTimelineSlots + 2 + 15] = globaltimer_ns();
  }
  if (STATS && d == 0 && g < a.M) finish_stats<(VPT <= 4 ? 8 : 6), TL>(a, g, G);
  if constexpr (TL) {
    if (lane == 0) a.timeline[(size_t)g * kTimelineSlots + 2 + d] = globaltimer_ns();
  }
}

// The gather: register use left to the compiler under the CTA-size bound
// (54 and 62 registers at 3 and 4 vectors per lane: 4 CTAs of 256 threads
// per SM).
template <typename V, int VPT, bool PREF, int MAXT, bool TL = false>
__global__ void __launch_bounds__(MAXT) gather_kernel(const __grid_constant__ GatherArgs a) {
  gather_body<V, VPT, PREF, MAXT, false, TL>(a);
}

// The gather with row statistics (tp <= 16): held to 64 registers, so that 4
// CTAs of 256 threads fit per SM as for the plain gather.
template <typename V, int VPT, bool PREF, bool TL = false>
__global__ void __launch_bounds__(512, 2) gather_stats_kernel(const __grid_constant__ GatherArgs a) {
  gather_body<V, VPT, PREF, 512, true, TL>(a);
}

__global__ void fill_u32_kernel(uint32_t* p, size_t n, uint32_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

// Kernels for tp <= 16 (CTAs of up to 512 threads) take 1 to 6 elements per
// lane; larger tp (up to 1024 threads, 64 registers) 1 or 2. Row statistics
// exist for tp <= 16.
// Kernel of elements per lane VPT for a template pattern: the gather or the
// gather with statistics, with or without the timeline.
template <typename V, bool PREF, bool STATS, bool TL, int VPT>
const void* kernel_ptr() {
  if constexpr (STATS)
    return reinterpret_cast<const void*>(&gather_stats_kernel<V, VPT, PREF, TL>);
  else
    return reinterpret_cast<const void*>(&gather_kernel<V, VPT, PREF, 512, TL>);
}

template <typename V, bool PREF, bool STATS, bool TL>
const void* pick_512(int vpt) {
  switch (vpt) {
    case 1: return kernel_ptr<V, PREF, STATS, TL, 1>();
    case 2: return kernel_ptr<V, PREF, STATS, TL, 2>();
    case 3: return kernel_ptr<V, PREF, STATS, TL, 3>();
    case 4: return kernel_ptr<V, PREF, STATS, TL, 4>();
    case 5: return kernel_ptr<V, PREF, STATS, TL, 5>();
    case 6: return kernel_ptr<V, PREF, STATS, TL, 6>();
    default: return nullptr;
  }
}

// Kernels for tp <= 16 (CTAs of up to 512 threads) take 1 to 6 elements per
// lane; larger tp (up to 1024 threads, 64 registers) 1 or 2. Row statistics
// exist for tp <= 16; timeline builds for 16-byte vectors without prefetch.
template <typename V, bool PREF, bool STATS>
const void* pick_vpt(int vpt, int tp) {
  if (tp <= 16) return pick_512<V, PREF, STATS, false>(vpt);
  if (STATS) return nullptr;
  switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&gather_kernel<V, 1, PREF, 1024>);
    case 2: return reinterpret_cast<const void*>(&gather_kernel<V, 2, PREF, 1024>);
    default: return nullptr;
  }
}

template <typename V, bool PREF>
const void* pick_stats(const LaunchShape& s, int tp) {
  return s.stats ? pick_vpt<V, PREF, true>(s.vpt, tp) : pick_vpt<V, PREF, false>(s.vpt, tp);
}

const void* kernel_for(const LaunchShape& s, bool vec16, int tp) {
  if (s.timeline) {
    if (!vec16 || s.pref || tp > 16) return nullptr;
    return s.stats ? pick_512<uint4, false, true, true>(s.vpt)
                   : pick_512<uint4, false, false, true>(s.vpt);
  }
  if (vec16) return s.pref ? pick_stats<uint4, true>(s, tp) : pick_stats<uint4, false>(s, tp);
  return s.pref ? pick_stats<uint32_t, true>(s, tp) : pick_stats<uint32_t, false>(s, tp);
}

}  // namespace

cudaError_t gather_occupancy(const LaunchShape& s, bool vec16, int tp, int* ctas_per_sm) {
  const void* k = kernel_for(s, vec16, tp);
  if (!k) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, k, 32 * tp, 0);
}

cudaError_t launch_gather(const GatherArgs& a, const LaunchShape& s, bool vec16,
                          cudaStream_t stream, bool cooperative) {
  const void* k = kernel_for(s, vec16, a.tp);
  if (!k) return cudaErrorInvalidValue;
  GatherArgs args = a;
  args.late_trigger = s.late ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s.ctas);
  cfg.blockDim = dim3((unsigned)(32 * a.tp));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (cooperative) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* kargs[] = {&args};
  return cudaLaunchKernelExC(&cfg, k, kargs);
}

cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t v, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_u32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace hg
