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
// Polling. PIPE (single-wave launches, where the poll races the neighbour's
// push): two staggered loads per waiting element stay in flight, so a word
// that lands between two polls is seen about half an L2 round trip later
// rather than a whole one. Otherwise (multi-iteration launches, where the data
// was pushed an iteration earlier): load, check, re-load what is missing.
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
constexpr unsigned kPollStaggerNs = 256;  // delay between the two in-flight polls

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void sleep_ns(unsigned ns) {
  asm volatile("nanosleep.u32 %0;" :: "r"(ns));
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
  template <bool STREAM>
  static __device__ __forceinline__ void st_out(uint4* p, uint4 v) {
    if (STREAM)
      asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                   :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
    else
      asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
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
  template <bool STREAM>
  static __device__ __forceinline__ void st_out(uint32_t* p, uint32_t v) {
    if (STREAM)
      asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
    else
      asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
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
  UnitPos p;
  p.r = r;
  p.idx = c * 32 * VPT + lane;
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

// Take the arrived elements of q into res; true when this warp is done. A lane
// that waits too long (or sees an error raised elsewhere) gives up.
template <typename V, int VPT>
__device__ __forceinline__ bool take_arrived(const GatherArgs& a, const V (&q)[VPT],
                                             V (&res)[VPT], unsigned& todo,
                                             unsigned long long& t_wait, bool& gave_up, int u,
                                             int d, size_t dst) {
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    if ((todo >> v & 1) && Elem<V>::arrived(q[v])) {
      res[v] = q[v];
      todo &= ~(1u << v);
    }
  if (todo) {
    const unsigned long long now = globaltimer_ns();
    if (t_wait == 0) t_wait = now;
    if (now - t_wait > a.timeout_ns || ld_relaxed_s32(a.status) != kDevOk) {
      record_timeout(a, u, d, dst);
      gave_up = true;
      todo = 0;
    }
  }
  return __all_sync(kFull, todo == 0);
}

// Poll this lane's elements of unit u in mailbox `box` until none holds a
// sentinel word; res receives the data. The warp leaves together (vote).
// Returns false when the warp gave up.
template <typename V, int VPT, bool PIPE>
__device__ __forceinline__ bool poll_unit(const GatherArgs& a, const V* box, const UnitPos& p,
                                          int u, int d, V (&res)[VPT]) {
  unsigned todo = 0;  // bit v: slot v still waits
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    if (p.idx + 32 * v < a.wv) todo |= 1u << v;
  unsigned long long t_wait = 0;
  bool gave_up = false;
  V q0[VPT], q1[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) q0[v] = q1[v] = Elem<V>::sentinel();
  issue_polls<V, VPT>(box, p, todo, q0);
  if (PIPE) {
    // Two loads in flight, issued a stagger apart; the loop is unrolled by two
    // so that no register copy waits on a pending load.
    for (;;) {
      sleep_ns(kPollStaggerNs);
      issue_polls<V, VPT>(box, p, todo, q1);
      if (take_arrived<V, VPT>(a, q0, res, todo, t_wait, gave_up, u, d, p.dst)) break;
      sleep_ns(kPollStaggerNs);
      issue_polls<V, VPT>(box, p, todo, q0);
      if (take_arrived<V, VPT>(a, q1, res, todo, t_wait, gave_up, u, d, p.dst)) break;
    }
  } else {
    while (!take_arrived<V, VPT>(a, q0, res, todo, t_wait, gave_up, u, d, p.dst))
      issue_polls<V, VPT>(box, p, todo, q0);
  }
  return !__any_sync(kFull, gave_up);
}

// VPT: elements per lane per unit. PIPE: staggered double polls (single-wave
// launches). STREAM: evict-first stores of the outputs (multi-iteration
// launches, whose outputs L2 should not keep). MAXT: largest CTA (32 * tp).
template <typename V, int VPT, bool PIPE, bool STREAM, int MAXT>
__global__ void __launch_bounds__(MAXT) gather_kernel(const __grid_constant__ GatherArgs a) {
  using E = Elem<V>;
  // Programmatic dependent launch: wait until the previous kernel on the
  // stream has completed and its memory is visible. Nothing is read or
  // written before the wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int lane = (int)threadIdx.x & 31;
  const int d = (int)threadIdx.x >> 5;  // this warp's rank: mailbox and output
  const int N = a.M * a.tp * a.chunks;  // units
  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  const int cons = (g + 1 == G) ? 0 : g + 1;  // the CTA whose pushes we consume
  const int iters = (N + G - 1) / G;

  // The first push's shard loads do not depend on the parity: start them
  // before anything else, so that their latency overlaps the parity and
  // status reads.
  V x0[VPT];
  UnitPos p0{};
  const bool push0 = iters > 0 && g < N;
  if (push0) {
    p0 = unit_pos<VPT>(a, g, lane);
    if (p0.r != a.skip_rank) {
      const V* src = reinterpret_cast<const V*>(a.shard[p0.r]) + p0.src;
#pragma unroll
      for (int v = 0; v < VPT; ++v)
        if (p0.idx + 32 * v < a.wv) x0[v] = E::ld_shard(src + 32 * v);
    }
  }
  // Device-resident parity: this warp's own copy (one load per warp of one
  // address, so every lane sees the same value).
  const int reader = g * a.tp + d;
  int parity = 0;
  if (a.parity_words) parity = ld_relaxed_s32(a.parity_words + reader);
  // Let the next kernel on the stream start launching (it waits for this one
  // to complete before it touches memory).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // One load per warp of one address: every lane sees the same value.
  if (ld_relaxed_s32(a.status) != kDevOk) return;  // unrecovered error: no work

  V* const box = reinterpret_cast<V*>(a.box[d]) + (size_t)parity * a.parity_stride;
  V* const out = reinterpret_cast<V*>(a.out[d]);

  // Iteration 0's push, from the loads started above.
  if (push0 && p0.r != a.skip_rank) {
#pragma unroll
    for (int v = 0; v < VPT; ++v)
      if (p0.idx + 32 * v < a.wv) E::st_relaxed(box + p0.dst + 32 * v, E::rewrite(x0[v]));
  }

  for (int t = 0; t <= iters; ++t) {
    const int up = t * G + g;
    if (t >= 1 && t < iters && up < N) {
      const UnitPos p = unit_pos<VPT>(a, up, lane);
      if (p.r != a.skip_rank) {
        const V* src = reinterpret_cast<const V*>(a.shard[p.r]) + p.src;
        V x[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v)
          if (p.idx + 32 * v < a.wv) x[v] = E::ld_shard(src + 32 * v);
#pragma unroll
        for (int v = 0; v < VPT; ++v)
          if (p.idx + 32 * v < a.wv) E::st_relaxed(box + p.dst + 32 * v, E::rewrite(x[v]));
      }
    }
    const int uc = (t - 1) * G + cons;
    if (t >= 1 && uc < N) {
      const UnitPos p = unit_pos<VPT>(a, uc, lane);
      V res[VPT];
      if (!poll_unit<V, VPT, PIPE>(a, box, p, uc, d, res)) return;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (p.idx + 32 * v < a.wv) {
          E::template st_out<STREAM>(out + p.dst + 32 * v, res[v]);
          E::st_relaxed(box + p.dst + 32 * v, E::sentinel());
        }
      }
    }
  }
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
}

__global__ void fill_u32_kernel(uint32_t* p, size_t n, uint32_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

// Kernels for tp <= 16 (CTAs of up to 512 threads) take 1, 2 or 4 elements
// per lane; larger tp (up to 1024 threads, 64 registers) 1 or 2.
template <typename V, bool PIPE>
const void* pick_vpt(int vpt, int tp) {
  if (tp <= 16) {
    switch (vpt) {
      case 1: return reinterpret_cast<const void*>(&gather_kernel<V, 1, PIPE, !PIPE, 512>);
      case 2: return reinterpret_cast<const void*>(&gather_kernel<V, 2, PIPE, !PIPE, 512>);
      case 4: return reinterpret_cast<const void*>(&gather_kernel<V, 4, PIPE, !PIPE, 512>);
      default: return nullptr;
    }
  }
  switch (vpt) {
    case 1: return reinterpret_cast<const void*>(&gather_kernel<V, 1, PIPE, !PIPE, 1024>);
    case 2: return reinterpret_cast<const void*>(&gather_kernel<V, 2, PIPE, !PIPE, 1024>);
    default: return nullptr;
  }
}

const void* kernel_for(const LaunchShape& s, bool vec16, int tp) {
  if (vec16) return s.pipe ? pick_vpt<uint4, true>(s.vpt, tp) : pick_vpt<uint4, false>(s.vpt, tp);
  return s.pipe ? pick_vpt<uint32_t, true>(s.vpt, tp) : pick_vpt<uint32_t, false>(s.vpt, tp);
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
  void* args[] = {const_cast<GatherArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t v, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_u32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace hg
