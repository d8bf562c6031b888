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
// Work decomposition. A unit is (row m, source rank r, chunk c): blockDim.x
// consecutive elements (16-byte vectors, or 32-bit words when W % 8 != 0) of
// rank r's row m, one per thread. Units are dealt round-robin to the CTAs;
// in iteration t CTA g pushes unit t*G + g into all TP mailboxes and consumes,
// for every consumer rank d, the unit that CTA g+1 (mod G) pushed in iteration
// t-1. Every poll therefore waits on words that another CTA stores, and a
// CTA's push never depends on a poll, so with all CTAs co-resident (the
// launch is cooperative) every wait ends; each one is also bounded in time by
// %globaltimer and gives up with an error in the status word instead of
// spinning on. The one-iteration lag keeps the freshly pushed unit in L2
// until it is polled and decouples neighbouring CTAs.
//
// Memory ordering. Pushes and polls are relaxed at gpu scope (morally strong,
// per-word single-copy atomic; a vector access is one access per 32-bit word),
// so a polled word is either still the sentinel or the pushed data word, never
// a mix. A word is re-armed by the thread that read it, after reading it
// (same-address coherence). Calls are ordered by kernel boundaries on one
// stream; two calls in a row use different mailbox parities.

#include "hg_internal.cuh"

namespace hg {
namespace {

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
  static __device__ __forceinline__ uint4 ld_shard(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
  }
  static __device__ __forceinline__ uint4 ld_poll(const uint4* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
  }
  static __device__ __forceinline__ void st_push(uint4* p, uint4 v) {
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
  }
  static __device__ __forceinline__ void st_out(uint4* p, uint4 v) {
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
  static __device__ __forceinline__ uint4 none() { return make_uint4(0, 0, 0, 0); }
};

// One 32-bit word (shards whose width is not a multiple of 8 columns).
template <>
struct Elem<uint32_t> {
  static __device__ __forceinline__ uint32_t ld_shard(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
  static __device__ __forceinline__ uint32_t ld_poll(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  }
  static __device__ __forceinline__ void st_push(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
  }
  static __device__ __forceinline__ void st_out(uint32_t* p, uint32_t v) {
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
  }
  static __device__ __forceinline__ bool arrived(uint32_t v) { return v != kSentinel; }
  static __device__ __forceinline__ uint32_t rewrite(uint32_t v) {
    return v == kSentinel ? kSentAs : v;
  }
  static __device__ __forceinline__ uint32_t sentinel() { return kSentinel; }
  static __device__ __forceinline__ uint32_t none() { return 0u; }
};

// Where unit u's elements live for this thread.
struct UnitPos {
  int r;       // source rank
  size_t src;  // element offset in the shard of rank r
  size_t dst;  // element offset in a mailbox row block / output
  bool valid;  // this thread has an element in the unit
};

__device__ __forceinline__ UnitPos unit_pos(const GatherArgs& a, int tp, int u) {
  const int per_row = tp * a.chunks;
  const int m = u / per_row;
  const int rem = u - m * per_row;
  const int r = rem / a.chunks;
  const int c = rem - r * a.chunks;
  const int idx = c * (int)blockDim.x + (int)threadIdx.x;
  UnitPos p;
  p.r = r;
  p.valid = idx < a.wv;
  p.src = (size_t)m * a.wv + idx;
  p.dst = (size_t)m * tp * a.wv + (size_t)r * a.wv + idx;
  return p;
}

// Poll NB mailbox elements (consumer ranks d0 .. d0+nb-1) already loaded into
// x until none holds a sentinel word, then copy them to the outputs and
// re-arm. Warp-uniform loop: the warp spins until every lane's elements have
// arrived (warp vote), re-reading only what is still missing. Returns false if
// the poll gave up (timeout or an error raised elsewhere in the grid).
template <typename V, int NB>
__device__ __forceinline__ bool finish_consume(const GatherArgs& a, int d0, int nb,
                                               const UnitPos& p, V (&x)[NB], int u) {
  using E = Elem<V>;
  bool ok = true;
  unsigned long long t_wait = 0;  // start of this wait, read on the first miss
#pragma unroll
  for (int i = 0; i < NB; ++i)
    if (i < nb) ok = ok && E::arrived(x[i]);
  if (!p.valid) ok = true;
  bool gave_up = false;
  while (!__all_sync(0xffffffffu, ok)) {
    if (!ok) {
      ok = true;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i < nb && !E::arrived(x[i])) {
          x[i] = E::ld_poll(reinterpret_cast<const V*>(a.box[d0 + i]) + p.dst);
          ok = ok && E::arrived(x[i]);
        }
      }
      if (!ok && t_wait == 0) t_wait = globaltimer_ns();
      if (!ok && (globaltimer_ns() - t_wait > a.timeout_ns ||
                  ld_relaxed_s32(a.status) != kDevOk)) {
        if (atomicCAS(a.status, kDevOk, kDevTimeout) == kDevOk) {
          a.status[1] = u;
          a.status[2] = d0;
          a.status[3] = (int)p.dst;
        }
        gave_up = true;
        ok = true;
      }
    }
  }
  // Give up as a warp, so that no lane leaves while the others vote again.
  gave_up = __any_sync(0xffffffffu, gave_up);
  if (!p.valid || gave_up) return !gave_up;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (i < nb) {
      E::st_out(reinterpret_cast<V*>(a.out[d0 + i]) + p.dst, x[i]);
      E::st_push(reinterpret_cast<V*>(a.box[d0 + i]) + p.dst, E::sentinel());
    }
  }
  return true;
}

// TPC > 0: tp known at compile time, all TP consumer elements in flight at
// once. TPC == 0: any tp, consumer ranks in batches of 4.
template <typename V, int TPC>
__global__ void __launch_bounds__(512) gather_kernel(const __grid_constant__ GatherArgs a) {
  using E = Elem<V>;
  constexpr int NB = TPC > 0 ? TPC : 4;
  const int tp = TPC > 0 ? TPC : a.tp;
  const int N = a.M * tp * a.chunks;  // units
  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  const int cons = (g + 1 == G) ? 0 : g + 1;  // the CTA whose pushes we consume
  const int iters = (N + G - 1) / G;

  // One load per warp of one address: every lane sees the same value.
  const int status0 = ld_relaxed_s32(a.status);

  for (int t = 0; t <= iters; ++t) {
    // Loads first (push source of iteration t, poll of iteration t-1), so that
    // their latencies overlap; then the push stores; then the poll.
    const int up = t * G + g;
    const bool do_push = t < iters && up < N;
    UnitPos pp{};
    V xs = E::none();
    if (do_push) {
      pp = unit_pos(a, tp, up);
      if (pp.valid && pp.r != a.skip_rank)
        xs = E::ld_shard(reinterpret_cast<const V*>(a.shard[pp.r]) + pp.src);
    }
    const int uc = (t - 1) * G + cons;
    const bool do_cons = t >= 1 && uc < N;
    UnitPos pc{};
    V x[NB];
    if (do_cons) {
      pc = unit_pos(a, tp, uc);
#pragma unroll
      for (int i = 0; i < NB; ++i)
        x[i] = (pc.valid && i < tp) ? E::ld_poll(reinterpret_cast<const V*>(a.box[i]) + pc.dst)
                                    : E::none();
    }
    if (status0 != kDevOk) return;  // handle in error state: no device work
    if (do_push && pp.valid && pp.r != a.skip_rank) {
      const V y = E::rewrite(xs);
      for (int d = 0; d < tp; ++d) E::st_push(reinterpret_cast<V*>(a.box[d]) + pp.dst, y);
    }
    if (do_cons) {
      if (!finish_consume<V, NB>(a, 0, tp < NB ? tp : NB, pc, x, uc)) return;
      for (int d0 = NB; d0 < tp; d0 += NB) {  // only when TPC == 0 and tp > 4
        const int nb = tp - d0 < NB ? tp - d0 : NB;
#pragma unroll
        for (int i = 0; i < NB; ++i)
          x[i] = (pc.valid && i < nb)
                     ? E::ld_poll(reinterpret_cast<const V*>(a.box[d0 + i]) + pc.dst)
                     : E::none();
        if (!finish_consume<V, NB>(a, d0, nb, pc, x, uc)) return;
      }
    }
  }
}

__global__ void fill_u32_kernel(uint32_t* p, size_t n, uint32_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

template <typename V>
const void* pick_kernel(int tp) {
  switch (tp) {
    case 2: return reinterpret_cast<const void*>(&gather_kernel<V, 2>);
    case 4: return reinterpret_cast<const void*>(&gather_kernel<V, 4>);
    case 8: return reinterpret_cast<const void*>(&gather_kernel<V, 8>);
    case 16: return reinterpret_cast<const void*>(&gather_kernel<V, 16>);
    default: return reinterpret_cast<const void*>(&gather_kernel<V, 0>);
  }
}

const void* kernel_for(bool vec16, int tp) {
  return vec16 ? pick_kernel<uint4>(tp) : pick_kernel<uint32_t>(tp);
}

}  // namespace

cudaError_t gather_occupancy(bool vec16, int tp, int threads, int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kernel_for(vec16, tp),
                                                       threads, 0);
}

cudaError_t launch_gather(const GatherArgs& a, bool vec16, int ctas, int threads,
                          cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<GatherArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, kernel_for(vec16, a.tp), args);
}

cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t v, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_u32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace hg
