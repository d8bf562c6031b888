// Measurement kernels that bound the gather's latency from below (hg_probe).
//
// At decode sizes the gather moves a few megabytes that stay in L2, so its
// time per call is set by latency, not bandwidth: the dependent launch, and
// a chain of memory round trips (the shard read, the push, the poll that sees
// it, the output and re-arm stores). These kernels are launched exactly as
// the gather is (a programmatic dependent launch on the caller's stream, the
// same grid and CTA size) and keep only part of its work:
//
//   empty    wait for the previous kernel, let the next one launch, return;
//   handoff  one 16-byte vector per lane pushed into the CTA's slot, the slot
//            of CTA g + 1 polled until it arrives, copied to an output and
//            re-armed: the gather's push -> poll -> copy -> re-arm chain for
//            one vector per lane, with no shard read.
//
// A call stream of either, replayed back to back, gives the time per call
// that the gather cannot go below with the same launch and the same
// cross-CTA handoff. The handoff slots are Lamport cells like the mailboxes:
// armed with the sentinel word, written with relaxed stores, polled with
// relaxed loads (bounded by %globaltimer) and re-armed by their reader. One
// set of slots suffices: the next launch waits for this one to complete
// before it touches memory, and by then every slot has been re-armed.

#include "hg_internal.cuh"

namespace hg {
namespace {

constexpr int kProbeMaxThreads = 512;
constexpr unsigned long long kProbeTimeoutNs = 1000000000ull;

__device__ __forceinline__ unsigned long long probe_clock_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(kProbeMaxThreads) probe_empty_kernel() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 probe_ld(const uint4* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void probe_st(uint4* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// slots and outs: [gridDim.x * blockDim.x] vectors each; status: one word.
__global__ void __launch_bounds__(kProbeMaxThreads)
    probe_handoff_kernel(uint4* slots, uint4* outs, int* status) {
  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  const int cons = g + 1 == G ? 0 : g + 1;
  const size_t mine = (size_t)g * blockDim.x + threadIdx.x;
  const size_t theirs = (size_t)cons * blockDim.x + threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // A token that is never the sentinel word (its first word is g < 2^31).
  probe_st(slots + mine, make_uint4((uint32_t)g, threadIdx.x, 1u, 2u));
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int st;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(st) : "l"(status) : "memory");
  if (st != 0) return;
  uint4 v = probe_ld(slots + theirs);
  unsigned long long t0 = 0;
  bool gave_up = false;
  for (;;) {
    bool done = v.x != kSentinel && v.y != kSentinel && v.z != kSentinel && v.w != kSentinel;
    if (!done) {
      const unsigned long long now = probe_clock_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > kProbeTimeoutNs) {
        atomicExch(status, 1);
        gave_up = true;
        done = true;
      }
    }
    if (__all_sync(0xffffffffu, done)) break;
    if (!done) v = probe_ld(slots + theirs);
  }
  if (__any_sync(0xffffffffu, gave_up)) return;
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(outs + mine), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
  probe_st(slots + theirs, make_uint4(kSentinel, kSentinel, kSentinel, kSentinel));
}

__global__ void probe_arm_kernel(uint4* slots, size_t n, int* status) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    slots[i] = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0;
}

}  // namespace
}  // namespace hg

extern "C" size_t hg_probe_scratch_bytes(int ctas, int threads) {
  if (ctas < 1 || threads < 32) return 0;
  // slots and outputs (one vector per thread each), then the status word
  return 2 * (size_t)ctas * threads * 16 + 16;
}

extern "C" int hg_probe(int kind, int ctas, int threads, void* scratch, hg_stream_t stream) {
  if (kind < 0 || kind > 2 || ctas < 1 || threads < 32 || threads % 32 != 0 ||
      threads > hg::kProbeMaxThreads)
    return HG_ERR_ARG;
  if (kind != 0 && (!scratch || reinterpret_cast<uintptr_t>(scratch) % 16 != 0))
    return HG_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t n = (size_t)ctas * threads;
  uint4* slots = static_cast<uint4*>(scratch);
  uint4* outs = slots + n;
  int* status = reinterpret_cast<int*>(outs + n);
  if (kind == 2) {
    size_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    hg::probe_arm_kernel<<<(unsigned)blocks, 256, 0, s>>>(slots, n, status);
    return cudaGetLastError() == cudaSuccess ? HG_OK : HG_ERR_CUDA;
  }
  const void* k = kind == 0 ? reinterpret_cast<const void*>(&hg::probe_empty_kernel)
                            : reinterpret_cast<const void*>(&hg::probe_handoff_kernel);
  if (kind == 1) {
    // Every CTA waits on its neighbour's store: the whole grid must be resident.
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, 0) != cudaSuccess)
      return HG_ERR_CUDA;
    if ((long long)per_sm * sms < ctas) return HG_ERR_ARG;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (kind == 0) {
    e = cudaLaunchKernelEx(&cfg, hg::probe_empty_kernel);
  } else {
    e = cudaLaunchKernelEx(&cfg, hg::probe_handoff_kernel, slots, outs, status);
  }
  return e == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}
