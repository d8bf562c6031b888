// hg_gather_static: the logits gather for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc on their hot path or at all: a serving
// engine whose caching allocator has already reserved the GPU's free memory (a
// fresh cudaMalloc fails or fragments that pool), a plug-in loaded into a host
// framework that forbids allocations outside its own allocator, or a
// latency-critical loop that cannot afford cudaMalloc/cudaFree's implicit
// device synchronisation. hg_create allocates the mailboxes; this entry point
// instead keeps one mailbox set and the status words in a file-scope
// __device__ array of fixed size (HG_STATIC_MAILBOX_BYTES plus 256 bytes),
// which every GPU that loads the library holds until the process exits.
//
// Host code must not use the array's name as a device address: on the host it
// is only a stand-in. Its device address comes from cudaGetSymbolAddress, taken
// once per device, with that device current, by the first call made on that
// device (so the first call on a device should be made before any stream
// capture). The caller passes the shards and outputs as for hg_gather; they and
// the stream belong to the device that is current at the call (a stream of
// another device is refused).
//
// Every call shares the array and finds it as the last call left it. Each call
// therefore clears the status words and re-arms the mailbox region it uses
// (every word = the sentinel) before its gather kernel, all on the caller's
// stream. Calls whose work overlaps on the GPU (other streams, other threads)
// race on the array. The call allocates nothing: no cudaMalloc, no cudaFree,
// no allocating library routine.

#include <mutex>

#include "hg_internal.cuh"

namespace {

constexpr size_t kMailboxBytes = HG_STATIC_MAILBOX_BYTES;
constexpr size_t kStatusOffset = kMailboxBytes;  // status words follow the mailboxes
constexpr int kMaxDevices = 64;

// Mailboxes of all virtual ranks ([tp][M][V] bf16, one parity) and the status
// words. Aligned for 16-byte vector accesses.
static __device__ __align__(256) unsigned char g_scratch[kMailboxBytes + 256];

struct DeviceScratch {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_scratch on this device
  int sms = 0;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// Device address of g_scratch on the current device (set up on first use).
int scratch_for_current_device(DeviceScratch* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return HG_ERR_CUDA;
  if (dev >= kMaxDevices) return HG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& s = g_dev[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return HG_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
      return HG_ERR_CUDA;
    s.base = static_cast<unsigned char*>(p);
    s.sms = sms;
    s.ready = true;
  }
  *out = s;
  return HG_OK;
}

}  // namespace

extern "C" int hg_gather_static(int tp, int shard_cols, const void* const* shard_ptrs,
                                void* const* out_ptrs, int M, int* status_out,
                                hg_stream_t stream) {
  if (tp < 1 || tp > HG_MAX_TP || shard_cols < 2 || shard_cols % 2 != 0 || M < 1 ||
      !shard_ptrs || !out_ptrs)
    return HG_ERR_ARG;
  // Mailbox of this call: tp ranks x M rows x V = tp * W bf16 columns.
  const unsigned long long need =
      (unsigned long long)tp * (unsigned long long)M * tp * (unsigned long long)shard_cols * 2ull;
  if (need > kMailboxBytes) return HG_ERR_ARG;  // beyond HG_STATIC_MAILBOX_BYTES
  const bool vec16 = shard_cols % 8 == 0;
  const size_t align = vec16 ? 16 : 4;
  hg::GatherArgs a;
  for (int r = 0; r < tp; ++r) {
    if (!shard_ptrs[r] || !out_ptrs[r] ||
        reinterpret_cast<uintptr_t>(shard_ptrs[r]) % align != 0 ||
        reinterpret_cast<uintptr_t>(out_ptrs[r]) % align != 0)
      return HG_ERR_ARG;
    a.shard[r] = shard_ptrs[r];
    a.out[r] = out_ptrs[r];
  }
  DeviceScratch ds;
  int st = scratch_for_current_device(&ds);
  if (st != HG_OK) return st;
  // The array's address and the launches belong to the current device, so the
  // stream must too. The legacy and per-thread default streams always do.
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cs != nullptr && cs != cudaStreamLegacy && cs != cudaStreamPerThread) {
    int dev = -1, sdev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HG_ERR_CUDA;
    if (cudaStreamGetDevice(cs, &sdev) != cudaSuccess) {
      cudaGetLastError();  // an unknown stream handle: clear the error it set
      return HG_ERR_ARG;
    }
    if (sdev != dev) return HG_ERR_ARG;
  }

  const int wv = vec16 ? shard_cols / 8 : shard_cols / 2;
  const size_t rank_bytes = (size_t)M * tp * shard_cols * 2;  // one rank's [M][V]
  for (int d = 0; d < tp; ++d) a.box[d] = ds.base + (size_t)d * rank_bytes;
  for (int d = tp; d < HG_MAX_TP; ++d) {
    a.shard[d] = nullptr;
    a.out[d] = nullptr;
    a.box[d] = nullptr;
  }
  a.status = reinterpret_cast<int*>(ds.base + kStatusOffset);
  a.timeout_ns = 1000000000ull;
  a.tp = tp;
  a.wv = wv;
  a.M = M;
  a.skip_rank = -1;
  a.l2_prefetch = 1;

  // Launch shape: the library's fixed rule (elements per lane by tp and M,
  // widened from four rows on where that unloads the busiest SM; one CTA per
  // unit up to the co-resident maximum, beyond which the CTAs loop over the
  // units).
  hg::LaunchShape s;
  s.vpt = hg::default_vpt(tp, M);
  a.chunks = (wv + 32 * s.vpt - 1) / (32 * s.vpt);
  const long long units = (long long)M * tp * a.chunks;
  int per_sm = 0;
  if (hg::gather_occupancy(s, vec16, tp, &per_sm) != cudaSuccess || per_sm < 1) return HG_ERR_CUDA;
  const long long maxg = (long long)per_sm * ds.sms;
  s.ctas = (int)(units < maxg ? units : maxg);
  s.late = hg::trigger_late(s.ctas, units, maxg);
  if (hg::widen_units(tp, wv, M, ds.sms, vec16, &s, &a.chunks) != cudaSuccess)
    return HG_ERR_CUDA;

  // The array keeps the last call's contents: clear the status words and arm
  // this call's mailbox region, then gather, all in stream order.
  if (cudaMemsetAsync(a.status, 0, hg::kStatusWords * sizeof(int), stream) != cudaSuccess)
    return HG_ERR_CUDA;
  if (hg::launch_fill_u32(reinterpret_cast<uint32_t*>(ds.base), need / 4, hg::kSentinel,
                          stream) != cudaSuccess)
    return HG_ERR_CUDA;
  if (hg::launch_gather(a, s, vec16, stream, false) != cudaSuccess) return HG_ERR_CUDA;
  if (status_out &&
      cudaMemcpyAsync(status_out, a.status, sizeof(int), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return HG_ERR_CUDA;
  return HG_OK;
}
