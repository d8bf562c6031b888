// Fused LM-head producer: the vocab-parallel lm_head GEMM whose epilogue
// pushes its bf16 logits straight into every rank's Lamport mailbox, followed,
// in the same persistent kernel, by the poll / copy / re-arm of the gather.
//
// What it computes (vLLM API page "vllm.models.kimi_k3.nvidia.
// specialized_decode.runtime.logits_gather", module docstring: the
// vocab-parallel lm_head yields [M, V / TP] per rank, then the gather): for
// every virtual rank r,
//   logits_r[m][n] = bf16_rn( sum_k hidden_r[m][k] * weight_r[n][k] )
// with fp32 accumulation (weight_r in the nn.Linear layout [W, K]), and then
// exactly the gather of hg_gather on those logits: the sentinel word (+0, -0)
// is sent as (+0, +0) into row m, word column r * W / 2 of every rank's
// mailbox, and each rank polls, copies its row to the [M, V] output and
// re-arms.
//
// GEMM (tcgen05, swap-AB). The vocab is the MMA's M dimension (128 weight rows
// per tile) and the M <= 16 hidden rows, zero-padded, are its N = 16. Per
// 64-wide K block, TMA loads a [128 x 64] weight tile (16 KB) and the [16 x
// 64] hidden tile (2 KB) into one of kStages shared-memory stages with 128-byte
// swizzle (the canonical K-major layout of the shared-memory descriptors); one
// elected thread issues four 128x16x16 bf16 MMAs into an fp32 accumulator in
// tensor memory (two accumulators of 16 columns, so that the epilogue of one
// tile overlaps the MMAs of the next). Warp 0 is the TMA producer, warp 1 the
// MMA issuer (and owner of the TMEM allocation), warps 2..5 the epilogue: each
// reads its 32 TMEM lanes (= 32 vocab rows) with tcgen05.ld, rounds to bf16,
// packs column pairs into 32-bit words, stages them in shared memory, and
// stores them as 16-byte vectors, sentinel rewritten, into all TP mailboxes
// (kept in L2, evict-last). The GEMM streams each weight byte from HBM once
// (evict-first), so the kernel is bound by HBM bandwidth on the weights.
//
// Tail split. Tiles are dealt round-robin to the CTAs (one CTA per SM, all
// co-resident: cooperative launch): every CTA takes full_waves whole tiles.
// The tail tiles left over (fewer than the CTAs) would leave most SMs idle
// while a few stream one more tile, so when there are at most half as many
// tail tiles as CTAs each is split along K into `split` parts on `split`
// CTAs. The part-0 CTA (the owner) keeps its fp32 partial in registers; every
// other part writes its partial [128 x M] into a split cell, and the owner
// polls the cell, adds it, re-arms the cell, rounds and pushes. A split cell
// is a Lamport cell like a mailbox row: armed with 0xffffffff in every word
// (a NaN; a partial with that bit pattern is written as the NaN 0x7fffffff
// instead, the same value to the addition), written with relaxed stores,
// polled until no armed word is left, and re-armed by its reader.
//
// Gather. CTA g consumes the tiles that CTA g+1 (mod G) pushed (its whole
// tiles and the tail tile it owns): it polls them in every rank's mailbox,
// copies them to the outputs and re-arms, as the gather kernel does. The
// epilogue warps do this one item behind their own pushes, so the gather
// overlaps the weight stream; the last one or two tiles are consumed by all
// threads after the CTA's own tiles. Every wait in this kernel (mbarriers and
// polls) is bounded by %globaltimer; on expiry the kernel records the error
// in the status block and stops issuing work. Before it frees its tensor
// memory and returns, the TMA thread waits for every copy it issued to land
// (the full barrier of each stage it filled) and the MMA thread for every MMA
// it issued to complete (a final commit): those waits end because that work
// needs nothing from any other CTA, so they are bounded by time only.

#include <cuda.h>
#include <cuda_bf16.h>

#include "hg_internal.cuh"

namespace hg {
namespace fused {
namespace {

constexpr int kTileN = 128;      // weight rows (vocab columns) per tile: MMA M
constexpr int kBlockK = 64;      // K per stage: one 128-byte swizzle atom of bf16
constexpr int kMmaN = 16;        // padded hidden rows: MMA N
constexpr int kMmaK = 16;        // K per tcgen05.mma of kind::f16
constexpr int kStages = 8;
constexpr uint32_t kABytes = kTileN * kBlockK * 2;  // 16384
constexpr uint32_t kBBytes = kMmaN * kBlockK * 2;   // 2048
constexpr int kAccCols = 16;     // fp32 columns of one accumulator
constexpr uint32_t kTmemCols = 32;  // two accumulators (power of two >= 32)
constexpr int kThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kPollBatch = 8;    // gather phase: mailbox vectors per thread in flight
// Per epilogue warp, its [16 rows m][16 words] of packed logits, staged so that
// the push moves 16-byte vectors.
constexpr size_t kStageWordsPerWarp = (size_t)kMmaN * 16;
constexpr size_t kSmemBytes = (size_t)kStages * (kABytes + kBBytes) + 1024 /*align*/ + 256 +
                              4 * kStageWordsPerWarp * sizeof(uint32_t);

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A bf16 (bits 7-9 = 1), B bf16 (bits 10-12 = 1), A and B K-major (bits 15,
// 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(kMmaN >> 3) << 17) | ((uint32_t)(kTileN >> 4) << 24);

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// whose 8-row groups are 1024 bytes apart: start address >> 4 (bits 0-13),
// leading byte offset 16 >> 4 (bits 16-29, unused by this layout), stride
// byte offset 1024 >> 4 (bits 32-45), descriptor version 1 (bits 46-47),
// swizzle mode 128B = 2 (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void mma_bf16_f32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kInstrDesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}

__device__ __forceinline__ uint4 ld_poll_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Relaxed store into a mailbox or a split cell, kept in L2 ahead of the weight
// stream (evict-last): every call writes and re-arms the same mailbox lines,
// and written back to HBM they would be mixed into the weight stream (TP8,
// V=163840, K=7168: M=8 364.5 -> 357.7 us, M=16 384.2 -> 379.4 us per call).
__device__ __forceinline__ void st_relaxed_v4(uint4* p, uint4 v) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
      "st.relaxed.gpu.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, pol;\n\t}" ::"l"(p),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
      : "memory");
}

// Output store, evict-first: the caller reads the outputs once, and the L2 is
// better spent on the mailboxes (as in the gather kernel).
__device__ __forceinline__ void st_out_v4(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ bool arrived_v4(uint4 v) {
  return v.x != kSentinel && v.y != kSentinel && v.z != kSentinel && v.w != kSentinel;
}

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t failed;
};
static_assert(sizeof(Shared) <= 256, "barriers must fit the 256 bytes kept after the stages");
static_assert(kSmemBytes <= 227 * 1024, "dynamic shared memory above the per-CTA limit");

__device__ __forceinline__ void raise_error(const FusedArgs& a, int where) {
  if (atomicCAS(a.status, kDevOk, kDevTimeout) == kDevOk) {
    a.status[1] = -1;
    a.status[2] = where;
    a.status[3] = (int)blockIdx.x;
  }
}

// Bounded wait on an mbarrier phase. False: time limit or an error raised
// elsewhere (recorded in the status block).
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, const FusedArgs& a, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > a.timeout_ns || ld_relaxed_s32(a.status) != kDevOk) {
      raise_error(a, where);
      return false;
    }
  }
}

// Wait for work this CTA issued itself (TMA copies into its shared memory,
// its MMAs). That work completes without any other CTA, so the wait does not
// give up when another CTA raises an error; it is bounded by time alone, and
// on expiry it records the error and returns false (a last resort).
__device__ bool mbar_wait_own(uint64_t* bar, uint32_t parity, const FusedArgs& a, int where) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      raise_error(a, where);
      return false;
    }
  }
  return true;
}

// One work item of a CTA: a tile (rank r's vocab rows t * 128 ..) and the
// K-block range [kb0, kb1) it covers; part -1 for a whole tile, else the
// part of split tail tile j.
struct Item {
  int tile, kb0, kb1, part, j;
};

// Work items of CTA g: full_waves whole tiles, then at most one tail item.
__device__ __forceinline__ int item_count(const FusedArgs& a, int g) {
  const bool tail = a.split <= 1 ? g < a.tail : g < a.tail * a.split;
  return a.full_waves + (tail ? 1 : 0);
}

__device__ __forceinline__ Item item_at(const FusedArgs& a, int g, int G, int i, int kblocks) {
  if (i < a.full_waves) return Item{g + i * G, 0, kblocks, -1, -1};
  if (a.split <= 1) return Item{a.full_waves * G + g, 0, kblocks, -1, -1};
  const int j = g / a.split, p = g - j * a.split;
  return Item{a.full_waves * G + j, p * kblocks / a.split, (p + 1) * kblocks / a.split, p, j};
}

// Words of split cell (tail tile j, part p >= 1) for vocab row `row`.
__device__ __forceinline__ uint32_t* split_cell(const FusedArgs& a, int j, int p, int row) {
  return a.split_cells + ((size_t)(j * (a.split - 1) + (p - 1)) * 128 + (size_t)row) * 16;
}

// Tiles CTA c pushed (its whole tiles, then the tail tile it owns, if any):
// count, and the k-th of them.
__device__ __forceinline__ int own_tail_of(const FusedArgs& a, int c, int G) {
  if (a.split <= 1) return c < a.tail ? a.full_waves * G + c : -1;
  return (c % a.split == 0 && c / a.split < a.tail) ? a.full_waves * G + c / a.split : -1;
}

// Poll tile `it` (pushed by another CTA) in every rank's mailbox until it has
// arrived, copy it to the outputs and re-arm it: this thread's share is
// vectors tid, tid + nthr, ..., kPollBatch of them in flight at once. False
// when a poll gave up (recorded in the status block).
__device__ bool consume_tile(const FusedArgs& a, int it, size_t parity_off, int tid, int nthr) {
  const int V = a.tp * a.W;
  const int per_row = kTileN / 8;                  // 16-byte vectors of a tile row
  const int per_item = a.tp * a.M * per_row;       // 16-byte vectors of a tile, all ranks
  const int r = it / a.tiles_per_rank;
  const int t = it - r * a.tiles_per_rank;
  const uint4 sent = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  // Vector j: rank d's mailbox, row m, 16-byte vector vv of the tile.
  auto word_off = [&](int j, int* d) {
    *d = j / (a.M * per_row);
    const int rem = j - *d * (a.M * per_row);
    const int m = rem / per_row;
    const int vv = rem - m * per_row;
    return (size_t)m * (V / 2) + (size_t)r * (a.W / 2) + (size_t)t * (kTileN / 2) +
           (size_t)vv * 4;  // in words
  };
  for (int base = tid; base < per_item; base += nthr * kPollBatch) {
    uint4 x[kPollBatch];
#pragma unroll
    for (int k = 0; k < kPollBatch; ++k) {
      const int j = base + k * nthr;
      if (j < per_item) {
        int d;
        const size_t off = word_off(j, &d);
        x[k] = ld_poll_v4(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint32_t*>(a.box[d]) + parity_off + off));
      }
    }
#pragma unroll
    for (int k = 0; k < kPollBatch; ++k) {
      const int j = base + k * nthr;
      if (j >= per_item) continue;
      int d;
      const size_t off = word_off(j, &d);
      uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(a.box[d]) + parity_off + off);
      if (!arrived_v4(x[k])) {
        const unsigned long long t0 = globaltimer_ns();
        do {
          x[k] = ld_poll_v4(p);
          if (arrived_v4(x[k])) break;
          if (globaltimer_ns() - t0 > a.timeout_ns || ld_relaxed_s32(a.status) != kDevOk) {
            raise_error(a, 6);
            return false;
          }
        } while (true);
      }
      st_out_v4(reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(a.out[d]) + off), x[k]);
      st_relaxed_v4(p, sent);
    }
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned operand stages (the 128-byte swizzle repeats every 1024).
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sA = base;
  unsigned char* sB = base + (size_t)kStages * kABytes;
  Shared* sh = reinterpret_cast<Shared*>(sB + (size_t)kStages * kBBytes);
  uint32_t* const stage_words = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(sh) + 256);

  const int warp = (int)threadIdx.x >> 5;
  const int lane = (int)threadIdx.x & 31;
  // Timeline record (measurement only): slots of this CTA, written by one thread.
  unsigned long long* const tl =
      a.timeline ? a.timeline + (size_t)blockIdx.x * kTimelineSlots : nullptr;
  if (tl && threadIdx.x == 0) tl[kFusedTlEntry] = globaltimer_ns();

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Device-resident parity: this CTA's copy g (every thread reads it; the CTA
  // flips its share of the copies once every thread is past this point).
  int parity = 0;
  if (a.parity_words) parity = ld_relaxed_s32(a.parity_words + blockIdx.x);
  const size_t parity_off = (size_t)parity * a.parity_stride_words;  // in 32-bit words
  if (ld_relaxed_s32(a.status) != kDevOk) return;  // unrecovered error: no work

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->acc_full[b], 1);
      mbar_init(&sh->acc_empty[b], 4);  // one arrive per epilogue warp
    }
    mbar_init(&sh->drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  if (tl && threadIdx.x == 0) tl[kFusedTlSetup] = globaltimer_ns();

  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  const int kblocks = a.K / kBlockK;
  const int n_items = item_count(a, g);
  // The CTA whose pushes this one consumes, and its tiles.
  const int cons = (g + 1 == G) ? 0 : g + 1;
  const int cons_tail = own_tail_of(a, cons, G);
  const int n_cons = a.full_waves + (cons_tail >= 0 ? 1 : 0);
  auto cons_tile = [&](int k) { return k < a.full_waves ? cons + k * G : cons_tail; };

  if (warp == 0) {
    // TMA producer.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // stage fills issued; fill j goes to stage j % kStages
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item_at(a, g, G, i, kblocks);
        const int r = w.tile / a.tiles_per_rank;
        const int t = w.tile - r * a.tiles_per_rank;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(&sh->empty[stage], phase ^ 1u, a, 1)) { ok = false; break; }
          mbar_expect_tx(&sh->full[stage], kABytes + kBBytes);
          tma_load_2d(sA + (size_t)stage * kABytes, &a.tm_w[r], kb * kBlockK, t * kTileN,
                      &sh->full[stage], pol_w);
          tma_load_2d(sB + (size_t)stage * kBBytes, &a.tm_h[r], kb * kBlockK, 0,
                      &sh->full[stage], pol_h);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Every copy issued must land before the CTA's shared memory goes: wait
      // for the last fill of each stage (fill j completes the phase of parity
      // (j / kStages) & 1 of stage j % kStages; a stage is refilled only after
      // its previous fill was consumed, so no later phase can be pending).
      // After a normal run the MMA thread has already seen every fill land.
      const int last = issued - 1;
      for (int s = 0; s < kStages && s <= last; ++s) {
        const int j = last - (last - s) % kStages;
        mbar_wait_own(&sh->full[s], (uint32_t)((j / kStages) & 1), a, 8);
      }
    }
  } else if (warp == 1) {
    // MMA issuer.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item_at(a, g, G, i, kblocks);
        if (!mbar_wait(&sh->acc_empty[acc], acc_phase ^ 1u, a, 2)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * kAccCols);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(&sh->full[stage], phase, a, 3)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + (size_t)stage * kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + (size_t)stage * kBBytes));
#pragma unroll
          for (int k = 0; k < kBlockK / kMmaK; ++k) {
            // K step of 16 bf16 = 32 bytes = 2 in the start-address field.
            mma_bf16_f32(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                         (kb != w.kb0 || k != 0) ? 1u : 0u);
          }
          mma_commit(&sh->empty[stage]);  // stage free once these MMAs have read it
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&sh->acc_full[acc]);  // accumulator ready
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      // Every MMA this thread issued must complete before TMEM is freed (and
      // before the stages they read go): a commit tracks all of them.
      mma_commit(&sh->drain);
      mbar_wait_own(&sh->drain, 0, a, 4);
    }
  } else {
    // Epilogue: warps 2..5; warp w reads TMEM lanes 32 * (w % 4) ...
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // vocab row within the tile
    const int V = a.tp * a.W;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = 0; i < n_items; ++i) {
      const Item w = item_at(a, g, G, i, kblocks);
      // Every lane waits; the vote reconverges the warp before the warp-wide
      // tcgen05.ld and makes the give-up decision the same for all lanes.
      const bool ready = mbar_wait(&sh->acc_full[acc], acc_phase, a, 5);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      uint32_t v[16];
      tmem_ld_32x32b_x16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kAccCols), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

      const int nvec = (a.M + 3) / 4;  // 16-byte vectors of a cell row that hold rows m < M
      if (w.part > 0) {
        // A later part of a split tail tile: hand the fp32 partial to part 0.
        uint32_t* c = split_cell(a, w.j, w.part, row);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < nvec) {
            uint4 x;
            x.x = v[4 * q] == kSplitArmed ? kSplitArmedAs : v[4 * q];
            x.y = v[4 * q + 1] == kSplitArmed ? kSplitArmedAs : v[4 * q + 1];
            x.z = v[4 * q + 2] == kSplitArmed ? kSplitArmedAs : v[4 * q + 2];
            x.w = v[4 * q + 3] == kSplitArmed ? kSplitArmedAs : v[4 * q + 3];
            st_relaxed_v4(reinterpret_cast<uint4*>(c) + q, x);
          }
        }
      } else {
        if (w.part == 0) {
          // Part 0 of a split tail tile: add the other parts' partials (in part
          // order), polling their cells, and re-arm the cells.
          bool got = true;
          for (int p = 1; p < a.split && got; ++p) {
            uint4* c = reinterpret_cast<uint4*>(split_cell(a, w.j, p, row));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (q < nvec && got) {
                uint4 x = ld_poll_v4(c + q);
                const unsigned long long t0 = globaltimer_ns();
                while (x.x == kSplitArmed || x.y == kSplitArmed || x.z == kSplitArmed ||
                       x.w == kSplitArmed) {
                  if (globaltimer_ns() - t0 > a.timeout_ns || ld_relaxed_s32(a.status) != kDevOk) {
                    raise_error(a, 7);
                    got = false;
                    break;
                  }
                  x = ld_poll_v4(c + q);
                }
                if (got) {
                  v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) + __uint_as_float(x.x));
                  v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + __uint_as_float(x.y));
                  v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + __uint_as_float(x.z));
                  v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + __uint_as_float(x.w));
                  st_relaxed_v4(c + q, make_uint4(kSplitArmed, kSplitArmed, kSplitArmed, kSplitArmed));
                }
              }
            }
          }
          if (!__all_sync(0xffffffffu, got)) break;
        }

        const int r = w.tile / a.tiles_per_rank;
        const int t = w.tile - r * a.tiles_per_rank;
        uint32_t* lg = reinterpret_cast<uint32_t*>(a.logits[r]);
        // Pack column pairs (row, row + 1) into words (low half = even column) and
        // stage the warp's [M][16] words (its 32 vocab rows) in shared memory:
        // then lane l takes row m = l / 4 (and m + 8) and the 4 words, 8 vocab
        // rows, of group l % 4, and pushes them as one 16-byte vector per rank
        // instead of one 4-byte word per rank from every other lane.
        uint32_t* const stage = stage_words + (size_t)(warp - 2) * kStageWordsPerWarp;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          if (m < a.M) {
            const float mine = __uint_as_float(v[m]);
            const float next = __shfl_down_sync(0xffffffffu, mine, 1);
            if ((lane & 1) == 0) stage[m * 16 + (lane >> 1)] = pack_bf16x2(mine, next);
          }
        }
        __syncwarp();
        const int grp = lane & 3;
        // Word column of the group within rank r's row: tile t, this warp's 32
        // rows (16 words), group grp (4 words).
        const size_t wcol = (size_t)t * (kTileN / 2) + (size_t)quarter * 16 + (size_t)grp * 4;
        const bool lg_vec = lg && (reinterpret_cast<uintptr_t>(lg) & 15) == 0;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const int m = (lane >> 2) + pass * 8;
          if (m < a.M) {
            const uint4 x = *reinterpret_cast<const uint4*>(stage + m * 16 + grp * 4);
            if (lg) {
              uint32_t* dst = lg + (size_t)m * (a.W / 2) + wcol;
              if (lg_vec) {
                *reinterpret_cast<uint4*>(dst) = x;
              } else {
                dst[0] = x.x;
                dst[1] = x.y;
                dst[2] = x.z;
                dst[3] = x.w;
              }
            }
            uint4 y;
            y.x = x.x == kSentinel ? kSentAs : x.x;
            y.y = x.y == kSentinel ? kSentAs : x.y;
            y.z = x.z == kSentinel ? kSentAs : x.z;
            y.w = x.w == kSentinel ? kSentAs : x.w;
            const size_t off = (size_t)m * (V / 2) + (size_t)r * (a.W / 2) + wcol;
            if (r != a.skip_rank)
              for (int d = 0; d < a.tp; ++d)
                st_relaxed_v4(reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(a.box[d]) +
                                                       parity_off + off),
                              y);
          }
        }
        __syncwarp();  // the next item rewrites the staged words
      }  // whole tile or part 0
      if (tl && warp == 2 && lane == 0 && i < kFusedTlPushN) tl[kFusedTlPush + i] = globaltimer_ns();
      // One item behind, the gather of the neighbour's tiles: its item i - 1
      // was pushed about one tile of weight streaming ago, so these polls
      // rarely wait, and the copy overlaps this CTA's next tile.
      if (i >= 1 && i - 1 < n_cons) {
        const bool ok = consume_tile(a, cons_tile(i - 1), parity_off, (int)threadIdx.x - 64, 128);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (tl && warp == 2 && lane == 0 && i - 1 < kFusedTlConsumeN)
          tl[kFusedTlConsume + i - 1] = globaltimer_ns();
      }
    }
    if (tl && warp == 2 && lane == 0) tl[kFusedTlLoopDone] = globaltimer_ns();
  }

  // All roles done (or stopped on an error): free the tensor memory. One
  // thread reads the status so that every thread takes the same branch.
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) sh->failed = ld_relaxed_s32(a.status) != kDevOk ? 1u : 0u;
  __syncthreads();
  tc_fence_after();
  const bool failed = sh->failed != 0;
  if (a.parity_words && !failed) {
    // Every thread of this CTA read copy g before the barriers above: flip
    // copies g + k * G (each copy flips exactly once per call).
    for (int e = (int)blockIdx.x + (int)threadIdx.x * (int)gridDim.x; e < a.parity_entries;
         e += kThreads * (int)gridDim.x)
      asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(a.parity_words + e),
                   "r"(parity ^ 1)
                   : "memory");
  }
  // The TMA thread and the MMA thread waited for their own copies and MMAs
  // above, before the barrier: nothing is in flight into shared or tensor
  // memory here.
  if (warp == 1) {
    __syncwarp();  // the warp-wide dealloc needs the whole warp converged
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if (failed) return;

  // The rest of the gather: the neighbour's tiles the epilogue loop has not
  // consumed (its last one or two), by every thread.
  for (int k = n_items >= 1 ? n_items - 1 : 0; k < n_cons; ++k)
    if (!consume_tile(a, cons_tile(k), parity_off, (int)threadIdx.x, kThreads)) return;
  if (tl && threadIdx.x == 0) tl[kFusedTlDone] = globaltimer_ns();
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// 2-D bf16 tensor map of a row-major [rows, K] matrix, box [box_rows, 64],
// 128-byte swizzle; rows beyond `rows` read as zero.
bool encode(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t K, uint32_t box_rows) {
  EncodeTiled fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBlockK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int fused_limits(int* max_tp, int* max_m, int* k_multiple, int* w_multiple) {
  *max_tp = kFusedMaxTp;
  *max_m = kMmaN;
  *k_multiple = kBlockK;
  *w_multiple = kTileN;
  return 0;
}

size_t split_cells_needed(int sms) {
  // tail * (split - 1) < tail * split <= grid <= one CTA per SM
  return (size_t)(sms > 0 ? sms : 1);
}

cudaError_t fused_launch(const FusedLaunch& l, cudaStream_t stream, int sms) {
  FusedArgs a;  // copied into the launch by cudaLaunchKernelExC
  // The dynamic shared-memory limit is a per-device attribute of the kernel:
  // set it on every launch, on the current device (a host call of well under
  // a microsecond beside a launch that streams the weights for hundreds).
  cudaError_t e = cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  for (int r = 0; r < l.tp; ++r) {
    if (!encode(&a.tm_w[r], l.weight[r], (uint64_t)l.W, (uint64_t)l.K, kTileN) ||
        !encode(&a.tm_h[r], l.hidden[r], (uint64_t)l.M, (uint64_t)l.K, kMmaN))
      return cudaErrorInvalidValue;
    a.box[r] = l.box[r];
    a.out[r] = l.out[r];
    a.logits[r] = l.logits ? l.logits[r] : nullptr;
  }
  for (int r = l.tp; r < kFusedMaxTp; ++r) {
    a.box[r] = nullptr;
    a.out[r] = nullptr;
    a.logits[r] = nullptr;
  }
  a.status = l.status;
  a.timeout_ns = l.timeout_ns;
  a.parity_words = l.parity_words;
  a.parity_entries = l.parity_entries;
  a.parity_stride_words = l.parity_stride_words;
  a.skip_rank = l.skip_rank;
  a.timeline = nullptr;
  a.tp = l.tp;
  a.W = l.W;
  a.K = l.K;
  a.M = l.M;
  a.tiles_per_rank = l.W / kTileN;
  const int items = l.tp * a.tiles_per_rank;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel, kThreads, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = sms * per_sm;
  if (l.max_ctas > 0 && grid > l.max_ctas) grid = l.max_ctas;
  if (grid > items) grid = items;
  if (l.timeline && grid <= l.timeline_ctas) a.timeline = l.timeline;
  // Work split: whole tiles in full waves; a tail of at most half the grid is
  // split along K (at most kMaxSplit parts, each of at least one K block) if
  // the handle has split cells for it.
  a.full_waves = items / grid;
  a.tail = items - a.full_waves * grid;
  a.split = 1;
  a.split_cells = nullptr;
  if (a.tail > 0 && 2 * a.tail <= grid && l.split_cells) {
    int split = grid / a.tail;
    if (split > kMaxSplit) split = kMaxSplit;
    if (split > l.K / kBlockK) split = l.K / kBlockK;
    if (split >= 2 && (size_t)a.tail * (split - 1) <= l.split_cell_count) {
      a.split = split;
      a.split_cells = l.split_cells;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&fused_kernel), args);
}

}  // namespace fused
}  // namespace hg
