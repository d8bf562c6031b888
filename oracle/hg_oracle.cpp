// CPU oracle for the vocab-parallel LM-head logits gather on a two-parity
// Lamport mailbox.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
// statement of what the GPU path computes. Only the tests, the smoke check and
// the benchmark's CPU-baseline leg and reference arm may load it. It shares no code, header,
// constant or helper with the CUDA library, and the library never calls it.
//
// Source of the definition: the vLLM API page
// "vllm.models.kimi_k3.nvidia.specialized_decode.runtime.logits_gather"
// (module docstring, class HeadGather: docstring, __init__ and __call__), and
// the vLLM pull request "[Perf][Kimi-K3] Use the one-shot custom all-gather for
// TP logits" (section "Purpose": rank-order concat, padded-vocab slice).
//
// Readings taken where the pages leave a step open (all listed in the design
// notes of the repository):
//  * The sentinel word is the BF16 pair (+0, -0): element 2k = +0 = 0x0000 in
//    the low half of the little-endian 32-bit word, element 2k+1 = -0 = 0x8000
//    in the high half, so the word is 0x80000000.
//  * Only a data word exactly equal to the sentinel is rewritten, to the pair
//    (+0, +0) = 0x00000000. Every other word moves unchanged.
//  * The rank's own fragment also goes through its own mailbox (the push
//    targets every rank, the pushing rank included), so all TP outputs are
//    identical.
//  * Parity starts at 0 and flips on every served call; a call whose row count
//    is not served returns before the flip and changes nothing.
//  * The LM head multiplies hidden [M, K] by the rank's weight held in the
//    nn.Linear layout [W, K] (the page passes weight.shape[0] as the shard
//    width), i.e. logits[m][n] = sum_k hidden[m][k] * weight[n][k].
//
// Parity pinned by the tests: invariants I1-I7, an exhaustive brute force at
// TP=2, V=8, a hand-worked example; for the LM head closed forms and a library
// float64 matmul; for the row statistics numpy/scipy, closed forms and a
// hand-worked row. No function here is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// The two BF16 halves of the sentinel pair, written out from their IEEE-754
// bfloat16 encodings (sign bit 15, exponent 14..7, mantissa 6..0).
const uint32_t kBf16PosZero = 0x0000u;  // +0
const uint32_t kBf16NegZero = 0x8000u;  // -0: sign bit only

// Word = element 2k in bits 0..15, element 2k+1 in bits 16..31 (little endian).
uint32_t pair_word(uint32_t elem_even, uint32_t elem_odd) {
  return (elem_odd << 16) | elem_even;
}

const uint32_t kSentinel = pair_word(kBf16PosZero, kBf16NegZero);      // (+0, -0)
const uint32_t kSentinelSentAs = pair_word(kBf16PosZero, kBf16PosZero);  // (+0, +0)

struct OracleGather {
  int tp;         // TP virtual ranks
  int W;          // shard width in bf16 columns (even)
  int w;          // shard width in 32-bit words, W / 2
  int V;          // full vocab width in bf16 columns, tp * W
  int cap;        // mailbox rows
  std::vector<int> served;  // served[M] != 0 when row count M is served
  int parity;     // parity the next served call uses
  // box[d][q][m][k]: rank d's mailbox, parity q, row m, word k (k < tp * w).
  std::vector<uint32_t> box;

  size_t at(int d, int q, int m, int k) const {
    return (((size_t)d * 2 + q) * cap + m) * ((size_t)tp * w) + k;
  }
};

double bf16_to_double(uint16_t bits) {
  uint32_t f32 = (uint32_t)bits << 16;  // bf16 is the top half of an fp32
  float f;
  std::memcpy(&f, &f32, sizeof f);
  return (double)f;
}

}  // namespace

extern "C" {

uint32_t og_sentinel(void) { return kSentinel; }

// Construction: allocate every rank's [2, cap, V] mailbox and arm it with the
// sentinel (HeadGather.__init__: LamportRows(..., (2, cap, words * tp),
// PAIR_SENT)); parity starts at 0. rows lists the served row counts; cap must
// be at least max(rows) (the page sets cap = max(rows)). Returns NULL for
// arguments that describe no valid gather.
void* og_create(int tp, int shard_cols, int cap, const int* rows, int nrows) {
  if (tp < 1 || shard_cols < 2 || shard_cols % 2 != 0 || cap < 1) return nullptr;
  if (nrows < 0 || (nrows > 0 && rows == nullptr)) return nullptr;
  OracleGather* g = new OracleGather;
  g->tp = tp;
  g->W = shard_cols;
  g->w = shard_cols / 2;
  g->V = tp * shard_cols;
  g->cap = cap;
  g->served.assign(cap + 1, 0);
  if (nrows == 0) {
    for (int m = 1; m <= cap; ++m) g->served[m] = 1;
  } else {
    for (int i = 0; i < nrows; ++i) {
      if (rows[i] < 1 || rows[i] > cap) { delete g; return nullptr; }
      g->served[rows[i]] = 1;
    }
  }
  g->parity = 0;
  g->box.assign((size_t)tp * 2 * cap * tp * g->w, kSentinel);
  return g;
}

void og_destroy(void* h) { delete static_cast<OracleGather*>(h); }

int og_parity(const void* h) { return static_cast<const OracleGather*>(h)->parity; }

// Rank d's mailbox for parity q, [cap][tp * w] words, for inspection.
const uint32_t* og_mailbox(const void* h, int d, int q) {
  const OracleGather* g = static_cast<const OracleGather*>(h);
  return &g->box[g->at(d, q, 0, 0)];
}

// One gather call (HeadGather.__call__ and the kernel behaviour described in
// the module docstring).
//   shard: [tp][M][w] words, rank r's [M, W] bf16 logits viewed as int32.
//   out:   [tp][M][tp * w] words, rank d's [M, V] bf16 output.
// Returns 0 on success; -1 when M is not served (no state change: the page's
// call falls back to its stock gather there); -2 when some polled word is still
// the sentinel (the
// poll would never finish; cannot happen when every rank pushes).
int og_call(void* h, int M, const uint32_t* shard, uint32_t* out) {
  OracleGather* g = static_cast<OracleGather*>(h);
  if (M < 1 || M > g->cap || !g->served[M]) return -1;

  const int q = g->parity;  // box.view(self.parity)
  g->parity ^= 1;           // self.parity ^= 1

  const int tp = g->tp, w = g->w;
  const int row_words = tp * w;

  // Push: rank r's row m, word j, lands at column r * w + j of row m of every
  // rank's mailbox; the sentinel word is sent as (+0, +0).
  for (int r = 0; r < tp; ++r) {
    for (int m = 0; m < M; ++m) {
      for (int j = 0; j < w; ++j) {
        uint32_t x = shard[((size_t)r * M + m) * w + j];
        uint32_t y = (x == kSentinel) ? kSentinelSentAs : x;
        for (int d = 0; d < tp; ++d) g->box[g->at(d, q, m, r * w + j)] = y;
      }
    }
  }

  // Poll: every word of rows m < M of rank d's mailbox must have arrived
  // (differ from the sentinel) before it is read.
  for (int d = 0; d < tp; ++d)
    for (int m = 0; m < M; ++m)
      for (int k = 0; k < row_words; ++k)
        if (g->box[g->at(d, q, m, k)] == kSentinel) return -2;

  // Copy the row to the output and re-arm the mailbox word with the sentinel.
  for (int d = 0; d < tp; ++d) {
    for (int m = 0; m < M; ++m) {
      for (int k = 0; k < row_words; ++k) {
        out[((size_t)d * M + m) * row_words + k] = g->box[g->at(d, q, m, k)];
        g->box[g->at(d, q, m, k)] = kSentinel;
      }
    }
  }
  return 0;
}

// Padded-vocab slice after the gather (pull request, "Purpose"): keep the
// first v_real bf16 columns of each [M, V] row.
void og_slice_bf16(const uint16_t* out, int M, int V, int v_real, uint16_t* sliced) {
  for (int m = 0; m < M; ++m)
    for (int c = 0; c < v_real; ++c)
      sliced[(size_t)m * v_real + c] = out[(size_t)m * V + c];
}

// Sampler statistics of one gathered row. The API page's module docstring
// notes that the sentinel rewrite changes no value a sampler computes with
// (+0 and -0 compare, add and exponentiate alike); these are such values.
// Over the V bf16 values x_c of the row,
//   max_logit = max_c x_c
//   argmax    = the smallest c with x_c == max_logit
//   sum_exp   = sum over c with x_c != -inf of exp(x_c - max_logit)
// in double precision. A row of only -inf values has sum_exp 0.
void og_row_stats(const uint16_t* row, int V, double* max_logit, int* argmax, double* sum_exp) {
  double mx = -std::numeric_limits<double>::infinity();
  int arg = 0;
  for (int c = 0; c < V; ++c) {
    double x = bf16_to_double(row[c]);
    if (x > mx) { mx = x; arg = c; }
  }
  double s = 0.0;
  for (int c = 0; c < V; ++c) {
    double x = bf16_to_double(row[c]);
    if (x != -std::numeric_limits<double>::infinity()) s += std::exp(x - mx);
  }
  *max_logit = mx;
  *argmax = arg;
  *sum_exp = s;
}

// Vocab-parallel LM head of one rank, in double precision:
//   logits[m][n - n0] = sum_{k=0}^{K-1} hidden[m][k] * weight[n][k]
// for rows m < M and vocab columns n0 <= n < n1. hidden is [M][K] bf16 bits,
// weight is [W][K] bf16 bits (nn.Linear layout), logits is [M][n1 - n0].
// The sum runs over k in increasing order.
void og_lm_head_f64(const uint16_t* hidden, const uint16_t* weight, int M, int K,
                    int n0, int n1, double* logits) {
  for (int m = 0; m < M; ++m) {
    for (int n = n0; n < n1; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += bf16_to_double(hidden[(size_t)m * K + k]) *
               bf16_to_double(weight[(size_t)n * K + k]);
      logits[(size_t)m * (n1 - n0) + (n - n0)] = acc;
    }
  }
}

}  // extern "C"
