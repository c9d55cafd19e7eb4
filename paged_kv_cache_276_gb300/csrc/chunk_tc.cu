// Causal query chunks on the 5th-generation tensor cores: the 16-token chunk
// of a decode step, and prompt chunks of any length (chunked prefill).
//
// For one KV head, a query tile of 128 rows holds 128 / G tokens x the G query
// heads of the group (row r = token r / G, head r % G).  Over each tile of T
// keys of the paged cache (T = 128 in prefill, 64 in the decode chunk):
//     S  = Q K^T                     tcgen05.mma, M 128 x N T x K 128 -> TMEM
//     P  = exp2(S * scale*log2e - m)  softmax warps, one query row per thread,
//                                    bf16 in TMEM (prefill: over the scores)
//     O += P V                       tcgen05.mma, M 128 x N 128 x K T -> TMEM
// with the running max / sum of online softmax (x321.org "The serving
// bottleneck is not just FLOPs", section "First understand what the KV cache
// is storing"; the causal chunk and chunked prefill follow the same page's
// section "Continuous batching is the other half of the story").
//
// Two schedules drive the same pipeline (persistent grid, one CTA per SM):
//  * decode chunk (the newest q_len tokens of every sequence, q_len * G <= 128:
//    one query tile per sequence and KV head, its spare rows zero; a
//    single-token decode is q_len 1).
//    The (sequence, KV head, partition) items split each sequence's keys into
//    partitions and CTA c takes a contiguous range of them.  Consecutive items
//    of the same (sequence, KV head) accumulate into the same TMEM
//    accumulator; at the end of such a run the CTA writes one partial (max,
//    sum, unnormalised O) into the slot of the run's first partition and marks
//    the run's other partitions empty, and the split-K combine kernel merges
//    the slots.  A sequence with a single partition gets its bf16 output
//    directly.
//  * prefill (a chunk of its own length per sequence).  Batches of long
//    chunks: one item per (sequence, KV head, pair of query tiles), covering
//    every key the pair's last token sees; both query tiles are multiplied
//    against each key and value tile, so the key / value traffic per product
//    halves.  Batches of mostly short chunks (decode rows): one item per
//    (sequence, KV head, query tile).  Items of one (sequence, KV head) are
//    numbered together, longest first, and CTA c takes items c, c + grid,
//    c + 2 grid, ...  The CTAs that run at the same time then sweep the same
//    keys, so the re-reads hit L2.  Every item writes its bf16 output
//    directly; no workspace.
//
// Warp roles: 0-7 softmax (thread = row).  Warps 0-3 and 4-7 are two sets,
// each with its own running max / sum and its own TMEM accumulator: over a
// pair of query tiles set q takes query tile q against every key tile;
// otherwise set 0 takes the even key tiles of a run and set 1 the odd ones,
// merged exactly at the end of the run by set 0.  8 TMA producer of queries
// and keys, 9 score-product issuer (one lane) and tensor-memory owner, 10 P V
// product issuer (one lane), 11 TMA producer of values.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"
#include "merge.cuh"
#include "pkv.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;       // query rows per tile (tokens x group heads)
constexpr int kMaxStages = 5;    // K/V ring (at most)
constexpr int kTmemCols = 512;   // O: 2 x 128 columns (even / odd tiles), then the S (and P) buffers
constexpr int kKWarp = 8, kMmaWarp = 9, kPvWarp = 10, kVWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.f;    // lazy rescale threshold (log2 units)

// barrier indices (8 bytes each)
enum : int {
  B_Q_FULL0 = 0, B_Q_FULL1, B_Q_FREE0, B_Q_FREE1, B_O_FULL, B_O_FULL1, B_O_FREE, B_O_FREE1,
  B_S_FULL0, B_S_FULL1, B_S_FREE0, B_S_FREE1,
  B_P_FULL0, B_P_FULL1, B_P_LO0, B_P_LO1, B_PV_DONE0, B_PV_DONE1, B_STATS0, B_STATS1, B_STATS_FREE0,
  B_STATS_FREE1,
  B_K_FULL0, B_K_EMPTY0 = B_K_FULL0 + kMaxStages, B_V_FULL0 = B_K_EMPTY0 + kMaxStages,
  B_V_EMPTY0 = B_V_FULL0 + kMaxStages, B_COUNT = B_V_EMPTY0 + kMaxStages
};

// Tiles and shared-memory plan of each schedule.
//  * prefill (compute-bound): 128-key tiles.  S = Q K^T is one N = 128 product
//    per 16 head dims, and P V one K = 128 product.  Over single query tiles a
//    set writes its weights P over its own S buffer, so a score product waits
//    for the set's previous P V product (which reads that P); over pairs the
//    two sets share one S buffer and keep their P in columns of their own (the
//    kernel's tP0), so a score product only waits for the previous one to be
//    read.  Two key and two value stages.
//  * decode chunk (bandwidth-bound): 64-key tiles, 4 key and 4 value stages,
//    and P in its own buffers, so the score products run ahead of the P V
//    products: finer, deeper rings keep more copies in flight.
// Both keep two query tiles, then a ring of key tiles and a ring of value
// tiles.  A key stage is released as soon as its score product completes, a
// value stage after its P V product, so the keys can be fetched further ahead
// than the values.  The second query tile lets the producer load the next
// run's queries, and then its keys, while the current run is still in flight.
template <bool kPrefill, int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kHalves = D / 64;           // 64-column (128-byte) halves of a row
  static constexpr int kQHalf = kRows * 128;       // one half of the query tile
  static constexpr int kQBytes = kHalves * kQHalf;  // query tile: [half][128 rows][128 B]
  static constexpr int kTK = kPrefill ? 128 : 64;   // keys per tile
  static constexpr bool kPOverS = kPrefill;         // P stored over its S buffer
  static constexpr int kKVHalf = kTK * 128;         // one half of a key (or value) tile
  static constexpr int kKVBytes = kHalves * kKVHalf;  // key (or value) tile: [half][kTK rows][128 B]
  static constexpr int kStages = kPrefill ? 2 : 4;
  static constexpr int kQBufs = 2;
  static constexpr int kMaxSeqs = kPrefill ? 1024 : 2048;
  static constexpr int kSeqInts = kPrefill ? 4 : 2;  // per-sequence ints after the item prefix
  static constexpr int kSmemK = kQBufs * kQBytes;
  static constexpr int kSmemV = kSmemK + kStages * kKVBytes;
  static constexpr int kSmemStats = kSmemV + kStages * kKVBytes;  // float2 [2][128]: odd set's (max, sum)
  static constexpr int kSmemBars = kSmemStats + 2 * kRows * 8;
  static constexpr int kSmemSeq = kSmemBars + B_COUNT * 8 + 16;  // after the TMEM slot and the abort flag
  // tensor memory: O accumulators at 0 and D, S buffers at 2 D (+kTK); P in
  // the upper half of its S buffer (prefill: keys 0..63 over S columns 64..95,
  // keys 64..127 over 96..127, written after those scores are read) or after
  // the S buffers.  Prefill over pairs of query tiles uses the first S buffer
  // only and puts P where the second one starts (the kernel's tP0).
  static constexpr int kTmemS = 2 * D;
  static constexpr int kTmemP = kPOverS ? kTmemS + kTK / 2 : kTmemS + 2 * kTK;
  static constexpr int kPStride = kPOverS ? kTK : kTK / 2;        // columns between the two sets' P
  static_assert(kTmemP + kPStride + kTK / 2 <= kTmemCols, "tensor memory");
  static constexpr size_t bytes(int num_seqs) {
    return 1024 + kSmemSeq + (static_cast<size_t>(kSeqInts) * num_seqs + 1) * 4;
  }
};
static_assert(Layout<false, 128>::bytes(Layout<false, 128>::kMaxSeqs) <= 227 * 1024, "shared memory");
static_assert(Layout<true, 128>::bytes(Layout<true, 128>::kMaxSeqs) <= 227 * 1024, "shared memory");
static_assert(Layout<false, 128>::kStages <= kMaxStages && Layout<true, 128>::kStages <= kMaxStages, "stages");

struct TcParams {
  const int32_t *block_tables;
  const int32_t *seq_lens;
  const int32_t *q_start;  // prefill: [B + 1] first query row of each sequence
  __nv_bfloat16 *out;      // decode chunk: [B][q_len][Hq][D]; prefill: [total_q][Hq][D]
  float *ws_o;             // decode chunk: [B * q_len * Hq][P][D]
  float2 *ws_ml;           // decode chunk: [B * q_len * Hq][P]
  int32_t *status;
  int num_seqs, max_blocks, num_q_heads, num_kv_heads, num_blocks;
  int part_tokens, max_parts, oob_row;
  int total_q;             // prefill: query rows
  int group;               // query heads per KV head (G, 1..16)
  int tile_tok;            // query tokens per tile: floor(128 / G); rows tile_tok * G .. 127 are spare
  int q_len;               // decode chunk: query tokens per sequence (q_len * G <= 128)
  float scale_log2;
  // prefill: a host-built list of the items each CTA takes (null: CTA c takes
  // items c, c + grid, ...): [grid, n, offsets[grid + 1], item indices[n]]
  const int32_t *work;
};

// Walks (sequence, KV head, sub-item) in order; the sub-items of a sequence are
// its partitions (decode chunk) or its query tiles (prefill).
struct ItemWalker {
  int seq, head, part, nparts;
  __device__ void seek(const int *prefix, int num_seqs, int hkv, int it) {
    int lo = 0, hi = num_seqs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= it) lo = mid; else hi = mid;
    }
    seq = lo;
    nparts = (prefix[seq + 1] - prefix[seq]) / hkv;
    const int off = it - prefix[seq];
    head = off / nparts;
    part = off - head * nparts;
  }
  __device__ void next(const int *prefix, int num_seqs, int hkv) {
    if (++part < nparts) return;
    part = 0;
    if (++head < hkv) return;
    head = 0;
    if (++seq < num_seqs) nparts = (prefix[seq + 1] - prefix[seq]) / hkv;
  }
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Decode chunk: CTA c takes items [range_first(c), range_first(c + 1)): equal
// item counts.  (Equal key-tile counts were measured slower: the per-run
// cost at the end of every (sequence, KV head) run weighs as much as tiles.)
__device__ __forceinline__ int range_first(unsigned c, int total) {
  return static_cast<int>((static_cast<long long>(c) * total + gridDim.x - 1) / gridDim.x);
}

// Per-sequence values kept in shared memory.
struct SeqTab {
  const int *prefix;  // [B + 1] items before each sequence
  const int *lens;    // [B] clamped lengths
  const int *qs;      // prefill: [B] first query row
  const int *qc;      // prefill: [B] chunk length (0 for a bad q_start entry)
};

// One work item: a query tile (prefill: a pair of query tiles 2 qt and
// 2 qt + 1, the second one present when has_b) against the keys [k_lo, k_hi)
// of one sequence and KV head.  A run is a maximal sequence of items sharing
// one accumulator.
struct Item {
  int seq, head, qt, part, nparts, k_lo, k_hi;
  bool run_begin, run_end, has_b;
  bool skip;  // prefill split over keys: a partition past this query tile's keys (no work, no output)
};

// Prefill split over keys (part_tokens > 0): partitions per query tile of a
// sequence of L keys; 1 without the split.
__device__ __forceinline__ int split_parts(const TcParams &p, int L) {
  return p.part_tokens > 0 && L > 0 ? ceil_div(L, p.part_tokens) : 1;
}

// The items of this CTA in order (every role walks the same sequence).
// kPairs: prefill items are pairs of query tiles.
template <bool kPrefill, bool kPairs = false>
struct Sched {
  int it, end, step, total;
  ItemWalker w;
  Item x;

  __device__ void begin(const TcParams &p, const SeqTab &t, int total_items) {
    total = total_items;
    if (kPrefill && p.work) {
      // this CTA's range of the list; a list built for another grid size, or
      // a range outside it, is no work and sets PKV_STATUS_BAD_ITEM
      bool ok = p.work[0] == static_cast<int>(gridDim.x);  // only then are the offsets of this grid there
      int a = 0, b = 0;
      if (ok) {
        a = p.work[2 + blockIdx.x];
        b = p.work[3 + blockIdx.x];
        ok = 0 <= a && a <= b && b <= p.work[1];
      }
      if (!ok && threadIdx.x == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_ITEM);
      it = ok ? a : 0;
      end = ok ? b : 0;
      step = 1;
    } else if (kPrefill) {
      it = blockIdx.x;
      end = total_items;
      step = gridDim.x;
    } else {
      it = range_first(blockIdx.x, total_items);
      end = range_first(blockIdx.x + 1, total_items);
      step = 1;
    }
    if (it < end) {
      if (kPrefill) load(p, t);
      else {
        w.seek(t.prefix, p.num_seqs, p.num_kv_heads, it);
        fill(p, t, true);
      }
    }
  }
  // prefill: the item at position it (of the list, or of the batch)
  __device__ void load(const TcParams &p, const SeqTab &t) {
    const int idx = p.work ? p.work[3 + gridDim.x + it] : it;
    if (idx < 0 || idx >= total) {  // a list entry outside the batch: nothing to do
      if ((threadIdx.x & 31) == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_ITEM);
      x = Item{};
      x.skip = true;
      x.run_begin = x.run_end = true;
      return;
    }
    w.seek(t.prefix, p.num_seqs, p.num_kv_heads, idx);
    fill(p, t, true);
  }
  __device__ bool valid() const { return it < end; }
  __device__ void advance(const TcParams &p, const SeqTab &t) {
    it += step;
    if (it >= end) return;
    if (kPrefill) {
      load(p, t);
    } else {
      const int s0 = w.seq, h0 = w.head;
      w.next(t.prefix, p.num_seqs, p.num_kv_heads);
      fill(p, t, w.seq != s0 || w.head != h0);
    }
  }
  __device__ void fill(const TcParams &p, const SeqTab &t, bool begins) {
    const int L = t.lens[w.seq];
    x.seq = w.seq;
    x.head = w.head;
    x.run_begin = begins;
    if (kPrefill) {
      const int c = t.qc[w.seq];
      const int tile_tok = p.tile_tok;
      // split over keys: every query tile of the sequence has ps partitions of
      // part_tokens keys (the last tile's count); items past a tile's keys are empty
      const int ps = split_parts(p, L);
      x.qt = w.nparts / ps - 1 - w.part / ps;  // longest first
      const int span = kPairs ? 2 * tile_tok : tile_tok;  // query tokens per item
      const int k_hi = min(L, max(0, L - c + min(c, span * (x.qt + 1))));  // keys the tile's last row sees
      x.skip = false;
      if (ps == 1) {
        x.part = 0;
        x.nparts = 1;
        x.k_lo = 0;
        x.k_hi = k_hi;
      } else {
        x.part = w.part % ps;
        x.nparts = max(1, ceil_div(k_hi, p.part_tokens));  // this tile's partitions
        x.skip = x.part >= x.nparts;
        x.k_lo = x.skip ? 0 : x.part * p.part_tokens;
        x.k_hi = x.skip ? 0 : min(k_hi, x.k_lo + p.part_tokens);
      }
      x.has_b = kPairs && (2 * x.qt + 1) * tile_tok < c;
      x.run_end = true;
    } else {
      x.skip = false;
      x.qt = 0;
      x.has_b = false;
      x.part = w.part;
      x.nparts = w.nparts;
      x.k_lo = w.part * p.part_tokens;
      x.k_hi = max(x.k_lo, min(L, x.k_lo + p.part_tokens));
      ItemWalker nx = w;
      nx.next(t.prefix, p.num_seqs, p.num_kv_heads);
      x.run_end = it + 1 >= end || nx.seq != w.seq || nx.head != w.head;
    }
  }
};

// 32 bytes from eight 32-bit registers to global memory in one request
// (256-bit store, sm_100+); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *w) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
               "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// The largest (smallest, for a negative scale) of 64 raw scores: eight short
// chains of 3-input maxima.
__device__ __forceinline__ float extreme64(const uint32_t (&v)[64], bool neg) {
  float e[8];
  if (!neg) {
#pragma unroll
    for (int q = 0; q < 8; ++q) e[q] = fmax3(__uint_as_float(v[q]), __uint_as_float(v[q + 8]), __uint_as_float(v[q + 16]));
#pragma unroll
    for (int q = 0; q < 8; ++q) e[q] = fmax3(e[q], __uint_as_float(v[q + 24]), __uint_as_float(v[q + 32]));
#pragma unroll
    for (int q = 0; q < 8; ++q) e[q] = fmax3(e[q], __uint_as_float(v[q + 40]), __uint_as_float(v[q + 48]));
#pragma unroll
    for (int q = 0; q < 8; ++q) e[q] = fmaxf(e[q], __uint_as_float(v[q + 56]));
    return fmax3(fmax3(e[0], e[1], e[2]), fmax3(e[3], e[4], e[5]), fmaxf(e[6], e[7]));
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) e[q] = fmin3(__uint_as_float(v[q]), __uint_as_float(v[q + 8]), __uint_as_float(v[q + 16]));
#pragma unroll
  for (int q = 0; q < 8; ++q) e[q] = fmin3(e[q], __uint_as_float(v[q + 24]), __uint_as_float(v[q + 32]));
#pragma unroll
  for (int q = 0; q < 8; ++q) e[q] = fmin3(e[q], __uint_as_float(v[q + 40]), __uint_as_float(v[q + 48]));
#pragma unroll
  for (int q = 0; q < 8; ++q) e[q] = fminf(e[q], __uint_as_float(v[q + 56]));
  return fmin3(fmin3(e[0], e[1], e[2]), fmin3(e[3], e[4], e[5]), fminf(e[6], e[7]));
}

// Weights of 64 raw scores, p = 2^(s * scale * log2e - m), two at a time with a
// packed fp32 FMA, packed to bf16 pairs; returns the sum of the weights before
// their rounding to bf16 (the rounding errors, at most 2^-9 of each weight and
// of either sign, leave the sum's relative error far below the output's bf16
// step).  Masked keys hold -inf (or +inf for a negative scale): their weight
// is 2^-inf = 0.
__device__ __forceinline__ float weights64(const uint32_t (&v)[64], uint64_t ks2, uint64_t nm2, uint32_t (&pk)[32]) {
  uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};  // four packed partial sums (0 bits = +0.0)
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x0, x1;
    f32x2_split(ffma2(f32x2_bits(v[2 * c], v[2 * c + 1]), ks2, nm2), x0, x1);
    const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
    pk[c] = pack_bf16x2(e0, e1);
    ls[c & 3] = fadd2(ls[c & 3], f32x2_bits(__float_as_uint(e0), __float_as_uint(e1)));
  }
  float a0, a1, b0, b1, c0, c1, d0, d1;
  f32x2_split(ls[0], a0, a1);
  f32x2_split(ls[1], b0, b1);
  f32x2_split(ls[2], c0, c1);
  f32x2_split(ls[3], d0, d1);
  return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
}

// Bounded wait whose outcome every lane of the warp agrees on; try_wait
// parks the warp until the phase completes (or a short hardware window ends).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

template <int BS, bool kPrefill, int D, bool kPairs>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const TcParams p) {
  using Lay = Layout<kPrefill, D>;
  constexpr bool kP2 = kPrefill && kPairs;  // prefill over pairs of query tiles
  constexpr int kStages = Lay::kStages, kQBufs = Lay::kQBufs, kTileKeys = Lay::kTK, kKVBytes = Lay::kKVBytes;
  constexpr int kHalves = Lay::kHalves, kQBytes = Lay::kQBytes;
  // one TMA box per block of the tile (a block longer than the tile: the tile's piece of it)
  constexpr int kBoxRows = BS < kTileKeys ? BS : kTileKeys;
  constexpr int kBoxes = kTileKeys / kBoxRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kSmemBars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *prefix = reinterpret_cast<int *>(smem + Lay::kSmemSeq);  // [B + 1]
  int *lens = prefix + p.num_seqs + 1;                          // [B]
  int *qs = lens + p.num_seqs;                                  // prefill: [B]
  int *qc = qs + p.num_seqs;                                    // prefill: [B]
  const SeqTab tab{prefix, lens, qs, qc};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.num_seqs, hkv = p.num_kv_heads;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  // Wait for the kernel before this one, then let the grid queued behind this
  // one become resident (a merge grid still waits for our results).  In this
  // order a dependent grid that reads nothing of ours, such as the decode rows
  // of a mixed step, can skip its own wait: our inputs, which are its inputs
  // too, are complete once every CTA of this grid has passed this point.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {  // items per sequence -> exclusive prefix
    const int per = (B + 31) / 32;
    const int lo = min(B, lane * per), hi = min(B, lo + per);
    const int cap_tbl = p.max_blocks * BS, cap_grid = p.max_parts * p.part_tokens;
    // prefill without the key split has no partition grid
    const int cap = (kPrefill && p.part_tokens == 0) || cap_tbl < cap_grid ? cap_tbl : cap_grid;
    const int tile_tok = p.tile_tok;
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
      int L = p.seq_lens[i];
      if (L < 0 || L > cap) {
        if (blockIdx.x == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_LEN);
        L = L < 0 ? 0 : cap;
      }
      lens[i] = L;
      int n;
      if (kPrefill) {
        const int a = p.q_start[i], b = p.q_start[i + 1];
        int c = b - a;
        if (a < 0 || c < 0 || b > p.total_q) {
          if (blockIdx.x == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_QSTART);
          c = 0;
        }
        qs[i] = a;
        qc[i] = c;
        n = ceil_div(c, (kP2 ? 2 : 1) * tile_tok) * split_parts(p, L) * hkv;  // query tiles, pairs, or partitions
      } else {
        n = (L > 0 ? ceil_div(L, p.part_tokens) : 1) * hkv;
      }
      prefix[i + 1] = n;
      sum += n;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      run += prefix[i + 1];
      prefix[i + 1] = run;
    }
    if (lane == 0) prefix[0] = 0;
  }
  if (threadIdx.x == 32 * kKWarp) {
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(bar(B_Q_FULL0 + i), 1);
      mbar_init(bar(B_Q_FREE0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {  // decode chunk: index 0 only; prefill: one per query tile of the pair
      mbar_init(bar(B_O_FULL + i), 1);
      mbar_init(bar(B_O_FREE + i), kRows);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_STATS0 + i), kRows);
      mbar_init(bar(B_STATS_FREE0 + i), kRows);
      mbar_init(bar(B_S_FULL0 + i), 1);
      mbar_init(bar(B_S_FREE0 + i), kRows);
      mbar_init(bar(B_P_FULL0 + i), kRows);
      mbar_init(bar(B_P_LO0 + i), kRows);
      mbar_init(bar(B_PV_DONE0 + i), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_K_FULL0 + s), 1);
      mbar_init(bar(B_K_EMPTY0 + s), 1);
      mbar_init(bar(B_V_FULL0 + s), 1);
      mbar_init(bar(B_V_EMPTY0 + s), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tc::alloc(smem_u32(tmem_slot), kTmemCols);
    tc::relinquish();
  }
  if (kPrefill ? p.tile_tok * p.group < kRows : p.q_len * p.group < kRows) {
    // the loads fill the tile's first q_len * G (prefill: tile_tok * G) rows
    // only: the rest stay zero for the whole kernel, so their scores are
    // finite (and masked)
    for (int i = threadIdx.x; i < kQBufs * kQBytes / 16; i += kThreads)
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(smem_u32(smem) + i * 16), "r"(0u) : "memory");
    fence_proxy_async_shared();
  }
  if (threadIdx.x == 32 * kKWarp + 1) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const int I = prefix[B];
  const uint32_t sQ = smem_u32(smem), sK = smem_u32(smem + Lay::kSmemK), sV = smem_u32(smem + Lay::kSmemV);
  const uint32_t tS0 = tmem + Lay::kTmemS;  // S buffers after the two accumulators
  // P buffers: over pairs of query tiles the two sets share one S buffer (a
  // score product goes out once the previous one has been read) and write
  // their weights to columns of their own after it; otherwise over the S
  // buffers (prefill) or after them (decode chunk)
  const uint32_t tP0 = tmem + (kP2 ? Lay::kTmemS + kTileKeys : Lay::kTmemP);
  constexpr int kPStr = kP2 ? kTileKeys / 2 : Lay::kPStride;  // columns between the two sets' P
  static_assert(!kP2 || 2 * D + kTileKeys + 2 * (kTileKeys / 2) <= kTmemCols, "tensor memory");
  const bool has_work = kPrefill ? static_cast<int>(blockIdx.x) < I
                                 : range_first(blockIdx.x, I) < range_first(blockIdx.x + 1, I);

  if (has_work) {
    if (warp == kKWarp || warp == kVWarp) {
      // ------------------------------------------- producers: K (+ Q), V
      const bool is_v = warp == kVWarp;
      const CUtensorMap *tm = is_v ? &tmv : &tmk;
      const uint32_t ring = is_v ? sV : sK;
      const int full0 = is_v ? B_V_FULL0 : B_K_FULL0, empty0 = is_v ? B_V_EMPTY0 : B_K_EMPTY0;
      // decode: every key is read once; prefill: the CTAs beside this one read them too
      const uint64_t pol = kPrefill ? l2_policy_evict_normal() : l2_policy_evict_first();
      Sched<kPrefill, kP2> sc;
      sc.begin(p, tab, I);
      int g = 0, tpieces = 0;
      int tw_seq = -1, tw_base = 0, tw_val = -1;
      for (; sc.valid() && !*abort_flag; sc.advance(p, tab)) {
        const Item &x = sc.x;
        if (kP2 && !is_v && x.k_hi > x.k_lo) {  // the pair's query tiles, both into buffers 0 and 1
          const int qi = tpieces++;
          if (qi > 0 && !wait_warp(bar(B_Q_FREE0), (qi - 1) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if (lane == 0) {
            const int gsz = p.group, tile_tok = p.tile_tok;
            const int ntq = x.has_b ? 2 : 1;
            mbar_arrive_expect_tx(bar(B_Q_FULL0), ntq * tile_tok * gsz * D * 2);  // the boxes' bytes
            for (int q = 0; q < ntq; ++q)
              for (int hf = 0; hf < kHalves; ++hf)
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sQ + q * kQBytes + hf * Lay::kQHalf),
                    "l"(reinterpret_cast<uint64_t>(&tmq)), "r"(hf * 64), "r"(x.head * gsz),
                    "r"(qs[x.seq] + tile_tok * (2 * x.qt + q)), "r"(bar(B_Q_FULL0))
                    : "memory");
          }
        }
        if (!kP2 && !is_v && x.run_begin && x.k_hi > x.k_lo) {  // a run with keys: load its queries
          const int qi = tpieces++, qb = qi % kQBufs, use = qi / kQBufs;
          if (use > 0 && !wait_warp(bar(B_Q_FREE0 + qb), (use - 1) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if (lane == 0) {
            const int gsz = p.group;
            const int qz = kPrefill ? qs[x.seq] + p.tile_tok * x.qt : x.seq * p.q_len;
            // the box holds tile_tok * G (decode chunk: q_len * G) rows
            mbar_arrive_expect_tx(bar(B_Q_FULL0 + qb), (kPrefill ? p.tile_tok : p.q_len) * gsz * D * 2);
            for (int hf = 0; hf < kHalves; ++hf)
              asm volatile(
                  "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                  " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sQ + qb * kQBytes + hf * Lay::kQHalf),
                  "l"(reinterpret_cast<uint64_t>(&tmq)), "r"(hf * 64), "r"(x.head * gsz), "r"(qz),
                  "r"(bar(B_Q_FULL0 + qb))
                  : "memory");
          }
        }
        const int ntile = ceil_div(x.k_hi - x.k_lo, kTileKeys);
        const int nblk_seq = ceil_div(lens[x.seq], BS);
        for (int t = 0; t < ntile; ++t, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !wait_warp(bar(empty0 + s), ((g / kStages) - 1) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const int k0 = x.k_lo + t * kTileKeys;
          const int blk_first = k0 / BS;
          if (x.seq != tw_seq || blk_first < tw_base || blk_first + kBoxes > tw_base + 32) {
            tw_seq = x.seq;
            tw_base = blk_first;
            const int e = blk_first + lane;
            tw_val = e < p.max_blocks ? p.block_tables[static_cast<size_t>(x.seq) * p.max_blocks + e] : -1;
          }
          int bids[kBoxes];
#pragma unroll
          for (int j = 0; j < kBoxes; ++j) bids[j] = __shfl_sync(0xffffffffu, tw_val, blk_first + j - tw_base);
          if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), kKVBytes);
          // one lane per (box, half): the box copies go out in parallel
          if (lane < kBoxes * kHalves) {
            const int j = lane / kHalves, hf = lane % kHalves;
            const int b = bids[j];
            int row;
            if (blk_first + j < nblk_seq && b >= 0 && b < p.num_blocks) {
              row = (b * hkv + x.head) * BS + k0 % BS;
            } else {
              if (blk_first + j < nblk_seq && p.status && !is_v && hf == 0) atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
              row = p.oob_row;  // past the sequence, or a bad id: zeros
            }
            tma_load_2d(ring + s * kKVBytes + hf * Lay::kKVHalf + j * kBoxRows * 128, tm, hf * 64, row,
                        bar(full0 + s), pol);
          }
        }
      }
      // never leave a copy in flight into this CTA's shared memory
      if (lane == 0) {
        for (int y = g > kStages ? g - kStages : 0; y < g; ++y)
          mbar_wait_sleep(bar(full0 + (y % kStages)), (y / kStages) & 1);
        if (!is_v && kP2 && tpieces > 0) mbar_wait_sleep(bar(B_Q_FULL0), (tpieces - 1) & 1);
        if (!is_v && !kP2)
          for (int qi = tpieces > kQBufs ? tpieces - kQBufs : 0; qi < tpieces; ++qi)
            mbar_wait_sleep(bar(B_Q_FULL0 + qi % kQBufs), (qi / kQBufs) & 1);
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------- S = Q K^T issuer
      // A score product waits for its key stage and for its S buffer: in
      // prefill over single query tiles the buffer holds the set's previous P
      // until that tile's P V product completes; over pairs and in the decode
      // chunk it is free once the softmax has read it, so the score products
      // run ahead.  Each releases its key stage
      // when it completes.  The waits are plain try_wait loops (woken on
      // completion), so each issue follows its event closely.
      if (lane == 0) {
        constexpr uint32_t kIdS = tc::idesc_bf16(kRows, kTileKeys, false, false);
        Sched<kPrefill, kP2> sc;
        sc.begin(p, tab, I);
        int g = 0, tpieces = 0;
        bool ok = true;
        int ns = 0;  // pairs: score products into the shared S buffer so far
        for (; sc.valid() && ok; sc.advance(p, tab)) {
          const Item &x = sc.x;
          const int ntile = ceil_div(x.k_hi - x.k_lo, kTileKeys);
          if (ntile == 0) continue;
          if constexpr (kP2) {
            // both query tiles of the pair against each key tile, A then B,
            // into the one S buffer: each product goes out once the set that
            // owned the previous one has read its scores (the sets' weights
            // have their own columns), so a set's next score product runs
            // while it computes its softmax
            const int qi = tpieces++;
            if (!mbar_wait(bar(B_Q_FULL0), qi & 1)) { ok = false; break; }
            for (int t = 0; t < ntile && ok; ++t, ++g) {
              const int s = g % kStages;
              if (!mbar_wait(bar(B_K_FULL0 + s), (g / kStages) & 1)) { ok = false; break; }
              const uint32_t kb = sK + s * kKVBytes;
              for (int q = 0; q < (x.has_b ? 2 : 1); ++q) {
                if (ns > 0 && !mbar_wait(bar(B_S_FREE0), (ns - 1) & 1)) { ok = false; break; }
                tc::fence_after();
                const uint32_t sq = sQ + q * kQBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                  tc::mma(tS0, tc::desc_sw128(sq + (ks >> 2) * Lay::kQHalf + (ks & 3) * 32, 16, 1024),
                          tc::desc_sw128(kb + (ks >> 2) * Lay::kKVHalf + (ks & 3) * 32, 16, 1024), kIdS, ks > 0);
                tc::commit(bar(B_S_FULL0 + q));
                ++ns;
              }
              if (!ok) break;
              tc::commit(bar(B_K_EMPTY0 + s));  // the keys are read by these products only
              if (t == ntile - 1) tc::commit(bar(B_Q_FREE0));
            }
            continue;
          }
          int qb = (tpieces > 0 ? tpieces - 1 : 0) % kQBufs;
          if (x.run_begin) {
            const int qi = tpieces++;
            qb = qi % kQBufs;
            if (!mbar_wait(bar(B_Q_FULL0 + qb), (qi / kQBufs) & 1)) { ok = false; break; }
          }
          const uint32_t sq = sQ + qb * kQBytes;
          for (int t = 0; t < ntile; ++t, ++g) {
            const int s = g % kStages, sb = g & 1;
            if (!mbar_wait(bar(B_K_FULL0 + s), (g / kStages) & 1)) { ok = false; break; }
            // prefill: the buffer holds the set's previous P until its P V product
            // completes; decode chunk: the softmax has read the buffer's last scores
            if (g >= 2 && !mbar_wait(bar((Lay::kPOverS ? B_PV_DONE0 : B_S_FREE0) + sb), ((g >> 1) - 1) & 1)) {
              ok = false;
              break;
            }
            tc::fence_after();
            const uint32_t kb = sK + s * kKVBytes;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc::mma(tS0 + sb * kTileKeys, tc::desc_sw128(sq + (ks >> 2) * Lay::kQHalf + (ks & 3) * 32, 16, 1024),
                      tc::desc_sw128(kb + (ks >> 2) * Lay::kKVHalf + (ks & 3) * 32, 16, 1024), kIdS, ks > 0);
            tc::commit(bar(B_S_FULL0 + sb));
            tc::commit(bar(B_K_EMPTY0 + s));  // the keys are read by this product only
            if (x.run_end && t == ntile - 1) tc::commit(bar(B_Q_FREE0 + qb));  // read by MMAs issued so far only
          }
        }
        if (!ok) {
          if (p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
          *abort_flag = 1;
        }
      }
    } else if (warp == kPvWarp) {
      // ------------------------------------------------ O += P V issuer
      // Each product goes out, in tile order, as soon as its P is written and
      // its values have landed; its value stage is released when it completes.
      if (lane == 0) {
        constexpr uint32_t kIdO = tc::idesc_bf16(kRows, D, false, true);
        Sched<kPrefill, kP2> sc;
        sc.begin(p, tab, I);
        int g = 0, tpieces = 0, run_g0 = 0;
        int na = 0, nb = 0, ia = 0, ib = 0;  // prefill: P V products and items of each query tile of the pair
        bool ok = true;
        for (; sc.valid() && ok; sc.advance(p, tab)) {
          const Item &x = sc.x;
          const int ntile = ceil_div(x.k_hi - x.k_lo, kTileKeys);
          if (ntile == 0) continue;
          if constexpr (kP2) {
            // per key tile: tile A's product, then tile B's (so that B's
            // product follows A's zeroing of the value rows past the end)
            ++ia;
            if (x.has_b) ++ib;
            for (int t = 0; t < ntile && ok; ++t, ++g) {
              const int vs = g % kStages;
              if (!mbar_wait(bar(B_V_FULL0 + vs), (g / kStages) & 1)) { ok = false; break; }
              const uint32_t vb = sV + vs * kKVBytes;
              constexpr int kSteps = kTileKeys / 16;  // 16 keys = 8 packed columns of P
              for (int q = 0; q < (x.has_b ? 2 : 1); ++q) {
                int &n = q ? nb : na;
                const int items = q ? ib : ia;
                if (!mbar_wait(bar(B_P_FULL0 + q), n & 1)) { ok = false; break; }
                // the item's first product overwrites the accumulator: the previous epilogue must have read it
                if (t == 0 && items > 1 && !mbar_wait(bar(B_O_FREE + q), (items - 2) & 1)) { ok = false; break; }
                tc::fence_after();
                const uint32_t pa = tP0 + q * kPStr, acc = tmem + q * D;
                // keys kTK/2.. first (P_FULL), keys 0.. once weighted (P_LO)
#pragma unroll
                for (int ks = kSteps / 2; ks < kSteps; ++ks)
                  tc::mma_ta(acc, pa + ks * 8, tc::desc_sw128(vb + ks * 2048, Lay::kKVHalf, 1024), kIdO,
                             !(t == 0 && ks == kSteps / 2));
                if (!mbar_wait(bar(B_P_LO0 + q), n & 1)) { ok = false; break; }
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < kSteps / 2; ++ks)
                  tc::mma_ta(acc, pa + ks * 8, tc::desc_sw128(vb + ks * 2048, Lay::kKVHalf, 1024), kIdO, true);
                tc::commit(bar(B_PV_DONE0 + q));
                if (t == ntile - 1) tc::commit(bar(B_O_FULL + q));
                ++n;
              }
              if (!ok) break;
              tc::commit(bar(B_V_EMPTY0 + vs));
            }
            continue;
          }
          if (x.run_begin) {
            ++tpieces;
            run_g0 = g;
          }
          for (int t = 0; t < ntile; ++t, ++g) {
            const int pb = g & 1;  // the set (even / odd tiles): its P buffer and accumulator
            const bool first = g - run_g0 < 2, last = x.run_end && t == ntile - 1;
            if (!mbar_wait(bar(B_P_FULL0 + pb), (g >> 1) & 1)) { ok = false; break; }
            if (!mbar_wait(bar(B_V_FULL0 + g % kStages), (g / kStages) & 1)) { ok = false; break; }
            // the first products of run j overwrite the accumulators: run j-1's epilogue must have read them
            if (first && tpieces > 1 && !mbar_wait(bar(B_O_FREE), (tpieces - 2) & 1)) { ok = false; break; }
            tc::fence_after();
            const uint32_t pa = tP0 + pb * Lay::kPStride;
            const uint32_t vb = sV + (g % kStages) * kKVBytes;
            constexpr int kSteps = kTileKeys / 16;  // 16 keys = 8 packed columns of P
            if constexpr (Lay::kPOverS) {
              // the weights of keys kTK/2.. come first (P_FULL); those of keys
              // 0.. follow while this half's product runs (P_LO)
#pragma unroll
              for (int ks = kSteps / 2; ks < kSteps; ++ks)
                tc::mma_ta(tmem + pb * D, pa + ks * 8, tc::desc_sw128(vb + ks * 2048, Lay::kKVHalf, 1024), kIdO,
                           !(first && ks == kSteps / 2));
              if (!mbar_wait(bar(B_P_LO0 + pb), (g >> 1) & 1)) { ok = false; break; }
              tc::fence_after();
#pragma unroll
              for (int ks = 0; ks < kSteps / 2; ++ks)
                tc::mma_ta(tmem + pb * D, pa + ks * 8, tc::desc_sw128(vb + ks * 2048, Lay::kKVHalf, 1024), kIdO,
                           true);
            } else {
#pragma unroll
              for (int ks = 0; ks < kSteps; ++ks)
                tc::mma_ta(tmem + pb * D, pa + ks * 8, tc::desc_sw128(vb + ks * 2048, Lay::kKVHalf, 1024), kIdO,
                           !(first && ks == 0));
            }
            tc::commit(bar(B_PV_DONE0 + pb));
            tc::commit(bar(B_V_EMPTY0 + (g % kStages)));
            if (last) tc::commit(bar(B_O_FULL));
          }
        }
        if (!ok) {
          if (p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
          *abort_flag = 1;
        }
      }
    } else {
      // ------------------------------------------------------ softmax warps
      // decode chunk: set 0 takes the even tiles of a run, set 1 the odd ones;
      // prefill: set q takes every tile of query tile q of the pair
      const int set = warp >> 2;
      const int r = threadIdx.x & (kRows - 1);    // query row = TMEM lane
      const int tok = r / p.group, gh = r - tok * p.group;
      const int tile_tok = p.tile_tok;
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tO = tmem + set * D;         // this set's accumulator
      float2 *stats = reinterpret_cast<float2 *>(smem + Lay::kSmemStats);
      Sched<kPrefill, kP2> sc;
      sc.begin(p, tab, I);
      int g = 0, tpieces = 0;
      int n_set = 0, items_set = 0;  // prefill: this set's tiles and items so far
      float m = -INFINITY, l = 0.f;
      int run_first_part = 0;
      bool run_has_tiles = false, set_has_tiles = false;
      bool ok = true;
      for (; sc.valid() && ok; sc.advance(p, tab)) {
        const Item &x = sc.x;
        const int L = lens[x.seq];
        const int ntile = ceil_div(x.k_hi - x.k_lo, kTileKeys);
        if (kP2 && set == 1 && !x.has_b) continue;  // the pair has no second query tile
        if (x.skip) continue;                        // an empty partition: nothing to compute or store
        if (x.run_begin) {
          m = -INFINITY;
          l = 0.f;
          run_first_part = x.part;
          run_has_tiles = ntile > 0;
          set_has_tiles = false;
          if (run_has_tiles) ++tpieces;
        }
        // this row's token within the chunk, and the keys it sees: t < limit
        int row_tok, limit;
        bool row_valid;
        if (kPrefill) {
          const int c = qc[x.seq];
          row_tok = tile_tok * (kP2 ? 2 * x.qt + set : x.qt) + tok;
          row_valid = tok < tile_tok && row_tok < c;  // a spare row of the tile is never valid
          limit = row_valid ? L - c + 1 + row_tok : 0;
        } else {
          row_tok = tok;
          row_valid = tok < p.q_len;
          limit = row_valid ? L - p.q_len + 1 + tok : 0;
        }
        for (int t = 0; t < ntile; ++t, ++g) {
          if (!kP2 && (g & 1) != set) continue;  // the other set's tile
          const bool first_tile_of_set = !set_has_tiles;
          set_has_tiles = true;
          const int sb = set;
          const uint32_t sphase = kP2 ? (n_set++ & 1) : ((g >> 1) & 1);
          if (!wait_warp(bar(B_S_FULL0 + sb), sphase)) { ok = false; break; }
          const int k0 = x.k_lo + t * kTileKeys;
          const int vis = min(limit, x.k_hi) - k0;  // keys of this tile the row sees
          const uint32_t tSb = tS0 + (kP2 ? 0 : sb * kTileKeys) + lane_off;  // this row's scores
          const uint32_t tPb = tP0 + sb * kPStr + lane_off;                 // this row's weights
          // no row of this warp sees a key of the tile (rows past a short
          // chunk's end): its weights are zero and nothing else changes
          const bool skip = __all_sync(0xffffffffu, vis <= 0);
          const bool partial = !__all_sync(0xffffffffu, vis >= kTileKeys);
          // a negative scale turns the largest score into the smallest: take minima then
          const bool neg = p.scale_log2 < 0.f;
          const uint32_t masked = __float_as_uint(neg ? INFINITY : -INFINITY);
          bool scale_o = false;
          float alpha = 1.f;
          // move the reference max only when a score passes it by more than
          // kSlack (rare after a set's first tile); exact, since O and l share
          // it.  rm is the extreme raw score (times the scale: the largest scaled
          // score).  Returns the reference to subtract.
          auto new_reference = [&](float rm) {
            const float bm = rm * p.scale_log2;
            const bool move = bm > m + kSlack;
            scale_o = move && !first_tile_of_set && m != -INFINITY;
            alpha = scale_o ? fast_exp2(m - bm) : 1.f;
            if (move) {
              l = m == -INFINITY ? 0.f : l * exp2f(m - bm);
              m = bm;
            }
            return m == -INFINITY ? 0.f : m;
          };
          auto mask = [&](uint32_t(&sv)[64], int c0) {
            if (partial) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c0 + c >= vis) sv[c] = masked;
            }
          };
          auto rescale_o = [&]() {
            if (__any_sync(0xffffffffu, scale_o)) {  // warp-uniform: tcgen05.ld/st are warp-wide
#pragma unroll
              for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t ov[32];
                tc::ld32(tO + lane_off + ch * 32, ov);
                tc::wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                tc::st32(tO + lane_off + ch * 32, ov);
              }
            }
          };
          // value rows past the sequence end were never written: zero them
          // before any P V product of this tile reads the stage
          auto zero_tail_values = [&]() {
            const int exist = L - k0;
            // prefill: query tile A's set zeroes; B's P V product is issued after A's
            if (exist >= kTileKeys || (kP2 && set == 1)) return true;
            const int s = g % kStages;
            if (!wait_warp(bar(B_V_FULL0 + s), (g / kStages) & 1)) return false;
            const uint32_t vb = sV + s * kKVBytes;
            const int first = exist < 0 ? 0 : exist;
            for (int e = r; e < (kTileKeys - first) * kHalves * 8; e += kRows) {  // 16-byte chunks
              const int row = first + e / (kHalves * 8), rem = e % (kHalves * 8), hf = rem / 8, c = rem % 8;
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vb + hf * Lay::kKVHalf + row * 128 + c * 16),
                           "r"(0u)
                           : "memory");
            }
            return true;
          };
          // make this thread's P (tensor memory) and zeroed values (shared
          // memory) visible to the P V issuer, then count in at barrier bi
          auto publish = [&](int bi) {
            tc::wait_st();
            fence_proxy_async_shared();
            tc::fence_before();
            mbar_arrive(bar(bi));
          };
          tc::fence_after();
          if constexpr (Lay::kPOverS) {
            static_assert(kTileKeys == 128, "two 64-key halves");
            // pairs: this set's previous P V product must be complete before
            // its weights' columns and its accumulator are written (the score
            // product of this tile did not wait for it)
            auto previous_pv_done = [&]() {
              if (kP2 && n_set > 1 && !wait_warp(bar(B_PV_DONE0 + sb), (n_set - 2) & 1)) return false;
              tc::fence_after();
              return true;
            };
            if (skip) {
              if constexpr (kP2) {
                tc::fence_before();
                mbar_arrive(bar(B_S_FREE0));  // nothing to read: the next score product may go out
              }
              if (!previous_pv_done()) { ok = false; break; }
              uint32_t z[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) z[c] = 0u;
              tc::st32(tPb, z);
              tc::st32(tPb + 32, z);
              if (!zero_tail_values()) { ok = false; break; }
              publish(B_P_FULL0 + sb);
              mbar_arrive(bar(B_P_LO0 + sb));
            } else {
              if constexpr (kP2) {
                // the row's 128 scores in one load round; once they are in
                // registers the other set's score product may overwrite them
                uint32_t sl[64], sh[64];
                tc::ld32(tSb, *reinterpret_cast<uint32_t(*)[32]>(&sl[0]));
                tc::ld32(tSb + 32, *reinterpret_cast<uint32_t(*)[32]>(&sl[32]));
                tc::ld32(tSb + 64, *reinterpret_cast<uint32_t(*)[32]>(&sh[0]));
                tc::ld32(tSb + 96, *reinterpret_cast<uint32_t(*)[32]>(&sh[32]));
                tc::wait_ld();
                tc::fence_before();
                mbar_arrive(bar(B_S_FREE0));
                mask(sl, 0);
                mask(sh, 64);
                const float el = extreme64(sl, neg), eh = extreme64(sh, neg);
                const float msub = new_reference(neg ? fminf(el, eh) : fmaxf(el, eh));
                const uint64_t ks2 = f32x2_bits(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
                const uint64_t nm2 = f32x2_bits(__float_as_uint(-msub), __float_as_uint(-msub));
                // keys 64..127 first: their P V product starts while keys
                // 0..63 are weighted
                uint32_t pk[32];
                float lsum = weights64(sh, ks2, nm2, pk);
                if (!previous_pv_done()) { ok = false; break; }
                tc::st32(tPb + 32, pk);
                // none of this tile's P V products is issued before P_FULL:
                // the accumulator holds its final value and may be rescaled here
                rescale_o();
                if (!zero_tail_values()) { ok = false; break; }
                publish(B_P_FULL0 + sb);
                lsum += weights64(sl, ks2, nm2, pk);
                tc::st32(tPb, pk);
                tc::wait_st();
                tc::fence_before();
                mbar_arrive(bar(B_P_LO0 + sb));
                l += lsum;
              } else {
                // two load rounds (fewer registers, for the single-tile
                // schedule): the maximum over both halves, then the weights of
                // keys 64..127 from the scores still in registers and of keys
                // 0..63 after reloading them
                uint32_t sv[64];
                // pass 1: the row's extreme raw score, 64 columns at a time
                float rm = neg ? INFINITY : -INFINITY;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  tc::ld32(tSb + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                  tc::ld32(tSb + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                  tc::wait_ld();
                  mask(sv, hh * 64);
                  const float e = extreme64(sv, neg);
                  rm = neg ? fminf(rm, e) : fmaxf(rm, e);
                }
                const float msub = new_reference(rm);
                const uint64_t ks2 = f32x2_bits(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
                const uint64_t nm2 = f32x2_bits(__float_as_uint(-msub), __float_as_uint(-msub));
                // pass 2, keys 64..127 first (their scores are still in
                // registers): weights over score columns 96..127, already read;
                // their P V product starts while keys 0..63 are weighted
                uint32_t pk[32];
                float lsum = weights64(sv, ks2, nm2, pk);
                tc::st32(tPb + 32, pk);
                rescale_o();
                if (!zero_tail_values()) { ok = false; break; }
                publish(B_P_FULL0 + sb);
                // keys 0..63: weights over score columns 64..95
                tc::ld32(tSb, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                tc::ld32(tSb + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                tc::wait_ld();
                mask(sv, 0);
                lsum += weights64(sv, ks2, nm2, pk);
                tc::st32(tPb, pk);
                tc::wait_st();
                tc::fence_before();
                mbar_arrive(bar(B_P_LO0 + sb));
                l += lsum;
              }
            }
          } else {
            uint32_t pk[32];
            if (skip) {
              mbar_arrive(bar(B_S_FREE0 + sb));
#pragma unroll
              for (int c = 0; c < 32; ++c) pk[c] = 0u;
            } else {
              uint32_t sv[64];
              tc::ld32(tSb, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
              tc::ld32(tSb + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
              tc::wait_ld();
              tc::fence_before();
              mbar_arrive(bar(B_S_FREE0 + sb));  // the next score product may overwrite the buffer
              mask(sv, 0);
              const float msub = new_reference(extreme64(sv, neg));
              const uint64_t ks2 = f32x2_bits(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
              const uint64_t nm2 = f32x2_bits(__float_as_uint(-msub), __float_as_uint(-msub));
              l += weights64(sv, ks2, nm2, pk);
            }
            // this set's previous tile (g - 2) must be in the accumulator before a
            // rescale, and its P buffer free before the new P is written; the
            // weights above were computed while that product ran
            if (g >= 2 && !wait_warp(bar(B_PV_DONE0 + sb), ((g - 2) >> 1) & 1)) { ok = false; break; }
            tc::fence_after();
            rescale_o();
            tc::st32(tPb, pk);
            if (!zero_tail_values()) { ok = false; break; }
            publish(B_P_FULL0 + sb);
          }
        }
        if (!ok) break;
        // ---- end of a run
        if (!x.run_end) continue;
        if constexpr (kP2) {
          // this set's query tile: normalise its accumulator and store its rows
          float inv = 0.f;
          if (run_has_tiles) {
            ++items_set;
            if (!wait_warp(bar(B_O_FULL + set), (items_set - 1) & 1)) { ok = false; break; }
            tc::fence_after();
            inv = l > 0.f ? 1.f / l : 0.f;
          }
          const size_t orow = static_cast<size_t>(qs[x.seq] + row_tok) * p.num_q_heads + x.head * p.group + gh;
          // split over keys: this set's query tile has its own partitions (tile
          // A may end a partition before tile B); its rows take bf16 output from
          // their only partition, a partial from each of theirs, and nothing
          // from a partition past their keys
          int np_q = 1;
          if (p.part_tokens > 0) {
            const int c = qc[x.seq];
            const int kq = min(L, max(0, L - c + min(c, tile_tok * (2 * x.qt + set + 1))));
            np_q = max(1, ceil_div(kq, p.part_tokens));
          }
          const bool to_out = np_q == 1 && x.part == 0, to_ws = np_q > 1 && x.part < np_q;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = 0u;
            if (run_has_tiles) {
              tc::ld32(tO + lane_off + ch * 32, ov);
              tc::wait_ld();
            }
            if (!row_valid) continue;
            if (to_ws) {  // the unnormalised partial, against this set's reference m
              float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (orow * p.max_parts + x.part) * D + ch * 32);
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4)
                dst[c4] = make_float4(__uint_as_float(ov[c4 * 4]), __uint_as_float(ov[c4 * 4 + 1]),
                                      __uint_as_float(ov[c4 * 4 + 2]), __uint_as_float(ov[c4 * 4 + 3]));
              continue;
            }
            if (!to_out) continue;
            // a thread writes its own row: each store instruction touches one
            // line per lane, so 32-byte stores (when the output allows) halve
            // the requests of this epilogue, which sits between a set's items
            __nv_bfloat16 *dst = p.out + orow * D + ch * 32;
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              w[c] = pack_bf16x2(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv);
            if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {
#pragma unroll
              for (int h8 = 0; h8 < 2; ++h8) st_global_v8(dst + h8 * 16, &w[8 * h8]);
            } else {
#pragma unroll
              for (int c8 = 0; c8 < 4; ++c8)
                reinterpret_cast<uint4 *>(dst)[c8] = make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
            }
          }
          if (run_has_tiles) {
            tc::fence_before();
            mbar_arrive(bar(B_O_FREE + set));
          }
          if (to_ws && row_valid) p.ws_ml[orow * p.max_parts + x.part] = make_float2(m, l);
          continue;
        }
        const int rp = tpieces & 1;
        if (set == 1) {  // the odd set hands its (max, sum) to the even set
          if (run_has_tiles) {
            // slot rp was last filled two runs ago: wait until the even set read it
            const int use = (tpieces - 1) >> 1;
            if (use > 0 && !wait_warp(bar(B_STATS_FREE0 + rp), (use - 1) & 1)) { ok = false; break; }
            stats[rp * kRows + r] = make_float2(set_has_tiles ? m : -INFINITY, set_has_tiles ? l : 0.f);
            mbar_arrive(bar(B_STATS0 + rp));
          }
          continue;
        }
        const int nparts = x.nparts;
        const size_t orow =
            kPrefill ? static_cast<size_t>(qs[x.seq] + row_tok) * p.num_q_heads + x.head * p.group + gh
                     : (static_cast<size_t>(x.seq) * p.q_len + tok) * p.num_q_heads + x.head * p.group + gh;
        float fa = 0.f, fb = 0.f, M = -INFINITY, lt = 0.f;
        if (run_has_tiles) {
          if (!wait_warp(bar(B_O_FULL), (tpieces - 1) & 1)) { ok = false; break; }
          if (!wait_warp(bar(B_STATS0 + rp), ((tpieces - 1) >> 1) & 1)) { ok = false; break; }
          tc::fence_after();
          const float2 sb2 = stats[rp * kRows + r];
          mbar_arrive(bar(B_STATS_FREE0 + rp));
          const float ma = set_has_tiles ? m : -INFINITY, la = set_has_tiles ? l : 0.f;
          M = fmaxf(ma, sb2.x);
          fa = ma == -INFINITY ? 0.f : exp2f(ma - M);
          fb = sb2.x == -INFINITY ? 0.f : exp2f(sb2.x - M);
          lt = la * fa + sb2.y * fb;
        }
        // a set with no key for this row contributes nothing (its accumulator is not read)
        const bool use_a = __any_sync(0xffffffffu, fa != 0.f), use_b = __any_sync(0xffffffffu, fb != 0.f);
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          float ov[32];
          uint32_t ta[32], tb[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) ta[c] = tb[c] = 0u;
          // both sets' columns of this chunk in flight together, one wait
          if (use_a) tc::ld32(tmem + lane_off + ch * 32, ta);
          if (use_b) tc::ld32(tmem + D + lane_off + ch * 32, tb);
          if (use_a || use_b) tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            ov[c] = (fa != 0.f ? fa * __uint_as_float(ta[c]) : 0.f) + (fb != 0.f ? fb * __uint_as_float(tb[c]) : 0.f);
          if (!row_valid) continue;  // a spare row of the tile: nothing to store
          if (nparts == 1) {
            __nv_bfloat16 *dst = p.out + orow * D + ch * 32;
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) w[c] = pack_bf16x2(ov[2 * c] * inv, ov[2 * c + 1] * inv);
            if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {  // 32-byte stores, as in the pairs' epilogue
#pragma unroll
              for (int h8 = 0; h8 < 2; ++h8) st_global_v8(dst + h8 * 16, &w[8 * h8]);
            } else {
#pragma unroll
              for (int c8 = 0; c8 < 4; ++c8)
                reinterpret_cast<uint4 *>(dst)[c8] = make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
            }
          } else {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (orow * p.max_parts + run_first_part) * D + ch * 32);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              dst[c4] = make_float4(ov[c4 * 4], ov[c4 * 4 + 1], ov[c4 * 4 + 2], ov[c4 * 4 + 3]);
          }
        }
        if (run_has_tiles) {
          tc::fence_before();
          mbar_arrive(bar(B_O_FREE));
        }
        if (nparts > 1 && row_valid) {
          p.ws_ml[orow * p.max_parts + run_first_part] = make_float2(M, lt);
          for (int q = run_first_part + 1; q <= x.part; ++q)  // merged into the run's first slot
            p.ws_ml[orow * p.max_parts + q] = make_float2(-INFINITY, 0.f);
        }
      }
      if (!ok) {
        if (p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

// Prefill split over keys: one warp per (query row, query head) merges the
// partitions of the row's query tile.  The row's sequence is found by a binary
// search of q_start (copied to shared memory); rows of no valid sequence, and
// rows whose tile has one partition (written directly), are left alone.
template <int D>
__global__ void __launch_bounds__(256) prefill_combine_kernel(const TcParams p, int block_size) {
  extern __shared__ int sq[];  // q_start [B + 1]
  grid_launch_dependents();
  grid_dependency_wait();  // the partials come from the grid launched just before
  for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) sq[i] = p.q_start[i];
  __syncthreads();
  const long long wg = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wg >= static_cast<long long>(p.total_q) * p.num_q_heads) return;
  const int row = static_cast<int>(wg / p.num_q_heads);
  int lo = 0, hi = p.num_seqs;  // the last sequence whose first row is at most `row`
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sq[mid] <= row) lo = mid; else hi = mid;
  }
  const int a = sq[lo], b = sq[lo + 1];
  if (a < 0 || b < a || b > p.total_q || row < a || row >= b) return;
  const int cap = min(p.max_blocks * block_size, p.max_parts * p.part_tokens);  // as the main kernel clamps
  int L = p.seq_lens[lo];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int c = b - a, qt = (row - a) / p.tile_tok;
  const int k_hi = min(L, max(0, L - c + min(c, p.tile_tok * (qt + 1))));
  const int nparts = max(1, ceil_div(k_hi, p.part_tokens));
  if (nparts <= 1) return;
  merge_partials<D>(p.ws_ml + wg * p.max_parts, p.ws_o + wg * p.max_parts * D, nparts, p.out + wg * D, lane);
}

// ------------------------------------------------------------------ host
using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, TcParams);

template <bool kPrefill, int D, bool kPairs>
KernelFn pick_kernel(int block_size) {
  switch (block_size) {
    case 16: return chunk_tc_kernel<16, kPrefill, D, kPairs>;
    case 32: return chunk_tc_kernel<32, kPrefill, D, kPairs>;
    case 64: return chunk_tc_kernel<64, kPrefill, D, kPairs>;
    default: return chunk_tc_kernel<128, kPrefill, D, kPairs>;
  }
}

template <bool kPrefill, int D, bool kPairs>
int launch_tc_d(const CUtensorMap &tmq, const CUtensorMap &tmk, const CUtensorMap &tmv, const TcParams &p,
                int block_size, cudaStream_t stream, int max_ctas) {
  using Lay = Layout<kPrefill, D>;
  const KernelFn kernel = pick_kernel<kPrefill, D, kPairs>(block_size);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(Lay::bytes(Lay::kMaxSeqs)))) != cudaSuccess)
    return set_cuda_error(e), PKV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  // one persistent CTA per SM, or fewer when the caller leaves SMs to a concurrent grid
  cfg.gridDim = dim3(max_ctas > 0 && max_ctas < num_sms() ? max_ctas : num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lay::bytes(p.num_seqs);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, tmq, tmk, tmv, p);
  if (e != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
  return PKV_OK;
}

template <bool kPrefill, bool kPairs>
int launch_tc(const CUtensorMap &tmq, const CUtensorMap &tmk, const CUtensorMap &tmv, const TcParams &p,
              int block_size, int head_dim, cudaStream_t stream, int max_ctas = 0) {
  return head_dim == 64 ? launch_tc_d<kPrefill, 64, kPairs>(tmq, tmk, tmv, p, block_size, stream, max_ctas)
                        : launch_tc_d<kPrefill, 128, kPairs>(tmq, tmk, tmv, p, block_size, stream, max_ctas);
}

// The kernels compare raw scores before scaling them; a zero scale would turn
// the masked -inf scores into NaN, so it runs as the smallest normal float,
// whose products with finite scores round to the same weights (all 1).
float kernel_scale_log2(float scale) { return (scale == 0.f ? FLT_MIN : scale) * kLog2e; }

}  // namespace

bool chunk_tc_supported(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int part_tokens) {
  if (num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return false;
  const int group = num_q_heads / num_kv_heads;
  return (q_len == 1 || q_len == 16) && (group & (group - 1)) == 0 && group <= 16 && q_len * group <= kRows &&
         (head_dim == 64 || head_dim == 128) && num_seqs <= Layout<false, 128>::kMaxSeqs &&
         (block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128) &&
         part_tokens % Layout<false, 128>::kTK == 0 && part_tokens % block_size == 0;
}

int chunk_tc_launch(const ChunkTcArgs &a, cudaStream_t stream) {
  const int B = a.num_seqs;
  const int box_rows = a.block_size < Layout<false, 128>::kTK ? a.block_size : Layout<false, 128>::kTK;
  CUtensorMap tmq, tmk, tmv;
  const int group = a.num_q_heads / a.num_kv_heads;
  // q viewed as [B*q_len][Hq][128]: box = 64 columns x G heads x q_len tokens
  if (!make_tensor_map_3d(&tmq, a.q, a.head_dim, a.num_q_heads, static_cast<long long>(B) * a.q_len, 64, group,
                          a.q_len) ||
      !make_tensor_map_2d(&tmk, a.k_cache, a.head_dim, a.rows, 64, box_rows) ||
      !make_tensor_map_2d(&tmv, a.v_cache, a.head_dim, a.rows, 64, box_rows))
    return PKV_ERR_CUDA;
  TcParams p{};
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  p.ws_o = a.ws_o;
  p.ws_ml = static_cast<float2 *>(a.ws_ml);
  p.status = a.status;
  p.num_seqs = B;
  p.max_blocks = a.max_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.part_tokens = a.part_tokens;
  p.max_parts = a.max_parts;
  p.oob_row = static_cast<int>(a.rows);
  p.group = group;
  p.tile_tok = kRows / group;
  p.q_len = a.q_len;
  p.scale_log2 = kernel_scale_log2(a.scale);
  return launch_tc<false, false>(tmq, tmk, tmv, p, a.block_size, a.head_dim, stream);
}

}  // namespace pkv

namespace pkv {
namespace {

struct PrefillPlan {
  int part_tokens = 0, max_parts = 1;
  size_t ws_o_bytes = 0, ws_ml_bytes = 0;
  size_t ws_bytes() const { return part_tokens > 0 ? ws_o_bytes + ws_ml_bytes : 0; }
};

bool make_prefill_plan(int total_q, int num_q_heads, int head_dim, int max_seq_len, int partition_size,
                       PrefillPlan *plan) {
  if (total_q < 0 || num_q_heads < 1 || head_dim < 1 || max_seq_len < 0 || partition_size < 0) return false;
  if (partition_size == 0) return *plan = PrefillPlan{}, true;
  if (partition_size % Layout<true, 128>::kTK != 0) return false;  // whole key tiles
  const long long parts = max_seq_len > 0 ? (static_cast<long long>(max_seq_len) + partition_size - 1) / partition_size : 1;
  if (parts > 65535) return false;
  plan->part_tokens = partition_size;
  plan->max_parts = static_cast<int>(parts);
  const size_t rows = static_cast<size_t>(total_q) * num_q_heads;
  plan->ws_o_bytes = (rows * plan->max_parts * head_dim * sizeof(float) + 255) & ~size_t(255);
  plan->ws_ml_bytes = rows * plan->max_parts * sizeof(float2);
  return true;
}

}  // namespace

int prefill_entry(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *seq_lens, const int32_t *q_start, int num_seqs, int total_q,
                  int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                  int max_seq_len, int partition_size, pkv_bf16 *out, void *workspace, size_t workspace_bytes,
                  int32_t *d_status, void *stream, int max_ctas, const int32_t *work) {
  if (num_seqs < 0 || total_q < 0 || max_blocks_per_seq < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_blocks < 0 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_ARG;
  const int group = num_q_heads / num_kv_heads;
  if ((head_dim != 64 && head_dim != 128) || group > 16) return PKV_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > Layout<true, 128>::kMaxSeqs) return PKV_ERR_UNSUPPORTED;
  PrefillPlan plan;
  if (!make_prefill_plan(total_q, num_q_heads, head_dim, max_seq_len, partition_size, &plan)) return PKV_ERR_ARG;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_start || !out) return PKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(q_start) & 3u))
    return PKV_ERR_ARG;
  if (num_blocks == 0) return PKV_ERR_ARG;
  const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
  if (rows + block_size >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
  const int tile_tok = kRows / group;
  // the largest item count the kernel forms: every row its own query tile, split
  if (static_cast<long long>(total_q) * num_kv_heads * plan.max_parts >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= (1ll << 31)) return PKV_ERR_UNSUPPORTED;
  if (plan.ws_bytes() > 0 && (!workspace || workspace_bytes < plan.ws_bytes() || !aligned16(workspace)))
    return PKV_ERR_WORKSPACE;
  if (work && (plan.part_tokens > 0 || (reinterpret_cast<uintptr_t>(work) & 3u))) return PKV_ERR_ARG;

  const int box_rows = block_size < Layout<true, 128>::kTK ? block_size : Layout<true, 128>::kTK;
  CUtensorMap tmq, tmk, tmv;
  // q viewed as [total_q][Hq][128]: box = 64 columns x G heads x floor(128 / G)
  // tokens (G not a power of two: the tile's last 128 mod G rows are spare)
  if (!make_tensor_map_3d(&tmq, q, head_dim, num_q_heads, total_q, 64, group, tile_tok) ||
      !make_tensor_map_2d(&tmk, k_cache, head_dim, rows, 64, box_rows) ||
      !make_tensor_map_2d(&tmv, v_cache, head_dim, rows, 64, box_rows))
    return PKV_ERR_CUDA;
  TcParams p{};
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_start = q_start;
  p.out = reinterpret_cast<__nv_bfloat16 *>(out);
  p.status = d_status;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.part_tokens = plan.part_tokens;
  p.max_parts = plan.max_parts;
  p.oob_row = static_cast<int>(rows);
  p.total_q = total_q;
  p.group = group;
  p.tile_tok = tile_tok;
  p.scale_log2 = kernel_scale_log2(scale);
  p.work = work;
  cudaStream_t st = as_stream(stream);
  // Batches of long chunks run over pairs of query tiles, which share every
  // key and value tile (half the key / value traffic per product); batches
  // of mostly short chunks (decodes) split each query tile's keys between the
  // two softmax sets instead, so that both sets work on every item.
  const bool pairs = static_cast<long long>(total_q) >= 2ll * tile_tok * num_seqs;
  if (plan.part_tokens > 0) {
    // split over keys: the items of either schedule per key partition, then
    // the merge of each row's partitions
    p.ws_o = static_cast<float *>(workspace);
    p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + plan.ws_o_bytes);
    const int rc = pairs ? launch_tc<true, true>(tmq, tmk, tmv, p, block_size, head_dim, st, max_ctas)
                         : launch_tc<true, false>(tmq, tmk, tmv, p, block_size, head_dim, st, max_ctas);
    if (rc != PKV_OK) return rc;
    const long long warps = static_cast<long long>(total_q) * num_q_heads;
    const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
    const size_t smem = (static_cast<size_t>(num_seqs) + 1) * sizeof(int);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = head_dim == 128 ? cudaLaunchKernelEx(&cfg, prefill_combine_kernel<128>, p, block_size)
                                          : cudaLaunchKernelEx(&cfg, prefill_combine_kernel<64>, p, block_size);
    if (e != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
    return PKV_OK;
  }
  if (pairs) return launch_tc<true, true>(tmq, tmk, tmv, p, block_size, head_dim, st, max_ctas);
  return launch_tc<true, false>(tmq, tmk, tmv, p, block_size, head_dim, st, max_ctas);
}

}  // namespace pkv

// Host-built prefill work list (pkv.h).  The items and their order are the
// kernel's (Sched::fill): per sequence, per KV head, pairs (or single query
// tiles) longest first; an item's cost is its key tiles, the tiles of a lone
// query tile (no pair partner, or the single-tile schedule) weighing about half
// a pair's, plus a fixed cost per item for its start and its epilogue.
extern "C" int pkv_prefill_items(const int32_t *seq_lens, const int32_t *q_start, int num_seqs, int total_q,
                                 int num_q_heads, int num_kv_heads, int grid, int32_t *items_out, int max_ints,
                                 int *num_ints) {
  if (!seq_lens || !q_start || !items_out || !num_ints || num_seqs < 0 || total_q < 0 || num_q_heads < 1 ||
      num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || grid < 1 || max_ints < 0)
    return PKV_ERR_ARG;
  const int group = num_q_heads / num_kv_heads;
  if (group > 16) return PKV_ERR_UNSUPPORTED;
  constexpr double kItemCost = 2.0;    // key-tile periods lost at an item boundary
  constexpr double kLoneWeight = 0.55;  // a lone query tile's period against a pair's
  const int tile_tok = pkv::kRows / group;
  const bool pairs = static_cast<long long>(total_q) >= 2ll * tile_tok * num_seqs;  // as prefill_entry
  const long long span = pairs ? 2 * tile_tok : tile_tok;
  std::vector<std::pair<double, int>> cost;  // (cost, item index)
  long long n = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const long long a = q_start[s], b = q_start[s + 1];
    if (a < 0 || b < a || b > total_q) return PKV_ERR_ARG;
    const long long c = b - a, L = seq_lens[s] < 0 ? 0 : seq_lens[s];
    const long long np = (c + span - 1) / span;
    n += np * num_kv_heads;
    if (n > (1ll << 30)) return PKV_ERR_ARG;
    for (int h = 0; h < num_kv_heads; ++h)
      for (long long part = 0; part < np; ++part) {
        const long long qt = np - 1 - part;
        const long long k_hi = std::min(L, std::max(0ll, L - c + std::min(c, span * (qt + 1))));
        const bool pair = pairs && (2 * qt + 1) * tile_tok < c;
        const double tiles = static_cast<double>((k_hi + 127) / 128);
        cost.emplace_back((pair ? 1.0 : kLoneWeight) * tiles + kItemCost, static_cast<int>(cost.size()));
      }
  }
  const long long need = 3ll + grid + n;
  *num_ints = need > (1ll << 31) - 1 ? -1 : static_cast<int>(need);
  if (need > max_ints) return PKV_ERR_RANGE;
  // longest first (ties in item order), each to the least-loaded CTA
  std::stable_sort(cost.begin(), cost.end(),
                   [](const std::pair<double, int> &x, const std::pair<double, int> &y) { return x.first > y.first; });
  using Load = std::pair<double, int>;  // (load, CTA)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int g = 0; g < grid; ++g) heap.emplace(0.0, g);
  std::vector<std::vector<int>> lists(grid);
  for (const auto &it : cost) {
    Load l = heap.top();
    heap.pop();
    lists[l.second].push_back(it.second);
    l.first += it.first;
    heap.push(l);
  }
  items_out[0] = grid;
  items_out[1] = static_cast<int32_t>(n);
  int32_t *off = items_out + 2, *items = items_out + 3 + grid;
  int32_t pos = 0;
  for (int g = 0; g < grid; ++g) {
    off[g] = pos;
    for (int i : lists[g]) items[pos++] = i;
  }
  off[grid] = pos;
  return PKV_OK;
}

extern "C" size_t paged_attention_prefill_workspace_size(int total_q, int num_q_heads, int head_dim, int max_seq_len,
                                                         int partition_size) {
  pkv::PrefillPlan plan;
  if (!pkv::make_prefill_plan(total_q, num_q_heads, head_dim, max_seq_len, partition_size, &plan)) return 0;
  return plan.ws_bytes();
}

extern "C" int paged_attention_prefill(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                       const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                                       const int32_t *q_start, int num_seqs, int total_q, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                                       pkv_bf16 *out, int32_t *d_status, void *stream) {
  return pkv::prefill_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, q_start, num_seqs,
                            total_q, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, 0, 0, out,
                            nullptr, 0, d_status, stream, 0, nullptr);
}

extern "C" int paged_attention_prefill_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *seq_lens, const int32_t *q_start, int num_seqs, int total_q,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, int max_seq_len, int partition_size,
                                          pkv_bf16 *out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                                          void *stream) {
  return pkv::prefill_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, q_start, num_seqs,
                            total_q, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, max_seq_len,
                            partition_size, out, workspace, workspace_bytes, d_status, stream, 0, nullptr);
}
