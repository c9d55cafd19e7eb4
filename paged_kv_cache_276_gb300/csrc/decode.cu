// Paged attention over a block-paged KV cache (paged_attention_decode).
//
// Math: out = softmax(scale * q K^T) V  (x321.org "The serving bottleneck is
// not just FLOPs", section "First understand what the KV cache is storing"),
// with K/V rows fetched through the per-sequence block table (same page,
// "PagedAttention borrows an operating-system trick").
//
// Design (GB300, sm_103a):
//   * grid = (partition, kv head, sequence).  A partition is `part_blocks`
//     consecutive logical blocks of one sequence (split-K over the context).
//   * one producer lane per CTA walks the block table and issues 2-D TMA tile
//     loads (128-byte swizzle) of each (block, kv head) K and V tile into a
//     ring of shared-memory stages guarded by mbarriers.  Each tile is
//     block_size x head_dim contiguous bf16 in HBM.
//   * consumer warps compute, per block, S^T = K Q^T and O^T += V^T P^T with
//     warp-level bf16 MMA (m16n8k16): the keys of the block are the M
//     dimension and the query heads of the GQA group are N, so every K/V byte
//     is read once for the whole group.  Online softmax (running max / sum)
//     in fp32, exp2 with log2(e) folded into the scale.
//   * single-token decode: the 4 consumer warps take interleaved blocks and
//     are merged in shared memory at the end; the 16-token chunk variant gives
//     each of 8 consumer warps 16 query rows and all blocks.
//   * a sequence that spans one partition writes bf16 output directly; longer
//     ones write (max, sum, unnormalised O) partials that a second kernel
//     merges exactly (log-sum-exp) into bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <functional>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "pkv.h"
#include "attend.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace pkv {
namespace {

using namespace attend;

constexpr int kDecodeWarps = 4;  // consumer warps, q_len = 1
constexpr int kChunkWarps = 8;   // consumer warps, q_len = 16
constexpr int kChunkLen = 16;
constexpr int kDefaultPartition = 768;

struct Params {
  const __nv_bfloat16 *q;       // [B][q_len][Hq][D]
  const int32_t *block_tables;  // [B][max_blocks]
  const int32_t *seq_lens;      // [B]
  __nv_bfloat16 *out;           // [B][q_len][Hq][D]
  float *ws_o;                  // [B][q_len*Hq][P][D]   unnormalised partial outputs
  float2 *ws_ml;                // [B][q_len*Hq][P]      (running max in log2 units, sum)
  int32_t *status;
  int max_blocks;
  int num_q_heads;
  int num_kv_heads;
  int group;         // query heads per KV head
  int q_len;
  int num_blocks;
  int max_parts;     // P
  int part_blocks;   // blocks per partition
  int oob_row;       // a TMA row coordinate wholly outside the cache (reads zeros)
  int active_warps;  // chunk kernel: consumer warps that own at least one real row
  float scale_log2;  // scale * log2(e)
  // single-token decode with the new token's write folded in (k_new == nullptr: none):
  // sequence i's key / value rows [Hkv][D] go to slot slots[i] before the reads
  const uint4 *k_new, *v_new;
  const int64_t *slots;
  uint4 *k_cache, *v_cache;
  // single-token decode over a host-built work list (nullptr: the grid is
  // (partition, KV head, sequence)): items[0].x = item count, then one item per
  // CTA, {sequence, KV head | partition << 16, length, first physical block}
  const int4 *items;
  int num_seqs;
  // launched right behind a grid whose results this one does not read (the
  // chunk kernel of a mixed step), which waited for our inputs before it let
  // this grid start: no wait here, so the two grids run side by side
  int skip_dependency_wait;
  // nothing this grid reads is written by the kernels launched before it (the
  // layers of one decode step): it streams at once and waits for them only
  // before it writes its workspace or outputs, which they may still read
  int wait_before_writes;
};

// Keys are staged in "units" of 32 consecutive token rows of one partition,
// one unit per ring stage: two whole blocks for block size 16, the whole block
// for 32, 32-row pieces for 64 and 128 (whole tiles would leave too few ring
// stages for four consumer warps).  A unit is copied as kSub boxes of kBoxRows
// rows per tensor (one box per block for 16 and 32).  Measured with half the
// SMs streaming: 16-row units (one block of 16 per stage) 57 GB/s per SM,
// 32-row units 83.
template <int BS>
struct Unit {
  static_assert(BS == 16 || BS == 32 || BS == 64 || BS == 128, "block size 16, 32, 64 or 128");
  static constexpr int kRows = 32;
  static constexpr int kBoxRows = BS < 32 ? BS : 32;  // rows of one copy
  static constexpr int kSub = kRows / kBoxRows;        // copies per unit and tensor
  static constexpr int kPieces = BS / kBoxRows;        // copies per block
};

// Staged unit in shared memory, per tensor: [sub-box][half][kBoxRows rows][64
// bf16] with the 128-byte swizzle (R = kBoxRows rows per sub-box; one sub-box
// unless block 16).
template <int D, int ROWS, int R>
struct Tile {
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
  static_assert(ROWS % R == 0 && R % 16 == 0, "whole boxes of 16-row multiples");
  static constexpr int kHalves = D / 64;                  // 64-column (128-byte) halves of a row
  static constexpr int kHalfBytes = R * 128;              // one half of a box's rows
  static constexpr int kBoxBytes = kHalves * kHalfBytes;  // one copy
  static constexpr int kTileBytes = (ROWS / R) * kBoxBytes;  // K (or V) of one unit
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = (65536 / kStageBytes) < 8 ? (65536 / kStageBytes) : 8;
  static constexpr int kRingBytes = kStages * kStageBytes;
};

template <int D, int BS>
using UnitTile = Tile<D, Unit<BS>::kRows, Unit<BS>::kBoxRows>;

__device__ __forceinline__ int clamp_len(const Params &p, int seq, int block_size, bool report) {
  int L = p.seq_lens[seq];
  const long long cap_tbl = static_cast<long long>(p.max_blocks) * block_size;
  const long long cap_grid = static_cast<long long>(p.max_parts) * p.part_blocks * block_size;
  const long long cap = cap_tbl < cap_grid ? cap_tbl : cap_grid;
  if (L < 0 || L > cap) {
    if (report && p.status) atomicOr(p.status, PKV_STATUS_BAD_LEN);
    L = L < 0 ? 0 : static_cast<int>(cap);
  }
  return L;
}

// A work item's length: clamped like clamp_len, and checked against seq_lens
// (a list built for other lengths is reported, PKV_STATUS_BAD_ITEM).
__device__ __forceinline__ int clamp_item_len(const Params &p, int seq, int L, int block_size, bool report) {
  if (report && p.status && p.seq_lens[seq] != L) atomicOr(p.status, PKV_STATUS_BAD_ITEM);
  const long long cap_tbl = static_cast<long long>(p.max_blocks) * block_size;
  const long long cap_grid = static_cast<long long>(p.max_parts) * p.part_blocks * block_size;
  const long long cap = cap_tbl < cap_grid ? cap_tbl : cap_grid;
  if (L < 0 || L > cap) {
    if (report && p.status) atomicOr(p.status, PKV_STATUS_BAD_LEN);
    L = L < 0 ? 0 : static_cast<int>(cap);
  }
  return L;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// The first 32 block-table entries of a partition (lane i: entry blk0 + i),
// read before the sequence length is known so that the two loads overlap;
// entries past the sequence's end are dropped by the producer unused.
__device__ __forceinline__ int first_window(const Params &p, int seq, int part, int lane) {
  const int e = part * p.part_blocks + lane;
  return e < p.max_blocks ? p.block_tables[static_cast<size_t>(seq) * p.max_blocks + e] : -1;
}

// The new token of (seq, KV head h) when the decode stores it itself
// (paged_attention_decode_write).  Its slot must be the table position of
// token L - 1: returns that block (or -1: no store; a non-negative slot
// elsewhere is reported as PKV_STATUS_BAD_SLOT when report is set).
template <int BS>
__device__ __forceinline__ int new_token_block(const Params &p, int seq, int L, bool report) {
  const int64_t slot = p.slots[seq];
  if (slot < 0) return -1;
  const int last = L - 1, e = last / BS;
  const int entry = last >= 0 && e < p.max_blocks ? p.block_tables[static_cast<size_t>(seq) * p.max_blocks + e] : -1;
  if (entry < 0 || entry >= p.num_blocks || slot != static_cast<int64_t>(entry) * BS + last % BS) {
    if (report && p.status) atomicOr(p.status, PKV_STATUS_BAD_SLOT);
    return -1;
  }
  return entry;
}

// Lane l's 16-byte chunk of the new token's key row (l < D/8) or value row
// (D/8 <= l < D/4) for KV head h.
template <int D>
__device__ __forceinline__ uint4 new_token_chunk(const Params &p, int seq, int h, int lane) {
  constexpr int kChunks = D / 8;
  const size_t src = (static_cast<size_t>(seq) * p.num_kv_heads + h) * kChunks;
  if (lane < kChunks) return p.k_new[src + lane];
  if (lane < 2 * kChunks) return p.v_new[src + lane - kChunks];
  return make_uint4(0u, 0u, 0u, 0u);
}

// Producer (one whole warp): walk this partition's block-table entries and
// stream K/V tiles into the ring.  The warp reads 32 table entries with one
// coalesced load and lane 0 issues the copies.  Stages are released by the
// consumers through the empty barriers (count given at init).
// b0 >= 0: the partition's first block id, known from the work item, so the
// first copies go out before the table window has arrived; the window's first
// entry is checked against it afterwards (PKV_STATUS_BAD_ITEM if they differ).
template <int D, int BS>
__device__ void produce(const CUtensorMap *tmk, const CUtensorMap *tmv, const Params &p, int seq, int h,
                        int blk0, int ntok, int window0, int b0, uint32_t ring, uint32_t full0, uint32_t empty0,
                        volatile int *abort_flag, int lane) {
  using U = Unit<BS>;
  using T = UnitTile<D, BS>;
  constexpr int S = T::kStages;
  const uint64_t pol = l2_policy_evict_first();
  const int32_t *tbl = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + blk0;
  const int nunit = (ntok + U::kRows - 1) / U::kRows;
  const int nbox = (ntok + U::kBoxRows - 1) / U::kBoxRows;  // copies per tensor of this partition
  const int nblk = (ntok + BS - 1) / BS;                    // its table entries
  int issued = 0;
  int window = lane < nblk ? window0 : -1;
  // source row of copy q of the partition (past its end: the zero-fill row);
  // warp-uniform: the lanes hold the current window of 32 table entries
  auto source_row = [&](int q) {
    const int e = q / U::kPieces, piece = q - e * U::kPieces;  // table entry, copy within the block
    if (q < nbox && piece == 0 && (e & 31) == 0 && e > 0) window = e + lane < nblk ? tbl[e + lane] : -1;
    const int b = e == 0 && b0 >= 0 ? b0 : __shfl_sync(0xffffffffu, window, e & 31);
    if (q >= nbox) return p.oob_row;
    if (b >= 0 && b < p.num_blocks) return (b * p.num_kv_heads + h) * BS + piece * U::kBoxRows;
    if (lane == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
    return p.oob_row;  // zero fill
  };
  for (int j = 0; j < nunit; ++j) {
    const int row0 = source_row(j * U::kSub);
    const int s = j % S;
    bool ok = true;
    if (j >= S && !mbar_wait(empty0 + 8 * s, ((j / S) - 1) & 1)) ok = false;
    const bool timed_out = __any_sync(0xffffffffu, !ok);
    if (timed_out || __any_sync(0xffffffffu, *abort_flag != 0)) {  // warp-uniform decision
      if (lane == 0) {
        if (p.status && timed_out) atomicOr(p.status, PKV_STATUS_TIMEOUT);
        *abort_flag = 1;
      }
      break;
    }
    const uint32_t full = full0 + 8 * s;
    const uint32_t kdst = ring + s * T::kStageBytes;
    const uint32_t vdst = kdst + T::kTileBytes;
    if (lane == 0) mbar_arrive_expect_tx(full, T::kStageBytes);
    // one copy per box: with head_dim 128 the map's box holds both 64-column
    // halves of its rows, half after half (the layout the consumers read);
    // fewer, larger copies stream faster per SM than one per half.  A unit's
    // first copy goes out before the rows of its others are looked up.
#pragma unroll
    for (int k = 0; k < U::kSub; ++k) {
      const int row = k == 0 ? row0 : source_row(j * U::kSub + k);
      if (lane == 0) {
        if constexpr (T::kHalves == 2) {
          tma_load_3d(kdst + k * T::kBoxBytes, tmk, 0, row, 0, full, pol);
          tma_load_3d(vdst + k * T::kBoxBytes, tmv, 0, row, 0, full, pol);
        } else {
          tma_load_2d(kdst + k * T::kBoxBytes, tmk, 0, row, full, pol);
          tma_load_2d(vdst + k * T::kBoxBytes, tmv, 0, row, full, pol);
        }
      }
    }
    ++issued;
  }
  if (b0 >= 0 && nunit > 0) {
    const int first = __shfl_sync(0xffffffffu, lane < nblk ? window0 : -1, 0);
    if (lane == 0 && first != b0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_ITEM);
  }
  // never leave a copy in flight into this CTA's shared memory
  if (lane == 0)
    for (int j = issued > S ? issued - S : 0; j < issued; ++j) mbar_wait(full0 + 8 * (j % S), (j / S) & 1);
}

// ------------------------------------------------------------- q_len = 1
template <int D, int BS, int NT>
__global__ void __launch_bounds__((kDecodeWarps + 1) * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const Params p) {
  using U = Unit<BS>;
  using T = UnitTile<D, BS>;
  constexpr int S = T::kStages;
  constexpr int COLS = NT * 8;
  constexpr int DP = D + 4;  // padded row of the merge buffer
  static_assert(kDecodeWarps * COLS * DP * 4 + 2 * kDecodeWarps * COLS * 4 <= T::kRingBytes,
                "merge buffer must fit in the ring");
  // Unit j goes to stage j % S and to consumer warp j % kDecodeWarps.  Every
  // use of a stage must go to the same warp, else a warp could wait on a
  // stage two phases ahead of the barrier and pass the parity test early.
  static_assert(S % kDecodeWarps == 0, "ring stages must be a multiple of the consumer warps");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::kRingBytes);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * S);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Let the merge grid queued behind this one become resident now; it still
  // waits for this whole grid's results before it reads anything.
  grid_launch_dependents();
  // inputs may come from the kernel launched just before
  if (!p.skip_dependency_wait && !p.wait_before_writes) grid_dependency_wait();
  int part, h, seq, L, window0, b0 = -1;
  if (p.items) {
    // a host-built work list: one 16-byte load names this CTA's partition, its
    // length and its first block, so the first copy needs no other load
    const int4 it = p.items[1 + blockIdx.x];
    if (static_cast<int>(blockIdx.x) >= p.items[0].x) return;  // past the list (a grid sized for a bound)
    seq = it.x;
    h = it.y & 0xffff;
    part = static_cast<int>(static_cast<unsigned>(it.y) >> 16);
    if (seq < 0 || seq >= p.num_seqs || h >= p.num_kv_heads || part >= p.max_parts) {
      if (threadIdx.x == 0 && p.status) atomicOr(p.status, PKV_STATUS_BAD_ITEM);
      return;
    }
    window0 = warp == kDecodeWarps ? first_window(p, seq, part, lane) : -1;
    L = clamp_item_len(p, seq, it.z, BS, threadIdx.x == 0);
    b0 = it.w;
  } else {
    part = blockIdx.x;
    h = blockIdx.y;
    seq = blockIdx.z;
    // the producer's first 32 block-table entries load while the length does
    window0 = warp == kDecodeWarps ? first_window(p, seq, part, lane) : -1;
    L = clamp_len(p, seq, BS, part == 0 && threadIdx.x == 0);
  }
  const int part_tokens = p.part_blocks * BS;
  const int nparts = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
  if (part >= nparts) return;
  const int blk0 = part * p.part_blocks;
  const int tok0 = blk0 * BS;  // first key of the partition
  const int ntok = max(0, min(L, tok0 + p.part_blocks * BS) - tok0);
  const int nunit = (ntok + U::kRows - 1) / U::kRows;

  const uint32_t ring = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kDecodeWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();

  WarpAcc<D, NT> acc;
  if (warp == kDecodeWarps) {
    // The new token (paged_attention_decode_write): the CTA of the partition
    // holding it stores its rows to the cache.  No copy of this grid waits for
    // that store: the consumer warp of the token's unit puts the same rows into
    // its staged tile itself (below).
    if (p.k_new && part == nparts - 1) {
      const int entry = new_token_block<BS>(p, seq, L, h == 0 && lane == 0);
      if (entry >= 0 && lane < D / 4) {
        const size_t dst = (static_cast<size_t>(entry) * p.num_kv_heads + h) * BS + (L - 1) % BS;
        const uint4 c = new_token_chunk<D>(p, seq, h, lane);
        if (lane < D / 8) p.k_cache[dst * (D / 8) + lane] = c;
        else p.v_cache[dst * (D / 8) + lane - D / 8] = c;
      }
    }
    produce<D, BS>(&tmk, &tmv, p, seq, h, blk0, ntok, window0, b0, ring, full0, empty0, abort_flag, lane);
  } else {
    const int g4 = lane >> 2, c4 = lane & 3;
    uint32_t qf[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nt * 8 + g4;
      const bool real = col < p.group;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          p.q + (static_cast<size_t>(seq) * p.num_q_heads + h * p.group + (real ? col : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qf[nt][ks][0] = real ? qrow[ks * 8 + c4] : 0u;
        qf[nt][ks][1] = real ? qrow[ks * 8 + 4 + c4] : 0u;
      }
    }
    // the new token's unit: its rows come from the inputs (registers), not
    // from the copy, which may have read the slot before this grid's store
    int patch_unit = -1, patch_row = 0;
    uint4 patch = make_uint4(0u, 0u, 0u, 0u);
    if (p.k_new && part == nparts - 1 && nunit > 0 && warp == (nunit - 1) % kDecodeWarps &&
        new_token_block<BS>(p, seq, L, false) >= 0) {
      patch_unit = nunit - 1;
      patch_row = (L - 1) - (tok0 + patch_unit * U::kRows);
      patch = new_token_chunk<D>(p, seq, h, lane);
    }
    acc.init();
    for (int j = warp; j < nunit; j += kDecodeWarps) {
      const int s = j % S;
      if (!mbar_wait(full0 + 8 * s, (j / S) & 1)) {
        if (p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (j == patch_unit) {  // 128-byte swizzle: chunk c of row r sits at chunk c ^ (r % 8)
        if (lane < D / 4) {
          const int v = lane >= D / 8, c = v ? lane - D / 8 : lane;
          const int box = patch_row / U::kBoxRows, r = patch_row - box * U::kBoxRows;
          const uint32_t dst = ring + s * T::kStageBytes + v * T::kTileBytes + box * T::kBoxBytes +
                               (c >> 3) * T::kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(patch.x), "r"(patch.y),
                       "r"(patch.z), "r"(patch.w)
                       : "memory");
        }
        __syncwarp();
      }
      const int valid = min(U::kRows, ntok - j * U::kRows);  // a partition may end inside a unit
      int vis[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) vis[nt][0] = vis[nt][1] = valid;
      const uint32_t kb = ring + s * T::kStageBytes;
      attend_block<D, U::kRows, NT, U::kBoxRows>(acc, qf, kb, kb + T::kTileBytes, valid, vis, p.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (*abort_flag) break;
    }
  }
  __syncthreads();  // ring drained: reuse it as the merge buffer

  float *so = reinterpret_cast<float *>(smem);             // [warps][COLS][DP]
  float *sm = so + kDecodeWarps * COLS * DP;               // [warps][COLS]
  float *sl = sm + kDecodeWarps * COLS;                    // [warps][COLS]
  if (warp < kDecodeWarps) {
    const int g4 = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = acc.l[nt][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (g4 == 0) {
          sm[warp * COLS + nt * 8 + 2 * c4 + e] = acc.m[nt][e];
          sl[warp * COLS + nt * 8 + 2 * c4 + e] = l;
        }
      }
#pragma unroll
    for (int md = 0; md < D / 16; ++md)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          so[(warp * COLS + nt * 8 + 2 * c4 + (i & 1)) * DP + md * 16 + g4 + (i >> 1) * 8] = acc.o[md][nt][i];
  }
  __syncthreads();
  if (*abort_flag) return;
  if (p.wait_before_writes && !p.skip_dependency_wait) grid_dependency_wait();

  const int rows = p.num_q_heads;  // q_len == 1
  for (int idx = threadIdx.x; idx < p.group * D; idx += blockDim.x) {
    const int col = idx / D, d = idx - col * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sm[w * COLS + col]);
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float mw = sm[w * COLS + col];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      lt += sl[w * COLS + col] * f;
      ot += so[(w * COLS + col) * DP + d] * f;
    }
    const size_t row = static_cast<size_t>(seq) * rows + h * p.group + col;
    if (nparts == 1) {
      p.out[row * D + d] = __float2bfloat16_rn(lt > 0.f ? ot / lt : 0.f);
    } else {
      p.ws_o[(row * p.max_parts + part) * D + d] = ot;
      if (d == 0) p.ws_ml[row * p.max_parts + part] = make_float2(M, lt);
    }
  }
}

// ------------------------------------------------- q_len = 16 causal chunk
// Column c of the CTA is query row (r = c / G, g = c % G) of KV head h; warp w
// owns columns [16w, 16w + 16).  Row r sees keys t < L - 16 + 1 + r.
template <int D, int BS>
__global__ void __launch_bounds__((kChunkWarps + 1) * 32)
    chunk_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const Params p) {
  using U = Unit<BS>;
  using T = UnitTile<D, BS>;
  constexpr int S = T::kStages;
  constexpr int NT = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::kRingBytes);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * S);

  const int part = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Let the merge grid queued behind this one become resident now; it still
  // waits for this whole grid's results before it reads anything.
  grid_launch_dependents();
  grid_dependency_wait();  // inputs may come from the kernel launched just before
  // the producer's first 32 block-table entries load while the length does
  const int window0 = warp == kChunkWarps ? first_window(p, seq, part, lane) : -1;
  const int L = clamp_len(p, seq, BS, part == 0 && threadIdx.x == 0);
  const int part_tokens = p.part_blocks * BS;
  const int nparts = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
  if (part >= nparts) return;
  const int blk0 = part * p.part_blocks;
  const int tok0 = blk0 * BS;  // first key of the partition
  const int ntok = max(0, min(L, tok0 + p.part_blocks * BS) - tok0);
  const int nunit = (ntok + U::kRows - 1) / U::kRows;
  const int ncols = kChunkLen * p.group;

  const uint32_t ring = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, p.active_warps);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kChunkWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();

  if (warp == kChunkWarps) {
    produce<D, BS>(&tmk, &tmv, p, seq, h, blk0, ntok, window0, -1, ring, full0, empty0, abort_flag, lane);
    return;
  }
  if (warp >= p.active_warps) return;

  const int g4 = lane >> 2, c4 = lane & 3;
  const int rows = kChunkLen * p.num_q_heads;
  uint32_t qf[NT][D / 16][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = warp * 16 + nt * 8 + g4;
    const bool real = col < ncols;
    const int r = real ? col / p.group : 0, g = real ? col - (col / p.group) * p.group : 0;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        p.q + (static_cast<size_t>(seq) * rows + r * p.num_q_heads + h * p.group + g) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[nt][ks][0] = real ? qrow[ks * 8 + c4] : 0u;
      qf[nt][ks][1] = real ? qrow[ks * 8 + 4 + c4] : 0u;
    }
  }
  // keys visible to each of this thread's accumulator columns
  int nvis[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = warp * 16 + nt * 8 + 2 * c4 + e;
      nvis[nt][e] = col < ncols ? L - kChunkLen + 1 + col / p.group : 0;
    }

  WarpAcc<D, NT> acc;
  acc.init();
  bool ok = true;
  for (int j = 0; j < nunit; ++j) {
    const int s = j % S;
    if (!mbar_wait(full0 + 8 * s, (j / S) & 1)) {
      if (p.status) atomicOr(p.status, PKV_STATUS_TIMEOUT);
      *abort_flag = 1;
      ok = false;
      break;
    }
    const int key0 = tok0 + j * U::kRows;
    const int valid = min(U::kRows, ntok - j * U::kRows);  // a partition may end inside a unit
    int vis[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      vis[nt][0] = min(valid, nvis[nt][0] - key0);
      vis[nt][1] = min(valid, nvis[nt][1] - key0);
    }
    const uint32_t kb = ring + s * T::kStageBytes;
    attend_block<D, U::kRows, NT, U::kBoxRows>(acc, qf, kb, kb + T::kTileBytes, valid, vis, p.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (*abort_flag) {
      ok = false;
      break;
    }
  }
  if (!ok) return;

#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = acc.l[nt][e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      acc.l[nt][e] = l;
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = warp * 16 + nt * 8 + 2 * c4 + e;
      if (col >= ncols) continue;
      const int r = col / p.group, g = col - r * p.group;
      const size_t row = static_cast<size_t>(seq) * rows + r * p.num_q_heads + h * p.group + g;
      const float l = acc.l[nt][e];
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int md = 0; md < D / 16; ++md)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int d = md * 16 + g4 + hi * 8;
          const float o = acc.o[md][nt][e + 2 * hi];
          if (nparts == 1) {
            p.out[row * D + d] = __float2bfloat16_rn(o * inv);
          } else {
            p.ws_o[(row * p.max_parts + part) * D + d] = o;
          }
        }
      if (nparts > 1 && g4 == 0) p.ws_ml[row * p.max_parts + part] = make_float2(acc.m[nt][e], l);
    }
}

// ---------------------------------------------- cross-partition combine
// One warp per (sequence, query row): the exact merge of its partitions.  Over
// a work list only the sequences the list names (those with more than one
// partition) are merged, by a grid of a few CTAs per SM looping over their rows.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const Params p, int block_size, int total_rows,
                                                      int rows) {
  grid_launch_dependents();
  grid_dependency_wait();  // the partials come from the grid launched just before
  const int lane = threadIdx.x & 31;
  if (p.items) {
    const int4 hdr = p.items[0];
    const int *list = reinterpret_cast<const int *>(p.items + hdr.w);
    const long long n = static_cast<long long>(hdr.z) * rows;
    for (long long w = blockIdx.x * 4ll + (threadIdx.x >> 5); w < n; w += gridDim.x * 4ll) {
      const int k = static_cast<int>(w / rows), r = static_cast<int>(w - static_cast<long long>(k) * rows);
      const int seq = list[k];
      if (seq < 0 || seq >= p.num_seqs) continue;
      const int L = clamp_len(p, seq, block_size, false);
      const int part_tokens = p.part_blocks * block_size;
      const int nparts = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
      if (nparts <= 1) continue;
      const size_t wg = static_cast<size_t>(seq) * rows + r;
      merge_partials<D>(p.ws_ml + wg * p.max_parts, p.ws_o + wg * p.max_parts * D, nparts, p.out + wg * D, lane);
    }
    return;
  }
  const int wg = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (wg >= total_rows) return;
  const int seq = wg / rows;
  const int L = clamp_len(p, seq, block_size, false);
  const int part_tokens = p.part_blocks * block_size;
  const int nparts = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
  if (nparts <= 1) return;
  merge_partials<D>(p.ws_ml + static_cast<size_t>(wg) * p.max_parts, p.ws_o + static_cast<size_t>(wg) * p.max_parts * D,
                    nparts, p.out + static_cast<size_t>(wg) * D, lane);
}

// ------------------------------------------------------------------ host
// Single-token decodes go to the tensor-core kernel only when the caller's
// bound on the sequence length is at least this: its persistent CTAs pay a
// fixed cost at the end of every (sequence, KV head) run (the accumulators
// are read before the next run may write them), which long runs amortise and
// short ones do not.  Measured: 16 x 32768 tokens, block 16: 0.85 -> 0.91 of
// the copy bandwidth; 32 sequences of up to 4096: 0.72 -> 0.62.
constexpr int kTcDecodeMinLen = 16384;
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The cache as a bf16 tensor of rows = num_blocks * Hkv * block_size rows of
// head_dim elements, read box_rows rows at a time with the 128-byte swizzle
// (64 elements wide).  head_dim 64: 2-D, a box is box_rows x 64.  head_dim 128:
// 3-D (64 columns, rows at a 256-byte stride, the two halves of a row at a
// 128-byte stride), a box is 64 x box_rows x 2, so one copy stages a unit's
// rows as [half][row][64], the layout of two 2-D boxes side by side.
bool make_cache_map(CUtensorMap *map, const void *base, int head_dim, int box_rows, long long rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  if (head_dim == 128) {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), 2};
    cuuint64_t strides[2] = {256, 128};  // bytes, dimensions 1 and 2
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
  int part_tokens = 0;
  int max_parts = 0;
  size_t ws_o_bytes = 0;
  size_t ws_ml_bytes = 0;
  size_t ws_bytes() const { return max_parts > 1 ? ws_o_bytes + ws_ml_bytes : 0; }
};

bool make_plan(int num_seqs, int q_len, int num_q_heads, int head_dim, int max_seq_len,
               int partition_size, Plan *plan) {
  if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || head_dim < 1 || max_seq_len < 0) return false;
  const int part = partition_size == 0 ? kDefaultPartition : partition_size;
  if (part < 1) return false;
  plan->part_tokens = part;
  const long long parts = max_seq_len > 0 ? (static_cast<long long>(max_seq_len) + part - 1) / part : 1;
  if (parts > (1 << 20)) return false;
  plan->max_parts = static_cast<int>(parts);
  const size_t rows = static_cast<size_t>(num_seqs) * q_len * num_q_heads;
  plan->ws_o_bytes = rows * plan->max_parts * head_dim * sizeof(float);
  plan->ws_o_bytes = (plan->ws_o_bytes + 255) & ~size_t(255);
  plan->ws_ml_bytes = rows * plan->max_parts * sizeof(float2);
  return true;
}

template <int D, int BS>
constexpr size_t smem_bytes() {
  using T = UnitTile<D, BS>;
  return T::kRingBytes + 2 * T::kStages * 8 + 16 + 1024;
}

template <typename K>
cudaError_t raise_smem_limit(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// Launch with programmatic stream serialisation: the grid may start while the
// previous kernel in the stream drains; it waits (griddepcontrol.wait) before
// reading anything.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int D, int BS>
int launch(const CUtensorMap &tmk, const CUtensorMap &tmv, const Params &p, int num_seqs, int q_len,
           int grid_items, cudaStream_t stream, cudaEvent_t main_done) {
  const dim3 grid = p.items ? dim3(grid_items) : dim3(p.max_parts, p.num_kv_heads, num_seqs);
  constexpr size_t smem = smem_bytes<D, BS>();
  cudaError_t e;
  if (q_len == 1) {
    if (p.group <= 8) {
      auto k = decode_kernel<D, BS, 1>;
      if ((e = raise_smem_limit(k, smem)) != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
      e = launch_pdl(k, grid, dim3((kDecodeWarps + 1) * 32), smem, stream, tmk, tmv, p);
    } else {
      auto k = decode_kernel<D, BS, 2>;
      if ((e = raise_smem_limit(k, smem)) != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
      e = launch_pdl(k, grid, dim3((kDecodeWarps + 1) * 32), smem, stream, tmk, tmv, p);
    }
  } else {
    auto k = chunk_kernel<D, BS>;
    if ((e = raise_smem_limit(k, smem)) != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
    e = launch_pdl(k, grid, dim3((kChunkWarps + 1) * 32), smem, stream, tmk, tmv, p);
  }
  if (e == cudaSuccess && main_done) e = cudaEventRecord(main_done, stream);
  if (e != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
  if (p.max_parts <= 1) return PKV_OK;
  const int rows = q_len * p.num_q_heads;
  const int total = num_seqs * rows;
  // over a work list the merge loops over the listed sequences' rows: a few CTAs per SM at most
  const int ctas = p.items ? std::min((total + 3) / 4, 2 * num_sms()) : (total + 3) / 4;
  e = launch_pdl(combine_kernel<D>, dim3(ctas), dim3(128), 0, stream, p, BS, total, rows);
  if (e != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace

bool make_tensor_map_2d(void *map, const void *base, int dim0, long long dim1, int box0, int box1) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(dim0), static_cast<cuuint64_t>(dim1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(dim0) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1)};
  cuuint32_t estr[2] = {1, 1};
  return enc(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_3d(void *map, const void *base, int dim0, int dim1, long long dim2, int box0, int box1,
                        int box2) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim0), static_cast<cuuint64_t>(dim1),
                        static_cast<cuuint64_t>(dim2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim0) * 2, static_cast<cuuint64_t>(dim0) * dim1 * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1), static_cast<cuuint32_t>(box2)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The new token of every sequence, written by the decode itself
// (paged_attention_decode_write): rows [num_seqs][Hkv][D] and their slots.
struct NewTokens {
  const void *k, *v;
  const int64_t *slots;
  pkv_bf16 *k_cache, *v_cache;
};

int decode_entry(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
                 int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len, int q_len,
                 int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                 int partition_size, pkv_bf16 *out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                 void *stream, void *main_done_event, const NewTokens *nt, const int32_t *items = nullptr,
                 int grid_items = 0, bool skip_dependency_wait = false, bool wait_before_writes = false);

}  // namespace pkv

extern "C" {

size_t paged_attention_workspace_size(int num_seqs, int q_len, int num_q_heads, int head_dim,
                                      int max_seq_len, int partition_size) {
  pkv::Plan plan;
  if (!pkv::make_plan(num_seqs, q_len, num_q_heads, head_dim, max_seq_len, partition_size, &plan)) return 0;
  return plan.ws_bytes();
}

int paged_attention_decode(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                           const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                           int num_seqs, int max_seq_len, int q_len, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, float scale, int partition_size,
                           pkv_bf16 *out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                           void *stream) {
  return paged_attention_decode_ex(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                   max_seq_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                   scale, partition_size, out, workspace, workspace_bytes, d_status, stream, nullptr);
}

int paged_attention_decode_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                              int num_seqs, int max_seq_len, int q_len, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, int num_blocks, float scale, int partition_size,
                              pkv_bf16 *out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                              void *stream, void *main_done_event) {
  return pkv::decode_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                           q_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                           partition_size, out, workspace, workspace_bytes, d_status, stream, main_done_event,
                           nullptr);
}

int paged_attention_decode_write(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                 const int64_t *slot_mapping, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                                 int num_seqs, int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, float scale, int partition_size, pkv_bf16 *out,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status, void *stream,
                                 void *main_done_event) {
  if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping)) return PKV_ERR_ARG;
  if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ARG;
  const pkv::NewTokens nt{k_new, v_new, slot_mapping, k_cache, v_cache};
  return pkv::decode_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                           1, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                           out, workspace, workspace_bytes, d_status, stream, main_done_event, &nt);
}

}  // extern "C"

namespace pkv {
namespace {

// Predicted time of a decode work list with partitions of `part` tokens, from a
// model of one GB300 running the decode kernel: 152 SMs x 3 resident CTAs, the
// CTAs that stream at once share ~6.45 TB/s of HBM, one CTA alone streams at
// most ~40 GB/s, a CTA spends ~2.4 us before its first tile lands, and a list
// that splits any sequence adds ~4 us of merge.  Items go to the CTA slots
// longest first (as launched); every streaming CTA progresses at the same
// rate, so the slots' finishing order in bytes gives the number of CTAs
// streaming at each point and the time is the integral of bytes over rate.
// Only the comparison between partition sizes is used.
double predict_list_time(const int32_t *lens, int num_seqs, int num_kv_heads, int head_dim, int part,
                         std::vector<double> &rest, std::vector<double> &slot) {
  constexpr int kSlots = 456;
  constexpr double kBw = 6.45e3;  // bytes per ns, every streaming CTA together
  constexpr double kRmax = 40.0;  // bytes per ns, one CTA
  constexpr double kStartNs = 2400.0;
  constexpr double kMergeNs = 4000.0;
  const double per_tok = 4.0 * head_dim, start = kStartNs * kBw / kSlots;
  // Whole partitions all cost the same and come first (the longest), so they
  // go round the slots; then the sequences' last, shorter partitions (and the
  // empty sequences), longest first, each to the least loaded slot.
  long long full = 0;
  rest.clear();
  for (int i = 0; i < num_seqs; ++i) {
    const int L = lens[i];
    full += L / part;
    if (L % part != 0 || L == 0) rest.push_back((L % part) * per_tok + start);
  }
  const long long nfull = full * num_kv_heads;
  const double cfull = part * per_tok + start;
  slot.assign(kSlots, static_cast<double>(nfull / kSlots) * cfull);
  for (long long i = 0; i < nfull % kSlots; ++i) slot[i] += cfull;
  std::make_heap(slot.begin(), slot.end(), std::greater<double>());
  std::sort(rest.begin(), rest.end(), std::greater<double>());
  for (double c : rest)
    for (int h = 0; h < num_kv_heads; ++h) {
      std::pop_heap(slot.begin(), slot.end(), std::greater<double>());
      slot.back() += c;
      std::push_heap(slot.begin(), slot.end(), std::greater<double>());
    }
  std::sort(slot.begin(), slot.end());
  double t = 0.0, u = 0.0;
  for (int i = 0; i < kSlots; ++i) {
    const int busy = kSlots - i;
    t += (slot[i] - u) / std::min(kRmax, kBw / busy);
    u = slot[i];
  }
  for (int i = 0; i < num_seqs; ++i)
    if (lens[i] > part) return t + kMergeNs;
  return t;
}

// Whether two sequences' tables name the same physical block among the blocks
// their lengths use (a shared prefix, re-read from L2 by every sharer).
bool tables_share_blocks(const int32_t *lens, const int32_t *tables, int max_blocks, int num_seqs, int block_size) {
  if (!tables) return true;  // unknown: assume sharing
  long long total = 0;
  for (int i = 0; i < num_seqs; ++i) total += (static_cast<long long>(lens[i]) + block_size - 1) / block_size;
  if (total > (1ll << 20)) return true;  // not worth the sort: assume sharing
  std::vector<int32_t> ids;
  ids.reserve(static_cast<size_t>(total));
  for (int i = 0; i < num_seqs; ++i) {
    const long long nb = (static_cast<long long>(lens[i]) + block_size - 1) / block_size;
    for (long long j = 0; j < nb && j < max_blocks; ++j) {
      const int32_t b = tables[static_cast<size_t>(i) * max_blocks + j];
      if (b >= 0) ids.push_back(b);  // -1: an entry past the sequence's blocks
    }
  }
  std::sort(ids.begin(), ids.end());
  return std::adjacent_find(ids.begin(), ids.end()) != ids.end();
}

}  // namespace
}  // namespace pkv

extern "C" {

// Host: the work list of a single-token decode batch (see pkv.h).
int pkv_decode_items(const int32_t *seq_lens, const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
                     int num_kv_heads, int head_dim, int block_size, int partition_size, int32_t *items_out,
                     int max_items, int *num_items) {
  if (!num_items) return PKV_ERR_ARG;
  *num_items = 0;
  if (num_seqs < 0 || num_kv_heads < 1 || num_kv_heads > 65535 || block_size < 1 || max_blocks_per_seq < 0 ||
      max_items < 0 || partition_size < 0 || head_dim < 1 || (num_seqs > 0 && !seq_lens) || !items_out)
    return PKV_ERR_ARG;
  if (partition_size % block_size != 0) return PKV_ERR_ARG;
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  for (int i = 0; i < num_seqs; ++i)
    if (seq_lens[i] < 0 || seq_lens[i] > cap) return PKV_ERR_RANGE;
  int part = partition_size;
  if (part == 0) {
    // the candidate the schedule model predicts fastest (within 0.5 %: the
    // larger, fewer merges).  3072 and 4096 only without shared blocks: with a
    // shared prefix, re-read from L2, a partition that holds the prefix alone
    // streams fastest (measured on 512 sequences behind a 2043-token prefix:
    // 0.476 ms at 2048, 0.647 at 3072)
    const bool shared = pkv::tables_share_blocks(seq_lens, block_tables, max_blocks_per_seq, num_seqs, block_size);
    double best = 0.0;
    std::vector<double> rest, slot;
    rest.reserve(static_cast<size_t>(num_seqs));
    for (int cand : {768, 1024, 1536, 2048, 3072, 4096}) {
      if (cand % block_size != 0 || (shared && cand > 2048)) continue;
      const double t = pkv::predict_list_time(seq_lens, num_seqs, num_kv_heads, head_dim, cand, rest, slot);
      if (part == 0 || t <= best * 1.005) part = cand, best = std::min(best == 0.0 ? t : best, t);
    }
    if (part == 0) part = pkv::kDefaultPartition;
  }
  long long count = 0, merges = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int L = seq_lens[i];
    const long long np = L > 0 ? (static_cast<long long>(L) + part - 1) / part : 1;
    if (np > 65535) return PKV_ERR_UNSUPPORTED;
    count += np * num_kv_heads;
    merges += np > 1;
  }
  // rows after the header: the items, then the merge list, four sequences a row
  const long long rows = count + (merges + 3) / 4;
  if (rows > 0x7fffffffll) return PKV_ERR_UNSUPPORTED;
  *num_items = static_cast<int>(rows);
  if (rows > max_items) return PKV_ERR_RANGE;
  struct Piece {
    int ntok, seq, part, len;
  };
  std::vector<Piece> pieces;
  pieces.reserve(static_cast<size_t>(count / num_kv_heads));
  for (int i = 0; i < num_seqs; ++i) {
    const int L = seq_lens[i];
    const int np = L > 0 ? (L + part - 1) / part : 1;
    for (int j = 0; j < np; ++j) {
      const long long lo = static_cast<long long>(j) * part;
      const long long hi = std::min<long long>(L, lo + part);
      pieces.push_back({static_cast<int>(std::max<long long>(0, hi - lo)), i, j, L});
    }
  }
  // longest first: the CTAs launched first carry the most keys, the shortest fill the tail
  std::stable_sort(pieces.begin(), pieces.end(), [](const Piece &a, const Piece &b) { return a.ntok > b.ntok; });
  int32_t *o = items_out;
  o[0] = static_cast<int32_t>(count);
  o[1] = part;  // the partition the list was built for: pass it to the decode
  o[2] = static_cast<int32_t>(merges);      // sequences whose partitions the merge combines
  o[3] = static_cast<int32_t>(1 + count);   // the row where their list starts
  o += 4;
  const long long part_blocks = part / block_size;
  for (const Piece &pc : pieces) {
    const long long e = pc.part * part_blocks;
    const int b0 = block_tables && pc.ntok > 0 && e < max_blocks_per_seq
                       ? block_tables[static_cast<size_t>(pc.seq) * max_blocks_per_seq + e]
                       : -1;
    for (int h = 0; h < num_kv_heads; ++h, o += 4) {
      o[0] = pc.seq;
      o[1] = static_cast<int32_t>(static_cast<uint32_t>(h) | (static_cast<uint32_t>(pc.part) << 16));
      o[2] = pc.len;
      o[3] = b0;
    }
  }
  for (long long i = 0; i < (merges + 3) / 4 * 4; ++i) o[i] = -1;
  for (int i = 0, k = 0; i < num_seqs; ++i)
    if (seq_lens[i] > part) o[k++] = i;
  return PKV_OK;
}

int paged_attention_decode_items(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                 const int64_t *slot_mapping, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                                 int num_seqs, int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, float scale, int partition_size,
                                 const int32_t *items, int grid_items, pkv_bf16 *out, void *workspace,
                                 size_t workspace_bytes, int32_t *d_status, void *stream, void *main_done_event,
                                 int flags) {
  if ((flags & ~PKV_DECODE_OVERLAP) != 0) return PKV_ERR_ARG;
  if (num_seqs > 0 && (!items || grid_items < 1 || (reinterpret_cast<uintptr_t>(items) & 15u))) return PKV_ERR_ARG;
  const bool store = k_new || v_new || slot_mapping;
  if (store) {
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping)) return PKV_ERR_ARG;
    if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
      return PKV_ERR_ARG;
  }
  const pkv::NewTokens nt{k_new, v_new, slot_mapping, k_cache, v_cache};
  return pkv::decode_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                           1, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                           out, workspace, workspace_bytes, d_status, stream, main_done_event,
                           store ? &nt : nullptr, items, grid_items, false, (flags & PKV_DECODE_OVERLAP) != 0);
}

// One continuous-batching step (see pkv.h): the chunks on the tensor cores with
// a capped grid, the decode rows over their work list right behind it.
int paged_attention_mixed(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                          const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                          const int32_t *q_start, int num_seqs, int total_q, int num_decodes, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                          int max_decode_len, int decode_partition_size, const int32_t *decode_items,
                          int decode_grid, int prefill_ctas, const int32_t *prefill_items, pkv_bf16 *out,
                          void *workspace, size_t workspace_bytes, int32_t *d_status, void *stream) {
  if (num_decodes < 0 || num_decodes > num_seqs || num_decodes > total_q || prefill_ctas < 0 || max_blocks_per_seq < 0)
    return PKV_ERR_ARG;
  const int chunks = num_seqs - num_decodes;
  if (chunks > 0) {
    // the chunk sequences: rows q_start[num_decodes] ...; the decode rows are not theirs
    const int rc = pkv::prefill_entry(q, k_cache, v_cache,
                                      block_tables ? block_tables + static_cast<size_t>(num_decodes) * max_blocks_per_seq
                                                   : nullptr,
                                      max_blocks_per_seq, seq_lens ? seq_lens + num_decodes : nullptr,
                                      q_start ? q_start + num_decodes : nullptr, chunks, total_q, num_q_heads,
                                      num_kv_heads, head_dim, block_size, num_blocks, scale, 0, 0, out, nullptr, 0,
                                      d_status, stream, num_decodes > 0 || prefill_items ? prefill_ctas : 0,
                                      prefill_items);
    if (rc != PKV_OK) return rc;
  }
  if (num_decodes == 0) return PKV_OK;
  if (!decode_items || decode_grid < 1 || (reinterpret_cast<uintptr_t>(decode_items) & 15u)) return PKV_ERR_ARG;
  // rows 0 .. num_decodes-1 of q and out are [num_decodes][1][Hq][d]
  return pkv::decode_entry(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_decodes,
                           max_decode_len, 1, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                           decode_partition_size, out, workspace, workspace_bytes, d_status, stream, nullptr, nullptr,
                           decode_items, decode_grid, chunks > 0);
}

}  // extern "C"

namespace pkv {

// Every check of a decode call's arguments that does not involve the
// workspace, in the order the entry points apply them; on PKV_OK *plan holds
// the split-K partitioning (and *plan is set only then).
int decode_check(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
                 int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len, int q_len,
                 int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                 int partition_size, const pkv_bf16 *out, Plan *plan) {
  if (num_seqs < 0 || max_blocks_per_seq < 0 || max_seq_len < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_blocks < 0 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128) return PKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (q_len == 1) {
    if (group > 16) return PKV_ERR_UNSUPPORTED;
  } else if (q_len == kChunkLen) {
    if (group * kChunkLen > kChunkWarps * 16) return PKV_ERR_UNSUPPORTED;
  } else {
    return q_len < 1 ? PKV_ERR_ARG : PKV_ERR_UNSUPPORTED;
  }
  if (partition_size < 0 || (partition_size != 0 && partition_size % block_size != 0)) return PKV_ERR_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PKV_ERR_ARG;
  const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
  if (rows + block_size >= (1ll << 31) || num_blocks == 0) return num_blocks == 0 ? PKV_ERR_ARG : PKV_ERR_UNSUPPORTED;

  Plan pl;
  if (!make_plan(num_seqs, q_len, num_q_heads, head_dim, max_seq_len, partition_size, &pl)) return PKV_ERR_ARG;
  if (pl.max_parts > 65535) return PKV_ERR_UNSUPPORTED;
  *plan = pl;
  return PKV_OK;
}

int decode_entry(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
                 int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len, int q_len,
                 int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                 int partition_size, pkv_bf16 *out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                 void *stream, void *main_done_event, const NewTokens *nt, const int32_t *items, int grid_items,
                 bool skip_dependency_wait, bool wait_before_writes) {
  cudaEvent_t main_done = static_cast<cudaEvent_t>(main_done_event);
  Plan plan;
  const int checked = decode_check(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                   max_seq_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                   scale, partition_size, out, &plan);
  if (checked != PKV_OK || num_seqs == 0) return checked;
  const int group = num_q_heads / num_kv_heads;
  const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
  if (plan.ws_bytes() > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes() || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  }

  cudaStream_t st = as_stream(stream);
  if (chunk_tc_supported(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, plan.part_tokens) &&
      (q_len > 1 || max_seq_len >= kTcDecodeMinLen)) {
    if (nt) {  // the tensor-core kernel takes the new tokens from the cache: write them first
      const int rc = pkv_write(static_cast<const pkv_bf16 *>(nt->k), static_cast<const pkv_bf16 *>(nt->v), nt->slots,
                               num_seqs, nt->k_cache, nt->v_cache, num_blocks, block_size, num_kv_heads, head_dim,
                               d_status, stream);
      if (rc != PKV_OK) return rc;
    }
    ChunkTcArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.ws_o = plan.ws_bytes() ? static_cast<float *>(workspace) : nullptr;
    a.ws_ml = plan.ws_bytes() ? static_cast<char *>(workspace) + plan.ws_o_bytes : nullptr;
    a.status = d_status;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.part_tokens = plan.part_tokens;
    a.max_parts = plan.max_parts;
    a.rows = rows;
    a.scale = scale;
    int rc = chunk_tc_launch(a, st);
    if (rc == PKV_OK && main_done) {
      const cudaError_t er = cudaEventRecord(main_done, st);
      if (er != cudaSuccess) return set_cuda_error(er), PKV_ERR_CUDA;
    }
    if (rc != PKV_OK || plan.max_parts <= 1) return rc;
    Params pc{};
    pc.seq_lens = seq_lens;
    pc.out = reinterpret_cast<__nv_bfloat16 *>(out);
    pc.ws_o = static_cast<float *>(workspace);
    pc.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + plan.ws_o_bytes);
    pc.status = d_status;
    pc.max_blocks = max_blocks_per_seq;
    pc.max_parts = plan.max_parts;
    pc.part_blocks = plan.part_tokens / block_size;
    const int crows = q_len * num_q_heads, total = num_seqs * crows;
    cudaError_t e = head_dim == 128
                        ? launch_pdl(combine_kernel<128>, dim3((total + 3) / 4), dim3(128), 0, st, pc, block_size,
                                     total, crows)
                        : launch_pdl(combine_kernel<64>, dim3((total + 3) / 4), dim3(128), 0, st, pc, block_size,
                                     total, crows);
    if (e != cudaSuccess) return set_cuda_error(e), PKV_ERR_CUDA;
    return PKV_OK;
  }

  CUtensorMap tmk, tmv;
  const int tile_rows = block_size <= 32 ? block_size : 32;  // the kernels' Unit<BS>::kRows
  if (!make_cache_map(&tmk, k_cache, head_dim, tile_rows, rows) ||
      !make_cache_map(&tmv, v_cache, head_dim, tile_rows, rows))
    return PKV_ERR_CUDA;

  Params p{};
  p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = reinterpret_cast<__nv_bfloat16 *>(out);
  p.ws_o = plan.ws_bytes() ? static_cast<float *>(workspace) : nullptr;
  p.ws_ml = plan.ws_bytes() ? reinterpret_cast<float2 *>(static_cast<char *>(workspace) + plan.ws_o_bytes) : nullptr;
  p.status = d_status;
  p.max_blocks = max_blocks_per_seq;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.q_len = q_len;
  p.num_blocks = num_blocks;
  p.max_parts = plan.max_parts;
  p.part_blocks = plan.part_tokens / block_size;
  p.oob_row = static_cast<int>(rows);
  p.active_warps = (group * kChunkLen + 15) / 16;
  p.scale_log2 = scale * kLog2e;
  p.num_seqs = num_seqs;
  if (items) p.items = reinterpret_cast<const int4 *>(items);  // q_len == 1, grid_items >= 1 (entry checks)
  p.skip_dependency_wait = skip_dependency_wait ? 1 : 0;
  p.wait_before_writes = wait_before_writes ? 1 : 0;
  if (nt) {
    p.k_new = static_cast<const uint4 *>(nt->k);
    p.v_new = static_cast<const uint4 *>(nt->v);
    p.slots = nt->slots;
    p.k_cache = reinterpret_cast<uint4 *>(nt->k_cache);
    p.v_cache = reinterpret_cast<uint4 *>(nt->v_cache);
  }

  switch (head_dim * 1000 + block_size) {
    case 128016: return launch<128, 16>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 128032: return launch<128, 32>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 128064: return launch<128, 64>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 128128: return launch<128, 128>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 64016: return launch<64, 16>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 64032: return launch<64, 32>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    case 64064: return launch<64, 64>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
    default: return launch<64, 128>(tmk, tmv, p, num_seqs, q_len, grid_items, st, main_done);
  }
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// Allocation-free variant of paged_attention_decode.
//
// Some callers cannot allocate device memory at all: an engine that carves all
// of device memory into its own arena at start-up and forbids allocations
// afterwards, or a plugin whose host framework owns every allocation and gives
// the plugin no allocator.  For them the split-K scratch lives in this
// fixed-size array, which every GPU that loads this library keeps until the
// process exits.  Host code must not use the array's name as a device address
// (on the host it is only a stand-in); the real address is looked up once per
// device with cudaGetSymbolAddress, with that device current.
namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set up on first use).
int static_scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pkv::set_cuda_error(e);
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || !ptr) {
      pkv::set_cuda_error(e);
      return PKV_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_static_scratch(
    const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len, int q_len,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    int partition_size, pkv_bf16 *out, int32_t *d_status, void *stream) {
  // The same argument checks as paged_attention_decode first, so an unsupported
  // or malformed call gets the same error code here as there.
  pkv::Plan plan;
  const int checked = pkv::decode_check(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                        max_seq_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                        num_blocks, scale, partition_size, out, &plan);
  if (checked != PKV_OK || num_seqs == 0) return checked;
  if (plan.ws_bytes() > kStaticScratchBytes) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (plan.ws_bytes() > 0) {
    const int rc = static_scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
  }
  // No part of the scratch has to start at zero: every partial the combine
  // step reads is written by the same call first.
  return paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                max_seq_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, partition_size, out, scratch,
                                plan.ws_bytes() > 0 ? kStaticScratchBytes : 0, d_status, stream);
}
