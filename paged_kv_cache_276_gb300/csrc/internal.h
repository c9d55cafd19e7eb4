// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

void set_cuda_error(cudaError_t e);
int num_sms();

// 2-D / 3-D bf16 tensor maps with 128-byte swizzle (defined in decode.cu).
// dims are in elements, innermost first; rows of dim0 elements are contiguous.
bool make_tensor_map_2d(void *map, const void *base, int dim0, long long dim1, int box0, int box1);
bool make_tensor_map_3d(void *map, const void *base, int dim0, int dim1, long long dim2, int box0, int box1,
                        int box2);

// Chunked causal query on tcgen05 (chunk_tc.cu): q_len 16, 8 query heads per
// KV head, head_dim 128, block 16 or 32, partitions a multiple of 64 tokens.
struct ChunkTcArgs {
  const void *q, *k_cache, *v_cache;
  const int32_t *block_tables, *seq_lens;
  void *out;
  float *ws_o;
  void *ws_ml;
  int32_t *status;
  int num_seqs, q_len, max_blocks, num_q_heads, num_kv_heads, num_blocks, block_size, head_dim;
  int part_tokens, max_parts;
  long long rows;  // num_blocks * num_kv_heads * block_size
  float scale;
};
bool chunk_tc_supported(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int part_tokens);
int chunk_tc_launch(const ChunkTcArgs &a, cudaStream_t stream);

// Chunked prefill (chunk_tc.cu): paged_attention_prefill_ex with a cap on the
// persistent grid (max_ctas > 0: at most that many CTAs, one per SM) and an
// optional device copy of a pkv_prefill_items list (work; not with a split).
int prefill_entry(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *seq_lens, const int32_t *q_start, int num_seqs, int total_q,
                  int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                  int max_seq_len, int partition_size, pkv_bf16 *out, void *workspace, size_t workspace_bytes,
                  int32_t *d_status, void *stream, int max_ctas, const int32_t *work);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Returns PKV_OK or PKV_ERR_CUDA after a launch, recording the CUDA error text.
inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace pkv
