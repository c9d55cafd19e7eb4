// Slot write (pkv_write), copy-on-write block copy (pkv_block_copy) and block
// swap to and from page-locked host memory (pkv_swap_out / pkv_swap_in).
//
// All are pure data movement: 16-byte vector loads and stores, coalesced
// along head_dim, grid-stride loops sized to the SM count.
#include <cstdio>
#include <cuda_runtime.h>

#include "internal.h"
#include "pkv.h"

namespace pkv {

namespace {

thread_local char g_cuda_error[256] = "";

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

// One thread moves one 16-byte chunk of a token's key row and the same chunk
// of its value row.  idx enumerates (token, kv head, chunk) with chunk fastest,
// so a warp reads and writes whole contiguous rows.
__global__ void __launch_bounds__(256) kv_write_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int64_t *__restrict__ slots,
    int64_t total, uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots,
    int block_size, int num_kv_heads, int chunks, int32_t *status) {
  // the attention grid queued behind this one may become resident now (it
  // waits for this grid's writes before it reads the cache)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * chunks;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_token;
    const int64_t rem = idx - t * per_token;
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (rem == 0 && status) atomicOr(status, PKV_STATUS_BAD_SLOT);
      continue;
    }
    const int64_t h = rem / chunks;
    const int64_t c = rem - h * chunks;
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks + c;
    const uint4 kv = k[idx];
    const uint4 vv = v[idx];
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

// blockIdx.y walks the (src, dst) pairs; the x-dimension threads stride over
// the pair's contiguous block (all heads, slots, dims), four chunks in flight
// per thread.
__global__ void __launch_bounds__(256) block_copy_kernel(
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, const int32_t *__restrict__ pairs,
    int num_pairs, int num_blocks, int64_t chunks_per_block, int32_t *status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int pr = blockIdx.y; pr < num_pairs; pr += gridDim.y) {
    const int src = pairs[2 * pr];
    const int dst = pairs[2 * pr + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicOr(status, PKV_STATUS_BAD_BLOCK);
      continue;
    }
    const uint4 *ks = k_cache + static_cast<int64_t>(src) * chunks_per_block;
    const uint4 *vs = v_cache + static_cast<int64_t>(src) * chunks_per_block;
    uint4 *kd = k_cache + static_cast<int64_t>(dst) * chunks_per_block;
    uint4 *vd = v_cache + static_cast<int64_t>(dst) * chunks_per_block;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (; i + stride < chunks_per_block; i += 2 * stride) {
      const uint4 a = ks[i], b = ks[i + stride], c = vs[i], d = vs[i + stride];
      kd[i] = a;
      kd[i + stride] = b;
      vd[i] = c;
      vd[i + stride] = d;
    }
    for (; i < chunks_per_block; i += stride) {
      kd[i] = ks[i];
      vd[i] = vs[i];
    }
  }
}

// Whole blocks between the caches and a host buffer of n blocks: blockIdx.y
// walks the listed blocks, the x threads stride over a block's 16-byte chunks
// (all heads, slots and dims), K and V together.  to_host: cache -> buffer.
__global__ void __launch_bounds__(256) swap_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                   uint4 *__restrict__ buf_k, uint4 *__restrict__ buf_v,
                                                   const int32_t *__restrict__ ids, int n, int num_blocks,
                                                   int64_t chunks_per_block, int to_host, int32_t *status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.y; i < n; i += gridDim.y) {
    const int b = ids[i];
    if (b < 0 || b >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicOr(status, PKV_STATUS_BAD_BLOCK);
      continue;
    }
    uint4 *ck = k_cache + static_cast<int64_t>(b) * chunks_per_block;
    uint4 *cv = v_cache + static_cast<int64_t>(b) * chunks_per_block;
    uint4 *hk = buf_k + static_cast<int64_t>(i) * chunks_per_block;
    uint4 *hv = buf_v + static_cast<int64_t>(i) * chunks_per_block;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < chunks_per_block;
         c += stride) {
      if (to_host) {
        const uint4 a = ck[c], d = cv[c];
        hk[c] = a;
        hv[c] = d;
      } else {
        const uint4 a = hk[c], d = hv[c];
        ck[c] = a;
        cv[c] = d;
      }
    }
  }
}

// Device address of a buffer the caller says is page-locked host memory (or
// device memory); nullptr for pageable memory the device cannot address.
void *device_view(const void *p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of a failed query
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost && attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return nullptr;
  return attr.devicePointer;
}

int swap_blocks(const void *k_cache, const void *v_cache, const int32_t *block_ids, int n, const void *host_k,
                const void *host_v, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                int32_t *d_status, void *stream, bool to_host) {
  if (n < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 8 || head_dim % 8 != 0)
    return PKV_ERR_ARG;
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_ids || !host_k || !host_v) return PKV_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(host_k) || !aligned16(host_v) ||
      (reinterpret_cast<uintptr_t>(block_ids) & 3u))
    return PKV_ERR_ARG;
  void *dk = device_view(host_k), *dv = device_view(host_v);
  if (!dk || !dv) return PKV_ERR_ARG;
  const int64_t chunks_per_block = static_cast<int64_t>(num_kv_heads) * block_size * head_dim / 8;
  const int threads = 256;
  int64_t gx = (chunks_per_block + threads - 1) / threads;
  if (gx > 32) gx = 32;
  const int gy = n < 65535 ? n : 65535;
  swap_kernel<<<dim3(static_cast<unsigned>(gx), gy), threads, 0, as_stream(stream)>>>(
      reinterpret_cast<uint4 *>(const_cast<void *>(k_cache)), reinterpret_cast<uint4 *>(const_cast<void *>(v_cache)),
      reinterpret_cast<uint4 *>(dk), reinterpret_cast<uint4 *>(dv), block_ids, n, num_blocks, chunks_per_block,
      to_host ? 1 : 0, d_status);
  return check_launch();
}

}  // namespace

void set_cuda_error(cudaError_t e) {
  std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
}

int num_sms() { return sm_count(); }

}  // namespace pkv

extern "C" {

const char *pkv_error_string(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_ARG: return "invalid argument";
    case PKV_ERR_OOM: return "out of free blocks";
    case PKV_ERR_RANGE: return "index out of range";
    case PKV_ERR_UNSUPPORTED: return "unsupported size";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_TIMEOUT: return "device wait timed out";
    case PKV_ERR_SHARED: return "append into a shared block (copy it first)";
    case PKV_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown error";
  }
}

const char *pkv_last_cuda_error(void) { return pkv::g_cuda_error; }

int pkv_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping, int num_tokens,
              pkv_bf16 *k_cache, pkv_bf16 *v_cache, int num_blocks, int block_size,
              int num_kv_heads, int head_dim, int32_t *d_status, void *stream) {
  if (num_tokens < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 8 ||
      head_dim % 8 != 0)
    return PKV_ERR_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_ARG;
  if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) ||
      !pkv::aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ARG;
  const int chunks = head_dim / 8;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(pkv::num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  pkv::kv_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, pkv::as_stream(stream)>>>(
      reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), slot_mapping, total,
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
      static_cast<int64_t>(num_blocks) * block_size, block_size, num_kv_heads, chunks, d_status);
  return pkv::check_launch();
}

int pkv_block_copy(pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *src_dst_pairs,
                   int num_pairs, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                   int32_t *d_status, void *stream) {
  if (num_pairs < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 8 ||
      head_dim % 8 != 0)
    return PKV_ERR_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PKV_ERR_ARG;
  if (!pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(src_dst_pairs) & 3u))
    return PKV_ERR_ARG;
  const int64_t chunks_per_block = static_cast<int64_t>(num_kv_heads) * block_size * head_dim / 8;
  const int threads = 256;
  int64_t gx = (chunks_per_block + 2 * threads - 1) / (2 * threads);
  if (gx > 64) gx = 64;
  const int gy = num_pairs < 65535 ? num_pairs : 65535;
  pkv::block_copy_kernel<<<dim3(static_cast<unsigned>(gx), gy), threads, 0,
                           pkv::as_stream(stream)>>>(
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), src_dst_pairs,
      num_pairs, num_blocks, chunks_per_block, d_status);
  return pkv::check_launch();
}

int pkv_swap_out(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_ids, int n,
                 pkv_bf16 *host_k, pkv_bf16 *host_v, int num_blocks, int block_size, int num_kv_heads,
                 int head_dim, int32_t *d_status, void *stream) {
  return pkv::swap_blocks(k_cache, v_cache, block_ids, n, host_k, host_v, num_blocks, block_size, num_kv_heads,
                          head_dim, d_status, stream, true);
}

int pkv_swap_in(const pkv_bf16 *host_k, const pkv_bf16 *host_v, const int32_t *block_ids, int n,
                pkv_bf16 *k_cache, pkv_bf16 *v_cache, int num_blocks, int block_size, int num_kv_heads,
                int head_dim, int32_t *d_status, void *stream) {
  return pkv::swap_blocks(k_cache, v_cache, block_ids, n, host_k, host_v, num_blocks, block_size, num_kv_heads,
                          head_dim, d_status, stream, false);
}

}  // extern "C"
