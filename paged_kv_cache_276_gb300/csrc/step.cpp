// Decode step runner (pkv_step_*): the host side of one decode step of a batch
// through every layer, issued by one call.
//
// A step is the allocator's append and table fill (host), one copy of the
// step's inputs to the device, per layer the slot write and the paged decode,
// and one copy of the outputs back.  Issued one by one from a scripting
// language those are a dozen calls whose argument handling costs more than
// the copies; here they are one C call, and with graphs the device part is a
// single graph launch captured once per (batch size, partition count).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <tuple>
#include <utility>
#include <vector>

#include "internal.h"
#include "pkv.h"

namespace {

constexpr int kMaxGraphs = 32;
constexpr int kGridGranule = 256;  // decode CTAs a captured graph may launch beyond the item count
constexpr int kRepick = 64;  // steps between two picks of the work list's partition
constexpr int kDefaultPartition = 768;  // paged_attention_decode's default

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

bool pinned_host(const void *p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeHost;
}

}  // namespace

struct pkv_step {
  pkv_step_config cfg{};
  pkv_step_layout lay{};
  pkv_alloc *alloc = nullptr;
  std::vector<pkv_bf16 *> k, v;
  char *hs = nullptr, *ds = nullptr;
  char *dout = nullptr, *hout = nullptr;
  void *ws = nullptr;
  size_t ws_bytes = 0;
  int32_t *status = nullptr;
  int part = kDefaultPartition;
  cudaStream_t cap = nullptr;
  cudaStream_t copy = nullptr;  // the step's host <-> device copies, beside the kernels
  cudaEvent_t done = nullptr;
  cudaEvent_t start = nullptr, copied_out = nullptr;
  std::vector<cudaEvent_t> layer_in, layer_done;  // per group of layers: its inputs landed, its kernels finished
  bool pending = false;
  // (n, partitions, partition size, decode grid): the grid is the work list's
  // item count rounded up to kGridGranule, so a graph launches few idle CTAs
  // and is captured again only when the count passes its granule
  std::map<std::tuple<int, int, int, int>, cudaGraphExec_t> graphs;
  int auto_part = 0, auto_n = 0, auto_age = 0;  // the work list's partition pick, kept between steps
};

namespace {

void drop_graphs(pkv_step *s) {
  for (auto &g : s->graphs) cudaGraphExecDestroy(g.second);
  s->graphs.clear();
}

// Layers in groups for the copies: 1, 2, 4, then 8 at a time, shrinking again
// towards the end (never more than half of the layers left), so the first
// kernels start after a small copy, the last output returns in a small copy,
// and between groups consecutive layers' kernels overlap (an event between two
// kernels would make the second wait for the first to finish).  Returns the
// first layer of each group, then the layer count.
std::vector<int> layer_groups(int layers) {
  std::vector<int> first;
  for (int lo = 0, k = 1; lo < layers; k *= 2) {
    const int left = layers - lo;
    const int g = left <= 1 ? left : std::min(std::min(k, 8), std::max(1, left / 2));
    first.push_back(lo);
    lo += g;
  }
  first.push_back(layers);
  return first;
}

// One step on `st`: the common inputs (slots, tables, lengths, work list) and
// the layers' queries, keys and values go to the device on the runner's copy
// stream, group after group, while the kernels of the groups already copied
// run on `st`; each group's outputs go back as soon as its kernels finish.  So
// the copies overlap the kernels instead of preceding and following all of
// them.  q_len 1: the decode runs grid_items CTAs over the work list in the
// staging buffer, each layer overlapping the one before (PKV_DECODE_OVERLAP:
// the layers' inputs are independent).
int enqueue(pkv_step *s, cudaStream_t st, int n, int max_seq_len, int grid_items, int partition) {
  const pkv_step_config &c = s->cfg;
  const pkv_step_layout &L = s->lay;
  cudaError_t e;
  auto fail = [](cudaError_t err) { return pkv::set_cuda_error(err), PKV_ERR_CUDA; };
  const std::vector<int> groups = layer_groups(c.num_layers);
  const int ng = static_cast<int>(groups.size()) - 1;
  // the copies may overwrite the staging buffers only after the work before this step
  if ((e = cudaEventRecord(s->start, st)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(s->copy, s->start, 0)) != cudaSuccess) return fail(e);
  for (int gi = 0; gi < ng; ++gi) {
    // the first group comes with the common segment in front of it
    const size_t lo = gi == 0 ? 0 : L.q_offset + groups[gi] * L.layer_stride;
    const size_t hi = L.q_offset + groups[gi + 1] * L.layer_stride;
    if ((e = cudaMemcpyAsync(s->ds + lo, s->hs + lo, hi - lo, cudaMemcpyHostToDevice, s->copy)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(s->layer_in[gi], s->copy)) != cudaSuccess) return fail(e);
  }
  const auto *slots = reinterpret_cast<const int64_t *>(s->ds + L.slots_offset);
  const auto *tables = reinterpret_cast<const int32_t *>(s->ds + L.tables_offset);
  const auto *lens = reinterpret_cast<const int32_t *>(s->ds + L.lens_offset);
  for (int gi = 0, l = 0; gi < ng; ++gi) {
    if ((e = cudaStreamWaitEvent(st, s->layer_in[gi], 0)) != cudaSuccess) return fail(e);
    for (; l < groups[gi + 1]; ++l) {
      const char *layer = s->ds + L.q_offset + l * L.layer_stride;
      const auto *q = reinterpret_cast<const pkv_bf16 *>(layer);
      const auto *kn = reinterpret_cast<const pkv_bf16 *>(layer + (L.k_offset - L.q_offset));
      const auto *vn = reinterpret_cast<const pkv_bf16 *>(layer + (L.v_offset - L.q_offset));
      auto *out = reinterpret_cast<pkv_bf16 *>(s->dout + l * L.out_layer_bytes);
      int rc;
      if (c.q_len == 1) {  // the allocator's slots are the newest tokens' table positions: one grid
        const auto *items = reinterpret_cast<const int32_t *>(s->ds + L.items_offset);
        rc = paged_attention_decode_items(q, kn, vn, slots, s->k[l], s->v[l], tables, c.max_blocks_per_seq, lens, n,
                                          max_seq_len, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                          c.num_blocks, c.scale, partition, items, grid_items, out, s->ws,
                                          s->ws_bytes, s->status, st, nullptr, PKV_DECODE_OVERLAP);
      } else {
        rc = pkv_write(kn, vn, slots, n * c.q_len, s->k[l], s->v[l], c.num_blocks, c.block_size, c.num_kv_heads,
                       c.head_dim, s->status, st);
        if (rc != PKV_OK) return rc;
        rc = paged_attention_decode(q, s->k[l], s->v[l], tables, c.max_blocks_per_seq, lens, n, max_seq_len,
                                    c.q_len, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks,
                                    c.scale, c.partition_size, out, s->ws, s->ws_bytes, s->status, st);
      }
      if (rc != PKV_OK) return rc;
    }
    // the group's outputs, contiguous in the output buffer
    const size_t o0 = groups[gi] * L.out_layer_bytes, o1 = groups[gi + 1] * L.out_layer_bytes;
    if ((e = cudaEventRecord(s->layer_done[gi], st)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(s->copy, s->layer_done[gi], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaMemcpyAsync(s->hout + o0, s->dout + o0, o1 - o0, cudaMemcpyDeviceToHost, s->copy)) != cudaSuccess)
      return fail(e);
  }
  // the step ends on `st` once its last output has landed
  if ((e = cudaEventRecord(s->copied_out, s->copy)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(st, s->copied_out, 0)) != cudaSuccess) return fail(e);
  return PKV_OK;
}

int capture(pkv_step *s, int n, int max_seq_len, int grid_items, int partition, cudaGraphExec_t *exec) {
  cudaError_t e;
  if (!s->cap && (e = cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking)) != cudaSuccess)
    return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  // Relaxed: the launch helpers may set kernel attributes or look up driver
  // entry points while the stream is being captured.
  if ((e = cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeRelaxed)) != cudaSuccess)
    return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  const int rc = enqueue(s, s->cap, n, max_seq_len, grid_items, partition);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(s->cap, &g);
  if (rc != PKV_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    if (rc != PKV_OK) return rc;
    return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  }
  e = cudaGraphInstantiate(exec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_step_layout_of(const pkv_step_config *c, pkv_step_layout *o) {
  if (!c || !o) return PKV_ERR_ARG;
  if (c->num_layers < 1 || c->max_seqs < 1 || c->q_len < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 ||
      c->head_dim < 1 || c->block_size < 1 || c->num_blocks < 1 || c->max_blocks_per_seq < 1 ||
      c->partition_size < 0)
    return PKV_ERR_ARG;
  const long long cap = static_cast<long long>(c->max_blocks_per_seq) * c->block_size;
  if (cap >= (1ll << 31)) return PKV_ERR_ARG;
  // Every count below is a product of ints; bound them so no size_t product overflows.
  const double rows = static_cast<double>(c->max_seqs) * c->q_len;
  const double worst = rows * (c->num_q_heads + 2.0 * c->num_kv_heads) * c->head_dim * 2.0 * c->num_layers +
                       static_cast<double>(c->max_seqs) * c->max_blocks_per_seq * 4.0;
  if (worst > 9.0e15) return PKV_ERR_ARG;
  const size_t r = static_cast<size_t>(c->max_seqs) * c->q_len;
  const size_t qb = up256(r * c->num_q_heads * c->head_dim * 2);
  const size_t kvb = up256(r * c->num_kv_heads * c->head_dim * 2);
  std::memset(o, 0, sizeof(*o));
  // the segments every layer reads come first, then each layer's queries, keys and values
  o->slots_offset = 0;
  o->tables_offset = o->slots_offset + up256(r * sizeof(int64_t));
  o->lens_offset = o->tables_offset + up256(static_cast<size_t>(c->max_seqs) * c->max_blocks_per_seq * 4);
  size_t common = o->lens_offset + up256(static_cast<size_t>(c->max_seqs) * 4);
  if (c->q_len == 1) {  // the decode's work list: at most every sequence's partitions x KV heads
    const int part = c->partition_size > 0 ? c->partition_size : kDefaultPartition;
    // rows after the list's header: every sequence's partitions x KV heads, then the merge list
    const long long items = static_cast<long long>(c->max_seqs) * c->num_kv_heads * ((cap + part - 1) / part) +
                            (c->max_seqs + 3) / 4;
    if (items > 0x7ffffffell) return PKV_ERR_ARG;
    o->items_offset = common;
    o->max_items = static_cast<int>(items);
    common += up256(static_cast<size_t>(items + 1) * 16);
  }
  o->q_layer_bytes = qb;
  o->kv_layer_bytes = kvb;
  o->layer_stride = qb + 2 * kvb;
  o->q_offset = common;
  o->k_offset = o->q_offset + qb;
  o->v_offset = o->k_offset + kvb;
  o->stage_bytes = common + c->num_layers * o->layer_stride;
  o->out_layer_bytes = qb;
  o->out_bytes = c->num_layers * qb;
  o->workspace_bytes = paged_attention_workspace_size(c->max_seqs, c->q_len, c->num_q_heads, c->head_dim,
                                                      static_cast<int>(cap), c->partition_size);
  return PKV_OK;
}

int pkv_step_create(const pkv_step_config *cfg, pkv_alloc *alloc, pkv_bf16 *const *k_caches,
                    pkv_bf16 *const *v_caches, void *host_stage, void *dev_stage, pkv_bf16 *dev_out,
                    pkv_bf16 *host_out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                    pkv_step **out) {
  if (!out) return PKV_ERR_ARG;
  *out = nullptr;
  pkv_step_layout lay;
  int rc = pkv_step_layout_of(cfg, &lay);
  if (rc != PKV_OK) return rc;
  if (!alloc || !k_caches || !v_caches || !host_stage || !dev_stage || !dev_out || !host_out) return PKV_ERR_ARG;
  if (!pkv::aligned16(host_stage) || !pkv::aligned16(dev_stage) || !pkv::aligned16(dev_out) ||
      !pkv::aligned16(host_out))
    return PKV_ERR_ARG;
  if (lay.workspace_bytes > 0 && (!workspace || workspace_bytes < lay.workspace_bytes)) return PKV_ERR_WORKSPACE;
  for (int l = 0; l < cfg->num_layers; ++l)
    if (!k_caches[l] || !v_caches[l]) return PKV_ERR_ARG;
  if (!pinned_host(host_stage) || !pinned_host(host_out)) return PKV_ERR_ARG;

  auto *s = new (std::nothrow) pkv_step;
  if (!s) return PKV_ERR_OOM;
  s->cfg = *cfg;
  s->lay = lay;
  s->alloc = alloc;
  s->k.assign(k_caches, k_caches + cfg->num_layers);
  s->v.assign(v_caches, v_caches + cfg->num_layers);
  s->hs = static_cast<char *>(host_stage);
  s->ds = static_cast<char *>(dev_stage);
  s->dout = reinterpret_cast<char *>(dev_out);
  s->hout = reinterpret_cast<char *>(host_out);
  s->ws = workspace;
  s->ws_bytes = workspace_bytes;
  s->status = d_status;
  s->part = cfg->partition_size > 0 ? cfg->partition_size : kDefaultPartition;
  cudaError_t e = cudaEventCreateWithFlags(&s->done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->copied_out, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s->copy, cudaStreamNonBlocking);
  s->layer_in.assign(cfg->num_layers, nullptr);
  s->layer_done.assign(cfg->num_layers, nullptr);
  for (int l = 0; l < cfg->num_layers && e == cudaSuccess; ++l) {
    e = cudaEventCreateWithFlags(&s->layer_in[l], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->layer_done[l], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    pkv::set_cuda_error(e);
    pkv_step_destroy(s);
    return PKV_ERR_CUDA;
  }
  *out = s;
  return PKV_OK;
}

int pkv_step_wait(pkv_step *s) {
  if (!s) return PKV_ERR_ARG;
  if (!s->pending) return PKV_OK;
  const cudaError_t e = cudaEventSynchronize(s->done);
  if (e != cudaSuccess) return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  s->pending = false;
  return PKV_OK;
}

void pkv_step_destroy(pkv_step *s) {
  if (!s) return;
  pkv_step_wait(s);
  drop_graphs(s);
  if (s->cap) cudaStreamDestroy(s->cap);
  if (s->copy) cudaStreamDestroy(s->copy);
  for (cudaEvent_t ev : {s->done, s->start, s->copied_out})
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : s->layer_in)
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : s->layer_done)
    if (ev) cudaEventDestroy(ev);
  delete s;
}

int pkv_step_run(pkv_step *s, const int64_t *seq_ids, int n, void *stream) {
  if (!s || n < 0 || n > s->cfg.max_seqs || (n > 0 && !seq_ids)) return PKV_ERR_ARG;
  int rc = pkv_step_wait(s);
  if (rc != PKV_OK || n == 0) return rc;
  const pkv_step_config &c = s->cfg;
  const long long cap = static_cast<long long>(c.max_blocks_per_seq) * c.block_size;
  int max_len = 0;  // every length after this step's append
  for (int i = 0; i < n; ++i) {
    const int64_t len = pkv_seq_len(s->alloc, seq_ids[i]);
    if (len < 0) return static_cast<int>(len);
    if (len + c.q_len > cap) return PKV_ERR_RANGE;
    max_len = len + c.q_len > max_len ? static_cast<int>(len + c.q_len) : max_len;
  }
  // The work list (q_len 1) depends on the lengths after the append, which the
  // checks above already know; its partition size keys the graphs.
  auto *items = reinterpret_cast<int32_t *>(s->hs + s->lay.items_offset);
  auto *tables = reinterpret_cast<int32_t *>(s->hs + s->lay.tables_offset);
  auto *lens = reinterpret_cast<int32_t *>(s->hs + s->lay.lens_offset);
  int count = 0, partition = c.partition_size;
  if (c.q_len == 1) {
    for (int i = 0; i < n; ++i) lens[i] = static_cast<int32_t>(pkv_seq_len(s->alloc, seq_ids[i]) + c.q_len);
    // With partition_size 0 the list picks its partition from a schedule model;
    // the lengths move by one token a step, so the pick is kept for a while
    // and made again every kRepick steps or when the batch size changes.
    int want = c.partition_size;
    if (want == 0 && s->auto_part > 0 && s->auto_n == n && s->auto_age < kRepick) want = s->auto_part;
    // When the model picks, it may go past 2048-token partitions only if no
    // block serves two sequences: the tables before this step's append tell
    // (an append never makes a block shared), filled here into the staging
    // rows that the tables after the append overwrite below.
    const int32_t *share_tables = nullptr;
    if (want == 0) {
      std::vector<int32_t> pre_lens(static_cast<size_t>(n));
      if (pkv_block_table(s->alloc, seq_ids, n, tables, c.max_blocks_per_seq, pre_lens.data()) == PKV_OK)
        share_tables = tables;
    }
    // cannot fail: the lengths fit the tables and the list its segment (partitions of at least 768 tokens)
    if ((rc = pkv_decode_items(lens, share_tables, c.max_blocks_per_seq, n, c.num_kv_heads, c.head_dim, c.block_size,
                               want, items, s->lay.max_items, &count)) != PKV_OK)
      return rc;
    partition = items[1];
    count = items[0];  // the merge list follows the items; the decode's grid is the items
    if (c.partition_size == 0) {
      s->auto_age = want == 0 ? 0 : s->auto_age + 1;
      s->auto_part = partition;
      s->auto_n = n;
    }
  }
  // Everything that can fail without a CUDA fault (a graph capture included)
  // happens before the allocator changes; the append is the last host step.
  cudaStream_t st = pkv::as_stream(stream);
  cudaGraphExec_t exec = nullptr;
  const int part = partition > 0 ? partition : s->part;
  if (c.use_graph) {
    const int parts = max_len > 0 ? (max_len + part - 1) / part : 1;
    // the work list of any step with this key has at most n x KV heads x parts items
    const int most = c.q_len == 1 ? n * c.num_kv_heads * parts : 0;
    const int grid = c.q_len == 1 ? std::min(most, (count + kGridGranule - 1) / kGridGranule * kGridGranule) : 0;
    const auto key = std::make_tuple(n, parts, part, grid);
    auto it = s->graphs.find(key);
    if (it == s->graphs.end()) {
      if (static_cast<int>(s->graphs.size()) >= kMaxGraphs) drop_graphs(s);
      const long long bound = static_cast<long long>(parts) * part;
      rc = capture(s, n, bound < cap ? static_cast<int>(bound) : static_cast<int>(cap), grid, partition, &exec);
      if (rc != PKV_OK) return rc;
      it = s->graphs.emplace(key, exec).first;
    }
    exec = it->second;
  }
  auto *slots = reinterpret_cast<int64_t *>(s->hs + s->lay.slots_offset);
  if ((rc = pkv_seq_append_batch(s->alloc, seq_ids, n, c.q_len, slots)) != PKV_OK) return rc;
  // cannot fail: every id is resident (the append took it) and its table has room (checked above)
  if ((rc = pkv_block_table(s->alloc, seq_ids, n, tables, c.max_blocks_per_seq, lens)) != PKV_OK) return rc;
  if (c.q_len == 1) {  // the first blocks of the items, now that the tables are filled
    const int part_blocks = partition / c.block_size;
    for (int i = 1; i <= count; ++i) {
      int32_t *it = items + 4 * i;
      const int seq = it[0], pt = static_cast<int>(static_cast<uint32_t>(it[1]) >> 16);
      const long long e = static_cast<long long>(pt) * part_blocks;
      it[3] = it[2] > 0 && e < c.max_blocks_per_seq ? tables[static_cast<size_t>(seq) * c.max_blocks_per_seq + e] : -1;
    }
  }

  if (exec) {
    const cudaError_t e = cudaGraphLaunch(exec, st);
    if (e != cudaSuccess) return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  } else if ((rc = enqueue(s, st, n, max_len, count, partition)) != PKV_OK) {
    return rc;
  }
  const cudaError_t e = cudaEventRecord(s->done, st);
  if (e != cudaSuccess) return pkv::set_cuda_error(e), PKV_ERR_CUDA;
  s->pending = true;
  return PKV_OK;
}

}  // extern "C"
